// gemm_kernel.cuh -- C = A B (bf16 in, fp32 accumulate in TMEM, bf16 out) on
// the sm_103a tensor cores.  Used for the two projections of the multi-head
// layer: the fused QKV projection X W_QKV ("Self-Attention 机制", section
// "五步计算": the three projections merged into one GEMM) and the output
// projection Concat(heads) W_O.
//
//   A [M, K] row-major (K-major operand), B [K, N] row-major (N-major operand),
//   C [M, N] row-major.  Tiles of 256 x 256 computed by a pair of CTAs with
//   the two-SM form of tcgen05.mma (cta_group::2), K blocks of 64.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gb300 {

constexpr int GEMM_BM = 256;        // rows of a tile: 128 in each CTA of the pair
constexpr int GEMM_BM_CTA = 128;
constexpr int GEMM_BN = 256;        // columns of a tile: B split 128 / 128 over the pair
constexpr int GEMM_BN_CTA = 128;
constexpr int GEMM_BK = 64;
constexpr int GEMM_STAGES = 7;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t GEMM_TMEM_COLS = 512;
enum : unsigned int { GEMM_STATUS_TIMEOUT = 1u };

struct GemmLayout {
  static constexpr int A_BYTES = GEMM_BM_CTA * GEMM_BK * 2;    // 16 KB: this CTA's 128 rows
  static constexpr int B_CHUNK = GEMM_BK * 64 * 2;             // 64 K-rows x 64 N = 8 KB
  static constexpr int B_BYTES = GEMM_BK * GEMM_BN_CTA * 2;    // 16 KB: this CTA's 128 columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // per CTA
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = GEMM_STAGES * A_BYTES;
  static constexpr int BAR_OFF = B_OFF + GEMM_STAGES * B_BYTES;
  static constexpr int B_FULL = 0;                       // used in the even CTA
  static constexpr int B_EMPTY = GEMM_STAGES;            // both CTAs
  static constexpr int B_ACC_FULL = 2 * GEMM_STAGES;     // both CTAs
  static constexpr int B_ACC_EMPTY = B_ACC_FULL + 2;     // used in the even CTA
  static constexpr int B_DRAIN = B_ACC_EMPTY + 2;
  static constexpr int N_BARS = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
};

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  // The tile list: the first n_full tiles of the N-fastest order at full
  // width, then the rest split into two halves of GEMM_BN / 2 columns each
  // (entries n_full + 2 i and n_full + 2 i + 1), n_list entries in all.
  // The host splits the tiles of a last, partial wave when the halves still
  // fit in one wave, so that wave takes half as long.
  int n_full, n_list;
  __nv_bfloat16* C;
  int c_v8;  // C is 32-byte aligned: the epilogue writes 32-byte pieces
  unsigned int* status;
  unsigned long long wait_limit_ns;
};

// Output corner of list entry `tile`; returns its width in columns.
__device__ __forceinline__ int gemm_tile_coords(const GemmParams& p, int tile, int& m0, int& n0) {
  int t = tile, half = -1;
  if (tile >= p.n_full) {
    const int h = tile - p.n_full;
    t = p.n_full + (h >> 1);
    half = h & 1;
  }
  // N-fastest: the pairs of a wave share few rows of A, so the first wave
  // does not read all of A from DRAM at once
  const int mt = t / p.n_tiles;
  const int nt = t % p.n_tiles;
  m0 = mt * GEMM_BM;
  n0 = nt * GEMM_BN;
  if (half < 0) return GEMM_BN;
  n0 += half * (GEMM_BN / 2);
  return GEMM_BN / 2;
}

// One cluster = one pair of CTAs on a TPC; the pair computes 256 x 256 output
// tiles, persistent over the tile list.  Per CTA of the pair:
//   warp 0      TMA producer (one thread): its 128 rows of A and its 128
//               columns of B into a 7-stage ring; the completion of both
//               CTAs' loads is counted on the even CTA's full-barrier
//   warp 1      TMEM (both CTAs allocate the pair's 512 columns together);
//               in the even CTA also the MMA issuer (whole warp, one elected
//               lane issues tcgen05.mma.cta_group::2 with M = N = 256; its
//               commits arrive on the barriers of both CTAs)
//   warps 2-5   epilogue of this CTA's 128 rows: TMEM -> bf16 -> global
//               memory, each lane writing its row in whole 32-byte sectors;
//               the four warps of each CTA release an accumulator with one
//               arrival each on the even CTA's accumulator-empty barrier
// The epilogue of one tile runs while the next tile's operands stream in.
// Staging C in shared memory for TMA tensor stores made those stores compete
// with the operand loads (the tensor pipe idled ~8% more on the QKV shape);
// direct stores of whole sectors do not, and the freed 32 KB hold a seventh
// stage, which hides more of the DRAM latency of A's first reads.
// Per SM and 64-deep K block the tensor core reads 32 KB of operands from
// shared memory for 2 x 128 x 256 x 64 FLOPs, two thirds of what a one-CTA
// 128 x 256 tile needs.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using L = GemmLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: its peer
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int n_pairs = static_cast<int>(gridDim.x >> 1);
  const int n_tiles_total = p.n_list;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GEMM_STAGES; ++s) {
      mbar_init(&bars[L::B_FULL + s], 1);    // the even CTA's producer arrives (+ both CTAs' bytes)
      mbar_init(&bars[L::B_EMPTY + s], 1);   // one multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars[L::B_ACC_FULL + a], 1);  // one multicast commit
      mbar_init(&bars[L::B_ACC_EMPTY + a], 8);  // 4 epilogue warps x 2 CTAs
    }
    mbar_init(&bars[L::B_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, GEMM_TMEM_COLS);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised and the pair's TMEM is allocated
  // before either CTA signals the other
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns, GEMM_STATUS_TIMEOUT};
  // Set-up done (on-chip only).  Behind a dependent launch this overlapped
  // the previous kernel's tail; nothing in global memory is touched before
  // that kernel has completed.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint32_t full0 = mapa_shared(smem_u32(&bars[L::B_FULL]), 0u);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < n_tiles_total; tile += n_pairs) {
        int m0, n0;
        const int cw = gemm_tile_coords(p, tile, m0, n0) / 2;  // B columns this CTA stages
        const int row = m0 + static_cast<int>(rank) * GEMM_BM_CTA;
        const int col = n0 + static_cast<int>(rank) * cw;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int s = static_cast<int>(it % GEMM_STAGES);
          if (it >= static_cast<uint32_t>(GEMM_STAGES)) {
            ok = mbar_wait(&bars[L::B_EMPTY + s], ((it / GEMM_STAGES) - 1u) & 1u, ctl);
            if (!ok) break;
          }
          // the even CTA's full-barrier counts the bytes of both CTAs; the
          // odd CTA's bytes may land before this expect_tx (the count then
          // runs below zero until it does, and the phase cannot complete
          // without this arrival)
          if (rank == 0)
            mbar_arrive_expect_tx(&bars[L::B_FULL + s], 2 * (L::A_BYTES + (cw / 64) * L::B_CHUNK));
          const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
          tma_load_2d_pair(smem + L::A_OFF + s * L::A_BYTES, &tmA, fb, kb * GEMM_BK, row);
          for (int c = 0; c < cw / 64; ++c)
            tma_load_2d_pair(smem + L::B_OFF + s * L::B_BYTES + c * L::B_CHUNK, &tmB, fb,
                             col + 64 * c, kb * GEMM_BK);
        }
      }
      // Unwind: every commit that arrives on this CTA's empty-barriers, and
      // (even CTA) the loads of both CTAs, must have landed before the pair
      // leaves; on the normal path these phases completed long ago.
      for (int s = 0; s < GEMM_STAGES; ++s) {
        if (it <= static_cast<uint32_t>(s)) continue;
        const uint32_t n_s = (it - s + GEMM_STAGES - 1) / GEMM_STAGES;
        if (rank == 0) mbar_wait_drain(&bars[L::B_FULL + s], (n_s - 1u) & 1u, ctl.limit_ns);
        mbar_wait_drain(&bars[L::B_EMPTY + s], (n_s - 1u) & 1u, ctl.limit_ns);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      // The whole warp waits and computes operands; one elected lane issues,
      // so the operands stay warp-uniform and each MMA issues quickly.
      constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, GEMM_BN, true);
      constexpr uint32_t IDESC_HALF = idesc_bf16_f32(GEMM_BM, GEMM_BN / 2, true);
      constexpr unsigned FULL = 0xffffffffu;
      constexpr uint16_t BOTH = 0x3;
      const uint64_t a_desc = smem_desc_sw128(smem_u32(smem + L::A_OFF), 16, 1024);
      const uint64_t b_desc = smem_desc_sw128(smem_u32(smem + L::B_OFF), L::B_CHUNK, 1024);
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < n_tiles_total; tile += n_pairs, ++tcount) {
        const uint32_t acc = tcount & 1u;
        if (tcount >= 2u) {
          ok = __all_sync(FULL, mbar_wait(&bars[L::B_ACC_EMPTY + acc], ((tcount >> 1) - 1u) & 1u, ctl));
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t d_tmem = tmem + acc * GEMM_BN;
        int m0, n0;
        const uint32_t idesc =
            gemm_tile_coords(p, tile, m0, n0) == GEMM_BN ? IDESC : IDESC_HALF;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int s = static_cast<int>(it % GEMM_STAGES);
          ok = __all_sync(FULL, mbar_wait(&bars[L::B_FULL + s], (it / GEMM_STAGES) & 1u, ctl));
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = a_desc + static_cast<uint64_t>((s * L::A_BYTES) >> 4);
          const uint64_t bd = b_desc + static_cast<uint64_t>((s * L::B_BYTES) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < GEMM_BK / 16; ++kk)
              mma_bf16_ss_pair(d_tmem, ad + static_cast<uint64_t>((kk * 32) >> 4),
                               bd + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
                               (kb > 0 || kk > 0) ? 1u : 0u);
            mma_commit_pair_multicast(&bars[L::B_EMPTY + s], BOTH);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) mma_commit_pair_multicast(&bars[L::B_ACC_FULL + acc], BOTH);
        __syncwarp();
      }
      if (elect_one()) mma_commit_pair(&bars[L::B_DRAIN]);
      __syncwarp();
      mbar_wait_drain(&bars[L::B_DRAIN], 0u, ctl.limit_ns);
    }
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const int wq = warp & 3;  // TMEM lane quarter = rows 32 wq .. 32 wq + 31 of this CTA
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&bars[L::B_ACC_EMPTY]), 0u);
    uint32_t tcount = 0;
    bool ok = true;
    for (int tile = pair; tile < n_tiles_total; tile += n_pairs, ++tcount) {
      const uint32_t acc = tcount & 1u;
      ok = mbar_wait(&bars[L::B_ACC_FULL + acc], (tcount >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int m0, n0;
      const int width = gemm_tile_coords(p, tile, m0, n0);
      const int row0 = m0 + static_cast<int>(rank) * GEMM_BM_CTA + wq * 32;
      // M is a multiple of 128: this warp's 32 rows lie wholly inside or past M
      const bool rows_in = row0 < p.M;
#pragma unroll 1
      for (int c = 0; c < width / 64; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tmem + acc * GEMM_BN + lane_base + c * 64u, r0);
        tmem_ld_32x32b_x32(tmem + acc * GEMM_BN + lane_base + c * 64u + 32u, r1);
        tmem_ld_wait(r0);
        reg_fence(r1);
        if (rows_in) {
          // row `lane` of C, columns n0 + 64 c .. + 63
          __nv_bfloat16* crow = p.C + static_cast<size_t>(row0 + lane) * p.N + n0 + 64 * c;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t* f = (i < 2) ? &r0[16 * i] : &r1[16 * (i - 2)];
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__uint_as_float(f[2 * k]), __uint_as_float(f[2 * k + 1]));
            if (p.c_v8) {
              st_global_v8(crow + 16 * i, w);
            } else {
              st_global_v4(crow + 16 * i, w[0], w[1], w[2], w[3]);
              st_global_v4(crow + 16 * i + 8, w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + acc * 8u);
    }
  }

  // Neither CTA leaves (or frees TMEM) while the other may still signal it.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, GEMM_TMEM_COLS);
  }
}

}  // namespace gb300

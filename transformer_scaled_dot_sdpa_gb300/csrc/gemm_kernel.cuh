// gemm_kernel.cuh -- C = A B (bf16 in, fp32 accumulate in TMEM, bf16 out) on
// the sm_103a tensor cores.  Used for the two projections of the multi-head
// layer: the fused QKV projection X W_QKV ("Self-Attention 机制", section
// "五步计算": the three projections merged into one GEMM) and the output
// projection Concat(heads) W_O.
//
//   A [M, K] row-major (K-major operand), B [K, N] row-major (N-major operand),
//   C [M, N] row-major.  Tiles of 128 x 256, K blocks of 64.
//
// CTA organisation (persistent, one CTA per SM):
//   warp 0      TMA producer (one thread): A and B tiles into a 4-stage ring
//   warp 1      MMA issuer (whole warp, one elected lane issues) + TMEM
//               owner; two 256-column fp32 accumulators so the epilogue of
//               one tile overlaps the main loop of the next
//   warps 2-5   epilogue: TMEM -> registers -> bf16 -> global, one row each
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gb300 {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BN = 256;
constexpr int GEMM_BK = 64;
constexpr int GEMM_STAGES = 4;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t GEMM_TMEM_COLS = 512;
enum : unsigned int { GEMM_STATUS_TIMEOUT = 1u };

struct GemmLayout {
  static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;        // 16 KB
  static constexpr int B_CHUNK = GEMM_BK * 64 * 2;             // 64 K-rows x 64 N = 8 KB
  static constexpr int B_BYTES = GEMM_BK * GEMM_BN * 2;        // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = GEMM_STAGES * A_BYTES;
  static constexpr int BAR_OFF = B_OFF + GEMM_STAGES * B_BYTES;
  static constexpr int B_FULL = 0;
  static constexpr int B_EMPTY = GEMM_STAGES;
  static constexpr int B_ACC_FULL = 2 * GEMM_STAGES;
  static constexpr int B_ACC_EMPTY = B_ACC_FULL + 2;
  static constexpr int B_DRAIN = B_ACC_EMPTY + 2;
  static constexpr int N_BARS = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
};

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  __nv_bfloat16* C;
  unsigned int* status;
  unsigned long long wait_limit_ns;
};

__device__ __forceinline__ void gemm_tile_coords(const GemmParams& p, int tile, int& m0, int& n0) {
  const int mt = tile % p.m_tiles;
  const int nt = tile / p.m_tiles;
  m0 = mt * GEMM_BM;
  n0 = nt * GEMM_BN;
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
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
  const int n_tiles_total = p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GEMM_STAGES; ++s) {
      mbar_init(&bars[L::B_FULL + s], 1);
      mbar_init(&bars[L::B_EMPTY + s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars[L::B_ACC_FULL + a], 1);
      mbar_init(&bars[L::B_ACC_EMPTY + a], 128);
    }
    mbar_init(&bars[L::B_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, GEMM_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns, GEMM_STATUS_TIMEOUT};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x) {
        int m0, n0;
        gemm_tile_coords(p, tile, m0, n0);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int s = static_cast<int>(it % GEMM_STAGES);
          if (it >= static_cast<uint32_t>(GEMM_STAGES)) {
            ok = mbar_wait(&bars[L::B_EMPTY + s], ((it / GEMM_STAGES) - 1u) & 1u, ctl);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&bars[L::B_FULL + s], L::STAGE_BYTES);
          tma_load_2d(smem + L::A_OFF + s * L::A_BYTES, &tmA, &bars[L::B_FULL + s],
                      kb * GEMM_BK, m0);
#pragma unroll
          for (int c = 0; c < GEMM_BN / 64; ++c)
            tma_load_2d(smem + L::B_OFF + s * L::B_BYTES + c * L::B_CHUNK, &tmB,
                        &bars[L::B_FULL + s], n0 + 64 * c, kb * GEMM_BK);
        }
      }
      for (int s = 0; s < GEMM_STAGES; ++s) {
        if (it <= static_cast<uint32_t>(s)) continue;
        const uint32_t n_s = (it - s + GEMM_STAGES - 1) / GEMM_STAGES;
        mbar_wait_drain(&bars[L::B_FULL + s], (n_s - 1u) & 1u, ctl.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The whole warp waits and computes operands; one elected lane issues,
    // so the operands stay warp-uniform and each MMA issues quickly.
    constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, GEMM_BN, true);
    constexpr unsigned FULL = 0xffffffffu;
    const uint64_t a_desc = smem_desc_sw128(smem_u32(smem + L::A_OFF), 16, 1024);
    const uint64_t b_desc = smem_desc_sw128(smem_u32(smem + L::B_OFF), L::B_CHUNK, 1024);
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles_total; tile += gridDim.x, ++tcount) {
      const uint32_t acc = tcount & 1u;
      if (tcount >= 2u) {
        ok = __all_sync(FULL, mbar_wait(&bars[L::B_ACC_EMPTY + acc], ((tcount >> 1) - 1u) & 1u, ctl));
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t d_tmem = tmem + acc * GEMM_BN;
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
            mma_bf16_ss(d_tmem, ad + static_cast<uint64_t>((kk * 32) >> 4),
                        bd + static_cast<uint64_t>((kk * 2048) >> 4), IDESC,
                        (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars[L::B_EMPTY + s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&bars[L::B_ACC_FULL + acc]);
      __syncwarp();
    }
    if (elect_one()) mma_commit(&bars[L::B_DRAIN]);
    __syncwarp();
    mbar_wait_drain(&bars[L::B_DRAIN], 0u, ctl.limit_ns);
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int row = static_cast<int>((warp & 3) * 32 + lane);  // TMEM lane = tile row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t tcount = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles_total; tile += gridDim.x, ++tcount) {
      const uint32_t acc = tcount & 1u;
      ok = mbar_wait(&bars[L::B_ACC_FULL + acc], (tcount >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int m0, n0;
      gemm_tile_coords(p, tile, m0, n0);
      __nv_bfloat16* crow = p.C + static_cast<long long>(m0 + row) * p.N + n0;
#pragma unroll 1
      for (int cc = 0; cc < GEMM_BN / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + acc * GEMM_BN + lane_base + cc * 32u, r);
        tmem_ld_wait(r);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_global_v4(crow + cc * 32 + i * 8, w[4 * i], w[4 * i + 1], w[4 * i + 2],
                       w[4 * i + 3]);
      }
      tc_fence_before();
      mbar_arrive(&bars[L::B_ACC_EMPTY + acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, GEMM_TMEM_COLS);
  }
}

}  // namespace gb300

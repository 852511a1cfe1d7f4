// attn_fwd_t1_kernel.cuh -- attention forward, one 128-query tile per work
// item, with Q and P held in tensor memory and a double-buffered S, for sm_103a.
//
// It computes the same thing as attn_fwd_kernel.cuh (online softmax of
// "Self-Attention 机制", section "Softmax 的数值稳定性与 Online Softmax"; the n x
// n scores never leave the chip; key tiles above the causal diagonal are
// skipped) with a different schedule.  One thread issues a tcgen05.mma only
// about every 100-130 cycles, while a 128 x 128 x 16 step is 64 cycles of
// tensor time, so the tensor core needs two issuers working at once, and the
// softmax should never wait for an MMA to be issued:
//
//   S issuer  (warp 8):  S(j) = Q K_j^T into buffer j % 2 as soon as K_j has
//                        landed and P(j-2) V has been consumed from that
//                        buffer, i.e. up to two tiles ahead of the softmax
//   PV issuer (warp 10): O += P(j) V_j once the softmax has written P(j)
//   TMA       (warp 9):  Q and K through one ring of shared-memory slots
//             (warp 11): V through a second ring
//   softmax   (warps 0-7): two threads per query row (keys 0..63 / 64..127 of
//                        each tile); the two partial row maxima are swapped
//                        through shared memory
//
// P(j) is written over S(j) in its own buffer, so P is double-buffered too and
// the softmax never waits for a P.V before writing P; it waits only when it
// has to rescale O.  The row-max exchange is speculative: the exponentials of
// tile j are computed with the running maximum both halves already agree on,
// and redone only in the rare case that the tile raises it by more than the
// rescale threshold.
//
// Each issuer commits once per tile (S_FULL, PV_DONE).  K slots are handed
// back to the producer by one softmax thread once it has seen S_FULL, V slots
// by the S issuer once it has seen PV_DONE, which keeps the ~250-cycle commit
// off the issuers.
//
// TMEM (128 lanes x 512 columns of 32 bit):
//   [  0, D/2)   Q as bf16 pairs (A operand of S = Q K^T), copied from shared
//                memory with tcgen05.cp
//   [ 64, 192)   buffer 0: S(j) in fp32, then P(j) as bf16 pairs in its
//                first 64 columns (A operand of O += P V)
//   [192, 320)   buffer 1
//   [384, 384+D) O accumulator (fp32)
// An MMA never writes columns another MMA may still read: S(j+2) goes into a
// buffer only after P(j) V has completed; every ordering is an mbarrier.
#pragma once

#include <cuda_bf16.h>

#include "attn_fwd_kernel.cuh"
#include "ptx.cuh"

namespace gb300 {

constexpr int T1_THREADS = 384;
constexpr int T1_ROWS = 128;  // query rows per work item

template <int D>
struct T1Layout {
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;  // 128 rows x 64 bf16
  static constexpr int NCHUNK = D / 64;
  // Q passes through the K ring (it is needed only until it is in TMEM).
  static constexpr int KQ_STAGES = (D == 128) ? 3 : 6;
  static constexpr int V_STAGES = (D == 128) ? 3 : 6;
  static constexpr int KQ_OFF = 0;
  static constexpr int V_OFF = KQ_OFF + KQ_STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + V_STAGES * TILE_BYTES;
  static constexpr int B_KQ_FULL = 0;
  static constexpr int B_KQ_EMPTY = B_KQ_FULL + KQ_STAGES;
  static constexpr int B_V_FULL = B_KQ_EMPTY + KQ_STAGES;
  static constexpr int B_V_EMPTY = B_V_FULL + V_STAGES;
  // per S/P buffer: S(j) computed, P(j) written, P(j) V completed
  static constexpr int B_S_FULL = B_V_EMPTY + V_STAGES;  // [2]
  static constexpr int B_P_FULL = B_S_FULL + 2;           // [2]
  static constexpr int B_PV_DONE = B_P_FULL + 2;          // [2]
  static constexpr int B_DRAIN = B_PV_DONE + 2;  // [2], one per issuer
  static constexpr int B_XCHG = B_DRAIN + 2;     // [4], one per TMEM lane quarter
  static constexpr int N_BARS = B_XCHG + 4;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int XMAX_OFF = MISC_OFF + 16;               // float [2 parity][2 halves][128]
  static constexpr int XSUM_OFF = XMAX_OFF + 2 * 2 * 128 * 4;  // float [2 halves][128][2]
  static constexpr int SMEM_BYTES = XSUM_OFF + 2 * 128 * 2 * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
  // TMEM columns
  static constexpr uint32_t TQ = 0, TS0 = 64, TO = 384;
};

struct T1Item {
  int b, h, kvh, row0, nkv, kv_len, kv_len_raw;
};

// Item k of this CTA: one (b, h, 128-row query tile), heaviest first, dealt
// in a boustrophedon order like attn_get_item.
__device__ __forceinline__ bool t1_get_item(const AttnParams& p, int k, T1Item& it) {
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  const long long w = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (w >= p.n_items) return false;
  const int BH = p.B * p.H;
  const int rank = static_cast<int>(w / BH);
  const int bh = static_cast<int>(w - static_cast<long long>(rank) * BH);
  const int qt = p.n_qblocks - 1 - rank;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  it.kvh = it.h / p.kv_group;
  int kv_len = p.Lk;
  it.kv_len_raw = p.Lk;
  if (p.mask_kind & ATTN_MASK_PADDING_BIT) {
    const int raw = p.kv_lens[it.b];
    it.kv_len_raw = raw;
    kv_len = raw < 0 ? 0 : (raw > p.Lk ? p.Lk : raw);
  }
  it.kv_len = kv_len;
  it.row0 = qt * T1_ROWS;
  int n = 0;
  const bool all_padded = (p.mask_kind & ATTN_MASK_PADDING_BIT) && it.row0 >= kv_len;
  if (it.row0 < p.Lq && !all_padded) {
    int lim = kv_len;
    if (p.mask_kind & ATTN_MASK_CAUSAL_BIT) {
      const int last = min(it.row0 + T1_ROWS - 1, p.Lq - 1);
      lim = min(lim, max(last + 1 + p.causal_offset, 0));
    }
    n = (lim + ATTN_BLOCK_N - 1) / ATTN_BLOCK_N;
  }
  it.nkv = n;
  return true;
}

// Waits for the last load into each slot of a ring before the CTA exits (n
// loads were issued in ring order; `skip` is a running index never loaded).
__device__ __forceinline__ void t1_drain_ring(uint64_t* full, int stages, uint32_t n,
                                              long long skip, uint64_t limit_ns) {
  for (int s = 0; s < stages; ++s) {
    if (n <= static_cast<uint32_t>(s)) continue;
    const uint32_t uses = (n - s + stages - 1) / stages;
    const uint32_t last = s + (uses - 1u) * stages;
    if (static_cast<long long>(last) != skip) mbar_wait_drain(&full[s], (uses - 1u) & 1u, limit_ns);
  }
}

// ---------------------------------------------------------------------------
// TMA producers
// ---------------------------------------------------------------------------
// Q, then the item's K tiles, through the KQ ring.  `kv_it` counts K tiles
// only (the running index the debug hook refers to); `ring` counts slots.
template <int D>
__device__ __forceinline__ void t1_qk_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                               const AttnParams& p, uint8_t* smem,
                                               uint64_t* bars, const WaitCtl& ctl) {
  using L = T1Layout<D>;
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  uint32_t ring = 0, kv_it = 0;
  long long skip_ring = -1;
  bool ok = true;
  T1Item it;
  for (int k = 0; ok && t1_get_item(p, k, it); ++k) {
    if (it.nkv == 0) continue;
    for (int j = -1; j < it.nkv; ++j, ++ring) {
      const int s = static_cast<int>(ring % L::KQ_STAGES);
      const uint32_t reuse = ring / L::KQ_STAGES;
      if (reuse > 0) {
        ok = mbar_wait(&bars[L::B_KQ_EMPTY + s], (reuse - 1u) & 1u, ctl);
        if (!ok) break;
      }
      uint8_t* dst = smem + L::KQ_OFF + s * L::TILE_BYTES;
      if (j < 0) {
        mbar_arrive_expect_tx(&bars[L::B_KQ_FULL + s], L::TILE_BYTES);
        for (int c = 0; c < L::NCHUNK; ++c)
          attn_load_tile(tmQ, dst + c * L::CHUNK_BYTES, &bars[L::B_KQ_FULL + s], 64 * c,
                         it.row0, it.h, it.b, p.packed);
        continue;
      }
      const bool skip = static_cast<long long>(kv_it++) == p.debug_skip_kv_load;
      if (skip) {
        skip_ring = ring;
        continue;
      }
      mbar_arrive_expect_tx(&bars[L::B_KQ_FULL + s], L::TILE_BYTES);
      for (int c = 0; c < L::NCHUNK; ++c)
        attn_load_tile(tmK, dst + c * L::CHUNK_BYTES, &bars[L::B_KQ_FULL + s], 64 * c,
                       j * ATTN_BLOCK_N, it.kvh, it.b, p.packed);
    }
  }
  // Unwind: every load this thread issued lands before the CTA exits.
  t1_drain_ring(&bars[L::B_KQ_FULL], L::KQ_STAGES, ring, skip_ring, ctl.limit_ns);
}

template <int D>
__device__ __forceinline__ void t1_v_producer(const CUtensorMap* tmV, const AttnParams& p,
                                              uint8_t* smem, uint64_t* bars, const WaitCtl& ctl) {
  using L = T1Layout<D>;
  tma_prefetch_desc(tmV);
  uint32_t kv_it = 0;
  bool ok = true;
  T1Item it;
  for (int k = 0; ok && t1_get_item(p, k, it); ++k) {
    for (int j = 0; j < it.nkv; ++j, ++kv_it) {
      const int s = static_cast<int>(kv_it % L::V_STAGES);
      const uint32_t reuse = kv_it / L::V_STAGES;
      if (reuse > 0) {
        ok = mbar_wait(&bars[L::B_V_EMPTY + s], (reuse - 1u) & 1u, ctl);
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&bars[L::B_V_FULL + s], L::TILE_BYTES);
      for (int c = 0; c < L::NCHUNK; ++c)
        attn_load_tile(tmV, smem + L::V_OFF + s * L::TILE_BYTES + c * L::CHUNK_BYTES,
                       &bars[L::B_V_FULL + s], 64 * c, j * ATTN_BLOCK_N, it.kvh, it.b, p.packed);
    }
  }
  t1_drain_ring(&bars[L::B_V_FULL], L::V_STAGES, kv_it, -1, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// S issuer: Q -> TMEM once per item, then S(j) = Q K_j^T into buffer j % 2
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void t1_s_role(const AttnParams& p, uint8_t* smem, uint64_t* bars,
                                          uint32_t tmem, const WaitCtl& ctl) {
  using L = T1Layout<D>;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(128, ATTN_BLOCK_N, false);
  const uint32_t ring_base = smem_u32(smem + L::KQ_OFF);
  uint32_t ring = 0, s_idx = 0;
  bool ok = true;
  T1Item it;
  for (int k = 0; ok && t1_get_item(p, k, it); ++k) {
    if (it.kv_len_raw != it.kv_len) atomicOr(p.status, ATTN_STATUS_BAD_KVLEN);
    if (it.nkv == 0) continue;
    // Q of this item
    {
      const int s = static_cast<int>(ring % L::KQ_STAGES);
      ok = mbar_wait(&bars[L::B_KQ_FULL + s], (ring / L::KQ_STAGES) & 1u, ctl);
      if (!ok) break;
      if (s_idx > 0) {
        // the previous item's last S still reads the Q columns
        const uint32_t t = s_idx - 1u;
        ok = mbar_wait(&bars[L::B_S_FULL + (t & 1u)], (t >> 1) & 1u, ctl);
        if (!ok) break;
      }
      tc_fence_after();
      const uint32_t qa = ring_base + s * L::TILE_BYTES;
      // 128 rows x 16 bf16 (8 TMEM columns) per copy, K-major 128B-swizzled
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * L::CHUNK_BYTES + (kk & 3) * 32;
        tmem_cp_128x256b(tmem + L::TQ + kk * 8, smem_desc_sw128(qa + off, 16, 1024));
      }
      mma_commit(&bars[L::B_KQ_EMPTY + s]);  // the slot is free once the copies are done
      ++ring;
    }
    for (int j = 0; j < it.nkv; ++j, ++ring, ++s_idx) {
      const int s = static_cast<int>(ring % L::KQ_STAGES);
      ok = mbar_wait(&bars[L::B_KQ_FULL + s], (ring / L::KQ_STAGES) & 1u, ctl);
      if (!ok) break;
      const uint32_t buf = s_idx & 1u;
      if (s_idx >= 2) {
        // P(s_idx-2) V has read this buffer (and V_{s_idx-2}: free its slot)
        ok = mbar_wait(&bars[L::B_PV_DONE + buf], ((s_idx >> 1) - 1u) & 1u, ctl);
        if (!ok) break;
        mbar_arrive(&bars[L::B_V_EMPTY + (s_idx - 2u) % L::V_STAGES]);
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + L::TS0 + buf * 128u;
      const uint32_t ka = ring_base + s * L::TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * L::CHUNK_BYTES + (kk & 3) * 32;
        mma_bf16_ts(d_tmem, tmem + L::TQ + kk * 8, smem_desc_sw128(ka + off, 16, 1024), IDESC_S,
                    kk > 0 ? 1u : 0u);
      }
      mma_commit(&bars[L::B_S_FULL + buf]);
    }
  }
  // Unwind: all MMAs and copies issued by this thread complete before TMEM is freed.
  mma_commit(&bars[L::B_DRAIN + 0]);
  mbar_wait_drain(&bars[L::B_DRAIN + 0], 0u, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// P.V issuer: O += P(j) V_j
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void t1_pv_role(const AttnParams& p, uint8_t* smem, uint64_t* bars,
                                           uint32_t tmem, const WaitCtl& ctl) {
  using L = T1Layout<D>;
  constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
  const uint32_t v_base = smem_u32(smem + L::V_OFF);
  uint32_t kv_it = 0;
  bool ok = true;
  T1Item it;
  for (int k = 0; ok && t1_get_item(p, k, it); ++k) {
    for (int j = 0; j < it.nkv; ++j, ++kv_it) {
      const int s = static_cast<int>(kv_it % L::V_STAGES);
      ok = mbar_wait(&bars[L::B_V_FULL + s], (kv_it / L::V_STAGES) & 1u, ctl);
      if (!ok) break;
      const uint32_t buf = kv_it & 1u;
      ok = mbar_wait(&bars[L::B_P_FULL + buf], (kv_it >> 1) & 1u, ctl);
      if (!ok) break;
      tc_fence_after();
      const uint32_t va = v_base + s * L::TILE_BYTES;
      const uint32_t pa = tmem + L::TS0 + buf * 128u;
#pragma unroll
      for (int kk = 0; kk < ATTN_BLOCK_N / 16; ++kk)
        mma_bf16_ts(tmem + L::TO, pa + kk * 8,
                    smem_desc_sw128(va + kk * 2048, L::CHUNK_BYTES, 1024), IDESC_O,
                    (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&bars[L::B_PV_DONE + buf]);
    }
  }
  mma_commit(&bars[L::B_DRAIN + 1]);
  mbar_wait_drain(&bars[L::B_DRAIN + 1], 0u, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// softmax / correction / epilogue: 256 threads, two per query row
// ---------------------------------------------------------------------------
// p = 2^(s c - mb) for one thread's 64 scores, packed as bf16 pairs; sum_f is
// set to the fp32 sum of p, sum_b to the sum of the bf16-rounded p.
__device__ __forceinline__ void t1_exp_tile(const float (&s)[64], float c, float mb,
                                            uint32_t (&pk)[32], float& sum_f, float& sum_b) {
  const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-mb, -mb);
  uint64_t lf_a = 0ull, lf_b = 0ull;
  float lb_a = 0.f, lb_b = 0.f, lb_c = 0.f, lb_d = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float a0, a1, a2, a3;
    f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), c2, nm2), a0, a1);
    f2_unpack(f2_fma(f2_pack(s[2 * i + 2], s[2 * i + 3]), c2, nm2), a2, a3);
    const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
    const float p2 = ex2_approx(a2), p3 = ex2_approx(a3);
    pk[i] = pack_bf16x2(p0, p1);
    pk[i + 1] = pack_bf16x2(p2, p3);
    lf_a = f2_add(lf_a, f2_pack(p0, p1));
    lf_b = f2_add(lf_b, f2_pack(p2, p3));
    lb_a = add_bf16lo_f32(lb_a, pk[i]);
    lb_b = add_bf16hi_f32(lb_b, pk[i]);
    lb_c = add_bf16lo_f32(lb_c, pk[i + 1]);
    lb_d = add_bf16hi_f32(lb_d, pk[i + 1]);
  }
  float x0, x1;
  f2_unpack(f2_add(lf_a, lf_b), x0, x1);
  sum_f = x0 + x1;
  sum_b = (lb_a + lb_b) + (lb_c + lb_d);
}

// Thread (h, q, lane) owns row q * 32 + lane of the tile and keys / output
// columns of half h.  Thread 0 also returns K slots to the producer.
template <int D>
__device__ __forceinline__ void t1_softmax_role(const int h, const int q, const AttnParams& p,
                                                uint8_t* smem, uint64_t* bars, uint32_t tmem,
                                                const WaitCtl& ctl) {
  using L = T1Layout<D>;
  constexpr int DH = D / 2;  // output columns per thread
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const bool leader = threadIdx.x == 0;
  const int rloc = q * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t o_tmem = tmem + L::TO + lane_base + DH * h;
  float* xmax = reinterpret_cast<float*>(smem + L::XMAX_OFF);  // [par][h][128]
  float* xsum = reinterpret_cast<float*>(smem + L::XSUM_OFF);  // [h][128][2]
  uint64_t* xbar = &bars[L::B_XCHG + q];
  const float c = p.scale_log2;
  const bool causal = (p.mask_kind & ATTN_MASK_CAUSAL_BIT) != 0;
  const bool padding = (p.mask_kind & ATTN_MASK_PADDING_BIT) != 0;
  uint32_t n_t = 0;    // tiles consumed (S read, P written), over all items
  uint32_t x_cnt = 0;  // row exchanges
  uint32_t ring = 0;   // KQ ring position
  bool ok = true;
  T1Item it;
  for (int k = 0; ok && t1_get_item(p, k, it); ++k) {
    if (it.row0 >= p.Lq) continue;
    const int r = it.row0 + rloc;
    const int nkv = it.nkv;
    int limit = it.kv_len;
    if (causal) limit = min(limit, max(r + 1 + p.causal_offset, 0));
    const bool padded_row = padding && r >= it.kv_len;
    if (nkv > 0) ++ring;  // the item's Q slot
    float m = -INFINITY, l = 0.f, lb = 0.f;  // l, lb: this half's partial sums
    for (int j = 0; j < nkv; ++j, ++n_t, ++ring) {
      const uint32_t buf = n_t & 1u;
      ok = mbar_wait(&bars[L::B_S_FULL + buf], (n_t >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (leader) mbar_arrive(&bars[L::B_KQ_EMPTY + ring % L::KQ_STAGES]);  // K_j read
      tc_fence_after();
      const uint32_t s_tmem = tmem + L::TS0 + buf * 128u + lane_base;
      uint32_t ra[32], rb[32];
      tmem_ld_32x32b_x32(s_tmem + 64u * h, ra);
      tmem_ld_32x32b_x32(s_tmem + 64u * h + 32u, rb);
      tmem_ld_wait(ra);
      reg_fence(rb);
      float s[64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(ra[i]);
        s[32 + i] = __uint_as_float(rb[i]);
      }
      const int nvalid = limit - j * ATTN_BLOCK_N - 64 * h;
      if (nvalid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = (i < nvalid) ? s[i] : -INFINITY;
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int i = 8; i < 64; i += 8) {
        mx0 = fmax3(mx0, s[i], s[i + 1]);
        mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
        mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
        mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
      }
      // Offer this half's maximum to the other half.  The arrive also orders
      // this half's S loads before the other half's P stores, which overwrite
      // part of them.
      const int par = static_cast<int>(x_cnt & 1u);
      xmax[(par * 2 + h) * 128 + rloc] = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      tc_fence_before();
      mbar_arrive(xbar);
      uint32_t pk[32];
      float sf = 0.f, sb = 0.f;
      // Speculatively, with the running maximum of the previous tiles (both
      // halves hold the same m).
      if (j > 0) t1_exp_tile(s, c, (m == -INFINITY) ? 0.f : m, pk, sf, sb);
      ok = mbar_wait(xbar, x_cnt & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++x_cnt;
      tc_fence_after();
      const float mx = fmaxf(xmax[(par * 2 + 0) * 128 + rloc], xmax[(par * 2 + 1) * 128 + rloc]);
      const float m_new = fmaxf(m, mx * c);
      // Both halves see the same m and m_new, so they decide alike.
      const bool need = m_new > m + ATTN_RESCALE_THRESHOLD;
      float alpha = 1.0f;
      if (need) {
        alpha = ex2_approx(m - m_new);
        l *= alpha;
        lb *= alpha;
        m = m_new;
      }
      if (j == 0 || __any_sync(0xffffffffu, need)) {
        const float mb = (m == -INFINITY) ? 0.f : m;
        t1_exp_tile(s, c, mb, pk, sf, sb);
      }
      l += sf;
      lb += sb;
      // O holds P(0..j-1) V in the old scale: rescale it once P(j-1) V is done
      if (__any_sync(0xffffffffu, need && j > 0)) {
        const uint32_t pb = (n_t - 1u) & 1u;
        ok = mbar_wait(&bars[L::B_PV_DONE + pb], ((n_t - 1u) >> 1) & 1u, ctl);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
        for (int cc = 0; cc < DH / 32; ++cc) {
          uint32_t ro[32];
          tmem_ld_32x32b_x32(o_tmem + cc * 32u, ro);
          tmem_ld_wait(ro);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(ro[2 * i]), __uint_as_float(ro[2 * i + 1])),
                             a2),
                      x0, x1);
            ro[2 * i] = __float_as_uint(x0);
            ro[2 * i + 1] = __float_as_uint(x1);
          }
          tmem_st_32x32b_x32(o_tmem + cc * 32u, ro);
        }
      }
      // P(j) over the first 64 columns of S(j)'s buffer
      tmem_st_32x32b_x32(s_tmem + 32u * h, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[L::B_P_FULL + buf]);
    }
    if (!ok) break;
    // epilogue: combine the halves' sums, wait for the last P.V, write O and LSE
    if (nkv > 0) {
      xsum[(h * 128 + rloc) * 2 + 0] = l;
      xsum[(h * 128 + rloc) * 2 + 1] = lb;
      mbar_arrive(xbar);
      ok = mbar_wait(xbar, x_cnt & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++x_cnt;
      l = xsum[(0 * 128 + rloc) * 2 + 0] + xsum[(1 * 128 + rloc) * 2 + 0];
      lb = xsum[(0 * 128 + rloc) * 2 + 1] + xsum[(1 * 128 + rloc) * 2 + 1];
      const uint32_t pb = (n_t - 1u) & 1u;
      ok = mbar_wait(&bars[L::B_PV_DONE + pb], ((n_t - 1u) >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
    }
    const bool in_range = r < p.Lq;
    const bool zero_row = padded_row || nkv == 0 || limit <= 0 || !(lb > 0.f);
    const float inv_l = zero_row ? 0.f : 1.0f / lb;
    __nv_bfloat16* orow = p.O + it.b * p.o_stride_b + it.h * p.o_stride_h +
                          static_cast<long long>(r) * p.o_stride_l + DH * h;
#pragma unroll
    for (int cc = 0; cc < DH / 32; ++cc) {
      uint32_t ro[32];
      if (nkv > 0) {
        tmem_ld_32x32b_x32(o_tmem + cc * 32u, ro);
        tmem_ld_wait(ro);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) ro[i] = 0u;
      }
      if (in_range) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = zero_row ? 0u
                          : pack_bf16x2(__uint_as_float(ro[2 * i]) * inv_l,
                                        __uint_as_float(ro[2 * i + 1]) * inv_l);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_global_v4(orow + cc * 32 + i * 8, w[4 * i], w[4 * i + 1], w[4 * i + 2],
                       w[4 * i + 3]);
      }
    }
    if (p.LSE != nullptr && in_range && h == 0) {
      const float lse = zero_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
      p.LSE[(static_cast<long long>(it.b) * p.H + it.h) * p.Lq + r] = lse;
    }
    // The next item's first P.V overwrites O.  It waits for P_FULL, which
    // these threads give only after the loads above have completed.
    tc_fence_before();
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(T1_THREADS, 1)
    attn_fwd_t1_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using L = T1Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::KQ_STAGES; ++s) {
      mbar_init(&bars[L::B_KQ_FULL + s], 1);
      mbar_init(&bars[L::B_KQ_EMPTY + s], 1);
    }
    for (int s = 0; s < L::V_STAGES; ++s) {
      mbar_init(&bars[L::B_V_FULL + s], 1);
      mbar_init(&bars[L::B_V_EMPTY + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[L::B_S_FULL + b], 1);
      mbar_init(&bars[L::B_P_FULL + b], 256);
      mbar_init(&bars[L::B_PV_DONE + b], 1);
      mbar_init(&bars[L::B_DRAIN + b], 1);
    }
    for (int x = 0; x < 4; ++x) mbar_init(&bars[L::B_XCHG + x], 64);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, ATTN_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns, ATTN_STATUS_TIMEOUT};

  // Register split as in attn_fwd_kernel: softmax warpgroups 216, control 72;
  // together exactly the 384 x 168 registers of the launch.
  if (warp >= 8) {
    reg_dealloc<ATTN_REGS_CONTROL>();
    if (warp == 8) {
      if (lane == 0) t1_s_role<D>(p, smem, bars, tmem, ctl);
      __syncwarp();
    } else if (warp == 9) {
      if (lane == 0) t1_qk_producer<D>(&tmQ, &tmK, p, smem, bars, ctl);
    } else if (warp == 10) {
      if (lane == 0) t1_pv_role<D>(p, smem, bars, tmem, ctl);
      __syncwarp();
    } else {
      if (lane == 0) t1_v_producer<D>(&tmV, p, smem, bars, ctl);
    }
  } else {
    reg_alloc<ATTN_REGS_SOFTMAX>();
    // warps w and w + 4 hold the two halves of the same 32 rows (lane quarter w % 4)
    t1_softmax_role<D>(warp >> 2, warp & 3, p, smem, bars, tmem, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, ATTN_TMEM_COLS);
  }
}

}  // namespace gb300

// attn_fwd_split_kernel.cuh -- attention forward, one 128-query tile per work
// item, its key tiles dealt alternately to two softmax warpgroups, for sm_103a.
//
// It computes the same thing as attn_fwd_kernel.cuh (online softmax of
// "Self-Attention 机制", section "Softmax 的数值稳定性与 Online Softmax"; the n x
// n scores never leave the chip; key tiles above the causal diagonal are
// skipped).  The softmax of a 128 x 128 score tile is bound by the
// exponential unit (16 exp2 per clock per SM), and a warpgroup that handles
// one tile from start to end leaves that unit idle while it loads scores,
// reduces maxima and stores P.  Here the tiles of a query tile are split by
// parity between two warpgroups, each with its own running maximum, sums and
// O accumulator (a split of the key range inside the CTA, merged at the end
// of the item the way partial softmaxes combine), so one group's
// exponentials overlap the other group's loads, reductions and stores:
//
//   S issuer  (warp 8):  S(t) = Q K_t^T into S buffer t % 2 once K_t has
//                        landed and P(t-2) V has consumed that buffer
//   PV issuer (warp 10): O_{t % 2} += P(t) V_t once P(t) is written
//   TMA       (warp 9):  Q (one slot per item) and K through a ring
//             (warp 11): V through a second ring
//   softmax   (warps 0-3 / 4-7): warpgroup g takes the tiles t with
//                        t % 2 == g, one thread per query row
//
// P(t) is written over S(t) in its buffer.  The K slot of a tile is returned
// by the warpgroup that reads its S, the V slot by the S issuer once the
// tile's P.V has completed, so each issuer commits once per tile.
//
// TMEM (128 lanes x 512 columns of 32 bit):
//   [  0, 128)   buffer 0: S in fp32, then P as bf16 pairs in columns 0..63
//   [128, 256)   buffer 1
//   [256, 256+D) O_0     [384, 384+D) O_1
#pragma once

#include <cuda_bf16.h>

#include "attn_fwd_kernel.cuh"
#include "ptx.cuh"

namespace gb300 {

constexpr int SPLIT_ROWS = 128;  // query rows per work item

struct SplitItem {
  int b, h, kvh, row0, nkv, kv_len, kv_len_raw;
  int coff;   // causal offset of the sequence (attn_causal_offset)
  int k0;     // first key of the item's key range
  int chunk;  // decode: slot of the item's partial result among its pair's
  int qrow;   // decode: flat index of the first packed Q row
};

// Split-KV decode plan, computed alike by every role of every CTA and by the
// combine kernel from kv_lens: the visible key tiles of all (sequence, K/V
// head) pairs, laid end to end in pair order, are cut into gridDim.x ranges of
// ceil(T / gridDim.x) tiles.  CTA c takes range c; each part of a pair inside
// the range is one work item, whose partial result goes to slot
// c - (first CTA of the pair).  Every CTA gets the same number of key tiles
// (within one), whatever the cache lengths.
__device__ __forceinline__ int decode_seq_tiles(const AttnParams& p, int b) {
  int len = p.Lk;
  if (p.mask_kind & ATTN_MASK_PADDING_BIT) {
    const int raw = p.kv_lens[b];
    len = raw < 0 ? 0 : (raw > p.Lk ? p.Lk : raw);
  }
  // keys the last query row may see bound those of every row of the pair
  if (p.mask_kind & ATTN_MASK_CAUSAL_BIT)
    len = min(len, max(p.Lq + attn_causal_offset(p, len), 0));
  return (len + ATTN_BLOCK_N - 1) / ATTN_BLOCK_N;
}

struct DecodeSplit {
  long long total;  // key tiles of all pairs
  long long share;  // key tiles per CTA range
};

__device__ __forceinline__ DecodeSplit decode_split(const AttnParams& p, int grid) {
  const int hkv = p.H / p.kv_group;
  long long total = 0;
  for (int b = 0; b < p.B; ++b) total += static_cast<long long>(hkv) * decode_seq_tiles(p, b);
  return {total, total > 0 ? (total + grid - 1) / grid : 0};
}

// Item k of this CTA.  Attention: one (b, h, 128-row query tile), heaviest
// first, dealt in a boustrophedon order like attn_get_item.  Decode: the k-th
// pair part of this CTA's range of key tiles (see decode_split).
__device__ __forceinline__ bool split_get_item(const AttnParams& p, int k, SplitItem& it) {
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  if (p.decode) {
    const int hkv = p.H / p.kv_group;
    const DecodeSplit ds = decode_split(p, G);
    const long long lo = static_cast<long long>(c) * ds.share;
    const long long hi = min(ds.total, lo + ds.share);
    if (lo >= hi) return false;
    // the sequence holding tile lo (sequences without visible keys hold none)
    long long cum = 0;  // first tile of sequence b
    int b = 0, nt = 0;
    for (; b < p.B; ++b) {
      nt = decode_seq_tiles(p, b);
      if (lo < cum + static_cast<long long>(hkv) * nt) break;
      cum += static_cast<long long>(hkv) * nt;
    }
    long long x = lo;
    for (int i = 0;; ++i) {
      if (b >= p.B || nt <= 0) return false;  // unreachable while x < hi
      const long long off = x - cum;
      const int kvh = static_cast<int>(off / nt);
      const int t0 = static_cast<int>(off - static_cast<long long>(kvh) * nt);
      const long long pair0 = cum + static_cast<long long>(kvh) * nt;  // first tile of the pair
      const long long end = min(pair0 + nt, hi);
      if (i == k) {
        it.b = b;
        it.kvh = kvh;
        it.h = kvh * p.kv_group;
        it.chunk = static_cast<int>(c - pair0 / ds.share);
#ifdef GB300_CHECKED
        if (!check_ok(it.b < p.B && it.kvh < hkv && it.chunk >= 0 && it.chunk < p.n_chunks,
                      CHECK_ITEM))
          return false;
#endif
        it.qrow = (it.b * p.H + it.h) * p.Lq;
        int kv_len = p.Lk;
        it.kv_len_raw = p.Lk;
        if (p.mask_kind & ATTN_MASK_PADDING_BIT) {
          const int raw = p.kv_lens[it.b];
          it.kv_len_raw = raw;
          kv_len = raw < 0 ? 0 : (raw > p.Lk ? p.Lk : raw);
        }
        it.kv_len = kv_len;
        it.coff = attn_causal_offset(p, kv_len);
        it.row0 = 0;
        it.k0 = t0 * ATTN_BLOCK_N;
        it.nkv = static_cast<int>(end - x);
        return true;
      }
      x = end;
      if (x >= hi) return false;
      if (x >= cum + static_cast<long long>(hkv) * nt) {  // on to the next sequence with tiles
        cum += static_cast<long long>(hkv) * nt;
        for (++b; b < p.B && (nt = decode_seq_tiles(p, b)) == 0; ++b) {
        }
      }
    }
  }
  const long long w = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (w >= p.n_items) return false;
  it.k0 = 0;
  it.chunk = 0;
  it.qrow = 0;
  const int BH = p.B * p.H;
  const int rank = static_cast<int>(w / BH);
  const int bh = static_cast<int>(w - static_cast<long long>(rank) * BH);
  const int qt = p.n_qblocks - 1 - rank;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  it.kvh = it.h / p.kv_group;
#ifdef GB300_CHECKED
  // every role decodes the same k, so all of them stop at the same item
  if (!check_ok(it.b >= 0 && it.b < p.B && it.h >= 0 && it.h < p.H && qt >= 0 &&
                    qt < p.n_qblocks && it.kvh < p.H / p.kv_group,
                CHECK_ITEM))
    return false;
#endif
  int kv_len = p.Lk;
  it.kv_len_raw = p.Lk;
  if (p.mask_kind & ATTN_MASK_PADDING_BIT) {
    const int raw = p.kv_lens[it.b];
    it.kv_len_raw = raw;
    kv_len = raw < 0 ? 0 : (raw > p.Lk ? p.Lk : raw);
  }
  it.kv_len = kv_len;
  it.coff = attn_causal_offset(p, kv_len);
  it.row0 = qt * SPLIT_ROWS;
  int n = 0;
  const bool all_padded = attn_padded_query(p, it.row0, kv_len);
  if (it.row0 < p.Lq && !all_padded) {
    int lim = kv_len;
    if (p.mask_kind & ATTN_MASK_CAUSAL_BIT) {
      const int last = min(it.row0 + SPLIT_ROWS - 1, p.Lq - 1);
      lim = min(lim, max(last + 1 + it.coff, 0));
    }
    n = (lim + ATTN_BLOCK_N - 1) / ATTN_BLOCK_N;
  }
  it.nkv = n;
  return true;
}

// Waits for the last load into each slot of a ring before the CTA exits (n
// loads were issued in ring order; `skip` is a running index never loaded).
__device__ __forceinline__ void split_drain_ring(uint64_t* full, int stages, uint32_t n,
                                              long long skip, uint64_t limit_ns) {
  for (int s = 0; s < stages; ++s) {
    if (n <= static_cast<uint32_t>(s)) continue;
    const uint32_t uses = (n - s + stages - 1) / stages;
    const uint32_t last = s + (uses - 1u) * stages;
    if (static_cast<long long>(last) != skip) mbar_wait_drain(&full[s], (uses - 1u) & 1u, limit_ns);
  }
}

template <int D>
struct SplitLayout {
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;  // 128 rows x 64 bf16
  static constexpr int NCHUNK = D / 64;
  static constexpr int K_STAGES = (D == 128) ? 3 : 5;
  static constexpr int V_STAGES = (D == 128) ? 2 : 4;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE_BYTES;
  static constexpr int V_OFF = K_OFF + K_STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + V_STAGES * TILE_BYTES;
  static constexpr int B_Q_FULL = 0;
  static constexpr int B_Q_EMPTY = 1;
  static constexpr int B_K_FULL = 2;
  static constexpr int B_K_EMPTY = B_K_FULL + K_STAGES;
  static constexpr int B_V_FULL = B_K_EMPTY + K_STAGES;
  static constexpr int B_V_EMPTY = B_V_FULL + V_STAGES;
  // per S/P buffer: S(t) computed, P(t) written, P(t) V completed
  static constexpr int B_S_FULL = B_V_EMPTY + V_STAGES;  // [2]
  static constexpr int B_P_FULL = B_S_FULL + 2;           // [2]
  static constexpr int B_PV_DONE = B_P_FULL + 2;          // [2]
  static constexpr int B_DRAIN = B_PV_DONE + 2;           // [2], one per issuer
  static constexpr int B_XCHG = B_DRAIN + 2;              // [4], one per TMEM lane quarter
  static constexpr int N_BARS = B_XCHG + 4;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int XCH_OFF = MISC_OFF + 16;  // float [2 groups][128 rows][4]
  static constexpr int SMEM_BYTES = XCH_OFF + 2 * 128 * 4 * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
  static constexpr uint32_t TS0 = 0, TO0 = 256;  // buffer b at TS0 + 128 b, O_b at TO0 + 128 b
};

// ---------------------------------------------------------------------------
// TMA producers
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void split_qk_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                               const AttnParams& p, uint8_t* smem,
                                               uint64_t* bars, const WaitCtl& ctl) {
  using L = SplitLayout<D>;
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  uint32_t q_loads = 0, kv_it = 0;
  bool ok = true;
  SplitItem it;
  for (int k = 0; ok && split_get_item(p, k, it); ++k) {
    if (it.nkv == 0) continue;
    if (q_loads > 0) {
      // the previous item's S MMAs have read Q
      ok = mbar_wait(&bars[L::B_Q_EMPTY], (q_loads - 1u) & 1u, ctl);
      if (!ok) break;
    }
    mbar_arrive_expect_tx(&bars[L::B_Q_FULL], L::TILE_BYTES);
    for (int c = 0; c < L::NCHUNK; ++c) {
      if (p.decode)  // 2-D map over the [B*H*Lq, D] query rows
        tma_load_2d(smem + L::Q_OFF + c * L::CHUNK_BYTES, tmQ, &bars[L::B_Q_FULL], 64 * c,
                    it.qrow);
      else
        attn_load_tile(tmQ, smem + L::Q_OFF + c * L::CHUNK_BYTES, &bars[L::B_Q_FULL], 64 * c,
                       it.row0, it.h, it.b, p.packed);
    }
    ++q_loads;
    for (int j = 0; j < it.nkv; ++j, ++kv_it) {
      const int s = static_cast<int>(kv_it % L::K_STAGES);
      const uint32_t reuse = kv_it / L::K_STAGES;
      if (reuse > 0) {
        ok = mbar_wait(&bars[L::B_K_EMPTY + s], (reuse - 1u) & 1u, ctl);
        if (!ok) break;
      }
      if (static_cast<long long>(kv_it) == p.debug_skip_kv_load) continue;
      mbar_arrive_expect_tx(&bars[L::B_K_FULL + s], L::TILE_BYTES);
      for (int c = 0; c < L::NCHUNK; ++c)
        attn_load_tile(tmK, smem + L::K_OFF + s * L::TILE_BYTES + c * L::CHUNK_BYTES,
                       &bars[L::B_K_FULL + s], 64 * c, it.k0 + j * ATTN_BLOCK_N, it.kvh, it.b,
                       p.packed);
    }
  }
  // Unwind: every load this thread issued lands before the CTA exits.
  if (q_loads > 0) mbar_wait_drain(&bars[L::B_Q_FULL], (q_loads - 1u) & 1u, ctl.limit_ns);
  split_drain_ring(&bars[L::B_K_FULL], L::K_STAGES, kv_it, p.debug_skip_kv_load, ctl.limit_ns);
}

template <int D>
__device__ __forceinline__ void split_v_producer(const CUtensorMap* tmV, const AttnParams& p,
                                              uint8_t* smem, uint64_t* bars, const WaitCtl& ctl) {
  using L = SplitLayout<D>;
  tma_prefetch_desc(tmV);
  uint32_t kv_it = 0;
  bool ok = true;
  SplitItem it;
  for (int k = 0; ok && split_get_item(p, k, it); ++k) {
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
                       &bars[L::B_V_FULL + s], 64 * c, it.k0 + j * ATTN_BLOCK_N, it.kvh, it.b,
                       p.packed);
    }
  }
  split_drain_ring(&bars[L::B_V_FULL], L::V_STAGES, kv_it, -1, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// S issuer (one warp): S(t) = Q K_t^T into buffer t % 2
// ---------------------------------------------------------------------------
// The whole warp runs the loop and waits; one elected lane issues.  Operands
// computed by all lanes stay warp-uniform, which keeps the issue of each
// tcgen05.mma short.
template <int D>
__device__ __forceinline__ void split_s_role(const AttnParams& p, uint8_t* smem, uint64_t* bars,
                                          uint32_t tmem, const WaitCtl& ctl) {
  using L = SplitLayout<D>;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(128, ATTN_BLOCK_N, false);
  const uint64_t q_desc = smem_desc_sw128(smem_u32(smem + L::Q_OFF), 16, 1024);
  const uint64_t k_desc = smem_desc_sw128(smem_u32(smem + L::K_OFF), 16, 1024);
  uint32_t t = 0, q_cnt = 0;  // running tile index, Q loads consumed
  bool ok = true;
  SplitItem it;
  for (int k = 0; ok && split_get_item(p, k, it); ++k) {
    if (it.kv_len_raw != it.kv_len && elect_one()) atomicOr(p.status, ATTN_STATUS_BAD_KVLEN);
    if (it.nkv == 0) continue;
    ok = __all_sync(0xffffffffu, mbar_wait(&bars[L::B_Q_FULL], q_cnt & 1u, ctl));
    if (!ok) break;
    ++q_cnt;
    for (int j = 0; j < it.nkv; ++j, ++t) {
      const uint32_t buf = t & 1u;
      if (t >= 2) {
        // P(t-2) V has read this buffer (and V_{t-2}: free its slot)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&bars[L::B_PV_DONE + buf], ((t >> 1) - 1u) & 1u, ctl));
        if (!ok) break;
        if (elect_one()) mbar_arrive(&bars[L::B_V_EMPTY + (t - 2u) % L::V_STAGES]);
      }
      const int s = static_cast<int>(t % L::K_STAGES);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[L::B_K_FULL + s], (t / L::K_STAGES) & 1u, ctl));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + L::TS0 + buf * 128u;
      const uint64_t kd = k_desc + static_cast<uint64_t>((s * L::TILE_BYTES) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          mma_bf16_ss(d_tmem, q_desc + off, kd + off, IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[L::B_S_FULL + buf]);
      }
      __syncwarp();
    }
    if (!ok) break;
    if (elect_one()) mma_commit(&bars[L::B_Q_EMPTY]);  // Q is free once the item's S complete
    __syncwarp();
  }
  // Unwind: all MMAs issued by this warp complete before TMEM is freed.
  if (elect_one()) mma_commit(&bars[L::B_DRAIN + 0]);
  __syncwarp();
  mbar_wait_drain(&bars[L::B_DRAIN + 0], 0u, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// P.V issuer (one warp): O_{t % 2} += P(t) V_t
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void split_pv_role(const AttnParams& p, uint8_t* smem, uint64_t* bars,
                                           uint32_t tmem, const WaitCtl& ctl) {
  using L = SplitLayout<D>;
  constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
  const uint64_t v_desc = smem_desc_sw128(smem_u32(smem + L::V_OFF), L::CHUNK_BYTES, 1024);
  uint32_t t = 0;
  bool ok = true;
  SplitItem it;
  for (int k = 0; ok && split_get_item(p, k, it); ++k) {
    for (int j = 0; j < it.nkv; ++j, ++t) {
      const int s = static_cast<int>(t % L::V_STAGES);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[L::B_V_FULL + s], (t / L::V_STAGES) & 1u, ctl));
      if (!ok) break;
      const uint32_t buf = t & 1u;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[L::B_P_FULL + buf], (t >> 1) & 1u, ctl));
      if (!ok) break;
      tc_fence_after();
      const uint64_t vd = v_desc + static_cast<uint64_t>((s * L::TILE_BYTES) >> 4);
      const uint32_t pa = tmem + L::TS0 + buf * 128u;
      const uint32_t o = tmem + L::TO0 + buf * 128u;
      // the first tile of each group in this item starts its accumulator
      const uint32_t first = j < 2 ? 1u : 0u;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < ATTN_BLOCK_N / 16; ++kk)
          mma_bf16_ts(o, pa + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4), IDESC_O,
                      (first && kk == 0) ? 0u : 1u);
        mma_commit(&bars[L::B_PV_DONE + buf]);
      }
      __syncwarp();
    }
  }
  if (elect_one()) mma_commit(&bars[L::B_DRAIN + 1]);
  __syncwarp();
  mbar_wait_drain(&bars[L::B_DRAIN + 1], 0u, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// softmax / correction / epilogue: warpgroup g, one thread per query row
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void split_softmax_role(const int g, const AttnParams& p, uint8_t* smem,
                                                uint64_t* bars, uint32_t tmem,
                                                const WaitCtl& ctl) {
  using L = SplitLayout<D>;
  constexpr int DH = D / 2;  // output columns written by each group
  const int rloc = static_cast<int>(threadIdx.x & 127u);
  const int q = (rloc >> 5);
  const bool leader = (threadIdx.x & 127u) == 0u;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t s_tmem = tmem + L::TS0 + static_cast<uint32_t>(g) * 128u + lane_base;
  const uint32_t o_own = tmem + L::TO0 + static_cast<uint32_t>(g) * 128u + lane_base;
  float* xch = reinterpret_cast<float*>(smem + L::XCH_OFF);  // [group][row][m, l, lb, n]
  uint64_t* xbar = &bars[L::B_XCHG + q];
  const float c = p.scale_log2;
  const bool causal = (p.mask_kind & ATTN_MASK_CAUSAL_BIT) != 0;
  uint32_t t0 = 0;     // running index of the item's first tile
  uint32_t x_cnt = 0;  // exchanges with the other group
  bool ok = true;
  SplitItem it;
  for (int k = 0; ok && split_get_item(p, k, it); ++k) {
    if (it.row0 >= p.Lq) continue;
    // query index of this thread's row: the tile's rows, or in decode the
    // packed (head, query) rows, of which the first q_rows are live
    const int r = p.decode ? rloc % p.Lq : it.row0 + rloc;
    const bool live_row = p.decode ? rloc < p.q_rows : r < p.Lq;
    const int nkv = it.nkv;
    int limit = it.kv_len;  // this row attends to keys [0, limit)
    if (causal) limit = min(limit, max(r + 1 + it.coff, 0));
    const bool padded_row = attn_padded_query(p, r, it.kv_len);
    float m = -INFINITY, l = 0.f, lb = 0.f;
    int cnt = 0;  // tiles of this item taken by this group
    // this group's first tile of the item
    const int jfirst = static_cast<int>((static_cast<uint32_t>(g) - t0) & 1u);
    for (int j = jfirst; j < nkv; j += 2) {
      const uint32_t t = t0 + static_cast<uint32_t>(j);
      ok = mbar_wait(&bars[L::B_S_FULL + g], (t >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (leader) mbar_arrive(&bars[L::B_K_EMPTY + t % L::K_STAGES]);  // K_t read
      tc_fence_after();
      uint32_t ra[32], rb[32], rc[32], rd[32];
      tmem_ld_32x32b_x32(s_tmem + 0u, ra);
      tmem_ld_32x32b_x32(s_tmem + 32u, rb);
      tmem_ld_32x32b_x32(s_tmem + 64u, rc);
      tmem_ld_32x32b_x32(s_tmem + 96u, rd);
      tmem_ld_wait(ra);
      reg_fence(rb);
      reg_fence(rc);
      reg_fence(rd);
      float s[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(ra[i]);
        s[32 + i] = __uint_as_float(rb[i]);
        s[64 + i] = __uint_as_float(rc[i]);
        s[96 + i] = __uint_as_float(rd[i]);
      }
      const int nvalid = limit - (it.k0 + j * ATTN_BLOCK_N);
      if (nvalid < ATTN_BLOCK_N) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = (i < nvalid) ? s[i] : -INFINITY;
      }
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
      float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int i = 8; i < 128; i += 8) {
        mx0 = fmax3(mx0, s[i], s[i + 1]);
        mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
        mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
        mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m, mx * c);  // scale > 0, so the max commutes with it
      const bool need = m_new > m + ATTN_RESCALE_THRESHOLD;
      if (__any_sync(0xffffffffu, need && cnt > 0)) {
        // O_g holds this group's earlier tiles in the old scale: rescale it
        // once its last P.V (tile t - 2) has completed
        ok = mbar_wait(&bars[L::B_PV_DONE + g], ((t >> 1) - 1u) & 1u, ctl);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ro[32];
          tmem_ld_32x32b_x32(o_own + cc * 32u, ro);
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
          tmem_st_32x32b_x32(o_own + cc * 32u, ro);
        }
      }
      if (need) {
        const float alpha = ex2_approx(m - m_new);
        l *= alpha;
        lb *= alpha;
        m = m_new;
      }
      const float mb = (m == -INFINITY) ? 0.f : m;
      // p = 2^(s c - m) as bf16 pairs over the first 64 columns of the
      // buffer; l sums the fp32 p (for the LSE), lb the bf16-rounded p that
      // the tensor core multiplies into V (for the normalisation of O)
      const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-mb, -mb);
      uint64_t lf_a = 0ull, lf_b = 0ull;
      float lb_a = 0.f, lb_b = 0.f, lb_c = 0.f, lb_d = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(s[64 * half + 2 * i], s[64 * half + 2 * i + 1]), c2, nm2), a0,
                    a1);
          f2_unpack(f2_fma(f2_pack(s[64 * half + 2 * i + 2], s[64 * half + 2 * i + 3]), c2, nm2),
                    a2, a3);
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
        tmem_st_32x32b_x32(s_tmem + 32u * half, pk);
      }
      {
        float x0, x1;
        f2_unpack(f2_add(lf_a, lf_b), x0, x1);
        l += x0 + x1;
        lb += (lb_a + lb_b) + (lb_c + lb_d);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[L::B_P_FULL + g]);
      ++cnt;
    }
    if (!ok) break;
    // epilogue: merge the two groups' partial softmaxes of every row
    //   m = max(m_0, m_1), w_g = 2^(m_g - m),
    //   O = (w_0 O_0 + w_1 O_1) / (w_0 lb_0 + w_1 lb_1),
    //   LSE = (m + log2(w_0 l_0 + w_1 l_1)) ln 2;
    // group g writes output columns [g D/2, (g+1) D/2)
    float mo = -INFINITY, lo = 0.f, lbo = 0.f;
    int cnt_o = 0;
    if (nkv > 0) {
      // all of the item's P.V (both groups') complete: commits are cumulative
      const uint32_t tl = t0 + static_cast<uint32_t>(nkv) - 1u;
      ok = mbar_wait(&bars[L::B_PV_DONE + (tl & 1u)], (tl >> 1) & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      float* mine = xch + (g * 128 + rloc) * 4;
      mine[0] = m;
      mine[1] = l;
      mine[2] = lb;
      mine[3] = __int_as_float(cnt);
      mbar_arrive(xbar);
      ok = mbar_wait(xbar, x_cnt & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++x_cnt;
      const float* other = xch + ((1 - g) * 128 + rloc) * 4;
      mo = other[0];
      lo = other[1];
      lbo = other[2];
      cnt_o = __float_as_int(other[3]);
      tc_fence_after();
    }
    const float mm = fmaxf(m, mo);
    const float w_own = (cnt > 0 && m != -INFINITY) ? ex2_approx(m - mm) : 0.f;
    const float w_oth = (cnt_o > 0 && mo != -INFINITY) ? ex2_approx(mo - mm) : 0.f;
    const float lsum = w_own * l + w_oth * lo;
    const float lbsum = w_own * lb + w_oth * lbo;
    const bool in_range = live_row;
    const bool zero_row = padded_row || nkv == 0 || limit <= it.k0 || !(lbsum > 0.f);
    // decode writes the chunk's partial unnormalised (the chunks are merged
    // by attn_decode_combine_kernel); attention divides by the row sum
    const float inv_l = zero_row ? 0.f : (p.decode ? 1.0f : 1.0f / lbsum);
    const float f0 = (g == 0 ? w_own : w_oth) * inv_l;  // weight of O_0
    const float f1 = (g == 0 ? w_oth : w_own) * inv_l;  // weight of O_1
    const bool has0 = (g == 0 ? cnt : cnt_o) > 0;
    const bool has1 = (g == 0 ? cnt_o : cnt) > 0;
    const long long part = static_cast<long long>(it.qrow + rloc) * p.n_chunks + it.chunk;
    __nv_bfloat16* orow = p.decode ? nullptr
                                   : p.O + it.b * p.o_stride_b + it.h * p.o_stride_h +
                                         static_cast<long long>(r) * p.o_stride_l + DH * g;
#pragma unroll
    for (int cc = 0; cc < DH / 32; ++cc) {
      const uint32_t col = static_cast<uint32_t>(DH * g + cc * 32);
      uint32_t r0[32], r1[32];
      if (has0) {
        tmem_ld_32x32b_x32(tmem + L::TO0 + lane_base + col, r0);
        tmem_ld_wait(r0);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r0[i] = 0u;
      }
      if (has1) {
        tmem_ld_32x32b_x32(tmem + L::TO0 + 128u + lane_base + col, r1);
        tmem_ld_wait(r1);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r1[i] = 0u;
      }
      if (in_range && p.decode) {
        // the workspace is 256-byte aligned and its rows are D floats: every
        // 8-float group is 32-byte aligned
        float* prow = p.part_o + part * D + DH * g + cc * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            y[e] = zero_row ? 0u
                            : __float_as_uint(__uint_as_float(r0[8 * i + e]) * f0 +
                                              __uint_as_float(r1[8 * i + e]) * f1);
          st_global_v8(prow + 8 * i, y);
        }
      } else if (in_range) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float y0 = __uint_as_float(r0[2 * i]) * f0 + __uint_as_float(r1[2 * i]) * f1;
          const float y1 =
              __uint_as_float(r0[2 * i + 1]) * f0 + __uint_as_float(r1[2 * i + 1]) * f1;
          w[i] = zero_row ? 0u : pack_bf16x2(y0, y1);
        }
        if (p.o_v8) {
          st_global_v8(orow + cc * 32, w);
          st_global_v8(orow + cc * 32 + 16, w + 8);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_global_v4(orow + cc * 32 + i * 8, w[4 * i], w[4 * i + 1], w[4 * i + 2],
                         w[4 * i + 3]);
        }
      }
    }
    if (p.decode && in_range && g == 0) {
      st_global_v4(p.part_ml + part * 4, __float_as_uint(zero_row ? -INFINITY : mm),
                   __float_as_uint(zero_row ? 0.f : lsum), __float_as_uint(zero_row ? 0.f : lbsum),
                   0u);
    } else if (p.LSE != nullptr && in_range && g == 0) {
      const float lse = zero_row ? -INFINITY : (mm + log2f(lsum)) * 0.69314718055994530942f;
      p.LSE[(static_cast<long long>(it.b) * p.H + it.h) * p.Lq + r] = lse;
    }
    if (nkv > 0) {
      // Neither group starts the next item (whose first P.V overwrites its
      // O) before both have read both accumulators.
      tc_fence_before();
      mbar_arrive(xbar);
      ok = mbar_wait(xbar, x_cnt & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++x_cnt;
    }
    t0 += static_cast<uint32_t>(nkv);
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_fwd_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using L = SplitLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);

  if (threadIdx.x == 0) {
    mbar_init(&bars[L::B_Q_FULL], 1);
    mbar_init(&bars[L::B_Q_EMPTY], 1);
    for (int s = 0; s < L::K_STAGES; ++s) {
      mbar_init(&bars[L::B_K_FULL + s], 1);
      mbar_init(&bars[L::B_K_EMPTY + s], 1);
    }
    for (int s = 0; s < L::V_STAGES; ++s) {
      mbar_init(&bars[L::B_V_FULL + s], 1);
      mbar_init(&bars[L::B_V_EMPTY + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[L::B_S_FULL + b], 1);
      mbar_init(&bars[L::B_P_FULL + b], 128);
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
  // Set-up done (on-chip only).  Behind a dependent launch this overlapped
  // the previous kernel's tail; nothing in global memory is touched before
  // that kernel has completed.
  grid_dependency_wait();
  grid_launch_dependents();

  // Register split as in attn_fwd_kernel: softmax warpgroups 216, control 72;
  // together exactly the 384 x 168 registers of the launch.
  if (warp >= 8) {
    reg_dealloc<ATTN_REGS_CONTROL>();
    if (warp == 8) {
      split_s_role<D>(p, smem, bars, tmem, ctl);
    } else if (warp == 9) {
      if (lane == 0) split_qk_producer<D>(&tmQ, &tmK, p, smem, bars, ctl);
    } else if (warp == 10) {
      split_pv_role<D>(p, smem, bars, tmem, ctl);
    } else {
      if (lane == 0) split_v_producer<D>(&tmV, p, smem, bars, ctl);
    }
  } else {
    reg_alloc<ATTN_REGS_SOFTMAX>();
    split_softmax_role<D>(warp >> 2, p, smem, bars, tmem, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, ATTN_TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// split-KV decode: merge the chunks' partial softmaxes of every query row
// ---------------------------------------------------------------------------
// One warp per query row (b, h, q).  With m = max_c m_c and w_c = 2^(m_c - m):
//   O = sum_c w_c Opart_c / sum_c w_c lb_c,   LSE = (m + log2 sum_c w_c l_c) ln 2,
// the identity by which the online softmax merges partial results
// ("Self-Attention 机制", Softmax 的数值稳定性与 Online Softmax).  Rows whose
// every chunk is empty (padded or without keys) get O = 0 and LSE = -inf.
// The row's pair has one partial per CTA range that overlaps its key tiles
// (decode_split, recomputed here from kv_lens): slots 0 .. last - first.
// Lane c reads the (m, l, lb) of slots c, c + 32, ... and the warp reduces
// them with shuffles, so the statistics cost one round trip to memory, not
// one per slot.  Then lane l accumulates output columns l, l + 32, ... over
// the slots in slot order, with several slots' loads in flight.
template <int D>
__global__ void __launch_bounds__(128)
    attn_decode_combine_kernel(const AttnParams p, int grid, long long rows,
                               __nv_bfloat16* __restrict__ O, float* __restrict__ LSE) {
  constexpr int PER = D / 32;
  constexpr unsigned FULL = 0xffffffffu;
  grid_dependency_wait();  // the partial results of the kernel ahead of it
  grid_launch_dependents();
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);
  if (row >= rows) return;  // uniform over the warp
  // the row's pair and the slots of its partial results
  const int hkv = p.H / p.kv_group;
  const int b = static_cast<int>(row / (static_cast<long long>(p.H) * p.Lq));
  const int kvh = static_cast<int>((row / p.Lq) % p.H) / p.kv_group;
  const DecodeSplit ds = decode_split(p, grid);
  long long cum = 0;
  for (int i = 0; i < b; ++i) cum += static_cast<long long>(hkv) * decode_seq_tiles(p, i);
  const int nt = decode_seq_tiles(p, b);
  int n_slots = 0;
  if (nt > 0) {
    const long long pair0 = cum + static_cast<long long>(kvh) * nt;
    n_slots = static_cast<int>((pair0 + nt - 1) / ds.share - pair0 / ds.share) + 1;
  }
  const float* part_o = p.part_o + row * p.n_chunks * D;
  const float4* ml = reinterpret_cast<const float4*>(p.part_ml + row * p.n_chunks * 4);
  float mm = -INFINITY;
  for (int c = lane; c < n_slots; c += 32) mm = fmaxf(mm, ml[c].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(FULL, mm, o));
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float l = 0.f, lb = 0.f;
  if (mm != -INFINITY) {
    for (int c0 = 0; c0 < n_slots; c0 += 32) {
      float w = 0.f;  // weight of slot c0 + lane; 0 for an empty partial
      if (c0 + lane < n_slots) {
        const float4 v = ml[c0 + lane];
        if (v.x != -INFINITY) {
          w = ex2_approx(v.x - mm);
          l += w * v.y;
          lb += w * v.z;
        }
      }
      const int nc = min(32, n_slots - c0);
      const float* po = part_o + static_cast<long long>(c0) * D + lane;
#pragma unroll 4
      for (int j = 0; j < nc; ++j) {
        const float wj = __shfl_sync(FULL, w, j);
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += wj * po[static_cast<long long>(j) * D + 32 * i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      l += __shfl_xor_sync(FULL, l, o);
      lb += __shfl_xor_sync(FULL, lb, o);
    }
  }
  const bool zero = !(lb > 0.f);
  const float inv = zero ? 0.f : 1.0f / lb;
#pragma unroll
  for (int i = 0; i < PER; ++i) O[row * D + lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  if (LSE != nullptr && lane == 0)
    LSE[row] = zero ? -INFINITY : (mm + log2f(l)) * 0.69314718055994530942f;
}

}  // namespace gb300

// attn_fwd_kernel.cuh -- fused multi-head scaled dot-product attention forward
// for sm_103a (tcgen05 tensor cores, TMEM accumulators, TMA staging).
//
//   O = softmax(Q K^T * scale + M) V,   LSE = log(sum_j exp(scale q.k_j + M_j))
//
// computed one 128-query x 128-key tile at a time with the online softmax of
// "Self-Attention 机制", section "Softmax 的数值稳定性与 Online Softmax"
// (running row max m and running sum d, rescaled by e^(m_old - m_new) when
// the max moves), so the n x n score matrix never leaves the chip
// (same page, section "瓶颈：两个项，两种场景").  Under the causal mask,
// key tiles that lie wholly above the diagonal are skipped (same page,
// section "Causal Mask").
//
// CTA organisation (one CTA per SM, persistent):
//   work item      = (batch b, head h, block of 256 query rows), taken
//                    longest-first and dealt to CTAs in a boustrophedon order
//   warps 0-3      = softmax group for Q tile 0 (rows 0..127 of the block)
//   warps 4-7      = softmax group for Q tile 1 (rows 128..255)
//   warp 8         = MMA issuer of Q tile 0 (one thread) + TMEM owner
//   warp 9         = TMA producer (one thread)
//   warp 10        = MMA issuer of Q tile 1 (one thread)
//   warp 11        = idle (it completes the third warpgroup, which the
//                    per-warpgroup register reallocation needs)
// TMEM (512 columns x 128 lanes, fp32):
//   [  0,128) S of tile 0, [128,256) S of tile 1
//   P (bf16 pairs) reuses the high 64 columns of its S;
//   [256,384) O accumulator of tile 0, [384,512) O of tile 1 (D = 64: the
//   first 80 columns of each, column 64 holding the row sum of P)
// Each Q tile has its own MMA issuer, and at D = 128 the two take turns: while
// one softmax group works on its S, the tensor core runs the other tile's P.V
// and next S.
//
// Softmax state per row (one thread per row = one TMEM lane): m in log2
// units (already multiplied by scale*log2 e) and two running sums: l of the
// fp32 probabilities (gives the LSE) and lb of the bf16-rounded
// probabilities that the tensor core multiplies into V (normalises O, so
// O / lb is an exactly normalised average of V rows and a one-hot row
// reproduces its V row; normalised by l instead, the peaked long-context
// rows drift just past the 1.5e-2 bound on O).  The max used
// for the exponentials is only moved when it grows by more than 8 (a factor
// 256); otherwise the stale max is kept, which is exact after the final
// division by l because O and l share it.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gb300 {

constexpr int ATTN_THREADS = 384;      // 3 warpgroups
constexpr int ATTN_REGS_AT_LAUNCH = 168;  // 65536 / 384, rounded down to 8
constexpr int ATTN_REGS_SOFTMAX = 216;
constexpr int ATTN_REGS_CONTROL = 72;
static_assert(2 * 128 * ATTN_REGS_SOFTMAX + 128 * ATTN_REGS_CONTROL <=
                  ATTN_THREADS * ATTN_REGS_AT_LAUNCH,
              "register split exceeds the registers the block is launched with");
constexpr int ATTN_BLOCK_M = 128;  // query rows per Q tile
constexpr int ATTN_BLOCK_N = 128;  // keys per KV tile
constexpr int ATTN_QTILES = 2;     // Q tiles per work item
constexpr int ATTN_ROWS_PER_ITEM = ATTN_BLOCK_M * ATTN_QTILES;
constexpr uint32_t ATTN_TMEM_COLS = 512;
constexpr float ATTN_RESCALE_THRESHOLD = 8.0f;  // log2 units
// Q tile 0 takes the lower 128 rows of even items and the upper 128 of odd
// ones (see attn_get_item)
constexpr bool ATTN_ALTERNATE_TILES = true;

enum : unsigned int { ATTN_STATUS_TIMEOUT = 1u, ATTN_STATUS_BAD_KVLEN = 2u };
enum : int { ATTN_MASK_CAUSAL_BIT = 1, ATTN_MASK_PADDING_BIT = 2 };

struct AttnParams {
  int B, H, Lq, Lk;
  int kv_group;            // query heads per K/V head (grouped-query attention)
  int causal_offset;       // causal: query i sees keys j <= i + causal_offset
  int mask_kind;           // bit 0 causal, bit 1 padding
  // 1: bottom-right causal with padding.  The queries are the last Lq tokens
  // of each sequence: sequence b's offset is kv_len_b - Lq (causal_offset is
  // unused) and no query row is padding by its index; rows before the
  // sequence's first token see no key.
  int offset_per_seq;
  int packed;              // 0: Q/K/V maps over [B,H,L,d]; 1: over [B,L,3,H,d]
  const int32_t* kv_lens;  // [B] valid lengths (padding) or nullptr
  float scale_log2;        // softmax scale * log2(e)
  __nv_bfloat16* O;
  long long o_stride_b, o_stride_h, o_stride_l;  // in elements
  int o_v8;                // 1: O and its strides are 32-byte aligned (256-bit stores)
  float* LSE;              // [B,H,Lq] natural-log LSE, or nullptr
  int n_qblocks;           // ceil(Lq / 256)
  int head_group;          // (b, h) pairs per group of the item order; B * H: one group
  int n_items;             // B * H * n_qblocks
  unsigned int* status;    // device status word
  unsigned long long wait_limit_ns;
  long long debug_skip_kv_load;  // test hook: skip this running K-tile load (-1: none)
  // split-KV decode (attn_fwd_split_kernel only; decode == 0 everywhere else):
  // an item is the part of one (b, K/V head) pair's key tiles that falls in
  // the CTA's share of all pairs' tiles; its Q tile packs the q_rows =
  // kv_group * Lq query rows of the heads that share the K/V head, and its
  // epilogue writes an unnormalised partial result to one of the row's slots
  int decode;
  int q_rows;
  int n_chunks;            // partial-result slots per query row
  float* part_o;           // [B*H*Lq][n_chunks][D]: w_0 O_0 + w_1 O_1 of the item
  float* part_ml;          // [B*H*Lq][n_chunks][4]: m (log2 units), l, lb, 0
};

// Causal offset of a sequence with kv_len valid keys: its query i sees the
// keys j <= i + offset ("04. Self-Attention", section 七: no token sees a
// later one).  Top-left: 0; bottom-right: Lk - Lq, or kv_len - Lq when each
// sequence has its own length, so that its queries sit at its own end.
__device__ __forceinline__ int attn_causal_offset(const AttnParams& p, int kv_len) {
  return p.offset_per_seq ? kv_len - p.Lq : p.causal_offset;
}

// A padded query row (O = 0, LSE = -inf): with the padding mask, rows at or
// past the sequence's length -- except under the bottom-right causal mask,
// whose queries end at the sequence's end.
__device__ __forceinline__ bool attn_padded_query(const AttnParams& p, int r, int kv_len) {
  return (p.mask_kind & ATTN_MASK_PADDING_BIT) && !p.offset_per_seq && r >= kv_len;
}

template <int D>
struct AttnLayout {
  static constexpr int TILE_BYTES = ATTN_BLOCK_M * D * 2;  // 128 rows x D bf16
  static constexpr int CHUNK_BYTES = ATTN_BLOCK_M * 128;   // 128 rows x 64 bf16
  static constexpr int NCHUNK = D / 64;
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + ATTN_QTILES * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  // Row sum on the tensor core (D = 64): the P.V MMA runs with N = D + 16,
  // its B operand's second 64-column atom a constant tile of ones (ONES_OFF,
  // reached from each V stage through the descriptor's leading-byte offset),
  // so O column D accumulates the sum of the bf16 P that the MMA multiplies
  // into V.  The softmax then keeps only the fp32 sum for the LSE.  At
  // D = 128 the two O accumulators leave no TMEM columns for it.
  static constexpr bool TC_ROWSUM = (D == 64);
  static constexpr int O_N = TC_ROWSUM ? D + 16 : D;  // N of the P.V MMA
  static constexpr int ONES_OFF = V_OFF + STAGES * TILE_BYTES;
  static constexpr int ONES_BYTES = TC_ROWSUM ? CHUNK_BYTES : 0;
  static constexpr int BAR_OFF = ONES_OFF + ONES_BYTES;
  // barrier indices
  static constexpr int B_Q_FULL = 0;
  static constexpr int B_Q_EMPTY = 2;
  static constexpr int B_K_FULL = 4;
  static constexpr int B_V_FULL = B_K_FULL + STAGES;
  // K and V of a stage are released separately: K once both Q tiles' S MMAs
  // that read it have completed, V once both P.V MMAs have
  static constexpr int B_K_EMPTY = B_V_FULL + STAGES;
  static constexpr int B_V_EMPTY = B_K_EMPTY + STAGES;
  static constexpr int B_S_FULL = B_V_EMPTY + STAGES;
  // [2 t + half]: P of keys [64 half, 64 half + 64) of tile t is in TMEM
  static constexpr int B_P_FULL = B_S_FULL + 2;
  static constexpr int B_O_DONE = B_P_FULL + 4;
  static constexpr int B_DRAIN = B_O_DONE + 2;  // one per MMA issuer
  static constexpr int B_TURN = B_DRAIN + 2;  // [issuer]: its turn to submit MMAs
  static constexpr int N_BARS = B_TURN + 2;
  // TMEM columns of tile t: S at 128 t; O at 256 + 128 t (D, or D + 16
  // with the row sum, of them used); P (bf16 pairs) in the high 64 columns
  // of S_t, which the softmax has read before it writes P
  static constexpr uint32_t O_STRIDE = 128u;
  static __device__ __forceinline__ uint32_t p_col(int t) {
    return 128u * static_cast<uint32_t>(t) + 64u;
  }
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
};

struct AttnItem {
  int b, h;
  int kvh;                // K/V head read by query head h
  int row0[ATTN_QTILES];  // first query row of each Q tile
  int nkv[ATTN_QTILES];   // KV tiles each Q tile needs (0: nothing to compute)
  int nkv_max;
  int kv_len;             // valid keys of this sequence (Lk without padding)
  int kv_len_raw;         // as given (for range reporting)
  int coff;               // causal offset of this sequence (attn_causal_offset)
};

// Item k of this CTA.  Items are ordered heaviest first (query blocks from
// the end of the sequence, which under the causal mask see the most keys)
// within each group of heads, and dealt to CTAs in a boustrophedon order,
// which balances the triangular work without any atomics.
__device__ __forceinline__ bool attn_get_item(const AttnParams& p, int k, AttnItem& it) {
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  const long long w = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (w >= p.n_items) return false;
  // Items go group by group of head_group (b, h) pairs (it divides B * H),
  // heaviest first within a group, so that the K/V a group streams can stay
  // in L2 while its items run.
  const int HG = p.head_group;
  const long long per_group = static_cast<long long>(HG) * p.n_qblocks;
  const int grp = static_cast<int>(w / per_group);
  const int rem = static_cast<int>(w - grp * per_group);
  const int rank = rem / HG;
  const int bh = grp * HG + (rem - rank * HG);
  const int qb = p.n_qblocks - 1 - rank;
  it.b = bh / p.H;
  it.h = bh - it.b * p.H;
  it.kvh = it.h / p.kv_group;
#ifdef GB300_CHECKED
  // every role decodes the same k, so all of them stop at the same item
  if (!check_ok(it.b >= 0 && it.b < p.B && it.h >= 0 && it.h < p.H && qb >= 0 &&
                    qb < p.n_qblocks && it.kvh < p.H / p.kv_group,
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
  it.nkv_max = 0;
#pragma unroll
  for (int t = 0; t < ATTN_QTILES; ++t) {
    const int r0 = qb * ATTN_ROWS_PER_ITEM + t * ATTN_BLOCK_M;
    it.row0[t] = r0;
    int n = 0;
    const bool all_padded = attn_padded_query(p, r0, kv_len);
    if (r0 < p.Lq && !all_padded) {
      int lim = kv_len;
      if (p.mask_kind & ATTN_MASK_CAUSAL_BIT) {
        const int last = min(r0 + ATTN_BLOCK_M - 1, p.Lq - 1);
        lim = min(lim, max(last + 1 + it.coff, 0));
      }
      n = (lim + ATTN_BLOCK_N - 1) / ATTN_BLOCK_N;
    }
    it.nkv[t] = n;
    it.nkv_max = max(it.nkv_max, n);
  }
  if (ATTN_ALTERNATE_TILES && (k & 1)) {
    // the upper 128 rows of a causal block need one key tile more than the
    // lower ones: the two Q tiles take them in turn, item by item
    const int r = it.row0[0], n = it.nkv[0];
    it.row0[0] = it.row0[1];
    it.nkv[0] = it.nkv[1];
    it.row0[1] = r;
    it.nkv[1] = n;
  }
  return true;
}

__device__ __forceinline__ void attn_load_tile(const CUtensorMap* m, void* dst, uint64_t* bar,
                                               int col, int row, int h, int b, int packed) {
  if (packed)
    tma_load_4d(dst, m, bar, col, h, row, b);
  else
    tma_load_4d(dst, m, bar, col, row, h, b);
}

// ---------------------------------------------------------------------------
// TMA producer (one thread)
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void attn_tma_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, const AttnParams& p,
                                              uint8_t* smem, uint64_t* bars, const WaitCtl& ctl) {
  using L = AttnLayout<D>;
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  tma_prefetch_desc(tmV);
  uint32_t q_loads[ATTN_QTILES] = {0u, 0u};
  uint32_t kv_it = 0;
  bool ok = true;
  AttnItem it;
  for (int k = 0; ok && attn_get_item(p, k, it); ++k) {
#pragma unroll
    for (int t = 0; t < ATTN_QTILES; ++t) {
      if (!ok || it.nkv[t] == 0) continue;
      if (q_loads[t] > 0) {
        ok = mbar_wait(&bars[L::B_Q_EMPTY + t], (q_loads[t] - 1u) & 1u, ctl);
        if (!ok) continue;
      }
      mbar_arrive_expect_tx(&bars[L::B_Q_FULL + t], L::TILE_BYTES);
      for (int c = 0; c < L::NCHUNK; ++c)
        attn_load_tile(tmQ, smem + L::Q_OFF + t * L::TILE_BYTES + c * L::CHUNK_BYTES,
                       &bars[L::B_Q_FULL + t], 64 * c, it.row0[t], it.h, it.b, p.packed);
      ++q_loads[t];
    }
    for (int j = 0; ok && j < it.nkv_max; ++j, ++kv_it) {
      const int s = static_cast<int>(kv_it % L::STAGES);
      // a K (V) slot is free once both MMA issuers released it; K slots come
      // free a whole Q tile step before V slots, so the next K tile lands
      // well before its S is issued
      if (kv_it >= static_cast<uint32_t>(L::STAGES)) {
        ok = mbar_wait(&bars[L::B_K_EMPTY + s], ((kv_it / L::STAGES) - 1u) & 1u, ctl);
        if (!ok) break;
      }
      if (static_cast<long long>(kv_it) != p.debug_skip_kv_load) {
        mbar_arrive_expect_tx(&bars[L::B_K_FULL + s], L::TILE_BYTES);
        for (int c = 0; c < L::NCHUNK; ++c)
          attn_load_tile(tmK, smem + L::K_OFF + s * L::TILE_BYTES + c * L::CHUNK_BYTES,
                         &bars[L::B_K_FULL + s], 64 * c, j * ATTN_BLOCK_N, it.kvh, it.b, p.packed);
      }
      if (kv_it >= static_cast<uint32_t>(L::STAGES)) {
        ok = mbar_wait(&bars[L::B_V_EMPTY + s], ((kv_it / L::STAGES) - 1u) & 1u, ctl);
        if (!ok) {
          // the K load of this index is in flight but not counted below
          if (static_cast<long long>(kv_it) != p.debug_skip_kv_load)
            mbar_wait_drain(&bars[L::B_K_FULL + s], (kv_it / L::STAGES) & 1u, ctl.limit_ns);
          break;
        }
      }
      mbar_arrive_expect_tx(&bars[L::B_V_FULL + s], L::TILE_BYTES);
      for (int c = 0; c < L::NCHUNK; ++c)
        attn_load_tile(tmV, smem + L::V_OFF + s * L::TILE_BYTES + c * L::CHUNK_BYTES,
                       &bars[L::B_V_FULL + s], 64 * c, j * ATTN_BLOCK_N, it.kvh, it.b, p.packed);
    }
  }
  // Unwind: every load this thread issued must land before the CTA exits.
  // On the normal path these phases completed long ago.
  for (int t = 0; t < ATTN_QTILES; ++t)
    if (q_loads[t] > 0)
      mbar_wait_drain(&bars[L::B_Q_FULL + t], (q_loads[t] - 1u) & 1u, ctl.limit_ns);
  for (int s = 0; s < L::STAGES; ++s) {
    if (kv_it <= static_cast<uint32_t>(s)) continue;
    const uint32_t n_s = (kv_it - s + L::STAGES - 1) / L::STAGES;  // loads into stage s
    const uint32_t last = s + (n_s - 1u) * L::STAGES;                 // running index
    if (static_cast<long long>(last) != p.debug_skip_kv_load)
      mbar_wait_drain(&bars[L::B_K_FULL + s], (n_s - 1u) & 1u, ctl.limit_ns);
    mbar_wait_drain(&bars[L::B_V_FULL + s], (n_s - 1u) & 1u, ctl.limit_ns);
  }
}

// ---------------------------------------------------------------------------
// MMA issuers: one warp per Q tile, taking turns
// ---------------------------------------------------------------------------
// Issuer t, per KV tile j:  [wait P_t(j), keys 0-63]    O_t += P V_j (keys 0-63)
//                           [wait P_t(j), keys 64-127]  O_t += P V_j (keys 64-127)
//                           S_t(j+1) = Q_t K_{j+1}^T
// The softmax hands P over in two halves, so the tensor core multiplies the
// first 64 keys of P into V while the softmax still finishes the second (at
// D = 128 the rest of its exponentials, at D = 64 its store to TMEM).
// S_t(j+1) overwrites the TMEM columns that hold P_t(j).  Both MMAs
// come from the same thread in that order, and the tensor core executes one
// thread's MMAs in issue order, so P_t(j) has been read before S_t(j+1)
// writes.  The S_FULL commit after S_t(j+1) fires only when every earlier
// MMA of the thread, including P_t(j) V_j, has completed, so the softmax may
// rescale O_t once it sees S_t(j+1).
//
// Turns (D = 128): the issuers submit their blocks of MMAs (an item's first
// S, then per KV tile the P.V and next S) strictly in turn, A B A B ..., by
// passing a token through the TURN barriers.  The tensor core then runs one
// tile's block to its end before the other's, and each tile's softmax
// overlaps the other tile's block.  Left to themselves the two issuers'
// MMAs interleaved on the tensor core: both S tiles completed together and
// both softmax groups then ran at the same time while the tensor core
// waited (a clock trace showed ~3,550 cycles per step against 2,048 of
// tensor work).  An issuer waits for its own operands (P, K, V) before it
// takes the token, so those waits overlap the other tile's submissions.  A
// block with nothing to compute (a tile that needs fewer KV tiles than the
// other) still waits for its turn and hands the token straight on, which
// keeps the strict alternation; a lock taken by whichever issuer is ready
// first measured 8-13% slower.
//
// A stage's K and V slots are released separately, each when both issuers
// have arrived: K with a commit after the issuer's S that read it, V with a
// commit after its P.V, or, for a KV tile the issuer's Q tile does not need
// (causal tails), with a plain arrive after waiting for the tile to land, so
// that an arrival can never count towards an earlier use of the slot.
// O_DONE is signalled only after an item's last P.V, for the epilogue.
template <int D>
__device__ __forceinline__ void attn_mma_role(const int t, const AttnParams& p, uint8_t* smem,
                                              uint64_t* bars, uint32_t tmem, const WaitCtl& ctl) {
  // Run by a whole warp: every lane waits and computes the operands, one
  // elected lane issues.  Operands computed by all lanes stay warp-uniform,
  // which keeps the issue of each tcgen05.mma short.
  using L = AttnLayout<D>;
  // (turns at D = 128 only: at D = 64 a tile's MMAs take a fraction of its
  // softmax, and the two softmax groups run better side by side)
  constexpr bool TURNS = (D == 128);
  constexpr uint32_t IDESC_S = idesc_bf16_f32(ATTN_BLOCK_M, ATTN_BLOCK_N, false);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(ATTN_BLOCK_M, L::O_N, true);
  const uint64_t q_desc = smem_desc_sw128(smem_u32(smem + L::Q_OFF) + t * L::TILE_BYTES, 16, 1024);
  const uint64_t k_desc = smem_desc_sw128(smem_u32(smem + L::K_OFF), 16, 1024);
  const uint64_t v_desc = smem_desc_sw128(smem_u32(smem + L::V_OFF), L::CHUNK_BYTES, 1024);
  const uint32_t s_tmem = tmem + static_cast<uint32_t>(t * ATTN_BLOCK_N);
  const uint32_t p_tmem = tmem + L::p_col(t);
  const uint32_t o_tmem = tmem + 256u + static_cast<uint32_t>(t) * L::O_STRIDE;
  constexpr unsigned FULL = 0xffffffffu;
  uint32_t q_uses = 0, p_cnt = 0;
  uint32_t turns = 0;     // blocks this issuer has submitted (TURNS only)
  uint32_t kv_it = 0;     // running KV tile index (stage = kv_it % STAGES)
  bool ok = true;
  AttnItem it;
  // S_t = Q_t K^T for the K tile in stage s
  auto issue_s = [&](int s) {
    const uint64_t kd = k_desc + static_cast<uint64_t>((s * L::TILE_BYTES) >> 4);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::CHUNK_BYTES + (kk & 3) * 32) >> 4);
      mma_bf16_ss(s_tmem, q_desc + off, kd + off, IDESC_S, kk > 0 ? 1u : 0u);
    }
  };
  // the token: tile 0 submits first; each issuer waits for the other's
  // previous block and hands its own on afterwards
  bool have_turn = false;
  auto take_turn = [&]() -> bool {
    if (!TURNS || have_turn) return true;
    have_turn = true;
    if (t == 0 && turns == 0) return true;
    const uint32_t parity = (t == 0 ? turns - 1u : turns) & 1u;
    return __all_sync(FULL, mbar_wait(&bars[L::B_TURN + t], parity, ctl));
  };
  auto pass_turn = [&]() -> bool {
    if (!TURNS) return true;
    bool r = take_turn();  // a block with nothing to compute still waits its turn
    if (r) {
      if (elect_one()) mbar_arrive(&bars[L::B_TURN + (1 - t)]);
      __syncwarp();
    }
    ++turns;
    have_turn = false;
    return r;
  };
  for (int k = 0; ok && attn_get_item(p, k, it); ++k) {
    if (t == 0 && it.kv_len_raw != it.kv_len && elect_one())
      atomicOr(p.status, ATTN_STATUS_BAD_KVLEN);
    if (it.nkv_max == 0) continue;
    const int nkv = t ? it.nkv[1] : it.nkv[0];
    // S_t(0), or the release of the item's first K tile
    {
      const int s = static_cast<int>(kv_it % L::STAGES);
      ok = __all_sync(FULL, mbar_wait(&bars[L::B_K_FULL + s], (kv_it / L::STAGES) & 1u, ctl));
      if (ok && nkv > 0) {
        ok = __all_sync(FULL, mbar_wait(&bars[L::B_Q_FULL + t], q_uses & 1u, ctl));
        ++q_uses;
        if (ok) ok = take_turn();
        if (ok) {
          tc_fence_after();
          if (elect_one()) {
            issue_s(s);
            mma_commit(&bars[L::B_S_FULL + t]);
            mma_commit(&bars[L::B_K_EMPTY + s]);
            if (nkv == 1) mma_commit(&bars[L::B_Q_EMPTY + t]);
          }
          __syncwarp();
        }
      } else if (ok) {
        if (elect_one()) mbar_arrive(&bars[L::B_K_EMPTY + s]);
        __syncwarp();
      }
      if (ok) ok = pass_turn();
    }
    for (int j = 0; ok && j < it.nkv_max; ++j, ++kv_it) {
      const int s = static_cast<int>(kv_it % L::STAGES);
      const uint32_t kv1 = kv_it + 1u;
      const int s1 = static_cast<int>(kv1 % L::STAGES);
      // V of stage s; with the row sum its second N atom is the ones tile
      const uint64_t vd =
          L::TC_ROWSUM
              ? smem_desc_sw128(smem_u32(smem + L::V_OFF) + s * L::TILE_BYTES,
                                static_cast<uint32_t>(L::ONES_OFF - L::V_OFF - s * L::TILE_BYTES),
                                1024)
              : v_desc + static_cast<uint64_t>((s * L::TILE_BYTES) >> 4);
      // O_t += P_t(j) V_j for the keys of one half of P
      auto issue_pv = [&](int half) {
#pragma unroll
        for (int kk = 4 * half; kk < 4 * half + 4; ++kk)
          mma_bf16_ts(o_tmem, p_tmem + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4),
                      IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
      };
      {
        // every operand of the block is waited for before the turn is taken,
        // so that the block's MMAs then go out back to back
        const bool has_k1 = j + 1 < it.nkv_max;
        ok = __all_sync(FULL, mbar_wait(&bars[L::B_V_FULL + s], (kv_it / L::STAGES) & 1u, ctl));
        if (ok && has_k1)
          ok = __all_sync(FULL, mbar_wait(&bars[L::B_K_FULL + s1], (kv1 / L::STAGES) & 1u, ctl));
        if (!ok) break;
        if (j < nkv) {
          const bool s_next = j + 1 < nkv;
          ok = __all_sync(FULL, mbar_wait(&bars[L::B_P_FULL + 2 * t], p_cnt & 1u, ctl));
          if (ok) ok = take_turn();
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) issue_pv(0);
          __syncwarp();
          ok = __all_sync(FULL, mbar_wait(&bars[L::B_P_FULL + 2 * t + 1], p_cnt & 1u, ctl));
          if (!ok) break;
          ++p_cnt;
          tc_fence_after();
          if (elect_one()) {
            issue_pv(1);
            // S_t(j+1) = Q_t K_{j+1}^T, after P_t(j) V_j
            if (s_next) issue_s(s1);
          }
          __syncwarp();
          // the other tile's block may follow on the tensor core (handing the
          // token on earlier, or through a spin on a shared word instead of
          // an mbarrier, measured no faster)
          ok = pass_turn();
          if (elect_one()) {
            if (s_next) mma_commit(&bars[L::B_S_FULL + t]);
            // V_j is free once this P.V completes, K_{j+1} once S_t(j+1) has;
            // O_t is final after the item's last P.V
            mma_commit(&bars[L::B_V_EMPTY + s]);
            if (j == nkv - 1) mma_commit(&bars[L::B_O_DONE + t]);
            if (s_next) {
              mma_commit(&bars[L::B_K_EMPTY + s1]);
              if (j + 2 == nkv) mma_commit(&bars[L::B_Q_EMPTY + t]);
            } else if (has_k1) {
              mbar_arrive(&bars[L::B_K_EMPTY + s1]);
            }
          }
          __syncwarp();
        } else {
          // nothing to compute for this Q tile: release V_j and K_{j+1}
          if (elect_one()) {
            mbar_arrive(&bars[L::B_V_EMPTY + s]);
            if (has_k1) mbar_arrive(&bars[L::B_K_EMPTY + s1]);
          }
          __syncwarp();
          ok = pass_turn();
        }
      }
    }
  }
  // Unwind: all MMAs issued by this warp complete before TMEM is freed.
  if (elect_one()) mma_commit(&bars[L::B_DRAIN + t]);
  __syncwarp();
  mbar_wait_drain(&bars[L::B_DRAIN + t], 0u, ctl.limit_ns);
}

// ---------------------------------------------------------------------------
// softmax / correction / epilogue group (128 threads, one query row each)
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void attn_softmax_role(const int t, const AttnParams& p,
                                                  uint64_t* bars, uint32_t tmem,
                                                  const WaitCtl& ctl) {
  using L = AttnLayout<D>;
  const int rloc = static_cast<int>(threadIdx.x & 127u);
  const uint32_t lane_base = static_cast<uint32_t>(threadIdx.x & 96u) << 16;
  const uint32_t s_tmem = tmem + static_cast<uint32_t>(t * ATTN_BLOCK_N) + lane_base;
  const uint32_t p_tmem = tmem + L::p_col(t) + lane_base;
  const uint32_t o_tmem = tmem + 256u + static_cast<uint32_t>(t) * L::O_STRIDE + lane_base;
  const float c = p.scale_log2;
  const bool causal = (p.mask_kind & ATTN_MASK_CAUSAL_BIT) != 0;
  uint32_t s_cnt = 0, o_cnt = 0;  // completions seen of S_FULL[t], O_DONE[t]
  bool ok = true;
  AttnItem it;
  for (int k = 0; ok && attn_get_item(p, k, it); ++k) {
    const int row0 = t ? it.row0[1] : it.row0[0];
    const int nkv = t ? it.nkv[1] : it.nkv[0];
    if (row0 >= p.Lq) continue;  // tile wholly past the end of the sequence
    const int r = row0 + rloc;
    int limit = it.kv_len;  // this row attends to keys [0, limit)
    if (causal) limit = min(limit, max(r + 1 + it.coff, 0));
    const bool padded_row = attn_padded_query(p, r, it.kv_len);
    float m = -INFINITY, l = 0.f, lb = 0.f;
    for (int j = 0; j < nkv; ++j) {
      ok = mbar_wait(&bars[L::B_S_FULL + t], s_cnt & 1u, ctl);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++s_cnt;
      tc_fence_after();
      uint32_t ra[32], rb[32], rc[32], rd[32];
      // d = 128: one load of the 128 columns (+0.5-1.5% over four of 32);
      // d = 64: two of 64 (+1-1.3%; one of 128 was from 1% faster to 4%
      // slower there)
      if constexpr (D == 128) {
        tmem_ld_32x32b_x128(s_tmem, ra, rb, rc, rd);
      } else {
        tmem_ld_32x32b_x64(s_tmem + 0u, ra, rb);
        tmem_ld_32x32b_x64(s_tmem + 64u, rc, rd);
      }
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
      // mask: keys at or past `limit` (causal diagonal, padding, end of keys)
      const int nvalid = limit - j * ATTN_BLOCK_N;
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
      const float m_tile = mx * c;  // scale > 0, so the max commutes with it
      const float m_new = fmaxf(m, m_tile);
      const bool need = m_new > m + ATTN_RESCALE_THRESHOLD;
      if (__any_sync(0xffffffffu, need && j > 0)) {
        // rescale this row's O accumulator.  P_t(j-1) V has completed: the
        // commit that signalled S_t(j) covers every earlier MMA of the issuer.
        const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
        const uint64_t a2 = f2_pack(alpha, alpha);
        // a rolled loop: the rescale is rare, and the softmax loop's code
        // stays small (bit-identical; unrolled it cost 1-6% at d = 128 in
        // instruction fetch)
#pragma unroll 1
        for (int cc = 0; cc < (L::O_N + 31) / 32; ++cc) {
          uint32_t ro[32];
          tmem_ld_32x32b_x32(o_tmem + cc * 32u, ro);
          tmem_ld_wait(ro);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(ro[2 * i]), __uint_as_float(ro[2 * i + 1])), a2),
                      x0, x1);
            ro[2 * i] = __float_as_uint(x0);
            ro[2 * i + 1] = __float_as_uint(x1);
          }
          tmem_st_32x32b_x32(o_tmem + cc * 32u, ro);
        }
        tmem_st_wait();
      }
      if (need) {
        const float alpha = ex2_approx(m - m_new);
        l *= alpha;
        lb *= alpha;
        m = m_new;
      }
      const float mb = (m == -INFINITY) ? 0.f : m;
      // p = 2^(s*c - m); P goes to TMEM as bf16 pairs.  Two row sums: l of
      // the fp32 p (for the LSE) and lb of the bf16-rounded p that the tensor
      // core multiplies into V (for the normalisation of O).
      const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-mb, -mb);
      uint64_t lf_a = 0ull, lf_b = 0ull;
      float lb_a = 0.f, lb_b = 0.f, lb_c = 0.f, lb_d = 0.f;
      // exponentials of the pairs [i0, i1) of one half (64 keys) of the tile
      auto exps = [&](int half, int i0, int i1, uint32_t* pk) {
#pragma unroll
        for (int i = i0; i < i1; i += 2) {
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
          if constexpr (!L::TC_ROWSUM) {
            lb_a = add_bf16lo_f32(lb_a, pk[i]);
            lb_b = add_bf16hi_f32(lb_b, pk[i]);
            lb_c = add_bf16lo_f32(lb_c, pk[i + 1]);
            lb_d = add_bf16hi_f32(lb_d, pk[i + 1]);
          }
        }
      };
      // Half 0 of P is stored, then exponentials of half 1 run while that
      // store completes; only then is half 0 handed to the MMA issuer, which
      // multiplies it into V while the rest of half 1 is computed.  Waiting
      // for the store right after it cost a store latency per half.  At
      // d = 128 half 0 goes after 32 of half 1's 64 exponentials; at d = 64
      // after all of them, just before half 1 is stored (measured: d = 64
      // +2-3%, d = 128 +0.2-0.6% over the per-half wait; at d = 64, handing
      // half 0 over only after half 1's store was 9-11% slower).
      constexpr int P_SPLIT = (D == 64) ? 32 : 16;  // pairs of half 1 before half 0 goes
      uint32_t pk0[32], pk1[32];
      exps(0, 0, 32, pk0);
      tmem_st_32x32b_x32(p_tmem, pk0);
      exps(1, 0, P_SPLIT, pk1);
      tmem_st_wait();
      reg_fence(pk0);  // the store has read pk0 before its registers are reused
      tc_fence_before();
      mbar_arrive(&bars[L::B_P_FULL + 2 * t]);
      exps(1, P_SPLIT, 32, pk1);
      tmem_st_32x32b_x32(p_tmem + 32u, pk1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[L::B_P_FULL + 2 * t + 1]);
      {
        float x0, x1;
        f2_unpack(f2_add(lf_a, lf_b), x0, x1);
        l += x0 + x1;
        lb += (lb_a + lb_b) + (lb_c + lb_d);
      }
    }
    if (!ok) break;
    // epilogue: O / lb (bf16), LSE; padded and empty rows are exactly 0 / -inf
    if (nkv > 0) {
      ok = mbar_wait(&bars[L::B_O_DONE + t], o_cnt & 1u, ctl);
      ++o_cnt;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
    }
    if constexpr (L::TC_ROWSUM) {
      // the sum of the bf16 P, from column D of the accumulator
      lb = 0.f;
      if (nkv > 0) {
        uint32_t rs[32];
        tmem_ld_32x32b_x32(o_tmem + static_cast<uint32_t>(D), rs);
        tmem_ld_wait(rs);
        lb = __uint_as_float(rs[0]);
      }
    }
    const bool in_range = r < p.Lq;
    const bool zero_row = padded_row || nkv == 0 || limit <= 0 || !(lb > 0.f);
    const float inv_l = zero_row ? 0.f : 1.0f / lb;
    __nv_bfloat16* orow = p.O + it.b * p.o_stride_b + it.h * p.o_stride_h +
                          static_cast<long long>(r) * p.o_stride_l;
#pragma unroll 1  // once per item: kept rolled, like the rescale
    for (int cc = 0; cc < D / 32; ++cc) {
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
        // one row per thread: a 32-byte store fills whole sectors
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
    if (p.LSE != nullptr && in_range) {
      const float lse = zero_row ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
      p.LSE[(static_cast<long long>(it.b) * p.H + it.h) * p.Lq + r] = lse;
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using L = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);

  if (threadIdx.x == 0) {
    for (int t = 0; t < ATTN_QTILES; ++t) {
      mbar_init(&bars[L::B_Q_FULL + t], 1);
      mbar_init(&bars[L::B_Q_EMPTY + t], 1);
      mbar_init(&bars[L::B_S_FULL + t], 1);
      mbar_init(&bars[L::B_P_FULL + 2 * t], 128);
      mbar_init(&bars[L::B_P_FULL + 2 * t + 1], 128);
      mbar_init(&bars[L::B_O_DONE + t], 1);
    }
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&bars[L::B_K_FULL + s], 1);
      mbar_init(&bars[L::B_V_FULL + s], 1);
      mbar_init(&bars[L::B_K_EMPTY + s], ATTN_QTILES);  // one arrival per MMA issuer
      mbar_init(&bars[L::B_V_EMPTY + s], ATTN_QTILES);
    }
    for (int t = 0; t < ATTN_QTILES; ++t) {
      mbar_init(&bars[L::B_DRAIN + t], 1);
      mbar_init(&bars[L::B_TURN + t], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (L::TC_ROWSUM) {
    // the ones operand of the row sum: bf16 1.0 everywhere (so its swizzle
    // does not matter), written once and read by the tensor core
    uint4* ones = reinterpret_cast<uint4*>(smem + L::ONES_OFF);
    for (int i = static_cast<int>(threadIdx.x); i < L::ONES_BYTES / 16; i += ATTN_THREADS)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
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

  // Register split: the two softmax warpgroups take 216 registers per
  // thread, the control warpgroup (MMA, TMA and two idle warps) 72; together
  // exactly the 384 x 168 registers the block is launched with (the host
  // refuses to launch a build whose launch register count differs).
  if (warp >= 8) {
    reg_dealloc<ATTN_REGS_CONTROL>();
    if (warp == 9) {
      if (lane == 0) attn_tma_role<D>(&tmQ, &tmK, &tmV, p, smem, bars, ctl);
    } else if (warp == 8 || warp == 10) {
      attn_mma_role<D>(warp == 8 ? 0 : 1, p, smem, bars, tmem, ctl);
    }
  } else {
    reg_alloc<ATTN_REGS_SOFTMAX>();
    attn_softmax_role<D>(warp >> 2, p, bars, tmem, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, ATTN_TMEM_COLS);
  }
}

// Output for sequences with no keys at all (Lk == 0): O = 0, LSE = -inf.
__global__ void attn_empty_keys_kernel(__nv_bfloat16* O, long long o_stride_b,
                                       long long o_stride_h, long long o_stride_l, float* LSE,
                                       int B, int H, int Lq, int D) {
  const long long rows = static_cast<long long>(B) * H * Lq;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < rows * D;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / D;
    const int col = static_cast<int>(i - row * D);
    const int r = static_cast<int>(row % Lq);
    const long long bh = row / Lq;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    O[b * o_stride_b + h * o_stride_h + static_cast<long long>(r) * o_stride_l + col] =
        __float2bfloat16(0.f);
    if (col == 0 && LSE != nullptr) LSE[row] = -INFINITY;
  }
}

}  // namespace gb300

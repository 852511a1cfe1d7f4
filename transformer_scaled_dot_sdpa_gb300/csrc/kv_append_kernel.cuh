// kv_append_kernel.cuh -- writes the new tokens' key and value rows into a
// device-resident K/V cache, the first step of a decode step with host
// buffers (attn_decode_host).  Sequence b holds kv_len_b valid keys after the
// step, the new ones last: new row i of (b, K/V head) goes to position
// kv_len_b - Lq + i ("Self-Attention 机制", section "Causal Mask": each new
// query then sees the cache up to and including its own key).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

// knew, vnew: [B, h_kv, Lq, d] staged new rows; K, V: [B, h_kv, Lk, d] caches;
// kv_lens: [B] (nullptr: every sequence fills the cache, kv_len = Lk).  One
// thread moves one 16-byte piece (8 bf16) of a row; rows whose position falls
// before the start of the cache (kv_len_b < Lq) are not written.
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ knew, const uint4* __restrict__ vnew,
                     uint4* __restrict__ K, uint4* __restrict__ V,
                     const int32_t* __restrict__ kv_lens, int B, int h_kv, int Lq, int Lk,
                     int pieces_per_row) {
  grid_dependency_wait();
  grid_launch_dependents();
  const long long n = static_cast<long long>(B) * h_kv * Lq * pieces_per_row;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / pieces_per_row;  // (b, K/V head, i)
    const int piece = static_cast<int>(idx - row * pieces_per_row);
    const int i = static_cast<int>(row % Lq);
    const long long bk = row / Lq;  // b * h_kv + K/V head
    const int b = static_cast<int>(bk / h_kv);
    int len = Lk;
    if (kv_lens != nullptr) {
      const int raw = kv_lens[b];
      len = raw < 0 ? 0 : (raw > Lk ? Lk : raw);
    }
    const int pos = len - Lq + i;  // < Lk because len <= Lk and i < Lq
    if (pos < 0) continue;
    const long long dst = (bk * Lk + pos) * pieces_per_row + piece;
    K[dst] = knew[idx];
    V[dst] = vnew[idx];
  }
}

}  // namespace gb300

// attn_weights_kernel.cuh -- the attention matrix A = softmax(Q K^T * scale + M)
// for inspection of small problems, rebuilt from the LSE that the forward
// kernel produced: A_ij = exp(scale * q_i . k_j - LSE_i) for a visible key,
// 0 for a masked one.  The tutorial snippets return A next to the output
// ("attention-mechanism" page, section "最小实现"; "多模态大模型学习笔记（十四）",
// section 2.3); the forward kernel never forms it, so this separate, plain
// CUDA-core kernel does, one (query, key) pair per thread.
#pragma once

#include <cuda_bf16.h>

namespace gb300 {

struct WeightsParams {
  const __nv_bfloat16* Q;  // [B, H, Lq, d]
  const __nv_bfloat16* K;  // [B, Hkv, Lk, d]
  const float* LSE;        // [B, H, Lq]
  float* A;                // [B, H, Lq, Lk]
  int B, H, Hkv, Lq, Lk, d;
  int mask_kind;           // bit 0 causal, bit 1 padding
  int causal_offset;       // causal: query i sees keys j <= i + causal_offset
  int offset_per_seq;      // 1: bottom-right causal with padding, offset kv_len_b - Lq
  const int32_t* kv_lens;
  float scale;
};

constexpr int WEIGHTS_TJ = 32;  // keys per block
constexpr int WEIGHTS_TI = 8;   // queries per block

// grid: (ceil(Lk/32), ceil(Lq/8), B*H); block: (32, 8); smem: (8 + 32) x d floats
__global__ void attn_weights_kernel(const WeightsParams p) {
  extern __shared__ float sh[];
  float* qs = sh;                       // [8][d]
  float* ks = sh + WEIGHTS_TI * p.d;    // [32][d]
  const int bh = static_cast<int>(blockIdx.z);
  const int b = bh / p.H, h = bh - b * p.H;
  const int kvh = h / (p.H / p.Hkv);
  const int i0 = static_cast<int>(blockIdx.y) * WEIGHTS_TI;
  const int j0 = static_cast<int>(blockIdx.x) * WEIGHTS_TJ;
  const int tid = static_cast<int>(threadIdx.y * blockDim.x + threadIdx.x);
  const int nthr = static_cast<int>(blockDim.x * blockDim.y);
  const __nv_bfloat16* qb = p.Q + (static_cast<long long>(bh) * p.Lq) * p.d;
  const __nv_bfloat16* kb = p.K + (static_cast<long long>(b) * p.Hkv + kvh) * p.Lk * p.d;
  for (int e = tid; e < WEIGHTS_TI * p.d; e += nthr) {
    const int ii = e / p.d, c = e - ii * p.d;
    qs[e] = (i0 + ii < p.Lq) ? __bfloat162float(qb[static_cast<long long>(i0 + ii) * p.d + c]) : 0.f;
  }
  for (int e = tid; e < WEIGHTS_TJ * p.d; e += nthr) {
    const int jj = e / p.d, c = e - jj * p.d;
    ks[e] = (j0 + jj < p.Lk) ? __bfloat162float(kb[static_cast<long long>(j0 + jj) * p.d + c]) : 0.f;
  }
  __syncthreads();
  const int i = i0 + static_cast<int>(threadIdx.y);
  const int j = j0 + static_cast<int>(threadIdx.x);
  if (i >= p.Lq || j >= p.Lk) return;
  // the same visible-key rule as the forward kernels (attn_causal_offset,
  // attn_padded_query): keys [0, limit) of row i
  int limit = p.Lk;
  int coff = p.causal_offset;
  if (p.mask_kind & 2) {
    int kl = p.kv_lens[b];
    kl = kl < 0 ? 0 : (kl > p.Lk ? p.Lk : kl);
    limit = (i >= kl && !p.offset_per_seq) ? 0 : kl;
    if (p.offset_per_seq) coff = kl - p.Lq;
  }
  if (p.mask_kind & 1) limit = min(limit, max(i + 1 + coff, 0));
  const float lse = p.LSE[static_cast<long long>(bh) * p.Lq + i];
  float a = 0.f;
  if (j < limit && lse > -INFINITY) {
    float dot = 0.f;
    for (int c = 0; c < p.d; ++c) dot = fmaf(qs[threadIdx.y * p.d + c], ks[threadIdx.x * p.d + c], dot);
    a = expf(dot * p.scale - lse);
  }
  p.A[(static_cast<long long>(bh) * p.Lq + i) * p.Lk + j] = a;
}

}  // namespace gb300

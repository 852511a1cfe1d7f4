// capi.cu -- host side of libgb300attn.so: argument validation, TMA tensor
// maps, kernel launch, and the device status word.  See include/gb300attn.h
// for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gb300attn.h"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_split_kernel.cuh"
#include "attn_weights_kernel.cuh"
#include "kv_append_kernel.cuh"
#include "gemm_kernel.cuh"
#include "probe_kernel.cuh"

namespace {

// Device status word: bits set by kernels (timeout, bad kv_len), read and
// cleared by attn_check_device_status().  One copy per device.
__device__ unsigned int g_status_word;

// Fixed scratch of mha_layer_fwd_noalloc (the layer's QKV projection and
// concatenated heads), for callers that cannot allocate device memory.  Host
// code must not use this name as a device pointer: the device address comes
// from cudaGetSymbolAddress (see noalloc_scratch_address).
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  long long l2_bytes = 0;
  unsigned int* status = nullptr;
  // one-time kernel set-up, done under g_mutex and published by the flags
  std::atomic<bool> attn_attr[4] = {false, false, false, false};
  std::atomic<bool> gemm_attr{false};
  int gemm_pairs = 0;  // CTA pairs of the GEMM kernel resident at once
  // attn_fwd_host: copy-in, copy-out and a second compute stream, and the
  // events that order them (created on first use)
  cudaStream_t host_in = nullptr, host_out = nullptr, host_comp = nullptr;
  cudaEvent_t host_ev[2 * 16 + 2] = {};
  void* noalloc_scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_mutex;
std::mutex g_host_mutex;  // one attn_fwd_host enqueue at a time (shared events)
DeviceState g_dev[kMaxDevices];
unsigned long long g_wait_limit_ns = kDefaultWaitLimitNs;
long long g_debug_skip_kv_load = -1;
int g_schedule = ATTN_SCHEDULE_AUTO;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

attn_status_t get_encode() {
  if (g_encode) return ATTN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return ATTN_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return ATTN_OK;
}

// Per-device state for the current device (lazily initialised).
attn_status_t device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    s.l2_bytes = l2;
    if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return ATTN_ERR_CUDA;
    s.status = static_cast<unsigned int*>(p);
    if (get_encode() != ATTN_OK) return ATTN_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  if (dev_out) *dev_out = dev;
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 4-D bf16 tensor map with a 64 x 128 box (the 128-row dimension is `row_dim`),
// 128-byte swizzle, zero fill out of bounds.
attn_status_t make_map_4d(CUtensorMap* m, const void* base, const cuuint64_t dims[4],
                          const cuuint64_t strides_bytes[3], const cuuint32_t box[4]) {
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Tensor map over a contiguous [B, H, L, d] bf16 tensor.
attn_status_t map_bhld(CUtensorMap* m, const void* base, int B, int H, int L, int d) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t str[3] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2,
                             (cuuint64_t)H * L * d * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  return make_map_4d(m, base, dims, str, box);
}

// Tensor map over one of the Q/K/V blocks of a packed [B, L, 3, H, d] tensor
// (base already offset to the block); dimension order (d, H, L, B).
attn_status_t map_packed(CUtensorMap* m, const void* base, int B, int H, int L, int d) {
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  const cuuint64_t str[3] = {(cuuint64_t)d * 2, (cuuint64_t)3 * H * d * 2,
                             (cuuint64_t)L * 3 * H * d * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  return make_map_4d(m, base, dims, str, box);
}

// Launch `kernel`; with `dependent`, as a programmatic dependent launch: it
// may start while the kernel ahead of it in the stream finishes, and waits
// for that kernel's completion (grid_dependency_wait) before it touches
// global memory.  Used between the library's own back-to-back kernels (the
// layer's three, the decode step's), where it hides the launch and set-up.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                          cudaStream_t stream, bool dependent, Args... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  std::memset(attr, 0, sizeof attr);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1u : 0u;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

template <int D, int SCHEDULE>
attn_status_t launch_attn(DeviceState* ds, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const gb300::AttnParams& p,
                          cudaStream_t stream, bool dependent = false) {
  constexpr bool split = SCHEDULE == ATTN_SCHEDULE_SPLIT_KEYS;
  const int attr_idx = (D == 64 ? 0 : 1) + (split ? 2 : 0);
  const int smem = split ? gb300::SplitLayout<D>::SMEM_BYTES : gb300::AttnLayout<D>::SMEM_BYTES;
  void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, gb300::AttnParams) =
      split ? gb300::attn_fwd_split_kernel<D> : gb300::attn_fwd_kernel<D>;
  if (!ds->attn_attr[attr_idx].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    // re-checked under the lock: of threads racing here, the first does the
    // set-up and the others find it done
    if (!ds->attn_attr[attr_idx].load(std::memory_order_relaxed)) {
      // The kernels hand registers between warpgroups (setmaxnreg); the split
      // adds up to exactly ATTN_THREADS x ATTN_REGS_AT_LAUNCH, so a build with
      // a different launch register count could wait forever: refuse it.
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return ATTN_ERR_CUDA;
      if (fa.numRegs != gb300::ATTN_REGS_AT_LAUNCH || fa.maxThreadsPerBlock < gb300::ATTN_THREADS)
        return ATTN_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return ATTN_ERR_CUDA;
      ds->attn_attr[attr_idx].store(true, std::memory_order_release);
    }
  }
  const int grid = p.n_items < ds->num_sms ? p.n_items : ds->num_sms;
  if (launch_kernel(kernel, static_cast<unsigned>(grid), gb300::ATTN_THREADS,
                    static_cast<size_t>(smem), stream, dependent, mq, mk, mv, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// Heads per group of the two-Q-tile item order.  One group (the plain
// heaviest-first order) unless the K/V of all heads exceeds three times the
// L2; then the largest divisor of B * H whose K/V (shared by kv_group query
// heads) fits in L2, provided each group still has at least four waves of
// items.  Measured at d = 128, causal, in 135.5 MB of L2:
//   B1 h32 L32768 (537 MB of K/V): groups of 8 heads 1401 TFLOP/s against
//     1372 under sustained load (1484 against 1502 in a short run); groups of
//     7, which leave a partial last group, 1240;
//   B1 h32 L16384 (268 MB): one group 1438, groups of 16 1320, of 8 1415;
//   B2 h32 L16384 (537 MB): groups of 16 1425, one group 1410.
int item_head_group(const DeviceState* ds, int B, int H, int H_kv, int Lk, int d,
                    int n_qblocks) {
  const int BH = B * H;
  const int kv_group = H / H_kv;
  const long long kv_head_bytes = 2ll * Lk * d * 2;  // K and V of one K/V head
  const long long min_items = 4ll * ds->num_sms;
  if (static_cast<long long>(B) * H_kv * kv_head_bytes <= 3 * ds->l2_bytes) return BH;
  for (int hg = BH; hg >= 1; --hg) {
    if (BH % hg != 0) continue;
    // K/V heads the group's query heads touch (one more when the group does
    // not start on a K/V head boundary)
    const long long kv_heads = hg / kv_group + (hg % kv_group != 0 ? 1 : 0);
    if (kv_heads * kv_head_bytes > ds->l2_bytes) continue;
    return static_cast<long long>(hg) * n_qblocks >= min_items ? hg : BH;
  }
  return BH;
}

// Bottom-right causal with per-sequence lengths: the queries are the last Lq
// tokens of each sequence, so each sequence has its own causal offset
// kv_len_b - Lq ("04. Self-Attention", section 七: a new token never sees a
// later one).
int bottom_right_per_sequence(int mask_kind) {
  return (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT) && (mask_kind & ATTN_MASK_PADDING) ? 1 : 0;
}

// Shared by attn_fwd and the layer: launch attention with prepared maps.
attn_status_t run_attention(DeviceState* ds, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, int packed, int B, int H, int H_kv, int Lq,
                            int Lk, int d, int mask_kind, const int32_t* kv_lens, float scale,
                            void* O, long long osb, long long osh, long long osl, float* LSE,
                            cudaStream_t stream, bool dependent = false) {
  gb300::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.kv_group = H / H_kv;
  // both causal alignments are one bit in the kernel plus an offset
  p.causal_offset = (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT) ? (Lk - Lq) : 0;
  p.offset_per_seq = bottom_right_per_sequence(mask_kind);
  p.mask_kind = (mask_kind & ATTN_MASK_PADDING) |
                ((mask_kind & (ATTN_MASK_CAUSAL | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) ? 1 : 0);
  p.packed = packed;
  p.kv_lens = kv_lens;
  const double sc = scale > 0.f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(d));
  p.scale_log2 = static_cast<float>(sc * 1.4426950408889634074);
  p.O = static_cast<__nv_bfloat16*>(O);
  p.o_stride_b = osb;
  p.o_stride_h = osh;
  p.o_stride_l = osl;
  // 256-bit O stores need every row start 32-byte aligned (the API asks for 16)
  p.o_v8 = aligned(O, 32) && (osb * 2) % 32 == 0 && (osh * 2) % 32 == 0 && (osl * 2) % 32 == 0;
  p.LSE = LSE;
  p.status = ds->status;
  int schedule;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    p.wait_limit_ns = g_wait_limit_ns;
    p.debug_skip_kv_load = g_debug_skip_kv_load;
    schedule = g_schedule;
  }
  if (schedule == ATTN_SCHEDULE_AUTO) {
    // Too few 256-row items to give every SM one: take the schedule with
    // 128-row items, which has twice as many (measured: 1.6-1.7x faster on
    // causal 1x8x4096 and 1x4x8192 at d = 128, slower from 256 items up).
    const long long items_two = static_cast<long long>(B) * H *
                                ((Lq + gb300::ATTN_ROWS_PER_ITEM - 1) / gb300::ATTN_ROWS_PER_ITEM);
    schedule = items_two < ds->num_sms ? ATTN_SCHEDULE_SPLIT_KEYS : ATTN_SCHEDULE_TWO_QTILES;
  }
  const bool split = schedule == ATTN_SCHEDULE_SPLIT_KEYS;
  const int rows = split ? gb300::SPLIT_ROWS : gb300::ATTN_ROWS_PER_ITEM;
  p.n_qblocks = (Lq + rows - 1) / rows;
  p.n_items = static_cast<int>(static_cast<long long>(B) * H * p.n_qblocks);
  p.head_group = split ? B * H : item_head_group(ds, B, H, H_kv, Lk, d, p.n_qblocks);
  if (split)
    return d == 64 ? launch_attn<64, ATTN_SCHEDULE_SPLIT_KEYS>(ds, mq, mk, mv, p, stream, dependent)
                   : launch_attn<128, ATTN_SCHEDULE_SPLIT_KEYS>(ds, mq, mk, mv, p, stream, dependent);
  return d == 64 ? launch_attn<64, ATTN_SCHEDULE_TWO_QTILES>(ds, mq, mk, mv, p, stream, dependent)
                 : launch_attn<128, ATTN_SCHEDULE_TWO_QTILES>(ds, mq, mk, mv, p, stream, dependent);
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box cols_box x rows_box.
attn_status_t map_2d(CUtensorMap* m, const void* base, int rows, int cols, int cols_box,
                     int rows_box) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)cols_box, (cuuint32_t)rows_box};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        str, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// C[M,N] = A[M,K] B[K,N]; sizes already validated.
attn_status_t run_gemm(DeviceState* ds, const void* A, const void* Bm, void* C, int M, int N,
                       int K, cudaStream_t stream, bool dependent = false) {
  CUtensorMap ma, mb;
  attn_status_t st;
  if ((st = map_2d(&ma, A, M, K, gb300::GEMM_BK, gb300::GEMM_BM_CTA)) != ATTN_OK) return st;
  if ((st = map_2d(&mb, Bm, K, N, 64, gb300::GEMM_BK)) != ATTN_OK) return st;
  if (!ds->gemm_attr.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    // re-checked under the lock, as in launch_attn
    if (!ds->gemm_attr.load(std::memory_order_relaxed)) {
      if (cudaFuncSetAttribute(gb300::gemm_bf16_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               gb300::GemmLayout::SMEM_BYTES) != cudaSuccess)
        return ATTN_ERR_CUDA;
      // The kernel is persistent: launch only as many pairs as can be resident
      // together (a TPC with one SM enabled cannot host a pair).
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof cfg);
      cfg.gridDim = dim3(static_cast<unsigned>(ds->num_sms & ~1), 1, 1);
      cfg.blockDim = dim3(gb300::GEMM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = gb300::GemmLayout::SMEM_BYTES;  // cluster size: the kernel's (2)
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, gb300::gemm_bf16_kernel, &cfg) !=
              cudaSuccess ||
          clusters < 1)
        return ATTN_ERR_CUDA;
      ds->gemm_pairs = clusters;
      ds->gemm_attr.store(true, std::memory_order_release);
    }
  }
  gb300::GemmParams p;
  std::memset(&p, 0, sizeof p);
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = (M + gb300::GEMM_BM - 1) / gb300::GEMM_BM;
  p.n_tiles = N / gb300::GEMM_BN;
  p.k_blocks = K / gb300::GEMM_BK;
  p.C = static_cast<__nv_bfloat16*>(C);
  p.c_v8 = aligned(C, 32) ? 1 : 0;  // rows are N * 2 bytes apart, a multiple of 512
  p.status = ds->status;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    p.wait_limit_ns = g_wait_limit_ns;
  }
  // A last wave that would leave pairs idle is run as half-width tiles when
  // those still fit in one wave: it then takes half as long.  Measured with
  // L2 flushed: 16384 x 1024 x 1024 (256 tiles on 76 pairs, 28 in the last
  // wave) and 16384 x 3072 x 1024 (768 tiles, 8 in the last wave).
  const int tiles = p.m_tiles * p.n_tiles;
  const int rem = tiles % ds->gemm_pairs;
  p.n_full = tiles;
  p.n_list = tiles;
  if (rem != 0 && 2 * rem <= ds->gemm_pairs) {
    p.n_full = tiles - rem;
    p.n_list = p.n_full + 2 * rem;
  }
  const int pairs = p.n_list < ds->gemm_pairs ? p.n_list : ds->gemm_pairs;
  if (launch_kernel(gb300::gemm_bf16_kernel, static_cast<unsigned>(2 * pairs),
                    gb300::GEMM_THREADS, gb300::GemmLayout::SMEM_BYTES, stream, dependent, ma, mb,
                    p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_TOO_LARGE: return "ATTN_ERR_TOO_LARGE";
    case ATTN_ERR_SELF_CHECK: return "ATTN_ERR_SELF_CHECK";
  }
  return "ATTN_STATUS_UNKNOWN";
}

void attn_set_wait_limit_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_wait_limit_ns = ns ? static_cast<unsigned long long>(ns) : kDefaultWaitLimitNs;
}

attn_status_t attn_set_schedule(int schedule) {
  if (schedule < ATTN_SCHEDULE_AUTO || schedule > ATTN_SCHEDULE_SPLIT_KEYS)
    return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_schedule = schedule;
  return ATTN_OK;
}

attn_status_t attn_probe_ex2(int blocks, int threads, int iters,
                             unsigned long long* timing_out, float* sink, void* stream) {
  static_assert(gb300::PROBE_CHAINS * gb300::PROBE_EX2_PER_LINK == ATTN_PROBE_EX2_PER_THREAD_ITER,
                "exp2 per thread and iteration");
  if (blocks < 1 || iters < 1 || threads < 32 || threads > 1024 || threads % 32 != 0 ||
      timing_out == nullptr || sink == nullptr)
    return ATTN_ERR_INVALID_ARG;
  gb300::ex2_probe_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      iters, timing_out, sink);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

void attn_debug_skip_kv_load(long long index) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_debug_skip_kv_load = index < 0 ? -1 : index;
}

attn_status_t attn_fwd(const void* Q, const void* K, const void* V, int B, int h, int Lq, int Lk,
                       int d_k, int d_v, int mask_kind, const int32_t* kv_lens, float scale,
                       void* O, float* LSE, void* stream) {
  return attn_fwd_gqa(Q, K, V, B, h, h, Lq, Lk, d_k, d_v, mask_kind, kv_lens, scale, O, LSE,
                      stream);
}

}  // extern "C"

namespace {

// Checks shared by attn_fwd_gqa and attn_fwd_host on everything but the
// pointers (no CUDA call).
attn_status_t check_attn_shape(int B, int h, int h_kv, int Lq, int Lk, int d_k, int d_v,
                               int mask_kind, float scale) {
  if (B < 0 || h < 0 || Lq < 0 || Lk < 0) return ATTN_ERR_INVALID_ARG;
  if (h_kv < 1 || (h > 0 && h % h_kv != 0)) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_PADDING | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_CAUSAL) && (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_k != d_v) return ATTN_ERR_UNSUPPORTED;
  if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
  // work items of the finer schedule (128 query rows each) must fit an int
  const long long n_qblocks = (static_cast<long long>(Lq) + gb300::SPLIT_ROWS - 1) / gb300::SPLIT_ROWS;
  if (static_cast<long long>(B) * h * n_qblocks >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Attention over contiguous [B, h, L, d] device buffers.
attn_status_t attn_device(DeviceState* ds, const void* Q, const void* K, const void* V, int B,
                          int h, int h_kv, int Lq, int Lk, int d, int mask_kind,
                          const int32_t* kv_lens, float scale, void* O, float* LSE,
                          cudaStream_t s) {
  const long long osl = d, osh = static_cast<long long>(Lq) * d, osb = osh * h;
  attn_status_t st;
  CUtensorMap mq, mk, mv;
  if ((st = map_bhld(&mq, Q, B, h, Lq, d)) != ATTN_OK) return st;
  if ((st = map_bhld(&mk, K, B, h_kv, Lk, d)) != ATTN_OK) return st;
  if ((st = map_bhld(&mv, V, B, h_kv, Lk, d)) != ATTN_OK) return st;
  return run_attention(ds, mq, mk, mv, 0, B, h, h_kv, Lq, Lk, d, mask_kind, kv_lens, scale, O,
                       osb, osh, osl, LSE, s);
}

// attn_fwd_host: where the device copies of Q, K, V, O, LSE and kv_lens live
// in the caller's workspace (byte offsets, 256-aligned).
struct HostLayout {
  size_t q, k, v, o, lse, kv, total;
};
constexpr int kHostMaxChunks = 16;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

HostLayout host_layout(int B, int h, int h_kv, int Lq, int Lk, int d) {
  HostLayout l;
  size_t off = 0;
  l.q = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * d * 2);
  l.k = off;
  off = align256(off + static_cast<size_t>(B) * h_kv * Lk * d * 2);
  l.v = off;
  off = align256(off + static_cast<size_t>(B) * h_kv * Lk * d * 2);
  l.o = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * d * 2);
  l.lse = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * 4);
  l.kv = off;
  off = align256(off + static_cast<size_t>(B) * 4);
  l.total = off;
  return l;
}

// The five-step layer on device buffers (arguments already validated).
attn_status_t layer_device(DeviceState* ds, const void* X, const void* W_QKV, const void* W_O,
                           int B, int L, int d_model, int h, int mask_kind,
                           const int32_t* kv_lens, float scale, void* Y, uint8_t* ws,
                           cudaStream_t s) {
  const int dk = d_model / h;
  const long long rows = static_cast<long long>(B) * L;
  const size_t qkv_bytes = static_cast<size_t>(rows) * 3 * d_model * 2;
  uint8_t* qkv = ws;
  uint8_t* cat = ws + ((qkv_bytes + 255) & ~static_cast<size_t>(255));
  attn_status_t st;
  // The three kernels go out as dependent launches: each starts while the
  // one ahead of it drains (measured on 8 x 2048 tokens, d_model 1024,
  // causal: 190.5 -> 185.4 us per layer).
  // step 1: QKV = X W_QKV  -> [B, L, 3, h, d_k]
  if ((st = run_gemm(ds, X, W_QKV, qkv, static_cast<int>(rows), 3 * d_model, d_model, s,
                     true)) != ATTN_OK)
    return st;
  // steps 2-4: split heads (strided tensor maps), attention, concat (strided store)
  CUtensorMap mq, mk, mv;
  const size_t blk = static_cast<size_t>(d_model) * 2;
  if ((st = map_packed(&mq, qkv, B, h, L, dk)) != ATTN_OK) return st;
  if ((st = map_packed(&mk, qkv + blk, B, h, L, dk)) != ATTN_OK) return st;
  if ((st = map_packed(&mv, qkv + 2 * blk, B, h, L, dk)) != ATTN_OK) return st;
  if ((st = run_attention(ds, mq, mk, mv, 1, B, h, h, L, L, dk, mask_kind, kv_lens, scale, cat,
                          static_cast<long long>(L) * d_model, dk, d_model, nullptr, s,
                          true)) != ATTN_OK)
    return st;
  // step 5: Y = Concat W_O
  return run_gemm(ds, cat, W_O, Y, static_cast<int>(rows), d_model, d_model, s, true);
}

// mha_layer_fwd_host: chunks of whole batch elements of at least 4096 tokens
// (so the projection GEMMs keep several waves of 256 x 256 tiles), at most 8;
// the workspace holds the device copies of X and Y, kv_lens and one layer
// scratch per compute stream.
struct LayerHostPlan {
  int per_b;
  size_t x, y, kv, scratch[2], total;
};

LayerHostPlan layer_host_plan(int B, int L, int d_model, int h) {
  LayerHostPlan pl;
  const long long rows = static_cast<long long>(B) * L;
  long long chunks = rows / 4096;
  chunks = chunks < 1 ? 1 : (chunks > 8 ? 8 : chunks);
  int per_b = static_cast<int>((B + chunks - 1) / chunks);
  // every chunk's rows must stay a multiple of the GEMM's 128-row tiles
  while (per_b < B && (static_cast<long long>(per_b) * L) % gb300::GEMM_BM_CTA != 0) ++per_b;
  if ((static_cast<long long>(per_b) * L) % gb300::GEMM_BM_CTA != 0) per_b = B;
  pl.per_b = per_b;
  const size_t xy = static_cast<size_t>(rows) * d_model * 2;
  const size_t scratch = mha_layer_workspace_bytes(per_b, L, d_model, h);
  size_t off = 0;
  pl.x = off;
  off = align256(off + xy);
  pl.y = off;
  off = align256(off + xy);
  pl.kv = off;
  off = align256(off + static_cast<size_t>(B) * 4);
  pl.scratch[0] = off;
  off = align256(off + scratch);
  pl.scratch[1] = off;
  off = align256(off + scratch);
  pl.total = off;
  return pl;
}

attn_status_t host_streams(DeviceState* ds) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (ds->host_in != nullptr) return ATTN_OK;
  cudaStream_t st[3] = {nullptr, nullptr, nullptr};
  for (auto& x : st)
    if (cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) != cudaSuccess) return ATTN_ERR_CUDA;
  for (auto& e : ds->host_ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return ATTN_ERR_CUDA;
  ds->host_out = st[1];
  ds->host_comp = st[2];
  ds->host_in = st[0];  // last: marks the set as ready
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd_gqa(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                           int Lq, int Lk, int d_k, int d_v, int mask_kind,
                           const int32_t* kv_lens, float scale, void* O, float* LSE,
                           void* stream) {
  // ---- host-side validation (no CUDA call before this point) ----
  attn_status_t st = check_attn_shape(B, h, h_kv, Lq, Lk, d_k, d_v, mask_kind, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || h == 0 || Lq == 0) return ATTN_OK;
  if (!O) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (Lk > 0 && (!Q || !K || !V)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(O, 16) || (LSE && !aligned(LSE, 4)) || (kv_lens && !aligned(kv_lens, 4)))
    return ATTN_ERR_MISALIGNED;
  if (Lk > 0 && (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16)))
    return ATTN_ERR_MISALIGNED;

  DeviceState* ds = nullptr;
  st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lk == 0) {
    const long long osl = d_v, osh = static_cast<long long>(Lq) * d_v, osb = osh * h;
    gb300::attn_empty_keys_kernel<<<256, 256, 0, s>>>(static_cast<__nv_bfloat16*>(O), osb, osh,
                                                     osl, LSE, B, h, Lq, d_v);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  return attn_device(ds, Q, K, V, B, h, h_kv, Lq, Lk, d_k, mask_kind, kv_lens, scale, O, LSE, s);
}

size_t attn_fwd_host_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d_k, int d_v) {
  if (check_attn_shape(B, h, h_kv, Lq, Lk, d_k, d_v, 0, 0.f) != ATTN_OK) return 0;
  return host_layout(B, h, h_kv, Lq, Lk, d_k).total;
}

attn_status_t attn_fwd_host(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                            int Lq, int Lk, int d_k, int d_v, int mask_kind,
                            const int32_t* kv_lens, float scale, void* O, float* LSE,
                            void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t st = check_attn_shape(B, h, h_kv, Lq, Lk, d_k, d_v, mask_kind, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || h == 0 || Lq == 0) return ATTN_OK;
  if (!O || (Lk > 0 && (!Q || !K || !V))) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  const HostLayout lay = host_layout(B, h, h_kv, Lq, Lk, d_k);
  if (!workspace || workspace_bytes < lay.total) return ATTN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != ATTN_OK) return st;
  if ((st = host_streams(ds)) != ATTN_OK) return st;
  std::lock_guard<std::mutex> host_lock(g_host_mutex);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* dQ = reinterpret_cast<__nv_bfloat16*>(ws + lay.q);
  __nv_bfloat16* dK = reinterpret_cast<__nv_bfloat16*>(ws + lay.k);
  __nv_bfloat16* dV = reinterpret_cast<__nv_bfloat16*>(ws + lay.v);
  __nv_bfloat16* dO = reinterpret_cast<__nv_bfloat16*>(ws + lay.o);
  float* dL = LSE ? reinterpret_cast<float*>(ws + lay.lse) : nullptr;
  int32_t* dkv = (mask_kind & ATTN_MASK_PADDING) ? reinterpret_cast<int32_t*>(ws + lay.kv) : nullptr;
  const int d = d_k;
  const int grp = h / h_kv;

  // Chunks of (b, K/V head) units, each with its query heads: whole batch
  // elements, or a group of K/V heads of one element.  Either way the
  // chunk's Q, K, V, O and LSE are contiguous, and every chunk has the same
  // work.  About kHostMaxChunks chunks, of at least 8 MB each.
  const size_t unit_bytes = static_cast<size_t>(grp) * Lq * d * 2 * 2 +
                            static_cast<size_t>(Lk) * d * 2 * 2;
  const size_t total_bytes = unit_bytes * B * h_kv;
  size_t target = total_bytes / (8u << 20);
  target = target < 1 ? 1 : (target > static_cast<size_t>(kHostMaxChunks) ? kHostMaxChunks : target);
  int per_b = 1, per_k = h_kv;  // batch elements / K/V heads per chunk
  if (target <= static_cast<size_t>(B)) {
    per_b = static_cast<int>((B + target - 1) / target);
  } else {
    const int groups = static_cast<int>((target + B - 1) / B);
    per_k = (h_kv + groups - 1) / groups;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = ds->host_ev;  // [0] start, [1] end, [2 + c % 16] inputs of chunk c, [18 + c % 16] chunk c done
  cudaError_t e = cudaEventRecord(ev[0], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_in, ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_out, ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_comp, ev[0], 0);
  if (e == cudaSuccess && dkv)
    e = cudaMemcpyAsync(dkv, kv_lens, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice,
                        ds->host_in);
  int c = 0;
  for (int b0 = 0; b0 < B && e == cudaSuccess && st == ATTN_OK; b0 += per_b) {
    const int nb = (b0 + per_b <= B) ? per_b : B - b0;
    for (int k0 = 0; k0 < h_kv && e == cudaSuccess && st == ATTN_OK; k0 += per_k, ++c) {
      const int nk = (k0 + per_k <= h_kv) ? per_k : h_kv - k0;
      const int hq = nk * grp;  // query heads of each batch element of the chunk
      const size_t q_off = (static_cast<size_t>(b0) * h + static_cast<size_t>(k0) * grp) * Lq;
      const size_t kv_off = (static_cast<size_t>(b0) * h_kv + k0) * static_cast<size_t>(Lk);
      const size_t q_rows = static_cast<size_t>(nb) * hq * Lq;
      const size_t kv_rows = static_cast<size_t>(nb) * nk * Lk;
      const size_t rb = static_cast<size_t>(d) * 2;
      // inputs
      e = cudaMemcpyAsync(dQ + q_off * d, static_cast<const uint8_t*>(Q) + q_off * rb, q_rows * rb,
                          cudaMemcpyHostToDevice, ds->host_in);
      if (e == cudaSuccess && kv_rows > 0)
        e = cudaMemcpyAsync(dK + kv_off * d, static_cast<const uint8_t*>(K) + kv_off * rb,
                            kv_rows * rb, cudaMemcpyHostToDevice, ds->host_in);
      if (e == cudaSuccess && kv_rows > 0)
        e = cudaMemcpyAsync(dV + kv_off * d, static_cast<const uint8_t*>(V) + kv_off * rb,
                            kv_rows * rb, cudaMemcpyHostToDevice, ds->host_in);
      if (e == cudaSuccess) e = cudaEventRecord(ev[2 + c % 16], ds->host_in);
      // compute: chunks alternate between two streams, so one chunk's last
      // CTAs and the next chunk's first ones share the GPU
      cudaStream_t cs = (c & 1) ? ds->host_comp : s;
      if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[2 + c % 16], 0);
      if (e != cudaSuccess) break;
      float* lse_c = dL ? dL + q_off : nullptr;
      if (Lk == 0) {
        const long long osl = d, osh = static_cast<long long>(Lq) * d, osb = osh * hq;
        gb300::attn_empty_keys_kernel<<<256, 256, 0, cs>>>(dO + q_off * d, osb, osh, osl, lse_c,
                                                            nb, hq, Lq, d);
        e = cudaGetLastError();
      } else {
        st = attn_device(ds, dQ + q_off * d, dK + kv_off * d, dV + kv_off * d, nb, hq, nk, Lq, Lk,
                         d, mask_kind, dkv ? dkv + b0 : nullptr, scale, dO + q_off * d, lse_c,
                         cs);
      }
      if (e == cudaSuccess && st == ATTN_OK) e = cudaEventRecord(ev[18 + c % 16], cs);
      // outputs
      if (e == cudaSuccess && st == ATTN_OK) e = cudaStreamWaitEvent(ds->host_out, ev[18 + c % 16], 0);
      if (e == cudaSuccess && st == ATTN_OK)
        e = cudaMemcpyAsync(static_cast<uint8_t*>(O) + q_off * rb, dO + q_off * d, q_rows * rb,
                            cudaMemcpyDeviceToHost, ds->host_out);
      if (e == cudaSuccess && st == ATTN_OK && LSE)
        e = cudaMemcpyAsync(LSE + q_off, lse_c, q_rows * 4, cudaMemcpyDeviceToHost, ds->host_out);
    }
  }
  // the caller's stream completes with the last copy out (which follows
  // every chunk's kernel)
  cudaError_t e2 = cudaEventRecord(ev[1], ds->host_out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev[1], 0);
  if (st != ATTN_OK) return st;
  return (e == cudaSuccess && e2 == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

namespace {

// Split-KV decode: the kernel cuts all (sequence, K/V head) pairs' key tiles
// into one equal range per CTA (decode_split in attn_fwd_split_kernel.cuh), so
// a pair's tiles are spread over at most min(CTAs, its tiles + 1) ranges: the
// partial-result slots each query row needs.
int decode_slots(int grid, int Lk) {
  const long long tiles = (static_cast<long long>(Lk) + gb300::ATTN_BLOCK_N - 1) / gb300::ATTN_BLOCK_N;
  return static_cast<int>(tiles + 1 < grid ? tiles + 1 : grid);
}

size_t decode_part_o_bytes(long long rows, int n_chunks, int d) {
  return (static_cast<size_t>(rows) * n_chunks * d * 4 + 255) / 256 * 256;
}

// attn_decode's scratch on a device with num_sms SMs: the partial O of every
// slot, then its (m, l, lb, 0)
size_t decode_workspace_bytes(int num_sms, int B, int h, int Lq, int Lk, int d) {
  const int slots = decode_slots(num_sms, Lk);
  const long long rows = static_cast<long long>(B) * h * Lq;
  return decode_part_o_bytes(rows, slots, d) + static_cast<size_t>(rows) * slots * 4 * sizeof(float);
}

// Argument checks shared by attn_decode and attn_decode_host (no CUDA call).
attn_status_t check_decode_shape(int B, int h, int h_kv, int Lq, int Lk, int d, int mask_kind,
                                 float scale) {
  if (B < 0 || h < 0 || Lq < 0 || Lk < 0) return ATTN_ERR_INVALID_ARG;
  if (h_kv < 1 || (h > 0 && h % h_kv != 0)) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_PADDING | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_CAUSAL) && (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (h > 0 && static_cast<long long>(h / h_kv) * Lq > gb300::SPLIT_ROWS)
    return ATTN_ERR_UNSUPPORTED;  // the query rows of one K/V head fill one 128-row tile
  if (static_cast<long long>(B) * h * Lq >= (1ll << 31) ||
      static_cast<long long>(B) * h_kv * ((static_cast<long long>(Lk) + 127) / 128) >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// attn_decode_host's workspace: staging for the new query rows and K/V rows,
// kv_lens, O and LSE; attn_decode's own workspace follows at `total`.
struct DecodeHostLayout {
  size_t q, knew, vnew, kv, o, lse, total;
};

DecodeHostLayout decode_host_layout(int B, int h, int h_kv, int Lq, int d) {
  DecodeHostLayout l;
  size_t off = 0;
  l.q = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * d * 2);
  l.knew = off;
  off = align256(off + static_cast<size_t>(B) * h_kv * Lq * d * 2);
  l.vnew = off;
  off = align256(off + static_cast<size_t>(B) * h_kv * Lq * d * 2);
  l.kv = off;
  off = align256(off + static_cast<size_t>(B) * 4);
  l.o = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * d * 2);
  l.lse = off;
  off = align256(off + static_cast<size_t>(B) * h * Lq * 4);
  l.total = off;
  return l;
}

// Split-KV decode on validated device buffers: the split kernel over
// (sequence, K/V head, key chunk) items, then the merge of the chunks.
attn_status_t decode_device(DeviceState* ds, const void* Q, const void* K, const void* V, int B,
                            int h, int h_kv, int Lq, int Lk, int d, int mask_kind,
                            const int32_t* kv_lens, float scale, void* O, float* LSE,
                            uint8_t* ws, cudaStream_t s);


attn_status_t decode_device(DeviceState* ds, const void* Q, const void* K, const void* V, int B,
                            int h, int h_kv, int Lq, int Lk, int d, int mask_kind,
                            const int32_t* kv_lens, float scale, void* O, float* LSE,
                            uint8_t* ws, cudaStream_t s) {
  attn_status_t st;
  if (Lk == 0) {
    const long long osl = d, osh = static_cast<long long>(Lq) * d, osb = osh * h;
    gb300::attn_empty_keys_kernel<<<256, 256, 0, s>>>(static_cast<__nv_bfloat16*>(O), osb, osh,
                                                     osl, LSE, B, h, Lq, d);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const int grid = ds->num_sms;
  const int slots = decode_slots(grid, Lk);
  const long long rows = static_cast<long long>(B) * h * Lq;

  CUtensorMap mq, mk, mv;
  if ((st = map_2d(&mq, Q, static_cast<int>(rows), d, 64, 128)) != ATTN_OK) return st;
  if ((st = map_bhld(&mk, K, B, h_kv, Lk, d)) != ATTN_OK) return st;
  if ((st = map_bhld(&mv, V, B, h_kv, Lk, d)) != ATTN_OK) return st;

  gb300::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.B = B;
  p.H = h;
  p.Lq = Lq;
  p.Lk = Lk;
  p.kv_group = h / h_kv;
  p.causal_offset = (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT) ? (Lk - Lq) : 0;
  p.offset_per_seq = bottom_right_per_sequence(mask_kind);
  p.mask_kind = (mask_kind & ATTN_MASK_PADDING) |
                ((mask_kind & (ATTN_MASK_CAUSAL | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) ? 1 : 0);
  p.kv_lens = kv_lens;
  const double sc = scale > 0.f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(d));
  p.scale_log2 = static_cast<float>(sc * 1.4426950408889634074);
  p.status = ds->status;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    p.wait_limit_ns = g_wait_limit_ns;
    p.debug_skip_kv_load = g_debug_skip_kv_load;
  }
  p.decode = 1;
  p.q_rows = p.kv_group * Lq;
  p.n_chunks = slots;
  p.n_qblocks = 1;
  p.n_items = grid;  // one CTA per SM; the kernel splits the key tiles among them
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float*>(ws + decode_part_o_bytes(rows, slots, d));
  // both kernels as dependent launches: the key split behind whatever the
  // caller (or attn_decode_host's cache append) ran last, the combine
  // behind the key split
  st = d == 64 ? launch_attn<64, ATTN_SCHEDULE_SPLIT_KEYS>(ds, mq, mk, mv, p, s, true)
               : launch_attn<128, ATTN_SCHEDULE_SPLIT_KEYS>(ds, mq, mk, mv, p, s, true);
  if (st != ATTN_OK) return st;
  const unsigned cgrid = static_cast<unsigned>((rows + 3) / 4);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(O);
  const cudaError_t e =
      d == 64 ? launch_kernel(gb300::attn_decode_combine_kernel<64>, cgrid, 128u, 0, s, true, p,
                              grid, rows, o, LSE)
              : launch_kernel(gb300::attn_decode_combine_kernel<128>, cgrid, 128u, 0, s, true, p,
                              grid, rows, o, LSE);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t attn_decode_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d) {
  if (B <= 0 || h <= 0 || h_kv <= 0 || Lq <= 0 || Lk <= 0 || (d != 64 && d != 128)) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds, nullptr) != ATTN_OK) return 0;
  return decode_workspace_bytes(ds->num_sms, B, h, Lq, Lk, d);
}

attn_status_t attn_decode(const void* Q, const void* K, const void* V, int B, int h, int h_kv,
                          int Lq, int Lk, int d, int mask_kind, const int32_t* kv_lens,
                          float scale, void* O, float* LSE, void* workspace,
                          size_t workspace_bytes, void* stream) {
  // ---- host-side validation (no CUDA call before this point) ----
  attn_status_t st = check_decode_shape(B, h, h_kv, Lq, Lk, d, mask_kind, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || h == 0 || Lq == 0) return ATTN_OK;
  if (!O) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (Lk > 0 && (!Q || !K || !V || !workspace)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(O, 16) || (LSE && !aligned(LSE, 4)) || (kv_lens && !aligned(kv_lens, 4)))
    return ATTN_ERR_MISALIGNED;
  if (Lk > 0 && (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) ||
                 !aligned(workspace, 256)))
    return ATTN_ERR_MISALIGNED;

  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != ATTN_OK) return st;
  if (Lk > 0 && workspace_bytes < attn_decode_workspace_bytes(B, h, h_kv, Lq, Lk, d))
    return ATTN_ERR_INVALID_ARG;
  return decode_device(ds, Q, K, V, B, h, h_kv, Lq, Lk, d, mask_kind, kv_lens, scale, O, LSE,
                       static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
}

size_t attn_decode_host_workspace_bytes(int B, int h, int h_kv, int Lq, int Lk, int d) {
  if (check_decode_shape(B, h, h_kv, Lq, Lk, d, 0, 0.f) != ATTN_OK || B == 0 || h == 0 ||
      Lq == 0 || Lk == 0)
    return 0;
  const size_t dec = attn_decode_workspace_bytes(B, h, h_kv, Lq, Lk, d);
  if (dec == 0) return 0;
  return decode_host_layout(B, h, h_kv, Lq, d).total + align256(dec);
}

attn_status_t attn_decode_host(const void* Q, const void* K_new, const void* V_new, void* K_cache,
                               void* V_cache, int B, int h, int h_kv, int Lq, int Lk, int d,
                               int mask_kind, const int32_t* kv_lens, float scale, void* O,
                               float* LSE, void* workspace, size_t workspace_bytes,
                               void* stream) {
  // ---- host-side validation: the arguments alone, then the device's SM
  // count (device_state, the first CUDA call) for the workspace size ----
  attn_status_t st = check_decode_shape(B, h, h_kv, Lq, Lk, d, mask_kind, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || h == 0 || Lq == 0) return ATTN_OK;
  if (Lk == 0) return ATTN_ERR_INVALID_ARG;  // the new rows need a cache to go into
  if (!Q || !K_new || !V_new || !K_cache || !V_cache || !O || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (!aligned(K_cache, 16) || !aligned(V_cache, 16) || !aligned(workspace, 256))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds, nullptr)) != ATTN_OK) return st;
  if (workspace_bytes < decode_host_layout(B, h, h_kv, Lq, d).total +
                            align256(decode_workspace_bytes(ds->num_sms, B, h, Lq, Lk, d)))
    return ATTN_ERR_INVALID_ARG;

  const DecodeHostLayout lay = decode_host_layout(B, h, h_kv, Lq, d);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_bytes = static_cast<size_t>(B) * h * Lq * d * 2;
  const size_t kv_bytes = static_cast<size_t>(B) * h_kv * Lq * d * 2;
  const bool padding = (mask_kind & ATTN_MASK_PADDING) != 0;
  int32_t* dkv = padding ? reinterpret_cast<int32_t*>(ws + lay.kv) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // inputs in: four copies on the caller's stream
  cudaError_t e = cudaMemcpyAsync(ws + lay.q, Q, q_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + lay.knew, K_new, kv_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + lay.vnew, V_new, kv_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && padding)
    e = cudaMemcpyAsync(dkv, kv_lens, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  // the new rows into the cache, then attention over it
  {
    const long long pieces = static_cast<long long>(B) * h_kv * Lq * (d / 8);
    const unsigned grid =
        static_cast<unsigned>(pieces / 256 + 1 < 4 * ds->num_sms ? pieces / 256 + 1 : 4 * ds->num_sms);
    gb300::kv_append_kernel<<<grid, 256, 0, s>>>(
        reinterpret_cast<const uint4*>(ws + lay.knew), reinterpret_cast<const uint4*>(ws + lay.vnew),
        static_cast<uint4*>(K_cache), static_cast<uint4*>(V_cache), dkv, B, h_kv, Lq, Lk, d / 8);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  float* dL = LSE ? reinterpret_cast<float*>(ws + lay.lse) : nullptr;
  st = decode_device(ds, ws + lay.q, K_cache, V_cache, B, h, h_kv, Lq, Lk, d, mask_kind, dkv,
                     scale, ws + lay.o, dL, ws + lay.total, s);
  if (st != ATTN_OK) return st;
  // outputs out
  e = cudaMemcpyAsync(O, ws + lay.o, q_bytes, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && LSE)
    e = cudaMemcpyAsync(LSE, dL, static_cast<size_t>(B) * h * Lq * 4, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_weights(const void* Q, const void* K, const float* LSE, int B, int h,
                           int h_kv, int Lq, int Lk, int d_k, int mask_kind,
                           const int32_t* kv_lens, float scale, float* A, void* stream) {
  if (B < 0 || h < 0 || Lq < 0 || Lk < 0 || d_k < 1 || d_k > 256) return ATTN_ERR_INVALID_ARG;
  if (h_kv < 1 || (h > 0 && h % h_kv != 0)) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_PADDING | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_CAUSAL) && (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || h == 0 || Lq == 0 || Lk == 0) return ATTN_OK;
  if (!Q || !K || !LSE || !A) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * h >= 65536 || static_cast<long long>(Lq) / 8 >= 65535)
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned(Q, 2) || !aligned(K, 2) || !aligned(LSE, 4) || !aligned(A, 4))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  gb300::WeightsParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.LSE = LSE;
  p.A = A;
  p.B = B;
  p.H = h;
  p.Hkv = h_kv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.d = d_k;
  p.mask_kind = (mask_kind & ATTN_MASK_PADDING) |
                ((mask_kind & (ATTN_MASK_CAUSAL | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) ? 1 : 0);
  p.causal_offset = (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT) ? (Lk - Lq) : 0;
  p.offset_per_seq = bottom_right_per_sequence(mask_kind);
  p.kv_lens = kv_lens;
  p.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  const dim3 grid((Lk + gb300::WEIGHTS_TJ - 1) / gb300::WEIGHTS_TJ,
                  (Lq + gb300::WEIGHTS_TI - 1) / gb300::WEIGHTS_TI, B * h);
  const dim3 block(gb300::WEIGHTS_TJ, gb300::WEIGHTS_TI);
  const size_t shm = static_cast<size_t>(gb300::WEIGHTS_TI + gb300::WEIGHTS_TJ) * d_k * sizeof(float);
  gb300::attn_weights_kernel<<<grid, block, shm, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t mha_layer_workspace_bytes(int B, int L, int d_model, int h) {
  if (B <= 0 || L <= 0 || d_model <= 0 || h <= 0 || d_model % h != 0) return 0;
  const size_t rows = static_cast<size_t>(B) * L;
  const size_t qkv = rows * 3 * d_model * 2;
  const size_t cat = rows * d_model * 2;
  const size_t qkv_aligned = (qkv + 255) & ~static_cast<size_t>(255);
  return qkv_aligned + cat;
}

attn_status_t attn_gemm_bf16(const void* A, const void* Bm, void* C, int M, int N, int K,
                             void* stream) {
  if (M < 0 || N < 0 || K < 0) return ATTN_ERR_INVALID_ARG;
  if (M % gb300::GEMM_BM_CTA != 0 || N % gb300::GEMM_BN != 0 || K % gb300::GEMM_BK != 0)
    return ATTN_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return ATTN_OK;
  if (K == 0) return ATTN_ERR_UNSUPPORTED;
  if (!A || !Bm || !C) return ATTN_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(Bm, 16) || !aligned(C, 16)) return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  return run_gemm(ds, A, Bm, C, M, N, K, static_cast<cudaStream_t>(stream));
}

attn_status_t mha_layer_fwd(const void* X, const void* W_QKV, const void* W_O, int B, int L,
                            int d_model, int h, int mask_kind, const int32_t* kv_lens,
                            float scale, void* Y, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (B < 0 || L < 0 || d_model <= 0 || h <= 0) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_PADDING | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_CAUSAL) && (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_model % h != 0) return ATTN_ERR_INVALID_ARG;
  const int dk = d_model / h;
  if (dk != 64 && dk != 128) return ATTN_ERR_UNSUPPORTED;
  if (d_model % gb300::GEMM_BN != 0) return ATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * L;
  if (rows % gb300::GEMM_BM_CTA != 0 || rows >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (!X || !W_QKV || !W_O || !Y || !workspace) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < mha_layer_workspace_bytes(B, L, d_model, h)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(W_QKV, 16) || !aligned(W_O, 16) || !aligned(Y, 16) ||
      !aligned(workspace, 256) || (kv_lens && !aligned(kv_lens, 4)))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  return layer_device(ds, X, W_QKV, W_O, B, L, d_model, h, mask_kind, kv_lens, scale, Y,
                      static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
}

size_t mha_layer_host_workspace_bytes(int B, int L, int d_model, int h) {
  const size_t one = mha_layer_workspace_bytes(B, L, d_model, h);
  if (one == 0) return 0;
  const LayerHostPlan pl = layer_host_plan(B, L, d_model, h);
  return pl.total;
}

attn_status_t mha_layer_fwd_host(const void* X, const void* W_QKV, const void* W_O, int B, int L,
                                 int d_model, int h, int mask_kind, const int32_t* kv_lens,
                                 float scale, void* Y, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (B < 0 || L < 0 || d_model <= 0 || h <= 0) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_PADDING | ATTN_MASK_CAUSAL_BOTTOM_RIGHT)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_CAUSAL) && (mask_kind & ATTN_MASK_CAUSAL_BOTTOM_RIGHT))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_model % h != 0) return ATTN_ERR_INVALID_ARG;
  const int dk = d_model / h;
  if (dk != 64 && dk != 128) return ATTN_ERR_UNSUPPORTED;
  if (d_model % gb300::GEMM_BN != 0) return ATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * L;
  if (rows % gb300::GEMM_BM_CTA != 0 || rows >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (!X || !W_QKV || !W_O || !Y || !workspace) return ATTN_ERR_INVALID_ARG;
  if ((mask_kind & ATTN_MASK_PADDING) && !kv_lens) return ATTN_ERR_INVALID_ARG;
  const LayerHostPlan pl = layer_host_plan(B, L, d_model, h);
  if (workspace_bytes < pl.total) return ATTN_ERR_INVALID_ARG;
  if (!aligned(W_QKV, 16) || !aligned(W_O, 16) || !aligned(workspace, 256))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  if ((st = host_streams(ds)) != ATTN_OK) return st;
  std::lock_guard<std::mutex> host_lock(g_host_mutex);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dX = ws + pl.x;
  uint8_t* dY = ws + pl.y;
  int32_t* dkv = (mask_kind & ATTN_MASK_PADDING) ? reinterpret_cast<int32_t*>(ws + pl.kv) : nullptr;
  const size_t row_bytes = static_cast<size_t>(d_model) * 2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = ds->host_ev;  // as in attn_fwd_host
  cudaError_t e = cudaEventRecord(ev[0], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_in, ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_out, ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_comp, ev[0], 0);
  if (e == cudaSuccess && dkv)
    e = cudaMemcpyAsync(dkv, kv_lens, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice,
                        ds->host_in);
  int c = 0;
  for (int b0 = 0; b0 < B && e == cudaSuccess && st == ATTN_OK; b0 += pl.per_b, ++c) {
    const int nb = (b0 + pl.per_b <= B) ? pl.per_b : B - b0;
    const size_t off = static_cast<size_t>(b0) * L * row_bytes;
    const size_t bytes = static_cast<size_t>(nb) * L * row_bytes;
    e = cudaMemcpyAsync(dX + off, static_cast<const uint8_t*>(X) + off, bytes,
                        cudaMemcpyHostToDevice, ds->host_in);
    if (e == cudaSuccess) e = cudaEventRecord(ev[2 + c % 16], ds->host_in);
    // the two compute streams alternate, each with its own layer scratch
    cudaStream_t cs = (c & 1) ? ds->host_comp : s;
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[2 + c % 16], 0);
    if (e != cudaSuccess) break;
    st = layer_device(ds, dX + off, W_QKV, W_O, nb, L, d_model, h, mask_kind,
                      dkv ? dkv + b0 : nullptr, scale, dY + off, ws + pl.scratch[c & 1], cs);
    if (st != ATTN_OK) break;
    e = cudaEventRecord(ev[18 + c % 16], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->host_out, ev[18 + c % 16], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(Y) + off, dY + off, bytes, cudaMemcpyDeviceToHost,
                          ds->host_out);
  }
  cudaError_t e2 = cudaEventRecord(ev[1], ds->host_out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev[1], 0);
  if (st != ATTN_OK) return st;
  return (e == cudaSuccess && e2 == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t mha_layer_fwd_noalloc(const void* X, const void* W_QKV, const void* W_O, int B,
                                    int L, int d_model, int h, int mask_kind,
                                    const int32_t* kv_lens, float scale, void* Y, void* stream) {
  const size_t need = mha_layer_workspace_bytes(B, L, d_model, h);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_TOO_LARGE;
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  void* scratch = nullptr;
  {
    // once per device, with that device current: the array's device address
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ds->noalloc_scratch == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return ATTN_ERR_CUDA;
      ds->noalloc_scratch = p;
    }
    scratch = ds->noalloc_scratch;
  }
  return mha_layer_fwd(X, W_QKV, W_O, B, L, d_model, h, mask_kind, kv_lens, scale, Y, scratch,
                       ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

attn_status_t attn_check_device_status(void* stream) {
  DeviceState* ds = nullptr;
  attn_status_t st = device_state(&ds, nullptr);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
#ifdef GB300_CHECKED
  unsigned int checks = 0;
  if (cudaMemcpyFromSymbol(&checks, gb300::g_check_word, sizeof checks) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (checks != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(gb300::g_check_word, &zero, sizeof zero) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_ERR_SELF_CHECK;
  }
#endif
  if (word & gb300::ATTN_STATUS_TIMEOUT) return ATTN_ERR_TIMEOUT;
  if (word & gb300::ATTN_STATUS_BAD_KVLEN) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int attn_is_checked_build(void) {
#ifdef GB300_CHECKED
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"

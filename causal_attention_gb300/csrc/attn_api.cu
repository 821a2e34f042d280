// C ABI of the attention library: argument checks, TMA descriptors, launches and
// the device error word.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "kernels.h"

namespace attn {

// Written by kernels whose bounded waits expire; read and cleared by
// attn_check_device_error. Kernels receive its device address as a parameter.
__device__ uint32_t g_error_word = 0;

namespace {

thread_local char g_last_cuda_error[256] = "";

attn_status cuda_fail(cudaError_t e, attn_status code) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return code;
}

constexpr int kMaxDevices = 32;

// Makes the current device's primary context current in this thread (once per
// thread and device), so that driver calls such as cuTensorMapEncodeTiled work in
// threads where only the runtime's device was set (e.g. autograd worker threads).
cudaError_t bind_device() {
  thread_local int bound = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (bound == dev) return cudaSuccess;
  e = cudaSetDevice(dev);
  if (e == cudaSuccess) bound = dev;
  return e;
}

uint32_t* error_word_ptr(cudaError_t* e) {
  static uint32_t* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  *e = bind_device();
  if (*e != cudaSuccess) return nullptr;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    *e = cudaGetSymbolAddress(&p, g_error_word);
    if (*e != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

// Streaming multiprocessors of the current device (cached per device).
int num_sms(cudaError_t* e) {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    *e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (*e != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so that the
// library does not link libcuda (it loads on machines without a GPU driver).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(cudaError_t* e) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t once_err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    once_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (once_err == cudaSuccess && q != cudaDriverEntryPointSuccess) once_err = cudaErrorSymbolNotFound;
    if (once_err == cudaSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  *e = once_err;
  return fn;
}

// A 3-D map over a [B*H, T, d] bf16 tensor with 128-row boxes of one swizzle
// width of columns. Rows past T (and heads past B*H) read as zero.
attn_status make_map(CUtensorMap* m, const void* ptr, int BH, int T, int d) {
  cudaError_t e = bind_device();
  if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
  EncodeTiledFn fn = encode_fn(&e);
  if (!fn) return cuda_fail(e, ATTN_ERR_CUDA);
  const int row_bytes = d * 2 >= 128 ? 128 : d * 2;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
  const cuuint32_t box[3] = {(cuuint32_t)(row_bytes / 2), 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle swz = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape limits: every index the kernels form stays in 32-bit where they use int,
// and every TMA dimension and stride within its encoding.
constexpr long long kMaxT = 1LL << 24;
constexpr long long kMaxBH = 1LL << 24;
constexpr long long kMaxElems = 1LL << 40;

attn_status check_shape(int B, int H, int T, int d) {
  if (B < 1 || H < 1 || T < 1) return ATTN_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > kMaxBH || T > kMaxT || bh * T * 128 > kMaxElems) return ATTN_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 80 && d != 128) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Grouped key/value heads: 1 <= H_kv <= H and H_kv divides H.
attn_status check_kv_heads(int H, int H_kv) {
  if (H_kv < 1 || H_kv > H || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status check_scale(float scale, int causal) {
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p) return ATTN_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

size_t workspace_bytes_for(int B, int H, int T) {
  return 2 * sizeof(float) * (size_t)B * H * (size_t)pad_rows(T);
}

// The fused dQ (d <= 64) appends the fp32 dQ tiles (B*H*T_pad*d floats) and one int32
// ordering counter per 128-row query tile, rounded up to 256 bytes.
size_t fused_workspace_bytes_for(int B, int H, int T, int d) {
  const size_t rows = (size_t)B * H * (size_t)pad_rows(T);
  const size_t cnt = ((size_t)B * H * (size_t)(pad_rows(T) / 128) * sizeof(int) + 255) / 256 * 256;
  return workspace_bytes_for(B, H, T) + rows * (size_t)d * sizeof(float) + cnt;
}

// Grouped key/value heads with few key/value heads: when there are fewer dK/dV work items
// (key tiles x key/value slices) than kSplitBelowItems (the SMs of a GB300), each item is
// split over the G query heads of its slice until there are at least kMinDkdvItems of them,
// so that the persistent kernel fills the device. Above one item per SM the fp32 partial
// sums and their reduction cost more than the better balance gains (measured at 256 items:
// 141.5 us split in two against 135 us unsplit). Fixed counts, not the device's, keep the
// result the same on every device.
constexpr int kSplitBelowItems = 152;
constexpr int kMinDkdvItems = 304;
int gqa_splits(int B, int H, int H_kv, int T) {
  const int G = H / H_kv;
  const long long items = (long long)B * H_kv * ((T + 127) / 128);
  if (G == 1 || items >= kSplitBelowItems) return 1;
  return (int)std::min<long long>(G, (kMinDkdvItems + items - 1) / items);
}

size_t gqa_workspace_bytes_for(int B, int H, int H_kv, int T, int d) {
  const int S = gqa_splits(B, H, H_kv, T);
  const size_t part = S > 1 ? 2 * (size_t)S * B * H_kv * (size_t)pad_rows(T) * d * sizeof(float) : 0;
  return workspace_bytes_for(B, H, T) + part;
}

bool fused_dq_ok(int d, size_t workspace_bytes, int B, int H, int T) {
  return d <= 64 && workspace_bytes >= fused_workspace_bytes_for(B, H, T, d);
}

attn_status check_workspace(const void* ws, size_t bytes, int B, int H, int T) {
  if (!ws || bytes < workspace_bytes_for(B, H, T)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(ws)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

#define ATTN_TRY(x)                   \
  do {                                \
    attn_status _s = (x);             \
    if (_s != ATTN_OK) return _s;     \
  } while (0)

// Backward arguments shared by the three stages (maps built only when needed).
attn_status bwd_args(BwdArgs* a, const void* q, const void* k, const void* v, const void* dO,
                     const void* workspace, int B, int H, int T, int d, float scale, int causal,
                     CUtensorMap* maps, bool need_maps) {
  memset(a, 0, sizeof(*a));
  a->T = T;
  a->T_pad = pad_rows(T);
  a->BH = B * H;
  a->G = 1;  // attn_bwd_gqa sets the group size
  a->S = 1;
  a->d = d;
  a->causal = causal;
  a->scale = scale;
  a->ws_nlse2 = static_cast<float*>(const_cast<void*>(workspace));
  a->ws_D = a->ws_nlse2 + (size_t)a->BH * a->T_pad;
  // fused-dQ parts (used only where the workspace is large enough and d <= 64)
  a->dq_acc = a->ws_D + (size_t)a->BH * a->T_pad;
  a->dq_cnt = reinterpret_cast<int*>(a->dq_acc + (size_t)a->BH * a->T_pad * d);
  cudaError_t e;
  a->err = error_word_ptr(&e);
  if (!a->err) return cuda_fail(e, ATTN_ERR_CUDA);
  a->num_sms = num_sms(&e);
  if (a->num_sms <= 0) return cuda_fail(e, ATTN_ERR_CUDA);
  if (need_maps) {
    ATTN_TRY(make_map(&maps[0], q, a->BH, T, d));
    ATTN_TRY(make_map(&maps[1], k, a->BH, T, d));  // remade over B * H_kv slices for grouped heads
    ATTN_TRY(make_map(&maps[2], v, a->BH, T, d));
    ATTN_TRY(make_map(&maps[3], dO, a->BH, T, d));
    a->tmQ = &maps[0];
    a->tmK = &maps[1];
    a->tmV = &maps[2];
    a->tmdO = &maps[3];
  }
  return ATTN_OK;
}

// dK and dV as tensor maps, for the d <= 64 dK/dV kernel's TMA-store epilogue.
attn_status bwd_map_dkdv(BwdArgs* a, const void* dk, const void* dv, CUtensorMap* maps) {
  if (a->d > 64) return ATTN_OK;
  ATTN_TRY(make_map(&maps[0], dk, a->BH / a->G, a->T, a->d));  // dK, dV: one per key/value slice
  ATTN_TRY(make_map(&maps[1], dv, a->BH / a->G, a->T, a->d));
  a->tmdK = &maps[0];
  a->tmdV = &maps[1];
  return ATTN_OK;
}

// O as a fifth tensor map, for the d <= 64 dQ kernel that stages it to form D itself.
attn_status bwd_map_o(BwdArgs* a, const void* o, CUtensorMap* map) {
  if (a->d > 64) return ATTN_OK;
  ATTN_TRY(make_map(map, o, a->BH, a->T, a->d));
  a->tmO = map;
  a->o = static_cast<const __nv_bfloat16*>(o);
  return ATTN_OK;
}

attn_status launched(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : cuda_fail(e, ATTN_ERR_LAUNCH); }

// ---------------------------------------------------------------------------
// Fixed scratch for attn_bwd_noalloc: the backward's two fp32 arrays of B*H*T_pad
// entries live in this array instead of a caller-allocated workspace. It is part of
// the library image, so every device that loads the library holds it until the
// process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB: B*H*T_pad <= 1,048,576
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device. Host code cannot use the
// symbol itself (on the host it names a stand-in, not device memory); the address is
// looked up once per device, with that device current, and cached.
void* noalloc_scratch_ptr(cudaError_t* e) {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  *e = bind_device();
  if (*e != cudaSuccess) return nullptr;
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    *e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*e != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

cudaError_t ensure_smem_attr(const void* func, int bytes, uint32_t* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint32_t bit = 1u << (dev & 31);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
  return e;
}

}  // namespace attn

using namespace attn;

extern "C" {

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int T, int d, float scale, int causal, void* stream) {
  return attn_fwd_gqa(q, k, v, o, lse, B, H, H, T, d, scale, causal, stream);
}

attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int H_kv, int T, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_kv_heads(H, H_kv));
  ATTN_TRY(check_scale(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, o, lse}));
  CUtensorMap maps[3];
  FwdArgs a;
  a.BH = B * H;
  a.G = H / H_kv;
  ATTN_TRY(make_map(&maps[0], q, a.BH, T, d));
  ATTN_TRY(make_map(&maps[1], k, B * H_kv, T, d));
  ATTN_TRY(make_map(&maps[2], v, B * H_kv, T, d));
  a.tmQ = &maps[0];
  a.tmK = &maps[1];
  a.tmV = &maps[2];
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.T = T;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  cudaError_t e;
  a.err = error_word_ptr(&e);
  if (!a.err) return cuda_fail(e, ATTN_ERR_CUDA);
  a.num_sms = num_sms(&e);
  if (a.num_sms <= 0) return cuda_fail(e, ATTN_ERR_CUDA);
  return launched(launch_fwd(a, static_cast<cudaStream_t>(stream)));
}

size_t attn_bwd_workspace_size(int B, int H, int T, int d) {
  if (check_shape(B, H, T, d) != ATTN_OK) return 0;
  return workspace_bytes_for(B, H, T);
}

size_t attn_bwd_gqa_workspace_size(int B, int H, int H_kv, int T, int d) {
  if (check_shape(B, H, T, d) != ATTN_OK || check_kv_heads(H, H_kv) != ATTN_OK) return 0;
  return gqa_workspace_bytes_for(B, H, H_kv, T, d);
}

size_t attn_bwd_fused_workspace_size(int B, int H, int T, int d) {
  if (check_shape(B, H, T, d) != ATTN_OK || d > 64) return 0;
  return fused_workspace_bytes_for(B, H, T, d);
}

attn_status attn_bwd_preprocess(const void* o, const void* dO, const float* lse, void* workspace,
                                size_t workspace_bytes, int B, int H, int T, int d, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_ptrs({o, dO, lse}));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  BwdArgs a;
  ATTN_TRY(bwd_args(&a, nullptr, nullptr, nullptr, dO, workspace, B, H, T, d, 1.f, 1, nullptr, false));
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dO = static_cast<const __nv_bfloat16*>(dO);
  a.lse = lse;
  if (!fused_dq_ok(d, workspace_bytes, B, H, T)) a.dq_cnt = nullptr;  // no counters to reset
  return launched(launch_bwd_preprocess(a, static_cast<cudaStream_t>(stream)));
}

attn_status attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                          void* dv, const void* workspace, size_t workspace_bytes, int B, int H,
                          int T, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_scale(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, dO, dk, dv}));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  BwdArgs a;
  CUtensorMap maps[6];
  ATTN_TRY(bwd_args(&a, q, k, v, dO, workspace, B, H, T, d, scale, causal, maps, true));
  ATTN_TRY(bwd_map_dkdv(&a, dk, dv, &maps[4]));
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  return launched(launch_bwd_dkdv(a, static_cast<cudaStream_t>(stream)));
}

attn_status attn_bwd_dkdv_dq(const void* q, const void* k, const void* v, const void* dO, void* dk,
                             void* dv, void* workspace, size_t workspace_bytes, int B, int H, int T,
                             int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_scale(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, dO, dk, dv}));
  if (d > 64) return ATTN_ERR_UNSUPPORTED;
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  if (!fused_dq_ok(d, workspace_bytes, B, H, T)) return ATTN_ERR_WORKSPACE;
  BwdArgs a;
  CUtensorMap maps[4];
  ATTN_TRY(bwd_args(&a, q, k, v, dO, workspace, B, H, T, d, scale, causal, maps, true));
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  return launched(launch_bwd_dkdv_dq(a, static_cast<cudaStream_t>(stream)));
}

attn_status attn_bwd_dq_finish(void* dq, const void* workspace, size_t workspace_bytes, int B, int H,
                               int T, int d, float scale, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_scale(scale, 1));
  ATTN_TRY(check_ptrs({dq}));
  if (d > 64) return ATTN_ERR_UNSUPPORTED;
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  if (!fused_dq_ok(d, workspace_bytes, B, H, T)) return ATTN_ERR_WORKSPACE;
  BwdArgs a;
  ATTN_TRY(bwd_args(&a, nullptr, nullptr, nullptr, nullptr, workspace, B, H, T, d, scale, 1, nullptr, false));
  a.dq = static_cast<__nv_bfloat16*>(dq);
  return launched(launch_bwd_dq_finish(a, static_cast<cudaStream_t>(stream)));
}

attn_status attn_bwd_dq(const void* q, const void* k, const void* v, const void* o, const void* dO,
                        const float* lse, void* dq, void* workspace, size_t workspace_bytes, int B, int H,
                        int T, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_scale(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, o, dO, lse, dq}));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  BwdArgs a;
  CUtensorMap maps[5];
  ATTN_TRY(bwd_args(&a, q, k, v, dO, workspace, B, H, T, d, scale, causal, maps, true));
  ATTN_TRY(bwd_map_o(&a, o, &maps[4]));
  a.lse = lse;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  return launched(launch_bwd_dq(a, static_cast<cudaStream_t>(stream)));
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int T, int d, float scale, int causal,
                     void* stream) {
  return attn_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, T, d, scale, causal,
                      stream);
}

attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, void* workspace,
                         size_t workspace_bytes, int B, int H, int H_kv, int T, int d, float scale,
                         int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  ATTN_TRY(check_kv_heads(H, H_kv));
  ATTN_TRY(check_scale(scale, causal));
  ATTN_TRY(check_ptrs({q, k, v, o, dO, lse, dq, dk, dv}));
  ATTN_TRY(check_workspace(workspace, workspace_bytes, B, H, T));
  BwdArgs a;
  CUtensorMap maps[7];
  ATTN_TRY(bwd_args(&a, q, k, v, dO, workspace, B, H, T, d, scale, causal, maps, true));
  a.G = H / H_kv;
  ATTN_TRY(make_map(&maps[1], k, B * H_kv, T, d));  // K, V: one slice per key/value head
  ATTN_TRY(make_map(&maps[2], v, B * H_kv, T, d));
  // few key/value heads: split dK/dV over the query heads when the workspace has room for
  // the partial sums (else one work item per key tile and key/value head)
  if (workspace_bytes >= gqa_workspace_bytes_for(B, H, H_kv, T, d)) {
    a.S = gqa_splits(B, H, H_kv, T);
    a.part = a.ws_D + (size_t)a.BH * a.T_pad;
  }
  ATTN_TRY(bwd_map_o(&a, o, &maps[4]));
  ATTN_TRY(bwd_map_dkdv(&a, dk, dv, &maps[5]));
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dO = static_cast<const __nv_bfloat16*>(dO);
  a.lse = lse;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  a.dq_cnt = nullptr;  // the fused dQ's counters are not used here
  if (d <= 64) {
    // the dQ kernel writes D and -LSE*log2(e) itself, then dK/dV reads them
    ATTN_TRY(launched(launch_bwd_dq(a, s)));
    return launched(launch_bwd_dkdv(a, s));
  }
  ATTN_TRY(launched(launch_bwd_preprocess(a, s)));
  ATTN_TRY(launched(launch_bwd_dkdv(a, s)));
  return launched(launch_bwd_dq(a, s));
}

attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                             int H, int T, int d, float scale, int causal, void* stream) {
  ATTN_TRY(check_shape(B, H, T, d));
  const size_t need = workspace_bytes_for(B, H, T);
  if (need > kNoAllocScratchBytes) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
             "attn_bwd_noalloc: B*H*T_pad = %zu rows needs %zu bytes of scratch; the fixed scratch "
             "holds %zu bytes (B*H*T_pad <= %zu, T_pad = T rounded up to 128); use attn_bwd",
             need / 8, need, kNoAllocScratchBytes, kNoAllocScratchBytes / 8);
    return ATTN_ERR_WORKSPACE;
  }
  cudaError_t e;
  void* scratch = noalloc_scratch_ptr(&e);
  if (!scratch) return cuda_fail(e, ATTN_ERR_CUDA);
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, T, d, scale,
                  causal, stream);
}

attn_status attn_check_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
  uint32_t word = 0;
  e = cudaMemcpyFromSymbolAsync(&word, g_error_word, sizeof(word), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "device error word 0x%x", word);
    return ATTN_ERR_DEVICE_TIMEOUT;
  }
  return ATTN_OK;
}

const char* attn_status_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension (d must be 32, 64, 80 or 128)";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel wait expired on the device";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
  }
  return "unknown status";
}

const char* attn_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"

// C ABI of the attention library: argument checks, TMA descriptors, launches and
// the device error word.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

// Written by kernels whose bounded waits expire; read and cleared by
// attn_check_device_error. Kernels receive its device address as a parameter.
__device__ uint32_t g_error_word = 0;

// Self-test of the bounded waits: one warp waits, through the same wait the kernels use,
// on an mbarrier that nothing ever arrives on. The wait runs out after its time limit,
// records the failure in the error word and returns; nothing faults or hangs.
__global__ void wait_timeout_selftest_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag, err};
  mbar_wait_warp(smem_u32(&bar), 0, ab, kErrTimeoutElem);
}

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

// ---------------------------------------------------------------------------
// Projections (training GEMMs around the attention)
// ---------------------------------------------------------------------------
attn_status encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box) {
  cudaError_t e = bind_device();
  if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
  EncodeTiledFn fn = encode_fn(&e);
  if (!fn) return cuda_fail(e, ATTN_ERR_CUDA);
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// A bf16 [Bn, Z, T, W] tensor as a 4-D map (W, T, Z, Bn) with boxes of 64 features x
// box_t tokens (128-byte swizzle): one map of a token view.
attn_status tok_map(CUtensorMap* m, const void* ptr, int W, int T, int Z, int Bn, int box_t) {
  const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)T, (cuuint64_t)Z, (cuuint64_t)Bn};
  const cuuint64_t strides[3] = {(cuuint64_t)W * 2, (cuuint64_t)T * W * 2, (cuuint64_t)Z * T * W * 2};
  const cuuint32_t box[4] = {64u, (cuuint32_t)box_t, 1u, 1u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box);
}

// A bf16 row-major [rows, cols] matrix as a 2-D map with boxes of 64 columns x box_r rows.
attn_status mat_map(CUtensorMap* m, const void* ptr, int cols, int rows, int box_r) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_r};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box);
}

// fp32 [S, M, N] partial sums (or the [M, N] result when S = 1) with 32 x 32 store boxes.
attn_status f32_out_map(CUtensorMap* m, void* ptr, int N, int M, int S) {
  const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)S};
  const cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)M * N * 4};
  const cuuint32_t box[3] = {32u, 32u, 1u};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box);
}

// A token view over one plain [Bn, T, F] activation.
attn_status plain_view(CUtensorMap* maps, TokView* v, const void* ptr, int Bn, int T, int F, int box_t) {
  v->W = F;
  v->f1 = v->f2 = INT_MAX;
  return tok_map(&maps[0], ptr, F, T, 1, Bn, box_t);
}

// A token view over head tensors: p0 [Bn, H0, T, d], then (optionally) p1 and p2
// [Bn, H1, T, d]: features h*d + c of p0, then of p1, then of p2.
attn_status head_view(CUtensorMap* maps, TokView* v, int Bn, int T, int d, int box_t, const void* p0, int H0,
                      const void* p1 = nullptr, const void* p2 = nullptr, int H1 = 0) {
  v->W = d;
  v->f1 = p1 ? H0 * d : INT_MAX;
  v->f2 = p2 ? (H0 + H1) * d : INT_MAX;
  ATTN_TRY(tok_map(&maps[0], p0, d, T, H0, Bn, box_t));
  if (p1) ATTN_TRY(tok_map(&maps[1], p1, d, T, H1, Bn, box_t));
  if (p2) ATTN_TRY(tok_map(&maps[2], p2, d, T, H1, Bn, box_t));
  return ATTN_OK;
}

constexpr int kGemmBM = 128, kGemmBK = 64;
// tn products with fewer output tiles than this (the SMs of a GB300) are split over K so
// that the persistent grid fills the device; the tile width is chosen against the same
// count. A fixed count, not the device's, keeps the result the same on every device.
constexpr int kGemmFillTiles = 152;

// The split count of a tn product with `tiles` output tiles and k_iters K-steps, and the
// K-steps of each split: at most one split per whole multiple of the output tiles that
// fits in kGemmFillTiles, at least 8 K-steps per split, at most 16 splits.
int gemm_splits(int tiles, int k_iters, int* k_per_split) {
  int S = std::max(1, kGemmFillTiles / tiles);
  S = std::min(S, std::max(1, k_iters / 8));
  S = std::min(S, 16);
  const int kps = (k_iters + S - 1) / S;
  *k_per_split = kps;
  return (k_iters + kps - 1) / kps;  // no empty split
}

// The output tile width of a product: 256 or 192 columns, whichever ends it in less
// tile-time: (waves of kGemmFillTiles work items) x (K-steps per item) x (the tile's cost:
// a 192-wide tile was measured at 0.9 of a 256-wide one, not 0.75); 256 on ties. For tn
// the split count follows the width's tile count.
int gemm_bn(int layout, int m_tiles, int N, int k_iters) {
  long long best = -1;
  int best_bn = 256;
  for (int bn : {256, 192}) {
    const long long tiles = (long long)m_tiles * ((N + bn - 1) / bn);
    long long items = tiles, iters = k_iters;
    if (layout == kGemmTN) {
      int kps;
      items = tiles * gemm_splits((int)std::min<long long>(tiles, INT_MAX), k_iters, &kps);
      iters = kps;
    }
    const long long cost = (items + kGemmFillTiles - 1) / kGemmFillTiles * iters * (bn == 256 ? 10 : 9);
    if (best < 0 || cost < best) {
      best = cost;
      best_bn = bn;
    }
  }
  return best_bn;
}

size_t tn_workspace_bytes(int M, int N, int k_iters) {
  const int m_tiles = (M + kGemmBM - 1) / kGemmBM;
  const int bn = gemm_bn(kGemmTN, m_tiles, N, k_iters);
  int kps;
  const int S = gemm_splits(m_tiles * ((N + bn - 1) / bn), k_iters, &kps);
  return S > 1 ? (size_t)S * M * N * sizeof(float) : 0;
}

// Sizes, tile counts and the error word of a product; the caller fills the maps and views.
attn_status gemm_params(GemmParams* p, int layout, int M, int N, int K, int T, int Bn, int* sms) {
  memset(p, 0, sizeof(*p));
  p->M = M;
  p->N = N;
  p->K = K;
  p->T = T;
  p->splits = 1;
  if (layout == kGemmTN) {
    p->nT = (T + kGemmBK - 1) / kGemmBK;  // 64-token K-steps per sequence
    p->m_tiles = (M + kGemmBM - 1) / kGemmBM;
    p->k_iters = Bn * p->nT;
  } else {
    p->nT = (T + kGemmBM - 1) / kGemmBM;  // 128-token row tiles per sequence
    p->m_tiles = Bn * p->nT;
    p->k_iters = (K + kGemmBK - 1) / kGemmBK;
  }
  p->bn = gemm_bn(layout, p->m_tiles, N, p->k_iters);
  p->n_tiles = (N + p->bn - 1) / p->bn;
  p->k_per_split = p->k_iters;
  if (layout == kGemmTN) p->splits = gemm_splits(p->m_tiles * p->n_tiles, p->k_iters, &p->k_per_split);
  cudaError_t e;
  p->err = error_word_ptr(&e);
  if (!p->err) return cuda_fail(e, ATTN_ERR_CUDA);
  *sms = num_sms(&e);
  if (*sms <= 0) return cuda_fail(e, ATTN_ERR_CUDA);
  return ATTN_OK;
}

// Runs a tn product into out (fp32 [M, N]): straight, or through S partial slices in the
// workspace and the in-order reduction.
attn_status run_tn(GemmParams* p, void* out, void* ws, size_t ws_bytes, int sms, cudaStream_t s) {
  const size_t need = p->splits > 1 ? (size_t)p->splits * p->M * p->N * sizeof(float) : 0;
  if (need > 0 && (!ws || ws_bytes < need)) return ATTN_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return ATTN_ERR_MISALIGNED;
  ATTN_TRY(f32_out_map(&p->c[0], need > 0 ? ws : out, p->N, p->M, p->splits));
  ATTN_TRY(launched(launch_gemm(kGemmTN, *p, sms, s)));
  if (need > 0)
    ATTN_TRY(launched(launch_splitk_reduce(static_cast<const float*>(ws), static_cast<float*>(out),
                                           (long long)p->M * p->N, p->splits, sms, s)));
  return ATTN_OK;
}

// Shape checks of the projections: every size >= 1, head dim 64 or 128 (a 64-feature box
// never straddles two heads), model width a multiple of 8 (16-byte rows).
attn_status check_proj(int B, int T, int C, int H, int H_kv, int d) {
  if (B < 1 || T < 1 || C < 1 || H < 1) return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_kv_heads(H, H_kv));
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (C % 8 != 0) return ATTN_ERR_INVALID_ARG;
  const long long tokens = (long long)B * T, feats = (long long)(H + 2 * H_kv) * d;
  if (T > kMaxT || tokens > kMaxBH || feats > kMaxBH || C > kMaxBH || tokens * std::max<long long>(feats, C) > kMaxElems)
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

size_t proj_bwd_workspace_bytes(int B, int T, int C, int H, int H_kv, int d) {
  const int k_iters = B * ((T + kGemmBK - 1) / kGemmBK);
  const size_t dwo = tn_workspace_bytes(C, H * d, k_iters);
  const size_t dwqkv = tn_workspace_bytes((H + 2 * H_kv) * d, C, k_iters);
  // the rotated-back dQ and dK (bf16) come first when RoPE is used
  const size_t rot = (size_t)B * (H + H_kv) * (size_t)T * d * 2;
  const size_t rot_pad = (rot + 255) / 256 * 256;
  return std::max(dwo, rot_pad + dwqkv);
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
    return (word & kErrBounds) ? ATTN_ERR_DEVICE_BOUNDS : ATTN_ERR_DEVICE_TIMEOUT;
  }
  return ATTN_OK;
}

const char* attn_status_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED:
      return "unsupported head dimension (attention: d in {32, 64, 80, 128}; projections: d in {64, 128})";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel wait expired on the device";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case ATTN_ERR_DEVICE_BOUNDS: return "a kernel found an index out of range (bounds-checked build)";
  }
  return "unknown status";
}

const char* attn_last_cuda_error(void) { return g_last_cuda_error; }

attn_status attn_selftest_wait_timeout(void* stream) {
  cudaError_t e;
  uint32_t* err = error_word_ptr(&e);
  if (!err) return cuda_fail(e, ATTN_ERR_CUDA);
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  return launched(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Projections
// ---------------------------------------------------------------------------
size_t attn_gemm_workspace_size(int M, int N, int K, int layout) {
  if (M < 1 || N < 1 || K < 1 || layout < 0 || layout > 2) return 0;
  if (layout != kGemmTN) return 0;
  return tn_workspace_bytes(M, N, (K + kGemmBK - 1) / kGemmBK);
}

attn_status attn_gemm(const void* a, const void* b, void* c, int M, int N, int K, int layout, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || layout < 0 || layout > 2) return ATTN_ERR_INVALID_ARG;
  if (M % 8 || N % 8 || K % 8) return ATTN_ERR_INVALID_ARG;
  if ((long long)M * K > kMaxElems || (long long)N * K > kMaxElems || (long long)M * N > kMaxElems ||
      M > kMaxT || N > kMaxT || K > kMaxT)
    return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_ptrs({a, b, c}));
  GemmParams p;
  int sms = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (layout == kGemmTN) {
    // A [K, M] and B [K, N]: K plays the token dimension (one sequence of K tokens)
    ATTN_TRY(gemm_params(&p, layout, M, N, K, K, 1, &sms));
    ATTN_TRY(plain_view(p.a, &p.va, a, 1, K, M, kGemmBK));
    ATTN_TRY(plain_view(p.b, &p.vb, b, 1, K, N, kGemmBK));
    return run_tn(&p, c, workspace, workspace_bytes, sms, s);
  }
  // A [M, K]: M plays the token dimension
  ATTN_TRY(gemm_params(&p, layout, M, N, K, M, 1, &sms));
  ATTN_TRY(plain_view(p.a, &p.va, a, 1, M, K, kGemmBM));
  if (layout == kGemmNT)
    ATTN_TRY(mat_map(&p.b[0], b, K, N, p.bn / 2));  // B [N, K]
  else
    ATTN_TRY(mat_map(&p.b[0], b, N, K, 64));  // B [K, N]
  ATTN_TRY(plain_view(p.c, &p.vc, c, 1, M, N, 32));
  return launched(launch_gemm(layout, p, sms, s));
}

attn_status attn_rope_table(float* tab, int T, int d, void* stream) {
  if (T < 1 || T > kMaxT || d < 2 || d % 8 != 0 || d > 1024) return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_ptrs({tab}));
  cudaError_t e = bind_device();
  if (e != cudaSuccess) return cuda_fail(e, ATTN_ERR_CUDA);
  return launched(launch_rope_table(tab, T, d, static_cast<cudaStream_t>(stream)));
}

attn_status attn_rope(const void* x, void* y, const float* rope_tab, int B, int H, int T, int d, int inverse,
                      void* stream) {
  if (B < 1 || H < 1 || T < 1 || T > kMaxT || (long long)B * H > kMaxBH) return ATTN_ERR_INVALID_ARG;
  if (d < 8 || d % 8 != 0 || (inverse != 0 && inverse != 1)) return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_ptrs({x, y, rope_tab}));
  cudaError_t e;
  const int sms = num_sms(&e);
  if (sms <= 0) return cuda_fail(e, ATTN_ERR_CUDA);
  return launched(launch_rope_apply(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), H, nullptr,
                                    nullptr, 0, rope_tab, B, T, d, inverse, sms, static_cast<cudaStream_t>(stream)));
}

attn_status attn_qkv_proj(const void* x, const void* w_qkv, void* q, void* k, void* v, const float* rope_tab, int B,
                          int T, int C, int H, int H_kv, int d, void* stream) {
  ATTN_TRY(check_proj(B, T, C, H, H_kv, d));
  ATTN_TRY(check_ptrs({x, w_qkv, q, k, v}));
  if (rope_tab && !aligned16(rope_tab)) return ATTN_ERR_MISALIGNED;
  const int N = (H + 2 * H_kv) * d;
  GemmParams p;
  int sms = 0;
  ATTN_TRY(gemm_params(&p, kGemmNT, B * T, N, C, T, B, &sms));
  ATTN_TRY(plain_view(p.a, &p.va, x, B, T, C, kGemmBM));
  ATTN_TRY(mat_map(&p.b[0], w_qkv, C, N, p.bn / 2));
  ATTN_TRY(head_view(p.c, &p.vc, B, T, d, 32, q, H, k, v, H_kv));
  if (rope_tab) {
    p.rope_features = (H + H_kv) * d;  // q and k
    p.rope_half = d / 2;
    p.rope_tab = rope_tab;
  }
  return launched(launch_gemm(kGemmNT, p, sms, static_cast<cudaStream_t>(stream)));
}

attn_status attn_out_proj(const void* o, const void* w_o, void* y, int B, int T, int H, int d, int C, void* stream) {
  ATTN_TRY(check_proj(B, T, C, H, H, d));
  ATTN_TRY(check_ptrs({o, w_o, y}));
  GemmParams p;
  int sms = 0;
  ATTN_TRY(gemm_params(&p, kGemmNT, B * T, C, H * d, T, B, &sms));
  ATTN_TRY(head_view(p.a, &p.va, B, T, d, kGemmBM, o, H));
  ATTN_TRY(mat_map(&p.b[0], w_o, H * d, C, p.bn / 2));
  ATTN_TRY(plain_view(p.c, &p.vc, y, B, T, C, 32));
  return launched(launch_gemm(kGemmNT, p, sms, static_cast<cudaStream_t>(stream)));
}

size_t attn_proj_bwd_workspace_size(int B, int T, int C, int H, int H_kv, int d) {
  if (check_proj(B, T, C, H, H_kv, d) != ATTN_OK) return 0;
  return proj_bwd_workspace_bytes(B, T, C, H, H_kv, d);
}

attn_status attn_out_proj_bwd(const void* dy, const void* o, const void* w_o, void* d_o, float* dw_o, void* workspace,
                              size_t workspace_bytes, int B, int T, int H, int d, int C, void* stream) {
  ATTN_TRY(check_proj(B, T, C, H, H, d));
  ATTN_TRY(check_ptrs({dy, o, w_o, d_o, dw_o}));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmParams p;
  int sms = 0;
  // dO = split(dY W_o): nn, M = tokens, N = H d, K = C
  ATTN_TRY(gemm_params(&p, kGemmNN, B * T, H * d, C, T, B, &sms));
  ATTN_TRY(plain_view(p.a, &p.va, dy, B, T, C, kGemmBM));
  ATTN_TRY(mat_map(&p.b[0], w_o, H * d, C, 64));  // W_o [C, H d] as [K, N]
  ATTN_TRY(head_view(p.c, &p.vc, B, T, d, 32, d_o, H));
  ATTN_TRY(launched(launch_gemm(kGemmNN, p, sms, s)));
  // dW_o = dY^T merge(O): tn, M = C, N = H d, K = tokens
  ATTN_TRY(gemm_params(&p, kGemmTN, C, H * d, B * T, T, B, &sms));
  ATTN_TRY(plain_view(p.a, &p.va, dy, B, T, C, kGemmBK));
  ATTN_TRY(head_view(p.b, &p.vb, B, T, d, kGemmBK, o, H));
  return run_tn(&p, dw_o, workspace, workspace_bytes, sms, s);
}

attn_status attn_qkv_proj_bwd(const void* dq, const void* dk, const void* dv, const void* x, const void* w_qkv,
                              const float* rope_tab, void* dx, float* dw_qkv, void* workspace, size_t workspace_bytes,
                              int B, int T, int C, int H, int H_kv, int d, void* stream) {
  ATTN_TRY(check_proj(B, T, C, H, H_kv, d));
  ATTN_TRY(check_ptrs({dq, dk, dv, x, w_qkv, dx, dw_qkv}));
  if (rope_tab && !aligned16(rope_tab)) return ATTN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = (H + 2 * H_kv) * d;
  size_t rot_pad = 0;
  if (rope_tab) {
    // dQ and dK rotated back (the inverse rotation) into the front of the workspace
    const size_t rq = (size_t)B * H * T * d, rk = (size_t)B * H_kv * T * d;
    rot_pad = ((rq + rk) * 2 + 255) / 256 * 256;
    if (!workspace || workspace_bytes < rot_pad) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
    __nv_bfloat16* wq = static_cast<__nv_bfloat16*>(workspace);
    __nv_bfloat16* wk = wq + rq;
    cudaError_t e;
    const int sms = num_sms(&e);
    if (sms <= 0) return cuda_fail(e, ATTN_ERR_CUDA);
    ATTN_TRY(launched(launch_rope_apply(static_cast<const __nv_bfloat16*>(dq), wq, H,
                                        static_cast<const __nv_bfloat16*>(dk), wk, H_kv, rope_tab, B, T, d, 1, sms, s)));
    dq = wq;
    dk = wk;
  }
  GemmParams p;
  int sms = 0;
  // dX = merge(dQ, dK, dV) W_qkv: nn, M = tokens, N = C, K = (H + 2 H_kv) d
  ATTN_TRY(gemm_params(&p, kGemmNN, B * T, C, N, T, B, &sms));
  ATTN_TRY(head_view(p.a, &p.va, B, T, d, kGemmBM, dq, H, dk, dv, H_kv));
  ATTN_TRY(mat_map(&p.b[0], w_qkv, C, N, 64));  // W_qkv [N, C] as [K, N]
  ATTN_TRY(plain_view(p.c, &p.vc, dx, B, T, C, 32));
  ATTN_TRY(launched(launch_gemm(kGemmNN, p, sms, s)));
  // dW_qkv = merge(dQ, dK, dV)^T X: tn, M = (H + 2 H_kv) d, N = C, K = tokens
  ATTN_TRY(gemm_params(&p, kGemmTN, N, C, B * T, T, B, &sms));
  ATTN_TRY(head_view(p.a, &p.va, B, T, d, kGemmBK, dq, H, dk, dv, H_kv));
  ATTN_TRY(plain_view(p.b, &p.vb, x, B, T, C, kGemmBK));
  void* ws_tn = workspace ? static_cast<char*>(workspace) + rot_pad : nullptr;
  const size_t ws_tn_bytes = workspace_bytes > rot_pad ? workspace_bytes - rot_pad : 0;
  return run_tn(&p, dw_qkv, ws_tn, ws_tn_bytes, sms, s);
}

}  // extern "C"

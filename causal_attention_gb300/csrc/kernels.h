// Host-side launch interface between the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

namespace attn {

struct FwdArgs {
  const CUtensorMap* tmQ;  // 3-D maps over [B*H, T, d] bf16, 128-row boxes
  const CUtensorMap* tmK;
  const CUtensorMap* tmV;
  __nv_bfloat16* o;
  float* lse;
  int T, BH, d, causal;
  int G;          // query heads per key/value head (grouped key/value heads; 1 without)
  float scale;
  uint32_t* err;  // device error word
  int num_sms;    // streaming multiprocessors of the device (persistent grids)
};

// Work items of the persistent attention kernels are sorted longest first and dealt to the
// CTAs in a snake order (round r left to right when r is even, right to left when odd), so
// that every CTA gets about the same total work. Items of every slice (b, h) run side by
// side, so the L2 holds the tiles that all items of a slice read again (K, V in the
// forward and the dQ kernel, Q and dO in dK/dV) for all slices at once. When those exceed
// the budget below (d >= 80 only), the kernels deal their items in two groups of half the
// slices each instead, one group after the other, and each group's tiles stay in L2 while
// it runs. Returns the slices per group: half the slices when all of them re-read more
// than the budget, else all (one group). Two groups dealt as HeadGroupSched does balance
// the CTAs' work as well as one; with four or more, the per-group rounds leave the CTAs up
// to a few per cent apart.
inline int slices_per_group(int n_slices, long long bytes_per_slice) {
  const long long budget = 40ll << 20;
  return (n_slices % 2 == 0 && (long long)n_slices * bytes_per_slice > budget) ? n_slices / 2 : n_slices;
}

#ifdef __CUDACC__
// One group: returns the r-th item of this CTA in the snake order, or -1 past its last.
struct SnakeSched {
  int n_items;
  __device__ __forceinline__ int item(int r) const {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int u = r * G + ((r & 1) ? (G - 1 - c) : c);
    return u < n_items ? u : -1;
  }
};

// Two groups of n_group items each (items [0, n_group) of the first group's slices, then
// the second's): each group is dealt in the snake order, the second with the CTAs in
// reverse order, so that the CTAs left short by the first group's last round are the ones
// that the second group serves first. Returns the r-th item of this CTA, or -1.
struct HeadGroupSched {
  int n_items;  // 2 n_group
  int n_group;
  __device__ __forceinline__ int item(int r) const {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int full = n_group / G, rem = n_group % G;
    const int n0 = full + (((full & 1) ? G - 1 - c : c) < rem ? 1 : 0);
    if (r < n0) return r * G + ((r & 1) ? G - 1 - c : c);
    r -= n0;
    const int c1 = G - 1 - c;
    const int n1 = full + (((full & 1) ? G - 1 - c1 : c1) < rem ? 1 : 0);
    return r < n1 ? n_group + r * G + ((r & 1) ? G - 1 - c1 : c1) : -1;
  }
};

// The scheduler of a kernel compiled with or without the grouped item order: the grouped
// form is a separate instantiation, so that one-group launches run the plain snake's code.
template <bool GROUPED>
__device__ __forceinline__ auto make_sched(int n_items, int n_group) {
  if constexpr (GROUPED)
    return HeadGroupSched{n_items, n_group};
  else
    return SnakeSched{n_items};
}
#endif

// Workspace of the backward: two fp32 arrays of [B*H, T_pad], T_pad = T rounded
// up to 128. ws_nlse2 = -LSE * log2(e) (-inf on padding rows), ws_D = rowsum(dO*O)
// (0 on padding rows). The fused dQ (d <= 64) adds dq_acc, one fp32 128 x d tile per
// (b*h, query tile), and dq_cnt, one int32 ordering counter per such tile.
struct BwdArgs {
  const CUtensorMap* tmQ;
  const CUtensorMap* tmK;
  const CUtensorMap* tmV;
  const CUtensorMap* tmdO;
  const CUtensorMap* tmO;  // O as a tensor map (the d <= 64 dQ kernel stages it), else null
  const CUtensorMap* tmdK;  // dK, dV as tensor maps (the d <= 64 dK/dV kernel stores through
  const CUtensorMap* tmdV;  // them), else null
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* ws_nlse2;
  float* ws_D;
  float* dq_acc;  // fused dQ only, else null
  int* dq_cnt;    // fused dQ only, else null
  int T, T_pad, BH, d, causal;  // BH = B * H query slices
  int G;                         // query heads per key/value head (1 without grouping)
  int S;                         // dK/dV splits of each key/value head's query heads (1: none)
  float* part;                   // S > 1: fp32 partial dK then dV, [S][B*H/G][T_pad][d] each
  float scale;
  uint32_t* err;  // device error word
  int num_sms;    // streaming multiprocessors of the device (persistent grids)
};

inline int pad_rows(int T) { return (T + 127) / 128 * 128; }

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream);  // + the partial-sum reduction when S > 1
// dQ; at d <= 64 it also writes D and -LSE*log2(e) into the workspace (needs tmO, lse),
// so it runs first and replaces the preprocess launch
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dkdv_dq(const BwdArgs& a, cudaStream_t stream);  // fused dK, dV, dQ (d <= 64)
cudaError_t launch_bwd_dq_finish(const BwdArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Training GEMMs around the attention (QKV and output projections)
// ---------------------------------------------------------------------------
// Orientation of C = op(A) op(B): NT C = A B^T (A [M, K], B [N, K]); NN C = A B (A [M, K],
// B [K, N]); TN C = A^T B (A [K, M], B [K, N]).
enum GemmLayout : int { kGemmNT = 0, kGemmNN = 1, kGemmTN = 2 };

// A token x feature operand stored as one to three 4-D tensors [Bn, Z, T, W] (dims W, T,
// Z, Bn for TMA): feature f of token (b, t) is element (b, f' / W, t, f' % W) of map
// m(f), f' = f - first feature of that map. A plain [Bn, T, F] activation is one map with
// W = F, Z = 1; the heads of Q / K / V ([Bn, H, T, d]) are W = d, Z = H, up to three
// maps (Q, K, V) for the concatenated QKV features.
struct TokView {
  int W;       // features per row of a map
  int f1, f2;  // first feature of map 1 and of map 2 (INT_MAX where absent)
};

struct GemmParams {
  CUtensorMap a[3];  // A: token view (NT / NN: K-major boxes of 64 features x 128 tokens;
                     // TN: MN-major boxes of 64 features x 64 tokens)
  CUtensorMap b[3];  // B: NT a 2-D [N, K] map (64 x bn/2 boxes); NN a 2-D [K, N] map (64 x 64);
                     // TN a token view (64 features x 64 tokens)
  CUtensorMap c[3];  // C: NT / NN a token view (bf16 stores of 64 features x 32 tokens);
                     // TN a 3-D fp32 [S, M, N] map (stores of 32 x 32)
  TokView va, vb, vc;
  int M, N, K;        // logical sizes of the product
  int T;              // tokens per sequence (the token dimension of the views)
  int nT;             // NT / NN: 128-token row tiles per sequence; TN: 64-token K-steps
  int m_tiles, n_tiles, k_iters, splits, k_per_split;
  int bn;             // output tile width: 256 or 192 (NT: B boxes of bn / 2 rows)
  int rope_features;  // NT epilogue: features below this are rotated (RoPE), 0 for none
  int rope_half;      // d / 2: entries of one position's row of the rotation table
  const float* rope_tab;  // [T][d/2][2] fp32 (cos, sin), or null
  uint32_t* err;          // device error word
};

// C = op(A) op(B); with p.splits > 1 (TN only) C is the [splits, M, N] partial-sum stack.
cudaError_t launch_gemm(int layout, const GemmParams& p, int num_sms, cudaStream_t stream);
// out[m, n] = sum over s = 0, 1, ... of part[s, m, n] (fp32, in split order)
cudaError_t launch_splitk_reduce(const float* part, float* out, long long mn, int splits, int num_sms,
                                 cudaStream_t stream);
// tab[t][k] = (cos, sin)(t * 10000^(-2k/d)), computed in fp64 and rounded to fp32
cudaError_t launch_rope_table(float* tab, int T, int d, cudaStream_t stream);
// dst_i = rope(src_i) (inverse: the rotation by -t theta_k) for [B, H_i, T, d] bf16 tensors,
// i = 0, 1 (H1 = 0: one tensor)
cudaError_t launch_rope_apply(const __nv_bfloat16* src0, __nv_bfloat16* dst0, int H0, const __nv_bfloat16* src1,
                              __nv_bfloat16* dst1, int H1, const float* tab, int B, int T, int d, int inverse,
                              int num_sms, cudaStream_t stream);

// Launches a kernel with programmatic stream serialization: its CTAs may be scheduled
// while the previous kernel in the stream drains; every kernel of the library waits for
// the previous kernels (griddep_begin) before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Launches a kernel cooperatively: the runtime starts it only when every CTA of its grid
// can be resident at once (the launch fails if the grid is larger than that), which a
// kernel whose CTAs wait on one another needs to make progress. No programmatic
// dependency: it starts after the previous kernel in the stream has completed.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                        Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Sets the max dynamic shared memory of a kernel once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, uint32_t* done_mask);

}  // namespace attn

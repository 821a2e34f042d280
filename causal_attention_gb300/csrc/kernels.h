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

// Sets the max dynamic shared memory of a kernel once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, uint32_t* done_mask);

}  // namespace attn

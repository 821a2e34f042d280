/*
 * attn.h - C ABI of the GB300 (sm_103a) fused causal attention library.
 *
 * The library computes multi-head attention with an optional causal mask, forward
 * and backward, for bf16 inputs with fp32 accumulation, on one GPU. Definitions
 * (Forge RESEARCH.md, section 6 "Fused attention design (flash-style)", and the
 * Forge paper, sections "Attention kernel design" and "Ecosystem survey"):
 *
 *   forward   S = Q K^T * scale;  key j is visible to query i iff j <= i (causal);
 *             P = softmax(S) over visible keys;  O = P V;
 *             LSE_i = log sum_j exp(S_ij)   (natural log, saved for the backward)
 *   backward  D = rowsum(dO * O);  P = exp(S - LSE);  dV = P^T dO;  dP = dO V^T;
 *             dS = P * (dP - D);  dQ = dS K * scale;  dK = dS^T Q * scale
 *
 * Layout and types. Every matrix argument is a contiguous row-major device
 * tensor [B, H, T, d] of bf16 (16-bit brain floats): element (b, h, t, c) is at
 * offset ((b*H + h)*T + t)*d + c. LSE is fp32 [B, H, T]. Pointers must be device
 * (or managed) memory visible to the current CUDA device and 16-byte aligned.
 * Head dimensions: d = 32, 64, 80 or 128 (Forge RESEARCH.md section 6, the layout
 * paragraph, lists 64, 80 and 128 as the head dimensions a fused kernel serves; 32 is
 * the small case). Any T >= 1.
 *
 * Ownership. The caller allocates and owns every buffer, including the backward's
 * workspace. The library allocates no device memory and keeps no per-call state
 * beyond a cached function pointer of the CUDA driver.
 *
 * Execution. Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and does not synchronise the host. Outputs are fully
 * overwritten. Results are bitwise deterministic run to run (no atomics).
 *
 * Errors. Arguments are checked before anything is launched; an invalid call
 * returns a status and launches nothing. Kernel waits are bounded: if one expires
 * the kernel records it in a device error word and returns early (its outputs are
 * then undefined); attn_check_device_error() reports and clears that word.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 3

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,     /* null pointer, B/H/T < 1, bad scale or causal flag, sizes too large */
  ATTN_ERR_UNSUPPORTED = 2,     /* head dimension d not in {32, 64, 80, 128} (projections: {64, 128}) */
  ATTN_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = 4,       /* workspace missing or smaller than attn_bwd_workspace_size() */
  ATTN_ERR_LAUNCH = 5,          /* the CUDA runtime rejected a launch (see attn_last_cuda_error) */
  ATTN_ERR_DEVICE_TIMEOUT = 6,  /* a kernel's bounded wait expired (attn_check_device_error) */
  ATTN_ERR_CUDA = 7,            /* another CUDA runtime or driver call failed */
  ATTN_ERR_DEVICE_BOUNDS = 8    /* bounds-checked build only: a kernel found an index out of its
                                   range and skipped the access (attn_check_device_error) */
} attn_status;

/* ABI version of the loaded library (ATTN_ABI_VERSION at build time). */
int attn_abi_version(void);

/*
 * Forward. Cited definition: Forge RESEARCH.md section 6, the online-softmax
 * algorithm and "L = m + log(l) (one f32/row, saved for backward)".
 *   q, k, v : bf16 [B, H, T, d] inputs
 *   o       : bf16 [B, H, T, d] output, O = softmax(Q K^T * scale) V
 *   lse     : fp32 [B, H, T] output, natural-log logsumexp of the scaled scores
 *   scale   : finite, > 0 (typically 1/sqrt(d));  causal: 1 masks keys j > i, 0 none
 * One kernel launch.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int T, int d, float scale, int causal, void* stream);

/*
 * Forward with grouped key/value heads (GQA; MQA when H_kv = 1). Cited mapping: Forge
 * RESEARCH.md section 6, its GQA index mapping: query head h reads
 * key/value head h / (H / H_kv), with no repeated copies of K and V.
 *   q, o : bf16 [B, H, T, d];  k, v : bf16 [B, H_kv, T, d];  lse : fp32 [B, H, T]
 *   H_kv : 1 <= H_kv <= H, dividing H (ATTN_ERR_INVALID_ARG otherwise)
 * attn_fwd(...) is attn_fwd_gqa(..., H_kv = H, ...). One kernel launch.
 */
attn_status attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int H_kv, int T, int d, float scale, int causal, void* stream);

/* Bytes of device workspace attn_bwd (and its stages) need: two fp32 arrays of
 * B*H*T_pad entries, T_pad = T rounded up to a multiple of 128. 0 if the sizes
 * are invalid. */
size_t attn_bwd_workspace_size(int B, int H, int T, int d);

/* Bytes of device workspace the fused-dQ stages (attn_bwd_dkdv_dq, attn_bwd_dq_finish)
 * need: the attn_bwd workspace, then B*H*T_pad*d fp32 dQ partial sums, then one int32
 * counter per 128-row query tile (4*B*H*T_pad/128 bytes, rounded up to 256). 0 if the
 * sizes are invalid or d > 64. */
size_t attn_bwd_fused_workspace_size(int B, int H, int T, int d);

/*
 * Backward. Cited definition: Forge RESEARCH.md section 6, the bullet on the D term
 * and "Backward (training)"; the three-stage atomic-free structure of the Forge
 * paper's "Ecosystem survey". Equivalent to, on the same stream: at d <= 64
 * attn_bwd_dq (which also forms D) then attn_bwd_dkdv; at d >= 80 attn_bwd_preprocess,
 * attn_bwd_dkdv, attn_bwd_dq.
 *   q, k, v, o, dO : bf16 [B, H, T, d] (o and lse as written by attn_fwd)
 *   lse            : fp32 [B, H, T]
 *   dq, dk, dv     : bf16 [B, H, T, d] outputs
 *   workspace      : >= attn_bwd_workspace_size(B, H, T, d) bytes of device memory,
 *                    16-byte aligned; its contents on entry do not matter
 * Two kernel launches at d <= 64, three at d >= 80.
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int T, int d, float scale, int causal,
                     void* stream);

/*
 * Backward with grouped key/value heads (the mapping of attn_fwd_gqa). dK and dV of a
 * key/value head are the sums over its H / H_kv query heads, accumulated inside the
 * dK/dV kernel (one CTA per key tile of each key/value head loops over the query tiles
 * of all of them), so the result is deterministic.
 *   q, o, dO, dq : bf16 [B, H, T, d];  k, v, dk, dv : bf16 [B, H_kv, T, d];  lse : [B, H, T]
 *   workspace    : >= attn_bwd_workspace_size(B, H, T, d) bytes (query heads)
 * attn_bwd(...) is attn_bwd_gqa(..., H_kv = H, ...). The stage entry points below are
 * for H_kv = H.
 */
/* Bytes of device workspace for attn_bwd_gqa's fastest path: the attn_bwd workspace, plus,
 * when the key/value heads are too few to fill the device with dK/dV work items (B * H_kv
 * * ceil(T / 128) < 304), fp32 partial dK and dV for S splits of each key/value head's
 * query heads (2 * S * B * H_kv * T_pad * d * 4 bytes, S = min(H / H_kv, ceil(304 / items))),
 * which a last launch adds in split order (deterministic). With only the attn_bwd
 * workspace, attn_bwd_gqa runs unsplit. 0 if the sizes are invalid. */
size_t attn_bwd_gqa_workspace_size(int B, int H, int H_kv, int T, int d);

attn_status attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, void* workspace,
                         size_t workspace_bytes, int B, int H, int H_kv, int T, int d, float scale,
                         int causal, void* stream);

/* Backward stage 1: D = rowsum(dO * O) and LSE * log2(e) into the workspace
 * (Forge RESEARCH.md section 6, the bullet on the D term). Memory-bound. With d <= 64 and a
 * workspace of attn_bwd_fused_workspace_size bytes it also zeroes the fused dQ's
 * counters, so it must run before every attn_bwd_dkdv_dq. */
attn_status attn_bwd_preprocess(const void* o, const void* dO, const float* lse, void* workspace,
                                size_t workspace_bytes, int B, int H, int T, int d, void* stream);

/* Backward stage 2: dK and dV, one CTA per 128-key tile looping over query tiles
 * (Forge paper, "Attention kernel design": transposes by operand-role swap).
 * Reads the D / LSE workspace written by stage 1 or, at d <= 64, by attn_bwd_dq. */
attn_status attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                          void* dv, const void* workspace, size_t workspace_bytes, int B, int H,
                          int T, int d, float scale, int causal, void* stream);

/* Backward stage 3: dQ, one CTA per 128-query tile looping over key tiles
 * (deterministic; Forge RESEARCH.md section 6, the production structure it surveys: a
 * separate dQ launch over query tiles, heads and batches).
 * At d >= 80 it reads the workspace written by stage 1. At d <= 64 it does stage 1's
 * work for its own query tile (D = rowsum(dO * O) from a staged O tile, -LSE * log2(e)
 * from lse) and writes both into the workspace, so it needs no stage 1 before it and
 * attn_bwd_dkdv may follow it; o and lse are read only at d <= 64 but are always
 * checked. */
attn_status attn_bwd_dq(const void* q, const void* k, const void* v, const void* o, const void* dO,
                        const float* lse, void* dq, void* workspace, size_t workspace_bytes, int B, int H,
                        int T, int d, float scale, int causal, void* stream);

/*
 * Backward stage 2 with dQ fused (d <= 64 only; an alternative to attn_bwd_dkdv followed
 * by attn_bwd_dq, which attn_bwd uses because it is faster on GB300): dK and dV as
 * attn_bwd_dkdv, and the products dQ_ij = dS_ij K_j formed in the same kernel from the
 * same dS tile, so the two GEMMs the separate dQ kernel recomputes (S and dP) are never
 * run. Each dQ_ij is added
 * to an fp32 tile of the workspace in the fixed order j = 0, 1, 2, ... (a per-tile
 * counter, bounded waits), never with atomics, so the result is the same on every run
 * (Iron "Kernel Engineering Guide", section 3.4 "Determinism": partial sums combined in a
 * fixed order; Forge RESEARCH.md section 8, pitfall 20: no atomic gradient
 * accumulation in deterministic mode). The ordering needs the launch's CTAs (one per SM,
 * at most the SM count) to be resident together, so the kernel is launched cooperatively:
 * the runtime starts it only once the whole grid fits on the device (kernels already
 * running on other streams finish first), and every counter wait is on a running CTA.
 * A wait that still ran out would be reported by attn_check_device_error as
 * ATTN_ERR_DEVICE_TIMEOUT; nothing hangs.
 *   workspace : attn_bwd_fused_workspace_size(B, H, T, d) bytes (ATTN_ERR_WORKSPACE if
 *               smaller), written by attn_bwd_preprocess just before
 *   dk, dv    : bf16 [B, H, T, d] outputs; dQ is left in the workspace for
 *               attn_bwd_dq_finish
 * d > 64 returns ATTN_ERR_UNSUPPORTED. One kernel launch.
 */
attn_status attn_bwd_dkdv_dq(const void* q, const void* k, const void* v, const void* dO, void* dk,
                             void* dv, void* workspace, size_t workspace_bytes, int B, int H, int T,
                             int d, float scale, int causal, void* stream);

/* Backward, last step of the fused path: dq (bf16 [B, H, T, d]) = scale times the fp32
 * dQ sums attn_bwd_dkdv_dq left in the workspace. d <= 64; memory-bound; one launch. */
attn_status attn_bwd_dq_finish(void* dq, const void* workspace, size_t workspace_bytes, int B, int H,
                               int T, int d, float scale, void* stream);

/*
 * Backward without a workspace argument. The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory for the workspace:
 * code running inside a host framework that owns every device allocation and gives a
 * plug-in no way to ask for scratch, and latency-critical callers that must not call
 * cudaMalloc/cudaFree on the step path because those calls can synchronise the whole
 * device. It computes exactly what attn_bwd computes (same kernels, same results), but
 * keeps the D / LSE scratch in a fixed 8 MiB array that is part of the library's device
 * image (every GPU that loads the library holds it until the process exits), and it
 * calls no allocating routine.
 *   Limit: B*H*T_pad <= 1,048,576 (T_pad = T rounded up to 128); larger shapes return
 *   ATTN_ERR_WORKSPACE without launching anything (use attn_bwd with a workspace).
 *   Set-up: the first call on each device looks up the array's device address (with
 *   that device current) and caches it. Under lazy module loading (the CUDA runtime's
 *   default) that lookup may also be what loads the library's device code, and with it
 *   the array, onto the device: the first call on a device can allocate device memory and
 *   synchronise. Treat it as a warm-up: make it before any stream capture and outside
 *   the region that must not allocate; later calls allocate nothing.
 *   Sharing: every call on a device uses the same array, and the array keeps the last
 *   call's contents. Nothing in it has to start at zero (each call overwrites every
 *   entry it reads), but calls whose executions overlap on the GPU (different streams,
 *   no ordering between them) race on the array and must be serialised by the caller.
 * Arguments are those of attn_bwd without workspace and workspace_bytes.
 */
attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                             int H, int T, int d, float scale, int causal, void* stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device. Returns ATTN_ERR_DEVICE_BOUNDS if (in the bounds-checked build,
 * libattn_debug.so) a kernel found an index outside its range since the last check,
 * else ATTN_ERR_DEVICE_TIMEOUT if a kernel's bounded wait expired, ATTN_ERR_CUDA if
 * the synchronisation failed. */
attn_status attn_check_device_error(void* stream);

/* Static description of a status code. */
const char* attn_status_string(attn_status status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* attn_last_cuda_error(void);

/* Self-test of the failure path: launches one warp that waits, through the kernels' own
 * bounded wait, on a barrier that nothing arrives on. After the wait's time limit (2 s)
 * it records the expiry in the device error word and returns, so that the next
 * attn_check_device_error on the stream reports ATTN_ERR_DEVICE_TIMEOUT (and clears the
 * word) and the context stays usable. Nothing faults, traps or hangs. One launch. */
attn_status attn_selftest_wait_timeout(void* stream);

/* ------------------------------------------------------------------------------------
 * Projections around the attention: the training GEMMs of the attention block.
 *
 * Cited definitions: the GEMM orientations a training step needs, nt (forward
 * Y = X W^T), nn (dX = dY W) and tn (dW = dY^T X), with split-K for the dW shape into
 * fp32 partials and a separate reduction, no atomics (Forge RESEARCH.md section 5 "GEMM
 * design"; the Forge paper's GEMM table, section "Results"); rotary position embedding
 * on q and k, interleaved pairs (2k, 2k+1) of a head row at position t rotated by
 * t * 10000^(-2k/d), backward = the rotation by minus that angle (Forge RESEARCH.md
 * section 7, model formulas).
 *
 * The attention block: x [B, T, C] bf16 -> q [B, H, T, d], k, v [B, H_kv, T, d] =
 * split(x W_qkv^T) (W_qkv bf16 [(H + 2 H_kv) d, C]: the rows of Q's heads, then K's,
 * then V's) -> attention -> o [B, H, T, d] -> y [B, T, C] = merge(o) W_o^T (W_o bf16
 * [C, H d]). split / merge move between token rows and [B, heads, T, d] through the
 * TMA tensor maps: no copy pass. Weight gradients are fp32; every other tensor is bf16
 * with fp32 accumulation. Projections need d in {64, 128} (else ATTN_ERR_UNSUPPORTED),
 * C a multiple of 8 (else ATTN_ERR_INVALID_ARG). Asynchronous on `stream`; pointers
 * 16-byte aligned; the caller owns every buffer. Results are bitwise deterministic.
 * ---------------------------------------------------------------------------------- */

/* Layouts of attn_gemm. */
#define ATTN_GEMM_NT 0 /* C [M, N] bf16 = A [M, K] . B [N, K]^T */
#define ATTN_GEMM_NN 1 /* C [M, N] bf16 = A [M, K] . B [K, N] */
#define ATTN_GEMM_TN 2 /* C [M, N] fp32 = A [K, M]^T . B [K, N] (split over K when M x N is small) */

/* Bytes of workspace attn_gemm needs (the tn split-K partial sums; 0 for nt / nn, or
 * when the tn product is not split, or for invalid sizes). */
size_t attn_gemm_workspace_size(int M, int N, int K, int layout);

/* A plain GEMM: row-major bf16 operands, M, N, K multiples of 8. C is bf16 for nt / nn
 * and fp32 for tn. One launch (two when a tn product is split over K). */
attn_status attn_gemm(const void* a, const void* b, void* c, int M, int N, int K, int layout, void* workspace,
                      size_t workspace_bytes, void* stream);

/* The rotation table of RoPE: tab fp32 [T][d/2][2] = (cos, sin) of t * 10000^(-2k/d),
 * computed in fp64 and rounded. d a multiple of 8. One launch; make it once per (T, d). */
attn_status attn_rope_table(float* tab, int T, int d, void* stream);

/* y = RoPE(x) (inverse = 1: the rotation by the negative angle, i.e. the backward) for
 * bf16 [B, H, T, d] tensors; y may be x. One launch. */
attn_status attn_rope(const void* x, void* y, const float* rope_tab, int B, int H, int T, int d, int inverse,
                      void* stream);

/* Forward QKV projection: q, k, v = split(x W_qkv^T), and with rope_tab (non-null) q and k
 * rotated in the GEMM's epilogue before rounding to bf16. One launch. */
attn_status attn_qkv_proj(const void* x, const void* w_qkv, void* q, void* k, void* v, const float* rope_tab, int B,
                          int T, int C, int H, int H_kv, int d, void* stream);

/* Forward output projection: y = merge(o) W_o^T. One launch. */
attn_status attn_out_proj(const void* o, const void* w_o, void* y, int B, int T, int H, int d, int C, void* stream);

/* Bytes of workspace attn_out_proj_bwd and attn_qkv_proj_bwd need (either may use all of
 * it; calls on one stream may share it). 0 for invalid sizes. */
size_t attn_proj_bwd_workspace_size(int B, int T, int C, int H, int H_kv, int d);

/* Backward of the output projection given dy [B, T, C]: d_o [B, H, T, d] = split(dy W_o)
 * (nn) and dw_o fp32 [C, H d] = dy^T merge(o) (tn). Two or three launches. */
attn_status attn_out_proj_bwd(const void* dy, const void* o, const void* w_o, void* d_o, float* dw_o, void* workspace,
                              size_t workspace_bytes, int B, int T, int H, int d, int C, void* stream);

/* Backward of the QKV projection given dq [B, H, T, d], dk, dv [B, H_kv, T, d] (the
 * gradients of the tensors attn_qkv_proj wrote): with rope_tab, dq and dk are rotated
 * back first (into the workspace); then dx [B, T, C] = merge(dq, dk, dv) W_qkv (nn) and
 * dw_qkv fp32 [(H + 2 H_kv) d, C] = merge(dq, dk, dv)^T x (tn). Up to four launches. */
attn_status attn_qkv_proj_bwd(const void* dq, const void* dk, const void* dv, const void* x, const void* w_qkv,
                              const float* rope_tab, void* dx, float* dw_qkv, void* workspace, size_t workspace_bytes,
                              int B, int T, int C, int H, int H_kv, int d, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */

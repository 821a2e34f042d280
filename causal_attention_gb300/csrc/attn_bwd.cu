// Causal attention backward for sm_103a, three kernels, no atomics:
//
//  1. preprocess: D = rowsum(dO * O) in fp32 (Forge RESEARCH.md, section 6, "The D
//     term is free": D_i = sum_j P_ij dP_ij = dO_i . O_i) and -LSE * log2(e), both
//     written to a [B*H, T_pad] workspace (padding rows: D = 0, -LSE*log2e = -inf,
//     so that padded queries contribute P = 0). With the sign folded in, P is one
//     fused multiply-add and an exp2 away from S.
//  2. dK/dV: one CTA per 128-key tile j, looping over query tiles i (i >= j when
//     causal): S^T = K_j Q_i^T, P^T = exp2(S^T * scale * log2e - LSE_i * log2e),
//     dV_j += P^T dO_i, dP^T = V_j dO_i^T, dS^T = P^T * (dP^T - D_i),
//     dK_j += dS^T Q_i; dK *= scale at the end. The transposes come from swapping
//     operand roles, not from moving data (Forge paper, section "Attention kernel
//     design").
//  3. dQ: one CTA per 128-query tile i, looping over key tiles j (j <= i):
//     S = Q_i K_j^T, P = exp2(S * scale * log2e - LSE * log2e), dP = dO_i V_j^T,
//     dS = P * (dP - D), dQ_i += dS K_j; dQ *= scale at the end. Each dQ tile is
//     owned by one CTA, so the result is deterministic.
// The dQ-parallel / dKV-parallel split with a D preprocess is the three-stage,
// atomic-free structure of the Forge paper's section "Ecosystem survey".
//
// Roles in the two tensor-core kernels (608 threads):
//   warps 0-15 elementwise, four warpgroups: thread = row of the CTA's own tile (TMEM
//              lane), warpgroup h = columns [32h, 32h+32) of the 128-column tiles
//              (four warps per scheduler to hide the exp / TMEM / barrier latencies)
//   warp  16   TMA producer
//   warp  17   TMEM allocator and MMA issuer (S and dP)
//   warp  18   second MMA issuer (dV and dK, or dQ) where the elementwise results have
//              their own TMEM columns. A tcgen05.mma issue blocks until the tensor core
//              can take it, and any wait of the issuing thread drains the queue, so two
//              issuers keep the tensor core fed while either one waits.
// Tensor memory: S or S^T [0,128), dP or dP^T [128,256), accumulators from 256.
// P^T and dS^T (bf16) go to their own TMEM columns where they fit, else over the S^T
// and dP^T regions (each warpgroup into the first 16 columns of its own 32-column
// quarter), and are fed back to the tensor core from TMEM as the A operand.
#include "kernels.h"
#include "tile.cuh"

namespace attn {

namespace {

// warps 0-15 elementwise, 16 producer, 17 and 18 MMA issuers, 19 (fused dQ) reducer or
// (dQ kernel at d >= 80) third MMA issuer
constexpr int kBwdThreads = 608;
constexpr int kWarpProd = 16, kWarpMmaA = 17, kWarpMmaB = 18, kWarpRed = 19, kWarpMmaC = 19;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
// With the fused dQ it also zeroes the per-tile ordering counters (dq_cnt, n_cnt entries).
//
// HBM-bound. CTA c takes rows t = 64x .. 64x + 63 of slice bh, c = bh * (T_pad / 64) + x
// (padding rows t >= T included), TPR threads per row reading 16-byte granules. Every load of a thread
// (its granules of O and dO in PRE_U rows, and LSE) is issued before any of them is used,
// so one round trip to memory serves the whole CTA.
constexpr int kPreRows = 64, kPreThreads = 256;

template <int D>
__global__ void __launch_bounds__(kPreThreads) attn_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
    const float* __restrict__ lse, float* __restrict__ ws_nlse2, float* __restrict__ ws_D, int* __restrict__ dq_cnt,
    int n_cnt, int T, int T_pad) {
  constexpr int NG = D / 8;                             // 16-byte granules per row
  constexpr int TPR = (NG & (NG - 1)) == 0 ? NG : 8;    // threads per row (a power of two)
  constexpr int RPP = kPreThreads / TPR;                // rows per pass
  constexpr int U = kPreRows / RPP;                     // rows per thread
  constexpr int GPT = (NG + TPR - 1) / TPR;             // granules per thread and row
  griddep_begin();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_cnt;
       i += (long long)gridDim.x * blockDim.x)
    dq_cnt[i] = 0;
  const int n_ch = T_pad / kPreRows;
  const int bh = (int)(blockIdx.x / n_ch), sub = threadIdx.x % TPR;
  const int t0 = (int)(blockIdx.x % n_ch) * kPreRows + threadIdx.x / TPR;
  const __nv_bfloat16* ob = o + (size_t)bh * T * D;
  const __nv_bfloat16* db = dO + (size_t)bh * T * D;
  uint4 a[U][GPT], b[U][GPT];
  float L[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int t = t0 + u * RPP;
    L[u] = (sub == 0 && t < T) ? lse[(size_t)bh * T + t] : 0.f;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      const int gi = sub + k * TPR;
      a[u][k] = make_uint4(0u, 0u, 0u, 0u);
      b[u][k] = a[u][k];
      if (t < T && gi < NG) {
        a[u][k] = ldg_stream(ob + (size_t)t * D + gi * 8);
        b[u][k] = ldg_stream(db + (size_t)t * D + gi * 8);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int k = 0; k < GPT; ++k) {
      fma_bf16x2_f32(a[u][k].x, b[u][k].x, a0, a1);
      fma_bf16x2_f32(a[u][k].y, b[u][k].y, a0, a1);
      fma_bf16x2_f32(a[u][k].z, b[u][k].z, a0, a1);
      fma_bf16x2_f32(a[u][k].w, b[u][k].w, a0, a1);
    }
    float acc = a0 + a1;
#pragma unroll
    for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    const int t = t0 + u * RPP;
    if (sub == 0 && t < T_pad) {
      ws_D[(size_t)bh * T_pad + t] = acc;  // 0 on padding rows
      ws_nlse2[(size_t)bh * T_pad + t] = t < T ? -L[u] * kLog2e : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------
// shared-memory plan of the two tensor-core kernels
// ---------------------------------------------------------------------------
// NFIX: tiles fixed for a whole work item (K_j, V_j for dK/dV; Q_i, dO_i and, when the
// dQ kernel computes D itself, O_i). NEPI: bf16 output tiles staged in shared memory for
// a TMA store in the epilogue (dV and dK).
// KRING, VRING (dQ kernel): separate rings of K and V tiles instead of the stages.
template <int D, bool FUSE = false, int NFIX = 2, int NEPI = 0, int KRING = 0, int VRING = 0>
struct BwdCfg {
  using TL = Tile<D>;
  static constexpr int STAGES = (D > 64) ? 2 : (D == 64 ? 3 : 4);
  // fixed tiles of a work item (K_j, V_j for dK/dV; Q_i, dO_i for dQ), in NSLOT slots:
  // with two (persistent kernels at d <= 64) the next item's tiles load during this one
  static constexpr int NSLOT = (D <= 64 && !FUSE) ? 2 : 1;
  static constexpr int OFF_FIX = 0;
  // per stage: two tiles (+ for dK/dV, 128 fp32 -LSE*log2e and 128 fp32 D)
  static constexpr int STAGE_BYTES = 2 * TL::BYTES + 1024;
  static constexpr int SLOT_BYTES = NFIX * TL::BYTES;
  static constexpr int OFF_STAGE = OFF_FIX + NSLOT * SLOT_BYTES;
  // fused dQ only: dS^T as a bf16 128x128 shared-memory tile (A operand of dK += dS^T Q_i
  // and, read transposed, of dQ_ij = dS K_j), then the fp32 staging tile of dQ_ij on its
  // way to the workspace
  static constexpr int DS_BYTES = FUSE ? kTileRows * kTileRows * 2 : 0;
  static constexpr int DQS_BYTES = FUSE ? kTileRows * D * 4 : 0;
  static constexpr int STAGE_AREA = KRING ? (KRING + VRING) * TL::BYTES : STAGES * STAGE_BYTES;
  static constexpr int OFF_DS = OFF_STAGE + STAGE_AREA;
  static constexpr int OFF_DQS = OFF_DS + DS_BYTES;
  static constexpr int OFF_EPI = OFF_DQS + DQS_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + NEPI * TL::BYTES;
  // barrier rings: st_full / st_empty (the stages, or the K ring) and v_full / v_empty
  static constexpr int RB = KRING > STAGES ? KRING : STAGES;
  static constexpr int NBAR = 1 + 2 * RB + 22 + 2 * VRING;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // at least 116 KB so that one CTA occupies an SM: each CTA allocates all 512
  // TMEM columns, and a second resident CTA would only wait for them
  static constexpr int SMEM_RAW = OFF_MISC + 16 + 1024;
  static constexpr int SMEM_BYTES = SMEM_RAW > 116 * 1024 ? SMEM_RAW : 116 * 1024;
  // The dK/dV kernel gives P^T and dS^T their own TMEM columns when they fit (d <= 64);
  // then two threads issue its MMAs.
  static constexpr bool SEP_DKDV = D <= 64;
  static constexpr uint32_t COL_P = 384, COL_DS = 448;
  // tensor-memory plan of the dK/dV kernel: S^T [0, 128), dP^T [128, 256), dV and dK from
  // 256, and (d <= 64) P^T, dS^T in 64 columns each after them
  static_assert(256 + 2 * TL::ACC_COLS <= (SEP_DKDV ? COL_P : 512u), "dV, dK columns");
  static_assert(COL_DS + 64 <= 512, "P^T, dS^T columns");
  // fused dQ: dQ_ij (fp32, d columns) takes the columns of dS^T, which lives in shared memory
  static constexpr uint32_t COL_DQ = 448;
  static constexpr int THREADS = FUSE ? kBwdThreads + 32 : kBwdThreads;
  static_assert(!FUSE || SEP_DKDV, "the fused dQ needs the separate P^T columns (d <= 64)");
};

// Barriers (one 8-byte mbarrier each). Per work item: fix_full / fix_empty (the item's
// fixed tiles), acc_full / acc_free (its accumulators). Per stage: st_full / st_empty.
// Per iteration (global count over the CTA's items): s_full, dp_full (MMA results),
// s_free, dp_free (read out by the elementwise warps), p_full, ds_full (their results
// written to TMEM), dv_done, dk_done (the MMAs reading those results finished).
struct BwdSmem {
  uint32_t base;
  uint8_t* gbase;
  uint32_t bar0;
  int st, vr;
  __device__ uint32_t fix_full(int b) const { return b ? bar0 + 8u * (20 + 2 * st) : bar0; }
  __device__ uint32_t st_full(int s) const { return bar0 + 8u * (1 + s); }
  __device__ uint32_t st_empty(int s) const { return bar0 + 8u * (1 + st + s); }
  __device__ uint32_t s_full() const { return bar0 + 8u * (1 + 2 * st); }
  __device__ uint32_t dp_full() const { return bar0 + 8u * (2 + 2 * st); }
  __device__ uint32_t p_full() const { return bar0 + 8u * (3 + 2 * st); }
  __device__ uint32_t ds_full() const { return bar0 + 8u * (4 + 2 * st); }
  __device__ uint32_t acc_full() const { return bar0 + 8u * (5 + 2 * st); }
  __device__ uint32_t drain() const { return bar0 + 8u * (6 + 2 * st); }
  __device__ uint32_t s_free() const { return bar0 + 8u * (7 + 2 * st); }
  __device__ uint32_t dp_free() const { return bar0 + 8u * (8 + 2 * st); }
  __device__ uint32_t dv_done() const { return bar0 + 8u * (9 + 2 * st); }
  __device__ uint32_t dk_done() const { return bar0 + 8u * (10 + 2 * st); }
  __device__ uint32_t drain2() const { return bar0 + 8u * (11 + 2 * st); }
  __device__ uint32_t fix_empty(int b) const { return bar0 + 8u * (b ? 21 + 2 * st : 12 + 2 * st); }
  __device__ uint32_t acc_free() const { return bar0 + 8u * (13 + 2 * st); }
  // fused dQ: the dQ_ij MMA finished (dS^T tile and TMEM columns read) / its TMEM columns
  // were read out / the staging tile is written / the staging tile was read by the copy
  __device__ uint32_t dq_done() const { return bar0 + 8u * (14 + 2 * st); }
  __device__ uint32_t dq_free() const { return bar0 + 8u * (15 + 2 * st); }
  __device__ uint32_t dqs_full() const { return bar0 + 8u * (16 + 2 * st); }
  __device__ uint32_t dqs_free() const { return bar0 + 8u * (17 + 2 * st); }
  __device__ uint32_t drain3() const { return bar0 + 8u * (18 + 2 * st); }
  // epilogue through shared memory: the TMA stores of the previous item read its tiles
  __device__ uint32_t epi_free() const { return bar0 + 8u * (19 + 2 * st); }
  // dQ kernel: the V ring (its K ring uses st_full / st_empty)
  __device__ uint32_t v_full(int s) const { return bar0 + 8u * (23 + 2 * st + s); }
  __device__ uint32_t v_empty(int s) const { return bar0 + 8u * (23 + 2 * st + vr + s); }
};

constexpr int kEwThreads = 512;  // four elementwise warpgroups

// fix_empty_count: arrivals that release an item's fixed tiles (the MMA commits, plus the
// elementwise threads where they read a fixed tile themselves). issuers: MMA-issuing
// threads whose commits each release a stage and complete an item's accumulators.
template <int D, bool FUSE = false, int NFIX = 2, int NEPI = 0, int KRING = 0, int VRING = 0>
__device__ __forceinline__ BwdSmem bwd_smem_setup(uint8_t* smem_raw, uint32_t*& tmem_slot,
                                                  volatile int*& abort, uint32_t fix_empty_count = 1,
                                                  uint32_t issuers = 1) {
  using C = BwdCfg<D, FUSE, NFIX, NEPI, KRING, VRING>;
  BwdSmem s;
  const uint32_t raw = smem_u32(smem_raw);
  s.base = (raw + 1023u) & ~1023u;
  s.gbase = smem_raw + (s.base - raw);
  s.bar0 = s.base + C::OFF_BAR;
  s.st = C::RB;
  s.vr = VRING;
  tmem_slot = reinterpret_cast<uint32_t*>(s.gbase + C::OFF_MISC);
  abort = reinterpret_cast<volatile int*>(s.gbase + C::OFF_MISC + 4);
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(s.fix_full(b), 1);
      mbar_init(s.fix_empty(b), fix_empty_count);
    }
    for (int i = 0; i < C::RB; ++i) {
      mbar_init(s.st_full(i), 1);
      mbar_init(s.st_empty(i), issuers);
    }
    for (int i = 0; i < VRING; ++i) {
      mbar_init(s.v_full(i), 1);
      mbar_init(s.v_empty(i), 1);
    }
    mbar_init(s.s_full(), 1);
    mbar_init(s.dp_full(), 1);
    mbar_init(s.p_full(), kEwThreads);
    mbar_init(s.ds_full(), kEwThreads);
    mbar_init(s.s_free(), kEwThreads);
    mbar_init(s.dp_free(), kEwThreads);
    mbar_init(s.dv_done(), 1);
    mbar_init(s.dk_done(), 1);
    mbar_init(s.acc_full(), issuers);
    mbar_init(s.acc_free(), kEwThreads);
    mbar_init(s.drain(), 1);
    mbar_init(s.drain2(), 1);
    mbar_init(s.epi_free(), 1);
    if (FUSE) {
      mbar_init(s.dq_done(), 1);
      mbar_init(s.dq_free(), kEwThreads);
      mbar_init(s.dqs_full(), kEwThreads);
      mbar_init(s.dqs_free(), 1);
    }
    mbar_init(s.drain3(), 1);
    *abort = 0;
    fence_barrier_init();
  }
  if ((threadIdx.x >> 5) == kWarpMmaA) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_begin();  // the inputs may come from the previous kernel in the stream
  return s;
}

// Converts 16 fp32 accumulator columns to bf16 (times `mul`) and stores them.
__device__ __forceinline__ void store_row16(__nv_bfloat16* dst, const uint32_t (&u)[16], float mul) {
  uint4 pk[2];
  uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    pw[i] = pack_bf16(__uint_as_float(u[2 * i]) * mul, __uint_as_float(u[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = pk[0];
  d4[1] = pk[1];
}

// Epilogue of one accumulator row (d fp32 TMEM columns from `tacc`): the warpgroup hc
// of four converts its quarter, columns [hc*d/4, (hc+1)*d/4), to bf16 (times `mul`) and
// stores it to `dst_row` (a [d] bf16 row) when `valid`.
template <int D>
__device__ __forceinline__ void store_acc_quarter(uint32_t tacc, __nv_bfloat16* dst_row, int hc, float mul,
                                                  bool valid) {
  constexpr int QW = D / 4;  // 8, 16 or 32 columns
  if constexpr (D % 64 != 0 && D > 32) {
    // d = 80: five 16-column blocks; warpgroup hc takes block hc, warpgroup 0 also block 4
    for (int b = hc; b < D / 16; b += 4) {
      uint32_t u[16];
      tmem_ld16(tacc + (uint32_t)(16 * b), u);
      tmem_wait_ld();
      if (valid) store_row16(dst_row + 16 * b, u, mul);
    }
  } else if constexpr (QW == 8) {
    uint32_t u[8];
    tmem_ld8(tacc + (uint32_t)(hc * QW), u);
    tmem_wait_ld();
    if (valid) {
      uint4 pk;
      pk.x = pack_bf16(__uint_as_float(u[0]) * mul, __uint_as_float(u[1]) * mul);
      pk.y = pack_bf16(__uint_as_float(u[2]) * mul, __uint_as_float(u[3]) * mul);
      pk.z = pack_bf16(__uint_as_float(u[4]) * mul, __uint_as_float(u[5]) * mul);
      pk.w = pack_bf16(__uint_as_float(u[6]) * mul, __uint_as_float(u[7]) * mul);
      *reinterpret_cast<uint4*>(dst_row + hc * QW) = pk;
    }
  } else {
#pragma unroll
    for (int cb = 0; cb < QW / 16; ++cb) {
      const int col = hc * QW + 16 * cb;
      uint32_t u[16];
      tmem_ld16(tacc + (uint32_t)col, u);
      tmem_wait_ld();
      if (valid) store_row16(dst_row + col, u, mul);
    }
  }
}

// Epilogue of a split work item: the warpgroup hc of four stores its quarter of one
// accumulator row (d fp32 TMEM columns from `tacc`) as fp32 to `dst_row` (a [d] row).
template <int D>
__device__ __forceinline__ void store_acc_quarter_f32(uint32_t tacc, float* dst_row, int hc) {
  if constexpr (D % 64 != 0 && D > 32) {
    // d = 80: five 16-column blocks; warpgroup hc takes block hc, warpgroup 0 also block 4
    for (int b = hc; b < D / 16; b += 4) {
      uint32_t u[16];
      tmem_ld16(tacc + (uint32_t)(16 * b), u);
      tmem_wait_ld();
      uint4* d4 = reinterpret_cast<uint4*>(dst_row + 16 * b);
#pragma unroll
      for (int k = 0; k < 4; ++k) d4[k] = make_uint4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
    }
  } else {
    constexpr int QW = D / 4;  // 8, 16 or 32 columns
    uint32_t u[QW];
    if constexpr (QW == 32) tmem_ld32(tacc + (uint32_t)(hc * QW), u);
    else if constexpr (QW == 16) tmem_ld16(tacc + (uint32_t)(hc * QW), u);
    else tmem_ld8(tacc + (uint32_t)(hc * QW), u);
    tmem_wait_ld();
    uint4* d4 = reinterpret_cast<uint4*>(dst_row + hc * QW);
#pragma unroll
    for (int k = 0; k < QW / 4; ++k) d4[k] = make_uint4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
  }
}

// Epilogue through shared memory: the warpgroup hc of four converts its quarter of one
// accumulator row (d fp32 TMEM columns from `tacc`, times `mul`) to bf16 and writes it
// into row r of a Tile<D>-layout shared tile (the layout a TMA store of the tile reads).
template <int D>
__device__ __forceinline__ void stage_acc_quarter(uint32_t tacc, uint32_t tile, int r, int hc, float mul) {
  using TL = Tile<D>;
  constexpr int QW = D / 4;  // 8, 16 or 32 columns = 1, 2 or 4 granules of 16 bytes
  uint32_t u[QW];
  if constexpr (QW == 32) tmem_ld32(tacc + (uint32_t)(hc * QW), u);
  else if constexpr (QW == 16) tmem_ld16(tacc + (uint32_t)(hc * QW), u);
  else tmem_ld8(tacc + (uint32_t)(hc * QW), u);
  tmem_wait_ld();
  const int c = (hc * QW) / TL::CHUNK_ELEMS, g0 = ((hc * QW) % TL::CHUNK_ELEMS) / 8;
#pragma unroll
  for (int k = 0; k < QW / 8; ++k)
    sts128(tile + TL::granule_off(r, c, g0 + k),
           pack_bf16(__uint_as_float(u[8 * k + 0]) * mul, __uint_as_float(u[8 * k + 1]) * mul),
           pack_bf16(__uint_as_float(u[8 * k + 2]) * mul, __uint_as_float(u[8 * k + 3]) * mul),
           pack_bf16(__uint_as_float(u[8 * k + 4]) * mul, __uint_as_float(u[8 * k + 5]) * mul),
           pack_bf16(__uint_as_float(u[8 * k + 6]) * mul, __uint_as_float(u[8 * k + 7]) * mul));
}

// Number of items the schedule gives this CTA.
template <class SchedT>
__device__ __forceinline__ int sched_count(const SchedT& s) {
  int n = 0;
  while (s.item(n) >= 0) ++n;
  return n;
}

// Producer drain after an abort: every copy issued must land before the CTA exits.
__device__ __forceinline__ void drain_loads(const BwdSmem& sm, int fix_issued, int nslot, int st_issued, int st,
                                            const Abort& ab) {
  for (int x = max(0, fix_issued - nslot); x < fix_issued; ++x)
    mbar_wait_drain(sm.fix_full(x % nslot), (x / nslot) & 1, ab);
  for (int g = max(0, st_issued - st); g < st_issued; ++g) mbar_wait_drain(sm.st_full(g % st), (g / st) & 1, ab);
}

// Fused dQ: waits until the workspace tile's counter shows `want` contributions (all key
// tiles before this one). Bounded like the mbarrier waits.
__device__ __forceinline__ bool wait_turn(const int* cnt, int want, const Abort& ab) {
  if (ld_acquire_gpu(cnt) == want) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(cnt) == want) return true;
    if ((it & 15u) == 0) {
      if (*ab.flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        atomicOr(ab.err, kErrTimeoutOrder);
        *ab.flag = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2. dK / dV (and, fused, dQ)
// ---------------------------------------------------------------------------
// Work item = one 128-key tile j of one (b, h); its iterations run over the query tiles
// i (i >= j when causal). Persistent. With separate P^T / dS^T columns (d <= 64) two
// threads issue MMAs:
//   warp 17: S_i (= S^T, K_j Q_i^T) as soon as S_{i-1} was read out, dP_i likewise;
//   warp 18: dV += P_i^T dO_i once P_i^T is in TMEM, dK += dS_i^T Q_i once dS_i^T is.
// The next item's S and dP run while the elementwise warps store this item's dK, dV.
// At d = 128 (TMEM full, P^T / dS^T written over S^T / dP^T) one thread issues in the
// order S_0, dP_0 | P_0: dV_0, S_1 | dS_0: dK_0, dP_1 | ..., which relies on same-thread
// MMAs executing in issue order; persistent too (the next item's K_j, V_j and first S,
// dP overlap this item's epilogue).
//
// FUSE (d <= 64): the dQ contributions are formed here too, so the separate dQ kernel and
// its two recomputed GEMMs (S and dP) go away. The elementwise warps write dS^T to shared
// memory instead of TMEM; warp 18 then issues dK += dS^T Q_i from there and
// dQ_ij = dS K_j (the same tile read transposed) into the TMEM columns dS^T used to take.
// The elementwise warps move dQ_ij into a shared fp32 staging tile, and warp 19 adds it
// to the fp32 workspace tile of query tile i with one bulk shared->global copy (a plain
// copy for key tile 0, an fp32 reduce-add for the others). Each workspace tile has a
// counter of the contributions already added; the contribution of key tile j is added
// when the counter reads j, so every tile sums its terms in the order j = 0, 1, 2, ...
// and the result is the same on every run. Items run longest (smallest j) first, so a
// wait is only ever on an item that started no later; all CTAs of the persistent grid
// are resident together (one per SM).
template <int D, bool CAUSAL, bool FUSE, bool SPLIT, bool GROUPED>
__global__ void __launch_bounds__(BwdCfg<D, FUSE>::THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                         const float* __restrict__ ws_nlse2, const float* __restrict__ ws_D,
                         __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, float* __restrict__ dq_acc,
                         int* __restrict__ dq_cnt, float* __restrict__ part, int T, int T_pad, int BH, int G,
                         int S_, int HG, float scale, float scale_log2, uint32_t* __restrict__ err) {
  // persistent d <= 64: dV and dK leave through shared memory and TMA stores (not when
  // SPLIT: then each work item writes fp32 partial sums)
  constexpr bool EPI = BwdCfg<D>::SEP_DKDV && !FUSE && !SPLIT;
  const int S = SPLIT ? S_ : 1;  // splits of each key/value head's query heads
  constexpr int NEPI = EPI ? 2 : 0;
  using C = BwdCfg<D, FUSE, 2, NEPI>;
  using TL = Tile<D>;
  using TD = Tile<128>;  // the dS^T tile: 128 key rows x 128 query columns
  constexpr int ST = C::STAGES;
  constexpr bool SEP = C::SEP_DKDV;
  extern __shared__ uint8_t smem_raw[];
  uint32_t* tmem_slot;
  volatile int* abort;
  const BwdSmem sm = bwd_smem_setup<D, FUSE, 2, NEPI>(smem_raw, tmem_slot, abort);
  const Abort ab{abort, err};
  const uint32_t tmem = *tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_q = (T + kTileRows - 1) / kTileRows;
  // BH counts key/value slices; each is shared by G query heads (grouped key/value heads,
  // G = 1 without), whose query tiles all feed its dK and dV. With S > 1 (few key/value
  // heads) the G query heads are split over S work items, each writing fp32 partial sums
  // that a second launch adds in split order.
  // item u: key tile u / (BH S) (small j = most work first), key/value slice
  // (u % (BH S)) / S, split u % S over query heads [sp G / S, (sp + 1) G / S);
  // iteration it: query head kv * G + h0 + it / n_per, query tile i0 + it % n_per.
  // GROUPED (S = 1; two groups of HG = BH / 2 key/value slices, slices_per_group): group
  // g = u >= n_q HG, v = u - g n_q HG, key tile v / HG, key/value slice g HG + v % HG
  static_assert(!(GROUPED && (SPLIT || FUSE)), "grouped order: unsplit, unfused items");
  const int n_group = n_q * HG;
  const auto sched = make_sched<GROUPED>(n_q * BH * S, n_group);
  auto key_tile = [&](int u) {
    if constexpr (GROUPED) return (u >= n_group ? u - n_group : u) / HG;
    else return u / (BH * S);
  };
  auto kv_slice = [&](int u) {
    if constexpr (GROUPED) return u >= n_group ? HG + (u - n_group) % HG : u % HG;
    else return (u % (BH * S)) / S;
  };
  auto head0 = [&](int u) { return (u % S) * G / S; };
  auto n_iters = [&](int u) {
    return ((u % S + 1) * G / S - head0(u)) * (n_q - (CAUSAL ? key_tile(u) : 0));
  };
  constexpr bool epi = EPI;  // TMA-store epilogue (else plain or partial stores)

  constexpr int NS = C::NSLOT;
  auto sKf = [&](int slot) { return sm.base + C::OFF_FIX + slot * C::SLOT_BYTES; };  // K_j, then V_j
  auto sQ = [&](int s) { return sm.base + C::OFF_STAGE + s * C::STAGE_BYTES; };
  auto sdO = [&](int s) { return sQ(s) + TL::BYTES; };
  auto sL = [&](int s) { return sQ(s) + 2 * TL::BYTES; };  // 128 fp32 -LSE*log2e, then 128 fp32 D
  const uint32_t sDS = sm.base + C::OFF_DS, sDQS = sm.base + C::OFF_DQS, sEPI = sm.base + C::OFF_EPI;

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      // Q_i and dO_i are read by every key tile of their head: keep them in L2; K_j, V_j once
      const uint64_t keep = l2_evict_last(), once = l2_evict_first();
      bool ok = true;
      int g = 0, r = 0, fix_issued = 0;
      for (int u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int kt = key_tile(u), bh = kv_slice(u), i0 = CAUSAL ? kt : 0, n_it = n_iters(u);
        const int slot = r % NS;
        if (r >= NS && !(ok = mbar_wait(sm.fix_empty(slot), (r / NS - 1) & 1, ab, kErrTimeoutLoad))) break;
        if (!(ok = in_bounds(kt * kTileRows < T && bh < BH, ab))) break;
        ++fix_issued;
        mbar_arrive_expect_tx(sm.fix_full(slot), 2 * TL::BYTES);
        TL::load(sKf(slot), &tmK, kt * kTileRows, bh, sm.fix_full(slot), once);
        TL::load(sKf(slot) + TL::BYTES, &tmV, kt * kTileRows, bh, sm.fix_full(slot), once);
        for (int it = 0, qi = i0, bq = bh * G + head0(u); it < n_it; ++it, ++g) {
          const int s = g % ST, n = g / ST;
          if (g >= ST && !(ok = mbar_wait(sm.st_empty(s), (n - 1) & 1, ab, kErrTimeoutLoad))) break;
          const size_t woff = (size_t)bq * T_pad + (size_t)qi * kTileRows;
          if (!(ok = in_bounds(qi * kTileRows < T && bq < BH * G && woff + kTileRows <= (size_t)BH * G * T_pad, ab)))
            break;
          mbar_arrive_expect_tx(sm.st_full(s), 2 * TL::BYTES + 1024);
          TL::load(sQ(s), &tmQ, qi * kTileRows, bq, sm.st_full(s), keep);
          TL::load(sdO(s), &tmdO, qi * kTileRows, bq, sm.st_full(s), keep);
          bulk_load(sL(s), ws_nlse2 + woff, 512, sm.st_full(s));
          bulk_load(sL(s) + 512, ws_D + woff, 512, sm.st_full(s));
          if (++qi == n_q) {  // the next query head of the group
            qi = i0;
            ++bq;
          }
        }
      }
      if (!ok) drain_loads(sm, fix_issued, C::NSLOT, g, ST, ab);
    }
  } else if (warp == kWarpMmaA) {
    // ------------------------------------------------------------ MMA issuer (S, dP)
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, 0, 1);
      const uint32_t tS = tmem, tDP = tmem + 128u, tDV = tmem + 256u, tDK = tmem + 256u + (uint32_t)TL::ACC_COLS;
      // K-step-0 descriptors: K_j / V_j per item (their slot), stage s adds s stages
      uint64_t dKk = 0, dVk = 0;
      const uint64_t dQk0 = TL::desc_kmajor0(sQ(0)), dQm0 = TL::desc_mnmajor0(sQ(0));
      const uint64_t dOk0 = TL::desc_kmajor0(sdO(0)), dOm0 = TL::desc_mnmajor0(sdO(0));
      constexpr uint64_t kStageOff = TL::bytes_off(C::STAGE_BYTES);
      auto issue_S = [&](int s) {  // S^T = K_j Q_i^T (M = keys, N = queries, K = d)
        mma_chain_ss<TL, TL::KSTEPS_D>(tS, dKk, dQk0 + (uint64_t)s * kStageOff, idesc_s, 0u);
      };
      auto issue_dP = [&](int s) {  // dP^T = V_j dO_i^T
        mma_chain_ss<TL, TL::KSTEPS_D>(tDP, dVk, dOk0 + (uint64_t)s * kStageOff, idesc_s, 0u);
      };
      bool ok = true;
      int g = 0;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int n_it = n_iters(u), slot = r % NS;
        if (!(ok = mbar_wait(sm.fix_full(slot), (r / NS) & 1, ab, kErrTimeoutMma))) break;
        dKk = TL::desc_kmajor0(sKf(slot));
        dVk = TL::desc_kmajor0(sKf(slot) + TL::BYTES);
        if constexpr (SEP) {
          for (int it = 0; it < n_it; ++it, ++g) {
            const int s = g % ST;
            if (g > 0 && !(ok = mbar_wait(sm.s_free(), (g - 1) & 1, ab, kErrTimeoutMma))) break;
            if (!(ok = mbar_wait(sm.st_full(s), (g / ST) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            issue_S(s);
            mma_commit(sm.s_full());
            if (g > 0 && !(ok = mbar_wait(sm.dp_free(), (g - 1) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            issue_dP(s);
            mma_commit(sm.dp_full());
            // K_j, V_j are no longer read (with FUSE, K_j is read by the dQ MMAs of warp 18,
            // which releases them)
            if (!FUSE && it == n_it - 1) mma_commit(sm.fix_empty(slot));
          }
        } else {
          // P^T / dS^T written over S^T / dP^T: same-thread issue order is the guard
          if (!(ok = mbar_wait(sm.st_full(g % ST), (g / ST) & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          issue_S(g % ST);
          mma_commit(sm.s_full());
          issue_dP(g % ST);
          mma_commit(sm.dp_full());
          for (int it = 0; it < n_it; ++it, ++g) {
            const int s = g % ST, s1 = (g + 1) % ST;
            const bool more = it + 1 < n_it;
            if (!(ok = mbar_wait(sm.p_full(), g & 1, ab, kErrTimeoutMma))) break;
            if (it == 0 && r > 0 && !(ok = mbar_wait(sm.acc_free(), (r - 1) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            mma_chain_ts<TL, true>(tDV, tS, dOm0 + (uint64_t)s * kStageOff, idesc_acc, it > 0 ? 1u : 0u);
            if (more) {
              if (!(ok = mbar_wait(sm.st_full(s1), ((g + 1) / ST) & 1, ab, kErrTimeoutMma))) break;
              tc_fence_after();
              issue_S(s1);
              mma_commit(sm.s_full());
            }
            if (!(ok = mbar_wait(sm.ds_full(), g & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            mma_chain_ts<TL, true>(tDK, tDP, dQm0 + (uint64_t)s * kStageOff, idesc_acc, it > 0 ? 1u : 0u);
            mma_commit(sm.st_empty(s));
            if (more) {
              issue_dP(s1);
              mma_commit(sm.dp_full());
            }
          }
          if (!ok) break;
          mma_commit(sm.fix_empty(slot));
          mma_commit(sm.acc_full());
        }
      }
      if (!ok) {
        mma_commit(sm.drain());
        mbar_wait_drain(sm.drain(), 0, ab);
      }
    }
  } else if (warp == kWarpMmaB) {
    // ------------------------------------------------------------ MMA issuer (dV, dK)
    if (lane == 0 && SEP) {
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, 0, 1);
      const uint32_t tDV = tmem + 256u, tDK = tmem + 256u + (uint32_t)TL::ACC_COLS;
      const uint64_t dQm0 = TL::desc_mnmajor0(sQ(0)), dOm0 = TL::desc_mnmajor0(sdO(0));
      constexpr uint64_t kStageOff = TL::bytes_off(C::STAGE_BYTES);
      // EPI: the previous item's dV / dK tiles, staged by the elementwise warps before they
      // arrived on acc_free, go out with TMA stores (rows past T are clipped by the maps)
      auto store_epi = [&](int u_prev) {
#pragma unroll
        for (int c = 0; c < TL::NCHUNK; ++c) {
          const int row0 = key_tile(u_prev) * kTileRows, bh_prev = kv_slice(u_prev);
          if (!in_bounds(row0 >= 0 && row0 < T && bh_prev < BH, ab)) continue;
          tma_store_3d(&tmdV, sEPI + c * TL::CHUNK_BYTES, c * TL::CHUNK_ELEMS, row0, bh_prev);
          tma_store_3d(&tmdK, sEPI + TL::BYTES + c * TL::CHUNK_BYTES, c * TL::CHUNK_ELEMS, row0, bh_prev);
        }
        bulk_commit();
      };
      bool ok = true;
      int g = 0, u_prev = -1;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int n_it = n_iters(u);
        for (int it = 0; it < n_it; ++it, ++g) {
          const int s = g % ST;
          if (!(ok = mbar_wait(sm.p_full(), g & 1, ab, kErrTimeoutMma))) break;
          // the accumulators still hold the previous item until its epilogue read them
          if (it == 0 && r > 0 && !(ok = mbar_wait(sm.acc_free(), (r - 1) & 1, ab, kErrTimeoutMma))) break;
          if (epi && it == 0 && r > 0) store_epi(u_prev);
          tc_fence_after();
          // dV += P^T dO_i (M = keys, N = d, K = queries)
          mma_chain_ts<TL, false>(tDV, tmem + C::COL_P, dOm0 + (uint64_t)s * kStageOff, idesc_acc, it > 0 ? 1u : 0u);
          mma_commit(sm.dv_done());
          if (!(ok = mbar_wait(sm.ds_full(), g & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          if constexpr (FUSE) {
            // dK += dS^T Q_i, dS^T from shared memory (K-major: key rows, query columns)
            const uint64_t a0 = TD::desc_kmajor0(sDS), b0 = dQm0 + (uint64_t)s * kStageOff;
#pragma unroll
            for (int k = 0; k < kTileRows / 16; ++k)
              mma_ss(tDK, a0 + TD::kmajor_off(k), b0 + TL::mnmajor_off(k), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
            // dQ_ij = dS K_j (M = queries, N = d, K = keys): the same tile as an M-major A
            // operand; its TMEM columns must have been read out by the elementwise warps
            if (g > 0 && !(ok = mbar_wait(sm.dq_free(), (g - 1) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            constexpr uint32_t idesc_dq = idesc_bf16(128, D, 1, 1);
            const uint64_t q0 = TD::desc_mnmajor0(sDS), k0 = TL::desc_mnmajor0(sKf(0));  // FUSE: one slot
#pragma unroll
            for (int k = 0; k < kTileRows / 16; ++k)
              mma_ss(tmem + C::COL_DQ, q0 + TD::mnmajor_off(k), k0 + TL::mnmajor_off(k), idesc_dq, k > 0 ? 1u : 0u);
            mma_commit(sm.dq_done());  // dS^T tile and dQ_ij columns
          } else {
            // dK += dS^T Q_i
            mma_chain_ts<TL, false>(tDK, tmem + C::COL_DS, dQm0 + (uint64_t)s * kStageOff, idesc_acc,
                                    it > 0 ? 1u : 0u);
            mma_commit(sm.dk_done());
          }
          // S_i and dP_i (warp 17) were read out before P_i / dS_i were signalled, so this
          // commit covers every MMA that reads stage s
          mma_commit(sm.st_empty(s));
        }
        if (ok) mma_commit(sm.acc_full());
        if (FUSE && ok) mma_commit(sm.fix_empty(0));  // K_j (dQ MMAs) and V_j are no longer read
        if (epi && ok && r > 0) {
          // the previous item's stores have read the staging tiles: the next epilogue may
          // overwrite them
          bulk_wait_read_all();
          mbar_arrive(sm.epi_free());
        }
        u_prev = u;
      }
      if (epi && ok && u_prev >= 0) {
        // the last item: wait for its epilogue to fill the staging tiles, store them
        if ((ok = mbar_wait(sm.acc_free(), (sched_count(sched) - 1) & 1, ab, kErrTimeoutMma))) store_epi(u_prev);
      }
      if (EPI) bulk_wait_all();  // every store has landed before the CTA exits
      if (!ok) {
        mma_commit(sm.drain2());
        mbar_wait_drain(sm.drain2(), 0, ab);
      }
    }
  } else if (FUSE && warp == kWarpRed) {
    // ------------------------------------------------------------ dQ reducer (fused)
    // adds each staged dQ_ij to workspace tile (b, h, i) in key-tile order
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int kt = key_tile(u), bh = kv_slice(u), i0 = CAUSAL ? kt : 0, n_it = n_iters(u);
        for (int it = 0; it < n_it; ++it, ++g) {
          const int qi = i0 + it;
          if (!(ok = mbar_wait(sm.dqs_full(), g & 1, ab, kErrTimeoutMma))) break;
          int* cnt = dq_cnt + (size_t)bh * n_q + qi;
          if (kt > 0 && !(ok = wait_turn(cnt, kt, ab))) break;
          fence_proxy_async_global();
          float* dst = dq_acc + ((size_t)bh * n_q + qi) * (kTileRows * D);
          if (kt == 0)
            bulk_store(dst, sDQS, C::DQS_BYTES);  // the first term of this tile
          else
            bulk_reduce_add_f32(dst, sDQS, C::DQS_BYTES);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(sm.dqs_free());
          bulk_wait_all();
          fence_proxy_async_global();
          st_release_gpu(cnt, kt + 1);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // thread owns key row kt*128 + r and query columns [32*hc, 32*hc + 32)
    const int hc = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lo = warp_lane_base();
    const uint32_t tSh = tmem + lo + 32u * hc, tDPh = tmem + lo + 128u + 32u * hc;
    const uint32_t tP = tmem + lo + (SEP ? C::COL_P + 16u * hc : 32u * hc);
    const uint32_t tDS = tmem + lo + (SEP ? C::COL_DS + 16u * hc : 128u + 32u * hc);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    // FUSE: this thread's part of the dS^T tile (key row r, query columns 32hc..32hc+31)
    // is 16-byte granules 4(hc%2)..4(hc%2)+3 of row r in chunk hc/2, in the 128-byte
    // swizzle (granule position XOR r%8) that the tensor core reads
    const uint32_t ds_row = sDS + (uint32_t)(hc >> 1) * TD::CHUNK_BYTES + (uint32_t)r * 128u;
    const uint32_t ds_g0 = 4u * (uint32_t)(hc & 1);
    // FUSE: dQ_ij readout; here the TMEM lane r is a query row and the thread takes d
    // columns [QW hc, QW hc + QW). The staging tile is [granule c4][row][4 floats], so a
    // warp's 16-byte stores cover 512 contiguous bytes.
    constexpr int QW = D / 4;
    const uint32_t tDQ = tmem + lo + C::COL_DQ + (uint32_t)(QW * hc);
    bool ok = true;
    auto dq_readout = [&](int x) {  // moves iteration x's dQ_ij into the staging tile
      if constexpr (FUSE) {
      if (!(ok = mbar_wait_warp(sm.dq_done(), x & 1, ab, kErrTimeoutElem))) return;
      tc_fence_after();
      uint32_t v[QW];
      if constexpr (QW == 32) tmem_ld32(tDQ, v);
      else if constexpr (QW == 16) tmem_ld16(tDQ, v);
      else tmem_ld8(tDQ, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(sm.dq_free());
      if (x > 0 && !(ok = mbar_wait_warp(sm.dqs_free(), (x - 1) & 1, ab, kErrTimeoutElem))) return;
#pragma unroll
      for (int k = 0; k < QW / 4; ++k)
        sts128(sDQS + (uint32_t)(((QW / 4) * hc + k) * kTileRows + r) * 16u, v[4 * k], v[4 * k + 1], v[4 * k + 2],
               v[4 * k + 3]);
      fence_proxy_async_smem();
      mbar_arrive(sm.dqs_full());
      }
    };
    // ---- epilogue of item ri_e (work item u_e): dV, dK (x scale) out of the accumulators,
    // then free them. In the persistent kernel (not split: its fp32 partials would spill
    // there) it is deferred into the next item's first iteration (after that iteration's P
    // is computed, before it is written), so that the wait for the item's last dK MMA
    // overlaps that computation.
    constexpr bool DEFER = SEP && !FUSE && !SPLIT;
    auto epilogue = [&](int ri_e, int u_e) {
      if (!(ok = mbar_wait_warp(sm.acc_full(), ri_e & 1, ab, kErrTimeoutElem))) return;
      tc_fence_after();
      const int bh_e = kv_slice(u_e), key = key_tile(u_e) * kTileRows + r;
      const bool key_ok = key < T && in_bounds(bh_e < BH && key >= 0, ab);
      const uint32_t tDV = tmem + lo + 256u, tDK = tmem + lo + 256u + (uint32_t)TL::ACC_COLS;
      if constexpr (SPLIT) {
        // fp32 partial sums of this split (unscaled), [S][key/value slice][T_pad][d] for dK
        // then the same for dV; rows past T are written too and never read
        const size_t off = (((size_t)(u_e % S) * BH + bh_e) * T_pad + key) * D;
        if (in_bounds(off + D <= (size_t)S * BH * T_pad * D, ab)) {
          store_acc_quarter_f32<D>(tDK, part + off, hc);
          store_acc_quarter_f32<D>(tDV, part + (size_t)S * BH * T_pad * D + off, hc);
        }
      } else if constexpr (EPI) {
        // into the staging tiles (free once the previous item's TMA stores have read them);
        // warp 18 stores them once acc_free says every thread has written its part
        if (ri_e > 0 && !(ok = mbar_wait_warp(sm.epi_free(), (ri_e - 1) & 1, ab, kErrTimeoutElem))) return;
        stage_acc_quarter<D>(tDV, sEPI, r, hc, 1.f);  // (EPI: compile-time d <= 64)
        stage_acc_quarter<D>(tDK, sEPI + TL::BYTES, r, hc, scale);
        fence_proxy_async_smem();
      } else {
        store_acc_quarter<D>(tDV, dv + ((size_t)bh_e * T + key) * D, hc, 1.f, key_ok);
        store_acc_quarter<D>(tDK, dk + ((size_t)bh_e * T + key) * D, hc, scale, key_ok);
      }
      tc_fence_before();
      mbar_arrive(sm.acc_free());
    };
    int pend_ri = -1, pend_u = 0;  // an item whose epilogue is deferred (DEFER)
    int g = 0;
    for (int ri = 0, u; ok && (u = sched.item(ri)) >= 0; ++ri) {
      const int kt = key_tile(u), bh = kv_slice(u), i0 = CAUSAL ? kt : 0, n_it = n_iters(u);
      for (int it = 0, qi = i0; it < n_it; ++it, ++g, qi = (qi + 1 == n_q) ? i0 : qi + 1) {
        const int s = g % ST;
        if (!(ok = mbar_wait_warp(sm.s_full(), g & 1, ab, kErrTimeoutElem))) break;
        if (!(ok = mbar_wait_warp(sm.st_full(s), (g / ST) & 1, ab, kErrTimeoutElem))) break;
        tc_fence_after();
        const float* nl = reinterpret_cast<const float*>(sm.gbase + (sL(s) - sm.base)) + 32 * hc;
        const float* dd = nl + 128;
        // ---- P^T = exp2(S^T * scale*log2e - LSE_i*log2e), kept in fp32 for dS
        float p[32];
        {
          uint32_t u2[32];
          tmem_ld32(tSh, u2);
          tmem_wait_ld();
          if (SEP) {
            tc_fence_before();
            mbar_arrive(sm.s_free());  // S^T_i is in registers
          }
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 L = reinterpret_cast<const float4*>(nl)[i4];  // 128-bit shared loads
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = 2 * i4 + h;
              const uint64_t x = f2_fma(f2_pack(__uint_as_float(u2[2 * i]), __uint_as_float(u2[2 * i + 1])), c2,
                                        h ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y));
              float x0, x1;
              f2_unpack(x, x0, x1);
              p[2 * i] = ex2(x0);
              p[2 * i + 1] = ex2(x1);
            }
          }
        }
        if (CAUSAL && qi == kt) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (32 * hc + c < r) p[c] = 0.f;
        }
        {
          uint32_t pp[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pp[i] = pack_bf16(p[2 * i], p[2 * i + 1]);
          if (DEFER && it == 0 && pend_ri >= 0) {
            epilogue(pend_ri, pend_u);  // the previous item's dV, dK (warp 18 waits for them
            pend_ri = -1;               // before this item's first dV MMA)
            if (!ok) break;
          }
          // the previous dV read the P^T columns: it must be complete before they are rewritten
          if (SEP && g > 0 && !(ok = mbar_wait_warp(sm.dv_done(), (g - 1) & 1, ab, kErrTimeoutElem))) break;
          tc_fence_after();
          tmem_st16(tP, pp);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sm.p_full());
        if (FUSE && g > 0) {
          // the previous iteration's dQ_ij; this also frees the dS^T tile for this one
          dq_readout(g - 1);
          if (!ok) break;
        }
        // ---- dS^T = P^T * (dP^T - D_i)
        if (!(ok = mbar_wait_warp(sm.dp_full(), g & 1, ab, kErrTimeoutElem))) break;
        tc_fence_after();
        {
          uint32_t u2[32];
          tmem_ld32(tDPh, u2);
          tmem_wait_ld();
          if (SEP) {
            tc_fence_before();
            mbar_arrive(sm.dp_free());  // dP^T_i is in registers
          }
          uint32_t pd[16];
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 Dv = reinterpret_cast<const float4*>(dd)[i4];  // 128-bit shared loads
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = 2 * i4 + h;
              const uint64_t gg = f2_mul(f2_pack(p[2 * i], p[2 * i + 1]),
                                         f2_sub(f2_pack(__uint_as_float(u2[2 * i]), __uint_as_float(u2[2 * i + 1])),
                                                h ? f2_pack(Dv.z, Dv.w) : f2_pack(Dv.x, Dv.y)));
              float g0, g1;
              f2_unpack(gg, g0, g1);
              pd[i] = pack_bf16(g0, g1);
            }
          }
          if constexpr (FUSE) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              sts128(ds_row + (((ds_g0 + (uint32_t)k) ^ (uint32_t)(r & 7)) << 4), pd[4 * k], pd[4 * k + 1],
                     pd[4 * k + 2], pd[4 * k + 3]);
            fence_proxy_async_smem();
          } else {
            if (SEP && g > 0 && !(ok = mbar_wait_warp(sm.dk_done(), (g - 1) & 1, ab, kErrTimeoutElem))) break;
            tc_fence_after();
            tmem_st16(tDS, pd);
          }
        }
        if (!FUSE) tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sm.ds_full());
      }
      if (!ok) break;
      if constexpr (DEFER) {
        pend_ri = ri;
        pend_u = u;
      } else {
        epilogue(ri, u);
        if (!ok) break;
      }
    }
    if (DEFER && ok && pend_ri >= 0) epilogue(pend_ri, pend_u);  // the last item
    if (FUSE && ok && g > 0) dq_readout(g - 1);  // the last iteration's dQ_ij
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ
// ---------------------------------------------------------------------------
// K and V rings of the dQ kernel. K_j is read by S_j and, last, by dQ_j; V_j by dP_j
// alone, so a V slot turns over about one MMA group sooner than a K slot. At d >= 80 the
// K ring has a third slot: K_{j+3} loads while iteration j + 1 runs (two combined K/V
// stages left the S MMA waiting for its K tile).
template <int D>
struct DqRing {
  static constexpr int K = D > 64 ? 3 : BwdCfg<D>::STAGES;
  static constexpr int V = D > 64 ? 2 : BwdCfg<D>::STAGES;
};

// Work item = one 128-query tile i of one (b, h); its iterations run over the key tiles
// j (j <= i when causal). Persistent, two MMA issuers:
//   warp 17: S_j = Q_i K_j^T as soon as S_{j-1} was read out, dP_j = dO_i V_j^T likewise;
//   warp 18: dQ += dS_j K_j once dS_j (its own 64 TMEM columns) is written.
// At d <= 64 the dQ accumulator has two TMEM buffers (items alternate), and the
// elementwise warps store an item's dQ during the next item's first iteration, by when
// its last dQ MMA has finished, instead of waiting for it at the end of the item.
// PRE (d <= 64): the kernel also does the preprocess for its query tile, so that it runs
// first and no separate D launch is needed: O_i is staged with Q_i and dO_i, the
// elementwise threads form D_i = rowsum(dO_i * O_i) and -LSE_i * log2(e) themselves at the
// start of the item and write both to the workspace for the dK/dV kernel that follows.
// At d >= 80 the S and dP MMAs (eight K-steps each) get one thread each (warp 17 and a
// third issuer, warp 19): a thread issues one tcgen05.mma about every hundred cycles
// however short the MMA, and one thread issuing both bounded the iteration.
template <int D>
constexpr int dq_threads() { return D > 64 ? kBwdThreads + 32 : kBwdThreads; }

template <int D, bool CAUSAL, bool PRE, bool GROUPED>
__global__ void __launch_bounds__(dq_threads<D>(), 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmO, const float* __restrict__ lse,
                       float* __restrict__ ws_nlse2, float* __restrict__ ws_D, __nv_bfloat16* __restrict__ dq,
                       int T, int T_pad, int BH, int G, int HG, float scale, float scale_log2,
                       uint32_t* __restrict__ err) {
  constexpr int NFIX = PRE ? 3 : 2;
  constexpr int KR = DqRing<D>::K, VR = DqRing<D>::V;
  using C = BwdCfg<D, false, NFIX, 0, KR, VR>;
  using TL = Tile<D>;
  extern __shared__ uint8_t smem_raw[];
  uint32_t* tmem_slot;
  volatile int* abort;
  // with PRE the elementwise threads read O_i and dO_i themselves: they release them too;
  // with a separate dP issuer (d >= 80) Q_i and dO_i are released by two MMA threads
  constexpr bool SPLIT_SDP = D > 64;
  const BwdSmem sm = bwd_smem_setup<D, false, NFIX, 0, KR, VR>(smem_raw, tmem_slot, abort,
                                                               PRE ? 1u + kEwThreads : (SPLIT_SDP ? 2u : 1u));
  const Abort ab{abort, err};
  const uint32_t tmem = *tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_k = (T + kTileRows - 1) / kTileRows;
  // item u: query tile n_k - 1 - u / BH (largest, i.e. most work, first), slice u % BH;
  // GROUPED (two groups of HG = BH / 2 slices, slices_per_group): group g = u >= n_k HG,
  // v = u - g n_k HG, query tile n_k - 1 - v / HG, slice g HG + v % HG
  const int n_group = n_k * HG;
  const auto sched = make_sched<GROUPED>(n_k * BH, n_group);
  auto query_tile = [&](int u) {
    if constexpr (GROUPED) return n_k - 1 - (u >= n_group ? u - n_group : u) / HG;
    else return n_k - 1 - u / BH;
  };
  auto slice_of = [&](int u) {
    if constexpr (GROUPED) return u >= n_group ? HG + (u - n_group) % HG : u % HG;
    else return u % BH;
  };
  auto n_iters = [&](int u) { return CAUSAL ? query_tile(u) + 1 : n_k; };

  constexpr int NS = C::NSLOT;
  // fixed tiles of slot b: Q_i, dO_i (, O_i)
  auto sQf = [&](int b) { return sm.base + C::OFF_FIX + b * C::SLOT_BYTES; };
  // dQ accumulator buffers: [256, 256 + D) and, at d <= 64, [320 + D, 320 + 2D) after dS;
  // buffer 1's full / free barriers are the ones the dK/dV kernel uses for dv_done / p_full
  constexpr int NACC = D <= 64 ? 2 : 1;
  auto acc_col = [&](int b) { return 256u + (b ? (uint32_t)D + 64u : 0u); };
  // tensor-memory plan: S [0, 128), dP [128, 256), dQ buffer 0, dS (64 columns), dQ buffer 1
  static_assert(256 + TL::ACC_COLS + 64 + (NACC == 2 ? D : 0) <= 512, "dQ kernel columns");
  auto acc_full_b = [&](int b) { return b ? sm.dv_done() : sm.acc_full(); };
  auto acc_free_b = [&](int b) { return b ? sm.p_full() : sm.acc_free(); };
  auto sK = [&](int s) { return sm.base + C::OFF_STAGE + s * TL::BYTES; };
  auto sV = [&](int s) { return sm.base + C::OFF_STAGE + (KR + s) * TL::BYTES; };
  constexpr uint64_t kSlotOff = TL::bytes_off(TL::BYTES);

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      // K_j and V_j are read by every query tile of their head: keep them in L2; Q_i, dO_i once
      const uint64_t keep = l2_evict_last(), once = l2_evict_first();
      bool ok = true;
      int g = 0, r = 0, fix_issued = 0, nk = 0, nv = 0;
      for (int u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int qt = query_tile(u), bh = slice_of(u), n_it = n_iters(u);
        const int slot = r % NS;
        if (r >= NS && !(ok = mbar_wait(sm.fix_empty(slot), (r / NS - 1) & 1, ab, kErrTimeoutLoad))) break;
        if (!(ok = in_bounds(qt >= 0 && qt * kTileRows < T && bh < BH, ab))) break;
        ++fix_issued;
        mbar_arrive_expect_tx(sm.fix_full(slot), NFIX * TL::BYTES);
        TL::load(sQf(slot), &tmQ, qt * kTileRows, bh, sm.fix_full(slot), once);
        TL::load(sQf(slot) + TL::BYTES, &tmdO, qt * kTileRows, bh, sm.fix_full(slot), once);
        if (PRE) TL::load(sQf(slot) + 2 * TL::BYTES, &tmO, qt * kTileRows, bh, sm.fix_full(slot), once);
        for (int it = 0; it < n_it; ++it, ++g) {
          const int sk = g % KR, sv = g % VR;
          // query head bh reads key/value slice bh / G (grouped key/value heads; G = 1 without)
          if (g >= KR && !(ok = mbar_wait(sm.st_empty(sk), (g / KR - 1) & 1, ab, kErrTimeoutLoad))) break;
          if (!(ok = in_bounds(it * kTileRows < T && bh / G < BH / G, ab))) break;
          mbar_arrive_expect_tx(sm.st_full(sk), TL::BYTES);
          TL::load(sK(sk), &tmK, it * kTileRows, bh / G, sm.st_full(sk), keep);
          ++nk;
          if (g >= VR && !(ok = mbar_wait(sm.v_empty(sv), (g / VR - 1) & 1, ab, kErrTimeoutLoad))) break;
          mbar_arrive_expect_tx(sm.v_full(sv), TL::BYTES);
          TL::load(sV(sv), &tmV, it * kTileRows, bh / G, sm.v_full(sv), keep);
          ++nv;
        }
      }
      if (!ok) {
        drain_loads(sm, fix_issued, C::NSLOT, nk, KR, ab);  // fixed tiles and the K ring
        for (int x = max(0, nv - VR); x < nv; ++x) mbar_wait_drain(sm.v_full(x % VR), (x / VR) & 1, ab);
      }
    }
  } else if (warp == kWarpMmaA || (SPLIT_SDP && warp == kWarpMmaC)) {
    // ------------------------------------------------------------ MMA issuers (S, dP)
    // warp 17: S and dP (d <= 64), or S alone (d >= 80, with warp 19 issuing dP)
    if (lane == 0) {
      const bool do_S = warp == kWarpMmaA, do_dP = !SPLIT_SDP || warp == kWarpMmaC;
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      const uint32_t tS = tmem, tDP = tmem + 128u;
      const uint64_t dKk0 = TL::desc_kmajor0(sK(0)), dVk0 = TL::desc_kmajor0(sV(0));
      bool ok = true;
      int g = 0;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int n_it = n_iters(u), slot = r % NS;
        if (!(ok = mbar_wait(sm.fix_full(slot), (r / NS) & 1, ab, kErrTimeoutMma))) break;
        const uint64_t dQk = TL::desc_kmajor0(sQf(slot)), dOk = TL::desc_kmajor0(sQf(slot) + TL::BYTES);
        for (int it = 0; it < n_it; ++it, ++g) {
          const int sk = g % KR, sv = g % VR;
          if (do_S) {
            if (g > 0 && !(ok = mbar_wait(sm.s_free(), (g - 1) & 1, ab, kErrTimeoutMma))) break;  // S read out
            if (!(ok = mbar_wait(sm.st_full(sk), (g / KR) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            // S = Q_i K_j^T (M = queries, N = keys, K = d)
            mma_chain_ss<TL, TL::KSTEPS_D>(tS, dQk, dKk0 + (uint64_t)sk * kSlotOff, idesc_s, 0u);
            mma_commit(sm.s_full());
          }
          if (do_dP) {
            if (g > 0 && !(ok = mbar_wait(sm.dp_free(), (g - 1) & 1, ab, kErrTimeoutMma))) break;  // dP read out
            if (!(ok = mbar_wait(sm.v_full(sv), (g / VR) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            // dP = dO_i V_j^T
            mma_chain_ss<TL, TL::KSTEPS_D>(tDP, dOk, dVk0 + (uint64_t)sv * kSlotOff, idesc_s, 0u);
            mma_commit(sm.dp_full());
            mma_commit(sm.v_empty(sv));  // V_j is read by dP_j only
          }
          // Q_i (S) and dO_i (dP) are no longer read by this thread
          if (it == n_it - 1) mma_commit(sm.fix_empty(slot));
        }
      }
      if (!ok) {
        const uint32_t dr = do_S ? sm.drain() : sm.drain3();
        mma_commit(dr);
        mbar_wait_drain(dr, 0, ab);
      }
    }
  } else if (warp == kWarpMmaB) {
    // ------------------------------------------------------------ MMA issuer (dQ)
    if (lane == 0) {
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, 0, 1);
      const uint32_t tDS = tmem + 256u + (uint32_t)TL::ACC_COLS;
      const uint64_t dKm0 = TL::desc_mnmajor0(sK(0));
      bool ok = true;
      int g = 0;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int n_it = n_iters(u), b = r % NACC;
        for (int it = 0; it < n_it; ++it, ++g) {
          const int sk = g % KR;
          if (!(ok = mbar_wait(sm.ds_full(), g & 1, ab, kErrTimeoutMma))) break;
          // this accumulator buffer still holds item r - NACC until its epilogue read it
          if (it == 0 && r >= NACC && !(ok = mbar_wait(acc_free_b(b), (r / NACC - 1) & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          // dQ += dS K_j (M = queries, N = d, K = keys); dS has its own 64 columns
          mma_chain_ts<TL, false>(tmem + acc_col(b), tDS, dKm0 + (uint64_t)sk * kSlotOff, idesc_acc,
                                  it > 0 ? 1u : 0u);
          mma_commit(sm.dk_done());  // "dQ_j done": the dS columns may be rewritten
          // K_j: S_j (warp 17) was read out before dS_j was signalled, dQ_j is its last reader
          mma_commit(sm.st_empty(sk));
        }
        if (ok) mma_commit(acc_full_b(b));
      }
      if (!ok) {
        mma_commit(sm.drain2());
        mbar_wait_drain(sm.drain2(), 0, ab);
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // thread owns query row qt*128 + r and key columns [32*hc, 32*hc + 32)
    const int hc = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lo = warp_lane_base();
    const uint32_t tSh = tmem + lo + 32u * hc, tDPh = tmem + lo + 128u + 32u * hc;
    const uint32_t tDS = tmem + lo + 256u + (uint32_t)TL::ACC_COLS + 16u * hc;
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    bool ok = true;
    int g = 0;
    // the epilogue of an item: its dQ (x scale) to memory, then free its accumulator
    auto epilogue = [&](int ri_e, int bh_e, int row_e) {
      const int b = ri_e % NACC;
      if (!(ok = mbar_wait_warp(acc_full_b(b), (ri_e / NACC) & 1, ab, kErrTimeoutElem))) return;
      tc_fence_after();
      store_acc_quarter<D>(tmem + lo + acc_col(b), dq + ((size_t)bh_e * T + row_e) * D, hc, scale,
                           row_e < T && in_bounds(bh_e < BH, ab));
      tc_fence_before();
      mbar_arrive(acc_free_b(b));
    };
    int pend_ri = -1, pend_bh = 0, pend_row = 0;  // an item whose epilogue is deferred (NACC = 2)
    for (int ri = 0, u; ok && (u = sched.item(ri)) >= 0; ++ri) {
      const int qt = query_tile(u), bh = slice_of(u), n_it = n_iters(u);
      const int row = qt * kTileRows + r;
      float nl, Dr;
      if constexpr (PRE) {
        // D for this row from the staged O_i and dO_i rows (zero past T, as TMA fills them)
        const int slot = ri % NS;
        if (!(ok = mbar_wait_warp(sm.fix_full(slot), (ri / NS) & 1, ab, kErrTimeoutElem))) break;
        const uint32_t sdO = sQf(slot) + TL::BYTES, sO = sdO + TL::BYTES;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int c = 0; c < TL::NCHUNK; ++c)
#pragma unroll
          for (int gi = 0; gi < TL::ROW_BYTES / 16; ++gi) {
            const uint32_t off = TL::granule_off(r, c, gi);
            const uint4 ov = lds128(sO + off), dv4 = lds128(sdO + off);
            const uint32_t* ow = &ov.x;
            const uint32_t* dw = &dv4.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) fma_bf16x2_f32(ow[e], dw[e], a0, a1);
          }
        mbar_arrive(sm.fix_empty(slot));  // O_i, dO_i read (the MMA commit is the other arrival)
        Dr = a0 + a1;
        nl = row < T ? -lse[(size_t)bh * T + row] * kLog2e : -INFINITY;
        if (hc == 0 && in_bounds(bh < BH && row < T_pad, ab)) {
          ws_nlse2[(size_t)bh * T_pad + row] = nl;
          ws_D[(size_t)bh * T_pad + row] = Dr;
        }
      } else {
        const bool in = in_bounds(bh < BH && row < T_pad, ab);
        nl = in ? ws_nlse2[(size_t)bh * T_pad + row] : -INFINITY;
        Dr = in ? ws_D[(size_t)bh * T_pad + row] : 0.f;
      }
      const uint64_t nl2 = f2_pack(nl, nl), D2 = f2_pack(Dr, Dr);
      for (int it = 0; it < n_it; ++it, ++g) {
        if (!(ok = mbar_wait_warp(sm.s_full(), g & 1, ab, kErrTimeoutElem))) break;
        tc_fence_after();
        float p[32];
        {
          uint32_t u2[32];
          tmem_ld32(tSh, u2);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(sm.s_free());  // S_j is in registers: the tensor core may overwrite it
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(u2[2 * i]), __uint_as_float(u2[2 * i + 1])), c2, nl2);
            float x0, x1;
            f2_unpack(x, x0, x1);
            p[2 * i] = ex2(x0);
            p[2 * i + 1] = ex2(x1);
          }
        }
        if (CAUSAL && it == qt) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (32 * hc + c > r) p[c] = 0.f;
        }
        if (!CAUSAL) {
          const int lim = T - it * kTileRows - 32 * hc;  // key columns >= lim are padding
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= lim) p[c] = 0.f;
        }
        if (!(ok = mbar_wait_warp(sm.dp_full(), g & 1, ab, kErrTimeoutElem))) break;
        tc_fence_after();
        {
          uint32_t u2[32];
          tmem_ld32(tDPh, u2);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(sm.dp_free());  // dP_j is in registers
          uint32_t pd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t gg = f2_mul(f2_pack(p[2 * i], p[2 * i + 1]),
                                       f2_sub(f2_pack(__uint_as_float(u2[2 * i]), __uint_as_float(u2[2 * i + 1])), D2));
            float g0, g1;
            f2_unpack(gg, g0, g1);
            pd[i] = pack_bf16(g0, g1);
          }
          // the previous dQ MMA read the dS columns: it must be complete before they are rewritten
          if (g > 0 && !(ok = mbar_wait_warp(sm.dk_done(), (g - 1) & 1, ab, kErrTimeoutElem))) break;
          tc_fence_after();
          tmem_st16(tDS, pd);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sm.ds_full());
        if (NACC == 2 && it == 0 && pend_ri >= 0) {
          // the previous item's dQ: its last MMA has finished while this iteration ran
          epilogue(pend_ri, pend_bh, pend_row);
          pend_ri = -1;
          if (!ok) break;
        }
      }
      if (!ok) break;
      // ---- epilogue: deferred into the next item's first iteration (two buffers), or now
      if (NACC == 2) {
        pend_ri = ri;
        pend_bh = bh;
        pend_row = row;
      } else {
        epilogue(ri, bh, row);
        if (!ok) break;
      }
    }
    if (ok && pend_ri >= 0) epilogue(pend_ri, pend_bh, pend_row);  // the last item
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// 4. fused dQ, last step: dQ = bf16(scale * workspace tile) for rows t < T
// ---------------------------------------------------------------------------
// The workspace tile of (b*h, i) holds 128 x d fp32 as [granule c4][row][4 floats]. A
// thread converts 8 columns of one row; consecutive threads take consecutive rows, so the
// reads of a warp are 512 contiguous bytes.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dq_finish_kernel(const float* __restrict__ acc,
                                                                 __nv_bfloat16* __restrict__ dq, int T, int T_pad,
                                                                 int BH, float scale) {
  constexpr int C8 = D / 8;
  griddep_begin();
  const int n_q = T_pad / kTileRows;
  const long long total = (long long)BH * T_pad * C8;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx % kTileRows);
    const long long rest = idx / kTileRows;
    const int c8 = (int)(rest % C8);
    const long long tile = rest / C8;  // bh * n_q + i
    const int bh = (int)(tile / n_q), t = (int)(tile % n_q) * kTileRows + r;
    if (t >= T) continue;
    const float4* src = reinterpret_cast<const float4*>(acc + tile * (kTileRows * D));
    const float4 x = src[(2 * c8) * kTileRows + r], y = src[(2 * c8 + 1) * kTileRows + r];
    uint4 o;
    o.x = pack_bf16(x.x * scale, x.y * scale);
    o.y = pack_bf16(x.z * scale, x.w * scale);
    o.z = pack_bf16(y.x * scale, y.y * scale);
    o.w = pack_bf16(y.z * scale, y.w * scale);
    *reinterpret_cast<uint4*>(dq + ((size_t)bh * T + t) * D + 8 * c8) = o;
  }
}

// ---------------------------------------------------------------------------
// 5. split dK/dV (few key/value heads): dK = bf16(scale * sum_s part_K[s]), dV = bf16(
//    sum_s part_V[s]), the splits added in order s = 0, 1, ... (deterministic)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dkdv_reduce_kernel(const float* __restrict__ part,
                                                                   __nv_bfloat16* __restrict__ dk,
                                                                   __nv_bfloat16* __restrict__ dv, int T, int T_pad,
                                                                   int BHkv, int S, float scale) {
  constexpr int C8 = D / 8;  // 8 columns (two float4) per thread
  griddep_begin();
  const long long rows = (long long)BHkv * T;
  const size_t plane = (size_t)BHkv * T_pad * D;  // one split's partial sums
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < rows * C8;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(idx % C8);
    const long long rt = idx / C8;
    const int bh = (int)(rt / T), t = (int)(rt % T);
    const size_t off = ((size_t)bh * T_pad + t) * D + 8 * c8;
    float ak[8] = {0, 0, 0, 0, 0, 0, 0, 0}, av[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int sp = 0; sp < S; ++sp) {
      const float4* pk = reinterpret_cast<const float4*>(part + sp * plane + off);
      const float4* pv = reinterpret_cast<const float4*>(part + (size_t)S * plane + sp * plane + off);
      const float4 k0 = pk[0], k1 = pk[1], v0 = pv[0], v1 = pv[1];
      ak[0] += k0.x; ak[1] += k0.y; ak[2] += k0.z; ak[3] += k0.w;
      ak[4] += k1.x; ak[5] += k1.y; ak[6] += k1.z; ak[7] += k1.w;
      av[0] += v0.x; av[1] += v0.y; av[2] += v0.z; av[3] += v0.w;
      av[4] += v1.x; av[5] += v1.y; av[6] += v1.z; av[7] += v1.w;
    }
    uint4 ok4, ov4;
    ok4.x = pack_bf16(ak[0] * scale, ak[1] * scale);
    ok4.y = pack_bf16(ak[2] * scale, ak[3] * scale);
    ok4.z = pack_bf16(ak[4] * scale, ak[5] * scale);
    ok4.w = pack_bf16(ak[6] * scale, ak[7] * scale);
    ov4.x = pack_bf16(av[0], av[1]);
    ov4.y = pack_bf16(av[2], av[3]);
    ov4.z = pack_bf16(av[4], av[5]);
    ov4.w = pack_bf16(av[6], av[7]);
    const size_t o = ((size_t)bh * T + t) * D + 8 * c8;
    *reinterpret_cast<uint4*>(dk + o) = ok4;
    *reinterpret_cast<uint4*>(dv + o) = ov4;
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <int D>
cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  // one CTA per 64 rows of each slice (T_pad is a multiple of 64)
  const dim3 grid((unsigned)((long long)a.T_pad / kPreRows * a.BH));
  const int n_cnt = a.dq_cnt ? a.BH * (a.T_pad / kTileRows) : 0;
  return launch_pdl(attn_bwd_preprocess_kernel<D>, grid, dim3(kPreThreads), 0, stream, a.o, a.dO, a.lse, a.ws_nlse2,
                    a.ws_D, a.dq_cnt, n_cnt, a.T, a.T_pad);
}

template <int D, bool CAUSAL, bool FUSE, bool SPLIT = false, bool GROUPED = false>
cudaError_t launch_dkdv(const BwdArgs& a, cudaStream_t stream) {
  if (!SPLIT && a.S > 1) return launch_dkdv<D, CAUSAL, FUSE, true>(a, stream);
  // Q and dO of a key/value slice's G query heads are read by all its items: at d >= 80,
  // when all key/value slices' Q and dO exceed the L2 budget, two groups of slices
  int hg = a.BH / a.G;
  if constexpr (D > 64 && !FUSE && !SPLIT && !GROUPED) {
    hg = slices_per_group(a.BH / a.G, 2ll * a.G * a.T_pad * D * 2);
    if (hg != a.BH / a.G) return launch_dkdv<D, CAUSAL, FUSE, false, true>(a, stream);
  } else if constexpr (GROUPED) {
    hg = a.BH / a.G / 2;
  }
  constexpr bool EPI = BwdCfg<D>::SEP_DKDV && !FUSE && !SPLIT;
  using C = BwdCfg<D, FUSE, 2, EPI ? 2 : 0>;
  auto kern = attn_bwd_dkdv_kernel<D, CAUSAL, FUSE, SPLIT, GROUPED>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, &configured);
  if (e != cudaSuccess) return e;
  const int n_items = (a.T + kTileRows - 1) / kTileRows * (a.BH / a.G) * a.S;  // key tiles x slices x splits
  // persistent: one CTA per SM walks its share of the items. Split items (few key/value
  // heads) differ in length by the split's head count as well as by key tile, and there
  // the hardware's dynamic dealing of one item per CTA, longest first, balances better
  // than a fixed per-CTA share.
  const int grid = SPLIT ? n_items : min(n_items, a.num_sms);
  if (EPI && (!a.tmdK || !a.tmdV)) return cudaErrorInvalidValue;
  // the fused dQ's CTAs wait on one another's contributions (per-tile counters): it is
  // launched cooperatively, so that it starts only when its whole grid (one CTA per SM,
  // at most the SM count) can be resident and every wait is on a running CTA
  auto go = [&](auto launcher) {
    return launcher(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, *a.tmQ, *a.tmK, *a.tmV, *a.tmdO,
                    EPI ? *a.tmdK : *a.tmQ, EPI ? *a.tmdV : *a.tmQ, a.ws_nlse2, a.ws_D, a.dk, a.dv, a.dq_acc,
                    a.dq_cnt, a.part, a.T, a.T_pad, a.BH / a.G, a.G, a.S, hg, a.scale, a.scale * kLog2e, a.err);
  };
  if constexpr (FUSE)
    return go([](auto&&... x) { return launch_coop(static_cast<decltype(x)&&>(x)...); });
  else
    return go([](auto&&... x) { return launch_pdl(static_cast<decltype(x)&&>(x)...); });
}

template <int D>
cudaError_t launch_dq_finish(const BwdArgs& a, cudaStream_t stream) {
  const long long total = (long long)a.BH * a.T_pad * (D / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)a.num_sms * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(attn_bwd_dq_finish_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, stream, a.dq_acc, a.dq, a.T,
                    a.T_pad, a.BH, a.scale);
}

template <int D, bool CAUSAL, bool GROUPED>
cudaError_t launch_dq_as(const BwdArgs& a, cudaStream_t stream, int hg) {
  // d <= 64: the dQ kernel forms D itself (and runs before dK/dV)
  constexpr bool PRE = D <= 64;
  using C = BwdCfg<D, false, PRE ? 3 : 2, 0, DqRing<D>::K, DqRing<D>::V>;
  static_assert(C::SMEM_BYTES <= 227 * 1024, "dQ kernel shared memory");
  auto kern = attn_bwd_dq_kernel<D, CAUSAL, PRE, GROUPED>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, &configured);
  if (e != cudaSuccess) return e;
  if (PRE && (!a.tmO || !a.lse)) return cudaErrorInvalidValue;
  const int n_items = (a.T + kTileRows - 1) / kTileRows * a.BH;
  return launch_pdl(kern, dim3(min(n_items, a.num_sms)), dim3(dq_threads<D>()), C::SMEM_BYTES, stream, *a.tmQ, *a.tmK,
                    *a.tmV, *a.tmdO, PRE ? *a.tmO : *a.tmQ, a.lse, a.ws_nlse2, a.ws_D, a.dq, a.T, a.T_pad, a.BH, a.G,
                    hg, a.scale, a.scale * kLog2e, a.err);
}

template <int D, bool CAUSAL>
cudaError_t launch_dq(const BwdArgs& a, cudaStream_t stream) {
  // K and V of a slice are read by all its items: at d >= 80, when all slices' K and V
  // exceed the L2 budget, two groups of slices (grouped key/value heads: one group)
  if constexpr (D > 64) {
    const int hg = a.G == 1 ? slices_per_group(a.BH, 2ll * a.T_pad * D * 2) : a.BH;
    if (hg != a.BH) return launch_dq_as<D, CAUSAL, true>(a, stream, hg);
  }
  return launch_dq_as<D, CAUSAL, false>(a, stream, a.BH);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return launch_pre<32>(a, stream);
    case 64: return launch_pre<64>(a, stream);
    case 80: return launch_pre<80>(a, stream);
    case 128: return launch_pre<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_dkdv_reduce(const BwdArgs& a, cudaStream_t stream) {
  const long long total = (long long)(a.BH / a.G) * a.T * (D / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)a.num_sms * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(attn_bwd_dkdv_reduce_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, stream, a.part, a.dk, a.dv,
                    a.T, a.T_pad, a.BH / a.G, a.S, a.scale);
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream) {
  if (a.S > 1 && !a.part) return cudaErrorInvalidValue;
  cudaError_t e;
  switch (a.d) {
    case 32: e = a.causal ? launch_dkdv<32, true, false>(a, stream) : launch_dkdv<32, false, false>(a, stream); break;
    case 64: e = a.causal ? launch_dkdv<64, true, false>(a, stream) : launch_dkdv<64, false, false>(a, stream); break;
    case 80: e = a.causal ? launch_dkdv<80, true, false>(a, stream) : launch_dkdv<80, false, false>(a, stream); break;
    case 128: e = a.causal ? launch_dkdv<128, true, false>(a, stream) : launch_dkdv<128, false, false>(a, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || a.S <= 1) return e;
  // split work items: add their partial sums
  switch (a.d) {
    case 32: return launch_dkdv_reduce<32>(a, stream);
    case 64: return launch_dkdv_reduce<64>(a, stream);
    case 80: return launch_dkdv_reduce<80>(a, stream);
    default: return launch_dkdv_reduce<128>(a, stream);
  }
}

cudaError_t launch_bwd_dkdv_dq(const BwdArgs& a, cudaStream_t stream) {
  if (!a.dq_acc || !a.dq_cnt) return cudaErrorInvalidValue;
  switch (a.d) {
    case 32: return a.causal ? launch_dkdv<32, true, true>(a, stream) : launch_dkdv<32, false, true>(a, stream);
    case 64: return a.causal ? launch_dkdv<64, true, true>(a, stream) : launch_dkdv<64, false, true>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq_finish(const BwdArgs& a, cudaStream_t stream) {
  if (!a.dq_acc) return cudaErrorInvalidValue;
  switch (a.d) {
    case 32: return launch_dq_finish<32>(a, stream);
    case 64: return launch_dq_finish<64>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return a.causal ? launch_dq<32, true>(a, stream) : launch_dq<32, false>(a, stream);
    case 64: return a.causal ? launch_dq<64, true>(a, stream) : launch_dq<64, false>(a, stream);
    case 80: return a.causal ? launch_dq<80, true>(a, stream) : launch_dq<80, false>(a, stream);
    case 128: return a.causal ? launch_dq<128, true>(a, stream) : launch_dq<128, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn

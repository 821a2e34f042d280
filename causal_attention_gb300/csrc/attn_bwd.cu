// Causal attention backward for sm_103a, three kernels, no atomics:
//
//  1. preprocess: D = rowsum(dO * O) in fp32 (Forge RESEARCH.md, section 6, "The D
//     term is free": D_i = sum_j P_ij dP_ij = dO_i . O_i) and LSE * log2(e), both
//     written to a [B*H, T_pad] workspace (padding rows: D = 0, LSE = +inf, so
//     that padded queries contribute P = 0).
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
// Roles in the two tensor-core kernels (192 threads):
//   warps 0-3  elementwise (thread = row of the CTA's own tile = TMEM lane)
//   warp  4    TMA producer
//   warp  5    TMEM allocator and MMA issuer
// Tensor memory: S or S^T [0,128), dP or dP^T [128,256), accumulators from 256.
// P^T and dS^T (bf16) are written over the first 64 columns of the S^T and dP^T
// regions and fed back to the tensor core from TMEM as the A operand.
#include "kernels.h"
#include "tile.cuh"

namespace attn {

namespace {

constexpr int kBwdThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
    const float* __restrict__ lse, float* __restrict__ ws_lse2, float* __restrict__ ws_D, int T,
    int T_pad, int BH) {
  constexpr int TPR = D / 8;           // threads per row, 16 bytes each
  constexpr int RPW = 32 / TPR;        // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  const long long total = (long long)BH * T_pad;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long base = warp_id * RPW; base < total; base += n_warps * RPW) {
    const long long row = base + lane / TPR;
    float acc = 0.f;
    int t = 0, bh = 0;
    const bool in_range = row < total;
    if (in_range) {
      bh = (int)(row / T_pad);
      t = (int)(row % T_pad);
      if (t < T) {
        const size_t off = ((size_t)bh * T + t) * D + sub * 8;
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + off));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + off));
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 fa = __bfloat1622float2(pa[i]);
          const float2 fb = __bfloat1622float2(pb[i]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
      }
    }
#pragma unroll
    for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (in_range && sub == 0) {
      const bool valid = t < T;
      ws_D[row] = valid ? acc : 0.f;
      ws_lse2[row] = valid ? lse[(size_t)bh * T + t] * kLog2e : INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------
// shared-memory plan of the two tensor-core kernels
// ---------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  using TL = Tile<D>;
  static constexpr int STAGES = (D == 128) ? 2 : (D == 64 ? 3 : 4);
  // fixed tiles (K_j, V_j for dK/dV; Q_i, dO_i for dQ)
  static constexpr int OFF_FIX = 0;
  // per stage: two tiles (+ for dK/dV, 128 fp32 LSE and 128 fp32 D)
  static constexpr int STAGE_BYTES = 2 * TL::BYTES + 1024;
  static constexpr int OFF_STAGE = OFF_FIX + 2 * TL::BYTES;
  static constexpr int OFF_BAR = OFF_STAGE + STAGES * STAGE_BYTES;
  // barriers: fix_full, st_full[S], st_empty[S], s_full, p_full, done, drain
  static constexpr int NBAR = 1 + 2 * STAGES + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // at least 116 KB so that one CTA occupies an SM: each CTA allocates all 512
  // TMEM columns, and a second resident CTA would only wait for them
  static constexpr int SMEM_RAW = OFF_MISC + 16 + 1024;
  static constexpr int SMEM_BYTES = SMEM_RAW > 116 * 1024 ? SMEM_RAW : 116 * 1024;
};

struct BwdSmem {
  uint32_t base;
  uint8_t* gbase;
  uint32_t bar0;
  int st;
  __device__ uint32_t fix_full() const { return bar0; }
  __device__ uint32_t st_full(int s) const { return bar0 + 8u * (1 + s); }
  __device__ uint32_t st_empty(int s) const { return bar0 + 8u * (1 + st + s); }
  __device__ uint32_t s_full() const { return bar0 + 8u * (1 + 2 * st); }
  __device__ uint32_t p_full() const { return bar0 + 8u * (2 + 2 * st); }
  __device__ uint32_t done() const { return bar0 + 8u * (3 + 2 * st); }
  __device__ uint32_t drain() const { return bar0 + 8u * (4 + 2 * st); }
};

template <int D>
__device__ __forceinline__ BwdSmem bwd_smem_setup(uint8_t* smem_raw, uint32_t*& tmem_slot,
                                                  volatile int*& abort) {
  using C = BwdCfg<D>;
  BwdSmem s;
  const uint32_t raw = smem_u32(smem_raw);
  s.base = (raw + 1023u) & ~1023u;
  s.gbase = smem_raw + (s.base - raw);
  s.bar0 = s.base + C::OFF_BAR;
  s.st = C::STAGES;
  tmem_slot = reinterpret_cast<uint32_t*>(s.gbase + C::OFF_MISC);
  abort = reinterpret_cast<volatile int*>(s.gbase + C::OFF_MISC + 4);
  if (threadIdx.x == 0) {
    mbar_init(s.fix_full(), 1);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(s.st_full(i), 1);
      mbar_init(s.st_empty(i), 1);
    }
    mbar_init(s.s_full(), 1);
    mbar_init(s.p_full(), 128);
    mbar_init(s.done(), 1);
    mbar_init(s.drain(), 1);
    *abort = 0;
    fence_barrier_init();
  }
  if ((threadIdx.x >> 5) == 5) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return s;
}

// Converts 32 fp32 accumulator columns to bf16 (times `mul`) and stores them.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&u)[32], float mul) {
  uint4 pk[4];
  uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pw[i] = pack_bf16(__uint_as_float(u[2 * i]) * mul, __uint_as_float(u[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = pk[i];
}

// ---------------------------------------------------------------------------
// 2. dK / dV
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const float* __restrict__ ws_lse2, const float* __restrict__ ws_D,
                         __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int T,
                         int T_pad, int BH, float scale, float scale_log2, uint32_t* __restrict__ err) {
  using C = BwdCfg<D>;
  using TL = Tile<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint32_t* tmem_slot;
  volatile int* abort;
  const BwdSmem sm = bwd_smem_setup<D>(smem_raw, tmem_slot, abort);
  const Abort ab{abort, err};
  const uint32_t tmem = *tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_q = (T + kTileRows - 1) / kTileRows;
  const int kt = (int)(blockIdx.x / BH);  // key tile: small j = most work, launched first
  const int bh = (int)(blockIdx.x % BH);
  const int i0 = CAUSAL ? kt : 0;
  const int n_it = n_q - i0;

  const uint32_t sK = sm.base + C::OFF_FIX, sV = sK + TL::BYTES;
  auto sQ = [&](int s) { return sm.base + C::OFF_STAGE + s * C::STAGE_BYTES; };
  auto sdO = [&](int s) { return sQ(s) + TL::BYTES; };
  auto sL = [&](int s) { return sQ(s) + 2 * TL::BYTES; };  // 128 fp32 LSE*log2e, then 128 fp32 D

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(sm.fix_full(), 2 * TL::BYTES);
      TL::load(sK, &tmK, kt * kTileRows, bh, sm.fix_full());
      TL::load(sV, &tmV, kt * kTileRows, bh, sm.fix_full());
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % ST, n = it / ST, qi = i0 + it;
        if (it >= ST && !(ok = mbar_wait(sm.st_empty(s), (n - 1) & 1, ab, kErrTimeoutLoad))) break;
        mbar_arrive_expect_tx(sm.st_full(s), 2 * TL::BYTES + 1024);
        TL::load(sQ(s), &tmQ, qi * kTileRows, bh, sm.st_full(s));
        TL::load(sdO(s), &tmdO, qi * kTileRows, bh, sm.st_full(s));
        const size_t woff = (size_t)bh * T_pad + (size_t)qi * kTileRows;
        bulk_load(sL(s), ws_lse2 + woff, 512, sm.st_full(s));
        bulk_load(sL(s) + 512, ws_D + woff, 512, sm.st_full(s));
        issued = it + 1;
      }
      if (!ok) {
        mbar_wait_drain(sm.fix_full(), 0, ab);
        for (int it = max(0, issued - ST); it < issued; ++it)
          mbar_wait_drain(sm.st_full(it % ST), (it / ST) & 1, ab);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, 0, 1);
      const uint32_t tS = tmem, tDP = tmem + 128u, tDV = tmem + 256u, tDK = tmem + 256u + (uint32_t)D;
      bool ok = mbar_wait(sm.fix_full(), 0, ab, kErrTimeoutMma);
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it % ST, n = it / ST;
        if (!(ok = mbar_wait(sm.st_full(s), n & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T (M = keys, N = queries, K = d)
#pragma unroll
        for (int k = 0; k < TL::KSTEPS_D; ++k)
          mma_ss(tS, TL::desc_kmajor(sK, k), TL::desc_kmajor(sQ(s), k), idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < TL::KSTEPS_D; ++k)
          mma_ss(tDP, TL::desc_kmajor(sV, k), TL::desc_kmajor(sdO(s), k), idesc_s, k > 0 ? 1u : 0u);
        mma_commit(sm.s_full());
        if (!(ok = mbar_wait(sm.p_full(), it & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        // dV += P^T dO_i, dK += dS^T Q_i (M = keys, N = d, K = queries)
#pragma unroll
        for (int k = 0; k < kTileRows / 16; ++k)
          mma_ts(tDV, tS + 8u * k, TL::desc_mnmajor(sdO(s), k), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < kTileRows / 16; ++k)
          mma_ts(tDK, tDP + 8u * k, TL::desc_mnmajor(sQ(s), k), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(sm.st_empty(s));
      }
      if (ok) {
        mma_commit(sm.done());
      } else {
        mma_commit(sm.drain());
        mbar_wait_drain(sm.drain(), 0, ab);
      }
    }
  } else {
    // elementwise: thread r owns key row kt*128 + r
    const int r = threadIdx.x;
    const uint32_t lo = warp_lane_base();
    const uint32_t tS = tmem + lo, tDP = tmem + lo + 128u;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % ST, n = it / ST, qi = i0 + it;
      if (!(ok = mbar_wait_warp(sm.s_full(), it & 1, ab, kErrTimeoutElem))) break;
      if (!(ok = mbar_wait_warp(sm.st_full(s), n & 1, ab, kErrTimeoutElem))) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(sm.gbase + (sL(s) - sm.base));
      const float* dd = lse2 + 128;
      const bool diag = CAUSAL && qi == kt;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t us[32], ud[32];
        tmem_ld32(tS + 32u * cb, us);
        tmem_ld32(tDP + 32u * cb, ud);
        tmem_wait_ld();
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float p[2], g[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 32 * cb + 2 * i + h;  // query column
            float pv = ex2(fmaf(__uint_as_float(us[2 * i + h]), scale_log2, -lse2[c]));
            if (diag && c < r) pv = 0.f;
            p[h] = pv;
            g[h] = pv * (__uint_as_float(ud[2 * i + h]) - dd[c]);
          }
          pp[i] = pack_bf16(p[0], p[1]);
          pd[i] = pack_bf16(g[0], g[1]);
        }
        tmem_st16(tS + 16u * cb, pp);
        tmem_st16(tDP + 16u * cb, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sm.p_full());
    }
    if (ok && mbar_wait_warp(sm.done(), 0, ab, kErrTimeoutElem)) {
      tc_fence_after();
      const int key = kt * kTileRows + r;
      const uint32_t tDV = tmem + lo + 256u, tDK = tmem + lo + 256u + (uint32_t)D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t u[32];
        tmem_ld32(tDV + 32u * cb, u);
        tmem_wait_ld();
        if (key < T) store_row32(dv + ((size_t)bh * T + key) * D + 32 * cb, u, 1.f);
        tmem_ld32(tDK + 32u * cb, u);
        tmem_wait_ld();
        if (key < T) store_row32(dk + ((size_t)bh * T + key) * D + 32 * cb, u, scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const float* __restrict__ ws_lse2, const float* __restrict__ ws_D,
                       __nv_bfloat16* __restrict__ dq, int T, int T_pad, int BH, float scale,
                       float scale_log2, uint32_t* __restrict__ err) {
  using C = BwdCfg<D>;
  using TL = Tile<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint32_t* tmem_slot;
  volatile int* abort;
  const BwdSmem sm = bwd_smem_setup<D>(smem_raw, tmem_slot, abort);
  const Abort ab{abort, err};
  const uint32_t tmem = *tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_k = (T + kTileRows - 1) / kTileRows;
  const int qt = n_k - 1 - (int)(blockIdx.x / BH);  // largest query tile (most work) first
  const int bh = (int)(blockIdx.x % BH);
  const int n_it = CAUSAL ? qt + 1 : n_k;

  const uint32_t sQ = sm.base + C::OFF_FIX, sdO = sQ + TL::BYTES;
  auto sK = [&](int s) { return sm.base + C::OFF_STAGE + s * C::STAGE_BYTES; };
  auto sV = [&](int s) { return sK(s) + TL::BYTES; };

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(sm.fix_full(), 2 * TL::BYTES);
      TL::load(sQ, &tmQ, qt * kTileRows, bh, sm.fix_full());
      TL::load(sdO, &tmdO, qt * kTileRows, bh, sm.fix_full());
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % ST, n = it / ST;
        if (it >= ST && !(ok = mbar_wait(sm.st_empty(s), (n - 1) & 1, ab, kErrTimeoutLoad))) break;
        mbar_arrive_expect_tx(sm.st_full(s), 2 * TL::BYTES);
        TL::load(sK(s), &tmK, it * kTileRows, bh, sm.st_full(s));
        TL::load(sV(s), &tmV, it * kTileRows, bh, sm.st_full(s));
        issued = it + 1;
      }
      if (!ok) {
        mbar_wait_drain(sm.fix_full(), 0, ab);
        for (int it = max(0, issued - ST); it < issued; ++it)
          mbar_wait_drain(sm.st_full(it % ST), (it / ST) & 1, ab);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_acc = idesc_bf16(128, D, 0, 1);
      const uint32_t tS = tmem, tDP = tmem + 128u, tDQ = tmem + 256u;
      bool ok = mbar_wait(sm.fix_full(), 0, ab, kErrTimeoutMma);
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it % ST, n = it / ST;
        if (!(ok = mbar_wait(sm.st_full(s), n & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        // S = Q_i K_j^T and dP = dO_i V_j^T (M = queries, N = keys, K = d)
#pragma unroll
        for (int k = 0; k < TL::KSTEPS_D; ++k)
          mma_ss(tS, TL::desc_kmajor(sQ, k), TL::desc_kmajor(sK(s), k), idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < TL::KSTEPS_D; ++k)
          mma_ss(tDP, TL::desc_kmajor(sdO, k), TL::desc_kmajor(sV(s), k), idesc_s, k > 0 ? 1u : 0u);
        mma_commit(sm.s_full());
        if (!(ok = mbar_wait(sm.p_full(), it & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        // dQ += dS K_j (M = queries, N = d, K = keys)
#pragma unroll
        for (int k = 0; k < kTileRows / 16; ++k)
          mma_ts(tDQ, tDP + 8u * k, TL::desc_mnmajor(sK(s), k), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(sm.st_empty(s));
      }
      if (ok) {
        mma_commit(sm.done());
      } else {
        mma_commit(sm.drain());
        mbar_wait_drain(sm.drain(), 0, ab);
      }
    }
  } else {
    // elementwise: thread r owns query row qt*128 + r
    const int r = threadIdx.x;
    const int row = qt * kTileRows + r;
    const uint32_t lo = warp_lane_base();
    const uint32_t tS = tmem + lo, tDP = tmem + lo + 128u;
    const float lse2 = ws_lse2[(size_t)bh * T_pad + row];
    const float Dr = ws_D[(size_t)bh * T_pad + row];
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      if (!(ok = mbar_wait_warp(sm.s_full(), it & 1, ab, kErrTimeoutElem))) break;
      tc_fence_after();
      const bool diag = CAUSAL && it == qt;
      const int key_lim = T - it * kTileRows;  // keys at column >= key_lim are padding
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t us[32], ud[32];
        tmem_ld32(tS + 32u * cb, us);
        tmem_ld32(tDP + 32u * cb, ud);
        tmem_wait_ld();
        uint32_t pd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float g[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 32 * cb + 2 * i + h;  // key column
            float pv = ex2(fmaf(__uint_as_float(us[2 * i + h]), scale_log2, -lse2));
            if (diag && c > r) pv = 0.f;
            if (!CAUSAL && c >= key_lim) pv = 0.f;
            g[h] = pv * (__uint_as_float(ud[2 * i + h]) - Dr);
          }
          pd[i] = pack_bf16(g[0], g[1]);
        }
        tmem_st16(tDP + 16u * cb, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sm.p_full());
    }
    if (ok && mbar_wait_warp(sm.done(), 0, ab, kErrTimeoutElem)) {
      tc_fence_after();
      const uint32_t tDQ = tmem + lo + 256u;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t u[32];
        tmem_ld32(tDQ + 32u * cb, u);
        tmem_wait_ld();
        if (row < T) store_row32(dq + ((size_t)bh * T + row) * D + 32 * cb, u, scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <int D>
cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.BH * a.T_pad;
  constexpr int rows_per_block = 256 / (D / 8);
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = 152LL * 8;  // grid-stride beyond 8 blocks per SM
  if (blocks > cap) blocks = cap;
  attn_bwd_preprocess_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(a.o, a.dO, a.lse, a.ws_lse2, a.ws_D,
                                                                      a.T, a.T_pad, a.BH);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_dkdv(const BwdArgs& a, cudaStream_t stream) {
  auto kern = attn_bwd_dkdv_kernel<D, CAUSAL>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), BwdCfg<D>::SMEM_BYTES, &configured);
  if (e != cudaSuccess) return e;
  const int n_t = (a.T + kTileRows - 1) / kTileRows;
  kern<<<n_t * a.BH, kBwdThreads, BwdCfg<D>::SMEM_BYTES, stream>>>(
      *a.tmQ, *a.tmK, *a.tmV, *a.tmdO, a.ws_lse2, a.ws_D, a.dk, a.dv, a.T, a.T_pad, a.BH, a.scale,
      a.scale * kLog2e, a.err);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_dq(const BwdArgs& a, cudaStream_t stream) {
  auto kern = attn_bwd_dq_kernel<D, CAUSAL>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), BwdCfg<D>::SMEM_BYTES, &configured);
  if (e != cudaSuccess) return e;
  const int n_t = (a.T + kTileRows - 1) / kTileRows;
  kern<<<n_t * a.BH, kBwdThreads, BwdCfg<D>::SMEM_BYTES, stream>>>(
      *a.tmQ, *a.tmK, *a.tmV, *a.tmdO, a.ws_lse2, a.ws_D, a.dq, a.T, a.T_pad, a.BH, a.scale,
      a.scale * kLog2e, a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return launch_pre<32>(a, stream);
    case 64: return launch_pre<64>(a, stream);
    case 128: return launch_pre<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return a.causal ? launch_dkdv<32, true>(a, stream) : launch_dkdv<32, false>(a, stream);
    case 64: return a.causal ? launch_dkdv<64, true>(a, stream) : launch_dkdv<64, false>(a, stream);
    case 128: return a.causal ? launch_dkdv<128, true>(a, stream) : launch_dkdv<128, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return a.causal ? launch_dq<32, true>(a, stream) : launch_dq<32, false>(a, stream);
    case 64: return a.causal ? launch_dq<64, true>(a, stream) : launch_dq<64, false>(a, stream);
    case 128: return a.causal ? launch_dq<128, true>(a, stream) : launch_dq<128, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn

// Fused causal attention forward for sm_103a: tcgen05 MMAs into tensor memory,
// TMA-staged K/V ring, warp-specialised roles, online softmax with exp2.
//
// Computes, per (batch, head) and query row i (Forge RESEARCH.md, section 6
// "Fused attention design (flash-style)"):
//   S = Q K^T * scale, causal mask (key j visible iff j <= i), online softmax
//   m_new = max(m, rowmax S), P = exp2((S - m_new) * scale * log2 e),
//   l = l * corr + rowsum P, O = O * corr + P V, and at the end O /= l and the
//   per-row logsumexp L = m * scale + ln l (natural log).
//
// Work item = two 128-row query tiles (Q0 = tile 2t, Q1 = tile 2t+1) of one (b, h).
//   warps 0-3  softmax for Q0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for Q1
//   warp  8    TMA producer (Q per item; K_j, V_j through a STAGES-deep ring)
//   warp  9    TMEM allocator and MMA issuer (tile 0, or both tiles at d >= 80)
//   warp  10   MMA issuer of tile 1 (d <= 64)
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 and O1 from 256. P_q is
// packed bf16, read by the PV MMA straight from tensor memory (A operand in TMEM):
// at d <= 64 it has its own 64 columns (384 / 448), so S_{q,j+1} is issued as soon as
// the softmax warps have read S_{q,j} into registers and runs while they compute;
// at d = 80 and 128 (no free columns) P is written over S_q, S_{q,j+1} follows PV_{q,j}, and
// the two tiles ping-pong on the tensor core. O is normalised by the sum of the
// rounded P values (so O / l stays a convex combination of V rows whatever the
// rounding), the logsumexp by the exact fp32 sum.
// Output rescaling is conditional: the running max is only moved when it grows by
// more than 32 in exp2 units (P <= 2^32 stays far inside the fp32 and bf16 ranges, and
// the fp32 sums of at most T such values too), so most blocks skip touching O.
#include "kernels.h"
#include "tile.cuh"

namespace attn {

namespace {

constexpr int kFwdThreads = 352;
constexpr float kRescaleThreshold = 32.0f;  // log2 units

template <int D>
struct FwdCfg {
  using TL = Tile<D>;
  static constexpr int STAGES = (D > 64) ? 2 : (D == 64 ? 3 : 4);
  // P gets its own TMEM columns when they fit (d <= 64); then each query tile has its own
  // MMA issuer. At d = 80 and 128, S and O of both tiles leave no room for P: P is written
  // over S and one thread issues every MMA. Persistent either way: the next item's Q load
  // and first S MMAs overlap this item's epilogue.
  static constexpr bool SEP_P = D <= 64;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + TL::ACC_COLS;
  static constexpr uint32_t COL_P0 = SEP_P ? 384 : COL_S0, COL_P1 = SEP_P ? 448 : COL_S1;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * TL::BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * TL::BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * TL::BYTES;
  // barriers: q_full, q_empty, k_full[S], v_full[S], k_empty[S], v_empty[S], then per
  // tile: s_full, s_free, p_full, pv_done, o_final, o_free; then drain[2]
  static constexpr int NBAR = 2 + 4 * STAGES + 12 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  // tensor-memory plan: S0, S1, O0, O1 (and P0, P1 at d <= 64) inside the 512 columns
  static_assert(COL_O1 + TL::ACC_COLS <= (SEP_P ? COL_P0 : 512u), "O columns");
  static_assert(!SEP_P || COL_P1 + 64 <= 512, "P columns");
};

// Row max of 128 values: eight independent chains of 3-input max, then a short tree.
__device__ __forceinline__ float rowmax128(const float (&x)[128]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
  for (int c = 16; c < 128; c += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], x[c + 2 * k], x[c + 2 * k + 1]);
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(fmax3(m[3], m[4], m[5]), m[6], m[7]));
}

template <int D, bool CAUSAL, bool GROUPED>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse_out, int T, int BH, int G, int n_pairs, int HG, float scale,
                    float scale_log2, uint32_t* __restrict__ err) {
  using C = FwdCfg<D>;
  using TL = Tile<D>;
  constexpr int ST = C::STAGES;
  constexpr bool SEP = C::SEP_P;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + C::OFF_Q;
  const uint32_t sK = base + C::OFF_K;
  const uint32_t sV = base + C::OFF_V;
  const uint32_t bar0 = base + C::OFF_BAR;
  const uint32_t q_full = bar0, q_empty = bar0 + 8u;
  auto k_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (2 + ST + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (2 + 2 * ST + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (2 + 3 * ST + s); };
  auto s_full = [&](int q) { return bar0 + 8u * (2 + 4 * ST + 6 * q); };
  auto s_free = [&](int q) { return bar0 + 8u * (3 + 4 * ST + 6 * q); };
  auto p_full = [&](int q) { return bar0 + 8u * (4 + 4 * ST + 6 * q); };
  auto pv_done = [&](int q) { return bar0 + 8u * (5 + 4 * ST + 6 * q); };
  auto o_final = [&](int q) { return bar0 + 8u * (6 + 4 * ST + 6 * q); };
  auto o_free = [&](int q) { return bar0 + 8u * (7 + 4 * ST + 6 * q); };
  auto drain = [&](int q) { return bar0 + 8u * (14 + 4 * ST + q); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
  const Abort ab{abort, err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nkv = (T + kTileRows - 1) / kTileRows;
  // work items: a pair of query tiles of one (b, h). Item u: query tiles 2t, 2t+1 with
  // t = n_pairs - 1 - u / BH (longest first), slice u % BH; GROUPED (two groups of HG =
  // BH / 2 slices, slices_per_group): group g = u >= n_pairs HG, v = u - g n_pairs HG,
  // t = n_pairs - 1 - v / HG, slice g HG + v % HG
  const int n_group = n_pairs * HG;
  const auto sched = make_sched<GROUPED>(n_pairs * BH, n_group);
  auto pair_of = [&](int u) {
    if constexpr (GROUPED) return n_pairs - 1 - (u >= n_group ? u - n_group : u) / HG;
    else return n_pairs - 1 - u / BH;
  };
  auto slice_of = [&](int u) {
    if constexpr (GROUPED) return u >= n_group ? HG + (u - n_group) % HG : u % HG;
    else return u % BH;
  };
  auto n_blocks = [&](int u, int q) { return CAUSAL ? min(2 * pair_of(u) + q + 1, nkv) : nkv; };
  constexpr uint32_t kRelease = SEP ? 2u : 1u;  // arrivals that free a K/V stage or the Q tiles

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, kRelease);
    for (int s = 0; s < ST; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(k_empty(s), kRelease);
      mbar_init(v_empty(s), kRelease);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(s_full(q), 1);
      mbar_init(s_free(q), 128);
      mbar_init(p_full(q), 128);
      mbar_init(pv_done(q), 1);
      mbar_init(o_final(q), 1);
      mbar_init(o_free(q), 128);
      mbar_init(drain(q), 1);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_begin();  // the inputs may come from the previous kernel in the stream

  constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
  constexpr uint64_t kTileOff = TL::bytes_off(TL::BYTES);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      // K and V tiles are read by every item of their head: keep them in L2; Q once
      const uint64_t keep = l2_evict_last(), once = l2_evict_first();
      bool ok = true;
      int g = 0, r = 0, q_issued = 0, k_issued = 0, v_issued = 0;
      for (int u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int t = pair_of(u), bh = slice_of(u), nb = n_blocks(u, 1);
        if (r > 0 && !(ok = mbar_wait(q_empty, (r - 1) & 1, ab, kErrTimeoutLoad))) break;
        if (!(ok = in_bounds(t >= 0 && t < n_pairs && bh >= 0 && bh < BH, ab))) break;
        mbar_arrive_expect_tx(q_full, 2 * TL::BYTES);
        TL::load(sQ, &tmQ, 2 * t * kTileRows, bh, q_full, once);
        TL::load(sQ + TL::BYTES, &tmQ, (2 * t + 1) * kTileRows, bh, q_full, once);
        ++q_issued;
        for (int j = 0; j < nb; ++j, ++g) {
          const int s = g % ST, n = g / ST;
          if (g >= ST && !(ok = mbar_wait(k_empty(s), (n - 1) & 1, ab, kErrTimeoutLoad))) break;
          if (!(ok = in_bounds(j * kTileRows < T && bh / G < BH / G, ab))) break;
          mbar_arrive_expect_tx(k_full(s), TL::BYTES);
          // query head bh reads key/value slice bh / G (grouped key/value heads; G = 1 without)
          TL::load(sK + s * TL::BYTES, &tmK, j * kTileRows, bh / G, k_full(s), keep);
          ++k_issued;
          if (g >= ST && !(ok = mbar_wait(v_empty(s), (n - 1) & 1, ab, kErrTimeoutLoad))) break;
          mbar_arrive_expect_tx(v_full(s), TL::BYTES);
          TL::load(sV + s * TL::BYTES, &tmV, j * kTileRows, bh / G, v_full(s), keep);
          ++v_issued;
        }
      }
      if (!ok) {
        // drain: every copy issued must land before the CTA exits
        if (q_issued > 0) mbar_wait_drain(q_full, (q_issued - 1) & 1, ab);
        for (int x = max(0, k_issued - ST); x < k_issued; ++x) mbar_wait_drain(k_full(x % ST), (x / ST) & 1, ab);
        for (int x = max(0, v_issued - ST); x < v_issued; ++x) mbar_wait_drain(v_full(x % ST), (x / ST) & 1, ab);
      }
    }
  } else if (SEP && (warp == 9 || warp == 10)) {
    // ------------------------------------------------------------ MMA issuer of tile q
    // S_{q,j+1} as soon as S_{q,j} has been read out, then PV_{q,j} once P_{q,j} is in TMEM
    if (lane == 0) {
      const int q = warp - 9;
      const uint32_t tS = tmem + (q ? C::COL_S1 : C::COL_S0);
      const uint32_t tO = tmem + (q ? C::COL_O1 : C::COL_O0);
      const uint32_t tP = tmem + (q ? C::COL_P1 : C::COL_P0);
      const uint64_t dQ = TL::desc_kmajor0(sQ + q * TL::BYTES);
      const uint64_t dK0 = TL::desc_kmajor0(sK), dV0 = TL::desc_mnmajor0(sV);
      bool ok = true;
      int g = 0, gq = 0;
      auto issue_S = [&](int gb) {
        const int s = gb % ST;
        if (!(ok = mbar_wait(k_full(s), (gb / ST) & 1, ab, kErrTimeoutMma))) return;
        tc_fence_after();
        mma_chain_ss<TL, TL::KSTEPS_D>(tS, dQ, dK0 + (uint64_t)s * kTileOff, idesc_s, 0u);
        mma_commit(s_full(q));
        mma_commit(k_empty(s));
      };
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int nb = n_blocks(u, 1), nbq = n_blocks(u, q);
        if (!(ok = mbar_wait(q_full, r & 1, ab, kErrTimeoutMma))) break;
        if (gq > 0 && !(ok = mbar_wait(s_free(q), (gq - 1) & 1, ab, kErrTimeoutMma))) break;
        issue_S(g);
        if (!ok) break;
        if (nbq == 1) mma_commit(q_empty);
        for (int j = 0; j < nbq; ++j) {
          const int gj = gq + j, gb = g + j, s = gb % ST;
          if (j + 1 < nbq) {
            if (!(ok = mbar_wait(s_free(q), gj & 1, ab, kErrTimeoutMma))) break;
            issue_S(gb + 1);
            if (!ok) break;
            if (j + 2 == nbq) mma_commit(q_empty);  // the item's last S of this tile is issued
          }
          if (!(ok = mbar_wait(v_full(s), (gb / ST) & 1, ab, kErrTimeoutMma))) break;
          if (!(ok = mbar_wait(p_full(q), gj & 1, ab, kErrTimeoutMma))) break;
          // O still holds the previous item until its epilogue read it
          if (j == 0 && r > 0 && !(ok = mbar_wait(o_free(q), (r - 1) & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          mma_chain_ts<TL, false>(tO, tP, dV0 + (uint64_t)s * kTileOff, idesc_pv, j > 0 ? 1u : 0u);
          mma_commit(pv_done(q));
          mma_commit(v_empty(s));
          if (j == nbq - 1) mma_commit(o_final(q));
        }
        if (!ok) break;
        // blocks of the item this tile does not need (causal tile 0): release them too,
        // but only once they are loaded, so that the arrival counts toward this block's
        // phase of the two-arrival barrier and not toward the previous use of the stage
        for (int j = nbq; j < nb && ok; ++j) {
          const int gb = g + j, s = gb % ST;
          if (!(ok = mbar_wait(k_full(s), (gb / ST) & 1, ab, kErrTimeoutMma))) break;
          mma_commit(k_empty(s));
          if (!(ok = mbar_wait(v_full(s), (gb / ST) & 1, ab, kErrTimeoutMma))) break;
          mma_commit(v_empty(s));
        }
        if (!ok) break;
        g += nb;
        gq += nbq;
      }
      if (!ok) {
        mma_commit(drain(q));  // completes once every MMA issued so far is done
        mbar_wait_drain(drain(q), 0, ab);
      }
    }
  } else if (!SEP && warp == 9) {
    // ------------------------------------------------------------ single MMA issuer
    // P is written over S: S_{q,j+1} must follow PV_{q,j} (in-order execution); the two
    // tiles ping-pong: S0_{j+1} after PV0_j, S1_{j+1} after PV1_j.
    if (lane == 0) {
      const uint32_t tS[2] = {tmem + C::COL_S0, tmem + C::COL_S1};
      const uint32_t tO[2] = {tmem + C::COL_O0, tmem + C::COL_O1};
      const uint64_t dQ0 = TL::desc_kmajor0(sQ), dQ1 = TL::desc_kmajor0(sQ + TL::BYTES);
      const uint64_t dK0 = TL::desc_kmajor0(sK), dV0 = TL::desc_mnmajor0(sV);
      auto issue_S = [&](int q, int s) {
        mma_chain_ss<TL, TL::KSTEPS_D>(q ? tS[1] : tS[0], q ? dQ1 : dQ0, dK0 + (uint64_t)s * kTileOff, idesc_s, 0u);
      };
      auto issue_PV = [&](int q, int s, bool acc) {
        mma_chain_ts<TL, false>(q ? tO[1] : tO[0], q ? tS[1] : tS[0], dV0 + (uint64_t)s * kTileOff, idesc_pv,
                                acc ? 1u : 0u);
      };
      bool ok = true;
      int g = 0, g0 = 0, g1 = 0;
      for (int r = 0, u; ok && (u = sched.item(r)) >= 0; ++r) {
        const int nb0 = n_blocks(u, 0), nb1 = n_blocks(u, 1);
        if (!(ok = mbar_wait(q_full, r & 1, ab, kErrTimeoutMma))) break;
        if (!(ok = mbar_wait(k_full(g % ST), (g / ST) & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        issue_S(0, g % ST);
        mma_commit(s_full(0));
        issue_S(1, g % ST);
        mma_commit(s_full(1));
        mma_commit(k_empty(g % ST));
        for (int j = 0; j < nb1 && ok; ++j) {
          const int gb = g + j, s = gb % ST, n = gb / ST;
          const int sn = (gb + 1) % ST, nn = (gb + 1) / ST;
          const bool next = j + 1 < nb1;
          if (!(ok = mbar_wait(v_full(s), n & 1, ab, kErrTimeoutMma))) break;
          bool k_next = false;
          if (j < nb0) {
            if (!(ok = mbar_wait(p_full(0), (g0 + j) & 1, ab, kErrTimeoutMma))) break;
            if (j == 0 && r > 0 && !(ok = mbar_wait(o_free(0), (r - 1) & 1, ab, kErrTimeoutMma))) break;
            tc_fence_after();
            issue_PV(0, s, j > 0);
            if (j + 1 < nb0) {
              if (!(ok = mbar_wait(k_full(sn), nn & 1, ab, kErrTimeoutMma))) break;
              tc_fence_after();
              k_next = true;
              issue_S(0, sn);
              mma_commit(s_full(0));
            } else {
              mma_commit(o_final(0));
            }
          }
          if (!(ok = mbar_wait(p_full(1), (g1 + j) & 1, ab, kErrTimeoutMma))) break;
          if (j == 0 && r > 0 && !(ok = mbar_wait(o_free(1), (r - 1) & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          issue_PV(1, s, j > 0);
          mma_commit(v_empty(s));
          if (next) {
            if (!k_next) {
              if (!(ok = mbar_wait(k_full(sn), nn & 1, ab, kErrTimeoutMma))) break;
              tc_fence_after();
            }
            issue_S(1, sn);
            mma_commit(s_full(1));
            mma_commit(k_empty(sn));
          } else {
            mma_commit(o_final(1));
          }
        }
        if (!ok) break;
        mma_commit(q_empty);
        g += nb1;
        g0 += nb0;
        g1 += nb1;
      }
      if (!ok) {
        mma_commit(drain(0));
        mbar_wait_drain(drain(0), 0, ab);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int q = warp >> 2;  // 0 or 1
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = warp_lane_base();
    const uint32_t tS = tmem + lane_off + (q ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_off + (q ? C::COL_O1 : C::COL_O0);
    const uint32_t tP = tmem + lane_off + (q ? C::COL_P1 : C::COL_P0);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    bool ok = true;
    int gq = 0;
    for (int ri = 0, u; ok && (u = sched.item(ri)) >= 0; ++ri) {
      const int qt = 2 * pair_of(u) + q, bh = slice_of(u), nb = n_blocks(u, q);
      const int row = qt * kTileRows + r;
      float m = -INFINITY, l = 0.f, lr = 0.f;
      for (int j = 0; j < nb; ++j) {
        const int gj = gq + j;
        if (!(ok = mbar_wait_warp(s_full(q), gj & 1, ab, kErrTimeoutElem))) break;
        tc_fence_after();
        float x[128];
        {
          uint32_t u2[128];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32(tS + 32u * cb, *reinterpret_cast<uint32_t(*)[32]>(&u2[32 * cb]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(u2[i]);
        }
        if constexpr (SEP) {
          tc_fence_before();
          mbar_arrive(s_free(q));  // S_q,j is in registers: the tensor core may overwrite it
        }
        if (CAUSAL && j == qt) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) x[c] = -INFINITY;
        }
        if (!CAUSAL && (j + 1) * kTileRows > T) {
          const int lim = T - j * kTileRows;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        const float mx = rowmax128(x);
        float corr = 1.f;
        bool need = false;
        if (j == 0) {
          m = mx;
        } else {
          const float m_new = fmaxf(m, mx);
          need = (m_new - m) * scale_log2 > kRescaleThreshold;
          if (need) {
            corr = ex2((m - m_new) * scale_log2);
            m = m_new;
          }
        }
        // P = exp2(S*scale*log2e - m*scale*log2e), rounded to bf16 for the PV MMA. The
        // LSE uses the exact row sum l; O is divided by lr, the sum of the same rounded
        // values, so that O / lr stays a convex combination of V rows.
        const uint64_t nmc = f2_pack(-m * scale_log2, -m * scale_log2);
        uint32_t pk[64];
        uint64_t se[4] = {0, 0, 0, 0};
        float sr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float a, b;
          f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), c2, nmc), a, b);
          a = ex2(a);
          b = ex2(b);
          pk[i] = pack_bf16(a, b);
          se[i & 3] = f2_add(se[i & 3], f2_pack(a, b));
          add_bf16x2_f32(pk[i], sr[2 * (i & 1)], sr[2 * (i & 1) + 1]);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(f2_add(f2_add(se[0], se[1]), f2_add(se[2], se[3])), a0, a1);
          b0 = sr[0] + sr[2];
          b1 = sr[1] + sr[3];
          l = l * corr + (a0 + a1);
          lr = lr * corr + (b0 + b1);
        }
        if constexpr (SEP) {
          // the previous PV of this tile must be complete: it reads the P columns and,
          // within an item, writes O
          if (gj > 0 && !(ok = mbar_wait_warp(pv_done(q), (gj - 1) & 1, ab, kErrTimeoutElem))) break;
          tc_fence_after();
        }
        // (single issuer: S_q,j completing implies PV_{q,j-1} completed, issued before it)
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t v[32];
            tmem_ld32(tO + 32u * cb, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
            tmem_st32(tO + 32u * cb, v);
          }
          if constexpr (D % 32 != 0) {  // d = 80: the last 16 columns
            uint32_t v[16];
            tmem_ld16(tO + (uint32_t)(D - 16), v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
            tmem_st16(tO + (uint32_t)(D - 16), v);
          }
        }
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) tmem_st16(tP + 16u * cb, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * cb]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(q));
      }
      // ---- epilogue: O / lr -> bf16, LSE; then free O for the next item
      if (!ok || !(ok = mbar_wait_warp(o_final(q), ri & 1, ab, kErrTimeoutElem))) break;
      tc_fence_after();
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      const bool row_ok = row < T && in_bounds(bh < BH && row >= 0, ab);
      __nv_bfloat16* orow = out + ((size_t)bh * T + row) * D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t v[32];
        tmem_ld32(tO + 32u * cb, v);
        tmem_wait_ld();
        uint4 pkd[4];
        uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pw[i] = pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cb);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = pkd[i];
        }
      }
      if constexpr (D % 32 != 0) {  // d = 80: the last 16 columns
        uint32_t v[16];
        tmem_ld16(tO + (uint32_t)(D - 16), v);
        tmem_wait_ld();
        uint4 pkd[2];
        uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pw[i] = pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + (D - 16));
          dst[0] = pkd[0];
          dst[1] = pkd[1];
        }
      }
      if (row_ok) lse_out[(size_t)bh * T + row] = (m * scale_log2 + __log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
      mbar_arrive(o_free(q));
      gq += nb;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool GROUPED>
cudaError_t launch_as(const FwdArgs& a, cudaStream_t stream, int n_pairs, int hg) {
  using C = FwdCfg<D>;
  auto kern = attn_fwd_kernel<D, CAUSAL, GROUPED>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, &configured);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM walks its share of the items
  const int grid = min(n_pairs * a.BH, a.num_sms);
  return launch_pdl(kern, dim3(grid), dim3(kFwdThreads), C::SMEM_BYTES, stream, *a.tmQ, *a.tmK, *a.tmV, a.o, a.lse,
                    a.T, a.BH, a.G, n_pairs, hg, a.scale, a.scale * 1.4426950408889634f, a.err);
}

template <int D, bool CAUSAL>
cudaError_t launch(const FwdArgs& a, cudaStream_t stream) {
  const int n_pairs = (a.T + 2 * kTileRows - 1) / (2 * kTileRows);
  // K and V of a slice are read by all its items: at d >= 80, when all slices' K and V
  // exceed the L2 budget, two groups of slices (grouped key/value heads: one group, their
  // key/value slices being shared across query slices)
  if constexpr (D > 64) {
    const int hg = a.G == 1 ? slices_per_group(a.BH, 2ll * n_pairs * 2 * kTileRows * D * 2) : a.BH;
    if (hg != a.BH) return launch_as<D, CAUSAL, true>(a, stream, n_pairs, hg);
  }
  return launch_as<D, CAUSAL, false>(a, stream, n_pairs, a.BH);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 32: return a.causal ? launch<32, true>(a, stream) : launch<32, false>(a, stream);
    case 64: return a.causal ? launch<64, true>(a, stream) : launch<64, false>(a, stream);
    case 80: return a.causal ? launch<80, true>(a, stream) : launch<80, false>(a, stream);
    case 128: return a.causal ? launch<128, true>(a, stream) : launch<128, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn

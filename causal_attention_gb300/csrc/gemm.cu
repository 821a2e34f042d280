// Training GEMMs of the attention block for sm_103a: C = op(A) op(B) with bf16 operands
// and fp32 accumulation in tensor memory, tcgen05 MMAs fed by a TMA ring.
//
// The three orientations a training step needs (Forge RESEARCH.md, section 5 "GEMM
// design": nt for the forward X W^T, nn for dX = dY W, tn for dW = dY^T X; the Forge
// paper's GEMM table in section "Results"), with the attention's layouts folded into the
// TMA tensor maps instead of separate copy passes: the QKV projection stores Q, K and V
// straight into their [B, H, T, d] tensors (head split), the output projection and the
// backward GEMMs read the heads straight from them (head merge), and the QKV epilogue
// can rotate q and k (RoPE, Forge RESEARCH.md section 7, model formulas) in fp32 before
// rounding to bf16.
//
// Work item: a 128 x 256 (or 128 x 192) output tile, accumulated over K-steps of 64 (one
// 128-byte swizzle atom of bf16) through a ring of 48 KB (40 KB) stages; the host picks
// the width that ends the product in fewer tile-times. Persistent: one CTA per SM loops
// over the work items.
//   warp 0      TMA producer
//   warp 1      TMEM allocator (512 columns: two accumulators of up to 256 fp32 columns)
//               and MMA issuer (M = 128, N = 256 or 192, K = 16 per instruction)
//   warps 2-5   epilogue: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 of the
//               finished accumulator, converts them, stages 32-row x 128-byte tiles in
//               shared memory and writes them with TMA stores, while the MMAs of the next
//               work item fill the other accumulator.
// Split-K (tn, the dW shape: few output tiles, K = B T long): the work items also range
// over S contiguous K ranges; each writes fp32 partial sums into its own [M, N] slice and
// a second launch adds the slices in the order s = 0, 1, ... (no atomics: every run gives
// the same bits; the split / reduce structure of RESEARCH.md section 5).
#include <climits>

#include "kernels.h"
#include "tile.cuh"

namespace attn {

namespace {

constexpr int kGM = 128, kGK = 64;
constexpr int kGemmThreads = 192;
constexpr int kGABytes = kGM * kGK * 2;  // 16 KB
constexpr int kGChunk = kGK * 128;      // one MN-major chunk: 64 elements x 64 K-rows (8 KB)
constexpr int kGEpiBytes = 32 * 128;    // one epilogue staging tile: 32 rows x 128 bytes

// Shared-memory plan of an output tile width BN (256 or 192): the 256-wide tile has a
// 4-stage ring of 48 KB stages and two staging tiles per epilogue warp; the 192-wide tile
// (chosen where it gives fewer or fuller waves) a 5-stage ring of 40 KB stages and one.
template <int BN>
struct GemmTile {
  static_assert(BN == 256 || BN == 192, "tile width");
  static constexpr int ST = BN == 256 ? 4 : 5;
  static constexpr int EPIBUF = BN == 256 ? 2 : 1;
  static constexpr int B_BYTES = BN * kGK * 2;
  static constexpr int STAGE = kGABytes + B_BYTES;
  static constexpr int OFF_EPI = ST * STAGE;
  static constexpr int OFF_BAR = OFF_EPI + 4 * EPIBUF * kGEpiBytes;
  static constexpr int NBAR = 2 * ST + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(STAGE % 1024 == 0 && (B_BYTES / 2) % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

// Which map holds feature f of a token view, and its (x, z) coordinates there.
__device__ __forceinline__ void view_coord(const TokView& v, int f, int& map, int& x, int& z) {
  map = f >= v.f2 ? 2 : (f >= v.f1 ? 1 : 0);
  const int fl = f - (map == 2 ? v.f2 : (map == 1 ? v.f1 : 0));
  x = fl % v.W;
  z = fl / v.W;
}

// K-major operand (rows of 64 K-elements = 128 swizzled bytes, 8-row groups 1024 bytes
// apart): K-step k (16 elements) starts 32 bytes further.
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return smem_desc<128>(addr, 16, 1024); }
// MN-major operand (64-element MN chunks of 64 K-rows, kGChunk bytes apart; 8 K-rows per
// 1024 bytes): K-step k starts 16 rows (2 KB) further.
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr) { return smem_desc<128>(addr, kGChunk, 1024); }
constexpr uint64_t kStepK = 32 >> 4, kStepMN = (16 * 128) >> 4;

template <int LAYOUT, bool ROPE, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool A_MN = LAYOUT == kGemmTN, B_MN = LAYOUT != kGemmNT;
  using TC = GemmTile<BN>;
  constexpr int kGN = BN, kGST = TC::ST, kGBBytes = TC::B_BYTES, kGStageBytes = TC::STAGE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + TC::OFF_BAR;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kGST + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kGST + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kGST + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * kGST + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + TC::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + TC::OFF_MISC + 4);
  const Abort ab{abort, p.err};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGST; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_begin();  // the operands may come from the previous kernel in the stream

  // work item u: K range u % splits, output tile u / splits (n tiles fastest, so that
  // neighbouring CTAs share the A rows)
  const int n_items = p.m_tiles * p.n_tiles * p.splits;
  auto item_k0 = [&](int u) { return (u % p.splits) * p.k_per_split; };
  auto item_k1 = [&](int u) { return min(item_k0(u) + p.k_per_split, p.k_iters); };
  auto item_mt = [&](int u) { return (u / p.splits) / p.n_tiles; };
  auto item_nt = [&](int u) { return (u / p.splits) % p.n_tiles; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // One thread issues every copy, so the coordinates are worked out once per work
    // item and then advanced per K-step (no divisions in the K loop).
    if (lane == 0) {
      bool ok = true;
      int g = 0;
      for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x) {
        const int mt = item_mt(u), nt = item_nt(u), k0 = item_k0(u), k1 = item_k1(u);
        // NT / NN: A's token rows (fixed) and its K features 64 k0, 64 (k0 + 1), ...
        int a_b = 0, a_t = 0, a_f = 0, a_map = 0, a_x = 0, a_z = 0;
        // TN: the token K-step (b, t0) and the MN chunks' coordinates (fixed)
        int k_b = 0, k_t = 0;
        int am[2] = {0, 0}, ax[2] = {0, 0}, az[2] = {0, 0};
        int bm[kGN / 64], bx[kGN / 64], bz[kGN / 64];
        if constexpr (!A_MN) {
          a_b = mt / p.nT;
          a_t = (mt % p.nT) * kGM;
          a_f = k0 * kGK;
          view_coord(p.va, a_f, a_map, a_x, a_z);
        } else {
          k_b = k0 / p.nT;
          k_t = (k0 % p.nT) * kGK;
#pragma unroll
          for (int j = 0; j < kGM / 64; ++j) view_coord(p.va, mt * kGM + 64 * j, am[j], ax[j], az[j]);
#pragma unroll
          for (int j = 0; j < kGN / 64; ++j) view_coord(p.vb, nt * kGN + 64 * j, bm[j], bx[j], bz[j]);
        }
        for (int i = k0; i < k1; ++i, ++g) {
          const int s = g % kGST;
          if (g >= kGST && !(ok = mbar_wait(empty(s), (g / kGST - 1) & 1, ab, kErrTimeoutLoad))) break;
          mbar_arrive_expect_tx(full(s), kGStageBytes);
          const uint32_t sA = base + s * kGStageBytes, sB = sA + kGABytes;
          if constexpr (!A_MN) {
            // 128 tokens (one sequence's row tile) x features 64i .. 64i + 63
            tma_load_4d(sA, &p.a[a_map], a_x, a_t, a_z, a_b, full(s));
            a_f += kGK;
            if (a_f == p.va.f1 || a_f == p.va.f2) {  // into the next tensor of the view
              ++a_map;
              a_x = a_z = 0;
            } else if ((a_x += kGK) >= p.va.W) {  // into the next head
              a_x = 0;
              ++a_z;
            }
          } else {
            // features 128 mt .. 128 mt + 127 (two MN chunks) x the 64 tokens of K-step i
#pragma unroll
            for (int j = 0; j < kGM / 64; ++j) tma_load_4d(sA + j * kGChunk, &p.a[am[j]], ax[j], k_t, az[j], k_b, full(s));
          }
          if constexpr (LAYOUT == kGemmNT) {
            // rows BN nt .. BN nt + BN - 1 of B [N, K] (two boxes) x K-columns 64i .. 64i + 63
            tma_load_2d(sB, &p.b[0], i * kGK, nt * kGN, full(s));
            tma_load_2d(sB + kGBBytes / 2, &p.b[0], i * kGK, nt * kGN + kGN / 2, full(s));
          } else if constexpr (LAYOUT == kGemmNN) {
            // K-rows 64i .. 64i + 63 of B [K, N] x BN / 64 MN chunks of 64 columns
#pragma unroll
            for (int j = 0; j < kGN / 64; ++j) tma_load_2d(sB + j * kGChunk, &p.b[0], nt * kGN + 64 * j, i * kGK, full(s));
          } else {
#pragma unroll
            for (int j = 0; j < kGN / 64; ++j) tma_load_4d(sB + j * kGChunk, &p.b[bm[j]], bx[j], k_t, bz[j], k_b, full(s));
            if ((k_t += kGK) >= p.nT * kGK) {  // the next sequence
              k_t = 0;
              ++k_b;
            }
          }
        }
      }
      if (!ok)  // every copy issued must land before the CTA exits
        for (int x = max(0, g - kGST); x < g; ++x) mbar_wait_drain(full(x % kGST), (x / kGST) & 1, ab);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kGM, kGN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      constexpr uint64_t stepA = A_MN ? kStepMN : kStepK, stepB = B_MN ? kStepMN : kStepK;
      constexpr uint64_t kStageOff = (uint64_t)(kGStageBytes >> 4);
      const uint64_t da0 = A_MN ? desc_mn(base) : desc_k(base);
      const uint64_t db0 = B_MN ? desc_mn(base + kGABytes) : desc_k(base + kGABytes);
      bool ok = true;
      int g = 0, r = 0;
      for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x, ++r) {
        const int b = r & 1, k0 = item_k0(u), k1 = item_k1(u);
        // the accumulator still holds item r - 2 until the epilogue has read it
        if (r >= 2 && !(ok = mbar_wait(acc_empty(b), ((r >> 1) - 1) & 1, ab, kErrTimeoutMma))) break;
        tc_fence_after();
        const uint32_t tacc = tmem + 256u * (uint32_t)b;
        for (int i = k0; i < k1; ++i, ++g) {
          const int s = g % kGST;
          if (!(ok = mbar_wait(full(s), (g / kGST) & 1, ab, kErrTimeoutMma))) break;
          tc_fence_after();
          const uint64_t da = da0 + (uint64_t)s * kStageOff, db = db0 + (uint64_t)s * kStageOff;
#pragma unroll
          for (int k = 0; k < kGK / 16; ++k)
            mma_ss(tacc, da + stepA * k, db + stepB * k, idesc, (i > k0 || k > 0) ? 1u : 0u);
          mma_commit(empty(s));
        }
        if (!ok) break;
        mma_commit(acc_full(b));
      }
      if (!ok) {
        mma_commit(drain);  // completes once every MMA issued so far is done
        mbar_wait_drain(drain, 0, ab);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int eq = warp & 3;  // the TMEM lane quarter this warp may access
    const uint32_t lane_base = (uint32_t)(eq * 32) << 16;
    const uint32_t stage0 = base + TC::OFF_EPI + (uint32_t)eq * (uint32_t)(TC::EPIBUF * kGEpiBytes);
    const uint32_t srow = (uint32_t)lane * 128u;
    int cnt = 0;  // TMA stores this warp has issued (its staging tiles are used in turn)
    bool ok = true;
    // a staging tile may be rewritten once the store that last used it has read it
    auto take_buffer = [&]() {
      if (cnt >= TC::EPIBUF) {
        if (lane == 0) bulk_wait_read<TC::EPIBUF - 1>();
        __syncwarp();
      }
      return stage0 + (uint32_t)(cnt % TC::EPIBUF) * kGEpiBytes;
    };
    int r = 0;
    for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x, ++r) {
      const int b = r & 1, mt = item_mt(u), nt = item_nt(u);
      if (!(ok = mbar_wait_warp(acc_full(b), (r >> 1) & 1, ab, kErrTimeoutElem))) break;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_base + 256u * (uint32_t)b;
      // after its last accumulator load this warp frees the accumulator, so that the MMAs of
      // work item r + 2 can start while it still converts and stores the last chunk
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(b));
      };
      if constexpr (LAYOUT != kGemmTN) {
        // bf16 tokens x features through the token view of C
        const int bi = mt / p.nT, t0 = (mt % p.nT) * kGM + 32 * eq, t = t0 + lane;
        const bool rows = t0 < p.T;
        // RoPE: the (cos, sin) entries of this row for head columns cs_x .. cs_x + 63; every
        // 64-column chunk of a head at that offset reuses them (at d = 64, all chunks)
        float4 csv[16];
        int cs_x = -1;
        const int n_chunks = min(kGN / 64, (p.N - nt * kGN + 63) / 64);  // >= 1: nt < n_tiles
#pragma unroll 1
        for (int j = 0; j < n_chunks; ++j) {
          const int f = nt * kGN + 64 * j;
          int map, x, z;
          view_coord(p.vc, f, map, x, z);
          const bool rot = ROPE && f < p.rope_features;
          if (rot && x != cs_x) {
            // pairs (x + 2i, x + 2i + 1) of a head at position t: entries x/2 + i (issued
            // before the accumulator loads, so that the two latencies overlap)
            const float4* cs4 = reinterpret_cast<const float4*>(p.rope_tab) +
                                (((size_t)min(t, p.T - 1) * p.rope_half + (x >> 1)) >> 1);
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) csv[i2] = __ldg(cs4 + i2);
            cs_x = x;
          }
          uint32_t v[64];
          tmem_ld32(tacc + 64u * j, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tacc + 64u * j + 32u, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          if (j == n_chunks - 1) release();
          if (!rows) continue;
          uint32_t pk[32];
          if (rot) {
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              const float4 cs = csv[i2];
              const float a0 = __uint_as_float(v[4 * i2]), b0 = __uint_as_float(v[4 * i2 + 1]);
              const float a1 = __uint_as_float(v[4 * i2 + 2]), b1 = __uint_as_float(v[4 * i2 + 3]);
              pk[2 * i2] = pack_bf16(a0 * cs.x - b0 * cs.y, a0 * cs.y + b0 * cs.x);
              pk[2 * i2 + 1] = pack_bf16(a1 * cs.z - b1 * cs.w, a1 * cs.w + b1 * cs.z);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
          const uint32_t buf = take_buffer();
#pragma unroll
          for (int g = 0; g < 8; ++g)
            sts128(buf + srow + (((uint32_t)g ^ (uint32_t)(lane & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2],
                   pk[4 * g + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&p.c[map], buf, x, t0, z, bi);  // rows past T are not written
            bulk_commit();
          }
          ++cnt;
        }
      } else {
        // fp32 [split][M][N] through the 3-D map of C
        const int m0 = mt * kGM + 32 * eq, sp = u % p.splits;
        const bool rows = m0 < p.M;
        const int n_chunks = min(kGN / 32, (p.N - nt * kGN + 31) / 32);  // >= 1: nt < n_tiles
#pragma unroll 1
        for (int j = 0; j < n_chunks; ++j) {
          const int n = nt * kGN + 32 * j;
          uint32_t v[32];
          tmem_ld32(tacc + 32u * j, v);
          tmem_wait_ld();
          if (j == n_chunks - 1) release();
          if (!rows) continue;
          const uint32_t buf = take_buffer();
#pragma unroll
          for (int g = 0; g < 8; ++g)
            sts128(buf + srow + (((uint32_t)g ^ (uint32_t)(lane & 7)) << 4), v[4 * g], v[4 * g + 1], v[4 * g + 2],
                   v[4 * g + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&p.c[0], buf, n, m0, sp);  // rows past M, columns past N are not written
            bulk_commit();
          }
          ++cnt;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // every store has landed before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out = sum over s of part[s] (fp32, added in split order), 4 values per thread
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4* __restrict__ part, float4* __restrict__ out,
                                                            long long mn4, int splits) {
  griddep_begin();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < mn4;
       i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[(long long)s * mn4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    out[i] = a;
  }
}

// tab[t][k] = (cos, sin) of t * 10000^(-2k/d), in fp64, rounded to fp32
__global__ void __launch_bounds__(256) rope_table_kernel(float2* __restrict__ tab, int T, int d) {
  griddep_begin();
  const int half = d / 2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)T * half;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / half), k = (int)(i % half);
    const double ang = (double)t * pow(10000.0, -2.0 * k / d);
    double s, c;
    sincos(ang, &s, &c);
    tab[i] = make_float2((float)c, (float)s);
  }
}

// dst = src with each pair (2k, 2k+1) of a row at position t rotated by sgn * t theta_k,
// for up to two [B, H_i, T, d] bf16 tensors. One thread takes one 16-byte granule (four
// pairs) of one (b, t) in a group of four heads (of the two tensors' H0 + H1): the (cos,
// sin) entries, shared by all heads at that position, are loaded once, and the four
// granules are loaded before any is stored.
__global__ void __launch_bounds__(256) rope_apply_kernel(const uint4* __restrict__ src0, uint4* __restrict__ dst0,
                                                         int H0, const uint4* __restrict__ src1,
                                                         uint4* __restrict__ dst1, int H1,
                                                         const float4* __restrict__ tab, int B, int T, int d,
                                                         float sgn) {
  constexpr int HG = 4;  // heads per thread
  griddep_begin();
  const int gpr = d / 8, half = d / 2, Ht = H0 + H1, n_hg = (Ht + HG - 1) / HG;
  const long long n = (long long)B * n_hg * T * gpr;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    // i = ((b * n_hg + hg) * T + t) * gpr + gi: consecutive threads, consecutive granules
    const int gi = (int)(i % gpr);
    long long r = i / gpr;
    const int t = (int)(r % T);
    r /= T;
    const int hg = (int)(r % n_hg), b = (int)(r / n_hg);
    const float4* cs4 = tab + (((size_t)t * half + 4 * gi) >> 1);
    const float4 c01 = __ldg(cs4), c23 = __ldg(cs4 + 1);
    const float cs[8] = {c01.x, c01.y * sgn, c01.z, c01.w * sgn, c23.x, c23.y * sgn, c23.z, c23.w * sgn};
    uint4 in[HG];
    size_t gix[HG];
#pragma unroll
    for (int u = 0; u < HG; ++u) {
      const int h = hg * HG + u;
      if (h >= Ht) continue;
      const bool first = h < H0;
      gix[u] = (((size_t)b * (first ? H0 : H1) + (first ? h : h - H0)) * T + t) * gpr + gi;
      in[u] = first ? src0[gix[u]] : src1[gix[u]];
    }
#pragma unroll
    for (int u = 0; u < HG; ++u) {
      const int h = hg * HG + u;
      if (h >= Ht) continue;
      const uint32_t w[4] = {in[u].x, in[u].y, in[u].z, in[u].w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = __uint_as_float(w[q] << 16), bb = __uint_as_float(w[q] & 0xFFFF0000u);
        const float c = cs[2 * q], sn = cs[2 * q + 1];
        o[q] = pack_bf16(a * c - bb * sn, a * sn + bb * c);
      }
      (h < H0 ? dst0 : dst1)[gix[u]] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

int grid_for(long long work, int per_block, int num_sms) {
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

template <int LAYOUT, bool ROPE, int BN>
cudaError_t launch_gemm_bn(const GemmParams& p, int num_sms, cudaStream_t stream) {
  auto kern = gemm_kernel<LAYOUT, ROPE, BN>;
  static uint32_t configured = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), GemmTile<BN>::SMEM, &configured);
  if (e != cudaSuccess) return e;
  const int n_items = p.m_tiles * p.n_tiles * p.splits;
  return launch_pdl(kern, dim3(min(n_items, num_sms)), dim3(kGemmThreads), GemmTile<BN>::SMEM, stream, p);
}

template <int LAYOUT, bool ROPE>
cudaError_t launch_gemm_t(const GemmParams& p, int num_sms, cudaStream_t stream) {
  switch (p.bn) {
    case 256: return launch_gemm_bn<LAYOUT, ROPE, 256>(p, num_sms, stream);
    case 192: return launch_gemm_bn<LAYOUT, ROPE, 192>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(int layout, const GemmParams& p, int num_sms, cudaStream_t stream) {
  if (p.m_tiles < 1 || p.n_tiles < 1 || p.k_iters < 1 || p.splits < 1) return cudaErrorInvalidValue;
  switch (layout) {
    case kGemmNT:
      return p.rope_features > 0 ? launch_gemm_t<kGemmNT, true>(p, num_sms, stream)
                                 : launch_gemm_t<kGemmNT, false>(p, num_sms, stream);
    case kGemmNN: return launch_gemm_t<kGemmNN, false>(p, num_sms, stream);
    case kGemmTN: return launch_gemm_t<kGemmTN, false>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_splitk_reduce(const float* part, float* out, long long mn, int splits, int num_sms,
                                 cudaStream_t stream) {
  const long long mn4 = mn / 4;
  return launch_pdl(splitk_reduce_kernel, dim3(grid_for(mn4, 256, num_sms)), dim3(256), 0, stream,
                    reinterpret_cast<const float4*>(part), reinterpret_cast<float4*>(out), mn4, splits);
}

cudaError_t launch_rope_table(float* tab, int T, int d, cudaStream_t stream) {
  const long long n = (long long)T * (d / 2);
  return launch_pdl(rope_table_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream,
                    reinterpret_cast<float2*>(tab), T, d);
}

cudaError_t launch_rope_apply(const __nv_bfloat16* src0, __nv_bfloat16* dst0, int H0, const __nv_bfloat16* src1,
                              __nv_bfloat16* dst1, int H1, const float* tab, int B, int T, int d, int inverse,
                              int num_sms, cudaStream_t stream) {
  const long long n = (long long)B * ((H0 + H1 + 3) / 4) * T * (d / 8);
  return launch_pdl(rope_apply_kernel, dim3(grid_for(n, 256, num_sms)), dim3(256), 0, stream,
                    reinterpret_cast<const uint4*>(src0), reinterpret_cast<uint4*>(dst0), H0,
                    reinterpret_cast<const uint4*>(src1), reinterpret_cast<uint4*>(dst1), H1,
                    reinterpret_cast<const float4*>(tab), B, T, d, inverse ? -1.f : 1.f);
}

}  // namespace attn

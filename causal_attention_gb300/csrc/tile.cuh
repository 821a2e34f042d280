// Tile geometry shared by the attention kernels.
//
// Every operand tile is 128 rows of one (batch, head) slice of a [B, H, T, d] bf16
// tensor, staged by TMA into shared memory with the hardware swizzle. A row of d
// bf16 values is split into column chunks of ROW_BYTES (128 B, or 64 B when
// d = 32); chunk c of all 128 rows is stored contiguously ([chunk][row][elems]),
// every chunk 1024-byte aligned so that the address-based swizzle of TMA and of
// tcgen05 agree. At d = 80 the second chunk holds columns 64..79 and zeros (TMA fills
// the columns past d with zeros), so the tile takes the space of a d = 128 tile; the
// MMAs read only the first 80 columns (five K-steps, or N = 80).
#pragma once
#include "ptx.cuh"

namespace attn {

constexpr int kTileRows = 128;  // rows per Q tile and per K/V tile

template <int D>
struct Tile {
  static_assert(D == 32 || D == 64 || D == 80 || D == 128, "head dim");
  static constexpr int ROW_BYTES = (D * 2 >= 128) ? 128 : D * 2;  // swizzle width
  static constexpr int CHUNK_ELEMS = ROW_BYTES / 2;                // bf16 per chunk row
  static constexpr int NCHUNK = (D + CHUNK_ELEMS - 1) / CHUNK_ELEMS;
  static constexpr int CHUNK_BYTES = kTileRows * ROW_BYTES;
  static constexpr int BYTES = NCHUNK * CHUNK_BYTES;  // shared-memory bytes (and TMA bytes) of a tile
  // TMEM columns reserved for a d-column fp32 accumulator (d rounded up to 32)
  static constexpr int ACC_COLS = (D + 31) / 32 * 32;
  static constexpr int KSTEPS_D = D / 16;  // MMA K-steps when contracting over d

  // Operand whose contraction dimension is d (K-major): Q or K as the A or B of
  // S = Q K^T, and V / dO in dP = dO V^T. K-step k covers d-columns 16k..16k+15.
  static __device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int k) {
    const int e = 16 * k;
    const uint32_t addr = base + (e / CHUNK_ELEMS) * CHUNK_BYTES + (e % CHUNK_ELEMS) * 2;
    return smem_desc<ROW_BYTES>(addr, 16, 8 * ROW_BYTES);
  }

  // Operand whose contraction dimension is the tile's rows and whose N dimension
  // is d (MN-major B): V in O += P V, dO / Q in dV += P^T dO / dK += dS^T Q, K in
  // dQ += dS K. K-step k covers rows 16k..16k+15.
  static __device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int k) {
    const uint32_t addr = base + 16 * k * ROW_BYTES;
    return smem_desc<ROW_BYTES>(addr, CHUNK_BYTES, 8 * ROW_BYTES);
  }

  // Lean forms for the MMA issue loop: the descriptor of K-step 0 is computed once per
  // tile, and K-step k adds a compile-time offset (in the 16-byte units of the start
  // address field; shared-memory addresses stay below 2^18, so the add never carries
  // out of that 14-bit field). A single thread issues every MMA of the CTA, and at
  // K = 16 per instruction its own instruction count bounds the tensor-core rate.
  static __device__ __forceinline__ uint64_t desc_kmajor0(uint32_t base) {
    return smem_desc<ROW_BYTES>(base, 16, 8 * ROW_BYTES);
  }
  static __device__ __forceinline__ uint64_t desc_mnmajor0(uint32_t base) {
    return smem_desc<ROW_BYTES>(base, CHUNK_BYTES, 8 * ROW_BYTES);
  }
  static __host__ __device__ constexpr uint64_t kmajor_off(int k) {
    return (uint64_t)(((16 * k) / CHUNK_ELEMS) * CHUNK_BYTES + ((16 * k) % CHUNK_ELEMS) * 2) >> 4;
  }
  static __host__ __device__ constexpr uint64_t mnmajor_off(int k) { return (uint64_t)(16 * k * ROW_BYTES) >> 4; }
  // descriptor offset of a tile that starts `bytes` later
  static __host__ __device__ constexpr uint64_t bytes_off(uint32_t bytes) { return bytes >> 4; }

  // Byte offset, within a tile written by TMA, of 16-byte granule g of row r in column
  // chunk c: the 128-byte swizzle XORs the granule index with r mod 8, the 64-byte one
  // (d = 32) with (r / 2) mod 4 (address bits 4-6 / 4-5 with bits 7-9 / 7-8).
  static __device__ __forceinline__ uint32_t granule_off(int r, int c, int g) {
    const uint32_t sw = ROW_BYTES == 128 ? (uint32_t)(r & 7) : (uint32_t)((r >> 1) & 3);
    return (uint32_t)c * CHUNK_BYTES + (uint32_t)r * ROW_BYTES + (((uint32_t)g ^ sw) << 4);
  }

  // Issue the TMA loads of one tile (rows row0..row0+127 of slice bh).
  static __device__ __forceinline__ void load(uint32_t dst, const CUtensorMap* m, int row0, int bh,
                                              uint32_t bar) {
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) tma_load_3d(dst + c * CHUNK_BYTES, m, c * CHUNK_ELEMS, row0, bh, bar);
  }
  // The same with an L2 cache policy (l2_evict_last / l2_evict_first).
  static __device__ __forceinline__ void load(uint32_t dst, const CUtensorMap* m, int row0, int bh,
                                              uint32_t bar, uint64_t policy) {
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c)
      tma_load_3d_hint(dst + c * CHUNK_BYTES, m, c * CHUNK_ELEMS, row0, bh, bar, policy);
  }
};

// D[tmem] (+)= A[smem] B[smem] over NK K-steps of 16, both operands K-major (contraction
// over the head dimension d). acc0: accumulate at K-step 0.
template <class TL, int NK>
__device__ __forceinline__ void mma_chain_ss(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int k = 0; k < NK; ++k) mma_ss(d, a0 + TL::kmajor_off(k), b0 + TL::kmajor_off(k), idesc, k ? 1u : acc0);
}

// D[tmem] (+)= A[tmem] B[smem] over 8 K-steps of 16 (K = 128 tile rows), B MN-major.
// The A operand's K-step k starts at TMEM column a0 + 8k, or, with QUARTERS (bf16
// K-columns written by four warpgroups into the first 16 columns of their own 32-column
// quarters of a 128-column fp32 region), at a0 + 32(k div 2) + 8(k mod 2).
template <class TL, bool QUARTERS>
__device__ __forceinline__ void mma_chain_ts(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int k = 0; k < kTileRows / 16; ++k) {
    const uint32_t col = QUARTERS ? 32u * (k >> 1) + 8u * (k & 1) : 8u * k;
    mma_ts(d, a0 + col, b0 + TL::mnmajor_off(k), idesc, k ? 1u : acc0);
  }
}

// The TMEM lane offset of this warp within its warpgroup (a warp may only access
// the 32-lane quarter numbered warp_id % 4).
__device__ __forceinline__ uint32_t warp_lane_base() {
  return (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
}

}  // namespace attn

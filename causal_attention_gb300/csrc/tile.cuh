// Tile geometry shared by the attention kernels.
//
// Every operand tile is 128 rows of one (batch, head) slice of a [B, H, T, d] bf16
// tensor, staged by TMA into shared memory with the hardware swizzle. A row of d
// bf16 values is split into column chunks of ROW_BYTES (128 B, or 64 B when
// d = 32); chunk c of all 128 rows is stored contiguously ([chunk][row][elems]),
// every chunk 1024-byte aligned so that the address-based swizzle of TMA and of
// tcgen05 agree.
#pragma once
#include "ptx.cuh"

namespace attn {

constexpr int kTileRows = 128;  // rows per Q tile and per K/V tile

template <int D>
struct Tile {
  static_assert(D == 32 || D == 64 || D == 128, "head dim");
  static constexpr int ROW_BYTES = (D * 2 >= 128) ? 128 : D * 2;  // swizzle width
  static constexpr int CHUNK_ELEMS = ROW_BYTES / 2;                // bf16 per chunk row
  static constexpr int NCHUNK = D / CHUNK_ELEMS;
  static constexpr int CHUNK_BYTES = kTileRows * ROW_BYTES;
  static constexpr int BYTES = kTileRows * D * 2;
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

  // Issue the TMA loads of one tile (rows row0..row0+127 of slice bh).
  static __device__ __forceinline__ void load(uint32_t dst, const CUtensorMap* m, int row0, int bh,
                                              uint32_t bar) {
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) tma_load_3d(dst + c * CHUNK_BYTES, m, c * CHUNK_ELEMS, row0, bh, bar);
  }
};

// The TMEM lane offset of this warp within its warpgroup (a warp may only access
// the 32-lane quarter numbered warp_id % 4).
__device__ __forceinline__ uint32_t warp_lane_base() {
  return (uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16;
}

}  // namespace attn

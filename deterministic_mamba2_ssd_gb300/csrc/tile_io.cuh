// tile_io.cuh -- element access to the 128-byte swizzled bf16 operand
// panels shared by the fused kernels: rows of 128 bytes (64 bf16), the
// 16-byte chunk j of row r stored at position j ^ (r % 8).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {

__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float *f) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// v -> bf16 hi + lo (hi = round(v), lo = round(v - hi)) as packed pairs, and
// both stored as 8 consecutive elements of row r of two 64-column panels
__device__ __forceinline__ void st8_bf16_hilo(uint8_t *panel_hi, uint8_t *panel_lo, int r, int c0,
                                              const float (&v)[8]) {
  uint4 uh, ul;
  uint32_t *ph = reinterpret_cast<uint32_t *>(&uh), *pl = reinterpret_cast<uint32_t *>(&ul);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    ph[i] = *reinterpret_cast<const uint32_t *>(&h);
    pl[i] = *reinterpret_cast<const uint32_t *>(&l);
  }
  const uint32_t off = r * 128 + (((c0 >> 3) ^ (r & 7)) << 4);
  *reinterpret_cast<uint4 *>(panel_hi + off) = uh;
  *reinterpret_cast<uint4 *>(panel_lo + off) = ul;
}

// 8 consecutive elements (one 16-byte chunk) of row r, columns c0..c0+7 (c0 % 8 == 0)
__device__ __forceinline__ void ld8_bf16(const uint8_t *panel, int r, int c0, float (&v)[8]) {
  bf16x8_to_f32(*reinterpret_cast<const uint4 *>(panel + r * 128 + (((c0 >> 3) ^ (r & 7)) << 4)), v);
}

// Row-per-lane tiles in a warp's shared staging area: 32 rows of four 16-byte
// chunks (64 bytes), chunk i of row l kept at slot i ^ ((l >> 1) & 3).  Lane l
// writes its own row; after a warp barrier lane l reads chunk (l & 3) of row
// 8 i + (l >> 2), so that the four lanes of a row hold 64 contiguous bytes of
// it and one warp-wide store covers 8 rows.  Both access patterns are free of
// shared-memory bank conflicts (each phase of 8 lanes touches 32 distinct banks).
__device__ __forceinline__ uint4 *stage_slot(uint8_t *stg, int row, int chunk) {
  return reinterpret_cast<uint4 *>(stg + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

}  // namespace ssd

namespace ssd {

// fp32 view of one packed state tile (bf16 hi then lo, each [128][64] in the
// swizzled operand layout): out[p * pitch + n] = hi + lo for p < 64, n < 128.
// The tile passes through shared memory (t: 64 rows of 129 floats) so that
// the writes run along n, 128 contiguous floats per row of p; the whole CTA
// (a multiple of 32 threads) takes part.
__device__ __forceinline__ void unpack_state_tile(const uint8_t *__restrict__ in, float *__restrict__ out,
                                                  int64_t pitch, float (*t)[129]) {
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int n = i >> 3, c0 = 8 * (i & 7);
    float hi[8], lo[8];
    ld8_bf16(in, n, c0, hi);
    ld8_bf16(in + 16384, n, c0, lo);
#pragma unroll
    for (int e = 0; e < 8; ++e) t[c0 + e][n] = hi[e] + lo[e];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int p = threadIdx.x >> 5; p < 64; p += nw)
#pragma unroll
    for (int k = 0; k < 4; ++k) out[p * pitch + lane + 32 * k] = t[p][lane + 32 * k];
}

}  // namespace ssd

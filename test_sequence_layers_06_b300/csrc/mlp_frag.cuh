// Fragment helpers of the TTT-MLP tensor-core kernels (mlp_mma.cu,
// mlp_cluster.cu): m16n8k16 operand loads from 128-byte-swizzled bf16 matrices in
// shared memory, paired products, the tanh-GELU of Hendrycks and Gimpel (2016)
// and its derivative, and bf16 stores of C tiles.
#pragma once

#include "ttt_device.cuh"

namespace ttt {
namespace mlpf {

// Byte offset of 16-byte chunk `c` of row `r` in a matrix with `rb`-byte rows,
// XOR-swizzled within each 128-byte group (conflict-free 8-row ldmatrix).
__device__ __forceinline__ uint32_t swz(int r, int c, int rb) {
  return static_cast<uint32_t>(r * rb + (((c & ~7) | ((c ^ r) & 7)) << 4));
}

// Fragment loads (m16n8k16 operands) from a bf16 matrix in shared memory.
// A operand, 16 x 16, from storage [m][k]: rows r0.., k chunks c0, c0+1.
__device__ __forceinline__ void ldA(uint32_t* a, uint32_t base, int rb, int r0, int c0, int lane) {
  const int mi = lane >> 3, mr = lane & 7;
  ldsm_x4(a, base + swz(r0 + ((mi & 1) << 3) + mr, c0 + (mi >> 1), rb));
}
// A operand of the transpose of storage [k][m]: k rows r0.., m chunks c0, c0+1.
__device__ __forceinline__ void ldAT(uint32_t* a, uint32_t base, int rb, int r0, int c0, int lane) {
  const int mi = lane >> 3, mr = lane & 7;
  ldsm_x4_t(a, base + swz(r0 + ((mi >> 1) << 3) + mr, c0 + (mi & 1), rb));
}
// B operands of two 8-wide n-tiles, from storage [n][k]: n rows r0.., k chunks c0, c0+1.
__device__ __forceinline__ void ldB(uint32_t* b, uint32_t base, int rb, int r0, int c0, int lane) {
  const int mi = lane >> 3, mr = lane & 7;
  ldsm_x4(b, base + swz(r0 + ((mi >> 1) << 3) + mr, c0 + (mi & 1), rb));
}
// B operands of two 8-wide n-tiles, from storage [k][n]: k rows r0.., n chunks c0, c0+1.
__device__ __forceinline__ void ldBT(uint32_t* b, uint32_t base, int rb, int r0, int c0, int lane) {
  const int mi = lane >> 3, mr = lane & 7;
  ldsm_x4_t(b, base + swz(r0 + ((mi & 1) << 3) + mr, c0 + (mi >> 1), rb));
}

__device__ __forceinline__ void mma2(float (*acc)[4], const uint32_t* a, const uint32_t* b4) {
  const uint32_t b0[2] = {b4[0], b4[1]}, b1[2] = {b4[2], b4[3]};
  mma_bf16_16816(acc[0], a, b0);
  mma_bf16_16816(acc[1], a, b1);
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh-GELU and its derivative.
__device__ __forceinline__ void gelu2(float u, float& g, float& gp) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float th = tanh_fast(c * (u + a * u * u * u));
  g = 0.5f * u * (1.f + th);
  gp = 0.5f * (1.f + th) + 0.5f * u * (1.f - th * th) * c * (1.f + 3.f * a * u * u);
}
__device__ __forceinline__ float gelu1(float u) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return 0.5f * u * (1.f + tanh_fast(c * (u + a * u * u * u)));
}

// Store a 16 x 16 C tile (rows r0 + g, + 8; columns 16*cb + 2tg, +1 of n-tiles
// 0 and 1) as bf16 into storage with `rb`-byte rows.
__device__ __forceinline__ void st_tile(uint8_t* base, int rb, int r0, int cb, const float (*c)[4], int lane) {
  const int g = lane >> 2, tg = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int ch = 2 * cb + nt;
    *reinterpret_cast<uint32_t*>(base + swz(r0 + g, ch, rb) + 4 * tg) = pack_bf16(c[nt][0], c[nt][1]);
    *reinterpret_cast<uint32_t*>(base + swz(r0 + g + 8, ch, rb) + 4 * tg) = pack_bf16(c[nt][2], c[nt][3]);
  }
}

}  // namespace mlpf
}  // namespace ttt

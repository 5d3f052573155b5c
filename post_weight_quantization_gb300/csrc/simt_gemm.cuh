// FFMA micro-kernel shared by the factorization updates and the lazy block update.
#pragma once

#include "common.cuh"

namespace gptq {
namespace simt {

constexpr int TILE = 128;     // output tile edge
constexpr int KC = 32;        // k chunk staged in shared memory
constexpr int THREADS = 256;

// 128 x 128 FFMA micro-kernel: each of 256 threads owns rows {ty*4 + 0..3, 64 + ty*4 + 0..3}
// and columns {tx*4 + 0..3, 64 + tx*4 + 0..3}; As[k][i], Bs[k][j] are k-major.
struct Acc {
  float v[8][8];
};

__device__ __forceinline__ void mma_chunk(const float (*As)[TILE], const float (*Bs)[TILE], int kn, int tx, int ty,
                                          Acc& acc) {
#pragma unroll 4
  for (int k = 0; k < kn; ++k) {
    const float4 a0 = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
    const float4 a1 = *reinterpret_cast<const float4*>(&As[k][64 + ty * 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
    const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][64 + tx * 4]);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc.v[i][j] = fmaf(a[i], b[j], acc.v[i][j]);
  }
}

__device__ __forceinline__ int micro_row(int t, int ty) { return (t < 4) ? ty * 4 + t : 64 + ty * 4 + (t - 4); }


__device__ __forceinline__ void zero(Acc& acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc.v[i][j] = 0.0f;
}

}  // namespace simt
}  // namespace gptq

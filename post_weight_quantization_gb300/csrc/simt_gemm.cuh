// FP32 FFMA GEMM used by the factorization and the lazy block update:
//
//     C = beta * C + alpha * A B        (per batch z, 128 x 128 output tiles)
//
// with A(i, k) and B(k, j) read from row-major storage in either of two layouts:
//   K-major   A(i, k) = A[i * lda + k]      B(k, j) = B[j * ldb + k]
//   MN-major  A(i, k) = A[k * lda + i]      B(k, j) = B[k * ldb + j]
// Options: only the lower-triangular tiles of a square C; A read as lower triangular
// (a_tri = 1: A(i, k) taken as 0 for k > i) or upper triangular (a_tri = 2: 0 for
// k < i), whatever the other triangle holds (the k range is trimmed per tile and the
// elements are masked); B lower triangular with zeros stored (B(k, j) = 0 for k < j,
// k range trimmed); batches with a smaller last batch (ragged pairs).
//
// 256 threads per 128 x 128 tile, each an 8 x 8 register micro-tile (rows and
// columns split 4 + 4 so shared-memory float4 reads are conflict free); k chunks of
// 16 are double-buffered in shared memory and prefetched into registers while the
// previous chunk is multiplied. All arithmetic is IEEE fp32 fused multiply-add.
#pragma once

#include "common.cuh"

namespace gptq {
namespace simt {

constexpr int TILE = 128;
constexpr int BK = 16;
constexpr int THREADS = 256;
constexpr int SLD = TILE + 4;   // padded shared-memory row (floats)

struct GemmArgs {
  int M, N, K;            // extents of every batch but the last
  int M_last, K_last;     // extents of the last batch
  const float* A;
  long long lda, a_bs;    // leading dimension, batch stride (elements)
  const float* B;
  long long ldb, b_bs;
  float* C;
  long long ldc, c_bs;
  float alpha, beta;
  // Optional low parts for the tensor-core GEMM (K-major, same extents as A and B):
  // A_lo = A - tf32(A) and B_lo = B - tf32(B), tf32 = the 13 low mantissa bits cleared.
  // Given both, the operands are loaded pre-split and no conversion pass runs.
  const float* A_lo;
  long long lda_lo;
  const float* B_lo;
  long long ldb_lo;
  int lower_tiles;        // C square: only tiles with J <= I (1: row by row; 2: column by column,
                          // so tile column 0 is computed in the first round)
  int a_tri;              // 1: A lower triangular, 2: A upper triangular (masked)
  int b_lower;            // B(k, j) == 0 for k < j
  int vec;                // every operand 16-byte aligned with leading dimensions % 4 == 0
  const int* skip;        // non-null and non-zero: do nothing (an earlier step failed)
  // Tensor-core GEMM only (the FFMA GEMM ignores them):
  int max_ctas;           // > 0: at most this many persistent CTAs (leave SMs to the next kernel)
  unsigned* signal;       // lower_tiles == 2: +1 per epilogue warp (8 per tile) once a tile of
                          // tile column 0 is stored, after a gpu-scope fence
  int b_final;            // B (and B_lo) were final before the kernel ahead of this GEMM in the
                          // stream started: their first loads may start before the dependency
                          // wait (needs skip == nullptr)
};

struct Acc {
  float v[8][8];
};

__device__ __forceinline__ int micro_row(int t, int ty) { return (t < 4) ? ty * 4 + t : 64 + ty * 4 + (t - 4); }

// Load a BK x TILE chunk (k in [k0, k0 + BK), r in [r0, r0 + TILE)) of one operand into
// 8 registers per thread. Element (r, k) is P[k * ld + r] (MN-major) or P[r * ld + k].
// tri: 0 none, 1 keep k <= r, 2 keep k >= r (r, k: the element's row and k index)
__device__ __forceinline__ bool tri_keep(int tri, int r, int k) {
  return tri == 0 || (tri == 1 ? k <= r : k >= r);
}

template <bool KMAJ>
__device__ __forceinline__ void load_chunk(const float* __restrict__ P, long long ld, int r0, int R, int k0, int Kend,
                                           bool vec, float (&v)[8], int tri = 0) {
  const int t = threadIdx.x;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if constexpr (!KMAJ) {
      const int kk = t / 32 + 8 * h, r = (t % 32) * 4;
      const int k = k0 + kk, rr = r0 + r;
      if (vec && k < Kend && rr + 3 < R) {
        const float4 q = *reinterpret_cast<const float4*>(P + (long long)k * ld + rr);
        v[4 * h] = q.x; v[4 * h + 1] = q.y; v[4 * h + 2] = q.z; v[4 * h + 3] = q.w;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) v[4 * h + c] = (k < Kend && rr + c < R) ? P[(long long)k * ld + rr + c] : 0.0f;
      }
      if (tri) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (!tri_keep(tri, rr + c, k)) v[4 * h + c] = 0.0f;
      }
    } else {
      const int r = t / 4 + 64 * h, kk = (t % 4) * 4;
      const int k = k0 + kk, rr = r0 + r;
      if (vec && rr < R && k + 3 < Kend) {
        const float4 q = *reinterpret_cast<const float4*>(P + (long long)rr * ld + k);
        v[4 * h] = q.x; v[4 * h + 1] = q.y; v[4 * h + 2] = q.z; v[4 * h + 3] = q.w;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) v[4 * h + c] = (rr < R && k + c < Kend) ? P[(long long)rr * ld + k + c] : 0.0f;
      }
      if (tri) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (!tri_keep(tri, rr, k + c)) v[4 * h + c] = 0.0f;
      }
    }
  }
}

template <bool KMAJ>
__device__ __forceinline__ void store_chunk(float (*S)[SLD], const float (&v)[8]) {
  const int t = threadIdx.x;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if constexpr (!KMAJ) {
      const int kk = t / 32 + 8 * h, r = (t % 32) * 4;
      *reinterpret_cast<float4*>(&S[kk][r]) = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
    } else {
      const int r = t / 4 + 64 * h, kk = (t % 4) * 4;
#pragma unroll
      for (int c = 0; c < 4; ++c) S[kk + c][r] = v[4 * h + c];
    }
  }
}

template <bool A_KMAJ, bool B_KMAJ>
__global__ void __launch_bounds__(THREADS) gemm_kernel(GemmArgs g) {
  if (g.skip && *g.skip) return;
  __shared__ __align__(16) float As[2][BK][SLD];
  __shared__ __align__(16) float Bs[2][BK][SLD];
  const int z = blockIdx.z;
  const bool last = (z == (int)gridDim.z - 1);
  const int M = last ? g.M_last : g.M;
  const int K = last ? g.K_last : g.K;
  const int N = g.N;
  int I, J;
  if (g.lower_tiles) {
    const int t = blockIdx.x;
    I = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((I + 1) * (I + 2) / 2 <= t) ++I;
    while (I * (I + 1) / 2 > t) --I;
    J = t - I * (I + 1) / 2;
  } else {
    J = blockIdx.x;
    I = blockIdx.y;
  }
  const int i0 = I * TILE, j0 = J * TILE;
  if (i0 >= M || j0 >= N) return;
  const float* __restrict__ A = g.A + (long long)z * g.a_bs;
  const float* __restrict__ B = g.B + (long long)z * g.b_bs;
  float* __restrict__ C = g.C + (long long)z * g.c_bs;
  int kbeg = 0, kend = K;
  if (g.a_tri == 1) kend = min(kend, i0 + TILE);
  if (g.a_tri == 2) kbeg = i0;
  if (g.b_lower) kbeg = max(kbeg, j0);
  const bool vec = g.vec != 0;

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  Acc acc;
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc.v[a][b] = 0.0f;

  float va[8], vb[8];
  if (kbeg < kend) {
    load_chunk<A_KMAJ>(A, g.lda, i0, M, kbeg, kend, vec, va, g.a_tri);
    load_chunk<B_KMAJ>(B, g.ldb, j0, N, kbeg, kend, vec, vb);
    store_chunk<A_KMAJ>(As[0], va);
    store_chunk<B_KMAJ>(Bs[0], vb);
  }
  __syncthreads();
  int buf = 0;
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) {
      load_chunk<A_KMAJ>(A, g.lda, i0, M, k0 + BK, kend, vec, va, g.a_tri);
      load_chunk<B_KMAJ>(B, g.ldb, j0, N, k0 + BK, kend, vec, vb);
    }
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc.v[i][j] = fmaf(a[i], b[j], acc.v[i][j]);
    }
    if (more) {
      store_chunk<A_KMAJ>(As[buf ^ 1], va);
      store_chunk<B_KMAJ>(Bs[buf ^ 1], vb);
    }
    __syncthreads();
    buf ^= 1;
  }

  const float alpha = g.alpha, beta = g.beta;
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int i = i0 + micro_row(a, ty);
    if (i >= M) continue;
    float* crow = C + (long long)i * g.ldc;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int jb = j0 + hb * 64 + tx * 4;
      if (vec && jb + 3 < N) {
        float4* p = reinterpret_cast<float4*>(crow + jb);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (beta != 0.0f) o = *p;
        o.x = fmaf(alpha, acc.v[a][4 * hb + 0], beta * o.x);
        o.y = fmaf(alpha, acc.v[a][4 * hb + 1], beta * o.y);
        o.z = fmaf(alpha, acc.v[a][4 * hb + 2], beta * o.z);
        o.w = fmaf(alpha, acc.v[a][4 * hb + 3], beta * o.w);
        *p = o;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = jb + c;
          if (j < N) {
            const float old = (beta != 0.0f) ? crow[j] : 0.0f;
            crow[j] = fmaf(alpha, acc.v[a][4 * hb + c], beta * old);
          }
        }
      }
    }
  }
}

// Host-side launcher (grid from the tile mode); `batches` >= 1.
inline gptq_status gemm(const GemmArgs& g, int batches, bool a_kmaj, bool b_kmaj, cudaStream_t s) {
  const int mt = (g.M + TILE - 1) / TILE, nt = (g.N + TILE - 1) / TILE;
  if (g.M <= 0 || g.N <= 0 || batches <= 0) return GPTQ_OK;
  dim3 grid;
  if (g.lower_tiles) grid = dim3((unsigned)(mt * (mt + 1) / 2), 1, (unsigned)batches);
  else grid = dim3((unsigned)nt, (unsigned)mt, (unsigned)batches);
  if (a_kmaj && b_kmaj) gemm_kernel<true, true><<<grid, THREADS, 0, s>>>(g);
  else if (a_kmaj) gemm_kernel<true, false><<<grid, THREADS, 0, s>>>(g);
  else if (b_kmaj) gemm_kernel<false, true><<<grid, THREADS, 0, s>>>(g);
  else gemm_kernel<false, false><<<grid, THREADS, 0, s>>>(g);
  count_launch();
  return check_launch("gemm_kernel");
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace simt

// Same operation on the tensor cores (3 x TF32, tc_gemm.cu); falls back to simt::gemm
// when TMA cannot describe an operand, or when GPTQ_FFMA_GEMM=1.
gptq_status tc_gemm(const simt::GemmArgs& g, int batches, bool a_kmaj, bool b_kmaj, cudaStream_t s);
// True when tc_gemm runs its K-major, 16-byte-aligned, single-batch calls on the tensor
// cores (the driver's tensor-map entry point resolves and GPTQ_FFMA_GEMM is not set).
bool tc_gemm_available();

}  // namespace gptq

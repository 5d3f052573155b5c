// Stage 2: damping, act-order and Hinv1, the upper Cholesky factor of H_d^-1.
//
// Damping adds lambda = percdamp * mean(diag H) to every diagonal entry ("GPTQ, Line
// by Line", question "What does percdamp (dampening) do in GPTQ?"); act-order visits
// columns by decreasing H_qq ("The GPTQ Algorithm", ActOrder). The pages obtain Hinv1
// by three factorizations ("GPTQ, Line by Line", question "Why does GPTQ use Cholesky
// factorizations instead of inverting the Hessian directly?"): Cholesky of H_d, the
// inverse from it, then the upper Cholesky factor of the inverse.
//
// This file reaches the same matrix with one Cholesky factorization and one
// triangular inverse. With J the reversal permutation and P = J H_d J = L L^T,
// H_d = (J L J)(J L J)^T with J L J upper, so H_d^-1 = (J L^-1 J)^T (J L^-1 J) and, by
// uniqueness of the Cholesky factor with positive diagonal, Hinv1 = J L^-1 J.
// Cost 2/3 d^3 instead of 4/3 d^3 flops, and one fewer factorization to lose accuracy.
//
// Kernels (fp32, FFMA; no spin-waits):
//   diag_stats      lambda and the finiteness check of diag(H)
//   perm_rank       stable descending sort of diag(H) by rank counting (act-order)
//   gather          P[a][b] = H_d[p(d-1-a)][p(d-1-b)] (lower triangle), p = act-order
//   Cholesky, 64-wide blocks, right-looking:
//     chol_panel    one launch per 64-wide panel: every CTA factors the diagonal block
//                   together with 64 rows below it, right-looking in 8-column steps in
//                   shared memory; CTA 0 writes L11, the others their rows of L21
//     tc_gemm       trailing update A22 -= L21 L21^T (lower tiles; tensor cores,
//                   3 x TF32, both operands K-major)
//   Triangular inverse X = L^-1 (natural order, inside Hinv1):
//     diag_inverse  every 64 x 64 diagonal block at once (thread c solves L x = e_c)
//     tc_gemm x 2 + a transpose per level, recursive doubling over block pairs (A, C)
//                   with X below the diagonal and Y = X^T above it:
//                   T = Y[A][A] L[C][A]^T;  X[C][A] = -X[C][C] T^T;  Y[A][C] = X[C][A]^T
//                   (T lives in P's unused strict upper triangle; both operands K-major)
//     reverse       Hinv1 = J X J in place, lower triangle cleared
// A failed pivot sets a flag in the workspace header that every later kernel checks.

#include <algorithm>
#include <climits>
#include <cmath>
#include <utility>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {
namespace factor {

constexpr int NB = 64;        // panel width

struct Header {               // at the start of the factor workspace
  float lambda;
  int nonfinite;
  int fail_pivot;             // INT_MAX when the factorization succeeded
  int d;
  int failed;                 // non-zero once a pivot failed or diag(H) is not finite
};
constexpr size_t kHeaderBytes = 256;

// ---------------------------------------------------------------------------------
__global__ void diag_stats_kernel(const float* __restrict__ H, int d, float percdamp, Header* hdr) {
  __shared__ double part[32];
  __shared__ int bad_s;
  if (threadIdx.x == 0) bad_s = 0;
  __syncthreads();
  double s = 0.0;
  int bad = 0;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float v = H[(long long)i * d + i];
    if (!isfinite(v)) bad = 1;
    s += (double)v;
  }
  if (bad) atomicOr(&bad_s, 1);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
    hdr->lambda = (float)((double)percdamp * (t / (double)d));
    hdr->nonfinite = bad_s;
    hdr->fail_pivot = INT_MAX;
    hdr->d = d;
    hdr->failed = bad_s;
  }
}

// rank_j = #{k : h_k > h_j} + #{k < j : h_k == h_j};  perm[rank_j] = j
__global__ void perm_rank_kernel(const float* __restrict__ H, int d, int* __restrict__ perm) {
  __shared__ float tile[256];
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const float hj = (j < d) ? H[(long long)j * d + j] : 0.0f;
  int rank = 0;
  for (int k0 = 0; k0 < d; k0 += 256) {
    __syncthreads();
    if (k0 + threadIdx.x < d) tile[threadIdx.x] = H[(long long)(k0 + threadIdx.x) * d + (k0 + threadIdx.x)];
    __syncthreads();
    const int kn = min(256, d - k0);
    for (int t = 0; t < kn; ++t) {
      const float hk = tile[t];
      rank += (hk > hj) || (hk == hj && (k0 + t) < j);
    }
  }
  if (j < d) perm[min(rank, d - 1)] = j;
}

// P[a][b] (b <= a) = H_d[p(d-1-a)][p(d-1-b)], read from the upper triangle of H
__global__ void gather_kernel(const float* __restrict__ H, int d, const int* __restrict__ perm,
                              const Header* __restrict__ hdr, float* __restrict__ P) {
  const int a = blockIdx.y * 8 + threadIdx.y;
  const float lam = hdr->lambda;
  if (a >= d) return;
  const int xa = perm ? perm[d - 1 - a] : d - 1 - a;
  for (int b = blockIdx.x * 32 + threadIdx.x; b <= a; b += gridDim.x * 32) {
    const int xb = perm ? perm[d - 1 - b] : d - 1 - b;
    const int lo = min(xa, xb), hi = max(xa, xb);
    float v = H[(long long)lo * d + hi];
    if (a == b) v += lam;
    P[(long long)a * d + b] = v;
  }
}

// ---------------------------------------------------------------------------------
// One Cholesky step for the 64-wide panel at k0, in one launch. Every CTA factors the
// tall panel made of the 64 x 64 diagonal block and (CTA b >= 1) rows
// [k1 + 64 (b - 1), + 64) below it, right-looking in steps of 8 columns, all in shared
// memory:
//   (a) warp 0 factors the step's 8 columns of the diagonal block (lane i holding rows
//       i and i + 32, pivots and column values broadcast by shuffles);
//   (b) 64 threads solve the same 8 columns of the rows below (x L^T = a);
//   (c) all threads subtract the step's rank-8 product from the columns to its right.
// The diagonal block's arithmetic is the same in every CTA, so every copy agrees;
// CTA 0 writes it back, the others write their rows. A ragged last block is padded
// with the identity.
constexpr int PANEL_THREADS = 256;
constexpr int PLD = NB + 1;                    // padded row of the shared tiles
constexpr int PS = 8;                          // columns per step

// 1 / sqrt(x) for x > 0: the hardware estimate refined by one Newton step
// y <- y (3 - x y^2) / 2 (about one ulp); no call, no slow path.
__device__ __forceinline__ float rsqrt_nr(float x) {
  const float y = rsqrtf(x);
  return y * fmaf(-0.5f * x * y, y, 1.5f);
}

// 1 / x for a normal x: the hardware estimate refined by one Newton step
// y <- y + y (1 - x y).
__device__ __forceinline__ float rcp_nr(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return fmaf(y, fmaf(-x, y, 1.0f), y);
}

// Step (a): columns [pc, pc + 8) of the diagonal block, rows pc..63, by one warp.
template <int... Js>
__device__ __forceinline__ void panel8(std::integer_sequence<int, Js...>, float* A, float* dinv, int pc, int lane,
                                       int& fail) {
  const int r0 = lane, r1 = lane + 32;
  float v0[PS], v1[PS];
#pragma unroll
  for (int c = 0; c < PS; ++c) {
    v0[c] = (r0 >= pc + c) ? A[r0 * PLD + pc + c] : 0.0f;
    v1[c] = (r1 >= pc + c) ? A[r1 * PLD + pc + c] : 0.0f;
  }
  const bool hi = pc >= 32;                    // warp-uniform: the step's pivots lie in rows 32..63
  auto step = [&](auto jc) {
    constexpr int jj = decltype(jc)::value;
    const int j = pc + jj;
    const float piv = __shfl_sync(0xffffffffu, hi ? v1[jj] : v0[jj], j & 31);
    if (!(piv > 0.0f && piv < INFINITY) && fail < 0) fail = j;
    const float inv = rsqrt_nr(piv);
    const float l0 = v0[jj] * inv, l1 = v1[jj] * inv;
#pragma unroll
    for (int cc = jj + 1; cc < PS; ++cc) {
      const int c = pc + cc;
      const float lc = __shfl_sync(0xffffffffu, hi ? l1 : l0, c & 31);   // L[c][j]
      v0[cc] = (r0 >= c) ? fmaf(-l0, lc, v0[cc]) : v0[cc];
      v1[cc] = (r1 >= c) ? fmaf(-l1, lc, v1[cc]) : v1[cc];
    }
    v0[jj] = (r0 == j) ? piv * inv : ((r0 > j) ? l0 : v0[jj]);
    v1[jj] = (r1 == j) ? piv * inv : ((r1 > j) ? l1 : v1[jj]);
    if (lane == 0) dinv[j] = inv;
  };
  (step(std::integral_constant<int, Js>{}), ...);
#pragma unroll
  for (int c = 0; c < PS; ++c) {
    if (r0 >= pc + c) A[r0 * PLD + pc + c] = v0[c];
    if (r1 >= pc + c) A[r1 * PLD + pc + c] = v1[c];
  }
}

__global__ void __launch_bounds__(PANEL_THREADS) chol_panel_kernel(float* __restrict__ P, int d, int k0, Header* hdr) {
  extern __shared__ float psm[];
  float* A = psm;                      // 64 x PLD: the diagonal block, then L11 (lower)
  float* Xs = A + NB * PLD;            // 64 x PLD: this CTA's rows of the panel below
  float* dinv = Xs + NB * PLD;         // 64
  int* fail_s = reinterpret_cast<int*>(dinv + NB);
  grid_dep_wait();                     // the previous trailing update
  grid_dep_launch();
  if (hdr->failed) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tx = tid & 15, ty = tid >> 4;
  const int nb = min(NB, d - k0), k1 = k0 + nb;
  const bool below = blockIdx.x > 0;
  const int rbeg = k1 + (blockIdx.x - 1) * NB;              // first panel row of this CTA
  const int nr = below ? min(NB, d - rbeg) : 0;

  // many loads in flight per thread; zeros outside the block
  load_tile<PANEL_THREADS, NB, NB>(A, PLD, P + (long long)k0 * d + k0, d, nb, nb);
  if (below) load_tile<PANEL_THREADS, NB, NB>(Xs, PLD, P + (long long)rbeg * d + k0, d, nr, nb);
  if (tid == 0) *fail_s = -1;
  __syncthreads();
  if (tid >= nb && tid < NB) A[tid * PLD + tid] = 1.0f;   // identity padding of a ragged block
  __syncthreads();

#pragma unroll 1
  for (int pc = 0; pc < NB; pc += PS) {
    if (warp == 0) {
      int fail = -1;
      panel8(std::make_integer_sequence<int, PS>{}, A, dinv, pc, lane, fail);
      if (lane == 0 && fail >= 0 && fail < nb && *fail_s < 0) *fail_s = fail;
    }
    __syncthreads();
    if (*fail_s >= 0) break;
    const int q0 = pc + PS, rem = NB - q0;
    if (below && tid < NB) {
      // (b) row tid of Xs, columns [pc, pc + 8)
      float* xr = Xs + tid * PLD + pc;
      float x[PS];
#pragma unroll
      for (int c = 0; c < PS; ++c) x[c] = xr[c];
#pragma unroll
      for (int jj = 0; jj < PS; ++jj) {
        x[jj] *= dinv[pc + jj];
#pragma unroll
        for (int cc = jj + 1; cc < PS; ++cc) x[cc] = fmaf(-x[jj], A[(pc + cc) * PLD + pc + jj], x[cc]);
      }
#pragma unroll
      for (int c = 0; c < PS; ++c) xr[c] = x[c];
    }
    // (c) diagonal block: A[i][c] -= sum_k L[i][pc+k] L[c][pc+k], q0 <= c <= i
    for (int a = ty; a < rem; a += 16) {
      const int i = q0 + a;
      for (int b = tx; b <= a; b += 16) {
        const int c = q0 + b;
        float acc = A[i * PLD + c];
#pragma unroll
        for (int k = 0; k < PS; ++k) acc = fmaf(-A[i * PLD + pc + k], A[c * PLD + pc + k], acc);
        A[i * PLD + c] = acc;
      }
    }
    __syncthreads();
    if (below) {
      // (c) rows below: Xs[r][c] -= sum_k Xs[r][pc+k] L[c][pc+k], c >= q0
      for (int r = ty; r < NB; r += 16) {
        for (int b = tx; b < rem; b += 16) {
          const int c = q0 + b;
          float acc = Xs[r * PLD + c];
#pragma unroll
          for (int k = 0; k < PS; ++k) acc = fmaf(-Xs[r * PLD + pc + k], A[c * PLD + pc + k], acc);
          Xs[r * PLD + c] = acc;
        }
      }
      __syncthreads();
    }
  }
  if (*fail_s >= 0) {
    if (blockIdx.x == 0 && tid == 0) {
      atomicMin(&hdr->fail_pivot, k0 + *fail_s);
      hdr->failed = 1;
    }
    return;
  }
  if (!below) {
    for (int idx = tid; idx < NB * NB; idx += PANEL_THREADS) {
      const int i = idx >> 6, c = idx & 63;
      if (i < nb && c <= i) P[(long long)(k0 + i) * d + k0 + c] = A[i * PLD + c];
    }
  } else {
    for (int idx = tid; idx < NB * NB; idx += PANEL_THREADS) {
      const int i = idx >> 6, c = idx & 63;
      if (i < nr && c < nb) P[(long long)(rbeg + i) * d + k0 + c] = Xs[i * PLD + c];
    }
  }
}
constexpr size_t PANEL_SMEM = (size_t)(2 * NB * PLD + NB + 4) * sizeof(float);

// Inverse of every 64 x 64 diagonal block of L, written into X's diagonal blocks
// (X = L^-1 in natural order). Thread c solves L x = e_c (column c of the inverse).
template <int... Js>
__device__ __forceinline__ void inv_column(std::integer_sequence<int, Js...>, float (&x)[NB], const float (*L)[NB + 1],
                                           const float* invd) {
  auto step = [&](auto jc) {
    constexpr int j = decltype(jc)::value;
    x[j] *= invd[j];
#pragma unroll
    for (int q = j + 1; q < NB; ++q) x[q] = fmaf(-L[q][j], x[j], x[q]);
  };
  (step(std::integral_constant<int, Js>{}), ...);
}

__global__ void __launch_bounds__(64) diag_inverse_kernel(const float* __restrict__ P, float* __restrict__ X, int d,
                                                          const Header* hdr) {
  __shared__ float L[NB][NB + 1];
  __shared__ float invd[NB];
  if (hdr->failed) return;
  const int k0 = blockIdx.x * NB;
  const int nb = min(NB, d - k0);
  load_tile<NB, NB, NB>(&L[0][0], NB + 1, P + (long long)k0 * d + k0, d, nb, nb);
  __syncthreads();
  for (int idx = threadIdx.x; idx < NB * NB; idx += blockDim.x) {   // lower triangle; identity past the block
    const int i = idx / NB, c = idx % NB;
    if (c > i || i >= nb) L[i][c] = (i == c) ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < NB; j += blockDim.x) invd[j] = rcp_nr(L[j][j]);
  __syncthreads();
  const int c = threadIdx.x;
  float x[NB];
#pragma unroll
  for (int q = 0; q < NB; ++q) x[q] = (q == c) ? 1.0f : 0.0f;
  inv_column(std::make_integer_sequence<int, NB>{}, x, L, invd);
  if (c >= nb) return;
#pragma unroll
  for (int q = 0; q < NB; ++q) {
    if (q < nb && q >= c) X[(long long)(k0 + q) * d + k0 + c] = x[q];
    if (q < nb && q > c) X[(long long)(k0 + c) * d + k0 + q] = x[q];   // the transpose, above
  }
}

__global__ void zero_kernel(float* __restrict__ M, long long n) {
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n; idx += (long long)gridDim.x * blockDim.x)
    M[idx] = 0.0f;
}

// In place: M[a][b] <-> M[d-1-a][d-1-b], then the strict lower triangle cleared: turns
// X = L^-1 (lower, with its transpose stored above) into J X J (upper, lower zero).
__global__ void reverse_kernel(float* __restrict__ M, int d, const Header* hdr) {
  if (hdr->failed) return;
  const long long n = (long long)d * d;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n / 2;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long jdx = n - 1 - idx;         // the partner of idx
    const long long a = idx / d, b = idx - a * d;   // idx: row a, column b; jdx: d-1-a, d-1-b
    const float t = M[idx];
    M[idx] = (a <= b) ? M[jdx] : 0.0f;
    M[jdx] = (a >= b) ? t : 0.0f;
  }
}

// Y[a0 + j][c0 + i] = X[c0 + i][a0 + j] for every pair z of the doubling step: the
// transpose of the block just computed, stored above the diagonal.
__global__ void pair_transpose_kernel(float* __restrict__ M, int d, int sz, int np, int c_last,
                                      const Header* hdr) {
  __shared__ float tile[32][33];
  if (hdr->failed) return;
  const int z = blockIdx.z;
  const int a0 = 2 * z * sz, c0 = a0 + sz;
  const int nc = (z == np - 1) ? c_last : sz;
  const int bi = blockIdx.y * 32, bj = blockIdx.x * 32;      // i over C rows, j over A columns
  if (bi >= nc) return;
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int i = bi + yy, j = bj + threadIdx.x;
    tile[yy][threadIdx.x] = (i < nc && j < sz) ? M[(long long)(c0 + i) * d + a0 + j] : 0.0f;
  }
  __syncthreads();
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int j = bj + yy, i = bi + threadIdx.x;
    if (i < nc && j < sz) M[(long long)(a0 + j) * d + c0 + i] = tile[threadIdx.x][yy];
  }
}

}  // namespace factor

size_t factor_workspace_bytes(long long d) {
  return factor::kHeaderBytes + (((size_t)d * (size_t)d * sizeof(float) + 255) & ~(size_t)255);
}

gptq_status factor_launch(const float* H, long long d_, float percdamp, int act_order, int32_t* perm_out,
                          float* Hinv1, void* ws, cudaStream_t s) {
  using namespace factor;
  const int d = (int)d_;
  Header* hdr = reinterpret_cast<Header*>(ws);
  float* P = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kHeaderBytes);
  const int* failed = &hdr->failed;
  const bool vec = (d % 4 == 0) && simt::aligned16(P) && simt::aligned16(Hinv1);

  {
  ProfScope ps_setup("factor.setup", s);
  diag_stats_kernel<<<1, 1024, 0, s>>>(H, d, percdamp, hdr);
  count_launch();
  if (act_order) {
    perm_rank_kernel<<<(d + 255) / 256, 256, 0, s>>>(H, d, perm_out);
    count_launch();
  }
  {
    dim3 grid((unsigned)std::min(64, (d + 31) / 32), (unsigned)((d + 7) / 8));
    gather_kernel<<<grid, dim3(32, 8), 0, s>>>(H, d, act_order ? perm_out : nullptr, hdr, P);
    count_launch();
  }
  }
  if (gptq_status st = check_launch("factor setup kernels")) return st;

  if (cudaFuncSetAttribute(chol_panel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PANEL_SMEM) !=
      cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(chol_panel_kernel) failed");

  // ---- Cholesky P = L L^T, 64-wide blocks, right-looking
  for (int k0 = 0; k0 < d; k0 += NB) {
    const int nb = std::min(NB, d - k0), k1 = k0 + nb, below = d - k1;
    {
      ProfScope ps("factor.chol_panel", s);
      if (launch_pdl(chol_panel_kernel, dim3(1 + (below + NB - 1) / NB), dim3(PANEL_THREADS), PANEL_SMEM, s, P, d, k0,
                     hdr) != cudaSuccess)
        return check_launch("chol_panel_kernel");
      count_launch();
    }
    if (below > 0) {
      simt::GemmArgs g{};
      g.M = g.N = below; g.K = nb; g.M_last = below; g.K_last = nb;
      g.A = P + (long long)k1 * d + k0; g.lda = d;
      g.B = g.A; g.ldb = d;
      g.C = P + (long long)k1 * d + k1; g.ldc = d;
      g.alpha = -1.0f; g.beta = 1.0f;
      g.lower_tiles = 1;
      g.vec = vec;
      g.skip = failed;
      ProfScope ps("factor.chol_update_gemm", s);
      if (gptq_status st = tc_gemm(g, 1, true, true, s)) return st;
    }
  }
  if (gptq_status st = check_launch("Cholesky kernels")) return st;

  // ---- X = L^-1 in natural order inside Hinv1: diagonal blocks, then recursive doubling
  {
    ProfScope ps("factor.zero_diag_inverse", s);
    zero_kernel<<<std::max(1, std::min(4096, (int)(((long long)d * d + 255) / 256))), 256, 0, s>>>(Hinv1, (long long)d * d);
    diag_inverse_kernel<<<(d + NB - 1) / NB, NB, 0, s>>>(P, Hinv1, d, hdr);
  }
  count_launch(2);
  // Doubling over block pairs (A, C) = ([2p sz, 2p sz + sz), [2p sz + sz, ...)): with
  // X = L^-1 kept below the diagonal of Hinv1 and Y = X^T above it (shared diagonal),
  //   T = Y[A][A] L[C][A]^T           (= (L[C][A] X[A][A])^T, into P's unused upper part)
  //   X[C][A] = -X[C][C] T^T          (= -X[C][C] L[C][A] X[A][A])
  //   Y[A][C] = X[C][A]^T
  // so every product has both operands K-major (the tensor-core GEMM's layout); the
  // triangular operands are masked, since their other triangle holds the transpose.
  for (int sz = NB; sz < d; sz *= 2) {
    int np = 0;
    while (2LL * np * sz + sz < d) ++np;
    const int c_last = std::min(sz, d - (2 * (np - 1) * sz + sz));
    const long long pair = 2LL * sz * d + 2LL * sz;
    const int nfull = (c_last == sz) ? np : np - 1;
    ProfScope ps("factor.trtri_gemms", s);
    auto g1_for = [&](int p0, int nbatch, int ncol) {
      const long long a0 = 2LL * p0 * sz, c0 = a0 + sz;
      simt::GemmArgs g1{};
      g1.M = sz; g1.N = ncol; g1.K = sz; g1.M_last = sz; g1.K_last = sz;
      g1.A = Hinv1 + a0 * d + a0; g1.lda = d; g1.a_bs = pair; g1.a_tri = 2;
      g1.B = P + c0 * d + a0; g1.ldb = d; g1.b_bs = pair;
      g1.C = P + a0 * d + c0; g1.ldc = d; g1.c_bs = pair;
      g1.alpha = 1.0f; g1.beta = 0.0f;
      g1.vec = vec;
      g1.skip = failed;
      return tc_gemm(g1, nbatch, true, true, s);
    };
    if (nfull > 0)
      if (gptq_status st = g1_for(0, nfull, sz)) return st;
    if (nfull < np)
      if (gptq_status st = g1_for(np - 1, 1, c_last)) return st;
    simt::GemmArgs g2{};
    g2.M = sz; g2.N = sz; g2.K = sz; g2.M_last = c_last; g2.K_last = c_last;
    g2.A = Hinv1 + (long long)sz * d + sz; g2.lda = d; g2.a_bs = pair; g2.a_tri = 1;
    g2.B = P + sz; g2.ldb = d; g2.b_bs = pair;
    g2.C = Hinv1 + (long long)sz * d; g2.ldc = d; g2.c_bs = pair;
    g2.alpha = -1.0f; g2.beta = 0.0f;
    g2.vec = vec;
    g2.skip = failed;
    if (gptq_status st = tc_gemm(g2, np, true, true, s)) return st;
    dim3 tg((unsigned)((sz + 31) / 32), (unsigned)((sz + 31) / 32), (unsigned)np);
    pair_transpose_kernel<<<tg, dim3(32, 8), 0, s>>>(Hinv1, d, sz, np, c_last, hdr);
    count_launch();
  }
  ProfScope ps_rev("factor.reverse", s);
  reverse_kernel<<<std::max(1, std::min(4096, (int)(((long long)d * d / 2 + 255) / 256))), 256, 0, s>>>(Hinv1, d, hdr);
  count_launch();
  return check_launch("triangular-inverse kernels");
}

gptq_status factor_read_status(const void* ws, long long* info, cudaStream_t s) {
  factor::Header h;
  if (cudaStreamSynchronize(s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaStreamSynchronize failed");
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "reading the factor status failed");
  if (h.nonfinite) {
    if (info) *info = 0;
    return set_error(GPTQ_ERR_NONFINITE, "diag(H) holds a NaN or an Inf");
  }
  if (h.fail_pivot != INT_MAX) {
    // pivot a of the reversed matrix is processing column d - 1 - a
    const int col = h.d - 1 - h.fail_pivot;
    if (info) *info = col;
    return set_error(GPTQ_ERR_NOT_PD, "the pivot of column %d is not positive", col);
  }
  if (info) *info = -1;
  return GPTQ_OK;
}

}  // namespace gptq

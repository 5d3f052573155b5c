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
//                   in shared memory (16-column pieces), CTA 0 writes it back and the
//                   others solve 64 rows each below it (x L11^T = a, four lanes per row)
//     tc_gemm       trailing update A22 -= L21 L21^T (lower tiles; tensor cores,
//                   3 x TF32, both operands K-major)
//   Triangular inverse X = L^-1 (natural order, inside Hinv1):
//     diag_inverse  every 64 x 64 diagonal block at once (thread c solves L x = e_c)
//     gemm x 2 per level, recursive doubling over block pairs (A, C):
//                   T = L[C][A] X[A][A];  X[C][A] = -X[C][C] T   (T lives in P's unused
//                   strict upper triangle)
//     reverse       Hinv1 = J X J in place
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
// Cholesky of the 64 x 64 diagonal block at k0, blocked in 4 panels of 16 columns:
//   (a) warp 0 factors the panel's 16 x 16 diagonal piece, lane i holding row i in
//       registers; column values move between lanes by shuffles;
//   (b) one thread per row below solves that row against the piece (x L^T = a);
//   (c) all threads apply the rank-16 update to the lower part right of the panel.
// Three barriers per panel.
constexpr int DP = 16;   // panel width inside the diagonal block

template <int... Js>
__device__ __forceinline__ bool panel_factor(std::integer_sequence<int, Js...>, float (&R)[DP], int lane, int np,
                                             float* dpiv, int& fail) {
  bool ok = true;
  auto step = [&](auto jc) {
    constexpr int j = decltype(jc)::value;
    if (!ok || j >= np) return;
    const float piv = __shfl_sync(0xffffffffu, R[j], j);
    if (!(piv > 0.0f) || !isfinite(piv)) {
      ok = false;
      fail = j;
      return;
    }
    const float dj = sqrtf(piv);
    const float inv = __fdiv_rn(1.0f, dj);
    const float li = (lane > j) ? R[j] * inv : 0.0f;
#pragma unroll
    for (int c = j + 1; c < DP; ++c) {
      const float lc = __shfl_sync(0xffffffffu, li, c);      // L[c][j]
      if (lane >= c) R[c] = fmaf(-li, lc, R[c]);
    }
    if (lane == j) R[j] = dj;
    else if (lane > j) R[j] = li;
    if (lane == 0) dpiv[j] = inv;
  };
  (step(std::integral_constant<int, Js>{}), ...);
  return ok;
}

// Factor the nb x nb block held in A (lower triangle) in place; returns the failing
// pivot (block-relative) or -1. All 256 threads of the CTA take part.
__device__ int factor_diag_block(float (*A)[NB + 1], float* dinv, int* fail_s, int nb) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *fail_s = -1;
  __syncthreads();
  for (int p0 = 0; p0 < nb; p0 += DP) {
    const int np = min(DP, nb - p0);
    // (a) diagonal piece
    if (warp == 0) {
      float R[DP];
#pragma unroll
      for (int c = 0; c < DP; ++c) R[c] = (lane < np && c <= lane) ? A[p0 + lane][p0 + c] : 0.0f;
      int fail = -1;
      const bool ok = panel_factor(std::make_integer_sequence<int, DP>{}, R, lane, np, dinv, fail);
      if (!ok && lane == 0) *fail_s = p0 + fail;
      if (lane < np) {
#pragma unroll
        for (int c = 0; c < DP; ++c)
          if (c <= lane) A[p0 + lane][p0 + c] = R[c];
      }
    }
    __syncthreads();
    if (*fail_s >= 0) return *fail_s;
    // (b) rows below the piece: x L^T = a
    const int r = p0 + DP + tid;
    if (tid < NB - p0 - DP && r < nb) {
      float x[DP];
#pragma unroll
      for (int c = 0; c < DP; ++c) x[c] = (c < np) ? A[r][p0 + c] : 0.0f;
#pragma unroll
      for (int j = 0; j < DP; ++j) {
        x[j] *= dinv[j];
#pragma unroll
        for (int c = j + 1; c < DP; ++c) x[c] = fmaf(-x[j], A[p0 + c][p0 + j], x[c]);
      }
#pragma unroll
      for (int c = 0; c < DP; ++c)
        if (c < np) A[r][p0 + c] = x[c];
    }
    __syncthreads();
    // (c) rank-16 update of the lower part right of the panel
    const int q0 = p0 + np, rem = nb - q0;
    for (int idx = tid; idx < rem * rem; idx += 256) {
      const int i = q0 + idx / rem, c = q0 + idx % rem;
      if (c <= i) {
        float acc = A[i][c];
#pragma unroll
        for (int k = 0; k < DP; ++k)
          if (k < np) acc = fmaf(-A[i][p0 + k], A[c][p0 + k], acc);
        A[i][c] = acc;
      }
    }
    __syncthreads();
  }
  return -1;
}

// One Cholesky step for the 64-wide panel at k0, in one launch: every CTA factors the
// diagonal block in shared memory (the same arithmetic in each, so every copy is the
// same); CTA 0 writes it back and CTA b >= 1 solves rows [k1 + 64 (b - 1), + 64) of the
// panel below against it (x L11^T = a, four lanes per row, pivots broadcast by shuffle).
constexpr int TR_LANES = 4;
constexpr int TR_SLOTS = NB / TR_LANES;        // 16
constexpr int PANEL_THREADS = 256;             // 64 rows per CTA
constexpr int TR_ROWS = PANEL_THREADS / TR_LANES;

__global__ void __launch_bounds__(PANEL_THREADS) chol_panel_kernel(float* __restrict__ P, int d, int k0, Header* hdr) {
  __shared__ float A[NB][NB + 1];
  __shared__ float dinv[DP];
  __shared__ float invd[NB];
  __shared__ int fail_s;
  if (hdr->failed) return;
  const int nb = min(NB, d - k0), k1 = k0 + nb;
  const int tid = threadIdx.x;
  load_tile<PANEL_THREADS, NB, NB>(&A[0][0], NB + 1, P + (long long)k0 * d + k0, d, nb, nb);   // upper part unused
  __syncthreads();
  const int fail = factor_diag_block(A, dinv, &fail_s, nb);
  if (fail >= 0) {
    if (blockIdx.x == 0 && tid == 0) {
      atomicMin(&hdr->fail_pivot, k0 + fail);
      hdr->failed = 1;
    }
    return;
  }
  if (blockIdx.x == 0) {
    for (int idx = tid; idx < nb * nb; idx += PANEL_THREADS) {
      const int i = idx / nb, c = idx % nb;
      if (c <= i) P[(long long)(k0 + i) * d + k0 + c] = A[i][c];
    }
    return;
  }
  for (int j = tid; j < NB; j += PANEL_THREADS) invd[j] = (j < nb) ? __fdiv_rn(1.0f, A[j][j]) : 0.0f;
  __syncthreads();
  const int lane = tid & 31, q = lane & (TR_LANES - 1), qbase = lane - q;
  const int r = k1 + (blockIdx.x - 1) * TR_ROWS + tid / TR_LANES;
  const bool active = r < d;
  float* row = P + (long long)(active ? r : k0) * d + k0;
  float x[TR_SLOTS];
#pragma unroll
  for (int k = 0; k < TR_SLOTS; ++k) {
    const int c = TR_LANES * k + q;
    x[k] = (active && c < nb) ? row[c] : 0.0f;
  }
#pragma unroll 1
  for (int jb = 0; jb < nb; jb += TR_LANES) {
#pragma unroll
    for (int i = 0; i < TR_LANES; ++i) {
      const int j = jb + i;
      if (j < nb) {                                           // warp-uniform
        const float xj = __shfl_sync(0xffffffffu, x[0], qbase + i) * invd[j];
        if (q == i && active) row[j] = xj;
        // slot k holds column jb + 4k + q: later than j unless k == 0 and q <= i
#pragma unroll
        for (int k = 0; k < TR_SLOTS; ++k) {
          const int c = jb + TR_LANES * k + q;
          if ((k > 0 || q > i) && c < NB) x[k] = fmaf(-xj, A[c][j], x[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < TR_SLOTS - 1; ++k) x[k] = x[k + 1];
    x[TR_SLOTS - 1] = 0.0f;
  }
}

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
  for (int j = threadIdx.x; j < NB; j += blockDim.x) invd[j] = __fdiv_rn(1.0f, L[j][j]);
  __syncthreads();
  const int c = threadIdx.x;
  float x[NB];
#pragma unroll
  for (int q = 0; q < NB; ++q) x[q] = (q == c) ? 1.0f : 0.0f;
  inv_column(std::make_integer_sequence<int, NB>{}, x, L, invd);
  if (c >= nb) return;
#pragma unroll
  for (int q = 0; q < NB; ++q)
    if (q < nb && q >= c) X[(long long)(k0 + q) * d + k0 + c] = x[q];
}

__global__ void zero_kernel(float* __restrict__ M, long long n) {
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n; idx += (long long)gridDim.x * blockDim.x)
    M[idx] = 0.0f;
}

// In place: M[a][b] <-> M[d-1-a][d-1-b] (turns X = L^-1, lower, into J X J, upper).
__global__ void reverse_kernel(float* __restrict__ M, int d, const Header* hdr) {
  if (hdr->failed) return;
  const long long n = (long long)d * d;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n / 2;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long jdx = n - 1 - idx;         // the partner of idx
    const float t = M[idx];
    M[idx] = M[jdx];
    M[jdx] = t;
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

  // ---- Cholesky P = L L^T, 64-wide blocks, right-looking
  for (int k0 = 0; k0 < d; k0 += NB) {
    const int nb = std::min(NB, d - k0), k1 = k0 + nb, below = d - k1;
    {
      ProfScope ps("factor.chol_panel", s);
      chol_panel_kernel<<<1 + (below + TR_ROWS - 1) / TR_ROWS, PANEL_THREADS, 0, s>>>(P, d, k0, hdr);
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
  for (int sz = NB; sz < d; sz *= 2) {
    // pairs p: A block [2p sz, 2p sz + sz) (full), C block [2p sz + sz, min(2p sz + 2sz, d))
    int np = 0;
    while (2LL * np * sz + sz < d) ++np;
    const int c_last = std::min(sz, d - (2 * (np - 1) * sz + sz));
    const long long pair = 2LL * sz * d + 2LL * sz;
    // T_p = L[C][A] X[A][A], stored in P's strict upper triangle at rows p sz, columns d - sz
    simt::GemmArgs g1{};
    g1.M = sz; g1.N = sz; g1.K = sz; g1.M_last = c_last; g1.K_last = sz;
    g1.A = P + (long long)sz * d; g1.lda = d; g1.a_bs = pair;
    g1.B = Hinv1; g1.ldb = d; g1.b_bs = pair; g1.b_lower = 1;
    g1.C = P + (d - sz); g1.ldc = d; g1.c_bs = (long long)sz * d;
    g1.alpha = 1.0f; g1.beta = 0.0f;
    g1.vec = vec;
    g1.skip = failed;
    ProfScope ps("factor.trtri_gemms", s);
    if (gptq_status st = simt::gemm(g1, np, true, false, s)) return st;
    // X[C][A] = -X[C][C] T_p
    simt::GemmArgs g2{};
    g2.M = sz; g2.N = sz; g2.K = sz; g2.M_last = c_last; g2.K_last = c_last;
    g2.A = Hinv1 + (long long)sz * d + sz; g2.lda = d; g2.a_bs = pair; g2.a_lower = 1;
    g2.B = P + (d - sz); g2.ldb = d; g2.b_bs = (long long)sz * d;
    g2.C = Hinv1 + (long long)sz * d; g2.ldc = d; g2.c_bs = pair;
    g2.alpha = -1.0f; g2.beta = 0.0f;
    g2.vec = vec;
    g2.skip = failed;
    if (gptq_status st = simt::gemm(g2, np, true, false, s)) return st;
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

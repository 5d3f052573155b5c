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
// Kernels (fp32, FFMA; all bounded, no spin-waits):
//   diag_stats   lambda and the finiteness check of diag(H)
//   perm_rank    stable descending sort of diag(H) by rank counting (act-order)
//   gather       P[a][b] = H_d[p(d-1-a)][p(d-1-b)] (lower triangle), p = act-order
//   chol_panel   factor a 64-wide diagonal block in shared memory (every CTA) and
//                solve the panel below it (L21 = A21 L11^-T), one 64-row slab per CTA
//   chol_update  trailing A22 -= L21 L21^T, 128 x 128 tiles of the lower triangle
//   eye          Hinv1 = I
//   trtri_panel  block row K of X = L^-1: X[K][:k1] = L_KK^-1 X[K][:k1]
//   trtri_update X[rows > K][:k1] -= L[rows > K][K] X[K][:k1]
// X lives directly in Hinv1 at reversed coordinates: X[a][b] is Hinv1[d-1-a][d-1-b].
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {
namespace factor {

constexpr int NB = 64;        // panel width
using simt::TILE;
using simt::KC;
constexpr int UPD_THREADS = simt::THREADS;

struct Header {               // at the start of the factor workspace
  float lambda;
  int nonfinite;
  int fail_pivot;             // INT_MAX when the factorization succeeded
  int d;
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
// Cholesky panel: every CTA factors the diagonal block (nb <= 64) in shared memory;
// CTA 0 writes it back, CTA b >= 1 solves rows [k1 + 64 (b-1), +64) of the panel.
__global__ void __launch_bounds__(256) chol_panel_kernel(float* __restrict__ P, int d, int k0, Header* hdr) {
  __shared__ float A[NB][NB + 1];
  __shared__ float R[64][NB + 1];
  __shared__ int failed;
  if (hdr->fail_pivot != INT_MAX || hdr->nonfinite) return;   // an earlier panel failed
  const int nb = min(NB, d - k0);
  const int tid = threadIdx.x;
  for (int idx = tid; idx < nb * nb; idx += blockDim.x) {
    const int i = idx / nb, l = idx % nb;
    A[i][l] = (l <= i) ? P[(long long)(k0 + i) * d + k0 + l] : 0.0f;
  }
  if (tid == 0) failed = 0;
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    if (tid == 0) {
      const float piv = A[j][j];
      if (!(piv > 0.0f) || !isfinite(piv)) {
        failed = 1;
        if (blockIdx.x == 0) atomicMin(&hdr->fail_pivot, k0 + j);
      } else {
        A[j][j] = sqrtf(piv);
      }
    }
    __syncthreads();
    if (failed) return;
    const float djj = A[j][j];
    for (int i = j + 1 + tid; i < nb; i += blockDim.x) A[i][j] = __fdiv_rn(A[i][j], djj);
    __syncthreads();
    const int rem = nb - j - 1;
    for (int idx = tid; idx < rem * rem; idx += blockDim.x) {
      const int i = j + 1 + idx / rem, l = j + 1 + idx % rem;
      if (l <= i) A[i][l] = fmaf(-A[i][j], A[l][j], A[i][l]);
    }
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int idx = tid; idx < nb * nb; idx += blockDim.x) {
      const int i = idx / nb, l = idx % nb;
      if (l <= i) P[(long long)(k0 + i) * d + k0 + l] = A[i][l];
    }
    return;
  }
  // rows of the panel below: X L11^T = A21  (forward substitution over columns)
  const int r0 = k0 + nb + (blockIdx.x - 1) * 64;
  const int nr = min(64, d - r0);
  if (nr <= 0) return;
  for (int idx = tid; idx < nr * nb; idx += blockDim.x) {
    const int i = idx / nb, l = idx % nb;
    R[i][l] = P[(long long)(r0 + i) * d + k0 + l];
  }
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    const float djj = A[j][j];
    for (int i = tid; i < nr; i += blockDim.x) R[i][j] = __fdiv_rn(R[i][j], djj);
    __syncthreads();
    const int rem = nb - j - 1;
    for (int idx = tid; idx < nr * rem; idx += blockDim.x) {
      const int i = idx / rem, l = j + 1 + idx % rem;
      R[i][l] = fmaf(-R[i][j], A[l][j], R[i][l]);
    }
    __syncthreads();
  }
  for (int idx = tid; idx < nr * nb; idx += blockDim.x) {
    const int i = idx / nb, l = idx % nb;
    P[(long long)(r0 + i) * d + k0 + l] = R[i][l];
  }
}

// ---------------------------------------------------------------------------------
// trailing update of the Cholesky: for tiles (I, J), J <= I, of rows/cols >= k1:
//   P[i][j] -= sum_{l < nb} P[i][k0 + l] * P[j][k0 + l]
__global__ void __launch_bounds__(UPD_THREADS) chol_update_kernel(float* __restrict__ P, int d, int k0, int nb,
                                                                  const Header* __restrict__ hdr) {
  __shared__ __align__(16) float As[KC][TILE];
  __shared__ __align__(16) float Bs[KC][TILE];
  if (hdr->fail_pivot != INT_MAX || hdr->nonfinite) return;
  const int k1 = k0 + nb;
  // lower-triangular tile index -> (I, J)
  const long long t = blockIdx.x;
  int I = (int)((sqrt(8.0 * (double)t + 1.0) - 1.0) * 0.5);
  while ((long long)(I + 1) * (I + 2) / 2 <= t) ++I;
  while ((long long)I * (I + 1) / 2 > t) --I;
  const int J = (int)(t - (long long)I * (I + 1) / 2);
  const int i0 = k1 + I * TILE, j0 = k1 + J * TILE;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  simt::Acc acc;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc.v[i][j] = 0.0f;
  for (int kc = 0; kc < nb; kc += KC) {
    const int kn = min(KC, nb - kc);
    __syncthreads();
    for (int idx = threadIdx.x; idx < TILE * KC; idx += UPD_THREADS) {
      const int r = idx % TILE, k = idx / TILE;
      float va = 0.0f, vb = 0.0f;
      if (k < kn) {
        if (i0 + r < d) va = P[(long long)(i0 + r) * d + k0 + kc + k];
        if (j0 + r < d) vb = P[(long long)(j0 + r) * d + k0 + kc + k];
      }
      As[k][r] = va;
      Bs[k][r] = vb;
    }
    __syncthreads();
    simt::mma_chunk(As, Bs, kn, tx, ty, acc);
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int i = i0 + simt::micro_row(a, ty);
    if (i >= d) continue;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int j = j0 + simt::micro_row(b, tx);
      if (j <= i) P[(long long)i * d + j] -= acc.v[a][b];
    }
  }
}

// ---------------------------------------------------------------------------------
__global__ void eye_kernel(float* __restrict__ M, int d) {
  const long long n = (long long)d * d;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n; idx += (long long)gridDim.x * blockDim.x)
    M[idx] = (idx / d == idx % d) ? 1.0f : 0.0f;
}

__device__ __forceinline__ long long rev_index(int a, int b, int d) {
  return (long long)(d - 1 - a) * d + (d - 1 - b);
}

// X[K][c0 : c0 + 64) = L_KK^-1 X[K][c0 : c0 + 64), K = [k0, k0 + nb), columns < k1
__global__ void __launch_bounds__(256) trtri_panel_kernel(const float* __restrict__ P, float* __restrict__ U, int d,
                                                          int k0, const Header* __restrict__ hdr) {
  __shared__ float A[NB][NB + 1];
  __shared__ float Xs[NB][64 + 1];
  if (hdr->fail_pivot != INT_MAX || hdr->nonfinite) return;
  const int nb = min(NB, d - k0);
  const int k1 = k0 + nb;
  const int c0 = blockIdx.x * 64;
  const int nc = min(64, k1 - c0);
  const int tid = threadIdx.x;
  for (int idx = tid; idx < nb * nb; idx += blockDim.x) {
    const int i = idx / nb, l = idx % nb;
    A[i][l] = (l <= i) ? P[(long long)(k0 + i) * d + k0 + l] : 0.0f;
  }
  for (int idx = tid; idx < nb * 64; idx += blockDim.x) {
    const int i = idx / 64, c = idx % 64;
    Xs[i][c] = (c < nc) ? U[rev_index(k0 + i, c0 + c, d)] : 0.0f;
  }
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    const float djj = A[j][j];
    for (int c = tid; c < 64; c += blockDim.x) Xs[j][c] = __fdiv_rn(Xs[j][c], djj);
    __syncthreads();
    const int rem = nb - j - 1;
    for (int idx = tid; idx < rem * 64; idx += blockDim.x) {
      const int i = j + 1 + idx / 64, c = idx % 64;
      Xs[i][c] = fmaf(-A[i][j], Xs[j][c], Xs[i][c]);
    }
    __syncthreads();
  }
  for (int idx = tid; idx < nb * 64; idx += blockDim.x) {
    const int i = idx / 64, c = idx % 64;
    if (c < nc && c0 + c <= k0 + i) U[rev_index(k0 + i, c0 + c, d)] = Xs[i][c];
  }
}

// X[i][j] -= sum_{l < nb} L[i][k0 + l] X[k0 + l][j] for i >= k1, j < k1
__global__ void __launch_bounds__(UPD_THREADS) trtri_update_kernel(const float* __restrict__ P, float* __restrict__ U,
                                                                   int d, int k0, int nb,
                                                                   const Header* __restrict__ hdr) {
  __shared__ __align__(16) float As[KC][TILE];
  __shared__ __align__(16) float Bs[KC][TILE];
  if (hdr->fail_pivot != INT_MAX || hdr->nonfinite) return;
  const int k1 = k0 + nb;
  const int i0 = k1 + blockIdx.y * TILE;
  const int j0 = blockIdx.x * TILE;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  simt::Acc acc;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc.v[i][j] = 0.0f;
  for (int kc = 0; kc < nb; kc += KC) {
    const int kn = min(KC, nb - kc);
    __syncthreads();
    for (int idx = threadIdx.x; idx < TILE * KC; idx += UPD_THREADS) {
      const int r = idx % TILE, k = idx / TILE;
      float va = 0.0f, vb = 0.0f;
      if (k < kn) {
        if (i0 + r < d) va = P[(long long)(i0 + r) * d + k0 + kc + k];
        if (j0 + r < k1) vb = U[rev_index(k0 + kc + k, j0 + r, d)];
      }
      As[k][r] = va;
      Bs[k][r] = vb;
    }
    __syncthreads();
    simt::mma_chunk(As, Bs, kn, tx, ty, acc);
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int i = i0 + simt::micro_row(a, ty);
    if (i >= d) continue;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int j = j0 + simt::micro_row(b, tx);
      if (j < k1) U[rev_index(i, j, d)] -= acc.v[a][b];
    }
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
  if (gptq_status st = check_launch("factor setup kernels")) return st;

  for (int k0 = 0; k0 < d; k0 += NB) {
    const int nb = std::min(NB, d - k0);
    const int below = d - k0 - nb;
    chol_panel_kernel<<<1 + (below + 63) / 64, 256, 0, s>>>(P, d, k0, hdr);
    count_launch();
    if (below > 0) {
      const long long nt = (below + TILE - 1) / TILE;
      chol_update_kernel<<<(unsigned)(nt * (nt + 1) / 2), UPD_THREADS, 0, s>>>(P, d, k0, nb, hdr);
      count_launch();
    }
  }
  if (gptq_status st = check_launch("Cholesky kernels")) return st;

  eye_kernel<<<std::max(1, std::min(4096, (int)(((long long)d * d + 255) / 256))), 256, 0, s>>>(Hinv1, d);
  count_launch();
  for (int k0 = 0; k0 < d; k0 += NB) {
    const int nb = std::min(NB, d - k0);
    const int k1 = k0 + nb;
    trtri_panel_kernel<<<(k1 + 63) / 64, 256, 0, s>>>(P, Hinv1, d, k0, hdr);
    count_launch();
    const int below = d - k1;
    if (below > 0) {
      dim3 grid((unsigned)((k1 + TILE - 1) / TILE), (unsigned)((below + TILE - 1) / TILE));
      trtri_update_kernel<<<grid, UPD_THREADS, 0, s>>>(P, Hinv1, d, k0, nb, hdr);
      count_launch();
    }
  }
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

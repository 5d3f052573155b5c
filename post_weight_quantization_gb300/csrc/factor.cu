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
//                   (gather_rev4: natural order, 16-byte loads)
//   Cholesky, 128-wide blocks, right-looking with a look-ahead of one panel:
//     chol_panel    one launch per 128-wide panel: every CTA factors the diagonal block
//                   (32-column tall panels in one warp's registers) and solves 128 rows
//                   below it; CTA 0 writes L11, the others their rows of L21
//     tc_gemm       trailing update A22 -= L21 L21^T (tensor cores, 3 x TF32, both
//                   operands K-major) in two launches: the next panel's column block
//                   first, then the lower tiles right of it, which run on the SMs the
//                   next panel leaves free while that panel is factored
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


struct Header {               // at the start of the factor workspace
  float lambda;
  int nonfinite;
  int fail_pivot;             // INT_MAX when the factorization succeeded
  int d;
  int failed;                 // non-zero once a pivot failed or diag(H) is not finite
  int timeout;                // a bounded wait gave up
  unsigned ready;             // warps of trailing-update tiles of tile column 0 stored so far
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
    hdr->timeout = 0;
    hdr->ready = 0;
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

// Natural order, d % 4 == 0 and 16-byte aligned rows: P[a][b] (b <= a) = H_d[d-1-a][d-1-b]
// = H[d-1-a][d-1-b] (+ lambda on the diagonal), four columns per thread: P[a][4k..4k+3]
// is H[d-1-a][d-4-4k .. d-1-4k] reversed, one aligned 16-byte load. One warp per row a.
__global__ void gather_rev4_kernel(const float* __restrict__ H, int d, const Header* __restrict__ hdr,
                                   float* __restrict__ P) {
  const int a = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (a >= d) return;
  const float lam = hdr->lambda;
  const float* hrow = H + (long long)(d - 1 - a) * d;
  float* prow = P + (long long)a * d;
  for (int k = lane; 4 * k <= a; k += 32) {
    const int b = 4 * k;
    const float4 v = *reinterpret_cast<const float4*>(hrow + d - 4 - b);
    float4 o = make_float4(v.w, v.z, v.y, v.x);          // P[a][b + t] = H[d-1-a][d-1-b-t]
    if (b + 3 <= a) {
      if (b + 3 == a) o.w += lam;
      *reinterpret_cast<float4*>(prow + b) = o;
    } else {                                             // the piece holding the diagonal
      const float ov[4] = {o.x, o.y, o.z, o.w};
      for (int t = 0; b + t <= a; ++t) prow[b + t] = (b + t == a) ? ov[t] + lam : ov[t];
    }
  }
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
// One Cholesky step for the 128-wide panel at k0, in one launch. Every CTA factors the
// 128 x 128 diagonal block (the same arithmetic in every CTA, so every copy agrees;
// CTA 0 keeps it) and CTA b >= 1 also solves the RB rows [k1 + RB (b - 1), + RB) below
// it (R), all in shared memory. The diagonal block goes in four sub-panels of 32
// columns; for sub-panel p, with barriers between the phases:
//   A  warp 0: L[p][p] = chol(S[p][p]) in registers (lane i holds row i); column j of L
//      is broadcast through shared memory (Lt[j][*]), the next pivot's own update stays
//      in its lane, so a column costs one shuffle, one reciprocal square root and a few
//      dependent operations. Meanwhile warps 1-7 finish the previous sub-panel's
//      trailing update of the diagonal block (every block but the one factored now)
//      and bring column block p of R up to date with all earlier ones;
//   B  one warp per row group (sub-panels i > p of the diagonal block, then R): the
//      group's 32 x 32 piece of column block p solves x L[p][p]^T = a by forward
//      substitution, one row per lane;
//   C  the next diagonal sub-block loses the new sub-panel's product (the one update the
//      next Cholesky waits for).
// Values above the diagonal of S are never read as L. A ragged last block is padded
// with the identity.
constexpr int NB = 128;                        // panel width
constexpr int SB = 32;                         // sub-panel width
constexpr int RB = 64;                         // rows below per CTA (RB / SB row groups)
constexpr int PANEL_THREADS = 256;
constexpr int SLD = NB + 4;                    // padded row of the shared tiles (rows stay 16-byte aligned)
constexpr int TLD = SB + 4;                    // padded row of Lt

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

// Bulk asynchronous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// v[c] -= f * Lt[j][c] for c in (j, 32): float4 broadcasts from the aligned piece that
// holds column j + 1 on (columns <= j in that piece are left alone)
template <int J>
__device__ __forceinline__ void axpy_tail(float (&v)[SB], float f, const float* __restrict__ lrow) {
#pragma unroll
  for (int c4 = (J + 1) & ~3; c4 < SB; c4 += 4) {
    const float4 q = *reinterpret_cast<const float4*>(lrow + c4);
    if (c4 + 0 > J) v[c4 + 0] = fmaf(-f, q.x, v[c4 + 0]);
    if (c4 + 1 > J) v[c4 + 1] = fmaf(-f, q.y, v[c4 + 1]);
    if (c4 + 2 > J) v[c4 + 2] = fmaf(-f, q.z, v[c4 + 2]);
    if (c4 + 3 > J) v[c4 + 3] = fmaf(-f, q.w, v[c4 + 3]);
  }
}

// Phase A, warp 0: S[c0..][c0..] (32 x 32) -> its Cholesky factor (lower), Lt[j][c] =
// L[c][j], dinv[c0 + j] = 1 / L[j][j].
template <int... Js>
__device__ __forceinline__ void chol32(std::integer_sequence<int, Js...>, float* __restrict__ S, int c0,
                                       float* __restrict__ Lt, float* __restrict__ dinv, int lane, int& fail) {
  float v[SB];
  float* row = S + (c0 + lane) * SLD + c0;
#pragma unroll
  for (int c = 0; c < SB; c += 4) {
    const float4 q = *reinterpret_cast<const float4*>(row + c);
    v[c] = q.x; v[c + 1] = q.y; v[c + 2] = q.z; v[c + 3] = q.w;
  }
  float piv = __shfl_sync(0xffffffffu, v[0], 0);
  auto column = [&](auto jc) {
    constexpr int j = decltype(jc)::value;
    if (!(piv > 0.0f && piv < INFINITY) && fail < 0) fail = c0 + j;
    const float inv = rsqrt_nr(piv);
    const float l = v[j] * inv;                         // lane j: piv * inv = L[j][j]
    if constexpr (j + 1 < SB) {
      const float dn = fmaf(-l, l, v[j + 1]);           // lane j + 1: the next pivot
      const float pn = __shfl_sync(0xffffffffu, dn, j + 1);
      Lt[j * TLD + lane] = l;
      __syncwarp();
      axpy_tail<j>(v, l, Lt + j * TLD);
      piv = pn;
    }
    v[j] = l;                                           // L[lane][j] (lane >= j)
    if (lane == 0) dinv[c0 + j] = inv;
  };
  (column(std::integral_constant<int, Js>{}), ...);
#pragma unroll
  for (int c = 0; c < SB; c += 4) *reinterpret_cast<float4*>(row + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
}

// Phase B: row `lane` of a 32 x 32 piece (row stride SLD) solves x L^T = a, L = the
// current diagonal sub-block, read as Lt.
template <int... Js>
__device__ __forceinline__ void solve32(std::integer_sequence<int, Js...>, float* __restrict__ A,
                                        const float* __restrict__ Lt, const float* __restrict__ dinv, int lane) {
  float r[SB];
  float* row = A + lane * SLD;
#pragma unroll
  for (int c = 0; c < SB; c += 4) {
    const float4 q = *reinterpret_cast<const float4*>(row + c);
    r[c] = q.x; r[c + 1] = q.y; r[c + 2] = q.z; r[c + 3] = q.w;
  }
  auto column = [&](auto jc) {
    constexpr int j = decltype(jc)::value;
    r[j] *= dinv[j];
    if constexpr (j + 1 < SB) axpy_tail<j>(r, r[j], Lt + j * TLD);
  };
  (column(std::integral_constant<int, Js>{}), ...);
#pragma unroll
  for (int c = 0; c < SB; c += 4) *reinterpret_cast<float4*>(row + c) = make_float4(r[c], r[c + 1], r[c + 2], r[c + 3]);
}

struct BlockTask {
  float* C;
  const float* A;
  const float* B;
};

// C -= A B^T for one 4 x 4 piece of a 32 x 32 block (k < K, K a multiple of 4): rows
// ui + 8a and columns uj + 8b, so the float4 reads of a quarter-warp fall in distinct
// banks.
__device__ __forceinline__ void piece_update(const BlockTask& bt, int ui, int uj, int K) {
  float acc[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.0f;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 a[4], b[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      a[x] = *reinterpret_cast<const float4*>(bt.A + (ui + 8 * x) * SLD + k);
      b[x] = *reinterpret_cast<const float4*>(bt.B + (uj + 8 * x) * SLD + k);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        acc[x][y] = fmaf(a[x].x, b[y].x, acc[x][y]);
        acc[x][y] = fmaf(a[x].y, b[y].y, acc[x][y]);
        acc[x][y] = fmaf(a[x].z, b[y].z, acc[x][y]);
        acc[x][y] = fmaf(a[x].w, b[y].w, acc[x][y]);
      }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) bt.C[(ui + 8 * x) * SLD + uj + 8 * y] -= acc[x][y];
}

static_assert(RB % SB == 0 && RB <= PANEL_THREADS - NB, "one copy-issuing thread per row below");
static_assert(3 + RB / SB <= PANEL_THREADS / 32, "one warp per row group in phase B");

// The panel step; `plain` loads its tiles with ordinary loads (they were published by a
// counter, see chol_panel_kernel) instead of bulk asynchronous copies.
__device__ __noinline__ void chol_panel_body(float* __restrict__ P, float* __restrict__ Lsave, float* __restrict__ Plo,
                                                int d, int k0, int vec, bool plain, Header* hdr, int* err_word) {
  extern __shared__ __align__(16) float psm[];
  float* S = psm;                      // NB x SLD: the diagonal block, then L11 (lower)
  float* R = S + NB * SLD;             // RB x SLD: this CTA's rows below, then its rows of L21
  float* Lt = R + RB * SLD;            // SB x TLD: Lt[j][c] = L[c0 + c][c0 + j] of the current sub-panel
  float* dinv = Lt + SB * TLD;         // NB
  int* fail_s = reinterpret_cast<int*>(dinv + NB);
  uint64_t* bar = reinterpret_cast<uint64_t*>(dinv + NB + 2);   // 8-byte aligned
  if (hdr->failed) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = min(NB, d - k0), k1 = k0 + nb;
  const bool below = blockIdx.x > 0;
  const int rbeg = k1 + (blockIdx.x - 1) * RB;               // first row below handled here
  const int nr = below ? min(RB, d - rbeg) : 0;
  const int nrg = (nr + SB - 1) / SB;                        // row groups of R in use

  // The lower triangle of the diagonal block (pieces of four columns up to the
  // diagonal) and the rows below; the identity past a ragged end.
  if (vec && plain) {
    // whole rows (the part above the diagonal is never read as L), 16 bytes at a time,
    // from L2 (.cg): the rows were stored by the update kernel still running beside us
    constexpr int Q = NB / 4;
    for (int idx = tid; idx < nb * Q; idx += PANEL_THREADS) {
      const int i = idx / Q, c4 = 4 * (idx - i * Q);
      if (c4 < nb)
        *reinterpret_cast<float4*>(S + i * SLD + c4) =
            __ldcg(reinterpret_cast<const float4*>(P + (long long)(k0 + i) * d + k0 + c4));
    }
    for (int idx = tid; idx < nr * Q; idx += PANEL_THREADS) {
      const int i = idx / Q, c4 = 4 * (idx - i * Q);
      if (c4 < nb)
        *reinterpret_cast<float4*>(R + i * SLD + c4) =
            __ldcg(reinterpret_cast<const float4*>(P + (long long)(rbeg + i) * d + k0 + c4));
    }
  } else if (vec) {
    // one bulk asynchronous copy per row: row i of the diagonal block up to the end of
    // the four-column piece holding the diagonal, full rows of R
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int i = 0; i < nb; ++i) bytes += 4u * (uint32_t)min((i | 3) + 1, nb);
      bytes += 4u * (uint32_t)(nr * nb);
      mbar_arrive_expect_tx(bar, bytes);
    }
    __syncthreads();
    if (tid < nb) bulk_g2s(S + tid * SLD, P + (long long)(k0 + tid) * d + k0, 4u * (uint32_t)min((tid | 3) + 1, nb), bar);
    else if (tid >= NB && tid - NB < nr)
      bulk_g2s(R + (tid - NB) * SLD, P + (long long)(rbeg + tid - NB) * d + k0, 4u * (uint32_t)nb, bar);
    const bool landed = mbar_wait_bounded(bar, 0, nullptr);
    if (__syncthreads_or(!landed)) {
      // the copies did not land in time: nothing is written, later kernels skip their
      // work, and the status reports a timeout
      if (tid == 0) {
        report_device_error(err_word, DEVERR_TIMEOUT);
        hdr->timeout = 1;
        hdr->failed = 1;
      }
      return;
    }
  } else {
    for (int idx = tid; idx < nb * nb; idx += PANEL_THREADS) {
      const int i = idx / nb, c = idx - i * nb;
      if (c <= i) S[i * SLD + c] = P[(long long)(k0 + i) * d + k0 + c];
    }
    for (int idx = tid; idx < nr * nb; idx += PANEL_THREADS) {
      const int i = idx / nb, c = idx - i * nb;
      R[i * SLD + c] = P[(long long)(rbeg + i) * d + k0 + c];
    }
  }
  if (nb < NB || (below && nr < RB)) {                       // ragged: pad
    for (int idx = tid; idx < NB * NB; idx += PANEL_THREADS) {
      const int i = idx / NB, c = idx % NB;
      if ((i >= nb || c >= nb) && c <= i) S[i * SLD + c] = (i == c) ? 1.0f : 0.0f;
    }
    if (below)
      for (int idx = tid; idx < RB * NB; idx += PANEL_THREADS) {
        const int i = idx / NB, c = idx % NB;
        if (i >= nr || c >= nb) R[i * SLD + c] = 0.0f;
      }
  }
  if (tid == 0) *fail_s = -1;
  __syncthreads();

#pragma unroll 1
  for (int p = 0; p < 4; ++p) {
    const int c0 = SB * p;
    // ---- A: Cholesky of the sub-block; the rest of the previous trailing update
    if (warp == 0) {
      int fail = -1;
      chol32(std::make_integer_sequence<int, SB>{}, S, c0, Lt, dinv, lane, fail);
      fail = __reduce_min_sync(0xffffffffu, fail < 0 ? INT_MAX : fail);
      if (lane == 0 && fail != INT_MAX && fail < nb) *fail_s = fail;
    } else if (p > 0) {
      // Diagonal block, right-looking: blocks (I, J), p <= J <= I <= 3, but not (p, p),
      // against column block p - 1. Rows below, left-looking: R[g][p] against all of
      // R[g][0 .. p) at once (K = 32 p), one task per row group g; R's column blocks
      // beyond p wait for their own phase, which keeps every phase's share of this work
      // below the time of the sub-block Cholesky.
      // Warp 4 shares warp 0's scheduler and stays out, so the latency-bound Cholesky
      // issues alone there; warps 1-3 and 5-7 take the pieces.
      const int q0 = c0 - SB;
      const int ndiag = (4 - p) * (5 - p) / 2 - 1;
      const int ntask = ndiag + nrg;
      constexpr int TASK_THREADS = PANEL_THREADS - 64;
      const int tw = (warp < 4) ? warp - 1 : warp - 2;       // 0..5 for warps 1-3, 5-7
      for (int u = (warp == 4) ? ntask * 64 : tw * 32 + lane; u < ntask * 64; u += TASK_THREADS) {
        const int t = u >> 6;
        if (t < ndiag) {
          int I = p, n = t + 1;                                // skip (p, p)
          while (n > I - p) { n -= I - p + 1; ++I; }
          const int J = p + n;
          piece_update(BlockTask{S + SB * I * SLD + SB * J, S + SB * I * SLD + q0, S + SB * J * SLD + q0},
                       (u & 63) >> 3, u & 7, SB);
        } else {
          float* Rg = R + (t - ndiag) * SB * SLD;
          piece_update(BlockTask{Rg + c0, Rg, S + c0 * SLD}, (u & 63) >> 3, u & 7, c0);
        }
      }
    }
    __syncthreads();
    if (*fail_s >= 0) break;
    // ---- B: column block p of the row groups below the sub-block
    {
      const int ngrp = 3 - p;
      if (warp < ngrp) solve32(std::make_integer_sequence<int, SB>{}, S + (c0 + SB * (warp + 1)) * SLD + c0, Lt,
                               dinv + c0, lane);
      else if (warp - ngrp < nrg)
        solve32(std::make_integer_sequence<int, SB>{}, R + (warp - ngrp) * SB * SLD + c0, Lt, dinv + c0, lane);
    }
    __syncthreads();
    // ---- C: the next diagonal sub-block, 2 x 2 outputs per thread (rows ri + 16a,
    // columns rj + 16b)
    if (p < 3) {
      const int n0 = c0 + SB;
      const int ri = tid >> 4, rj = tid & 15;
      const float* A0 = S + n0 * SLD + c0;
      float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll 4
      for (int k = 0; k < SB; k += 4) {
        const float4 x0 = *reinterpret_cast<const float4*>(A0 + ri * SLD + k);
        const float4 x1 = *reinterpret_cast<const float4*>(A0 + (ri + 16) * SLD + k);
        const float4 y0 = *reinterpret_cast<const float4*>(A0 + rj * SLD + k);
        const float4 y1 = *reinterpret_cast<const float4*>(A0 + (rj + 16) * SLD + k);
        a00 = fmaf(x0.x, y0.x, fmaf(x0.y, y0.y, fmaf(x0.z, y0.z, fmaf(x0.w, y0.w, a00))));
        a01 = fmaf(x0.x, y1.x, fmaf(x0.y, y1.y, fmaf(x0.z, y1.z, fmaf(x0.w, y1.w, a01))));
        a10 = fmaf(x1.x, y0.x, fmaf(x1.y, y0.y, fmaf(x1.z, y0.z, fmaf(x1.w, y0.w, a10))));
        a11 = fmaf(x1.x, y1.x, fmaf(x1.y, y1.y, fmaf(x1.z, y1.z, fmaf(x1.w, y1.w, a11))));
      }
      float* C0 = S + n0 * SLD + n0;
      C0[ri * SLD + rj] -= a00;
      C0[ri * SLD + rj + 16] -= a01;
      C0[(ri + 16) * SLD + rj] -= a10;
      C0[(ri + 16) * SLD + rj + 16] -= a11;
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
      const int i = idx / NB, c = idx % NB;
      if (i < nb && c <= i) Lsave[(long long)(k0 + i) * d + k0 + c] = S[i * SLD + c];
    }
  } else if (vec) {
    // L21 rows, and their low parts for the trailing update's tensor-core product
    // (Plo[row][c] = x - x with the 13 low mantissa bits cleared)
    const int nq = nb >> 2;
    for (int idx = tid; idx < nr * nq; idx += PANEL_THREADS) {
      const int i = idx / nq, c4 = idx - i * nq;
      const float4 x = *reinterpret_cast<const float4*>(R + i * SLD + 4 * c4);
      *reinterpret_cast<float4*>(P + (long long)(rbeg + i) * d + k0 + 4 * c4) = x;
      float4 l;
      l.x = x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
      l.y = x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
      l.z = x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
      l.w = x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
      *reinterpret_cast<float4*>(Plo + (long long)(rbeg + i) * NB + 4 * c4) = l;
    }
  } else {
    for (int idx = tid; idx < RB * NB; idx += PANEL_THREADS) {
      const int i = idx / NB, c = idx % NB;
      if (i < nr && c < nb) P[(long long)(rbeg + i) * d + k0 + c] = R[i * SLD + c];
    }
  }
}
constexpr size_t PANEL_SMEM = (size_t)((NB + RB) * SLD + SB * TLD + NB + 4) * sizeof(float);   // + flag, mbarrier
// Shared memory reserved per panel CTA: more than half an SM's, so no two CTAs of the
// latency-bound panel share an SM (the trailing update leaves it a few free SMs at a time).
constexpr size_t PANEL_SMEM_RESERVED = PANEL_SMEM > 120 * 1024 ? PANEL_SMEM : 120 * 1024;

// One 128-wide panel step. Without `ready` it waits for the kernel before it (the
// previous trailing update) to complete. With it (look-ahead), that update is still
// running: it publishes its tiles of this panel's column block by adding to *ready,
// and this panel starts once *ready reaches ready_target; only the completion of this
// grid waits for the update's, so the next kernel still sees both.
__global__ void __launch_bounds__(PANEL_THREADS, 2) chol_panel_kernel(float* __restrict__ P, float* __restrict__ Lsave,
                                                                      float* __restrict__ Plo, int d, int k0, int vec,
                                                                      const unsigned* ready, unsigned ready_target,
                                                                      Header* hdr, int* err_word) {
  if (!ready) {
    grid_dep_wait();
    grid_dep_launch();
    chol_panel_body(P, Lsave, Plo, d, k0, vec, false, hdr, err_word);
    return;
  }
  grid_dep_launch();
  __shared__ int ok_s;
  if (threadIdx.x == 0) ok_s = wait_counter_bounded(ready, ready_target) ? 1 : 0;
  __syncthreads();
  if (ok_s) {
    chol_panel_body(P, Lsave, Plo, d, k0, vec, true, hdr, err_word);
  } else if (threadIdx.x == 0) {
    report_device_error(err_word, DEVERR_TIMEOUT);
    hdr->timeout = 1;
    hdr->failed = 1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) grid_dep_wait();
}

// P[k0 + i][k0 + c] = Lsave[k0 + i][k0 + c] for the lower triangle of every diagonal
// block (blockIdx.y = block, 8 rows per CTA in x)
__global__ void place_diag_kernel(float* __restrict__ P, const float* __restrict__ Lsave, int d, const Header* hdr) {
  grid_dep_wait();              // launched behind the kernel that wrote its inputs
  grid_dep_launch();
  if (hdr->failed) return;
  const int k0 = blockIdx.y * NB;
  const int nb = min(NB, d - k0);
  const int i = blockIdx.x * 8 + threadIdx.y;
  if (i >= nb) return;
  const long long row = (long long)(k0 + i) * d + k0;
  for (int c = threadIdx.x; c <= i; c += 32) P[row + c] = Lsave[row + c];
}

constexpr int NBI = 64;       // diagonal blocks inverted at once before the doubling steps

// Inverse of every 64 x 64 diagonal block of L, written into X's diagonal blocks
// (X = L^-1 in natural order). Thread c solves L x = e_c (column c of the inverse).
template <int... Js>
__device__ __forceinline__ void inv_column(std::integer_sequence<int, Js...>, float (&x)[NBI], const float (*L)[NBI + 1],
                                           const float* invd) {
  auto step = [&](auto jc) {
    constexpr int j = decltype(jc)::value;
    x[j] *= invd[j];
#pragma unroll
    for (int q = j + 1; q < NBI; ++q) x[q] = fmaf(-L[q][j], x[j], x[q]);
  };
  (step(std::integral_constant<int, Js>{}), ...);
}

__global__ void __launch_bounds__(64) diag_inverse_kernel(const float* __restrict__ P, float* __restrict__ X, int d,
                                                          const Header* hdr) {
  __shared__ float L[NBI][NBI + 1];
  __shared__ float invd[NBI];
  grid_dep_wait();              // launched behind the kernel that wrote its inputs
  grid_dep_launch();
  if (hdr->failed) return;
  const int k0 = blockIdx.x * NBI;
  const int nb = min(NBI, d - k0);
  load_tile<NBI, NBI, NBI>(&L[0][0], NBI + 1, P + (long long)k0 * d + k0, d, nb, nb);
  __syncthreads();
  for (int idx = threadIdx.x; idx < NBI * NBI; idx += blockDim.x) {   // lower triangle; identity past the block
    const int i = idx / NBI, c = idx % NBI;
    if (c > i || i >= nb) L[i][c] = (i == c) ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < NBI; j += blockDim.x) invd[j] = rcp_nr(L[j][j]);
  __syncthreads();
  const int c = threadIdx.x;
  float x[NBI];
#pragma unroll
  for (int q = 0; q < NBI; ++q) x[q] = (q == c) ? 1.0f : 0.0f;
  inv_column(std::make_integer_sequence<int, NBI>{}, x, L, invd);
  if (c >= nb) return;
#pragma unroll
  for (int q = 0; q < NBI; ++q) {
    if (q < nb && q >= c) X[(long long)(k0 + q) * d + k0 + c] = x[q];
    if (q < nb && q > c) X[(long long)(k0 + c) * d + k0 + q] = x[q];   // the transpose, above
  }
}

// In place: M[a][b] <-> M[d-1-a][d-1-b], then the strict lower triangle cleared: turns
// X = L^-1 (lower, with its transpose stored above) into J X J (upper, lower zero).
__global__ void reverse_kernel(float* __restrict__ M, int d, const Header* hdr) {
  grid_dep_wait();              // launched behind the kernel that wrote its inputs
  grid_dep_launch();
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

// The same for d % 4 == 0 and a 16-byte aligned M: elements idx .. idx + 3 (one row) swap
// with the 16-byte piece at n - 4 - idx, which holds their partners in reverse order.
__global__ void reverse4_kernel(float* __restrict__ M, int d, const Header* hdr) {
  grid_dep_wait();              // launched behind the kernel that wrote its inputs
  grid_dep_launch();
  if (hdr->failed) return;
  const long long n = (long long)d * d;
  float4* M4 = reinterpret_cast<float4*>(M);
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; 4 * k < n / 2;
       k += (long long)gridDim.x * blockDim.x) {
    const long long idx = 4 * k;
    const long long a = idx / d, b = idx - a * d;
    const float4 lo = M4[k];
    const float4 hi = M4[(n - 4 - idx) >> 2];          // partners of idx + 3, + 2, + 1, idx
    M4[k] = make_float4(a <= b ? hi.w : 0.0f, a <= b + 1 ? hi.z : 0.0f, a <= b + 2 ? hi.y : 0.0f,
                        a <= b + 3 ? hi.x : 0.0f);
    M4[(n - 4 - idx) >> 2] = make_float4(a >= b + 3 ? lo.w : 0.0f, a >= b + 2 ? lo.z : 0.0f,
                                         a >= b + 1 ? lo.y : 0.0f, a >= b ? lo.x : 0.0f);
  }
}

// Y[a0 + j][c0 + i] = X[c0 + i][a0 + j] for every pair z of the doubling step: the
// transpose of the block just computed, stored above the diagonal.
__global__ void pair_transpose_kernel(float* __restrict__ M, int d, int sz, int np, int c_last,
                                      const Header* hdr) {
  __shared__ float tile[32][33];
  grid_dep_wait();              // launched behind the product that wrote its input
  grid_dep_launch();
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

// header | P (d x d) | Plo[2] (d x 128 each: low parts of L21 of the even and the odd
// panels; a panel writes its own while the trailing update of the one before still reads
// the other)
size_t factor_workspace_bytes(long long d) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return factor::kHeaderBytes + al((size_t)d * (size_t)d * sizeof(float)) +
         2 * al((size_t)d * factor::NB * sizeof(float));
}

gptq_status factor_launch(const float* H, long long d_, float percdamp, int act_order, int32_t* perm_out,
                          float* Hinv1, void* ws, cudaStream_t s) {
  using namespace factor;
  const int d = (int)d_;
  Header* hdr = reinterpret_cast<Header*>(ws);
  float* P = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kHeaderBytes);
  float* Plo0 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kHeaderBytes +
                                         (((size_t)d * (size_t)d * sizeof(float) + 255) & ~(size_t)255));
  const size_t plo_stride = (((size_t)d * NB * sizeof(float) + 255) & ~(size_t)255) / sizeof(float);
  auto plo = [&](int k0) { return Plo0 + ((k0 / NB) & 1) * plo_stride; };
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
  if (!act_order && d % 4 == 0 && simt::aligned16(H) && simt::aligned16(P)) {
    gather_rev4_kernel<<<(unsigned)((d + 7) / 8), 256, 0, s>>>(H, d, hdr, P);
    count_launch();
  } else {
    dim3 grid((unsigned)std::min(64, (d + 31) / 32), (unsigned)((d + 7) / 8));
    gather_kernel<<<grid, dim3(32, 8), 0, s>>>(H, d, act_order ? perm_out : nullptr, hdr, P);
    count_launch();
  }
  }
  if (gptq_status st = check_launch("factor setup kernels")) return st;

  if (cudaFuncSetAttribute(chol_panel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PANEL_SMEM_RESERVED) !=
      cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(chol_panel_kernel) failed");

  // ---- Cholesky P = L L^T, 128-wide panels, right-looking with a look-ahead of one
  // panel. The trailing update after panel k computes its tiles column by column, so
  // panel k+1's column block comes first; each stored tile of it is published on
  // hdr->ready (8 per tile), and panel k+1, already resident, starts when all of them
  // are, while the rest of the update runs on the SMs it leaves free. (Through the FFMA
  // GEMM, which publishes nothing, the panels wait for whole kernels instead.)
  auto panel_ctas = [](int below) { return 1 + (below + RB - 1) / RB; };
  const bool lookahead = vec && tc_gemm_available();
  unsigned ready_target = 0;
  for (int k0 = 0; k0 < d; k0 += NB) {
    const int nb = std::min(NB, d - k0), k1 = k0 + nb, below = d - k1;
    const bool flagged = lookahead && k0 > 0;
    {
      ProfScope ps("factor.chol_panel", s);
      if (launch_pdl(chol_panel_kernel, dim3(panel_ctas(below)), dim3(PANEL_THREADS), PANEL_SMEM_RESERVED, s, P, Hinv1,
                     plo(k0), d, k0, vec ? 1 : 0, flagged ? &hdr->ready : nullptr, ready_target, hdr,
                     device_error_word()) != cudaSuccess)
        return check_launch("chol_panel_kernel");
      count_launch();
    }
    if (below > 0) {
      // A22 -= L21 L21^T over the lower tiles of P[k1:, k1:]
      simt::GemmArgs g{};
      g.M = g.N = below; g.K = nb; g.M_last = below; g.K_last = nb;
      g.A = P + (long long)k1 * d + k0; g.lda = d;
      g.B = g.A; g.ldb = d;
      g.A_lo = plo(k0) + (long long)k1 * NB; g.lda_lo = NB;
      g.B_lo = g.A_lo; g.ldb_lo = NB;
      g.C = P + (long long)k1 * d + k1; g.ldc = d;
      g.alpha = -1.0f; g.beta = 1.0f;
      g.lower_tiles = lookahead ? 2 : 1;
      g.vec = vec;
      g.skip = failed;
      if (lookahead) {
        const int below_next = below - std::min(NB, below);
        g.signal = &hdr->ready;
        g.max_ctas = std::max(1, sm_count() - panel_ctas(below_next));
        ready_target += 8u * (unsigned)((below + 127) / 128);   // tiles of tile column 0
      }
      ProfScope ps("factor.chol_update_gemm", s);
      if (gptq_status st = tc_gemm(g, 1, true, true, s)) return st;
    }
  }
  if (gptq_status st = check_launch("Cholesky kernels")) return st;

  // ---- X = L^-1 in natural order inside Hinv1: diagonal blocks, then recursive doubling
  {
    ProfScope ps("factor.zero_diag_inverse", s);
    if (launch_pdl(place_diag_kernel, dim3(NB / 8, (unsigned)((d + NB - 1) / NB)), dim3(32, 8), 0, s, P,
                   (const float*)Hinv1, d, (const Header*)hdr) != cudaSuccess)
      return check_launch("place_diag_kernel");
    count_launch();
    // No clearing pass: every element of Hinv1 is written below before anything reads
    // it (the diagonal blocks whole, then at every level each pair's X block below the
    // diagonal and its transpose above), and the masked triangles of the products'
    // operands are replaced by zeros, not multiplied, so what the buffer held is never
    // used.
    if (launch_pdl(diag_inverse_kernel, dim3((d + NBI - 1) / NBI), dim3(NBI), 0, s, (const float*)P, Hinv1, d,
                   (const Header*)hdr) != cudaSuccess)
      return check_launch("diag_inverse_kernel");
  }
  count_launch();
  // Doubling over block pairs (A, C) = ([2p sz, 2p sz + sz), [2p sz + sz, ...)): with
  // X = L^-1 kept below the diagonal of Hinv1 and Y = X^T above it (shared diagonal),
  //   T = Y[A][A] L[C][A]^T           (= (L[C][A] X[A][A])^T, into P's unused upper part)
  //   X[C][A] = -X[C][C] T^T          (= -X[C][C] L[C][A] X[A][A])
  //   Y[A][C] = X[C][A]^T
  // so every product has both operands K-major (the tensor-core GEMM's layout); the
  // triangular operands are masked, since their other triangle holds the transpose.
  for (int sz = NBI; sz < d; sz *= 2) {
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
    if (launch_pdl(pair_transpose_kernel, tg, dim3(32, 8), 0, s, Hinv1, d, sz, np, c_last, (const Header*)hdr) !=
        cudaSuccess)
      return check_launch("pair_transpose_kernel");
    count_launch();
  }
  ProfScope ps_rev("factor.reverse", s);
  {
    const bool v4 = vec;
    const long long work = v4 ? (long long)d * d / 8 : (long long)d * d / 2;
    const dim3 grid((unsigned)std::max(1, std::min(4096, (int)((work + 255) / 256))));
    if (launch_pdl(v4 ? reverse4_kernel : reverse_kernel, grid, dim3(256), 0, s, Hinv1, d, (const Header*)hdr) !=
        cudaSuccess)
      return check_launch("reverse_kernel");
  }
  count_launch();
  return check_launch("triangular-inverse kernels");
}

gptq_status factor_read_status(const void* ws, long long* info, cudaStream_t s) {
  factor::Header h;
  if (cudaStreamSynchronize(s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaStreamSynchronize failed");
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "reading the factor status failed");
  if (h.timeout) {
    if (info) *info = -1;
    return set_error(GPTQ_ERR_TIMEOUT, "a wait for the panel's copies gave up");
  }
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

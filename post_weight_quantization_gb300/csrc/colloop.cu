// Stage 3: the blocked GPTQ column loop.
//
// Per block of BS columns ("GPTQ, Line by Line", question "Why does GPTQ process the
// weight matrix in blocks of 128 columns?"):
//   * at a group's first column, per row: scale = (max - min) / (2^b - 1) (clamped
//     to >= 1e-8) and zero = clamp(round(-min / scale)) over the group's current
//     weights ("GPTQ-style round-to-nearest with Hessian weighting", listing);
//   * for each column j: q = clamp(round(w / scale + zero)), w_hat = (q - zero) * scale,
//     Err1 = (w - w_hat) / Hinv1[j][j], Losses1 = Err1^2 / 2, and the block's
//     remaining columns move by -Err1 * Hinv1[j][j+1:] (rank-one update);
//   * after the block, the columns right of it move by -Err1 @ Hinv1[block, rest]
//     (the lazy update, one matrix product).
//
// Kernels:
//   prep_kernel        fp32 working copy of W in processing order; NaN/Inf check
//   colblock_kernel<BS> one thread per row, the block as 32-column sub-blocks whose
//                      weights stay in registers (the block's later columns wait in
//                      shared memory); the Hinv1 diagonal block sits in shared memory
//                      (every thread reads the same entry: broadcast); codes are packed into the
//                      output bitstream as they are produced; Err1 is written
//                      column-major (coalesced) for the lazy update; per-column loss
//                      partial sums come from warp-shuffle reductions
//   lazy_update_kernel W[:, i2:] -= Err1 @ Hinv1[i1:i2, i2:], FFMA tiles 128 x 128
//   loss_finalize      col_losses = sum of partials in a fixed order, un-permuted
//   pack_perm          act-order: gather codes back to the original column order
//
// The quantizer uses correctly rounded quotients (see div_mk) and no fused
// multiply-add, so each step rounds exactly like the listing's float32 arithmetic.
#include <algorithm>
#include <utility>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {
namespace colloop {

struct QHeader {
  int nonfinite;
};
constexpr size_t kHeaderBytes = 256;
constexpr int ROWS_PER_CTA = 32;

__device__ __forceinline__ float load_w(const void* W, int w_dtype, long long idx) {
  if (w_dtype == 0) return reinterpret_cast<const float*>(W)[idx];
  const uint16_t b = reinterpret_cast<const uint16_t*>(W)[idx];
  return __uint_as_float(((uint32_t)b) << 16);
}

__global__ void prep_kernel(const void* __restrict__ W, int w_dtype, int m, int d, long long ldw,
                            const int* __restrict__ perm, float* __restrict__ Wf, QHeader* hdr) {
  int bad = 0;
  for (int r = blockIdx.y; r < m; r += gridDim.y) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < d; j += gridDim.x * blockDim.x) {
      const int src = perm ? perm[j] : j;
      const float v = load_w(W, w_dtype, (long long)r * ldw + src);
      bad |= !isfinite(v);
      Wf[(long long)r * d + j] = v;
    }
  }
  if (bad) atomicOr(&hdr->nonfinite, 1);
}

// Correctly rounded a / b from the correctly rounded reciprocal inv_b = RN(1 / b):
// q = RN(a * inv_b) is within one ulp of a / b; the remainder a - b q is exact with
// one fused multiply-add, and RN(q + (a - b q) inv_b) is the correctly rounded
// quotient (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990, Theorem 1), barring overflow
// and results below the normal range. Keeps IEEE division (and its out-of-line slow
// path) out of the register-resident column loop.
__device__ __forceinline__ float div_mk(float a, float b, float inv_b) {
  const float q = __fmul_rn(a, inv_b);
  const float r = __fmaf_rn(-q, b, a);
  return __fmaf_rn(r, inv_b, q);
}

// RN(1 / s) for a normal float s without a call: Newton-Raphson reciprocal iteration
// y <- y + y (1 - s y) in fp64 from the hardware approximation; two steps give a
// relative error near 2^-52, and a quotient of two floats lies at least 2^-49
// (relative) away from any midpoint between floats, so rounding the fp64 value to
// float gives the correctly rounded reciprocal.
__device__ __forceinline__ float rcp_rn(float s) {
  const double sd = (double)s;
  double y;
  asm("rcp.approx.ftz.f64 %0, %1;" : "=d"(y) : "d"(sd));
  double e = fma(-sd, y, 1.0);
  y = fma(y, e, y);
  e = fma(-sd, y, 1.0);
  y = fma(y, e, y);
  return __double2float_rn(y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// State of one row (one thread) while a block is processed.
struct RowState {
  const float* wrow;      // the row of the working copy (global)
  float* wsm;             // the row's block columns in shared memory (stride 1)
  float s, z, inv_s;      // current group's scale, zero and RN(1 / scale)
  uint64_t acc;           // code bits not yet stored
  int nacc, widx;         // bits held in acc; next output word
};

struct BlockArgs {
  const float* Us;        // Hinv1 diagonal block (shared memory), row-major BS x BS
  const float* inv_u;     // RN(1 / Hinv1[j][j]) of the block (shared memory)
  int m, d, i1, ncols, g, G, wpr, lde, bits, r, lane, bs;
  bool active, natural;
  float qmax, inv_qmax;
  uint32_t* qweight;
  uint8_t* codes8;
  float *scales, *zeros, *errT, *part;
};

constexpr int SUB = 32;   // columns per register-resident sub-block

// Column T of sub-block c0 (block-local column c0 + T). T is a compile-time constant so
// that w[] and e[] stay in registers; the sub-block's other columns live in w[].
template <int T>
__device__ __forceinline__ void column_step(float (&w)[SUB], float (&e)[SUB], RowState& st, const BlockArgs& a,
                                            int c0) {
  const int t = c0 + T;
  if (t >= a.ncols) return;
  const int j = a.i1 + t;
  if constexpr (T == 0) {
    if ((j % a.g) == 0) {
      // group statistics over the current weights of columns [j, j + g): this
      // sub-block (registers), the block's later columns (shared memory, already
      // updated by the earlier sub-blocks) and, for groups wider than the block, the
      // working copy (already updated by the lazy updates)
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < SUB; ++u)
        if (c0 + u < a.ncols && u < a.g) { mn = fminf(mn, w[u]); mx = fmaxf(mx, w[u]); }
      for (int u = c0 + SUB; u < a.ncols && u - c0 < a.g; ++u) {
        const float v = st.wsm[u];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      for (int c = a.i1 + a.ncols; c < j + a.g && c < a.d; ++c) {
        const float v = st.wrow[c];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      st.s = fmaxf(div_mk(__fsub_rn(mx, mn), a.qmax, a.inv_qmax), 1e-8f);
      st.inv_s = rcp_rn(st.s);
      st.z = fminf(fmaxf(rintf(div_mk(-mn, st.s, st.inv_s)), 0.0f), a.qmax);
      if (a.active) {
        a.scales[(long long)a.r * a.G + j / a.g] = st.s;
        a.zeros[(long long)a.r * a.G + j / a.g] = st.z;
      }
    }
  }
  const float x = w[T];
  const float q = fminf(fmaxf(rintf(__fadd_rn(div_mk(x, st.s, st.inv_s), st.z)), 0.0f), a.qmax);
  const float wq = __fmul_rn(__fsub_rn(q, st.z), st.s);
  const float err = a.active ? div_mk(__fsub_rn(x, wq), a.Us[t * a.bs + t], a.inv_u[t]) : 0.0f;
  e[T] = err;
  a.errT[(long long)t * a.lde + a.r] = err;
  const float lsum = warp_sum(__fmul_rn(__fmul_rn(err, err), 0.5f));
  if (a.lane == 0) a.part[(long long)blockIdx.x * a.d + j] = lsum;
  const uint32_t qi = (uint32_t)q;
  if (a.natural) {
    st.acc |= (uint64_t)qi << st.nacc;
    st.nacc += a.bits;
    if (st.nacc >= 32) {
      if (a.active) a.qweight[(long long)a.r * a.wpr + st.widx] = (uint32_t)st.acc;
      ++st.widx;
      st.acc >>= 32;
      st.nacc -= 32;
    }
  } else if (a.active) {
    a.codes8[(long long)a.r * a.d + j] = (uint8_t)qi;
  }
  // rank-one update of the sub-block's remaining columns (same rounding as w - e * u)
  const float4* urow = reinterpret_cast<const float4*>(a.Us + t * a.bs + c0);
#pragma unroll
  for (int u4 = (T + 1) / 4; u4 < SUB / 4; ++u4) {
    const float4 uv = urow[u4];
    if (4 * u4 + 0 > T) w[4 * u4 + 0] = __fsub_rn(w[4 * u4 + 0], __fmul_rn(err, uv.x));
    if (4 * u4 + 1 > T) w[4 * u4 + 1] = __fsub_rn(w[4 * u4 + 1], __fmul_rn(err, uv.y));
    if (4 * u4 + 2 > T) w[4 * u4 + 2] = __fsub_rn(w[4 * u4 + 2], __fmul_rn(err, uv.z));
    if (4 * u4 + 3 > T) w[4 * u4 + 3] = __fsub_rn(w[4 * u4 + 3], __fmul_rn(err, uv.w));
  }
}

template <int... Ts>
__device__ __forceinline__ void sub_block_steps(std::integer_sequence<int, Ts...>, float (&w)[SUB], float (&e)[SUB],
                                                RowState& st, const BlockArgs& a, int c0) {
  (column_step<Ts>(w, e, st, a, c0), ...);
}

// One row per thread. The block's BS columns are processed as BS / 32 sub-blocks: a
// sub-block's 32 weights sit in registers and take their rank-one updates there; when
// the sub-block is done its 32 errors are applied to the block's later columns, kept
// in shared memory, in the same per-column order (so the rounding matches updating
// every column after every step).
template <int BS>
__global__ void __launch_bounds__(ROWS_PER_CTA)
colblock_kernel(const float* __restrict__ Wf, int m, int d, const float* __restrict__ U, int i1, int bits, int g,
                uint32_t* __restrict__ qweight, int wpr, uint8_t* __restrict__ codes8, float* __restrict__ scales,
                float* __restrict__ zeros, int G, float* __restrict__ errT, int lde, float* __restrict__ part) {
  extern __shared__ __align__(16) float Us[];   // BS x BS Hinv1 block, BS reciprocals, 32 x (BS + 1) rows
  float* inv_u = Us + BS * BS;
  float* Wsm = inv_u + BS;
  constexpr int WLD = BS + 1;                    // padded row stride: lanes hit distinct banks
  const int lane = threadIdx.x;
  const int ncols = min(BS, d - i1);
  for (int idx = lane; idx < BS * BS; idx += ROWS_PER_CTA) {
    const int t = idx / BS, u = idx % BS;
    Us[idx] = (t < ncols && u < ncols && u >= t) ? U[(long long)(i1 + t) * d + i1 + u] : 0.0f;
  }
  // the CTA's 32 rows of the block, one coalesced row at a time
  const int r0 = blockIdx.x * ROWS_PER_CTA;
  for (int rr = 0; rr < ROWS_PER_CTA; ++rr) {
    const bool ok = r0 + rr < m;
    for (int c = lane; c < BS; c += ROWS_PER_CTA)
      Wsm[rr * WLD + c] = (ok && c < ncols) ? Wf[(long long)(r0 + rr) * d + i1 + c] : 0.0f;
  }
  __syncwarp();
  for (int t = lane; t < BS; t += ROWS_PER_CTA) inv_u[t] = (t < ncols) ? __frcp_rn(Us[t * BS + t]) : 0.0f;
  __syncwarp();

  BlockArgs a;
  a.Us = Us;
  a.inv_u = inv_u;
  a.m = m;
  a.d = d;
  a.i1 = i1;
  a.ncols = ncols;
  a.g = g;
  a.G = G;
  a.wpr = wpr;
  a.lde = lde;
  a.bits = bits;
  a.bs = BS;
  a.r = r0 + lane;
  a.lane = lane;
  a.active = a.r < m;
  a.natural = (codes8 == nullptr);
  a.qmax = (float)((1 << bits) - 1);
  a.inv_qmax = __frcp_rn(a.qmax);
  a.qweight = qweight;
  a.codes8 = codes8;
  a.scales = scales;
  a.zeros = zeros;
  a.errT = errT;
  a.part = part;

  RowState st;
  st.wrow = Wf + (long long)(a.active ? a.r : 0) * d;
  st.wsm = Wsm + lane * WLD;
  st.s = 1.0f;
  st.z = 0.0f;
  if ((i1 % g) != 0 && a.active) {   // the block continues a group that began in an earlier block
    st.s = scales[(long long)a.r * G + i1 / g];
    st.z = zeros[(long long)a.r * G + i1 / g];
  }
  st.inv_s = rcp_rn(st.s);
  st.acc = 0;
  st.nacc = 0;
  st.widx = (int)(((long long)i1 * bits) >> 5);

#pragma unroll 1
  for (int c0 = 0; c0 < ncols; c0 += SUB) {
    float w[SUB], e[SUB];
#pragma unroll
    for (int u = 0; u < SUB; ++u) w[u] = st.wsm[c0 + u];
    sub_block_steps(std::make_integer_sequence<int, SUB>{}, w, e, st, a, c0);
    // the sub-block's errors move the block's later columns, column by column
    const int nsub = min(SUB, ncols - c0);
#pragma unroll 1
    for (int c = c0 + SUB; c < ncols; ++c) {
      float x = st.wsm[c];
#pragma unroll
      for (int u = 0; u < SUB; ++u)
        if (u < nsub) x = __fsub_rn(x, __fmul_rn(e[u], Us[(c0 + u) * BS + c]));
      st.wsm[c] = x;
    }
  }

  if (a.natural && st.nacc > 0 && a.active) qweight[(long long)a.r * wpr + st.widx] = (uint32_t)st.acc;
}

// Wf[r][c] -= sum_{k < nb} errT[k][r] * U[i1 + k][c]  for r < m, c in [c0, d)
__global__ void __launch_bounds__(simt::THREADS)
lazy_update_kernel(float* __restrict__ Wf, int m, int d, const float* __restrict__ errT, int lde,
                   const float* __restrict__ U, int i1, int nb, int c0) {
  using simt::KC;
  using simt::TILE;
  __shared__ __align__(16) float As[KC][TILE];
  __shared__ __align__(16) float Bs[KC][TILE];
  const int r0 = blockIdx.y * TILE;
  const int j0 = c0 + blockIdx.x * TILE;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  simt::Acc acc;
  simt::zero(acc);
  for (int kc = 0; kc < nb; kc += KC) {
    const int kn = min(KC, nb - kc);
    __syncthreads();
    for (int idx = threadIdx.x; idx < TILE * KC; idx += simt::THREADS) {
      const int c = idx % TILE, k = idx / TILE;
      float va = 0.0f, vb = 0.0f;
      if (k < kn) {
        if (r0 + c < m) va = errT[(long long)(kc + k) * lde + r0 + c];
        if (j0 + c < d) vb = U[(long long)(i1 + kc + k) * d + j0 + c];
      }
      As[k][c] = va;
      Bs[k][c] = vb;
    }
    __syncthreads();
    simt::mma_chunk(As, Bs, kn, tx, ty, acc);
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int r = r0 + simt::micro_row(a, ty);
    if (r >= m) continue;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int c = j0 + simt::micro_row(b, tx);
      if (c < d) Wf[(long long)r * d + c] = __fsub_rn(Wf[(long long)r * d + c], acc.v[a][b]);
    }
  }
}

__global__ void loss_finalize_kernel(const float* __restrict__ part, int nrg, int d, const int* __restrict__ perm,
                                     float* __restrict__ col_losses) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= d) return;
  float s = 0.0f;
  for (int b = 0; b < nrg; ++b) s += part[(long long)b * d + j];
  col_losses[perm ? perm[j] : j] = s;
}

__global__ void invperm_kernel(const int* __restrict__ perm, int d, int* __restrict__ inv) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < d) inv[perm[j]] = j;
}

// word w of row r from the codes of original columns, codes8 indexed in processing order
__global__ void pack_perm_kernel(const uint8_t* __restrict__ codes8, int m, int d, const int* __restrict__ inv,
                                 int bits, uint32_t* __restrict__ qweight, int wpr) {
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)m * wpr) return;
  const int r = (int)(idx / wpr), wi = (int)(idx % wpr);
  const long long b0 = (long long)wi * 32;
  const int jfirst = (int)(b0 / bits);
  const int jlast = (int)min((long long)d - 1, (b0 + 31) / bits);
  uint64_t v = 0;
  for (int jo = jfirst; jo <= jlast; ++jo) {
    const uint64_t code = codes8[(long long)r * d + inv[jo]];
    const long long sh = (long long)jo * bits - b0;
    v |= (sh >= 0) ? (code << sh) : (code >> (-sh));
  }
  qweight[idx] = (uint32_t)v;
}

__global__ void unpack_kernel(const uint32_t* __restrict__ qweight, int m, int d, int bits, int wpr,
                              uint8_t* __restrict__ codes) {
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)m * d) return;
  const int r = (int)(idx / d), j = (int)(idx % d);
  const long long bp = (long long)j * bits;
  const int wi = (int)(bp >> 5), off = (int)(bp & 31);
  uint64_t v = qweight[(long long)r * wpr + wi] >> off;
  if (off + bits > 32) v |= (uint64_t)qweight[(long long)r * wpr + wi + 1] << (32 - off);
  codes[idx] = (uint8_t)(v & ((1u << bits) - 1u));
}

struct Layout {
  size_t hdr, wf, errT, part, codes8, inv, total;
  int lde, nrg;
};

Layout layout(long long m, long long d, int blocksize) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  Layout L;
  L.lde = (int)((m + 127) / 128 * 128);
  L.nrg = (int)((m + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
  L.hdr = 0;
  L.wf = kHeaderBytes;
  L.errT = L.wf + al((size_t)m * d * 4);
  L.part = L.errT + al((size_t)blocksize * L.lde * 4);
  L.codes8 = L.part + al((size_t)L.nrg * d * 4);
  L.inv = L.codes8 + al((size_t)m * d);
  L.total = L.inv + al((size_t)d * 4);
  return L;
}

template <int BS>
gptq_status run_blocks(float* Wf, int m, int d, const float* U, int bits, int g, uint32_t* qweight, int wpr,
                       uint8_t* codes8, float* scales, float* zeros, int G, float* errT, int lde, float* part,
                       cudaStream_t s) {
  const size_t smem = (size_t)(BS * BS + BS + ROWS_PER_CTA * (BS + 1)) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(colblock_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(colblock_kernel) failed");
    attr = true;
  }
  const int nrg = (m + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  for (int i1 = 0; i1 < d; i1 += BS) {
    const int nb = std::min(BS, d - i1);
    colblock_kernel<BS><<<nrg, ROWS_PER_CTA, smem, s>>>(Wf, m, d, U, i1, bits, g, qweight, wpr, codes8, scales,
                                                        zeros, G, errT, lde, part);
    count_launch();
    const int i2 = i1 + nb;
    if (i2 < d) {
      dim3 grid((unsigned)((d - i2 + simt::TILE - 1) / simt::TILE), (unsigned)((m + simt::TILE - 1) / simt::TILE));
      lazy_update_kernel<<<grid, simt::THREADS, 0, s>>>(Wf, m, d, errT, lde, U, i1, nb, i2);
      count_launch();
    }
  }
  return check_launch("column-loop kernels");
}

}  // namespace colloop

size_t quantize_workspace_bytes(long long m, long long d, int blocksize) {
  return colloop::layout(m, d, blocksize).total;
}

gptq_status quantize_launch(const void* W, int w_dtype, long long m_, long long d_, long long ldw, const float* Hinv1,
                            const int32_t* perm, int bits, int group_size, int blocksize, uint32_t* qweight,
                            float* scales, float* zeros, float* col_losses, void* ws, cudaStream_t s) {
  using namespace colloop;
  const int m = (int)m_, d = (int)d_;
  const Layout L = layout(m, d, blocksize);
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  QHeader* hdr = reinterpret_cast<QHeader*>(base + L.hdr);
  float* Wf = reinterpret_cast<float*>(base + L.wf);
  float* errT = reinterpret_cast<float*>(base + L.errT);
  float* part = reinterpret_cast<float*>(base + L.part);
  uint8_t* codes8 = perm ? base + L.codes8 : nullptr;
  int* inv = reinterpret_cast<int*>(base + L.inv);
  const int g = (group_size < 0) ? d : group_size;
  const int G = d / g;
  const int wpr = (int)(((long long)d * bits + 31) / 32);

  if (cudaMemsetAsync(hdr, 0, sizeof(QHeader), s) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaMemsetAsync failed");
  {
    dim3 grid((unsigned)std::min(8, (d + 255) / 256), (unsigned)std::min(m, 65535));
    prep_kernel<<<grid, 256, 0, s>>>(W, w_dtype, m, d, ldw, perm, Wf, hdr);
    count_launch();
  }
  gptq_status st;
  switch (blocksize) {
    case 32: st = run_blocks<32>(Wf, m, d, Hinv1, bits, g, qweight, wpr, codes8, scales, zeros, G, errT, L.lde, part, s); break;
    case 64: st = run_blocks<64>(Wf, m, d, Hinv1, bits, g, qweight, wpr, codes8, scales, zeros, G, errT, L.lde, part, s); break;
    default: st = run_blocks<128>(Wf, m, d, Hinv1, bits, g, qweight, wpr, codes8, scales, zeros, G, errT, L.lde, part, s); break;
  }
  if (st) return st;
  loss_finalize_kernel<<<(d + 255) / 256, 256, 0, s>>>(part, L.nrg, d, perm, col_losses);
  count_launch();
  if (perm) {
    invperm_kernel<<<(d + 255) / 256, 256, 0, s>>>(perm, d, inv);
    const long long nw = (long long)m * wpr;
    pack_perm_kernel<<<(unsigned)((nw + 255) / 256), 256, 0, s>>>(codes8, m, d, inv, bits, qweight, wpr);
    count_launch(2);
  }
  return check_launch("column-loop finalize kernels");
}

gptq_status quantize_read_status(const void* ws, long long* info, cudaStream_t s) {
  colloop::QHeader h;
  if (cudaStreamSynchronize(s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaStreamSynchronize failed");
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "reading the quantize status failed");
  if (info) *info = h.nonfinite ? 1 : 0;
  if (h.nonfinite) return set_error(GPTQ_ERR_NONFINITE, "W holds a NaN or an Inf");
  return GPTQ_OK;
}

gptq_status unpack_launch(const uint32_t* qweight, long long m, long long d, int bits, uint8_t* codes, cudaStream_t s) {
  const int wpr = (int)((d * bits + 31) / 32);
  const long long n = m * d;
  if (n == 0) return GPTQ_OK;
  colloop::unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(qweight, (int)m, (int)d, bits, wpr, codes);
  count_launch();
  return check_launch("unpack_kernel");
}

}  // namespace gptq

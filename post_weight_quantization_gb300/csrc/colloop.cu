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
//   colblock_kernel<BS> eight lanes per row (4 rows per warp, 32 per CTA), the block as
//                      32-column register sub-blocks (the block's later columns wait
//                      in shared memory), the Hinv1 diagonal block in shared memory,
//                      group min/max by shuffles; codes are packed into the
//                      output bitstream as they are produced; Err1 is written
//                      row-major for the lazy update; per-column loss partial
//                      sums of each CTA's 32 rows in a fixed order
//   transpose_kernel   Ut = Hinv1^T once per call
//   tc_gemm            lazy update W[:, i2:] -= Err1 @ Hinv1[i1:i2, i2:] on the tensor cores
//                      (3 x TF32, both operands K-major: Err1 rows, Ut rows)
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

// Column block, LANES lanes per row.
//
// A warp holds 32 / LANES rows; the LANES lanes of a row own the block's columns
// c = LANES k + q round-robin (q = lane % LANES). At each column the owner broadcasts
// the current weight with one shuffle and all lanes of the row quantize it
// identically, then each lane applies the rank-one update to its own later columns.
// Within a 32-column sub-block the lane's columns sit in registers and are rotated by
// one slot every LANES columns, so the column about to be quantized is always slot 0
// of its owner and the loop body stays a few hundred instructions long. When a sub-block is done, its 32
// errors update the block's later columns (kept in shared memory) column by column in
// the same order, so the rounding is that of updating every column after every step.
constexpr int LANES = 8;                             // lanes per row
constexpr int ROWS_PER_WARP = 32 / LANES;            // 4
constexpr int WARPS_PER_CTA = ROWS_PER_CTA / ROWS_PER_WARP;   // 8
constexpr int CB_THREADS = WARPS_PER_CTA * 32;      // 256
constexpr int SUB = 32;                              // columns per register sub-block
constexpr int SLOTS = SUB / LANES;                   // 4 registers per lane
constexpr int ELD = SUB + 1;                         // padded row stride of the error tile

template <int BS>
__global__ void __launch_bounds__(CB_THREADS)
colblock_kernel(const float* __restrict__ Wf, int m, int d, const float* __restrict__ U, int i1, int bits, int g,
                uint32_t* __restrict__ qweight, int wpr, uint8_t* __restrict__ codes8, float* __restrict__ scales,
                float* __restrict__ zeros, int G, float* __restrict__ err, float* __restrict__ part) {
  extern __shared__ __align__(16) float smem[];
  float* Us = smem;                                  // BS x BS: Us[t * BS + u] = Hinv1[i1 + t][i1 + u]
  float* inv_u = Us + BS * BS;                       // RN(1 / Hinv1[j][j])
  float* Wsm = inv_u + BS;                           // ROWS_PER_CTA x (BS + 1): the block's weights
  float* Es = Wsm + ROWS_PER_CTA * (BS + 1);         // ROWS_PER_CTA x ELD: the sub-block's errors
  constexpr int WLD = BS + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = lane % LANES;                        // position within the row's lanes
  const int qbase = lane - q;                        // lane owning the row's column 0
  const int row = warp * ROWS_PER_WARP + lane / LANES;  // row within the CTA
  const int r0 = blockIdx.x * ROWS_PER_CTA;
  const int r = r0 + row;
  const bool active = r < m;
  const int ncols = min(BS, d - i1);

  // the Hinv1 block (only its upper triangle is ever read) and the CTA's rows of W
  load_tile<CB_THREADS, BS, BS>(Us, BS, U + (long long)i1 * d + i1, d, ncols, ncols);
  load_tile<CB_THREADS, ROWS_PER_CTA, BS>(Wsm, WLD, Wf + (long long)r0 * d + i1, d, min(ROWS_PER_CTA, m - r0), ncols);
  __syncthreads();
  for (int t = tid; t < BS; t += CB_THREADS) inv_u[t] = (t < ncols) ? __frcp_rn(Us[t * BS + t]) : 0.0f;
  __syncthreads();

  float* wsm = Wsm + row * WLD;
  float* es = Es + row * ELD;
  const float* wrow = Wf + (long long)(active ? r : 0) * d;
  const float qmax = (float)((1 << bits) - 1);
  const float inv_qmax = __frcp_rn(qmax);
  float s = 1.0f, z = 0.0f;
  if ((i1 % g) != 0 && active) {   // the block continues a group that began in an earlier block
    s = scales[(long long)r * G + i1 / g];
    z = zeros[(long long)r * G + i1 / g];
  }
  float inv_s = rcp_rn(s);
  const bool natural = (codes8 == nullptr);
  const bool packer = natural && q == 0 && active;
  uint64_t acc = 0;
  int nacc = 0;
  int widx = (int)(((long long)i1 * bits) >> 5);

#pragma unroll 1
  for (int c0 = 0; c0 < ncols; c0 += SUB) {
    const int nsub = min(SUB, ncols - c0);
    float w[SLOTS];
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) w[k] = wsm[c0 + LANES * k + q];   // column c0 + LANES k + q (zero-padded)

    const int j0 = i1 + c0;
    if ((j0 % g) == 0) {
      // group statistics over the current weights of columns [j0, j0 + g), each lane over
      // its own columns, then combined across the row's lanes
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < SLOTS; ++k) {
        const int c = LANES * k + q;
        if (c < nsub && c < g) { mn = fminf(mn, w[k]); mx = fmaxf(mx, w[k]); }
      }
      for (int c = c0 + SUB + q; c < ncols && c - c0 < g; c += LANES) {
        const float v = wsm[c];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      for (int c = i1 + ncols + q; c < j0 + g && c < d; c += LANES) {
        const float v = wrow[c];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
#pragma unroll
      for (int o = 1; o < LANES; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      s = fmaxf(div_mk(__fsub_rn(mx, mn), qmax, inv_qmax), 1e-8f);
      inv_s = rcp_rn(s);
      z = fminf(fmaxf(rintf(div_mk(-mn, s, inv_s)), 0.0f), qmax);
      if (active && q == 0) {
        scales[(long long)r * G + j0 / g] = s;
        zeros[(long long)r * G + j0 / g] = z;
      }
    }

#pragma unroll 1
    for (int cb = c0; cb < c0 + nsub; cb += LANES) {   // LANES columns per iteration
#pragma unroll
      for (int i = 0; i < LANES; ++i) {
        const int t = cb + i;
        if (t < ncols) {                                 // warp-uniform
          const float x = __shfl_sync(0xffffffffu, w[0], qbase + i);
          const float qv = fminf(fmaxf(rintf(__fadd_rn(div_mk(x, s, inv_s), z)), 0.0f), qmax);
          const float wq = __fmul_rn(__fsub_rn(qv, z), s);
          const float e = active ? div_mk(__fsub_rn(x, wq), Us[t * BS + t], inv_u[t]) : 0.0f;
          if (q == 0) {
            es[t - c0] = e;
            err[(long long)(r0 + row) * BS + t] = e;
          }
          const uint32_t qi = (uint32_t)qv;
          if (packer) {
            acc |= (uint64_t)qi << nacc;
            nacc += bits;
            if (nacc >= 32) {
              qweight[(long long)r * wpr + widx] = (uint32_t)acc;
              ++widx;
              acc >>= 32;
              nacc -= 32;
            }
          } else if (!natural && q == 0 && active) {
            codes8[(long long)r * d + i1 + t] = (uint8_t)qi;
          }
          // rank-one update of the lane's later columns of the sub-block: slot k holds
          // column cb + LANES k + q, later than t unless k == 0 and q <= i
          const float* urow = Us + t * BS + cb + q;
#pragma unroll
          for (int k = 0; k < SLOTS; ++k)
            if (k > 0 || q > i) w[k] = __fsub_rn(w[k], __fmul_rn(e, urow[LANES * k]));
        }
      }
#pragma unroll
      for (int k = 0; k < SLOTS - 1; ++k) w[k] = w[k + 1];
      w[SLOTS - 1] = 0.0f;
    }
    __syncwarp();
    // the sub-block's errors move the block's later columns (this lane's share), in order
#pragma unroll 1
    for (int c = c0 + SUB + q; c < ncols; c += LANES) {
      float x = wsm[c];
#pragma unroll
      for (int u = 0; u < SUB; ++u)
        if (u < nsub) x = __fsub_rn(x, __fmul_rn(es[u], Us[(c0 + u) * BS + c]));
      wsm[c] = x;
    }
    __syncthreads();
    // per-column loss partial sums of the CTA's 32 rows, in a fixed order
    if (tid < nsub) {
      float lsum = 0.0f;
      for (int rr = 0; rr < ROWS_PER_CTA; ++rr) {
        const float e = Es[rr * ELD + tid];
        lsum = __fadd_rn(lsum, __fmul_rn(__fmul_rn(e, e), 0.5f));
      }
      part[(long long)blockIdx.x * d + i1 + c0 + tid] = lsum;
    }
    __syncthreads();
  }
  if (packer && nacc > 0) qweight[(long long)r * wpr + widx] = (uint32_t)acc;
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

// Ut = Hinv1^T (the lazy update reads Hinv1's rows as K-major operand columns)
__global__ void transpose_kernel(const float* __restrict__ U, float* __restrict__ Ut, int d) {
  __shared__ float tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int r = by + yy, c = bx + threadIdx.x;
    tile[yy][threadIdx.x] = (r < d && c < d) ? U[(long long)r * d + c] : 0.0f;
  }
  __syncthreads();
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int r = bx + yy, c = by + threadIdx.x;
    if (r < d && c < d) Ut[(long long)r * d + c] = tile[threadIdx.x][yy];
  }
}

struct Layout {
  size_t hdr, wf, err, ut, part, codes8, inv, total;
  int nrg;
};

Layout layout(long long m, long long d, int blocksize) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  Layout L;
  L.nrg = (int)((m + ROWS_PER_CTA - 1) / ROWS_PER_CTA);
  const size_t mpad = (size_t)L.nrg * ROWS_PER_CTA;
  L.hdr = 0;
  L.wf = kHeaderBytes;
  L.err = L.wf + al((size_t)m * d * 4);
  L.ut = L.err + al(mpad * (size_t)blocksize * 4);
  L.part = L.ut + al((size_t)d * d * 4);
  L.codes8 = L.part + al((size_t)L.nrg * d * 4);
  L.inv = L.codes8 + al((size_t)m * d);
  L.total = L.inv + al((size_t)d * 4);
  return L;
}

template <int BS>
gptq_status run_blocks(float* Wf, int m, int d, const float* U, const float* Ut, int bits, int g, uint32_t* qweight,
                       int wpr, uint8_t* codes8, float* scales, float* zeros, int G, float* err, float* part,
                       cudaStream_t s) {
  const size_t smem = (size_t)(BS * BS + BS + ROWS_PER_CTA * (BS + 1) + ROWS_PER_CTA * ELD) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(colblock_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(colblock_kernel) failed");
    attr = true;
  }
  const int nrg = (m + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  for (int i1 = 0; i1 < d; i1 += BS) {
    const int nb = std::min(BS, d - i1);
    {
      ProfScope ps("quantize.colblock", s);
      colblock_kernel<BS><<<nrg, CB_THREADS, smem, s>>>(Wf, m, d, U, i1, bits, g, qweight, wpr, codes8, scales,
                                                          zeros, G, err, part);
      count_launch();
    }
    const int i2 = i1 + nb;
    if (i2 < d) {
      // W[:, i2:] -= Err1 @ Hinv1[i1:i2, i2:];  A = Err1 (rows of BS), B(k, j) = Ut[i2 + j][i1 + k]
      simt::GemmArgs ga{};
      ga.M = m; ga.N = d - i2; ga.K = nb; ga.M_last = m; ga.K_last = nb;
      ga.A = err; ga.lda = BS;
      ga.B = Ut + (long long)i2 * d + i1; ga.ldb = d;
      ga.C = Wf + i2; ga.ldc = d;
      ga.alpha = -1.0f; ga.beta = 1.0f;
      ga.vec = (d % 4 == 0) && simt::aligned16(Wf) && simt::aligned16(Ut) && simt::aligned16(err);
      ProfScope ps2("quantize.lazy_gemm", s);
      if (gptq_status st = tc_gemm(ga, 1, true, true, s)) return st;
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
  float* err = reinterpret_cast<float*>(base + L.err);
  float* Ut = reinterpret_cast<float*>(base + L.ut);
  float* part = reinterpret_cast<float*>(base + L.part);
  uint8_t* codes8 = perm ? base + L.codes8 : nullptr;
  int* inv = reinterpret_cast<int*>(base + L.inv);
  const int g = (group_size < 0) ? d : group_size;
  const int G = d / g;
  const int wpr = (int)(((long long)d * bits + 31) / 32);

  if (cudaMemsetAsync(hdr, 0, sizeof(QHeader), s) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaMemsetAsync failed");
  {
    ProfScope ps("quantize.prep", s);
    dim3 grid((unsigned)std::min(8, (d + 255) / 256), (unsigned)std::min(m, 65535));
    prep_kernel<<<grid, 256, 0, s>>>(W, w_dtype, m, d, ldw, perm, Wf, hdr);
    dim3 tg((unsigned)((d + 31) / 32), (unsigned)((d + 31) / 32));
    transpose_kernel<<<tg, dim3(32, 8), 0, s>>>(Hinv1, Ut, d);
    count_launch(2);
  }
  gptq_status st;
  switch (blocksize) {
    case 32: st = run_blocks<32>(Wf, m, d, Hinv1, Ut, bits, g, qweight, wpr, codes8, scales, zeros, G, err, part, s); break;
    case 64: st = run_blocks<64>(Wf, m, d, Hinv1, Ut, bits, g, qweight, wpr, codes8, scales, zeros, G, err, part, s); break;
    default: st = run_blocks<128>(Wf, m, d, Hinv1, Ut, bits, g, qweight, wpr, codes8, scales, zeros, G, err, part, s); break;
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

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
//                      (prep_bf16x8_kernel: bf16 in natural order, 16-byte loads)
//   rowstats_kernel    per-channel mode: scale and zero of every row from W before any update
//   diag_info_kernel   per column: Hinv1[j][j], RN(1 / Hinv1[j][j]) and Hinv1[j][j+1]
//   colblock_kernel<BS, LANES> 8 or 16 lanes per row (32 rows per CTA); the whole
//                      block of each row in registers; Hinv1's diagonal block by bulk
//                      asynchronous copies; group min/max by shuffles; Err1, codes and
//                      per-column loss partials (the CTA's 32 rows in a fixed order)
//                      leave from shared memory at the end of the block
//   transpose_kernel   Ut = Hinv1^T once per call (transpose4_kernel: 16-byte accesses)
//   tc_gemm            lazy update W[:, i2:] -= Err1 @ Hinv1[i1:i2, i2:] on the tensor cores
//                      (3 x TF32, both operands K-major: Err1 rows, Ut rows)
//   loss_finalize      col_losses = sum of partials in a fixed order, un-permuted
//   pack_perm          act-order: gather codes back to the original column order
//
// The quantizer uses correctly rounded quotients (see div_mk) and no fused
// multiply-add, so each step rounds exactly like the listing's float32 arithmetic.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <string>
#include <utility>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();   // tc_gemm.cu

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

// The same for bf16 W in natural order, rows 16-byte aligned: eight columns per thread.
__global__ void prep_bf16x8_kernel(const uint16_t* __restrict__ W, int m, int d, long long ldw, float* __restrict__ Wf,
                                   QHeader* hdr) {
  const int q8 = d >> 3;
  const long long n = (long long)m * q8;
  int bad = 0;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long r = idx / q8;
    const int c = (int)(idx - r * q8) << 3;
    const uint4 v = *reinterpret_cast<const uint4*>(W + r * ldw + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(u[k] << 16);
      f[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) bad |= !isfinite(f[k]);
    float4* dst = reinterpret_cast<float4*>(Wf + r * d + c);
    dst[0] = make_float4(f[0], f[1], f[2], f[3]);
    dst[1] = make_float4(f[4], f[5], f[6], f[7]);
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

// Scale, its reciprocal and zero of one group from the group's min and max: the
// quantizer range of "GPTQ-style round-to-nearest with Hessian weighting", in float32
// with correctly rounded quotients.
__device__ __forceinline__ void group_params(float mn, float mx, float qmax, float inv_qmax, float& s, float& inv_s,
                                             float& z) {
  s = fmaxf(div_mk(__fsub_rn(mx, mn), qmax, inv_qmax), 1e-8f);
  inv_s = __frcp_rn(s);        // the correctly rounded reciprocal, as rcp_rn, without fp64 steps
  z = fminf(fmaxf(rintf(div_mk(-mn, s, inv_s)), 0.0f), qmax);
}

// Per-channel quantization (one group per row): statistics of W before any update,
// one warp per row.
__global__ void rowstats_kernel(const float* __restrict__ Wf, int m, int d, int bits, float* __restrict__ scales,
                                float* __restrict__ zeros) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= m) return;
  const float* row = Wf + (long long)r * d;
  float mn = INFINITY, mx = -INFINITY;
  for (int c = lane; c < d; c += 32) {
    const float v = row[c];
    mn = fminf(mn, v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    const float qmax = (float)((1 << bits) - 1);
    float s, inv_s, z;
    group_params(mn, mx, qmax, rcp_rn(qmax), s, inv_s, z);
    scales[r] = s;
    zeros[r] = z;
  }
}

// Per column j: {Hinv1[j][j], RN(1 / Hinv1[j][j]), Hinv1[j][j+1], 0}
__global__ void diag_info_kernel(const float* __restrict__ U, int d, float4* __restrict__ dinfo) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= d) return;
  const float u = U[(long long)j * d + j];
  dinfo[j] = make_float4(u, rcp_rn(u), (j + 1 < d) ? U[(long long)j * d + j + 1] : 0.0f, 0.0f);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------------
// Column block. LANES lanes per row (8 or 16), 32 / LANES rows per warp, 32 rows per
// CTA.
//
// The block's weights stay in registers for the whole block: lane q of a row holds
// columns KW k + 4 q + j (slot 4 k + j), KW = 4 LANES. Columns are visited in
// KW-column steps; after each step the slots move down by four, so the step's columns
// are always slots 0..3 and the loop body is the same for every step. Later phases
// drop the slots that no longer hold a live column (triangular work).
//
// At column t all lanes of a row hold its current value x and quantize it
// identically; every lane then moves all its slots by -Err1 * Hinv1[t][col]
// (multiply, then subtract: the listing's float32 rounding). The value of column t+1
// is fetched from its owner by a shuffle BEFORE that update and updated locally with
// the same two operations, so the shuffle is off the dependent chain of a column.
//
// Hinv1's diagonal block arrives by bulk asynchronous copies of each row's upper part,
// one mbarrier per step. Errors and codes collect in shared memory and leave at the
// end: Err1 row-major for the lazy update, codes packed into the output bitstream (or
// as bytes for act-order), per-column loss sums over the CTA's rows in a fixed order.
//
// Lanes per row (LANES): 16 for 128-column blocks whose groups start on 64-column
// steps (two rows per warp, 16 warps per CTA, so each scheduler has four warps to hide
// the column chain's latency), else 8. A step of 4 * LANES columns must fit in the
// block, and group statistics are taken at step starts.
template <int LANES> constexpr int cb_threads() { return ROWS_PER_CTA * LANES; }
// Steps per phase: a phase is one inlined copy of the step with a fixed number of live
// slots; with 16 lanes a block has only two steps, so each gets its own.
template <int LANES> constexpr int cb_steps_per_phase() { return LANES >= 16 ? 1 : 2; }

template <int BS, int LANES>
struct CBSmem {
  static constexpr int KW = 4 * LANES;               // columns per step
  static constexpr int ELD = BS + 1;                 // padded row of the error tile
  static constexpr int CLD = BS + 4;                 // padded row of the code tile (bytes)
  static constexpr size_t us = 0;
  static constexpr size_t dinfo = us + sizeof(float) * BS * BS;
  static constexpr size_t es = dinfo + sizeof(float4) * BS;
  static constexpr size_t cs = es + sizeof(float) * ROWS_PER_CTA * ELD;
  static constexpr size_t bars = (cs + ROWS_PER_CTA * CLD + 15) & ~(size_t)15;
  static constexpr size_t flag = bars + sizeof(uint64_t) * (BS / KW);
  static constexpr size_t total = flag + 16;
};

struct CBArgs {
  const float* Wf;
  int m, d;
  const float* U;
  const float4* dinfo;        // {U[j][j], RN(1 / U[j][j]), U[j][j+1], 0}
  int i1, bits, g;
  int stats_given;            // scale/zero of every group precomputed (per-channel)
  uint32_t* qweight;
  int wpr;
  uint8_t* codes8;            // non-null: act-order, codes as bytes in processing order
  float* scales;
  float* zeros;
  int G;
  float* err;                 // Err1 of the current outer block: mpad x eld, row-major
  float* err_lo;              // its low parts (err - err with the 13 low mantissa bits cleared)
  int eld;                    // row stride of err (the outer block width)
  int eoff;                   // this block's first column within err
  float* part;                // loss partials, one row of d per CTA
  int bulk;                   // U rows 16-byte aligned: bulk asynchronous copies
  int vecw;                   // Wf rows 16-byte aligned: vector loads
  int* err_word;
};

template <int NSA, int BS, int LANES>
__device__ __forceinline__ void cb_step(float (&w)[BS / LANES], float& x, int k, int q, int qbase, int row, float s,
                                        float inv_s, float z, float qmax, const float* __restrict__ Us,
                                        const float4* __restrict__ dinfo, float* __restrict__ Es,
                                        uint8_t* __restrict__ Cs) {
  using SL = CBSmem<BS, LANES>;
  constexpr int ELD = SL::ELD, CLD = SL::CLD, KW = SL::KW;
  // Branch-free column bodies, so the scheduler can overlap one column's updates with
  // the next column's shuffle, loads and quantization. Columns past the end of a ragged
  // block, and rows past m, run on dead values whose stores are never read back; their
  // reads stay inside the shared allocation (a row of Us is followed by the next row or
  // by dinfo).
#pragma unroll 1
  for (int i = 0; i < LANES; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = KW * k + 4 * i + j;
      // the next column before this column's update, from its owner
      float nsrc;
      if (j < 3) nsrc = w[j + 1];
      else if constexpr (NSA > 4) nsrc = (i < LANES - 1) ? w[0] : w[4];
      else nsrc = w[0];
      const int nowner = qbase + ((j < 3) ? i : ((i + 1) & (LANES - 1)));
      const float xn_pre = __shfl_sync(0xffffffffu, nsrc, nowner);
      const float* urow = Us + t * BS;
      const float4 di = dinfo[t];                            // U[t][t], 1 / U[t][t], U[t][t+1]
      // quantize, dequantize, error
      const float qv = fminf(fmaxf(rintf(__fadd_rn(div_mk(x, s, inv_s), z)), 0.0f), qmax);
      const float wq = __fmul_rn(__fsub_rn(qv, z), s);
      const float e = div_mk(__fsub_rn(x, wq), di.x, di.y);
      Es[row * ELD + t] = e;                                 // the row's lanes store the same value
      Cs[row * CLD + t] = (uint8_t)(int)qv;
      // move every slot by -e * U[t][col]; slots at or before t are dead and ignored
      const float* ucol = urow + KW * k + 4 * q;
#pragma unroll
      for (int kk = 0; kk < NSA / 4; ++kk) {
        const float4 u4 = *reinterpret_cast<const float4*>(ucol + KW * kk);
        w[4 * kk + 0] = __fsub_rn(w[4 * kk + 0], __fmul_rn(e, u4.x));
        w[4 * kk + 1] = __fsub_rn(w[4 * kk + 1], __fmul_rn(e, u4.y));
        w[4 * kk + 2] = __fsub_rn(w[4 * kk + 2], __fmul_rn(e, u4.z));
        w[4 * kk + 3] = __fsub_rn(w[4 * kk + 3], __fmul_rn(e, u4.w));
      }
      x = __fsub_rn(xn_pre, __fmul_rn(e, di.z));
    }
  }
  // the step is done: its slots retire, the rest move down
#pragma unroll
  for (int sl = 0; sl < NSA - 4; ++sl) w[sl] = w[sl + 4];
}

// Phase P covers steps [SPP P, SPP P + SPP) with the NS - 4 SPP P slots that can still
// hold a live column there.
template <int NS, int SPP, class F, int... P>
__device__ __forceinline__ void for_phases(F&& f, std::integer_sequence<int, P...>) {
  (f(std::integral_constant<int, NS - 4 * SPP * P>{}, SPP * P), ...);
}

template <int BS, int LANES>
__global__ void __launch_bounds__(cb_threads<LANES>(), 1) colblock_kernel(CBArgs a) {
  constexpr int ROWS_PER_WARP = 32 / LANES;
  constexpr int CB_THREADS = cb_threads<LANES>();
  constexpr int SPP = cb_steps_per_phase<LANES>();
  constexpr int KW = 4 * LANES;                      // columns per step
  constexpr int NS = BS / LANES;                     // slots per lane
  constexpr int KS = BS / KW;                        // steps
  static_assert(KS >= 1 && BS % KW == 0, "a block holds whole steps");
  using SL = CBSmem<BS, LANES>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* Us = reinterpret_cast<float*>(smem_raw + SL::us);      // Us[t * BS + c] = Hinv1[i1 + t][i1 + c], c >= t
  float4* dinfo = reinterpret_cast<float4*>(smem_raw + SL::dinfo);
  float* Es = reinterpret_cast<float*>(smem_raw + SL::es);
  uint8_t* Cs = smem_raw + SL::cs;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + SL::bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + SL::flag);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = lane & (LANES - 1), qbase = lane - q;
  const int row = warp * ROWS_PER_WARP + lane / LANES;
  const int r0 = blockIdx.x * ROWS_PER_CTA, r = r0 + row;
  const bool active = r < a.m;
  const int d = a.d, i1 = a.i1;
  const int ncols = min(BS, d - i1);
  const int nks = (ncols + KW - 1) / KW;

  // ---- Hinv1's diagonal block: row t from column (t & ~3) on
  if (tid == 0) {
    *abort_flag = 0;
    if (a.bulk) {
      for (int k = 0; k < KS; ++k) mbar_init(&bars[k], 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (a.bulk) {
    if (warp == 0) {
      if (lane < nks) {
        uint32_t bytes = 0;
        for (int t = KW * lane; t < min(KW * lane + KW, ncols); ++t) bytes += (uint32_t)(ncols - (t & ~3)) * 4u;
        mbar_arrive_expect_tx(&bars[lane], bytes);
      }
      __syncwarp();
      for (int t = lane; t < ncols; t += 32) {
        const int c0 = t & ~3;
        bulk_load(Us + t * BS + c0, a.U + (long long)(i1 + t) * d + i1 + c0, (uint32_t)(ncols - c0) * 4u,
                  &bars[t / KW]);
      }
    }
  } else {
    load_tile<CB_THREADS, BS, BS>(Us, BS, a.U + (long long)i1 * d + i1, d, ncols, ncols);
  }
  // Hinv1 is final before this kernel's stream predecessor starts; W, dinfo and the
  // statistics may come from the kernel just before (and Err1 is still being read by it)
  grid_dep_launch();
  grid_dep_wait();
  for (int t = tid; t < BS; t += CB_THREADS) dinfo[t] = (t < ncols) ? a.dinfo[i1 + t] : make_float4(1.f, 1.f, 0.f, 0.f);

  // ---- the row's block of W into registers: slot 4k + j <- column 16k + 4q + j
  float w[NS];
  {
    const float* wrow = a.Wf + (long long)(active ? r : 0) * d + i1;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const int c = KW * k + 4 * q;
      if (a.vecw && active && c < ncols) {
        const float4 v = *reinterpret_cast<const float4*>(wrow + c);
        w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[4 * k + j] = (active && c + j < ncols) ? wrow[c + j] : 0.0f;
      }
    }
  }

  const float qmax = (float)((1 << a.bits) - 1);
  const float inv_qmax = rcp_rn(qmax);
  float s = 1.0f, inv_s = 1.0f, z = 0.0f;
  if (active && (a.stats_given || (i1 % a.g) != 0)) {   // statistics from an earlier block or precomputed
    s = a.scales[(long long)r * a.G + i1 / a.g];
    z = a.zeros[(long long)r * a.G + i1 / a.g];
    inv_s = rcp_rn(s);
  }
  __syncthreads();                                    // dinfo (and the fallback tile) visible

  float x = __shfl_sync(0xffffffffu, w[0], qbase);    // column 0 (slot 0 of lane 0)

  // One phase: SPP steps of KW columns with NSA live slots per lane (inlined once per
  // phase; the phase's steps share the code).
  auto phase = [&](auto nsa_c, int kbeg) {
    constexpr int NSA = decltype(nsa_c)::value;
#pragma unroll 1
    for (int k = kbeg; k < kbeg + SPP && k < nks; ++k) {
      if (a.bulk) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[k], 0, abort_flag));
        if (!ok && lane == 0) {
          *abort_flag = 1;
          report_device_error(a.err_word, DEVERR_TIMEOUT);
        }
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) return;
      const int j0 = i1 + KW * k;
      if (!a.stats_given && (j0 % a.g) == 0) {
        // the group's current weights: this lane's live slots, then columns beyond the block
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int sl = 0; sl < NSA; ++sl) {
          const int c = KW * (k + sl / 4) + 4 * q + (sl & 3);
          if (c < ncols && c - KW * k < a.g) { mn = fminf(mn, w[sl]); mx = fmaxf(mx, w[sl]); }
        }
        const float* wrow = a.Wf + (long long)(active ? r : 0) * d;
        for (int c = i1 + ncols + q; c < j0 + a.g && c < d; c += LANES) {
          const float v = wrow[c];
          mn = fminf(mn, v);
          mx = fmaxf(mx, v);
        }
#pragma unroll
        for (int o = 1; o < LANES; o <<= 1) {
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        group_params(mn, mx, qmax, inv_qmax, s, inv_s, z);
        if (active && q == 0) {
          a.scales[(long long)r * a.G + j0 / a.g] = s;
          a.zeros[(long long)r * a.G + j0 / a.g] = z;
        }
      }
      cb_step<NSA, BS, LANES>(w, x, k, q, qbase, row, s, inv_s, z, qmax, Us, dinfo, Es, Cs);
    }
  };
  // each phase runs with the slots that can still hold a live column
  for_phases<NS, SPP>(phase, std::make_integer_sequence<int, (KS + SPP - 1) / SPP>{});

  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: copies armed on bars[0, nks) may still be landing in this CTA's
    // shared memory. Warp 0 waits for each of them (bounded) before the CTA exits.
    if (a.bulk && warp == 0 && lane < nks) mbar_wait_bounded(&bars[lane], 0, nullptr);
    __syncwarp();
    return;
  }

  // ---- Err1 out (row-major, BS per row), loss partials, codes
  constexpr int ELD = SL::ELD, CLD = SL::CLD;
  for (int idx = tid; idx < ROWS_PER_CTA * BS; idx += CB_THREADS) {
    const int rr = idx / BS, t = idx % BS;
    if (t < ncols && r0 + rr < a.m) {
      const float e = Es[rr * ELD + t];
      const long long o = (long long)(r0 + rr) * a.eld + a.eoff + t;
      a.err[o] = e;
      a.err_lo[o] = e - __uint_as_float(__float_as_uint(e) & 0xFFFFE000u);
    }
  }
  {
    // per column, LPC adjacent lanes sum RPL rows each, then combine in a fixed order
    constexpr int LPC = (CB_THREADS / BS) < 8 ? (CB_THREADS / BS) : 8;    // 2, 4 or 8
    constexpr int RPL = ROWS_PER_CTA / LPC;
    for (int base = 0; base < BS; base += CB_THREADS / LPC) {
      const int t = base + tid / LPC, part = tid % LPC;
      float lsum = 0.0f;
      if (t < ncols)
        for (int rr = part * RPL; rr < part * RPL + RPL; ++rr) {
          const float e = (r0 + rr < a.m) ? Es[rr * ELD + t] : 0.0f;
          lsum = __fadd_rn(lsum, __fmul_rn(__fmul_rn(e, e), 0.5f));
        }
#pragma unroll
      for (int o = 1; o < LPC; o <<= 1) lsum = __fadd_rn(lsum, __shfl_xor_sync(0xffffffffu, lsum, o));
      if (t < ncols && part == 0) a.part[(long long)blockIdx.x * d + i1 + t] = lsum;
    }
  }
  if (a.codes8) {
    for (int idx = tid; idx < ROWS_PER_CTA * BS; idx += CB_THREADS) {
      const int rr = idx / BS, t = idx % BS;
      if (t < ncols && r0 + rr < a.m) a.codes8[(long long)(r0 + rr) * d + i1 + t] = Cs[rr * CLD + t];
    }
  } else {
    // words [i1 b / 32, ceil((i1 + ncols) b / 32)) of each row; i1 b is a multiple of 32
    const int bits = a.bits;
    const int wb = (int)(((long long)i1 * bits) >> 5);
    const int we = (int)(((long long)(i1 + ncols) * bits + 31) >> 5);
    const int nw = we - wb;
    for (int idx = tid; idx < ROWS_PER_CTA * nw; idx += CB_THREADS) {
      const int rr = idx / nw, wi = wb + idx % nw;
      if (r0 + rr >= a.m) continue;
      const long long b0 = (long long)wi * 32;
      const int jf = (int)(b0 / bits);
      const int jl = min(i1 + ncols - 1, (int)((b0 + 31) / bits));
      uint64_t v = 0;
      for (int j = jf; j <= jl; ++j) {
        const uint64_t code = Cs[rr * CLD + (j - i1)];
        const long long sh = (long long)j * bits - b0;
        v |= (sh >= 0) ? (code << sh) : (code >> (-sh));
      }
      a.qweight[(long long)(r0 + rr) * a.wpr + wi] = (uint32_t)v;
    }
  }
}

// ---------------------------------------------------------------------------------
// Column block with one chain warp per 32 rows: 128-column blocks whose groups start
// on block boundaries (group_size a multiple of 128, or per-channel statistics).
//
// Lane r of warp 0 runs row r's dependent chain once: quantize, dequantize, error and
// the update of the next column. Warps 1-3 and 5-7 (update warps, lane = row too) hold
// the block's quads (4 columns) 4..31 in registers, quad q in update warp
// (q - 4) % 6, and move them by the errors of every finished quad. Warp 4 issues the
// copies and then only waits, so the chain warp has its scheduler to itself (warps w
// and w + 4 share one).
//
// Hand-over: at the start of quad j the chain takes quad j + 1 from the W tile in
// shared memory, where its update warp stored it as soon as it carried the errors of
// quads 0 .. j - 3 (quads 1-3 come straight from the loaded tile); the chain applies
// the errors of quads j - 2 and j - 1 to it (they are still in its registers) and,
// while it works through quad j, each of quad j's errors. An update warp therefore has
// two quads of the chain's time to deliver a quad. Every weight still receives every
// earlier column's correction -- the product rounded, then subtracted -- in column
// order, so a block rounds exactly like the blocked loop in float32.
//
// Errors and codes of a finished quad go to shared memory (one 16-byte and one 4-byte
// store per lane) and an mbarrier per quad tells the update warps; another mbarrier per
// quad hands the updated quad back. Every wait is bounded.
namespace chain {
constexpr int BS = 128;
constexpr int NQ = BS / 4;                 // quads per block
constexpr int THREADS = 256;
constexpr int NUPD = 6;                    // update warps
constexpr int FIRST_UPD = 4;               // first quad held by an update warp
constexpr int NSLOT = (NQ - FIRST_UPD + NUPD - 1) / NUPD;
constexpr int WLD = BS + 4;                // padded rows of the W, error and code tiles (floats)
struct Smem {
  static constexpr size_t us = 0;                                        // Hinv1[i1 + t][i1 + c]
  static constexpr size_t ws = us + sizeof(float) * BS * BS;             // W block, 32 x WLD
  static constexpr size_t es = ws + sizeof(float) * 32 * WLD;            // Err1, 32 x WLD
  static constexpr size_t cs = es + sizeof(float) * 32 * WLD;            // codes (as floats), 32 x WLD
  static constexpr size_t dinfo = cs + sizeof(float) * 32 * WLD;
  static constexpr size_t bars = dinfo + sizeof(float4) * BS;           // W, U x 4, errors x NQ, hand-over x NQ
  static constexpr int NBARS = 1 + 4 + 2 * NQ;
  static constexpr size_t flag = bars + sizeof(uint64_t) * NBARS;
  static constexpr size_t total = flag + 16;
};
static_assert(Smem::dinfo % 16 == 0 && Smem::bars % 8 == 0, "shared-memory layout alignment");

__device__ __forceinline__ float upd(float w, float e, float u) { return __fsub_rn(w, __fmul_rn(e, u)); }

// rint(v) (round half to even) for |v| < 2^22 by adding and removing 1.5 * 2^23: the
// sum lies in [2^23, 2^24), where floats are the integers. Outside that range the value
// differs from rint(v) but stays beyond the same end of [0, 2^b - 1] (b <= 8), so the
// clamped code is the same; two additions instead of a rounding instruction on the
// chain.
__device__ __forceinline__ float rint_small(float v) {
  constexpr float kShift = 12582912.0f;      // 1.5 * 2^23
  return __fsub_rn(__fadd_rn(v, kShift), kShift);
}

// v[k] -= e_i * U[row_i][col + k] for the four rows i of quad `pq`, in row order
__device__ __forceinline__ void apply_quad(float (&v)[4], const float (&e)[4], const float* __restrict__ Us, int pq,
                                          int col) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 u = *reinterpret_cast<const float4*>(Us + (4 * pq + i) * BS + col);
    v[0] = upd(v[0], e[i], u.x);
    v[1] = upd(v[1], e[i], u.y);
    v[2] = upd(v[2], e[i], u.z);
    v[3] = upd(v[3], e[i], u.w);
  }
}
}  // namespace chain

__global__ void __launch_bounds__(chain::THREADS, 1) colchain_kernel(CBArgs a) {
  using namespace chain;
  using SM = chain::Smem;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* Us = reinterpret_cast<float*>(smem_raw + SM::us);
  float* Ws = reinterpret_cast<float*>(smem_raw + SM::ws);
  float* Es = reinterpret_cast<float*>(smem_raw + SM::es);
  float* Qs = reinterpret_cast<float*>(smem_raw + SM::cs);
  float4* dinfo = reinterpret_cast<float4*>(smem_raw + SM::dinfo);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + SM::bars);
  uint64_t* wbar = bars;                      // the W block
  uint64_t* ubar = bars + 1;                  // Hinv1 rows [32k, 32k + 32)
  uint64_t* ebar = bars + 5;                  // errors of quad p are in Es
  uint64_t* hbar = bars + 5 + NQ;             // quad q is back in Ws, ready for the chain
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + SM::flag);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = blockIdx.x * 32, r = r0 + lane;
  const bool active = r < a.m;
  const int d = a.d, i1 = a.i1;
  const int ncols = min(BS, d - i1);          // a multiple of 4 on this path
  const int nq = ncols >> 2;
  const int nrows = min(32, a.m - r0);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(wbar, 1);
    for (int k = 0; k < 4; ++k) mbar_init(&ubar[k], 1);
    for (int q = 0; q < NQ; ++q) {
      mbar_init(&ebar[q], 32);
      mbar_init(&hbar[q], 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // Hinv1's diagonal block, final before this kernel's stream predecessor starts: row t
  // from column t & ~3 on, 32 rows per barrier
  if (warp == 4) {
    if (lane < 4) {
      uint32_t bytes = 0;
      for (int t = 32 * lane; t < min(32 * lane + 32, ncols); ++t) bytes += (uint32_t)(ncols - (t & ~3)) * 4u;
      mbar_arrive_expect_tx(&ubar[lane], bytes);
    }
    __syncwarp();
    for (int t = lane; t < ncols; t += 32) {
      const int c0 = t & ~3;
      bulk_load(Us + t * BS + c0, a.U + (long long)(i1 + t) * d + i1 + c0, (uint32_t)(ncols - c0) * 4u,
                &ubar[t >> 5]);
    }
  }
  // W, dinfo and the statistics may come from the kernel just before (which still reads
  // Err1, written below)
  grid_dep_launch();
  grid_dep_wait();
  if (warp == 4) {
    if (lane == 0) mbar_arrive_expect_tx(wbar, (uint32_t)(nrows * ncols) * 4u);
    __syncwarp();
    if (lane < nrows) bulk_load(Ws + lane * WLD, a.Wf + (long long)(r0 + lane) * d + i1, (uint32_t)ncols * 4u, wbar);
    else
      for (int c = 0; c < BS; c += 4) *reinterpret_cast<float4*>(Ws + lane * WLD + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int t = tid; t < BS; t += THREADS) dinfo[t] = (t < ncols) ? a.dinfo[i1 + t] : make_float4(1.f, 1.f, 0.f, 0.f);
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ the chain warp
    const float qmax = (float)((1 << a.bits) - 1);
    const float inv_qmax = rcp_rn(qmax);
    float s = 1.0f, inv_s = 1.0f, z = 0.0f;
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, abort_flag));
    if (ok) {
      if (a.stats_given || (i1 % a.g) != 0) {          // statistics from an earlier block or precomputed
        if (active) {
          s = a.scales[(long long)r * a.G + i1 / a.g];
          z = a.zeros[(long long)r * a.G + i1 / a.g];
        }
        inv_s = rcp_rn(s);
      } else {
        // the group starts here: min and max of the row's current weights over the group
        float mn = INFINITY, mx = -INFINITY;
        for (int c = 0; c < ncols; c += 4) {
          const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + c);
          mn = fminf(fminf(mn, v.x), fminf(fminf(v.y, v.z), v.w));
          mx = fmaxf(fmaxf(mx, v.x), fmaxf(fmaxf(v.y, v.z), v.w));
        }
        const float* wrow = a.Wf + (long long)(active ? r : 0) * d;
        for (int c = i1 + ncols; c < i1 + a.g && c < d; c += 4) {   // a group wider than the block
          const float4 v = *reinterpret_cast<const float4*>(wrow + c);
          mn = fminf(fminf(mn, v.x), fminf(fminf(v.y, v.z), v.w));
          mx = fmaxf(fmaxf(mx, v.x), fmaxf(fmaxf(v.y, v.z), v.w));
        }
        group_params(mn, mx, qmax, inv_qmax, s, inv_s, z);
        if (active) {
          a.scales[(long long)r * a.G + i1 / a.g] = s;
          a.zeros[(long long)r * a.G + i1 / a.g] = z;
        }
      }
      float cur[4], nxt[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f}, e2[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD);
        cur[0] = v.x; cur[1] = v.y; cur[2] = v.z; cur[3] = v.w;
      }
#pragma unroll 1
      for (int j = 0; j < nq; ++j) {
        // the waits first, so the quad's work below is one straight block of code the
        // compiler can interleave: the chain of each column with the independent updates
        if (j + 1 >= FIRST_UPD && j + 1 < nq) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&hbar[j + 1], 0, abort_flag));
          if (!ok) break;
        }
        if ((j & 7) == 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ubar[j >> 3], 0, abort_flag));
          if (!ok) break;
        }
        // quad j + 1 (past the last quad it reads padding and is never used); the errors
        // of quads j - 2 and j - 1 (zeros, against quad 0's rows, before there are any)
        {
          const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + 4 * (j + 1));
          nxt[0] = v.x; nxt[1] = v.y; nxt[2] = v.z; nxt[3] = v.w;
        }
        apply_quad(nxt, e2, Us, max(j - 2, 0), 4 * (j + 1));
        apply_quad(nxt, e1, Us, max(j - 1, 0), 4 * (j + 1));
        float ec[4], qc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int t = 4 * j + c;
          const float4 di = dinfo[t];                          // U[t][t], 1 / U[t][t]
          const float4 ua = *reinterpret_cast<const float4*>(Us + t * BS + 4 * j);       // this quad
          const float4 ub = *reinterpret_cast<const float4*>(Us + t * BS + 4 * j + 4);   // the next one
          const float x = cur[c];
          const float qv = fminf(fmaxf(rint_small(__fadd_rn(div_mk(x, s, inv_s), z)), 0.0f), qmax);
          const float wq = __fmul_rn(__fsub_rn(qv, z), s);
          const float e = div_mk(__fsub_rn(x, wq), di.x, di.y);
          ec[c] = e;
          qc[c] = qv;
          if (c < 1) cur[1] = upd(cur[1], e, ua.y);
          if (c < 2) cur[2] = upd(cur[2], e, ua.z);
          if (c < 3) cur[3] = upd(cur[3], e, ua.w);
          nxt[0] = upd(nxt[0], e, ub.x);
          nxt[1] = upd(nxt[1], e, ub.y);
          nxt[2] = upd(nxt[2], e, ub.z);
          nxt[3] = upd(nxt[3], e, ub.w);
        }
        *reinterpret_cast<float4*>(Es + lane * WLD + 4 * j) = make_float4(ec[0], ec[1], ec[2], ec[3]);
        *reinterpret_cast<float4*>(Qs + lane * WLD + 4 * j) = make_float4(qc[0], qc[1], qc[2], qc[3]);
        mbar_arrive(&ebar[j]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          e2[k] = e1[k];
          e1[k] = ec[k];
          cur[k] = nxt[k];
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_device_error(a.err_word, DEVERR_TIMEOUT);
    }
  } else if (warp != 4) {
    // ------------------------------------------------------------ update warps
    const int u = (warp < 4) ? warp - 1 : warp - 2;
    const int nslot = (nq - 1 - FIRST_UPD - u >= 0) ? (nq - 1 - FIRST_UPD - u) / NUPD + 1 : 0;
    const int qlast = FIRST_UPD + u + NUPD * (nslot - 1);
    float w[NSLOT][4];
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, abort_flag));
    if (ok && nslot > 0) {
#pragma unroll
      for (int k = 0; k < NSLOT; ++k) {
        if (k < nslot) {
          const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + 4 * (FIRST_UPD + u + NUPD * k));
          w[k][0] = v.x; w[k][1] = v.y; w[k][2] = v.z; w[k][3] = v.w;
        } else {
          w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0.0f;
        }
      }
#pragma unroll 1
      for (int p = 0; p + FIRST_UPD <= qlast; ++p) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ebar[p], 0, abort_flag));
        if (!ok) break;
        if ((p & 7) == 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ubar[p >> 3], 0, abort_flag));
          if (!ok) break;
        }
        float ep[4];
        {
          const float4 v = *reinterpret_cast<const float4*>(Es + lane * WLD + 4 * p);
          ep[0] = v.x; ep[1] = v.y; ep[2] = v.z; ep[3] = v.w;
        }
#pragma unroll
        for (int k = 0; k < NSLOT; ++k) {
          const int q = FIRST_UPD + u + NUPD * k;
          if (k < nslot && q >= p + FIRST_UPD) {
            apply_quad(w[k], ep, Us, p, 4 * q);
            if (q == p + FIRST_UPD) {                        // quad q now carries quads 0..q-4: hand it over
              *reinterpret_cast<float4*>(Ws + lane * WLD + 4 * q) = make_float4(w[k][0], w[k][1], w[k][2], w[k][3]);
              mbar_arrive(&hbar[q]);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_device_error(a.err_word, DEVERR_TIMEOUT);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: the copies armed on wbar and ubar[] may still be landing in this
    // CTA's shared memory. Warp 4 waits for them (bounded) before the CTA exits.
    if (warp == 4) {
      if (lane == 0) mbar_wait_bounded(wbar, 0, nullptr);
      if (lane < 4) mbar_wait_bounded(&ubar[lane], 0, nullptr);
    }
    __syncwarp();
    return;
  }

  // ---- Err1 out (row-major) with its low parts, 16 bytes at a time (the row stride and
  // the block's offset in it are multiples of 4)
  for (int idx = tid; idx < 32 * (BS / 4); idx += THREADS) {
    const int rr = idx / (BS / 4), c = 4 * (idx % (BS / 4));
    if (c < ncols && rr < nrows) {
      const float4 e = *reinterpret_cast<const float4*>(Es + rr * WLD + c);
      const long long o = (long long)(r0 + rr) * a.eld + a.eoff + c;
      *reinterpret_cast<float4*>(a.err + o) = e;
      *reinterpret_cast<float4*>(a.err_lo + o) =
          make_float4(e.x - __uint_as_float(__float_as_uint(e.x) & 0xFFFFE000u),
                      e.y - __uint_as_float(__float_as_uint(e.y) & 0xFFFFE000u),
                      e.z - __uint_as_float(__float_as_uint(e.z) & 0xFFFFE000u),
                      e.w - __uint_as_float(__float_as_uint(e.w) & 0xFFFFE000u));
    }
  }
  {
    // column t = tid / 2: rows 16 h .. 16 h + 15 in order, then the pair's two sums
    const int t = tid >> 1, h = tid & 1;
    float lsum = 0.0f;
    if (t < ncols)
      for (int rr = 16 * h; rr < 16 * h + 16; ++rr) {
        const float e = (rr < nrows) ? Es[rr * WLD + t] : 0.0f;
        lsum = __fadd_rn(lsum, __fmul_rn(__fmul_rn(e, e), 0.5f));
      }
    lsum = __fadd_rn(lsum, __shfl_xor_sync(0xffffffffu, lsum, 1));
    if (t < ncols && h == 0) a.part[(long long)blockIdx.x * d + i1 + t] = lsum;
  }
  auto code_at = [&](int rr, int t) -> uint32_t { return (uint32_t)(int)Qs[rr * WLD + t]; };
  const int bits = a.bits;
  if (a.codes8) {
    for (int idx = tid; idx < 32 * BS; idx += THREADS) {
      const int rr = idx / BS, t = idx % BS;
      if (t < ncols && rr < nrows) a.codes8[(long long)(r0 + rr) * d + i1 + t] = (uint8_t)code_at(rr, t);
    }
  } else if (32 % bits == 0) {
    // 2, 4 and 8 bits: word w of the block holds columns [w cpw, (w + 1) cpw); i1 bits is
    // a multiple of 32 (i1 is a multiple of 128)
    const int cpw = 32 / bits;
    const int nwb = (ncols + cpw - 1) / cpw, wb = (i1 * bits) >> 5;
    for (int idx = tid; idx < 32 * nwb; idx += THREADS) {
      const int rr = idx / nwb, w = idx - rr * nwb;
      if (rr >= nrows) continue;
      uint32_t v = 0;
      for (int k = 0, t = w * cpw; k < cpw && t < ncols; ++k, ++t) v |= code_at(rr, t) << (k * bits);
      a.qweight[(long long)(r0 + rr) * a.wpr + wb + w] = v;
    }
  } else {
    // words [i1 b / 32, ceil((i1 + ncols) b / 32)) of each row (d b < 2^20: int arithmetic)
    const int wb = (i1 * bits) >> 5;
    const int we = ((i1 + ncols) * bits + 31) >> 5;
    const int nw = we - wb;
    for (int idx = tid; idx < 32 * nw; idx += THREADS) {
      const int rr = idx / nw, wi = wb + idx % nw;
      if (rr >= nrows) continue;
      const int b0 = wi * 32;
      const int jf = b0 / bits;
      const int jl = min(i1 + ncols - 1, (b0 + 31) / bits);
      uint64_t v = 0;
      for (int j = jf; j <= jl; ++j) {
        const uint64_t code = code_at(rr, j - i1);
        const int sh = j * bits - b0;
        v |= (sh >= 0) ? (code << sh) : (code >> (-sh));
      }
      a.qweight[(long long)(r0 + rr) * a.wpr + wi] = (uint32_t)v;
    }
  }
}

// ---------------------------------------------------------------------------------
// An outer block on one SM per 32 rows: the chain column block of every 128-column
// block of the outer block, and the lazy updates inside the outer block on this SM's
// own tensor core.
//
// The column loop of a row depends on no other row, so the CTA that owns 32 rows can
// move its rows' later columns itself. After block b it computes, for every later
// 128-column tile t of the outer block, D[c][r] = sum_k Hinv1[i1 + k][tile col c] *
// Err1[r][k] as D = Ut_tile (M = 128 columns, K-major) x Err1^T (N = 32 rows,
// K-major), three TF32 passes (hi lo, lo hi, hi hi) per 32-deep k chunk, two 64-deep
// accumulators per tile added in registers, round to nearest, then W -= D: the same
// products, sums and rounding as the tensor-core lazy update of the two-level scheme.
// Tile b + 1 comes first and goes straight into the chain's shared-memory W tile, so
// the next block starts ~2 us after the chain of this one ends; the other tiles run
// while the next block's chain does (the tensor core is otherwise idle here).
//
// Warps: 0 the chain, 1-3 and 5-7 the update warps (as in colchain_kernel; after a
// block they split Err1 into the hi and lo parts of the MMA's B operand); 4 copies
// Hinv1's first diagonal block and the first W tile, then its lane 0 streams the Ut
// tiles (TMA, 3-stage ring of 32-deep chunks); 8-11 the tensor-memory epilogue (lane
// quadrant = warp % 4; thread = column of a tile); 12 allocates tensor memory and its
// lane 0 issues the MMAs.
//
// Per block b: the W tile (the bulk copy for b = 0, else the epilogue's tile) -> the
// chain, errors written over the consumed quads of the W tile, codes as bytes (two
// buffers by block parity) -> the split into the B operand once the previous block's
// operand is free -> the MMAs of tiles b + 1 .. -> epilogue: tile b + 1 into the W
// tile (held in registers since tile b's turn), Err1, losses and codes of block b,
// then the other tiles (tile b + 2 kept in registers, the rest read-modify-written in
// the fp32 working copy). Every wait is bounded.
namespace mchain {
using chain::BS;
using chain::FIRST_UPD;
using chain::NQ;
using chain::NSLOT;
using chain::NUPD;
using chain::WLD;
constexpr int THREADS = 416;
constexpr int COPY_WARP = 4;
constexpr int EPI_WARP0 = 8;
constexpr int MMA_WARP = 12;
constexpr int NWG = 224;                          // threads of warps 0-3 and 5-7
constexpr int STAGES = 3;
constexpr int NBUF = 4;                           // tensor-memory accumulators, 32 columns each
constexpr uint32_t TMEM_COLS = 128;
constexpr int QLD = BS + 4;                       // padded row of the code tile (bytes)
constexpr uint32_t A_BYTES = 128u * 32u * 4u;     // 128 tile columns x 32 k, one part
constexpr uint32_t STAGE_BYTES = 2u * A_BYTES;    // hi and lo
constexpr uint32_t BOP_BYTES = 32u * BS * 4u;     // 32 rows x 128 k, one part (four 4 KB k chunks)
struct Smem {
  static constexpr size_t us = 0;                                        // Hinv1[i1 + t][i1 + c]
  static constexpr size_t ws = us + sizeof(float) * BS * BS;             // W tile / errors, 32 x WLD
  static constexpr size_t qb = ws + sizeof(float) * 32 * WLD;            // codes, 2 x 32 x QLD bytes
  static constexpr size_t dinfo = qb + 2 * 32 * QLD;
  static constexpr size_t bop = (dinfo + sizeof(float4) * BS + 1023) & ~(size_t)1023;
  static constexpr size_t ring = bop + 2 * BOP_BYTES;
  static constexpr size_t bars = ring + STAGES * STAGE_BYTES;
  // wbar, wready, ubar[4], ebar[NQ], hbar[NQ], bop_full, bop_free, afull/aempty[STAGES],
  // tfull/tempty[NBUF], drain
  static constexpr int NBARS = 2 + 4 + 2 * NQ + 2 + 2 * STAGES + 2 * NBUF + 1;
  static constexpr size_t tslot = bars + sizeof(uint64_t) * NBARS;
  static constexpr size_t flag = tslot + 8;
  static constexpr size_t used = flag + 8;
  static constexpr size_t total = used + 1024;                           // the base is aligned up to 1024
};
static_assert(Smem::dinfo % 16 == 0 && Smem::ring % 1024 == 0 && Smem::bars % 8 == 0, "shared-memory layout");
static_assert(Smem::total <= 232448, "shared memory per CTA");

// byte offset of element (row r, k t) in a 128-byte-swizzled K-major operand of 32 rows
__device__ __forceinline__ uint32_t bop_off(int r, int t) {
  return (uint32_t)((t >> 5) * 4096 + r * 128 + ((((t & 31) >> 2) ^ (r & 7)) << 4) + ((t & 3) << 2));
}
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) { return umma_sdesc_sw128(base + kk * 32, 16, 1024); }
__device__ __forceinline__ void bar_wg() { asm volatile("bar.sync 1, %0;" ::"n"(NWG) : "memory"); }
__device__ __forceinline__ float lo_part(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

struct Args {
  CBArgs a;
  int o1;                     // first column of the outer block
  int nb;                     // 128-column blocks in it
};
}  // namespace mchain

__global__ void __launch_bounds__(mchain::THREADS, 1)
colmma_kernel(const __grid_constant__ CUtensorMap map_ut, const __grid_constant__ CUtensorMap map_utlo,
              const __grid_constant__ CUtensorMap map_u, const mchain::Args p) {
  using namespace mchain;
  using chain::apply_quad;
  using chain::rint_small;
  using chain::upd;
  const CBArgs& a = p.a;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* Us = reinterpret_cast<float*>(sm + Smem::us);
  float* Ws = reinterpret_cast<float*>(sm + Smem::ws);
  uint8_t* Qb = sm + Smem::qb;
  float4* dinfo = reinterpret_cast<float4*>(sm + Smem::dinfo);
  uint8_t* bop = sm + Smem::bop;
  uint8_t* ring = sm + Smem::ring;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::bars);
  uint64_t* wbar = bars;                      // W tile of block 0 (bulk copy)
  uint64_t* wready = bars + 1;                // W tile of block b >= 1 (epilogue), completion b - 1
  uint64_t* ubar = bars + 2;                  // Hinv1's diagonal block and dinfo, completion b
  uint64_t* ebar = ubar + 4;                  // errors of quad p in the W tile, completion b
  uint64_t* hbar = ebar + NQ;                 // quad q handed back to the chain, completion b
  uint64_t* bop_full = hbar + NQ;             // B operand of block b written (NWG arrivals), completion b
  uint64_t* bop_free = bop_full + 1;          // MMAs and epilogue done with block b's operand
  uint64_t* afull = bop_free + 1;
  uint64_t* aempty = afull + STAGES;
  uint64_t* tfull = aempty + STAGES;
  uint64_t* tempty = tfull + NBUF;
  uint64_t* drain = tempty + NBUF;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Smem::tslot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Smem::flag);
  volatile int* last_diag = abort_flag + 1;   // last block whose diagonal block was armed

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = blockIdx.x * 32;
  const int d = a.d, o1 = p.o1, nb = p.nb;
  const int nrows = min(32, a.m - r0);
  auto ncols_of = [&](int b) { return min(BS, d - (o1 + BS * b)); };
  auto fail = [&]() {
    *abort_flag = 1;
    report_device_error(a.err_word, DEVERR_TIMEOUT);
  };

  if (tid == 0) {
    *abort_flag = 0;
    *last_diag = 0;
    mbar_init(wbar, 1);
    mbar_init(wready, 4);
    mbar_init(ubar, 1);
    for (int q = 0; q < NQ; ++q) {
      mbar_init(&ebar[q], 32);
      mbar_init(&hbar[q], 32);
    }
    mbar_init(bop_full, NWG);                 // every converting thread, after its writes
    mbar_init(bop_free, 5);                   // the MMA thread and the four epilogue warps
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&afull[s], 1);
      mbar_init(&aempty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    prefetch_tmap(&map_ut);
    prefetch_tmap(&map_utlo);
    prefetch_tmap(&map_u);
  }
  if (warp == MMA_WARP) tmem_alloc(tslot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tslot;

  // Hinv1's diagonal block of block b (one 128 x 128 TMA box, zeros past d) and its
  // dinfo, by one thread: one request instead of a copy per row (128 row copies took
  // the issuing warp ~4 us); Hinv1 and dinfo are final before this kernel's stream
  // predecessor starts
  auto issue_diag = [&](int b) {
    const int i1 = o1 + BS * b, ncols = ncols_of(b);
    mbar_arrive_expect_tx(ubar, (uint32_t)(BS * BS * 4) + (uint32_t)ncols * 16u);
    tma_load_2d(Us, &map_u, ubar, i1, i1);
    bulk_load(dinfo, a.dinfo + i1, (uint32_t)ncols * 16u, ubar);
    *last_diag = b;
  };
  if (warp == COPY_WARP && lane == 0) issue_diag(0);
  // W and the statistics come from earlier kernels (the outer update before this one)
  grid_dep_launch();
  grid_dep_wait();
  if (warp == COPY_WARP) {
    const int ncols = ncols_of(0);
    if (lane >= nrows)                          // rows past m: zeros, stored before the barrier's arrival
      for (int c = 0; c < BS; c += 4) *reinterpret_cast<float4*>(Ws + lane * WLD + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(wbar, (uint32_t)(nrows * ncols) * 4u);
    __syncwarp();
    if (lane < nrows) bulk_load(Ws + lane * WLD, a.Wf + (long long)(r0 + lane) * d + o1, (uint32_t)ncols * 4u, wbar);
  }

  if (warp < EPI_WARP0 && warp != COPY_WARP) {
    // ------------------------------------------------------------ chain and update warps
    const int wtid = (warp < COPY_WARP) ? tid : tid - 32;     // 0 .. NWG - 1
    const float qmax = (float)((1 << a.bits) - 1);
    const float inv_qmax = rcp_rn(qmax);
    const int r = r0 + lane;
    const bool active = r < a.m;
    // per-channel statistics (precomputed, one group per row): read once, not per block
    float s_row = 1.0f, z_row = 0.0f;
    if (warp == 0 && a.stats_given && active) {
      s_row = a.scales[(long long)r * a.G];
      z_row = a.zeros[(long long)r * a.G];
    }
    const float inv_s_row = rcp_rn(s_row);
    for (int b = 0; b < nb; ++b) {
      const int i1 = o1 + BS * b, ncols = ncols_of(b), nq = ncols >> 2;
      const uint32_t par = (uint32_t)b & 1u;
      uint8_t* Qc = Qb + (b & 1) * 32 * QLD;
      bool ok = __all_sync(0xffffffffu, *abort_flag == 0);
      if (ok) ok = __all_sync(0xffffffffu, b == 0 ? mbar_wait_bounded(wbar, 0, abort_flag)
                                                  : mbar_wait_bounded(wready, (uint32_t)(b - 1) & 1u, abort_flag));
      if (ok && warp == 0) {
        // ---- the chain: row `lane`'s dependent sequence, once per column
        float s = s_row, inv_s = inv_s_row, z = z_row;
        const bool group_start = !a.stats_given;         // groups of 128: every block starts one
        if (group_start) {
          // min and max of the row over the block, four independent running values
          float mn4[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 2
          for (int c = 0; c < ncols; c += 16) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (c + 4 * u < ncols) {
                const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + c + 4 * u);
                mn4[u] = fminf(mn4[u], fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
                mx4[u] = fmaxf(mx4[u], fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
              }
          }
          const float mn = fminf(fminf(mn4[0], mn4[1]), fminf(mn4[2], mn4[3]));
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          group_params(mn, mx, qmax, inv_qmax, s, inv_s, z);
        }
        float cur[4], nxt[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f}, e2[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD);
          cur[0] = v.x; cur[1] = v.y; cur[2] = v.z; cur[3] = v.w;
        }
#pragma unroll 1
        for (int j = 0; j < nq; ++j) {
          if (j + 1 >= FIRST_UPD && j + 1 < nq) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&hbar[j + 1], par, abort_flag));
            if (!ok) break;
          }
          if (j == 0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(ubar, par, abort_flag));
            if (!ok) break;
          }
          {
            const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + 4 * (j + 1));
            nxt[0] = v.x; nxt[1] = v.y; nxt[2] = v.z; nxt[3] = v.w;
          }
          apply_quad(nxt, e2, Us, max(j - 2, 0), 4 * (j + 1));
          apply_quad(nxt, e1, Us, max(j - 1, 0), 4 * (j + 1));
          float ec[4], qc[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int t = 4 * j + c;
            const float4 di = dinfo[t];
            const float4 ua = *reinterpret_cast<const float4*>(Us + t * BS + 4 * j);
            const float4 ub = *reinterpret_cast<const float4*>(Us + t * BS + 4 * j + 4);
            const float x = cur[c];
            const float qv = fminf(fmaxf(rint_small(__fadd_rn(div_mk(x, s, inv_s), z)), 0.0f), qmax);
            const float wq = __fmul_rn(__fsub_rn(qv, z), s);
            const float e = div_mk(__fsub_rn(x, wq), di.x, di.y);
            ec[c] = e;
            qc[c] = qv;
            if (c < 1) cur[1] = upd(cur[1], e, ua.y);
            if (c < 2) cur[2] = upd(cur[2], e, ua.z);
            if (c < 3) cur[3] = upd(cur[3], e, ua.w);
            nxt[0] = upd(nxt[0], e, ub.x);
            nxt[1] = upd(nxt[1], e, ub.y);
            nxt[2] = upd(nxt[2], e, ub.z);
            nxt[3] = upd(nxt[3], e, ub.w);
          }
          // quad j of the W tile is consumed: its errors take its place
          *reinterpret_cast<float4*>(Ws + lane * WLD + 4 * j) = make_float4(ec[0], ec[1], ec[2], ec[3]);
          *reinterpret_cast<uchar4*>(Qc + lane * QLD + 4 * j) =
              make_uchar4((unsigned char)qc[0], (unsigned char)qc[1], (unsigned char)qc[2], (unsigned char)qc[3]);
          mbar_arrive(&ebar[j]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            e2[k] = e1[k];
            e1[k] = ec[k];
            cur[k] = nxt[k];
          }
        }
        // the group's scale and zero leave after the block's chain: a global store issued
        // before it stalled the chain's start while the epilogue warps' stores filled the
        // memory pipeline
        if (group_start && active) {
          a.scales[(long long)r * a.G + i1 / BS] = s;
          a.zeros[(long long)r * a.G + i1 / BS] = z;
        }
      } else if (ok) {
        // ---- update warps: quads FIRST_UPD + u, + NUPD, ... of the row in registers
        const int u = (warp < COPY_WARP) ? warp - 1 : warp - 2;
        const int nslot = (nq - 1 - FIRST_UPD - u >= 0) ? (nq - 1 - FIRST_UPD - u) / NUPD + 1 : 0;
        const int qlast = FIRST_UPD + u + NUPD * (nslot - 1);
        float w[NSLOT][4];
        if (nslot > 0) {
#pragma unroll
          for (int k = 0; k < NSLOT; ++k) {
            if (k < nslot) {
              const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + 4 * (FIRST_UPD + u + NUPD * k));
              w[k][0] = v.x; w[k][1] = v.y; w[k][2] = v.z; w[k][3] = v.w;
            } else {
              w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0.0f;
            }
          }
#pragma unroll 1
          for (int q0 = 0; q0 + FIRST_UPD <= qlast; ++q0) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ebar[q0], par, abort_flag));
            if (!ok) break;
            if (q0 == 0) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(ubar, par, abort_flag));
              if (!ok) break;
            }
            float ep[4];
            {
              const float4 v = *reinterpret_cast<const float4*>(Ws + lane * WLD + 4 * q0);
              ep[0] = v.x; ep[1] = v.y; ep[2] = v.z; ep[3] = v.w;
            }
#pragma unroll
            for (int k = 0; k < NSLOT; ++k) {
              const int q = FIRST_UPD + u + NUPD * k;
              if (k < nslot && q >= q0 + FIRST_UPD) {
                apply_quad(w[k], ep, Us, q0, 4 * q);
                if (q == q0 + FIRST_UPD) {
                  *reinterpret_cast<float4*>(Ws + lane * WLD + 4 * q) = make_float4(w[k][0], w[k][1], w[k][2], w[k][3]);
                  mbar_arrive(&hbar[q]);
                }
              }
            }
          }
        }
      }
      if (!ok && lane == 0 && !*abort_flag) fail();
      bar_wg();                                              // block b done: errors, codes in place
      if (b + 1 < nb && wtid == 32 && !*abort_flag) {
        fence_proxy_async_smem();                            // the diagonal block's reads before the copy
        issue_diag(b + 1);
      }
      // errors -> the MMA operand: hi (the fp32 value; the tensor core reads its tf32
      // part) and lo, 128-byte swizzled, once the previous block's operand is free
      bool okf = !*abort_flag;
      if (okf && b >= 1) okf = mbar_wait_bounded(bop_free, (uint32_t)(b - 1) & 1u, abort_flag);
      if (okf) {
        for (int idx = wtid; idx < 32 * (BS / 4); idx += NWG) {
          const int rr = idx >> 5, t = 4 * (idx & 31);
          const float4 e = *reinterpret_cast<const float4*>(Ws + rr * WLD + t);
          const uint32_t off = bop_off(rr, t);
          *reinterpret_cast<float4*>(bop + off) = e;
          *reinterpret_cast<float4*>(bop + BOP_BYTES + off) =
              make_float4(lo_part(e.x), lo_part(e.y), lo_part(e.z), lo_part(e.w));
        }
        fence_proxy_async_smem();                            // generic writes -> tensor-core reads
      } else if (!*abort_flag) {
        fail();
      }
      // each thread signals its own part (a single arrival after a group barrier reached
      // the MMA warp about 4 us late); the next block's chain cannot overwrite the errors
      // before every part is converted, since its W tile comes after these products
      mbar_arrive(bop_full);
    }
  } else if (warp == COPY_WARP) {
    // ------------------------------------------------------------ Ut tiles (TMA), lane 0
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, last_phase = 0;
      bool ok = true;
      for (int b = 0; ok && b < nb; ++b) {
        const int i1 = o1 + BS * b;
        for (int t = b + 1; ok && t < nb; ++t)
          for (int kc = 0; kc < 4; ++kc) {
            if (!mbar_wait_bounded(&aempty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* dst = ring + stage * STAGE_BYTES;
            mbar_arrive_expect_tx(&afull[stage], STAGE_BYTES);
            tma_load_2d(dst, &map_ut, &afull[stage], i1 + 32 * kc, o1 + BS * t);
            tma_load_2d(dst + A_BYTES, &map_utlo, &afull[stage], i1 + 32 * kc, o1 + BS * t);
            armed |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
      }
      if (!ok && !*abort_flag) fail();
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) mbar_wait_bounded(&afull[s], (last_phase >> s) & 1u, nullptr);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer, lane 0
    // A lean loop: the tensor core holds only a few MMAs in flight, so every cycle the
    // issuing thread spends between stages (warp-wide waits and votes cost ~550 cycles
    // per 12-MMA stage here) is a cycle the tensor pipe idles. Descriptors advance by
    // 32 bytes per k-step: +2 in the 16-byte address field.
    if (lane == 0) {
      constexpr uint32_t IDESC = umma_idesc(/*tf32*/ 2, false, false, 128, 32);
      const uint32_t ring_u = smem_u32(ring), bop_u = smem_u32(bop);
      int stage = 0;
      uint32_t phase = 0, it = 0;
      bool ok = true, issued_any = false;
      for (int b = 0; ok && b < nb; ++b) {
        if (!mbar_wait_poll(bop_full, (uint32_t)b & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool issued = false;
        for (int t = b + 1; ok && t < nb; ++t)
          for (int ch = 0; ok && ch < 2; ++ch) {
            const uint32_t buf = it & (NBUF - 1);
            if (!mbar_wait_bounded(&tempty[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dt = tmem_base + buf * 32u;
            for (int s2 = 0; s2 < 2; ++s2) {
              if (!mbar_wait_bounded(&afull[stage], phase, abort_flag)) {
                ok = false;
                break;
              }
              const uint32_t ah = ring_u + stage * STAGE_BYTES;
              const uint32_t bh = bop_u + (uint32_t)(2 * ch + s2) * 4096u;
              const uint64_t dah = desc_k(ah, 0), dal = desc_k(ah + A_BYTES, 0);
              const uint64_t dbh = desc_k(bh, 0), dbl = desc_k(bh + BOP_BYTES, 0);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                // Ut_lo Err1_hi, Ut_hi Err1_lo, Ut_hi Err1_hi: the order of the tensor-core
                // lazy update's three passes (Err1_hi Ut_lo, Err1_lo Ut_hi, Err1_hi Ut_hi)
                umma_tf32(dt, dal + 2 * kk, dbh + 2 * kk, IDESC, (s2 > 0 || kk > 0) ? 1u : 0u);
                umma_tf32(dt, dah + 2 * kk, dbl + 2 * kk, IDESC, 1u);
                umma_tf32(dt, dah + 2 * kk, dbh + 2 * kk, IDESC, 1u);
              }
              umma_commit(&aempty[stage]);
              issued = true;
              if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            umma_commit(&tfull[buf]);
            ++it;
          }
        if (!ok) break;
        if (issued) umma_commit(bop_free);          // arrives when this block's products are done
        else mbar_arrive(bop_free);
        issued_any |= issued;
      }
      if (!ok && !*abort_flag) fail();
      if (issued_any) {
        umma_commit(drain);
        mbar_wait_bounded(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ tensor-memory epilogue
    const int e = warp - EPI_WARP0;                        // lane quadrant (== warp % 4)
    const int etid = tid - EPI_WARP0 * 32;                 // 0 .. 127
    const int c = 32 * e + lane;                           // column within a tile
    const uint32_t taddr = tmem_base + ((uint32_t)(32 * e) << 16);
    uint32_t it = 0;
    bool ok = true;
    float rn[32];                                          // the next block's W tile column
    if (nb > 1) {
      const int col = o1 + BS + c;
#pragma unroll
      for (int rr = 0; rr < 32; ++rr)
        rn[rr] = (rr < nrows && col < d) ? __ldcg(a.Wf + (long long)(r0 + rr) * d + col) : 0.0f;
    }
    // Err1 with its low parts, the loss partials and the codes of block b
    auto block_out = [&](int b) {
      const int i1 = o1 + BS * b, ncols = ncols_of(b);
      if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(bop_full, (uint32_t)b & 1u, abort_flag))) {
        ok = false;
        if (!*abort_flag) fail();
      }
      if (!ok) return;
      if (c < ncols) {
        const long long o = (long long)r0 * a.eld + (i1 - o1) + c;
        float l[2] = {0.0f, 0.0f};
        // 16 rows at a time: all shared-memory reads before the global stores, which the
        // compiler cannot move them across
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float hv[16], lv[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint32_t off = bop_off(16 * h + k, c);
            hv[k] = *reinterpret_cast<const float*>(bop + off);
            lv[k] = *reinterpret_cast<const float*>(bop + BOP_BYTES + off);
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int rr = 16 * h + k;
            if (rr < nrows) {
              a.err[o + (long long)rr * a.eld] = hv[k];
              a.err_lo[o + (long long)rr * a.eld] = lv[k];
              l[h] = __fadd_rn(l[h], __fmul_rn(__fmul_rn(hv[k], hv[k]), 0.5f));
            }
          }
        }
        a.part[(long long)blockIdx.x * d + i1 + c] = __fadd_rn(l[0], l[1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bop_free);
      const uint8_t* Qc = Qb + (b & 1) * 32 * QLD;
      const int bits = a.bits;
      if (a.codes8) {
        for (int idx = etid; idx < 32 * BS; idx += 128) {
          const int rr = idx / BS, t = idx % BS;
          if (t < ncols && rr < nrows) a.codes8[(long long)(r0 + rr) * d + i1 + t] = Qc[rr * QLD + t];
        }
      } else if (32 % bits == 0) {
        const int cpw = 32 / bits;
        const int nwb = (ncols + cpw - 1) / cpw, wb = (i1 * bits) >> 5;
        for (int idx = etid; idx < 32 * nwb; idx += 128) {
          const int rr = idx / nwb, w = idx - rr * nwb;
          if (rr >= nrows) continue;
          uint32_t v = 0;
          for (int k = 0, t = w * cpw; k < cpw && t < ncols; ++k, ++t) v |= (uint32_t)Qc[rr * QLD + t] << (k * bits);
          a.qweight[(long long)(r0 + rr) * a.wpr + wb + w] = v;
        }
      } else {
        const int wb = (i1 * bits) >> 5;
        const int we = ((i1 + ncols) * bits + 31) >> 5;
        const int nw = we - wb;
        for (int idx = etid; idx < 32 * nw; idx += 128) {
          const int rr = idx / nw, wi = wb + idx % nw;
          if (rr >= nrows) continue;
          const int b0 = wi * 32;
          const int jf = b0 / bits;
          const int jl = min(i1 + ncols - 1, (b0 + 31) / bits);
          uint64_t v = 0;
          for (int j = jf; j <= jl; ++j) {
            const uint64_t code = Qc[rr * QLD + (j - i1)];
            const int sh = j * bits - b0;
            v |= (sh >= 0) ? (code << sh) : (code >> (-sh));
          }
          a.qweight[(long long)(r0 + rr) * a.wpr + wi] = (uint32_t)v;
        }
      }
    };
    for (int b = 0; ok && b < nb; ++b) {
      for (int t = b + 1; ok && t < nb; ++t) {
        float acc[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const uint32_t buf = it % NBUF;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tfull[buf], (it / NBUF) & 1u, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          float v[32];
          tmem_ld_32x32b_x32(taddr + buf * 32u, v);
#pragma unroll
          for (int rr = 0; rr < 32; ++rr) acc[rr] = (ch == 0) ? v[rr] : __fadd_rn(acc[rr], v[rr]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
          ++it;
        }
        if (!ok) {
          if (!*abort_flag) fail();
          break;
        }
        const int col = o1 + BS * t + c;
        if (t == b + 1) {
          // the next block's W tile: its column c, all 32 rows
#pragma unroll
          for (int rr = 0; rr < 32; ++rr) Ws[rr * WLD + c] = __fsub_rn(rn[rr], acc[rr]);
          __syncwarp();
          if (lane == 0) mbar_arrive(wready);
          block_out(b);
        } else {
          // 16 rows at a time: all loads in flight before any store (a store between
          // them would keep the compiler from moving the next load above it)
          float* wcol = const_cast<float*>(a.Wf) + (long long)r0 * d + col;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int rr = 16 * h + k;
              x[k] = (rr < nrows && col < d) ? __ldcg(wcol + (long long)rr * d) : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int rr = 16 * h + k;
              if (t == b + 2) {
                rn[rr] = __fsub_rn(x[k], acc[rr]);                     // the next critical tile
              } else if (rr < nrows && col < d) {
                __stcg(wcol + (long long)rr * d, __fsub_rn(x[k], acc[rr]));
              }
            }
          }
        }
      }
      if (ok && b == nb - 1) block_out(b);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: wait (bounded) for the copies still landing in shared memory
    if (warp == COPY_WARP && lane == 0) mbar_wait_bounded(wbar, 0, nullptr);
    if (warp == 1 && lane == 0) mbar_wait_bounded(ubar, (uint32_t)*last_diag & 1u, nullptr);
  }
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// col_losses[j] = sum over the CTAs' partials: 32 columns per CTA, the 8 warps each sum
// every 8th partial, then warp 0 adds the 8 sums (fixed order)
__global__ void loss_finalize_kernel(const float* __restrict__ part, int nrg, int d, const int* __restrict__ perm,
                                     float* __restrict__ col_losses) {
  __shared__ float acc[8][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (j < d)
    for (int b = w; b < nrg; b += 8) s += part[(long long)b * d + j];
  acc[w][lane] = s;
  __syncthreads();
  if (w == 0 && j < d) {
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += acc[k][lane];
    col_losses[perm ? perm[j] : j] = t;
  }
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

// The same for d % 4 == 0 and 16-byte aligned rows: 32 x 32 tiles, one 16-byte load and
// two 16-byte stores per thread (256 threads: 32 rows x 8 pieces of four).
__global__ void transpose4_kernel(const float* __restrict__ U, float* __restrict__ Ut, float* __restrict__ Ut_lo,
                                  int d) {
  __shared__ float tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  if (bx + 31 < by) return;     // Ut rows bx.., columns by..: above the diagonal, never read
  const int r = threadIdx.x >> 3, c4 = (threadIdx.x & 7) * 4;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (by + r < d && bx + c4 < d) v = *reinterpret_cast<const float4*>(U + (long long)(by + r) * d + bx + c4);
  tile[r][c4] = v.x; tile[r][c4 + 1] = v.y; tile[r][c4 + 2] = v.z; tile[r][c4 + 3] = v.w;
  __syncthreads();
  // output row bx + r, columns by + c4 .. + 3 = input column bx + r of rows by + c4 ..
  if (bx + r < d && by + c4 < d) {
    const float4 o = make_float4(tile[c4][r], tile[c4 + 1][r], tile[c4 + 2][r], tile[c4 + 3][r]);
    const long long off = (long long)(bx + r) * d + by + c4;
    *reinterpret_cast<float4*>(Ut + off) = o;
    *reinterpret_cast<float4*>(Ut_lo + off) =
        make_float4(o.x - __uint_as_float(__float_as_uint(o.x) & 0xFFFFE000u),
                    o.y - __uint_as_float(__float_as_uint(o.y) & 0xFFFFE000u),
                    o.z - __uint_as_float(__float_as_uint(o.z) & 0xFFFFE000u),
                    o.w - __uint_as_float(__float_as_uint(o.w) & 0xFFFFE000u));
  }
}

// Ut = Hinv1^T (the lazy update reads Hinv1's rows as K-major operand columns) and
// its low parts Ut_lo = Ut - Ut with the 13 low mantissa bits cleared. Hinv1 is upper
// triangular and every lazy update reads Ut[c][k] with c beyond the k block (the
// columns right of it), so only the 32 x 32 tiles on and below the diagonal are written.
__global__ void transpose_kernel(const float* __restrict__ U, float* __restrict__ Ut, float* __restrict__ Ut_lo,
                                 int d) {
  __shared__ float tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  if (bx + 31 < by) return;     // Ut rows bx.., columns by..: above the diagonal, never read
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int r = by + yy, c = bx + threadIdx.x;
    tile[yy][threadIdx.x] = (r < d && c < d) ? U[(long long)r * d + c] : 0.0f;
  }
  __syncthreads();
  for (int yy = threadIdx.y; yy < 32; yy += 8) {
    const int r = bx + yy, c = by + threadIdx.x;
    if (r < d && c < d) {
      const float x = tile[threadIdx.x][yy];
      Ut[(long long)r * d + c] = x;
      Ut_lo[(long long)r * d + c] = x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    }
  }
}

// The lazy update is blocked on two levels. After a block of BS columns, only the
// columns up to the end of its outer block of OUTER columns move (K = BS); after an
// outer block, every column right of it moves at once by Err1 of the whole outer block
// (K = OUTER). In exact arithmetic this is the pages' update, W[:, i2:] -= Err1 @
// Hinv1[i1:i2, i2:] after every block, summed in another order: each column still
// receives every earlier column's correction before it is quantized, and a group's
// columns are current when its statistics are read, because an outer block holds
// whole groups. The wide products read and write W's right part once per outer block
// instead of once per block.
// 640 = five 128-column blocks: every K = BS update after a block then has at most
// 4 x 128 columns, one round of 128 x 128 tiles on the GPU at m = 4096 (with 1024, the
// first three of seven took two rounds), for some more K = OUTER work.
constexpr int OUTER = 640;

// Outer block width: OUTER when it holds whole blocks and whole groups, else one block.
inline int outer_width(int BS, int g, int stats_given) {
  const bool groups_fit = stats_given || (g > 0 && OUTER % g == 0);
  return (OUTER % BS == 0 && groups_fit) ? OUTER : BS;
}

struct Layout {
  size_t hdr, wf, err, errlo, ut, utlo, part, codes8, inv, dinfo, total;
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
  L.errlo = L.err + al(mpad * (size_t)std::max(OUTER, blocksize) * 4);
  L.ut = L.errlo + al(mpad * (size_t)std::max(OUTER, blocksize) * 4);
  L.utlo = L.ut + al((size_t)d * d * 4);
  L.part = L.utlo + al((size_t)d * d * 4);
  L.codes8 = L.part + al((size_t)L.nrg * d * 4);
  L.inv = L.codes8 + al((size_t)m * d);
  L.dinfo = L.inv + al((size_t)d * 4);
  L.total = L.dinfo + al((size_t)d * 16);
  return L;
}

// W[:, c0:c1] -= Err1[:, e0:e0+K] @ Hinv1[k0:k0+K, c0:c1] on the tensor cores (Err1
// row-major with row stride a.eld; B(k, j) = Ut[c0 + j][k0 + k])
gptq_status lazy_update(const CBArgs& a, const float* Ut, const float* Ut_lo, int e0, int k0, int K, int c0, int c1,
                        cudaStream_t s) {
  const int m = a.m, d = a.d;
  simt::GemmArgs ga{};
  ga.M = m; ga.N = c1 - c0; ga.K = K; ga.M_last = m; ga.K_last = K;
  ga.A = a.err + e0; ga.lda = a.eld;
  ga.B = Ut + (long long)c0 * d + k0; ga.ldb = d;
  ga.A_lo = a.err_lo + e0; ga.lda_lo = a.eld;
  ga.B_lo = Ut_lo + (long long)c0 * d + k0; ga.ldb_lo = d;
  ga.C = const_cast<float*>(a.Wf) + c0; ga.ldc = d;
  ga.alpha = -1.0f; ga.beta = 1.0f;
  ga.vec = (d % 4 == 0) && simt::aligned16(a.Wf) && simt::aligned16(Ut) && simt::aligned16(a.err);
  ga.b_final = 1;             // Ut is written once, before the first column block
  ProfScope ps("quantize.lazy_gemm", s);
  return tc_gemm(ga, 1, true, true, s);
}

// Every block of BS columns: the column-block kernel (`kernel`, `threads` threads and
// `smem` bytes of dynamic shared memory per CTA of 32 rows), then the lazy updates.
gptq_status run_blocks(void (*kernel)(CBArgs), int threads, size_t smem, int BS, CBArgs a, const float* Ut,
                       const float* Ut_lo, cudaStream_t s) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(column-block kernel) failed");
  const int d = a.d;
  const int nrg = (a.m + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  const int OB = outer_width(BS, a.g, a.stats_given);
  a.eld = OB;
  auto lazy = [&](int e0, int k0, int K, int c0, int c1) { return lazy_update(a, Ut, Ut_lo, e0, k0, K, c0, c1, s); };
  for (int o1 = 0; o1 < d; o1 += OB) {
    const int o2 = std::min(o1 + OB, d);
    for (int i1 = o1; i1 < o2; i1 += BS) {
      const int nb = std::min(BS, o2 - i1), i2 = i1 + nb;
      a.i1 = i1;
      a.eoff = i1 - o1;
      {
        ProfScope ps("quantize.colblock", s);
        if (launch_pdl(kernel, dim3(nrg), dim3(threads), smem, s, a) != cudaSuccess)
          return check_launch("column-block kernel");
        count_launch();
      }
      if (i2 < o2)   // the rest of this outer block
        if (gptq_status st = lazy(i1 - o1, i1, nb, i2, o2)) return st;
    }
    if (o2 < d)      // everything right of the outer block
      if (gptq_status st = lazy(0, o1, o2 - o1, o2, d)) return st;
  }
  return check_launch("column-loop kernels");
}

template <int BS, int LANES>
gptq_status run_blocks_lanes(CBArgs a, const float* Ut, const float* Ut_lo, cudaStream_t s) {
  return run_blocks(colblock_kernel<BS, LANES>, cb_threads<LANES>(), CBSmem<BS, LANES>::total, BS, a, Ut, Ut_lo, s);
}

// 2-D map over Ut (d x d fp32, row-major): boxes of 32 k x 128 rows, 128-byte swizzle,
// rows past d read as zeros
bool make_ut_map(CUtensorMap* map, const float* base, int d, uint32_t box_inner = 32,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)d};
  cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  cuuint32_t box[2] = {box_inner, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 128-column blocks, groups of 128 or per-channel: one colmma_kernel launch per outer
// block (the blocks and the lazy updates inside it), then the update of everything
// right of the outer block.
gptq_status run_outer_blocks(CBArgs a, const float* Ut, const float* Ut_lo, cudaStream_t s) {
  using namespace mchain;
  if (cudaFuncSetAttribute(colmma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem::total) !=
      cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(colmma_kernel) failed");
  CUtensorMap mu, mul, mh;
  // Ut and its low parts: 32-deep k chunks of 128 rows, swizzled for the MMA; Hinv1:
  // the 128 x 128 diagonal block as plain rows
  if (!make_ut_map(&mu, Ut, a.d) || !make_ut_map(&mul, Ut_lo, a.d) ||
      !make_ut_map(&mh, a.U, a.d, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return set_error(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for Hinv1");
  const int d = a.d;
  const int nrg = (a.m + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  const int OB = outer_width(BS, a.g, a.stats_given);
  a.eld = OB;
  for (int o1 = 0; o1 < d; o1 += OB) {
    const int o2 = std::min(o1 + OB, d);
    Args p{a, o1, (o2 - o1 + BS - 1) / BS};
    {
      ProfScope ps("quantize.colblock", s);
      if (launch_pdl(colmma_kernel, dim3(nrg), dim3(THREADS), Smem::total, s, mu, mul, mh, p) != cudaSuccess)
        return check_launch("colmma_kernel");
      count_launch();
    }
    if (o2 < d)
      if (gptq_status st = lazy_update(a, Ut, Ut_lo, 0, o1, o2 - o1, o2, d, s)) return st;
  }
  return check_launch("column-loop kernels");
}

// GPTQ_COLUMN_KERNEL=chain selects the per-block chain kernel with the lazy updates as
// separate tensor-core GEMMs for every configuration that kernel serves.
static bool prefer_chain_kernel() {
  static const bool f = [] {
    const char* v = getenv("GPTQ_COLUMN_KERNEL");
    return v && std::string(v) == "chain";
  }();
  return f;
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
  float* err_lo = reinterpret_cast<float*>(base + L.errlo);
  float* Ut = reinterpret_cast<float*>(base + L.ut);
  float* Ut_lo = reinterpret_cast<float*>(base + L.utlo);
  float* part = reinterpret_cast<float*>(base + L.part);
  uint8_t* codes8 = perm ? base + L.codes8 : nullptr;
  int* inv = reinterpret_cast<int*>(base + L.inv);
  float4* dinfo = reinterpret_cast<float4*>(base + L.dinfo);
  const int g = (group_size < 0) ? d : group_size;
  const int G = d / g;
  const int wpr = (int)(((long long)d * bits + 31) / 32);

  if (cudaMemsetAsync(hdr, 0, sizeof(QHeader), s) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "cudaMemsetAsync failed");
  {
    ProfScope ps("quantize.prep", s);
    if (!perm && w_dtype == 1 && d % 8 == 0 && ldw % 8 == 0 && simt::aligned16(W) && simt::aligned16(Wf)) {
      prep_bf16x8_kernel<<<8 * sm_count(), 256, 0, s>>>(reinterpret_cast<const uint16_t*>(W), m, d, ldw, Wf, hdr);
    } else {
      dim3 grid((unsigned)std::min(8, (d + 255) / 256), (unsigned)std::min(m, 65535));
      prep_kernel<<<grid, 256, 0, s>>>(W, w_dtype, m, d, ldw, perm, Wf, hdr);
    }
    dim3 tg((unsigned)((d + 31) / 32), (unsigned)((d + 31) / 32));
    if (d % 4 == 0 && simt::aligned16(Hinv1) && simt::aligned16(Ut) && simt::aligned16(Ut_lo))
      transpose4_kernel<<<tg, 256, 0, s>>>(Hinv1, Ut, Ut_lo, d);
    else
      transpose_kernel<<<tg, dim3(32, 8), 0, s>>>(Hinv1, Ut, Ut_lo, d);
    diag_info_kernel<<<(d + 255) / 256, 256, 0, s>>>(Hinv1, d, dinfo);
    count_launch(3);
    if (group_size < 0) {
      rowstats_kernel<<<(m + 7) / 8, 256, 0, s>>>(Wf, m, d, bits, scales, zeros);
      count_launch();
    }
  }
  CBArgs a{};
  a.Wf = Wf; a.m = m; a.d = d; a.U = Hinv1; a.dinfo = dinfo;
  a.bits = bits; a.g = g; a.stats_given = group_size < 0;
  a.qweight = qweight; a.wpr = wpr; a.codes8 = codes8;
  a.scales = scales; a.zeros = zeros; a.G = G;
  a.err = err; a.err_lo = err_lo; a.part = part;
  a.bulk = (d % 4 == 0) && simt::aligned16(Hinv1);
  a.vecw = (d % 4 == 0) && simt::aligned16(Wf);
  a.err_word = device_error_word();
  gptq_status st;
  switch (blocksize) {
    case 32: st = run_blocks_lanes<32, 8>(a, Ut, Ut_lo, s); break;
    case 64: st = run_blocks_lanes<64, 8>(a, Ut, Ut_lo, s); break;
    default:
      if ((a.stats_given || g == 128) && a.bulk && a.vecw && tc_gemm_available() && !prefer_chain_kernel())
        // one launch per outer block, its lazy updates on each SM's own tensor core
        st = run_outer_blocks(a, Ut, Ut_lo, s);
      else if ((a.stats_given || g % 128 == 0) && a.bulk && a.vecw)
        // groups start on block boundaries: one chain warp per 32 rows
        st = run_blocks(colchain_kernel, chain::THREADS, chain::Smem::total, 128, a, Ut, Ut_lo, s);
      else if (a.stats_given || g % 64 == 0)   // 64-column steps need groups that start on them
        st = run_blocks_lanes<128, 16>(a, Ut, Ut_lo, s);
      else
        st = run_blocks_lanes<128, 8>(a, Ut, Ut_lo, s);
      break;
  }
  if (st) return st;
  loss_finalize_kernel<<<(d + 31) / 32, 256, 0, s>>>(part, L.nrg, d, perm, col_losses);
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

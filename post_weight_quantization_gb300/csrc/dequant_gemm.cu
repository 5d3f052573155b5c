// The stored layer used on many tokens: Y = X W_hat^T on the 5th-generation tensor cores,
// straight from the packed codes ("GPTQ: fixing errors as you go": once quantized, the
// stored low-bit weights with one scale and zero per group stand in for the layer's
// weights), and the propagation of calibration inputs through a quantized layer when
// layers are quantized one after another ("The GPTQ Algorithm", procedure steps 1-4).
//
//   w_hat[r][j] = (code[r][j] - zero[r][g]) * scale[r][g],   g = j / group_size
//   Y[t][r]     = sum_g scale[r][g] * sum_{j in g} X[t][j] * (code[r][j] - zero[r][g])
//
// code - zero is an integer in [-255, 255], exact in bf16, and X is bf16, so every
// product is exact in fp32 and the tensor core (kind::f16, bf16 operands, fp32
// accumulation) forms each group's partial sum from exact products. The partial leaves
// tensor memory at the end of every group and is added, times the group's scale, into
// fp32 registers; no operand is rounded to a lower precision than the stored layer.
//
// Kernels:
//   dq_int_kernel        B[r][j] = bf16(code[r][j] - zero[r][j / group_size]) into the
//                        caller's workspace (m x d bf16, one pass over the packed layer)
//   dequant_gemm_kernel  persistent, one CTA per SM, 128 x 256 output tiles (tokens x
//                        rows), token tiles outer so the tiles in flight share X's rows
//     warp 0      TMA producer: 64-deep k stages of X and B (128-byte swizzle), 4-stage ring
//     warp 1      MMA issuer: tcgen05.mma kind::f16, M = 128, N = 256, K = 16 (at N = 128
//                 the same products ran at a third of the rate on this GPU); one
//                 tensor-memory buffer per group unit (units of at most 256 columns
//                 inside a group), two buffers rotate
//     warps 2-9   epilogue: per unit, 128 accumulator columns per thread, times the
//                 unit's scales (staged per warp in shared memory), added in fp32;
//                 at the end of a tile each thread writes its token's 128 outputs as
//                 16-byte stores (fp32, or bf16 rounded to nearest even)
// Every wait is bounded; a timeout raises the device error word.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"

namespace gptq {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();   // tc_gemm.cu

namespace dqg {

constexpr int BM = 128, BN = 256, BK = 64;      // BK bf16 = 128 bytes: one swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB of X per stage
constexpr int B_BYTES = BN * BK * 2;            // 32 KB of the integer operand per stage
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NEPI = 8;
constexpr int EPI_WARP0 = 2;
constexpr int THREADS = (EPI_WARP0 + NEPI) * 32;
constexpr int NBUF = 2;
constexpr uint32_t TMEM_COLS = NBUF * BN;
constexpr int EPI_COLS = BN / 2;                // accumulator columns per epilogue thread
constexpr int SC_BYTES = NEPI * EPI_COLS * 4;   // one unit's scales per epilogue warp
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + SC_BYTES;

struct Params {
  int T, m, d;
  int mt, nt;             // token tiles, row tiles
  int unit;               // columns per tensor-memory unit (divides the group size)
  int upg;                // units per group
  int gs, G;              // group size (d for per-channel), groups per row
  const float* scales;
  float* Y;
  long long ldy;
  int y_bf16;
};

// B[r][j] = bf16(code - zero), eight columns per thread (d % 8 == 0).
__global__ void dq_int_kernel(const uint32_t* __restrict__ qweight, const float* __restrict__ zeros, int m, int d,
                              int bits, int gs, int G, int wpr, __nv_bfloat16* __restrict__ B) {
  const long long n8 = (long long)m * (d >> 3);
  const uint32_t mask = (1u << bits) - 1u;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n8;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / (d >> 3));
    const int j0 = (int)(idx - (long long)r * (d >> 3)) << 3;
    const uint32_t* row = qweight + (long long)r * wpr;
    const int p0 = j0 * bits, w0 = p0 >> 5, off = p0 & 31;
    uint64_t win = row[w0];
    if (w0 + 1 < wpr) win |= (uint64_t)row[w0 + 1] << 32;
    win >>= off;                        // 8 codes of at most 8 bits fit in the 64-bit window
    const float z = zeros[(long long)r * G + j0 / gs];
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = __float2bfloat16_rn((float)((uint32_t)(win >> (k * bits)) & mask) - z);
    *reinterpret_cast<uint4*>(B + (long long)r * d + j0) = *reinterpret_cast<const uint4*>(o);
  }
}

// K-major SW128 shared-memory descriptor (both operands): rows of 128 bytes along k,
// 8-row groups 1024 B apart; k-step kk of 16 bf16 (32 bytes) inside the swizzle row.
// (An MN-major integer operand, tried, ran no faster.)
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) { return umma_sdesc_sw128(base + kk * 32, 16, 1024); }

__global__ void __launch_bounds__(THREADS, 1)
dequant_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b, Params p,
                    int* __restrict__ err_word) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tmem_full = empty + STAGES;
  uint64_t* tmem_empty = tmem_full + NBUF;
  uint64_t* drain = tmem_empty + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sc_stage = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);      // NEPI x EPI_COLS

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], NEPI);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_x);
    prefetch_tmap(&map_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();                               // X and B come from earlier kernels
  const int ntiles = p.mt * p.nt;
  const int nstages = (p.d + BK - 1) / BK;       // k stages per tile
  const int nunits = p.d / p.unit;               // tensor-memory units per tile
  constexpr uint32_t IDESC = umma_idesc(/*bf16*/ 1, false, false, BM, BN);

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0, armed = 0, last_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      const int I = t / p.nt, J = t - I * p.nt;
      for (int ks = 0; ks < nstages; ++ks) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        tma_load_2d(sa, &map_x, &full[stage], ks * BK, I * BM);
        tma_load_2d(sa + A_BYTES, &map_b, &full[stage], ks * BK, J * BN);
        armed |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, nullptr);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0, it = 0;
    bool ok = true, issued = false;
    const uint32_t sbase = smem_u32(smem);
    // This one thread paces the pipeline: no division or modulo by a runtime value in
    // its loop (each is a long dependent instruction sequence); positions are counted.
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      int k = 0;                                   // next k of the tile
      int kin = 0;                                 // columns of the current unit issued so far
      for (int ks = 0; ok && ks < nstages; ++ks) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a = sbase + stage * STAGE_BYTES, b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk, k += 16) {
          if (k >= p.d) break;                     // d % 32 == 0: the last stage may hold 32 columns
          const uint32_t buf = it % NBUF;
          if (kin == 0) {
            if (!mbar_wait_bounded(&tmem_empty[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          umma_f16(tmem_base + buf * BN, desc_k(a, kk), desc_k(b, kk), IDESC, kin == 0 ? 0u : 1u);
          issued = true;
          kin += 16;
          if (kin == p.unit) {                     // the unit is complete
            umma_commit(&tmem_full[buf]);
            ++it;
            kin = 0;
          }
        }
        umma_commit(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    if (issued) {
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                        // tensor-memory lane quadrant: tokens 32 q ..
    const int h = (warp - EPI_WARP0) >> 2;         // 128-column half of the tile
    float* scs = sc_stage + (warp - EPI_WARP0) * EPI_COLS;
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      const int I = t / p.nt, J = t - I * p.nt;
      const int rcol0 = J * BN + h * EPI_COLS;     // this warp's 128 rows of W (columns of Y)
      float run[EPI_COLS];
#pragma unroll
      for (int x = 0; x < EPI_COLS; ++x) run[x] = 0.0f;
      // the scales of this warp's rows for group g: lane l holds rows rcol0 + l + 32 c
      const float* sp = p.scales + (long long)(rcol0 + lane) * p.G;
      const long long sstep = 32LL * p.G;
      const int nlive = p.m - (rcol0 + lane);      // rows rcol0 + lane + 32 c exist for 32 c < nlive
      float sn[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sn[c] = (32 * c < nlive) ? __ldg(sp + c * sstep) : 0.0f;
      int g_next = 0, u_in_g = 0;                  // group of unit u + 1 (counted, no division)
      for (int u = 0; u < nunits; ++u, ++it) {
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c) scs[32 * c + lane] = sn[c];
        if (++u_in_g == p.upg) {
          u_in_g = 0;
          ++g_next;
        }
        if (u + 1 < nunits) {
#pragma unroll
          for (int c = 0; c < 4; ++c) sn[c] = (32 * c < nlive) ? __ldg(sp + c * sstep + g_next) : 0.0f;
        }
        const uint32_t buf = it % NBUF;
        if (!mbar_wait_bounded(&tmem_full[buf], (it / NBUF) & 1u, abort_flag)) {
          *abort_flag = 1;
          report_device_error(err_word, DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        __syncwarp();                              // scs written by every lane
#pragma unroll
        for (int part = 0; part < EPI_COLS / 16; ++part) {
          uint32_t acc[16];
          tmem_ld_32x32b_x16_nowait(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + h * EPI_COLS + part * 16, acc);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 sv = *reinterpret_cast<const float4*>(scs + part * 16 + 4 * c4);
            run[part * 16 + 4 * c4 + 0] = fmaf(__uint_as_float(acc[4 * c4 + 0]), sv.x, run[part * 16 + 4 * c4 + 0]);
            run[part * 16 + 4 * c4 + 1] = fmaf(__uint_as_float(acc[4 * c4 + 1]), sv.y, run[part * 16 + 4 * c4 + 1]);
            run[part * 16 + 4 * c4 + 2] = fmaf(__uint_as_float(acc[4 * c4 + 2]), sv.z, run[part * 16 + 4 * c4 + 2]);
            run[part * 16 + 4 * c4 + 3] = fmaf(__uint_as_float(acc[4 * c4 + 3]), sv.w, run[part * 16 + 4 * c4 + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[buf]);
      }
      if (!ok) break;
      // Y: this thread's token row holds 128 consecutive outputs; whole rows of the tile go
      // out as 16-byte stores (bf16 rounded to nearest even, or fp32), a ragged edge one
      // value at a time
      const int tok = I * BM + q * 32 + lane;
      if (tok < p.T) {
        const bool vec = (rcol0 + EPI_COLS <= p.m) && ((p.ldy & 7) == 0) &&
                         ((reinterpret_cast<uintptr_t>(p.Y) & 15) == 0);
        if (p.y_bf16) {
          __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(p.Y) + (long long)tok * p.ldy + rcol0;
          if (vec) {
#pragma unroll
            for (int c8 = 0; c8 < EPI_COLS / 8; ++c8) {
              __align__(16) __nv_bfloat16 o[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) o[k] = __float2bfloat16_rn(run[8 * c8 + k]);
              *reinterpret_cast<uint4*>(yr + 8 * c8) = *reinterpret_cast<const uint4*>(o);
            }
          } else {
#pragma unroll
            for (int c = 0; c < EPI_COLS; ++c)
              if (rcol0 + c < p.m) yr[c] = __float2bfloat16_rn(run[c]);
          }
        } else {
          float* yr = p.Y + (long long)tok * p.ldy + rcol0;
          if (vec) {
#pragma unroll
            for (int c4 = 0; c4 < EPI_COLS / 4; ++c4)
              *reinterpret_cast<float4*>(yr + 4 * c4) =
                  make_float4(run[4 * c4], run[4 * c4 + 1], run[4 * c4 + 2], run[4 * c4 + 3]);
          } else {
#pragma unroll
            for (int c = 0; c < EPI_COLS; ++c)
              if (rcol0 + c < p.m) yr[c] = run[c];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// 2-D bf16 map over (inner, outer) with row stride ld elements and a {64, rows} box.
bool make_map_bf16(CUtensorMap* m, const void* base, long long inner, long long outer, long long ld, uint32_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {BK, rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dqg

size_t dequant_gemm_workspace_bytes(long long m, long long d) { return (size_t)((m * d * 2 + 255) & ~255LL); }

gptq_status dequant_gemm_launch(const uint32_t* qweight, const float* scales, const float* zeros, long long m,
                                long long d, int bits, int group_size, const uint16_t* X, long long T, long long ldx,
                                void* Y, int y_bf16, long long ldy, void* ws, cudaStream_t s) {
  using namespace dqg;
  const int gs = (group_size < 0) ? (int)d : group_size;
  const int G = (int)(d / gs);
  const int wpr = (int)((d * bits + 31) / 32);
  // tensor-memory units: the group itself up to 256 columns, else the largest power of
  // two up to 256 that divides it (group sizes and d are multiples of 32)
  int unit = gs;
  if (unit > 256) {
    unit = 256;
    while (gs % unit) unit >>= 1;
  }
  __nv_bfloat16* B = reinterpret_cast<__nv_bfloat16*>(ws);
  {
    ProfScope ps("dequant_gemm.int_operand", s);
    const long long n8 = m * (d >> 3);
    const int grid = (int)std::min<long long>((n8 + 255) / 256, 8LL * sm_count());
    dq_int_kernel<<<grid, 256, 0, s>>>(qweight, zeros, (int)m, (int)d, bits, gs, G, wpr, B);
    count_launch();
    if (gptq_status st = check_launch("dq_int_kernel")) return st;
  }
  CUtensorMap mx, mb;
  if (!make_map_bf16(&mx, X, d, T, ldx, BM) || !make_map_bf16(&mb, B, d, m, d, BN))
    return set_error(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for the dequant GEMM operands");
  Params p{};
  p.T = (int)T; p.m = (int)m; p.d = (int)d;
  p.mt = (int)((T + BM - 1) / BM);
  p.nt = (int)((m + BN - 1) / BN);
  p.unit = unit; p.upg = gs / unit; p.gs = gs; p.G = G;
  p.scales = scales;
  p.Y = reinterpret_cast<float*>(Y);
  p.ldy = ldy;
  p.y_bf16 = y_bf16;
  const long long ntiles = (long long)p.mt * p.nt;
  const int grid = (int)std::min<long long>(ntiles, sm_count());
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(dequant_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
      return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(dequant_gemm_kernel) failed");
    attr_done = true;
  }
  ProfScope ps("dequant_gemm.gemm", s);
  if (launch_pdl(dequant_gemm_kernel, dim3(grid), dim3(THREADS), SMEM_BYTES, s, mx, mb, p, device_error_word()) !=
      cudaSuccess)
    return check_launch("dequant_gemm_kernel");
  count_launch();
  return check_launch("dequant_gemm_kernel");
}

}  // namespace gptq

// Stage 1: Hessian accumulation H += alpha * X^T X on the 5th-generation tensor cores.
//
// The Hessian of the layer-wise squared error is H = 2 X X^T with X channels x tokens
// ("GPTQ: fixing errors as you go", Objective; "The GPTQ Algorithm", procedure step 2);
// calibration batches add their X^T X into one running H ("GPTQ-style round-to-nearest
// with Hessian weighting", section "Computing the Hessian"). Here X is token-major
// (n x d, bf16) and only the upper triangle of the symmetric H is produced.
//
// Design (sm_103a):
//   * H is cut into 128 x 256 tiles; only tiles that hold some (i, j) with j >= i are
//     computed. The token axis is cut into S parts; a work unit is (tile, part).
//   * A persistent grid of one CTA per SM takes units round-robin in part-major
//     order, so all CTAs sweep the same token range at the same time and each X slab
//     is fetched from HBM about once and re-served to the other tiles from L2.
//   * Warp 0 (one thread) streams X tiles with TMA (128-byte swizzle) into a 4-stage
//     shared-memory ring; warp 1 (one thread) issues tcgen05.mma kind::f16
//     (bf16 x bf16 -> fp32, M = 128, N = 256, K = 16), both operands MN-major since
//     X^T's rows are X's columns; the accumulator lives in tensor memory, two
//     buffers of 256 columns so the epilogue of one chunk overlaps the next chunk's
//     products. The tensor core accumulates only CHUNK k-iterations (512 tokens) in a
//     buffer; warps 2-9 read each chunk with tcgen05.ld and add it into fp32
//     registers with round-to-nearest, which keeps the Hessian's error near that of
//     rounded fp32 summation (the tensor core's own long accumulations drift low).
//     At the end of a unit the register sums, scaled by alpha, go into H with vector
//     fp32 reductions (units of the same tile from different token parts meet there).
//   * Every wait is bounded; on a timeout the CTA raises the library's device error
//     word, drains its own copies and products, frees tensor memory and returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace gptq {
namespace syrk {

constexpr int BM = 128;                       // rows of an H tile (channels i)
constexpr int BN = 256;                       // columns of an H tile (channels j)
constexpr int BK = 64;                        // tokens per pipeline stage
constexpr int STAGES = 4;
constexpr int BOX = 64;                       // TMA box: 64 channels (128 bytes) x BK tokens
constexpr int BOX_BYTES = BOX * BK * 2;       // 8 KB
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 320;                  // TMA, MMA, 8 epilogue warps
constexpr int CHUNK = 8;                      // k-iterations (512 tokens) per tensor-memory accumulation
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr uint32_t IDESC = umma_idesc(/*bf16*/ 1, /*A MN-major*/ true, /*B MN-major*/ true, BM, BN);
// Within one stage a 16-token MMA step advances 16 rows of 128 bytes.
constexpr uint32_t KSTEP_BYTES = 16 * 128;
// MN-major, 128-byte swizzle: 8-row groups along K are 1024 bytes apart (SBO); the
// next 64 channels (next TMA box) are BOX_BYTES apart (LBO).
constexpr uint32_t SBO = 1024;
constexpr uint32_t LBO = BOX_BYTES;

struct Geometry {
  int d, nr, nc, tiles, parts, kiters;
  int npairs;                 // paired mode: 256 x 256 pair-tiles (rows 2p, 2p + 1 of the 128-row tiles)
};

// number of upper-triangle tiles in row-tiles [0, r)
__device__ __forceinline__ int tiles_before_row(int r, int nc) {
  const int a = r >> 1;
  const int s = (r & 1) ? a * a : a * (a - 1);   // sum_{r' < r} floor(r' / 2)
  return r * nc - s;
}

__device__ __forceinline__ void decode_tile(int t, int nr, int nc, int& r, int& c) {
  int lo = 0, hi = nr - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (tiles_before_row(mid, nc) <= t) lo = mid; else hi = mid - 1;
  }
  r = lo;
  c = (lo >> 1) + (t - tiles_before_row(lo, nc));
}

struct Unit {
  int r, c;
  int k0, k1;
};

// pair-tiles (p, c), c >= p, row-major: sum_{p' < p} (nc - p')
__device__ __forceinline__ int pairs_before_row(int p, int nc) { return p * nc - (p * (p - 1)) / 2; }

// 32-bit arithmetic only (a 64-bit division is an out-of-line call that would force
// the epilogue's register sums to the stack): units < 2^31, parts <= 64 and
// k-iterations < 2^25 keep part * kiters below 2^32.
__device__ __forceinline__ Unit decode_unit(int u, const Geometry& g) {
  Unit w;
  const unsigned part = (unsigned)u / (unsigned)g.tiles;
  const int t = u - (int)part * g.tiles;
  decode_tile(t, g.nr, g.nc, w.r, w.c);
  const unsigned kit = (unsigned)g.kiters;
  w.k0 = (int)(part * kit / (unsigned)g.parts);
  w.k1 = (int)((part + 1u) * kit / (unsigned)g.parts);
  return w;
}

// Paired mode (d a multiple of 256): a cluster of two CTAs takes (pair-tile, part)
// units; CTA `rank` computes the 128 x 256 tile of row 2p + rank. Both tiles need the
// same 256 channels of X as their B operand, so each CTA loads half of that slab with
// a multicast copy into both CTAs' shared memory (one third less traffic from L2 than
// two independent tiles); a stage is free again once both CTAs' products have read it.
__device__ __forceinline__ Unit decode_pair_unit(int u, const Geometry& g, int rank) {
  Unit w;
  const unsigned part = (unsigned)u / (unsigned)g.npairs;
  const int t = u - (int)part * g.npairs;
  int lo = 0, hi = g.nr / 2 - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pairs_before_row(mid, g.nc) <= t) lo = mid; else hi = mid - 1;
  }
  w.r = 2 * lo + rank;
  w.c = lo + (t - pairs_before_row(lo, g.nc));
  const unsigned kit = (unsigned)g.kiters;
  w.k0 = (int)(part * kit / (unsigned)g.parts);
  w.k1 = (int)((part + 1u) * kit / (unsigned)g.parts);
  return w;
}

template <bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
syrk_kernel(const __grid_constant__ CUtensorMap tmap, float* __restrict__ H, long long ldh, Geometry g,
            float alpha, int* __restrict__ err_word) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tmem_full = empty + STAGES;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int cid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;       // cluster (or CTA) index
  const int ncl = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  auto unit_of = [&](int u) { return PAIR ? decode_pair_unit(u, g, rank) : decode_unit(u, g); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAIR ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (PAIR) cluster_sync();      // the peer's barriers exist before anything targets them
  const uint32_t tmem_base = *tmem_slot;

  const int num_units = (PAIR ? g.npairs : g.tiles) * g.parts;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0;            // stages that were ever armed
    uint32_t last_phase = 0;       // bit s: phase of stage s's last arming
    bool ok = true;
    for (int u = cid; ok && u < num_units; u += ncl) {
      Unit w = unit_of(u);
      for (int k = w.k0; k < w.k1; ++k) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        uint8_t* sB = sA + A_BYTES;
        mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        const int tok = k * BK;
#pragma unroll
        for (int h = 0; h < BM / BOX; ++h) tma_load_2d(sA + h * BOX_BYTES, &tmap, &full[stage], w.r * BM + h * BOX, tok);
        if constexpr (PAIR) {
#pragma unroll
          for (int h = 2 * rank; h < 2 * rank + 2; ++h)
            tma_load_2d_mc(sB + h * BOX_BYTES, &tmap, &full[stage], w.c * BN + h * BOX, tok, (uint16_t)3);
        } else {
#pragma unroll
          for (int h = 0; h < BN / BOX; ++h)
            tma_load_2d(sB + h * BOX_BYTES, &tmap, &full[stage], w.c * BN + h * BOX, tok);
        }
        armed |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    // every armed load lands whatever the consumer did; wait for them before exit
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, nullptr);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: one accumulator per chunk of CHUNK k-iterations ----------------
    int stage = 0;
    uint32_t phase = 0;
    uint32_t it = 0;               // chunks issued (tensor-memory buffer rotation)
    bool ok = true, issued = false;
    const uint32_t sbase = smem_u32(smem);
    for (int u = cid; ok && u < num_units; u += ncl) {
      Unit w = unit_of(u);
      for (int kc = w.k0; ok && kc < w.k1; kc += CHUNK, ++it) {
        const int ke = (kc + CHUNK < w.k1) ? kc + CHUNK : w.k1;
        const uint32_t buf = it & 1u;
        if (!mbar_wait_bounded(&tmem_empty[buf], ((it >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int k = kc; k < ke; ++k) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = sbase + stage * STAGE_BYTES;
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t da = umma_sdesc_sw128(a0 + kk * KSTEP_BYTES, LBO, SBO);
            const uint64_t db = umma_sdesc_sw128(b0 + kk * KSTEP_BYTES, LBO, SBO);
            umma_f16(d_tmem, da, db, IDESC, (k > kc || kk > 0) ? 1u : 0u);
          }
          issued = true;
          if constexpr (PAIR) umma_commit_mc(&empty[stage], (uint16_t)3);   // both CTAs' copies of the stage
          else umma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tmem_full[buf]);
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    if (issued) {
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else if (warp >= 2) {
    // ---------------- epilogue: chunk sums from tensor memory, added in fp32 registers
    // (round to nearest), then alpha * sum reduced into H once per unit ----------------
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int h = (warp - 2) >> 2;           // which 128-column half of the tile
    const int row = q * 32 + lane;
    uint32_t it = 0;
    bool ok = true;
    float acc[BN / 2];
    for (int u = cid; ok && u < num_units; u += ncl) {
      Unit w = unit_of(u);
      const int i = w.r * BM + row;
      const int i_warp = w.r * BM + q * 32;
      const int jh = w.c * BN + h * (BN / 2);
      for (int kc = w.k0; kc < w.k1; kc += CHUNK, ++it) {
        const uint32_t buf = it & 1u;
        if (!mbar_wait_bounded(&tmem_full[buf], (it >> 1) & 1u, abort_flag)) {
          *abort_flag = 1;
          report_device_error(err_word, DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const bool first = (kc == w.k0);
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc) {
          const int j0 = jh + cc * 32;
          if (j0 + 31 < i_warp || j0 >= g.d) continue;   // warp-uniform: nothing on or above the diagonal
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[16];
            tmem_ld_32x32b_x16_nowait(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + h * (BN / 2) + cc * 32 + hh * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const float f = __uint_as_float(v[x]);
              acc[cc * 32 + hh * 16 + x] = first ? f : acc[cc * 32 + hh * 16 + x] + f;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[buf]);
      }
      if (!ok) break;
      if (i < g.d) {
        float* hrow = H + (long long)i * ldh;
#pragma unroll
        for (int x = 0; x < BN / 2; ++x) acc[x] *= alpha;
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc) {
          const int j0 = jh + cc * 32;
          if (j0 + 31 < i_warp || j0 >= g.d) continue;
          if (j0 >= i_warp + 31 && j0 + 31 < g.d) {          // whole group above the diagonal
#pragma unroll
            for (int e = 0; e < 8; ++e)
              atomicAdd(reinterpret_cast<float4*>(hrow + j0 + 4 * e),
                        make_float4(acc[cc * 32 + 4 * e], acc[cc * 32 + 4 * e + 1], acc[cc * 32 + 4 * e + 2],
                                    acc[cc * 32 + 4 * e + 3]));
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (j0 + x >= i && j0 + x < g.d) atomicAdd(hrow + j0 + x, acc[cc * 32 + x]);
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
  // neither CTA leaves while the other may still deliver copies or arrivals to it
  if constexpr (PAIR) cluster_sync();
}

// zero the upper triangle (i <= j) of H
// H[i][j] = 0 for j >= i: one warp per row, a scalar head up to the first 16-byte
// boundary (vec: rows 16-byte aligned), then 16-byte stores
__global__ void zero_upper_kernel(float* __restrict__ H, long long ldh, int d, int vec) {
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= d) return;
  float* row = H + (long long)i * ldh;
  if (!vec) {
    for (int j = i + lane; j < d; j += 32) row[j] = 0.0f;
    return;
  }
  const int j4 = min(d, (i + 3) & ~3);
  if (i + lane < j4) row[i + lane] = 0.0f;
  const int q_end = d >> 2;
  for (int q = (j4 >> 2) + lane; q < q_end; q += 32) reinterpret_cast<float4*>(row)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = (q_end << 2) + lane; j < d; j += 32) if (j >= j4) row[j] = 0.0f;
}

}  // namespace syrk

namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int choose_parts(long long tiles, long long kiters, int grid) {
  // minimise the estimated makespan ceil(units / grid) * (kiters / parts + fill)
  int best = 1;
  double best_cost = 1e300;
  const int max_parts = (int)std::min<long long>(64, std::max<long long>(1, kiters / 8));
  for (int s = 1; s <= max_parts; ++s) {
    const long long units = tiles * s;
    const double rounds = std::ceil((double)units / grid);
    const double cost = rounds * ((double)kiters / s + 4.0);
    if (cost < best_cost * 0.999) { best_cost = cost; best = s; }
  }
  return best;
}
}  // namespace

gptq_status syrk_accumulate(const uint16_t* X, long long n, long long d, long long ldx, float* H, long long ldh,
                            float alpha, int zero_first, cudaStream_t stream) {
  using namespace syrk;
  if (zero_first) {
    const int vec = (ldh % 4 == 0) && (reinterpret_cast<uintptr_t>(H) % 16 == 0);
    zero_upper_kernel<<<(unsigned)((d + 7) / 8), 256, 0, stream>>>(H, ldh, (int)d, vec);
    count_launch();
    if (gptq_status st = check_launch("zero_upper_kernel")) return st;
  }
  if (n == 0) return GPTQ_OK;

  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (!encode) return set_error(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap tmap;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
  cuuint32_t box[2] = {BOX, BK};
  cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return set_error(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);

  Geometry g;
  g.d = (int)d;
  g.nr = (int)((d + BM - 1) / BM);
  g.nc = (int)((d + BN - 1) / BN);
  long long tiles = 0;
  for (int r = 0; r < g.nr; ++r) tiles += g.nc - (r * BM) / BN;
  g.tiles = (int)tiles;
  g.kiters = (int)((n + BK - 1) / BK);
  g.npairs = 0;
  const int sms = sm_count();

  static bool attr_set[2] = {false, false};
  for (int k = 0; k < 2; ++k)
    if (!attr_set[k]) {
      if (cudaFuncSetAttribute(k ? syrk_kernel<true> : syrk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES) != cudaSuccess)
        return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(syrk_kernel) failed");
      attr_set[k] = true;
    }

  // Paired mode when every 128-row tile has its partner: d a multiple of 256.
  int clusters = 0;
  if (d % BN == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * (sms / 2)));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&clusters, syrk_kernel<true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
  }
  ProfScope ps("hessian.syrk", stream);
  if (clusters > 0) {
    g.npairs = (g.nc * (g.nc + 1)) / 2;
    g.parts = choose_parts(g.npairs, g.kiters, clusters);
    const long long units = (long long)g.npairs * g.parts;
    const int ncl = (int)std::min<long long>(units, clusters);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * ncl));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, syrk_kernel<true>, tmap, H, ldh, g, alpha, device_error_word()) != cudaSuccess)
      return check_launch("syrk_kernel (paired)");
  } else {
    g.parts = choose_parts(tiles, g.kiters, sms);
    const long long units = tiles * g.parts;
    const int grid = (int)std::min<long long>(units, sms);
    syrk_kernel<false><<<grid, THREADS, SMEM_BYTES, stream>>>(tmap, H, ldh, g, alpha, device_error_word());
  }
  count_launch();
  return check_launch("syrk_kernel");
}

}  // namespace gptq

// FP32-accurate GEMM on the 5th-generation tensor cores (3 x TF32):
//
//     C = beta * C + alpha * A B        (per batch z, 128 x 128 output tiles)
//
// with A(i, k) = A[i * lda + k] and B(k, j) = B[j * ldb + k] (both K-major: the tf32
// tensor-core path reads only K-major operands; an MN-major tf32 operand yields zeros,
// so those calls take the FFMA GEMM of simt_gemm.cuh).
//
// Each fp32 operand x is split as x = hi + lo, hi = x with its 13 low mantissa bits
// cleared and lo = x - hi (exact); A B is formed as hi_A hi_B + hi_A lo_B + lo_A hi_B,
// which carries about 21 significant bits per product. The tf32 tensor-core path reads
// an fp32 word as its hi part (the low mantissa bits are ignored; checked against an
// fp64 product on this GPU), so the raw operand serves as hi and only lo is stored.
// Callers that already hold the lo parts pass them (GemmArgs::A_lo / B_lo) and the
// tiles are loaded pre-split; otherwise converter warps form lo in shared memory.
//
// Design (sm_103a), one persistent CTA per SM, tiles taken round-robin:
//   warp 0      TMA producer: 32-deep k chunks of A and B into a 3-stage ring
//   warps 2-5   converters (operands without lo parts): lo parts of each stage into
//               their own buffers (the 128-byte swizzle permutes 16-byte chunks, so an
//               elementwise pass keeps the layout), zeroing k past the extent of a
//               ragged last batch and outside a triangular operand
//   warp 1      MMA issuer: per chunk 4 k-steps x 3 products, tcgen05.mma kind::tf32
//               M = 128, N = 128, K = 8; two chunks (64 products) go into one
//               tensor-memory buffer, four buffers of 128 columns rotate, so the
//               products of the next tile run ahead of the epilogue's memory traffic
//   warps 6-13  epilogue: each buffer's partial product is added into fp32 registers
//               with round-to-nearest (the tensor core's own accumulator truncates, so
//               long accumulations in it drift), and at the end of a tile
//               C = beta C + alpha acc is written through a shared-memory staging
//               tile in 128-byte rows
// Every wait is bounded; a timeout raises the device error word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {
namespace tc {

constexpr int BM = 128, BN = 128, BK = 32;     // BK fp32 = 128 bytes: one swizzle row
constexpr int STAGES = 3;
constexpr int OP_BYTES = BM * BK * 4;          // 16 KB per operand per stage
constexpr int STAGE_BYTES = 4 * OP_BYTES;      // A, B, A_lo, B_lo
constexpr int CONV_WARP0 = 2, NCONV = 4;
constexpr int NEPI = 8;
// warps 0-1 TMA and MMA, then the converters (operands without lo parts), then the
// epilogue warps
template <bool PRESPLIT> constexpr int epi_warp0() { return PRESPLIT ? 2 : CONV_WARP0 + NCONV; }
template <bool PRESPLIT> constexpr int threads() { return (epi_warp0<PRESPLIT>() + NEPI) * 32; }
constexpr int NBUF = 4;                       // chunk accumulators in tensor memory
constexpr int ACC_CHUNKS = 2;                 // 32-deep chunks summed in one accumulator (64 products)
constexpr uint32_t TMEM_COLS = NBUF * BN;
constexpr int EPI_LD = 33;                    // padded row of an epilogue warp's 32 x 32 staging tile
constexpr int EPI_BYTES = NEPI * 32 * EPI_LD * 4;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256 + EPI_BYTES;

struct Params {
  int M, N, K, M_last, K_last, batches;
  int tiles_per_batch, mt, nt;
  int lower_tiles, a_tri, b_lower;
  unsigned* signal;
  int b_final;
  float alpha, beta;
  float* C;
  long long ldc, c_bs;
  const int* skip;
};

struct Tile {
  int z, I, J, kbeg, kend, M, K;
};

__device__ __forceinline__ Tile decode(int t, const Params& p) {
  Tile w;
  w.z = t / p.tiles_per_batch;
  const int u = t - w.z * p.tiles_per_batch;
  if (p.lower_tiles == 2) {
    // column by column: tile column J starts at J mt - J (J - 1) / 2
    int J = 0;
    while (J + 1 < p.mt && u >= (J + 1) * p.mt - (J + 1) * J / 2) ++J;
    w.J = J;
    w.I = J + (u - (J * p.mt - J * (J - 1) / 2));
  } else if (p.lower_tiles) {
    int I = (int)((sqrtf(8.0f * (float)u + 1.0f) - 1.0f) * 0.5f);
    while ((I + 1) * (I + 2) / 2 <= u) ++I;
    while (I * (I + 1) / 2 > u) --I;
    w.I = I;
    w.J = u - I * (I + 1) / 2;
  } else {
    w.I = u / p.nt;
    w.J = u - w.I * p.nt;
    // a lower-triangular A (a_tri 1) makes tile rows cost more as I grows: take them
    // from the bottom so tiles come in order of decreasing cost, as for a_tri 2
    if (p.a_tri == 1) w.I = p.mt - 1 - w.I;
  }
  const bool last = (w.z == p.batches - 1);
  w.M = last ? p.M_last : p.M;
  w.K = last ? p.K_last : p.K;
  w.kbeg = 0;
  w.kend = w.K;
  if (p.a_tri == 1) w.kend = min(w.kend, (w.I + 1) * BM);
  if (p.a_tri == 2) w.kbeg = w.I * BM;
  if (p.b_lower) w.kbeg = max(w.kbeg, w.J * BN);
  if (w.kbeg >= w.kend || w.I * BM >= w.M) w.kend = w.kbeg;   // nothing to multiply
  return w;
}

__device__ __forceinline__ int nchunks(const Tile& w) { return (w.kend - w.kbeg + BK - 1) / BK; }

// The k-th tile of CTA b: rounds alternate direction (b, then 2 grid - 1 - b, ...), so a
// CTA that drew an expensive tile in one round draws a cheap one in the next when tiles
// come in order of decreasing cost (triangular operands, see decode). The sequence is
// increasing in k, so the first index past the end ends every role's loop.
__device__ __forceinline__ int tile_at(int k, int b, int grid) { return (k & 1) ? (k + 1) * grid - 1 - b : k * grid + b; }

// smem descriptors: K-major SW128 (rows of 128 bytes along k, 8-row groups 1024 B
// apart) and MN-major SW128 (32-element MN chunks are separate TMA boxes 4 KB apart,
// 8-row k groups 1024 B apart).
__device__ __forceinline__ uint64_t desc_kmaj(uint32_t base, int kk) { return umma_sdesc_sw128(base + kk * 32, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mnmaj(uint32_t base, int kk) { return umma_sdesc_sw128(base + kk * 1024, 4096, 1024); }

// Load one operand's 32-deep chunk: K-major = one box {32 k, 128 rows};
// MN-major = four boxes {32 rows, 32 k}.
template <bool KMAJ>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int r0, int k0, int z) {
  if constexpr (KMAJ) {
    tma_load_3d(dst, map, bar, k0, r0, z);
  } else {
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_3d(dst + b * 4096, map, bar, r0 + 32 * b, k0, z);
  }
}

// x -> (hi, lo) for one operand's chunk, hi written in place; elements with k >= kend
// are zeroed in both buffers, and so are those outside the triangle `tri` (1: keep
// k <= row, 2: keep k >= row; K-major operands, rows counted from row0). `kbase` is the
// chunk's first k.
template <bool KMAJ>
__device__ __forceinline__ void split_operand(uint8_t* raw, uint8_t* lo, int kbase, int kend, int ctid, int tri = 0,
                                              int row0 = 0) {
  float4* r4 = reinterpret_cast<float4*>(raw);
  float4* l4 = reinterpret_cast<float4*>(lo);
  const bool ragged = kbase + BK > kend;
  // the chunk meets the tile's diagonal band only if [kbase, kbase + BK) overlaps [row0, row0 + BM)
  const bool diag = KMAJ && tri != 0 && kbase < row0 + BM && kbase + BK > row0;
  for (int idx = ctid; idx < OP_BYTES / 16; idx += NCONV * 32) {
    float4 x = r4[idx];
    if (diag) {
      const int row = idx >> 3, lc = (idx & 7) ^ (row & 7);
      const int k0 = kbase + 4 * lc, r = row0 + row;
      if (tri == 1) {
        if (k0 + 0 > r) x.x = 0.0f;
        if (k0 + 1 > r) x.y = 0.0f;
        if (k0 + 2 > r) x.z = 0.0f;
        if (k0 + 3 > r) x.w = 0.0f;
      } else {
        if (k0 + 0 < r) x.x = 0.0f;
        if (k0 + 1 < r) x.y = 0.0f;
        if (k0 + 2 < r) x.z = 0.0f;
        if (k0 + 3 < r) x.w = 0.0f;
      }
    }
    if (ragged) {
      // 16-byte chunk idx: byte offset idx * 16
      int k_of_elem0, step;
      if constexpr (KMAJ) {
        const int row = idx >> 3, pc = idx & 7;           // 8 chunks per 128-byte row
        const int lc = pc ^ (row & 7);                    // logical chunk (128-byte swizzle)
        k_of_elem0 = kbase + 4 * lc;
        step = 1;
      } else {
        const int krow = (idx >> 3) & 31;                 // 32 k-rows per 4 KB box
        k_of_elem0 = kbase + krow;
        step = 0;
      }
      if (k_of_elem0 + 0 * step >= kend) x.x = 0.0f;
      if (k_of_elem0 + 1 * step >= kend) x.y = 0.0f;
      if (k_of_elem0 + 2 * step >= kend) x.z = 0.0f;
      if (k_of_elem0 + 3 * step >= kend) x.w = 0.0f;
    }
    float4 l;
    l.x = x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
    l.y = x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
    l.z = x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
    l.w = x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
    if (ragged || diag) r4[idx] = x;   // the masked operand; untouched chunks stay as loaded
    l4[idx] = l;
  }
}

template <bool A_KMAJ, bool B_KMAJ, bool PRESPLIT>
__global__ void __launch_bounds__(threads<PRESPLIT>(), 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_alo, const __grid_constant__ CUtensorMap map_blo, Params p,
               int* __restrict__ err_word) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* conv = full + STAGES;
  uint64_t* empty = conv + STAGES;
  uint64_t* tmem_full = empty + STAGES;
  uint64_t* tmem_empty = tmem_full + NBUF;
  uint64_t* drain = tmem_empty + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_stage = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);   // NEPI x 32 x EPI_LD

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], NCONV);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], NEPI);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
    if constexpr (PRESPLIT) {
      prefetch_tmap(&map_alo);
      prefetch_tmap(&map_blo);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above touched no global data; the operands and C come from earlier kernels
  grid_dep_launch();
  const bool producer = (warp == 0 && lane == 0);
  // With a final B, the producer first loads the B parts of its first tile's first
  // stages (their barriers armed for the whole stage), then waits like everyone else.
  int pre = 0;
  if (producer && p.b_final && !p.skip && (int)blockIdx.x < p.tiles_per_batch * p.batches) {
    const Tile w = decode(blockIdx.x, p);
    pre = min(nchunks(w), STAGES);
    for (int c = 0; c < pre; ++c) {
      uint8_t* sa = smem + c * STAGE_BYTES;
      const int k0 = w.kbeg + c * BK;
      mbar_arrive_expect_tx(&full[c], (PRESPLIT ? 4 : 2) * OP_BYTES);
      load_operand<B_KMAJ>(sa + OP_BYTES, &map_b, &full[c], w.J * BN, k0, w.z);
      if constexpr (PRESPLIT) load_operand<B_KMAJ>(sa + 3 * OP_BYTES, &map_blo, &full[c], w.J * BN, k0, w.z);
    }
  }
  grid_dep_wait();
  const int ntiles = (p.skip && *p.skip) ? 0 : p.tiles_per_batch * p.batches;
  constexpr uint32_t IDESC = umma_idesc(/*tf32*/ 2, !A_KMAJ, !B_KMAJ, BM, BN);

  if (producer) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0, armed = 0, last_phase = 0;
    bool ok = true;
    int seq = 0;                                   // chunks issued so far
    for (int kt = 0, t = blockIdx.x; ok && t < ntiles; t = tile_at(++kt, blockIdx.x, gridDim.x)) {
      const Tile w = decode(t, p);
      for (int k0 = w.kbeg; k0 < w.kend; k0 += BK, ++seq) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        const bool preloaded = seq < pre;          // B parts already on their way
        if (!preloaded) mbar_arrive_expect_tx(&full[stage], (PRESPLIT ? 4 : 2) * OP_BYTES);
        load_operand<A_KMAJ>(sa, &map_a, &full[stage], w.I * BM, k0, w.z);
        if (!preloaded) load_operand<B_KMAJ>(sa + OP_BYTES, &map_b, &full[stage], w.J * BN, k0, w.z);
        if constexpr (PRESPLIT) {
          load_operand<A_KMAJ>(sa + 2 * OP_BYTES, &map_alo, &full[stage], w.I * BM, k0, w.z);
          if (!preloaded) load_operand<B_KMAJ>(sa + 3 * OP_BYTES, &map_blo, &full[stage], w.J * BN, k0, w.z);
        }
        armed |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, nullptr);
  } else if (!PRESPLIT && warp >= CONV_WARP0 && warp < CONV_WARP0 + NCONV) {
    // ---------------- converters: lo parts ----------------
    const int ctid = threadIdx.x - CONV_WARP0 * 32;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kt = 0, t = blockIdx.x; ok && t < ntiles; t = tile_at(++kt, blockIdx.x, gridDim.x)) {
      const Tile w = decode(t, p);
      for (int k0 = w.kbeg; k0 < w.kend; k0 += BK) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        split_operand<A_KMAJ>(sa, sa + 2 * OP_BYTES, k0, w.kend, ctid, p.a_tri, w.I * BM);
        split_operand<B_KMAJ>(sa + OP_BYTES, sa + 3 * OP_BYTES, k0, w.kend, ctid);
        fence_proxy_async_smem();   // generic-proxy writes must be visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    int stage = 0;
    uint32_t phase = 0, it = 0;
    bool ok = true, issued = false;
    const uint32_t sbase = smem_u32(smem);
    for (int kt = 0, t = blockIdx.x; ok && t < ntiles; t = tile_at(++kt, blockIdx.x, gridDim.x)) {
      const Tile w = decode(t, p);
      int cin = 0;                                 // chunk index within the tile
      for (int k0 = w.kbeg; k0 < w.kend; k0 += BK, ++cin) {
        const bool first = (cin % ACC_CHUNKS) == 0;
        const bool last = (cin % ACC_CHUNKS) == ACC_CHUNKS - 1 || k0 + BK >= w.kend;
        const uint32_t buf = it % NBUF;
        if (first && !mbar_wait_bounded(&tmem_empty[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        if (!mbar_wait_bounded(PRESPLIT ? &full[stage] : &conv[stage], phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        const uint32_t a = sbase + stage * STAGE_BYTES, b = a + OP_BYTES;
        const uint32_t alo = a + 2 * OP_BYTES, blo = a + 3 * OP_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint64_t da = A_KMAJ ? desc_kmaj(a, kk) : desc_mnmaj(a, kk);
          const uint64_t dal = A_KMAJ ? desc_kmaj(alo, kk) : desc_mnmaj(alo, kk);
          const uint64_t db = B_KMAJ ? desc_kmaj(b, kk) : desc_mnmaj(b, kk);
          const uint64_t dbl = B_KMAJ ? desc_kmaj(blo, kk) : desc_mnmaj(blo, kk);
          umma_tf32(d_tmem, da, dbl, IDESC, (kk > 0 || !first) ? 1u : 0u);
          umma_tf32(d_tmem, dal, db, IDESC, 1u);
          umma_tf32(d_tmem, da, db, IDESC, 1u);
        }
        issued = true;
        umma_commit(&empty[stage]);
        if (last) {
          umma_commit(&tmem_full[buf]);
          ++it;
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) { *abort_flag = 1; report_device_error(err_word, DEVERR_TIMEOUT); }
    if (issued) {
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else if (warp >= epi_warp0<PRESPLIT>()) {
    // ---------------- epilogue ----------------
    constexpr int EPI_WARP0 = epi_warp0<PRESPLIT>();
    const int q = warp & 3;                       // TMEM lane quadrant
    const int h = (warp - EPI_WARP0) >> 2;        // 64-column half of the tile
    uint32_t it = 0;
    bool ok = true;
    for (int kt = 0, t = blockIdx.x; ok && t < ntiles; t = tile_at(++kt, blockIdx.x, gridDim.x)) {
      const Tile w = decode(t, p);
      // Pull this thread's 64-column segment of C into L2 while the tile's products are
      // computed, so the read-modify-write below waits on L2 rather than on DRAM
      // (whole segments only; a ragged edge is read as it is).
      if (p.beta != 0.0f) {
        const int i = w.I * BM + q * 32 + lane, j0 = w.J * BN + h * 64;
        if (i < w.M && j0 + 64 <= p.N) {
          const float* seg = p.C + (long long)w.z * p.c_bs + (long long)i * p.ldc + j0;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], 256;" ::"l"(seg) : "memory");
        }
      }
      // Pre-split mode: this thread's C values of the first 32-column half are loaded
      // now, so their latency hides behind the tile's loads and products.
      float o_early[32];
      if constexpr (PRESPLIT) {
        const int j = w.J * BN + h * 64 + lane;
        const float* cb = p.C + (long long)w.z * p.c_bs;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const int i = w.I * BM + q * 32 + r;
          o_early[r] = (p.beta != 0.0f && i < w.M && j < p.N) ? __ldcg(cb + (long long)i * p.ldc + j) : 0.0f;
        }
      }
      float acc[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) acc[x] = 0.0f;
      const int nc = (nchunks(w) + ACC_CHUNKS - 1) / ACC_CHUNKS;   // accumulators of this tile
      for (int c = 0; c < nc; ++c, ++it) {
        const uint32_t buf = it % NBUF;
        if (!mbar_wait_bounded(&tmem_full[buf], (it / NBUF) & 1u, abort_flag)) {
          *abort_flag = 1;
          report_device_error(err_word, DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t v[16];
          tmem_ld_32x32b_x16_nowait(tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN + h * 64 + g * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x) acc[g * 16 + x] += __uint_as_float(v[x]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[buf]);
      }
      if (!ok) break;
      // C = beta C + alpha acc through a 32 x 32 staging tile per warp: lane = row while
      // reading tensor memory, lane = column while touching C, so every load and store
      // of C is one contiguous 128-byte row segment
      float* stg = epi_stage + (warp - EPI_WARP0) * 32 * EPI_LD;
      const int rbase = w.I * BM + q * 32;
      float* cbase = p.C + (long long)w.z * p.c_bs;
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
#pragma unroll
        for (int c = 0; c < 32; ++c) stg[lane * EPI_LD + c] = acc[32 * g2 + c];
        __syncwarp();
        const int j = w.J * BN + h * 64 + 32 * g2 + lane;
        float o[32];
        if (PRESPLIT && g2 == 0) {
#pragma unroll
          for (int r = 0; r < 32; ++r) o[r] = o_early[r];
        } else if (p.beta != 0.0f) {
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            const int i = rbase + r;
            o[r] = (i < w.M && j < p.N) ? __ldcg(cbase + (long long)i * p.ldc + j) : 0.0f;
          }
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) o[r] = 0.0f;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const int i = rbase + r;
          if (i < w.M && j < p.N)
            __stcg(cbase + (long long)i * p.ldc + j, fmaf(p.alpha, stg[r * EPI_LD + lane], p.beta * o[r]));
        }
        __syncwarp();
      }
      if (p.signal && w.J == 0) {
        // this warp's part of a tile of column 0 is stored: publish it (gpu scope)
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.signal, 1u);
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D fp32 map over (inner, outer, batch) with the given box.
bool make_map(CUtensorMap* m, const float* base, long long inner, long long outer, long long ld, int batches,
              long long bstride, uint32_t box_inner, uint32_t box_outer) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)std::max(1, batches)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)std::max<long long>(bstride, 1) * 4};
  if (batches <= 1) strides[1] = (cuuint64_t)ld * 4 * (cuuint64_t)std::max<long long>(outer, 1);
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

// Operand extents: A is M x K (K-major: rows M of k; MN-major: rows K of m), B is K x N.
// Falls back to the FFMA GEMM when an operand cannot be described to TMA (16-byte
// alignment of bases and strides).
static bool force_ffma() {
  static const bool f = [] {
    const char* v = getenv("GPTQ_FFMA_GEMM");
    return v && v[0] == '1';
  }();
  return f;
}

bool tc_gemm_available() { return !force_ffma() && tc::encode_fn() != nullptr; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return tc::encode_fn(); }
bool tensor_maps_available() { return tc::encode_fn() != nullptr; }

gptq_status tc_gemm(const simt::GemmArgs& g, int batches, bool a_kmaj, bool b_kmaj, cudaStream_t s) {
  using namespace tc;
  if (g.M <= 0 || g.N <= 0 || batches <= 0) return GPTQ_OK;
  if (force_ffma()) return simt::gemm(g, batches, a_kmaj, b_kmaj, s);
  if (batches > 1 && (g.M_last != g.M || g.K_last != g.K)) {
    // a ragged last batch gets its own launch with exact extents, so no tensor map
    // describes memory past the end of an operand
    simt::GemmArgs full = g;
    full.M_last = g.M;
    full.K_last = g.K;
    if (gptq_status st = tc_gemm(full, batches - 1, a_kmaj, b_kmaj, s)) return st;
    simt::GemmArgs last = g;
    last.A = g.A + (long long)(batches - 1) * g.a_bs;
    last.B = g.B + (long long)(batches - 1) * g.b_bs;
    last.C = g.C + (long long)(batches - 1) * g.c_bs;
    last.M = last.M_last = g.M_last;
    last.K = last.K_last = g.K_last;
    return tc_gemm(last, 1, a_kmaj, b_kmaj, s);
  }
  const bool aligned = g.vec && simt::aligned16(g.A) && simt::aligned16(g.B) && simt::aligned16(g.C) &&
                       (g.lda % 4 == 0) && (g.ldb % 4 == 0) && (g.ldc % 4 == 0) && (g.a_bs % 4 == 0) &&
                       (g.b_bs % 4 == 0) && (g.c_bs % 4 == 0);
  // pre-split operands: both lo parts given, aligned, one batch, no triangular masks
  const bool presplit = g.A_lo && g.B_lo && batches == 1 && !g.a_tri && !g.b_lower && simt::aligned16(g.A_lo) &&
                        simt::aligned16(g.B_lo) && (g.lda_lo % 4 == 0) && (g.ldb_lo % 4 == 0);
  // tcgen05 kind::tf32 reads K-major operands only (an MN-major tf32 operand yields
  // zeros), so other layouts and unaligned operands take the FFMA GEMM
  if (!aligned || !a_kmaj || !b_kmaj) return simt::gemm(g, batches, a_kmaj, b_kmaj, s);
  CUtensorMap ma, mb;
  // logical extents cover every batch (the last batch can only be smaller)
  bool ok;
  if (a_kmaj) ok = make_map(&ma, g.A, g.K, g.M, g.lda, batches, g.a_bs, BK, BM);
  else ok = make_map(&ma, g.A, g.M, g.K, g.lda, batches, g.a_bs, 32, BK);
  if (ok) {
    if (b_kmaj) ok = make_map(&mb, g.B, g.K, g.N, g.ldb, batches, g.b_bs, BK, BN);
    else ok = make_map(&mb, g.B, g.N, g.K, g.ldb, batches, g.b_bs, 32, BK);
  }
  if (!ok) return simt::gemm(g, batches, a_kmaj, b_kmaj, s);
  CUtensorMap malo = ma, mblo = mb;
  const bool split = presplit && make_map(&malo, g.A_lo, g.K, g.M, g.lda_lo, 1, 0, BK, BM) &&
                     make_map(&mblo, g.B_lo, g.K, g.N, g.ldb_lo, 1, 0, BK, BN);

  Params p{};
  p.M = g.M; p.N = g.N; p.K = g.K; p.M_last = g.M_last; p.K_last = g.K_last; p.batches = batches;
  p.mt = (g.M + BM - 1) / BM;
  p.nt = (g.N + BN - 1) / BN;
  p.tiles_per_batch = g.lower_tiles ? p.mt * (p.mt + 1) / 2 : p.mt * p.nt;
  p.lower_tiles = g.lower_tiles; p.a_tri = g.a_tri; p.b_lower = g.b_lower;
  p.signal = (g.lower_tiles == 2) ? g.signal : nullptr;
  p.b_final = (g.b_final && !g.skip) ? 1 : 0;
  p.alpha = g.alpha; p.beta = g.beta;
  p.C = g.C; p.ldc = g.ldc; p.c_bs = g.c_bs;
  p.skip = g.skip;
  const int ntiles = p.tiles_per_batch * batches;
  const int grid = std::min(ntiles, g.max_ctas > 0 ? std::min(g.max_ctas, sm_count()) : sm_count());

  auto launch = [&](auto kern, int key) -> gptq_status {
    static bool attr_done[2] = {false, false};
    if (!attr_done[key]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
        return set_error(GPTQ_ERR_CUDA, "cudaFuncSetAttribute(tc_gemm_kernel) failed");
      attr_done[key] = true;
    }
    if (launch_pdl(kern, dim3(grid), dim3(key ? threads<true>() : threads<false>()), SMEM_BYTES, s, ma, mb, malo,
                   mblo, p, device_error_word()) != cudaSuccess)
      return check_launch("tc_gemm_kernel");
    count_launch();
    return check_launch("tc_gemm_kernel");
  };
  return split ? launch(tc_gemm_kernel<true, true, true>, 1) : launch(tc_gemm_kernel<true, true, false>, 0);
}

}  // namespace gptq

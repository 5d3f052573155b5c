// The stored layer used again: Y = X W_hat^T straight from the packed codes.
//
// After quantization a layer keeps its b-bit codes and one (scale, zero) per group of
// columns and is used as before ("GPTQ: fixing errors as you go", on what changes at
// inference time): w_hat[r][j] = (code[r][j] - zero[r][G(j)]) * scale[r][G(j)], with
// G(j) = j / group_size, or g_idx[j] for act-order groups. For the few tokens of a
// decoding step this product reads every code once and is bound by HBM bandwidth.
//
// Two kernels: gemv_mma_kernel (below) for codes in natural groups, and this FMA kernel
// for act-order groups and groups narrower than that kernel's column blocks.
//
// dequant_gemv_kernel<BITS, GIDX>: one warp per row r; lane L takes the 32-column
// chunks L, L + 32, ... of the row (BITS words each, read as 16-byte vectors where the
// width allows; several chunks in flight per lane), unpacks the codes with compile-time
// shifts into biased floats (no integer conversion), dequantizes them with the
// chunk's (scale, zero) (a group spans whole chunks: group_size is a multiple of 32) or
// per column through g_idx, and accumulates x * w_hat for NT = 1, 2, 4 or 8 tokens in
// fp32 (a template constant: a runtime count would leave predicated-off work); the
// warp's partial sums meet by shuffles. X (bf16, token-major) is read through the
// read-only cache; every row reuses it.
#include <algorithm>
#include <cstdlib>
#include <string>

#include "common.cuh"

namespace gptq {
namespace dgemv {

constexpr int WARPS = 8;         // rows per CTA

template <int BITS>
__device__ __forceinline__ void load_chunk(const uint32_t* __restrict__ row, int chunk, uint32_t (&wv)[BITS]) {
  const uint32_t* p = row + (long long)chunk * BITS;
  if constexpr (BITS == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
  } else if constexpr (BITS == 8) {
    const uint4 a = *reinterpret_cast<const uint4*>(p), b = *reinterpret_cast<const uint4*>(p + 4);
    wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w; wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
  } else if constexpr (BITS == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    wv[0] = v.x; wv[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < BITS; ++k) wv[k] = __ldg(p + k);
  }
}

// Code i (0..31) of a 32-column chunk held in BITS words (little-endian bitstream), as
// the float 2^23 + code: the code's bits ORed into the mantissa of 2^23, so no
// integer-to-float conversion (a quarter-rate instruction) is needed; the caller
// subtracts 2^23 + zero, which is exact, and gets code - zero.
constexpr uint32_t kTwo23Bits = 0x4B000000u;
constexpr float kTwo23 = 8388608.0f;

template <int BITS, int I>
__device__ __forceinline__ float code_of(const uint32_t (&wv)[BITS]) {
  constexpr int O = I * BITS, W = O >> 5, SH = O & 31;
  uint32_t v = wv[W] >> SH;
  if constexpr (SH + BITS > 32) v |= wv[W + 1] << (32 - SH);
  return __uint_as_float(kTwo23Bits | (v & ((1u << BITS) - 1u)));
}

template <int BITS, bool GIDX, int NT, int... Is>
__device__ __forceinline__ void chunk_fma(const uint32_t (&wv)[BITS], const uint16_t* __restrict__ X, long long ldx,
                                          int c0, float s, float z, const float* __restrict__ srow,
                                          const float* __restrict__ zrow, const int* __restrict__ g_idx,
                                          float (&acc)[NT], std::integer_sequence<int, Is...>) {
  // eight columns at a time: one 16-byte load of X per token
  auto piece = [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    float w[8];
    auto one = [&](auto ic) {
      constexpr int I = decltype(ic)::value;
      const float q = code_of<BITS, 8 * P + I>(wv);
      if constexpr (GIDX) {
        const int gq = __ldg(g_idx + c0 + 8 * P + I);
        w[I] = __fmul_rn(__fsub_rn(q, __fadd_rn(kTwo23, __ldg(zrow + gq))), __ldg(srow + gq));
      } else {
        w[I] = __fmul_rn(__fsub_rn(q, z), s);                // z = 2^23 + zero
      }
    };
    one(std::integral_constant<int, 0>{}); one(std::integral_constant<int, 1>{});
    one(std::integral_constant<int, 2>{}); one(std::integral_constant<int, 3>{});
    one(std::integral_constant<int, 4>{}); one(std::integral_constant<int, 5>{});
    one(std::integral_constant<int, 6>{}); one(std::integral_constant<int, 7>{});
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(X + (long long)t * ldx + c0 + 8 * P));
      const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[t] = fmaf(__uint_as_float(u[k] << 16), w[2 * k], acc[t]);
        acc[t] = fmaf(__uint_as_float(u[k] & 0xFFFF0000u), w[2 * k + 1], acc[t]);
      }
    }
  };
  (piece(std::integral_constant<int, Is>{}), ...);
}

template <int BITS, bool GIDX, int NT>
__global__ void __launch_bounds__(WARPS * 32) dequant_gemv_kernel(const uint32_t* __restrict__ qweight, int wpr,
                                                                  const float* __restrict__ scales,
                                                                  const float* __restrict__ zeros, int G, int cpg,
                                                                  uint32_t cpg_mul, const int* __restrict__ g_idx, int m,
                                                                  int d,
                                                                  const uint16_t* __restrict__ X, long long ldx,
                                                                  float* __restrict__ Y, long long ldy) {
  const int r = blockIdx.x * WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= m) return;
  const uint32_t* row = qweight + (long long)r * wpr;
  const float* srow = scales + (long long)r * G;
  const float* zrow = zeros + (long long)r * G;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
  const int nchunk = d >> 5;
  // UNR chunks per lane are loaded before any is used, so their loads overlap
  constexpr int UNR = BITS >= 8 ? 2 : 4;
  for (int ch0 = lane; ch0 < nchunk; ch0 += 32 * UNR) {
    uint32_t wv[UNR][BITS];
#pragma unroll
    for (int u = 0; u < UNR; ++u)
      if (ch0 + 32 * u < nchunk) load_chunk<BITS>(row, ch0 + 32 * u, wv[u]);
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int ch = ch0 + 32 * u;
      if (ch >= nchunk) break;
      const int c0 = ch << 5;
      float s = 0.0f, z = 0.0f;
      if constexpr (!GIDX) {
        // group of chunk ch: ch / cpg (chunks per group) as a multiply-high by
        // ceil(2^32 / cpg), exact since ch * cpg < 2^32
        const int grp = cpg == 1 ? ch : (int)__umulhi((uint32_t)ch, cpg_mul);
        s = __ldg(srow + grp);
        z = __fadd_rn(kTwo23, __ldg(zrow + grp));
      }
      chunk_fma<BITS, GIDX, NT>(wv[u], X, ldx, c0, s, z, srow, zrow, g_idx, acc, std::make_integer_sequence<int, 4>{});
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) Y[(long long)t * ldy + r] = acc[t];
  }
}

template <int BITS, int NT>
void launch_nt(const uint32_t* qweight, int wpr, const float* scales, const float* zeros, const int* g_idx, int m,
               int d, int G, int gsize, const uint16_t* X, long long ldx, float* Y, long long ldy, cudaStream_t s) {
  const dim3 grid((unsigned)((m + WARPS - 1) / WARPS));
  const int cpg = gsize >> 5;                              // 32-column chunks per group
  const uint32_t cpg_mul = cpg == 1 ? 0u : (uint32_t)((0x100000000ULL + (unsigned long long)cpg - 1) / cpg);
  if (g_idx)
    dequant_gemv_kernel<BITS, true, NT><<<grid, WARPS * 32, 0, s>>>(qweight, wpr, scales, zeros, G, cpg, cpg_mul, g_idx,
                                                                    m, d, X, ldx, Y, ldy);
  else
    dequant_gemv_kernel<BITS, false, NT><<<grid, WARPS * 32, 0, s>>>(qweight, wpr, scales, zeros, G, cpg, cpg_mul,
                                                                     g_idx, m, d, X, ldx, Y, ldy);
  count_launch();
}

// Tokens go in pieces of 8, then one of 4, 2 and 1 as needed (the token count is fixed
// per instantiation, so no instruction is spent on absent tokens).
template <int BITS>
gptq_status launch(const uint32_t* qweight, const float* scales, const float* zeros, const int* g_idx, int m, int d,
                   int G, int gsize, const uint16_t* X, long long ldx, int T, float* Y, long long ldy,
                   cudaStream_t s) {
  const int wpr = (d >> 5) * BITS;
  int t0 = 0;
  for (; t0 + 8 <= T; t0 += 8)
    launch_nt<BITS, 8>(qweight, wpr, scales, zeros, g_idx, m, d, G, gsize, X + (long long)t0 * ldx, ldx,
                       Y + (long long)t0 * ldy, ldy, s);
  if (T - t0 >= 4) {
    launch_nt<BITS, 4>(qweight, wpr, scales, zeros, g_idx, m, d, G, gsize, X + (long long)t0 * ldx, ldx,
                       Y + (long long)t0 * ldy, ldy, s);
    t0 += 4;
  }
  if (T - t0 >= 2) {
    launch_nt<BITS, 2>(qweight, wpr, scales, zeros, g_idx, m, d, G, gsize, X + (long long)t0 * ldx, ldx,
                       Y + (long long)t0 * ldy, ldy, s);
    t0 += 2;
  }
  if (T - t0 >= 1)
    launch_nt<BITS, 1>(qweight, wpr, scales, zeros, g_idx, m, d, G, gsize, X + (long long)t0 * ldx, ldx,
                       Y + (long long)t0 * ldy, ldy, s);
  return check_launch("dequant_gemv_kernel");
}

// ---------------------------------------------------------------------------------
// The same product with the dot products on the tensor cores: for codes in natural
// groups the FMA version above spends about six instructions per code
// (unpack, dequantize, convert the token, FMA) and is bound by instruction issue at a
// quarter of the HBM rate; here the unpacked codes go from registers straight into
// mma.sync (m16n8k16, bf16 operands, fp32 accumulation), which takes eight tokens at the
// cost of one. (The tcgen05 MMA reads its operands from shared memory; staging the
// dequantized codes there would add four bytes of shared-memory traffic per code, more
// than the code's half byte from HBM.)
//
// Per row, code - zero is an integer with |code - zero| <= 255, exact in bf16. At 2, 3
// and 4 bits a pair of codes is taken out of the packed words and OR-ed into the
// mantissas of a bf16 pair of 128 (0x4300: bf16 holds 128 ... 255 exactly), and a bf16
// subtraction of 128 + zero leaves code - zero exactly; 8-bit codes go through fp32
// (see code_pair). The product with a bf16 token is exact; each block of columns that
// shares one (scale, zero) is summed by the tensor core in fp32 and then scaled and
// added in fp32.
//
// Layout: a CTA takes 16 rows, its 8 warps split the row's column blocks. The packed
// row is read in units: one word (CPW = 32 / bits codes) at 2 and 4 bits, three words
// (32 codes) at 3 bits, whose codes straddle words, and two words (8 codes) at 8 bits.
// A block is 4 x UPT units; lane (g, t) of a warp (g = lane / 4, t = lane % 4) holds
// units t*UPT ... t*UPT + UPT - 1 of the block for rows g and g + 8 (the A fragment's
// rows) and the same columns of token g (the B fragment's column). Code pair p of a unit of UC codes is the codes p and
// p + UC/2, which the A fragment's bf16 pair puts at two consecutive k; the B fragment
// pairs the token's values of the same two columns with one byte permute. The order of
// k inside an MMA is thereby a fixed permutation of the block's columns, applied to
// both operands.
namespace tcv {

// GPTQ_GEMV_KERNEL=fma selects the FMA kernel for every case (to compare the two).
inline bool gemv_fma_forced() {
  static const bool forced = [] {
    const char* v = getenv("GPTQ_GEMV_KERNEL");
    return v && std::string(v) == "fma";
  }();
  return forced;
}

constexpr int WARPS = 8, ROWS = 16;
constexpr uint32_t kBf16Pair128 = 0x43004300u;

template <int BITS> constexpr int unit_words() { return BITS == 3 ? 3 : BITS == 8 ? 2 : 1; }
template <int BITS> constexpr int unit_codes() { return BITS == 3 ? 32 : BITS == 8 ? 8 : 32 / BITS; }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// a - c for bf16 pairs as a * 1 + (-c), one fused instruction; exact here (integers
// below 256).
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t neg_c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3F803F80u), "r"(neg_c));
  return d;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Codes p and p + UC/2 of a unit, minus the row's zero, as an exact bf16 pair (p is a
// compile-time constant once the callers' loops are unrolled). neg_z is the bf16 pair
// -(128 + zero) and zf the float 2^23 + zero.
//   2 and 4 bits: the two codes sit 16 bits apart in one word: one shift and one
//     mask-and-OR give the pair (128 + code, 128 + code'), one bf16 subtraction the rest.
//   3 bits: code p starts at bit 3p of the unit's 96 bits and code p + 16 at bit
//     48 + 3p; a funnel shift brings each to bit 0 and 16 of a word, then as above.
//   8 bits (128 + code would need 9 significant bits): byte p of each of the unit's two
//     words is permuted into the mantissa of 2^23, 2^23 + zero is subtracted in fp32
//     (exact), and the two results |code - zero| <= 255 convert to bf16 exactly.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* w, int p, uint32_t neg_z, float zf) {
  if constexpr (BITS == 8) {
    const uint32_t sel = 0x7650u | (uint32_t)p;      // byte p, then the bytes 00 00 4B of 2^23
    const float lo = __fsub_rn(__uint_as_float(prmt(w[0], 0x4B000000u, sel)), zf);
    const float hi = __fsub_rn(__uint_as_float(prmt(w[1], 0x4B000000u, sel)), zf);
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
  } else if constexpr (BITS == 3) {
    const uint32_t lo = (3 * p < 32) ? __funnelshift_r(w[0], w[1], 3 * p) : (w[1] >> (3 * p - 32));
    const uint32_t hi = (3 * p < 32) ? __funnelshift_r(w[1], w[2], 3 * p) : (w[2] >> (3 * p - 32));
    return sub_bf16x2((lo & 0x00000007u) | (hi & 0x00070000u) | kBf16Pair128, neg_z);
  } else {
    constexpr uint32_t MASK2 = ((1u << BITS) - 1u) * 0x00010001u;
    return sub_bf16x2(((w[0] >> (BITS * p)) & MASK2) | kBf16Pair128, neg_z);
  }
}

// N consecutive words (vector loads as wide as the alignment allows: 16 bytes for 4- and
// 8-bit rows, 8 for 2-bit, single words for 3-bit), or zeros for a row past the end.
template <int BITS, int N>
__device__ __forceinline__ void load_words(const uint32_t* __restrict__ p, uint32_t (&w)[N], bool valid) {
  if (!valid) {
#pragma unroll
    for (int u = 0; u < N; ++u) w[u] = 0u;
    return;
  }
  if constexpr ((BITS == 4 || BITS == 8) && N % 4 == 0) {
#pragma unroll
    for (int u = 0; u < N; u += 4) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p + u));
      w[u] = v.x; w[u + 1] = v.y; w[u + 2] = v.z; w[u + 3] = v.w;
    }
  } else if constexpr (BITS != 3 && N >= 2) {
#pragma unroll
    for (int u = 0; u < N; u += 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p + u));
      w[u] = v.x; w[u + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int u = 0; u < N; ++u) w[u] = __ldg(p + u);
  }
}

// bf16 pair (-(128 + zero), -(128 + zero)); zero is an integer in [0, 2^bits - 1], so
// for bits <= 4 128 + zero has at most 8 significant bits and its fp32 encoding's upper
// half is its bf16 (the 8-bit path uses 2^23 + zero instead).
__device__ __forceinline__ uint32_t neg_zero_pair(float z) {
  return ((__float_as_uint(128.0f + z) >> 16) * 0x00010001u) | 0x80008000u;
}

template <int BITS, int UPT>
__global__ void __launch_bounds__(WARPS * 32) gemv_mma_kernel(const uint32_t* __restrict__ qweight, int wpr,
                                                              const float* __restrict__ scales,
                                                              const float* __restrict__ zeros, int G, int bpg,
                                                              uint32_t bpg_mul, int m, int d,
                                                              const uint16_t* __restrict__ X, long long ldx, int T,
                                                              float* __restrict__ Y, long long ldy) {
  constexpr int UW = unit_words<BITS>();          // words of a unit
  constexpr int UC = unit_codes<BITS>();          // codes of a unit
  constexpr int TW = UPT * UW;                    // words of a row per thread and block
  constexpr int VBW = 4 * TW;                     // words of a row in one block
  constexpr int VBC = 4 * UPT * UC;               // columns of one block
  constexpr int SPU = UC / 4;                     // MMAs per unit (two code pairs each)
  constexpr int NB = (16 / TW) > 0 ? 16 / TW : 1; // blocks loaded at once: 2 * TW * NB <= 32 words
  __shared__ float red[WARPS][ROWS][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int r0 = blockIdx.x * ROWS, ra = r0 + g, rb = r0 + g + 8;
  const bool va = ra < m, vb = rb < m, tok = g < T;
  const uint32_t* rowa = qweight + (long long)(va ? ra : 0) * wpr + t * TW;
  const uint32_t* rowb = qweight + (long long)(vb ? rb : 0) * wpr + t * TW;
  const uint16_t* xrow = X + (long long)(tok ? g : 0) * ldx + t * UPT * UC;
  const float* sca = scales + (long long)(va ? ra : 0) * G;
  const float* scb = scales + (long long)(vb ? rb : 0) * G;
  const float* zra = zeros + (long long)(va ? ra : 0) * G;
  const float* zrb = zeros + (long long)(vb ? rb : 0) * G;
  const int nvb = d / VBC;
  float tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  // This warp's blocks v = warp + 8 k, in batches of NB whose words are all requested
  // before the first is multiplied.
  for (int v0 = warp; v0 < nvb; v0 += WARPS * NB) {
    uint32_t wa[NB][TW], wb[NB][TW];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int v = v0 + WARPS * i;
      load_words<BITS, TW>(rowa + v * VBW, wa[i], va && v < nvb);
      load_words<BITS, TW>(rowb + v * VBW, wb[i], vb && v < nvb);
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int v = v0 + WARPS * i;
      if (v >= nvb) continue;
      // group of block v: v / bpg (blocks per group) as a multiply-high by
      // ceil(2^32 / bpg), exact since v * bpg < 2^32
      const int grp = bpg == 1 ? v : (int)__umulhi((uint32_t)v, bpg_mul);
      const float sa = va ? __ldg(sca + grp) : 0.0f, sb = vb ? __ldg(scb + grp) : 0.0f;
      const float zfa = va ? __ldg(zra + grp) : 0.0f, zfb = vb ? __ldg(zrb + grp) : 0.0f;
      const uint32_t za = neg_zero_pair(zfa), zb = neg_zero_pair(zfb);
      const float z23a = __fadd_rn(8388608.0f, zfa), z23b = __fadd_rn(8388608.0f, zfb);
      float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int u = 0; u < UPT; ++u) {
        uint32_t xw[UC / 2];                     // token g's UC columns of unit u, bf16 pairs
#pragma unroll
        for (int q = 0; q < UC / 8; ++q) {
          uint4 xv = make_uint4(0u, 0u, 0u, 0u);
          if (tok) xv = __ldg(reinterpret_cast<const uint4*>(xrow + (v * VBC + u * UC + 8 * q)));
          xw[4 * q] = xv.x; xw[4 * q + 1] = xv.y; xw[4 * q + 2] = xv.z; xw[4 * q + 3] = xv.w;
        }
        const uint32_t* ua = wa[i] + u * UW;
        const uint32_t* ub = wb[i] + u * UW;
#pragma unroll
        for (int j = 0; j < SPU; ++j) {
          // code pairs 2j and 2j + 1: codes (2j, 2j + UC/2) and (2j + 1, 2j + 1 + UC/2)
          const uint32_t a0 = code_pair<BITS>(ua, 2 * j, za, z23a);
          const uint32_t a2 = code_pair<BITS>(ua, 2 * j + 1, za, z23a);
          const uint32_t a1 = code_pair<BITS>(ub, 2 * j, zb, z23b);
          const uint32_t a3 = code_pair<BITS>(ub, 2 * j + 1, zb, z23b);
          const uint32_t b0 = prmt(xw[j], xw[j + UC / 4], 0x5410u);
          const uint32_t b1 = prmt(xw[j], xw[j + UC / 4], 0x7632u);
          mma_bf16(c, a0, a1, a2, a3, b0, b1);
        }
      }
      tot[0] = fmaf(sa, c[0], tot[0]);
      tot[1] = fmaf(sa, c[1], tot[1]);
      tot[2] = fmaf(sb, c[2], tot[2]);
      tot[3] = fmaf(sb, c[3], tot[3]);
    }
  }
  // c[0], c[1]: row g, tokens 2t and 2t + 1; c[2], c[3]: row g + 8
  red[warp][g][2 * t] = tot[0];
  red[warp][g][2 * t + 1] = tot[1];
  red[warp][g + 8][2 * t] = tot[2];
  red[warp][g + 8][2 * t + 1] = tot[3];
  __syncthreads();
  if (threadIdx.x < ROWS * 8) {
    const int i = threadIdx.x >> 3, tk = threadIdx.x & 7;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[w][i][tk];
    if (tk < T && r0 + i < m) Y[(long long)tk * ldy + r0 + i] = sum;
  }
}

// Units of a row per thread in one block (1, 2 or 4), or 0 when the tensor-core path
// does not apply: 2-, 3- and 4-bit codes, natural groups whose width is a multiple of
// four threads' units (a block never straddles two groups), and a width that blocks
// cover. At 3 bits a thread takes one unit of three words.
inline int units_per_thread(int bits, int group_size, long long d) {
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return 0;
  const long long cols4 = 4LL * (bits == 3 ? 32 : bits == 8 ? 8 : 32 / bits);   // four threads' single units
  const long long span = group_size == -1 ? d : group_size;
  if (span % cols4) return 0;
  if (bits == 3) return 1;
  const long long q = span / cols4;
  return (q % 4 == 0) ? 4 : (q % 2 == 0) ? 2 : 1;
}

template <int BITS, int UPT>
gptq_status launch(const uint32_t* qweight, const float* scales, const float* zeros, int m, int d, int G, int gsize,
                   const uint16_t* X, long long ldx, int T, float* Y, long long ldy, cudaStream_t s) {
  const int wpr = d * BITS / 32;
  const int bpg = gsize / (4 * UPT * unit_codes<BITS>());          // blocks per group (a block never straddles two)
  const uint32_t bpg_mul = bpg == 1 ? 0u : (uint32_t)((0x100000000ULL + (unsigned long long)bpg - 1) / bpg);
  const dim3 grid((unsigned)((m + ROWS - 1) / ROWS));
  for (int t0 = 0; t0 < T; t0 += 8) {
    gemv_mma_kernel<BITS, UPT><<<grid, WARPS * 32, 0, s>>>(qweight, wpr, scales, zeros, G, bpg, bpg_mul, m, d,
                                                          X + (long long)t0 * ldx, ldx, std::min(8, T - t0),
                                                          Y + (long long)t0 * ldy, ldy);
    count_launch();
  }
  return check_launch("gemv_mma_kernel");
}

template <int BITS>
gptq_status launch_bits(int upt, const uint32_t* qweight, const float* scales, const float* zeros, int m, int d, int G,
                        int gsize, const uint16_t* X, long long ldx, int T, float* Y, long long ldy, cudaStream_t s) {
  switch (upt) {
    case 4: return launch<BITS, 4>(qweight, scales, zeros, m, d, G, gsize, X, ldx, T, Y, ldy, s);
    case 2: return launch<BITS, 2>(qweight, scales, zeros, m, d, G, gsize, X, ldx, T, Y, ldy, s);
    default: return launch<BITS, 1>(qweight, scales, zeros, m, d, G, gsize, X, ldx, T, Y, ldy, s);
  }
}

}  // namespace tcv

}  // namespace dgemv

gptq_status dequant_gemv_launch(const uint32_t* qweight, const float* scales, const float* zeros, const int32_t* g_idx,
                                long long m, long long d, int bits, int group_size, const uint16_t* X, long long T,
                                long long ldx, float* Y, long long ldy, cudaStream_t s) {
  using namespace dgemv;
  const int G = (group_size == -1) ? 1 : (int)(d / group_size);
  const int gsize = (group_size == -1) ? (int)d : group_size;
  // act-order groups (g_idx) and groups narrower than a block take the FMA kernel
  const int upt = (g_idx && G > 1) ? 0 : tcv::units_per_thread(bits, group_size, d);
  if (upt && !tcv::gemv_fma_forced()) {
    if (bits == 4) return tcv::launch_bits<4>(upt, qweight, scales, zeros, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    if (bits == 3) return tcv::launch<3, 1>(qweight, scales, zeros, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    if (bits == 8) return tcv::launch_bits<8>(upt, qweight, scales, zeros, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    return tcv::launch_bits<2>(upt, qweight, scales, zeros, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
  }
  switch (bits) {
    case 2: return launch<2>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    case 3: return launch<3>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    case 4: return launch<4>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    default: return launch<8>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
  }
}

}  // namespace gptq

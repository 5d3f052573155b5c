// The stored layer used again: Y = X W_hat^T straight from the packed codes.
//
// After quantization a layer keeps its b-bit codes and one (scale, zero) per group of
// columns and is used as before ("GPTQ: fixing errors as you go", on what changes at
// inference time): w_hat[r][j] = (code[r][j] - zero[r][G(j)]) * scale[r][G(j)], with
// G(j) = j / group_size, or g_idx[j] for act-order groups. For the few tokens of a
// decoding step this product reads every code once and is bound by HBM bandwidth.
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
                                                                  const float* __restrict__ zeros, int G, int gsize,
                                                                  const int* __restrict__ g_idx, int m, int d,
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
        const int grp = c0 / gsize;
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
  if (g_idx)
    dequant_gemv_kernel<BITS, true, NT><<<grid, WARPS * 32, 0, s>>>(qweight, wpr, scales, zeros, G, gsize, g_idx, m, d,
                                                                    X, ldx, Y, ldy);
  else
    dequant_gemv_kernel<BITS, false, NT><<<grid, WARPS * 32, 0, s>>>(qweight, wpr, scales, zeros, G, gsize, g_idx, m,
                                                                     d, X, ldx, Y, ldy);
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

}  // namespace dgemv

gptq_status dequant_gemv_launch(const uint32_t* qweight, const float* scales, const float* zeros, const int32_t* g_idx,
                                long long m, long long d, int bits, int group_size, const uint16_t* X, long long T,
                                long long ldx, float* Y, long long ldy, cudaStream_t s) {
  using namespace dgemv;
  const int G = (group_size == -1) ? 1 : (int)(d / group_size);
  const int gsize = (group_size == -1) ? (int)d : group_size;
  switch (bits) {
    case 2: return launch<2>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    case 3: return launch<3>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    case 4: return launch<4>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
    default: return launch<8>(qweight, scales, zeros, g_idx, (int)m, (int)d, G, gsize, X, ldx, (int)T, Y, ldy, s);
  }
}

}  // namespace gptq

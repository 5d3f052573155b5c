// C ABI of the GPTQ library: argument validation, dispatch to the stage kernels,
// status codes and the small host-side state (thread-local error text, launch
// counter, the device error word that bounded waits raise).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "simt_gemm.cuh"

namespace gptq {

// stage entry points (defined in the stage files)
gptq_status syrk_accumulate(const uint16_t* X, long long n, long long d, long long ldx, float* H, long long ldh,
                            float alpha, int zero_first, cudaStream_t stream);
size_t factor_workspace_bytes(long long d);
gptq_status factor_launch(const float* H, long long d, float percdamp, int act_order, int32_t* perm_out, float* Hinv1,
                          void* ws, cudaStream_t s);
gptq_status factor_read_status(const void* ws, long long* info, cudaStream_t s);
size_t quantize_workspace_bytes(long long m, long long d, int blocksize);
gptq_status quantize_launch(const void* W, int w_dtype, long long m, long long d, long long ldw, const float* Hinv1,
                            const int32_t* perm, int bits, int group_size, int blocksize, uint32_t* qweight,
                            float* scales, float* zeros, float* col_losses, void* ws, cudaStream_t s);
gptq_status quantize_read_status(const void* ws, long long* info, cudaStream_t s);
gptq_status unpack_launch(const uint32_t* qweight, long long m, long long d, int bits, uint8_t* codes, cudaStream_t s);
gptq_status dequant_gemv_launch(const uint32_t* qweight, const float* scales, const float* zeros, const int32_t* g_idx,
                                long long m, long long d, int bits, int group_size, const uint16_t* X, long long T,
                                long long ldx, float* Y, long long ldy, cudaStream_t s);
size_t dequant_gemm_workspace_bytes(long long m, long long d);
bool tensor_maps_available();
gptq_status dequant_gemm_launch(const uint32_t* qweight, const float* scales, const float* zeros, long long m,
                                long long d, int bits, int group_size, const uint16_t* X, long long T, long long ldx,
                                void* Y, int y_bf16, long long ldy, void* ws, cudaStream_t s);

namespace {
thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_launches{0};
__device__ int g_device_error_word = 0;

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
int* g_err_addr[kMaxDevices] = {nullptr};
std::mutex g_mu;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

gptq_status set_error(gptq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = 0; }

void count_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

gptq_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return GPTQ_OK;
}

// ---- opt-in launch timing ----
namespace {
struct ProfEntry {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::vector<ProfEntry>* g_prof = nullptr;
int g_prof_state = -1;   // -1 unknown, 0 off, 1 on

void profile_dump() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof) return;
  cudaDeviceSynchronize();
  std::map<std::string, std::pair<int, double>> tot;
  for (const ProfEntry& e : *g_prof) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, e.start, e.stop) == cudaSuccess) {
      auto& t = tot[e.name];
      t.first += 1;
      t.second += ms;
    }
  }
  double all = 0.0;
  for (auto& kv : tot) all += kv.second.second;
  fprintf(stderr, "[gptq profile] %zu scopes, %.3f ms total\n", g_prof->size(), all);
  for (auto& kv : tot)
    fprintf(stderr, "[gptq profile] %-28s %6d x  %10.3f ms  (%8.2f us each)\n", kv.first.c_str(), kv.second.first,
            kv.second.second, 1e3 * kv.second.second / kv.second.first);
}
}  // namespace

bool profiling_enabled() {
  if (g_prof_state < 0) {
    const char* v = getenv("GPTQ_PROFILE");
    g_prof_state = (v && v[0] == '1') ? 1 : 0;
    if (g_prof_state) {
      g_prof = new std::vector<ProfEntry>();
      atexit(profile_dump);
    }
  }
  return g_prof_state == 1;
}

cudaEvent_t profile_event() {
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void profile_record(const char* name, cudaEvent_t start, cudaEvent_t stop) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof) g_prof->push_back({name, start, stop});
}

int sm_count() {
  const int dev = current_device();
  if (!g_sm_count[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 1;
  }
  return g_sm_count[dev];
}

int* device_error_word() {
  const int dev = current_device();
  if (!g_err_addr[dev]) {
    std::lock_guard<std::mutex> lk(g_mu);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) == cudaSuccess) g_err_addr[dev] = reinterpret_cast<int*>(p);
  }
  return g_err_addr[dev];
}

gptq_status check_quantize_settings(long long m, long long d, int w_dtype, int bits, int group_size, int blocksize) {
  if (m < 1 || m > (1LL << 30) || d < 1 || d > 65536 || m * d > (1LL << 36))
    return set_error(GPTQ_ERR_INVALID_ARG, "m or d out of range");
  if (w_dtype != 0 && w_dtype != 1) return set_error(GPTQ_ERR_INVALID_ARG, "w_dtype must be 0 (fp32) or 1 (bf16)");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return set_error(GPTQ_ERR_INVALID_ARG, "bits must be 2, 3, 4 or 8");
  if (blocksize < 1 || blocksize > 256) return set_error(GPTQ_ERR_INVALID_ARG, "blocksize must be in [1, 256]");
  if (group_size != -1) {
    if (group_size < 1 || d % group_size) return set_error(GPTQ_ERR_INVALID_ARG, "d must be a multiple of group_size");
    if (group_size % blocksize && blocksize % group_size)
      return set_error(GPTQ_ERR_INVALID_ARG, "group_size and blocksize must divide one another");
  }
  if (blocksize != 32 && blocksize != 64 && blocksize != 128)
    return set_error(GPTQ_ERR_UNSUPPORTED, "this build runs blocksize 32, 64 or 128");
  if (group_size != -1 && group_size % 32)
    return set_error(GPTQ_ERR_UNSUPPORTED, "this build runs group sizes that are multiples of 32 (or -1)");
  return GPTQ_OK;
}

// ---- self-test of the bounded waits ----
namespace {
__device__ unsigned g_selftest_counter = 0;   // nothing ever publishes on it
__device__ int g_selftest_gave_up = 0;

// One thread runs one of the library's bounded waits on something that never
// completes, with a short limit: which = 0 the counter wait the Cholesky panels use
// (acquire loads of a counter in global memory), which = 1 the mbarrier wait every
// copy and tensor-core hand-over uses (a barrier that nothing arrives on). Nothing is
// in flight when it gives up; it reports the timeout like the real kernels do.
__global__ void wait_selftest_kernel(int which, unsigned long long limit_ns, int* err_word) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  bool done;
  if (which == 0) {
    done = wait_counter_bounded(&g_selftest_counter, 1u, limit_ns);
  } else {
    mbar_init(&bar, 1);
    fence_mbar_init();
    done = mbar_wait_bounded(&bar, 0, nullptr, limit_ns);
  }
  g_selftest_gave_up = done ? 0 : 1;
  if (!done) report_device_error(err_word, DEVERR_TIMEOUT);
}
}  // namespace

}  // namespace gptq

using namespace gptq;

extern "C" {

gptq_status gptq_wait_selftest(int which, int64_t limit_ns, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (which != 0 && which != 1) return set_error(GPTQ_ERR_INVALID_ARG, "which must be 0 (counter) or 1 (mbarrier)");
  if (limit_ns < 1000 || limit_ns > 1000000000)
    return set_error(GPTQ_ERR_INVALID_ARG, "limit_ns must be in [1e3, 1e9]");
  int* word = device_error_word();
  if (!word) return set_error(GPTQ_ERR_CUDA, "device error word is not available");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  wait_selftest_kernel<<<1, 32, 0, s>>>(which, (unsigned long long)limit_ns, word);
  count_launch();
  if (gptq_status st = check_launch("wait_selftest_kernel")) return st;
  if (cudaStreamSynchronize(s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaStreamSynchronize failed");
  int gave_up = 0;
  if (cudaMemcpyFromSymbol(&gave_up, g_selftest_gave_up, sizeof(int)) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "reading the self-test result failed");
  if (gave_up) return set_error(GPTQ_ERR_TIMEOUT, "the %s wait gave up after %lld ns", which ? "mbarrier" : "counter",
                                (long long)limit_ns);
  return GPTQ_OK;
}

const char* gptq_status_string(int status) {
  switch (status) {
    case GPTQ_OK: return "GPTQ_OK";
    case GPTQ_ERR_INVALID_ARG: return "GPTQ_ERR_INVALID_ARG";
    case GPTQ_ERR_NOT_PD: return "GPTQ_ERR_NOT_PD";
    case GPTQ_ERR_NONFINITE: return "GPTQ_ERR_NONFINITE";
    case GPTQ_ERR_UNSUPPORTED: return "GPTQ_ERR_UNSUPPORTED";
    case GPTQ_ERR_CUDA: return "GPTQ_ERR_CUDA";
    case GPTQ_ERR_TIMEOUT: return "GPTQ_ERR_TIMEOUT";
    default: return "GPTQ_ERR_UNKNOWN";
  }
}

const char* gptq_last_error(void) { return g_last_error; }

int gptq_version(void) { return 100; }

uint64_t gptq_launch_count(void) { return (uint64_t)g_launches.load(); }

gptq_status gptq_device_check(gptq_stream_t stream) {
  int* word = device_error_word();
  if (!word) return set_error(GPTQ_ERR_CUDA, "device error word is not available");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaStreamSynchronize failed");
  int v = 0;
  if (cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "reading the device error word failed");
  if (v) {
    const int zero = 0;
    cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
  }
  if (v & DEVERR_TIMEOUT) return set_error(GPTQ_ERR_TIMEOUT, "an on-device wait gave up");
  if (v & DEVERR_NONFINITE) return set_error(GPTQ_ERR_NONFINITE, "a kernel met a NaN or an Inf");
  return GPTQ_OK;
}

gptq_status gptq_hessian_accumulate(const uint16_t* X, int64_t n, int64_t d, int64_t ldx, float* H, int64_t ldh,
                                    float alpha, int zero_first, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!H) return set_error(GPTQ_ERR_INVALID_ARG, "H is NULL");
  if (d < 1 || d > 65536 || d % 8) return set_error(GPTQ_ERR_INVALID_ARG, "d must be in [8, 65536] and a multiple of 8");
  if (n < 0 || n > (int64_t)0x7FFFFF00) return set_error(GPTQ_ERR_INVALID_ARG, "n out of range");
  if (ldh < d || ldh % 4 || !aligned(H, 16))
    return set_error(GPTQ_ERR_INVALID_ARG, "H must be 16-byte aligned with ldh >= d and ldh %% 4 == 0");
  if (n > 0) {
    if (!X) return set_error(GPTQ_ERR_INVALID_ARG, "X is NULL");
    if (ldx < d || ldx % 8 || !aligned(X, 16))
      return set_error(GPTQ_ERR_INVALID_ARG, "X must be 16-byte aligned with ldx >= d and ldx %% 8 == 0");
  }
  if (!(alpha == alpha)) return set_error(GPTQ_ERR_INVALID_ARG, "alpha is NaN");
  if (n == 0 && !zero_first) return GPTQ_OK;
  return syrk_accumulate(X, n, d, ldx, H, ldh, alpha, zero_first, reinterpret_cast<cudaStream_t>(stream));
}

size_t gptq_workspace_size(int which, int64_t m, int64_t d, int bits, int group_size, int blocksize) {
  (void)bits;
  (void)group_size;
  if (d < 1 || d > 65536) return 0;
  if (which == GPTQ_WS_FACTOR) return factor_workspace_bytes(d);
  if (which == GPTQ_WS_QUANTIZE) {
    if (m < 1 || m > (int64_t)1 << 30) return 0;
    if (blocksize != 32 && blocksize != 64 && blocksize != 128) return 0;
    return quantize_workspace_bytes(m, d, blocksize);
  }
  if (which == GPTQ_WS_DEQUANT_GEMM) {
    if (m < 1 || m > (int64_t)1 << 30 || d % 32) return 0;
    return dequant_gemm_workspace_bytes(m, d);
  }
  return 0;
}

gptq_status gptq_factor(const float* H, int64_t d, float percdamp, int act_order, int32_t* perm_out, float* Hinv1,
                        void* ws, size_t ws_bytes, int64_t* info, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!H || !Hinv1 || !ws) return set_error(GPTQ_ERR_INVALID_ARG, "H, Hinv1 and ws must not be NULL");
  if (d < 1 || d > 65536) return set_error(GPTQ_ERR_INVALID_ARG, "d must be in [1, 65536]");
  if (!(percdamp >= 0.0f) || percdamp > 1e30f) return set_error(GPTQ_ERR_INVALID_ARG, "percdamp must be finite and >= 0");
  if (act_order && !perm_out) return set_error(GPTQ_ERR_INVALID_ARG, "act_order needs perm_out");
  if (!aligned(ws, 256)) return set_error(GPTQ_ERR_INVALID_ARG, "ws must be 256-byte aligned");
  if (ws_bytes < factor_workspace_bytes(d))
    return set_error(GPTQ_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, factor_workspace_bytes(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gptq_status st = factor_launch(H, d, percdamp, act_order, perm_out, Hinv1, ws, s);
  if (st) return st;
  if (!info) return GPTQ_OK;
  long long inf = -1;
  st = factor_read_status(ws, &inf, s);
  *info = inf;
  return st;
}

gptq_status gptq_factor_status(const void* ws, int64_t* info, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!ws) return set_error(GPTQ_ERR_INVALID_ARG, "ws is NULL");
  long long inf = -1;
  gptq_status st = factor_read_status(ws, &inf, reinterpret_cast<cudaStream_t>(stream));
  if (info) *info = inf;
  return st;
}

gptq_status gptq_quantize_layer(const void* W, int w_dtype, int64_t m, int64_t d, int64_t ldw, const float* Hinv1,
                                const int32_t* perm, int bits, int group_size, int blocksize, uint32_t* qweight,
                                float* scales, float* zeros, float* col_losses, void* ws, size_t ws_bytes,
                                int64_t* info, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!W || !Hinv1 || !qweight || !scales || !zeros || !col_losses || !ws)
    return set_error(GPTQ_ERR_INVALID_ARG, "a required pointer is NULL");
  if (gptq_status st = check_quantize_settings(m, d, w_dtype, bits, group_size, blocksize)) return st;
  if (ldw < d) return set_error(GPTQ_ERR_INVALID_ARG, "ldw < d");
  if (!aligned(ws, 256)) return set_error(GPTQ_ERR_INVALID_ARG, "ws must be 256-byte aligned");
  const size_t need = quantize_workspace_bytes(m, d, blocksize);
  if (ws_bytes < need) return set_error(GPTQ_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gptq_status st = quantize_launch(W, w_dtype, m, d, ldw, Hinv1, perm, bits, group_size, blocksize, qweight, scales,
                                   zeros, col_losses, ws, s);
  if (st || !info) return st;
  long long inf = 0;
  st = quantize_read_status(ws, &inf, s);
  *info = inf;
  return st;
}

gptq_status gptq_unpack_codes(const uint32_t* qweight, int64_t m, int64_t d, int bits, uint8_t* codes,
                              gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!qweight || !codes) return set_error(GPTQ_ERR_INVALID_ARG, "NULL pointer");
  if (m < 0 || m > ((int64_t)1 << 30) || d < 0 || d > 65536 || m * d > ((int64_t)1 << 36))
    return set_error(GPTQ_ERR_INVALID_ARG, "m in [0, 2^30], d in [0, 65536] and m * d <= 2^36 are required");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return set_error(GPTQ_ERR_INVALID_ARG, "bits must be 2, 3, 4 or 8");
  return unpack_launch(qweight, m, d, bits, codes, reinterpret_cast<cudaStream_t>(stream));
}

gptq_status gptq_dequant_gemv(const uint32_t* qweight, const float* scales, const float* zeros, const int32_t* g_idx,
                              int64_t m, int64_t d, int bits, int group_size, const uint16_t* X, int64_t T,
                              int64_t ldx, float* Y, int64_t ldy, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!qweight || !scales || !zeros || (T > 0 && (!X || !Y))) return set_error(GPTQ_ERR_INVALID_ARG, "NULL pointer");
  if (m < 1 || m > ((int64_t)1 << 30) || d < 32 || d > 65536 || d % 32)
    return set_error(GPTQ_ERR_INVALID_ARG, "m >= 1 and d a multiple of 32 in [32, 65536] are required");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return set_error(GPTQ_ERR_INVALID_ARG, "bits must be 2, 3, 4 or 8");
  if (group_size != -1 && (group_size < 32 || group_size % 32 || d % group_size))
    return set_error(GPTQ_ERR_INVALID_ARG, "group_size must be -1 or a multiple of 32 that divides d");
  if (T < 0 || T > 0x7FFFFFFF || ldx < d || ldx % 8 || ldy < m)
    return set_error(GPTQ_ERR_INVALID_ARG, "bad T, ldx or ldy");
  const size_t qa = (bits == 4 || bits == 8) ? 16 : (bits == 2 ? 8 : 4);
  if (!aligned(qweight, qa) || (T > 0 && !aligned(X, 16)) || !aligned(scales, 4) || !aligned(zeros, 4))
    return set_error(GPTQ_ERR_INVALID_ARG, "qweight (16 bytes for 4 and 8 bits, 8 for 2) or X (16 bytes) misaligned");
  if (T == 0) return GPTQ_OK;
  return dequant_gemv_launch(qweight, scales, zeros, g_idx, m, d, bits, group_size, X, T, ldx, Y, ldy,
                             reinterpret_cast<cudaStream_t>(stream));
}

gptq_status gptq_dequant_gemm(const uint32_t* qweight, const float* scales, const float* zeros, int64_t m, int64_t d,
                              int bits, int group_size, const uint16_t* X, int64_t T, int64_t ldx, void* Y, int y_bf16,
                              int64_t ldy, void* ws, size_t ws_bytes, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!qweight || !scales || !zeros || !ws || (T > 0 && (!X || !Y))) return set_error(GPTQ_ERR_INVALID_ARG, "NULL pointer");
  if (m < 1 || m > ((int64_t)1 << 30) || d < 32 || d > 65536 || d % 32)
    return set_error(GPTQ_ERR_INVALID_ARG, "m >= 1 and d a multiple of 32 in [32, 65536] are required");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8) return set_error(GPTQ_ERR_INVALID_ARG, "bits must be 2, 3, 4 or 8");
  if (group_size != -1 && (group_size < 32 || group_size % 32 || d % group_size))
    return set_error(GPTQ_ERR_INVALID_ARG, "group_size must be -1 or a multiple of 32 that divides d");
  if (y_bf16 != 0 && y_bf16 != 1) return set_error(GPTQ_ERR_INVALID_ARG, "y_bf16 must be 0 (fp32) or 1 (bf16)");
  if (T < 0 || T > 0x7FFFFFFF || ldx < d || ldx % 8 || ldy < m)
    return set_error(GPTQ_ERR_INVALID_ARG, "bad T, ldx or ldy");
  if (((T + 127) / 128) * ((m + 127) / 128) > 0x7FFFFFFF) return set_error(GPTQ_ERR_INVALID_ARG, "too many output tiles");
  if (!aligned(qweight, 4) || !aligned(scales, 4) || !aligned(zeros, 4) || (T > 0 && !aligned(X, 16)))
    return set_error(GPTQ_ERR_INVALID_ARG, "X must be 16-byte aligned (qweight, scales, zeros 4-byte)");
  if (!aligned(ws, 256)) return set_error(GPTQ_ERR_INVALID_ARG, "ws must be 256-byte aligned");
  if (ws_bytes < dequant_gemm_workspace_bytes(m, d))
    return set_error(GPTQ_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes,
                     dequant_gemm_workspace_bytes(m, d));
  if (T == 0) return GPTQ_OK;
  if (!tensor_maps_available()) return set_error(GPTQ_ERR_UNSUPPORTED, "the tensor-map encoder is not available");
  return dequant_gemm_launch(qweight, scales, zeros, m, d, bits, group_size, X, T, ldx, Y, y_bf16, ldy, ws,
                             reinterpret_cast<cudaStream_t>(stream));
}

gptq_status gptq_gemm_f32(int engine, int a_kmajor, int b_kmajor, int64_t M, int64_t N, int64_t K, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float* C, int64_t ldc, float alpha, float beta,
                          int lower_tiles, gptq_stream_t stream) {
  g_last_error[0] = 0;
  if (!A || !B || !C) return set_error(GPTQ_ERR_INVALID_ARG, "NULL pointer");
  if (M < 0 || N < 0 || K < 0 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30))
    return set_error(GPTQ_ERR_INVALID_ARG, "size out of range");
  if (lower_tiles && M != N) return set_error(GPTQ_ERR_INVALID_ARG, "lower_tiles needs M == N");
  if (ldc < N || lda < (a_kmajor ? K : M) || ldb < (b_kmajor ? K : N))
    return set_error(GPTQ_ERR_INVALID_ARG, "leading dimension too small");
  if (engine != 0 && engine != 1) return set_error(GPTQ_ERR_INVALID_ARG, "engine must be 0 or 1");
  simt::GemmArgs g{};
  g.M = (int)M; g.N = (int)N; g.K = (int)K; g.M_last = (int)M; g.K_last = (int)K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc;
  g.alpha = alpha; g.beta = beta;
  g.lower_tiles = lower_tiles;
  g.vec = simt::aligned16(A) && simt::aligned16(B) && simt::aligned16(C) && lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0 || N == 0) return GPTQ_OK;
  return engine == 0 ? tc_gemm(g, 1, a_kmajor != 0, b_kmajor != 0, s) : simt::gemm(g, 1, a_kmajor != 0, b_kmajor != 0, s);
}

}  // extern "C"

// gptq_factor_static: the stage-2 factor with its scratch in library-owned device
// memory, for callers that cannot allocate device memory themselves.
//
// Who needs this: code that runs inside a host process whose runtime owns the GPU's
// memory budget (a serving engine or framework plugin that has reserved the device
// through its own pool and forbids side allocations), and pipelines that cannot
// afford cudaMalloc's implicit device-wide synchronization between their launches.
// Such callers can still hand over the inputs and outputs they already own (H,
// Hinv1, perm_out), but not a d x d workspace.
//
// The scratch is one file-scope device array sized for d <= kStaticMaxD. Every GPU
// that loads this library holds it until the process exits. Host code cannot use the
// array's name as a device address (in host code it names a host-side stand-in), so
// the first call on each device, with that device current, asks the runtime for the
// array's device address with cudaGetSymbolAddress and caches it; kernels receive that
// address as their workspace pointer.
#include <mutex>

#include "common.cuh"

namespace gptq {

gptq_status factor_launch(const float* H, long long d, float percdamp, int act_order, int32_t* perm_out, float* Hinv1,
                          void* ws, cudaStream_t s);
gptq_status factor_read_status(const void* ws, long long* info, cudaStream_t s);
size_t factor_workspace_bytes(long long d);

namespace {

constexpr long long kStaticMaxD = 2048;
// status header (256 bytes) + the d x d fp32 matrix the factorization works in + the
// low parts of two 128-column panels (2 x d x 128 fp32)
constexpr size_t kStaticScratchBytes =
    256 + (size_t)kStaticMaxD * kStaticMaxD * sizeof(float) + 2 * (size_t)kStaticMaxD * 128 * sizeof(float);

static __device__ __align__(256) unsigned char g_factor_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_factor_scratch on the current device (set up once per device).
gptq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_error(GPTQ_ERR_CUDA, "gptq_factor_static: no usable current device");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_factor_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(GPTQ_ERR_CUDA, "gptq_factor_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GPTQ_OK;
}

}  // namespace
}  // namespace gptq

using namespace gptq;

extern "C" gptq_status gptq_factor_static(const float* H, int64_t d, float percdamp, int act_order,
                                          int32_t* perm_out, float* Hinv1, int64_t* info, gptq_stream_t stream) {
  clear_error();
  if (!H || !Hinv1) return set_error(GPTQ_ERR_INVALID_ARG, "H and Hinv1 must not be NULL");
  if (d < 1) return set_error(GPTQ_ERR_INVALID_ARG, "d must be >= 1");
  if (d > kStaticMaxD)
    return set_error(GPTQ_ERR_INVALID_ARG, "gptq_factor_static: d = %lld exceeds the static scratch limit d <= %lld",
                     (long long)d, kStaticMaxD);
  if (!(percdamp >= 0.0f) || percdamp > 1e30f) return set_error(GPTQ_ERR_INVALID_ARG, "percdamp must be finite and >= 0");
  if (act_order && !perm_out) return set_error(GPTQ_ERR_INVALID_ARG, "act_order needs perm_out");
  // The outcome (pivot failure, NaN/Inf, timeout) stays in the shared scratch's header,
  // which the next call overwrites: it is read back here, so info is required.
  if (!info) return set_error(GPTQ_ERR_INVALID_ARG, "gptq_factor_static needs info (its outcome is read back at once)");
  if (factor_workspace_bytes(d) > kStaticScratchBytes)
    return set_error(GPTQ_ERR_INVALID_ARG, "gptq_factor_static: scratch too small for d = %lld", (long long)d);
  void* scratch = nullptr;
  gptq_status st = scratch_address(&scratch);
  if (st) return st;
  // Nothing in the scratch has to start at zero: the first kernel of the factor writes
  // the status header, and the matrix is fully written before it is read.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = factor_launch(H, d, percdamp, act_order, perm_out, Hinv1, scratch, s);
  if (st) return st;
  long long inf = -1;
  st = factor_read_status(scratch, &inf, s);
  *info = inf;
  return st;
}

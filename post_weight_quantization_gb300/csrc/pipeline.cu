// One layer end to end from host memory: the calibration tokens stream to the GPU in
// chunks on a copy stream while the Hessian of the chunk before runs on the caller's
// stream, then W is copied, the factor and the column loop run, and the outputs go back
// to host memory ("The GPTQ Algorithm", procedure steps 2-4 for one layer;
// "GPTQ-style round-to-nearest with Hessian weighting", section "Computing the
// Hessian", where H is summed batch by batch).
//
// The pipeline is host code over the library's own entry points. Its device memory is
// one allocation made at creation, carved into 256-byte aligned pieces; a run enqueues
// copies and launches and returns, ordered against the run before it by an event.
#include <cstring>
#include <new>

#include "common.cuh"

namespace gptq {
size_t factor_workspace_bytes(long long d);
size_t quantize_workspace_bytes(long long m, long long d, int blocksize);
gptq_status factor_read_status(const void* ws, long long* info, cudaStream_t s);
gptq_status quantize_read_status(const void* ws, long long* info, cudaStream_t s);

namespace {
constexpr long long kMaxChunk = 1LL << 24;
// The last chunk of a run is cut into four pieces when it holds at least this many
// tokens: no copy overlaps the Hessian of the final piece, so that piece is kept short.
constexpr long long kSplitLast = 4096;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace
}  // namespace gptq

struct gptq_pipeline {
  int device = 0;
  long long m = 0, d = 0, chunk = 0, words = 0, G = 0;
  int w_dtype = 0, bits = 0, group_size = 0, blocksize = 0, act_order = 0;
  float percdamp = 0.0f;
  char* arena = nullptr;
  uint16_t* xbuf[2] = {nullptr, nullptr};
  void* W = nullptr;
  float* H = nullptr;
  float* Hinv1 = nullptr;
  int32_t* perm = nullptr;
  void* ws_f = nullptr;
  void* ws_q = nullptr;
  size_t ws_f_bytes = 0, ws_q_bytes = 0;
  uint32_t* qweight = nullptr;
  float* scales = nullptr;
  float* zeros = nullptr;
  float* col_losses = nullptr;
  cudaStream_t copy = nullptr;
  cudaEvent_t start = nullptr, w_copied = nullptr, copy_end = nullptr, done = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr}, consumed[2] = {nullptr, nullptr};
};

using namespace gptq;

namespace {

void release(gptq_pipeline* p) {
  if (p->copy) cudaStreamSynchronize(p->copy);
  if (p->done) cudaEventSynchronize(p->done);
  cudaEvent_t evs[] = {p->start,     p->w_copied,   p->copy_end,   p->done,
                       p->copied[0], p->copied[1], p->consumed[0], p->consumed[1]};
  for (cudaEvent_t e : evs)
    if (e) cudaEventDestroy(e);
  if (p->copy) cudaStreamDestroy(p->copy);
  if (p->arena) cudaFree(p->arena);
  delete p;
}

// Host rows -> device rows (device row stride = width): one copy when the host rows are
// dense, else a pitched copy.
cudaError_t copy_rows_h2d(void* dst, const void* src, long long rows, size_t row_bytes, size_t src_pitch,
                          cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (src_pitch == row_bytes) return cudaMemcpyAsync(dst, src, (size_t)rows * row_bytes, cudaMemcpyHostToDevice, s);
  return cudaMemcpy2DAsync(dst, row_bytes, src, src_pitch, row_bytes, (size_t)rows, cudaMemcpyHostToDevice, s);
}

}  // namespace

extern "C" {

gptq_status gptq_pipeline_create(int64_t m, int64_t d, int w_dtype, int bits, int group_size, int blocksize,
                                 float percdamp, int act_order, int64_t chunk_tokens, gptq_pipeline** out) {
  clear_error();
  if (!out) return set_error(GPTQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (gptq_status st = check_quantize_settings(m, d, w_dtype, bits, group_size, blocksize)) return st;
  if (d < 8 || d % 8) return set_error(GPTQ_ERR_INVALID_ARG, "d must be a multiple of 8");
  if (!(percdamp >= 0.0f) || percdamp > 1e30f) return set_error(GPTQ_ERR_INVALID_ARG, "percdamp must be finite and >= 0");
  if (chunk_tokens < 1 || chunk_tokens > kMaxChunk)
    return set_error(GPTQ_ERR_INVALID_ARG, "chunk_tokens must be in [1, 2^24]");

  gptq_pipeline* p = new (std::nothrow) gptq_pipeline();
  if (!p) return set_error(GPTQ_ERR_CUDA, "out of host memory");
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return set_error(GPTQ_ERR_CUDA, "cudaGetDevice failed");
  }
  p->m = m;
  p->d = d;
  p->chunk = chunk_tokens;
  p->w_dtype = w_dtype;
  p->bits = bits;
  p->group_size = group_size;
  p->blocksize = blocksize;
  p->act_order = act_order ? 1 : 0;
  p->percdamp = percdamp;
  p->words = (d * bits + 31) / 32;
  p->G = group_size == -1 ? 1 : d / group_size;
  p->ws_f_bytes = factor_workspace_bytes(d);
  p->ws_q_bytes = quantize_workspace_bytes(m, d, blocksize);

  // arena: chunk buffers, W, H, Hinv1, perm, workspaces, outputs
  const size_t sizes[] = {
      (size_t)chunk_tokens * d * 2, (size_t)chunk_tokens * d * 2,  // xbuf[0], xbuf[1]
      (size_t)m * d * (w_dtype ? 2 : 4),                           // W
      (size_t)d * d * 4, (size_t)d * d * 4,                        // H, Hinv1
      (size_t)d * 4,                                               // perm
      p->ws_f_bytes, p->ws_q_bytes,                                // workspaces
      (size_t)m * p->words * 4,                                    // qweight
      (size_t)m * p->G * 4, (size_t)m * p->G * 4,                  // scales, zeros
      (size_t)d * 4};                                              // col_losses
  constexpr int kParts = sizeof(sizes) / sizeof(sizes[0]);
  size_t off[kParts], total = 0;
  for (int i = 0; i < kParts; ++i) {
    off[i] = total;
    total += round256(sizes[i]);
  }
  if (cudaMalloc(&p->arena, total) != cudaSuccess) {
    cudaGetLastError();
    p->arena = nullptr;
    release(p);
    return set_error(GPTQ_ERR_CUDA, "cudaMalloc of %zu bytes failed", total);
  }
  char* a = p->arena;
  p->xbuf[0] = reinterpret_cast<uint16_t*>(a + off[0]);
  p->xbuf[1] = reinterpret_cast<uint16_t*>(a + off[1]);
  p->W = a + off[2];
  p->H = reinterpret_cast<float*>(a + off[3]);
  p->Hinv1 = reinterpret_cast<float*>(a + off[4]);
  p->perm = reinterpret_cast<int32_t*>(a + off[5]);
  p->ws_f = a + off[6];
  p->ws_q = a + off[7];
  p->qweight = reinterpret_cast<uint32_t*>(a + off[8]);
  p->scales = reinterpret_cast<float*>(a + off[9]);
  p->zeros = reinterpret_cast<float*>(a + off[10]);
  p->col_losses = reinterpret_cast<float*>(a + off[11]);

  // A non-blocking copy stream: no implicit ordering against the legacy default stream,
  // so a caller on the NULL stream still gets copies that overlap the Hessian.
  bool ok = cudaStreamCreateWithFlags(&p->copy, cudaStreamNonBlocking) == cudaSuccess;
  cudaEvent_t* evs[] = {&p->start,     &p->w_copied,  &p->copy_end,    &p->done,
                        &p->copied[0], &p->copied[1], &p->consumed[0], &p->consumed[1]};
  for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release(p);
    return set_error(GPTQ_ERR_CUDA, "creating the copy stream or its events failed");
  }
  *out = p;
  return GPTQ_OK;
}

gptq_status gptq_pipeline_run(gptq_pipeline* p, const void* W, int64_t ldw, const uint16_t* X, int64_t n, int64_t ldx,
                              uint32_t* qweight, float* scales, float* zeros, float* col_losses, int32_t* perm,
                              gptq_stream_t stream) {
  clear_error();
  if (!p) return set_error(GPTQ_ERR_INVALID_ARG, "pipeline is NULL");
  if (!W || !qweight || !scales || !zeros || !col_losses || (n > 0 && !X))
    return set_error(GPTQ_ERR_INVALID_ARG, "a required host pointer is NULL");
  if (ldw < p->d || (n > 0 && ldx < p->d)) return set_error(GPTQ_ERR_INVALID_ARG, "ldw and ldx must be >= d");
  if (n < 0 || n > (1LL << 40)) return set_error(GPTQ_ERR_INVALID_ARG, "n out of range");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device)
    return set_error(GPTQ_ERR_INVALID_ARG, "the pipeline belongs to device %d, the current device is %d", p->device, dev);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long d = p->d;
  const size_t xrow = (size_t)d * 2;

  // After the previous run on this pipeline, whatever stream it used; the copies follow
  // everything enqueued on `s` before this call.
  if (cudaStreamWaitEvent(s, p->done, 0) != cudaSuccess || cudaEventRecord(p->start, s) != cudaSuccess ||
      cudaStreamWaitEvent(p->copy, p->start, 0) != cudaSuccess)
    return set_error(GPTQ_ERR_CUDA, "ordering the run after the previous one failed");

  gptq_status st = GPTQ_OK;
  bool first = true;
  int piece = 0;
  auto hessian_piece = [&](long long t0, long long t1) -> gptq_status {
    const int b = piece & 1;
    if (piece >= 2 && cudaStreamWaitEvent(p->copy, p->consumed[b], 0) != cudaSuccess)
      return set_error(GPTQ_ERR_CUDA, "waiting for a chunk buffer failed");
    if (copy_rows_h2d(p->xbuf[b], X + t0 * ldx, t1 - t0, xrow, (size_t)ldx * 2, p->copy) != cudaSuccess ||
        cudaEventRecord(p->copied[b], p->copy) != cudaSuccess || cudaStreamWaitEvent(s, p->copied[b], 0) != cudaSuccess)
      return set_error(GPTQ_ERR_CUDA, "copying tokens %lld..%lld to the device failed", t0, t1);
    if (gptq_status e = gptq_hessian_accumulate(p->xbuf[b], t1 - t0, d, d, p->H, d, 2.0f, first ? 1 : 0, stream))
      return e;
    if (cudaEventRecord(p->consumed[b], s) != cudaSuccess) return set_error(GPTQ_ERR_CUDA, "cudaEventRecord failed");
    first = false;
    ++piece;
    return GPTQ_OK;
  };
  for (long long t0 = 0; t0 < n && !st; t0 += p->chunk) {
    const long long t1 = t0 + p->chunk < n ? t0 + p->chunk : n;
    if (t1 == n && t1 - t0 >= kSplitLast) {
      const long long q = (t1 - t0) / 4;
      for (int k = 0; k < 4 && !st; ++k) st = hessian_piece(t0 + k * q, k < 3 ? t0 + (k + 1) * q : t1);
    } else {
      st = hessian_piece(t0, t1);
    }
  }
  if (!st && first) st = gptq_hessian_accumulate(nullptr, 0, d, d, p->H, d, 2.0f, 1, stream);   // no tokens: H = 0

  // W behind the last token chunk on the copy stream
  if (!st) {
    const size_t wrow = (size_t)d * (p->w_dtype ? 2 : 4);
    if (copy_rows_h2d(p->W, W, p->m, wrow, (size_t)ldw * (p->w_dtype ? 2 : 4), p->copy) != cudaSuccess ||
        cudaEventRecord(p->w_copied, p->copy) != cudaSuccess)
      st = set_error(GPTQ_ERR_CUDA, "copying W to the device failed");
  }
  if (!st) st = gptq_factor(p->H, d, p->percdamp, p->act_order, p->perm, p->Hinv1, p->ws_f, p->ws_f_bytes, nullptr, stream);
  if (!st && cudaStreamWaitEvent(s, p->w_copied, 0) != cudaSuccess)
    st = set_error(GPTQ_ERR_CUDA, "waiting for the copy of W failed");
  if (!st)
    st = gptq_quantize_layer(p->W, p->w_dtype, p->m, d, d, p->Hinv1, p->act_order ? p->perm : nullptr, p->bits,
                             p->group_size, p->blocksize, p->qweight, p->scales, p->zeros, p->col_losses, p->ws_q,
                             p->ws_q_bytes, nullptr, stream);
  if (!st) {
    const size_t sg = (size_t)p->m * p->G * 4;
    bool ok = cudaMemcpyAsync(qweight, p->qweight, (size_t)p->m * p->words * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(scales, p->scales, sg, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(zeros, p->zeros, sg, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(col_losses, p->col_losses, (size_t)d * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    if (ok && p->act_order && perm)
      ok = cudaMemcpyAsync(perm, p->perm, (size_t)d * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    if (!ok) st = set_error(GPTQ_ERR_CUDA, "copying the outputs to the host failed");
  }
  // The next run waits for this one, also when this one stopped early: its copy stream
  // joins `s` so nothing of this run is still writing a device buffer afterwards.
  if (cudaEventRecord(p->copy_end, p->copy) == cudaSuccess) cudaStreamWaitEvent(s, p->copy_end, 0);
  if (cudaEventRecord(p->done, s) != cudaSuccess && !st) st = set_error(GPTQ_ERR_CUDA, "cudaEventRecord failed");
  return st;
}

gptq_status gptq_pipeline_status(gptq_pipeline* p, int64_t* info, gptq_stream_t stream) {
  clear_error();
  if (!p) return set_error(GPTQ_ERR_INVALID_ARG, "pipeline is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  long long inf = -1;
  gptq_status st = factor_read_status(p->ws_f, &inf, s);
  if (!st) {
    long long qinf = 0;
    st = quantize_read_status(p->ws_q, &qinf, s);
    if (st) inf = qinf;
  }
  if (info) *info = inf;
  return st;
}

gptq_status gptq_pipeline_destroy(gptq_pipeline* p) {
  clear_error();
  if (!p) return GPTQ_OK;
  release(p);
  return GPTQ_OK;
}

}  // extern "C"

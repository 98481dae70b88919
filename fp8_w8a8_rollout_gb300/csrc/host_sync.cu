// host_sync.cu -- weight sync from host memory to host memory.
//
// The trainer's bf16 weights live in host memory; every RL step they are
// quantised to E4M3 with 128x128 block scales and handed to the rollout
// engine ("FP8-RL", "Method steps", step 2).  fp8rl_quant_weight_host_batched
// does the whole transfer in one call: every matrix is cut into chunks of
// whole 128-row block rows (the codes and scale rows of a chunk are exactly
// those of the whole matrix), and each chunk is copied into a staging slot of
// the caller's device buffer, quantised there by the weight quantiser, and its
// codes and scales copied back.  Copy-in, quantise and copy-out run on three
// streams of the library's own, chained by events per slot, so that both
// directions of the host link and the kernels overlap; the call is ordered
// after earlier work on the caller's stream, and later work on that stream
// waits for the last copy out.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace fp8rl {
namespace {

constexpr int kMaxSlots = 8;

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// staging bytes of one chunk of `rows` rows and `k` columns: bf16 in, E4M3
// out and the scale rows, each region 256-byte aligned
size_t chunk_bytes(int64_t rows, int64_t k, size_t scale_bytes) {
  const int64_t rb = (rows + kBlock - 1) / kBlock, kb = (k + kBlock - 1) / kBlock;
  return align256((size_t)rows * k * 2) + align256((size_t)rows * k) + align256((size_t)rb * kb * scale_bytes);
}

// rows x width bytes between pitched buffers: one linear copy when both sides
// are contiguous (a pitched copy of contiguous rows measured about half the
// link rate on GB300), else a pitched copy
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (dpitch == width && spitch == width) return cudaMemcpyAsync(dst, src, width * rows, kind, s);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

// The library's streams and events of one device, made once per context.
struct SyncState {
  uint64_t ctx = 0;
  bool ok = false;
  cudaStream_t s_in = nullptr, s_q = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t ev_in[kMaxSlots] = {}, ev_q[kMaxSlots] = {}, ev_out[kMaxSlots] = {};
};

SyncState g_state[64];
std::mutex g_sync_mu[64];

bool make_state(SyncState& st, uint64_t ctx) {
  st = SyncState{};
  st.ctx = ctx;
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&st.s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&st.s_q, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&st.s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&st.start, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&st.done, ef) == cudaSuccess;
  for (int i = 0; ok && i < kMaxSlots; ++i)
    ok = cudaEventCreateWithFlags(&st.ev_in[i], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&st.ev_q[i], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&st.ev_out[i], ef) == cudaSuccess;
  st.ok = ok;
  if (!ok) cudaGetLastError();
  return ok;
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API size_t fp8rl_host_sync_staging_bytes(int64_t rows, int64_t k, int32_t slots,
                                                          fp8rl_scale_fmt fmt) {
  if (rows < 1 || k < 1 || slots < 2 || slots > kMaxSlots) return 0;
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return 0;
  return (size_t)slots * chunk_bytes(rows, k, fmt == FP8RL_SCALE_FP32 ? 4 : 1);
}

extern "C" FP8RL_API fp8rl_status fp8rl_quant_weight_host_batched(const fp8rl_weight_desc* descs, int32_t count,
                                                                  fp8rl_scale_fmt fmt, void* d_staging,
                                                                  size_t staging_bytes, int32_t slots,
                                                                  void* stream) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  if (count < 0 || (count > 0 && !descs)) return FP8RL_ERR_INVALID_ARG;
  if (slots < 2 || slots > kMaxSlots || !d_staging) return FP8RL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_staging) & 255) return FP8RL_ERR_ALIGNMENT;
  const size_t sb = fmt == FP8RL_SCALE_FP32 ? 4 : 1;
  const size_t slot_bytes = staging_bytes / (size_t)slots / 256 * 256;
  // every matrix must fit at least one 128-row block row (or all its rows) per slot
  for (int32_t i = 0; i < count; ++i) {
    const fp8rl_weight_desc& d = descs[i];
    if (d.n < 0 || d.k < 0 || d.ldw < d.k || d.ldq < d.k) return FP8RL_ERR_INVALID_ARG;
    if (d.n == 0 || d.k == 0) continue;
    if (!d.w_bf16 || !d.q_e4m3 || !d.w_scale) return FP8RL_ERR_INVALID_ARG;
    if (chunk_bytes(std::min<int64_t>(d.n, kBlock), d.k, sb) > slot_bytes) return FP8RL_ERR_SHAPE;
  }
  if (count == 0) return FP8RL_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8RL_ERR_CUDA;
  const uint64_t ctx = current_context_id();
  if (!ctx) return FP8RL_ERR_CUDA;
  // one sync at a time per device: the streams and events are shared
  std::lock_guard<std::mutex> lock(g_sync_mu[dev]);
  SyncState& st = g_state[dev];
  if ((!st.ok || st.ctx != ctx) && !make_state(st, ctx)) return FP8RL_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // after the caller's earlier work, and after the previous sync of this
  // device has left its staging slots (it may have been ordered on another
  // caller stream); an event never recorded is complete
  if (cudaEventRecord(st.start, cs) != cudaSuccess || cudaStreamWaitEvent(st.s_in, st.done, 0) != cudaSuccess ||
      cudaStreamWaitEvent(st.s_in, st.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(st.s_q, st.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(st.s_out, st.start, 0) != cudaSuccess)
    return FP8RL_ERR_CUDA;
  char* staging = static_cast<char*>(d_staging);
  auto enqueue = [&]() -> fp8rl_status {
    int64_t chunk = 0;  // chunks issued so far (slot = chunk mod slots)
    for (int32_t i = 0; i < count; ++i) {
      const fp8rl_weight_desc& d = descs[i];
      if (d.n == 0 || d.k == 0) continue;
      const int64_t kb = (d.k + kBlock - 1) / kBlock;
      // the most whole 128-row block rows that fit one slot
      int64_t rows = std::min<int64_t>(d.n, kBlock);
      while (rows < d.n && chunk_bytes(std::min<int64_t>(d.n, rows + kBlock), d.k, sb) <= slot_bytes)
        rows = std::min<int64_t>(d.n, rows + kBlock);
      for (int64_t r0 = 0; r0 < d.n; r0 += rows, ++chunk) {
        const int64_t r = std::min(rows, d.n - r0);
        const int j = (int)(chunk % slots);
        char* dw = staging + (size_t)j * slot_bytes;
        char* dq = dw + align256((size_t)r * d.k * 2);
        char* ds = dq + align256((size_t)r * d.k);
        const size_t scale_off = (size_t)(r0 / kBlock) * kb * sb;
        const size_t scale_len = (size_t)((r + kBlock - 1) / kBlock) * kb * sb;
        // the slot's previous chunk must have left the device before it is overwritten
        if (chunk >= slots && cudaStreamWaitEvent(st.s_in, st.ev_out[j], 0) != cudaSuccess) return FP8RL_ERR_CUDA;
        if (copy_rows(dw, (size_t)d.k * 2, static_cast<const char*>(d.w_bf16) + (size_t)r0 * d.ldw * 2,
                      (size_t)d.ldw * 2, (size_t)d.k * 2, (size_t)r, cudaMemcpyHostToDevice, st.s_in) != cudaSuccess ||
            cudaEventRecord(st.ev_in[j], st.s_in) != cudaSuccess ||
            cudaStreamWaitEvent(st.s_q, st.ev_in[j], 0) != cudaSuccess)
          return FP8RL_ERR_CUDA;
        const fp8rl_status qs = fp8rl_quant_weight_blockwise(dw, r, d.k, d.k, dq, d.k, ds, fmt, st.s_q);
        if (qs != FP8RL_OK) return qs;
        if (cudaEventRecord(st.ev_q[j], st.s_q) != cudaSuccess ||
            cudaStreamWaitEvent(st.s_out, st.ev_q[j], 0) != cudaSuccess ||
            copy_rows(static_cast<char*>(d.q_e4m3) + (size_t)r0 * d.ldq, (size_t)d.ldq, dq, (size_t)d.k,
                      (size_t)d.k, (size_t)r, cudaMemcpyDeviceToHost, st.s_out) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char*>(d.w_scale) + scale_off, ds, scale_len, cudaMemcpyDeviceToHost,
                            st.s_out) != cudaSuccess ||
            cudaEventRecord(st.ev_out[j], st.s_out) != cudaSuccess)
          return FP8RL_ERR_CUDA;
      }
    }
    return FP8RL_OK;
  };
  fp8rl_status status = enqueue();
  if (status != FP8RL_OK) cudaGetLastError();
  // every copy-in feeds a quantisation that feeds a copy-out: the copy-out
  // stream finishing means the whole sync has.  The caller's stream is joined
  // even when enqueueing stopped early, so that nothing the call did enqueue
  // runs unordered against the caller's later work.
  if (cudaEventRecord(st.done, st.s_out) != cudaSuccess || cudaStreamWaitEvent(cs, st.done, 0) != cudaSuccess)
    return FP8RL_ERR_CUDA;
  return status;
}

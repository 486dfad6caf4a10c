// smla_host.cu — smla_fwd_host: the forward for inputs and outputs that live
// in host memory, with the host<->device copies overlapped with the kernels.
//
// The tokens are processed in chunks.  Three streams run side by side: a
// library-owned copy-in stream (q, indices and valid_len of chunk i + 1), the
// caller's stream (the forward of chunk i, through smla_fwd_ws) and a
// library-owned copy-out stream (O and LSE of chunk i - 1).  The device
// staging buffers are double-buffered in the caller's workspace; events order
// each slot's reuse (a slot's inputs are overwritten only after the forward
// that read them, its outputs only after they were copied out).  The call
// ends with the caller's stream waiting for the last copies, so a
// synchronisation of that stream covers the whole call.
#include <cstdint>
#include <mutex>

#include "../../include/smla.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Per-device copy streams and events, created once with the device current.
struct HostPipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
};
std::mutex g_host_mutex;   // one pipeline per device: calls are serialised
HostPipe g_pipe[kMaxDevices];

smla_status host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return SMLA_ERR_CUDA;
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.ev_start, ef) != cudaSuccess)
      return SMLA_ERR_CUDA;
    for (int s = 0; s < 2; ++s)
      if (cudaEventCreateWithFlags(&hp.ev_in[s], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.ev_comp[s], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.ev_out[s], ef) != cudaSuccess)
        return SMLA_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return SMLA_OK;
}

// Tokens per chunk: the caller's choice, else about a sixteenth of the batch
// (at least 256 tokens, a multiple of 64), so a long batch has enough chunks
// to overlap and each chunk still fills the GPU.  (8192-token prefill on
// GB300: 512-token chunks 8.3 ms a step, 256: 8.9, 1024: 8.9, 2048: 10.1.)
int chunk_of(int T, int chunk_tokens) {
  int c = chunk_tokens > 0 ? chunk_tokens : (T + 15) / 16;
  if (chunk_tokens <= 0) {
    c = (c + 63) / 64 * 64;
    if (c < 256) c = 256;
  }
  return c < T ? c : (T > 0 ? T : 1);
}

// Byte sizes of one slot's staging buffers and of the split workspace.
struct Layout {
  size_t q, idx, vl, out, lse, slot, split, total;
};
// (The split workspace covers both chunk sizes that occur: C and the last,
// shorter chunk, whose plan may split its top-k ranges.)
Layout layout_of(int T, int C, int h, int d_qk, int d_v, int topk, int kv_dtype) {
  Layout L{};
  L.q = round_up((size_t)C * h * d_qk * 2);
  L.idx = round_up((size_t)C * topk * 4);
  L.vl = round_up((size_t)C * 4);
  L.out = round_up((size_t)C * h * d_v * 2);
  L.lse = round_up((size_t)C * h * 4);
  L.slot = L.q + L.idx + L.vl + L.out + L.lse;
  const int last = T - (T - 1) / C * C;
  const size_t w_full = smla_workspace_size(C, h, d_qk, d_v, topk, kv_dtype);
  const size_t w_last = smla_workspace_size(last, h, d_qk, d_v, topk, kv_dtype);
  L.split = round_up(w_full > w_last ? w_full : w_last);
  L.total = 2 * L.slot + L.split;
  return L;
}

}  // namespace

extern "C" {

size_t smla_fwd_host_workspace_size(int T, int h, int d_qk, int d_v, int topk,
                                    int kv_dtype, int chunk_tokens) {
  if (T <= 0 || h < 1 || topk < 1) return 0;
  return layout_of(T, chunk_of(T, chunk_tokens), h, d_qk, d_v, topk, kv_dtype).total;
}

smla_status smla_fwd_host(const void* q_host, const void* kv_cache, int kv_dtype,
                          const float* k_scale, const int32_t* indices_host,
                          const int32_t* valid_len_host, int T, int h, int d_qk,
                          int d_v, int topk, int64_t num_slots, float sm_scale,
                          void* out_host, float* lse_host, int chunk_tokens,
                          void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  if (T < 0 || h < 1 || topk < 1 || num_slots < 1 || chunk_tokens < 0)
    return SMLA_ERR_INVALID_ARG;
  // The shape checks of smla_fwd, before anything is queued.
  int kind = 0, splits = 0;
  size_t split_bytes = 0;
  const int C = chunk_of(T, chunk_tokens);
  smla_status st = smla_plan_info(C, h, d_qk, d_v, topk, kv_dtype, &kind, &splits, &split_bytes);
  if (st != SMLA_OK) return st;
  if (T == 0) return SMLA_OK;
  if (!q_host || !kv_cache || !indices_host || !out_host) return SMLA_ERR_INVALID_ARG;
  if (kv_dtype != SMLA_KV_BF16 && kv_dtype != SMLA_KV_FP8_DS_MLA && !k_scale)
    return SMLA_ERR_INVALID_ARG;
  const Layout L = layout_of(T, C, h, d_qk, d_v, topk, kv_dtype);
  if (!workspace || workspace_bytes < L.total) return SMLA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return SMLA_ERR_INVALID_ARG;

  std::lock_guard<std::mutex> lk(g_host_mutex);
  HostPipe* hp = nullptr;
  if ((st = host_pipe(&hp)) != SMLA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* slot[2] = {ws, ws + L.slot};
  void* split_ws = L.split ? ws + 2 * L.slot : nullptr;
  const uint8_t* qh = static_cast<const uint8_t*>(q_host);
  uint8_t* oh = static_cast<uint8_t*>(out_host);
  const size_t q_row = (size_t)h * d_qk * 2, o_row = (size_t)h * d_v * 2;

  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // On an error after copies were queued, wait for them before returning,
  // so that no queued copy touches the caller's host buffers afterwards.
  auto fail = [&](smla_status code) {
    cudaStreamSynchronize(hp->s_in);
    cudaStreamSynchronize(hp->s_out);
    return code;
  };
  // Nothing of this call starts before the caller's earlier work on `stream`.
  if (!ok(cudaEventRecord(hp->ev_start, stream)) ||
      !ok(cudaStreamWaitEvent(hp->s_in, hp->ev_start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->s_out, hp->ev_start, 0)))
    return SMLA_ERR_CUDA;
  const int n_chunks = (T + C - 1) / C;
  for (int i = 0; i < n_chunks; ++i) {
    const int s = i & 1;
    const int t0 = i * C, n = T - t0 < C ? T - t0 : C;
    uint8_t* q_d = slot[s];
    int32_t* idx_d = reinterpret_cast<int32_t*>(slot[s] + L.q);
    int32_t* vl_d = reinterpret_cast<int32_t*>(slot[s] + L.q + L.idx);
    uint8_t* out_d = slot[s] + L.q + L.idx + L.vl;
    float* lse_d = reinterpret_cast<float*>(slot[s] + L.q + L.idx + L.vl + L.out);
    // copy in (after the forward that last read this slot)
    if (i >= 2 && !ok(cudaStreamWaitEvent(hp->s_in, hp->ev_comp[s], 0)))
      return fail(SMLA_ERR_CUDA);
    if (!ok(cudaMemcpyAsync(q_d, qh + (size_t)t0 * q_row, (size_t)n * q_row,
                            cudaMemcpyHostToDevice, hp->s_in)) ||
        !ok(cudaMemcpyAsync(idx_d, indices_host + (size_t)t0 * topk, (size_t)n * topk * 4,
                            cudaMemcpyHostToDevice, hp->s_in)) ||
        (valid_len_host && !ok(cudaMemcpyAsync(vl_d, valid_len_host + t0, (size_t)n * 4,
                                               cudaMemcpyHostToDevice, hp->s_in))) ||
        !ok(cudaEventRecord(hp->ev_in[s], hp->s_in)))
      return fail(SMLA_ERR_CUDA);
    // forward (after its inputs, and after the copy-out that last read this slot)
    if (!ok(cudaStreamWaitEvent(stream, hp->ev_in[s], 0)) ||
        (i >= 2 && !ok(cudaStreamWaitEvent(stream, hp->ev_out[s], 0))))
      return fail(SMLA_ERR_CUDA);
    st = smla_fwd_ws(q_d, kv_cache, kv_dtype, k_scale, idx_d, valid_len_host ? vl_d : nullptr,
                     n, h, d_qk, d_v, topk, num_slots, sm_scale, out_d,
                     lse_host ? lse_d : nullptr, split_ws, L.split, stream);
    if (st != SMLA_OK) return fail(st);
    if (!ok(cudaEventRecord(hp->ev_comp[s], stream))) return fail(SMLA_ERR_CUDA);
    // copy out
    if (!ok(cudaStreamWaitEvent(hp->s_out, hp->ev_comp[s], 0)) ||
        !ok(cudaMemcpyAsync(oh + (size_t)t0 * o_row, out_d, (size_t)n * o_row,
                            cudaMemcpyDeviceToHost, hp->s_out)) ||
        (lse_host && !ok(cudaMemcpyAsync(lse_host + (size_t)t0 * h, lse_d, (size_t)n * h * 4,
                                         cudaMemcpyDeviceToHost, hp->s_out))) ||
        !ok(cudaEventRecord(hp->ev_out[s], hp->s_out)))
      return fail(SMLA_ERR_CUDA);
  }
  // The caller's stream waits for the last copies out of both slots.
  if (!ok(cudaStreamWaitEvent(stream, hp->ev_out[(n_chunks - 1) & 1], 0)) ||
      (n_chunks > 1 && !ok(cudaStreamWaitEvent(stream, hp->ev_out[n_chunks & 1], 0))))
    return fail(SMLA_ERR_CUDA);
  return SMLA_OK;
}

}  // extern "C"

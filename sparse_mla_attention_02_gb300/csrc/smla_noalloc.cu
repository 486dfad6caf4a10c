// smla_noalloc.cu — smla_fwd_noalloc: the forward for callers that cannot
// allocate device memory.  The split partial results live in a fixed device
// array of this file instead of memory that someone allocates.
//
// The array is a file-scope __device__ object, so the library's module
// carries it: each GPU that loads the library's kernels holds its
// SMLA_NOALLOC_SCRATCH_BYTES until the process exits.  In host code the name
// g_noalloc_scratch is only a host-side stand-in for the symbol; its device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and cached, and only that address is handed to kernels.
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace {

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[SMLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (first call per
// device does the lookup).  Returns nullptr on a CUDA error.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
      return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" SMLA_API smla_status smla_fwd_noalloc(
    const void* q, const void* kv_cache, int kv_dtype, const float* k_scale,
    const int32_t* indices, const int32_t* valid_len, int T, int h, int d_qk,
    int d_v, int topk, int64_t num_slots, float sm_scale, void* out,
    float* lse, cudaStream_t stream) {
  if (T == 0)
    return smla_fwd_ws(q, kv_cache, kv_dtype, k_scale, indices, valid_len, T,
                       h, d_qk, d_v, topk, num_slots, sm_scale, out, lse,
                       nullptr, 0, stream);
  // smla_fwd's own argument checks first, so that a shape or argument that
  // smla_fwd rejects gets the same code here.
  const int chk = smla::check_fwd_args_code(q, kv_cache, kv_dtype, k_scale, indices,
                                            valid_len, T, h, d_qk, d_v, topk, num_slots,
                                            out, lse);
  if (chk != SMLA_OK) return (smla_status)chk;
  void* scratch = scratch_on_current_device();
  if (!scratch) return SMLA_ERR_CUDA;
  // The split plan's need for this shape; larger than the fixed array means
  // this entry point cannot serve the shape (the caller gets a clear code).
  const size_t need =
      smla_workspace_size(T, h, d_qk, d_v, topk, kv_dtype);
  if (need > (size_t)SMLA_NOALLOC_SCRATCH_BYTES) return SMLA_ERR_WORKSPACE;
  // Every partial a call reads is written earlier in the same call, so the
  // previous call's leftovers in the array are never read: nothing to clear.
  return smla_fwd_ws(q, kv_cache, kv_dtype, k_scale, indices, valid_len, T, h,
                     d_qk, d_v, topk, num_slots, sm_scale, out, lse, scratch,
                     (size_t)SMLA_NOALLOC_SCRATCH_BYTES, stream);
}

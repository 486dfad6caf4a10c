// smla_api.cu — the C ABI of libsmla: argument checks, the split plan,
// workspace handling, the device status word, and kernel launches.
//
// Boundary as stated by the pages: FlashMLA's sparse forward takes
// (q, kv, indices, sm_scale, d_v, topk_length) and returns (out, lse)
// (vLLM API docs flashmla_sparse, FlashMLASparseImpl._bf16_flash_mla_kernel);
// FlashInfer's run takes (q_nope, q_pe, ckv, kpe, ckv_scale, kpe_scale)
// (flashinfer_mla_sparse_sm90.py, forward_mqa).  smla_fwd takes the
// concatenated q, the cache, its scales, the slot ids and valid counts.
#include <mutex>
#include <vector>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace {

__device__ int g_smla_status = 0;  // device status word (first error wins)
// Bumped by every bounded wait that gives up; a launch's blocks compare it
// with its value when they started (never reset).
__device__ int g_smla_abort = 0;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int* status = nullptr;      // device address of g_smla_status
  int* abort_ctr = nullptr;   // device address of g_smla_abort
  int stall = 0;              // smla_test_set_stall
  uint64_t wait_limit_ns = 0; // 0: the default limit
  void* workspace = nullptr;  // library-owned workspace for smla_fwd
  size_t workspace_bytes = 0;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, looked up once with that device current.
smla_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return SMLA_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return SMLA_ERR_CUDA;
    void* st = nullptr;
    void* ab = nullptr;
    if (cudaGetSymbolAddress(&st, g_smla_status) != cudaSuccess ||
        cudaGetSymbolAddress(&ab, g_smla_abort) != cudaSuccess)
      return SMLA_ERR_CUDA;
    d.num_sms = sms;
    d.status = static_cast<int*>(st);
    d.abort_ctr = static_cast<int*>(ab);
    d.ready = true;
  }
  *out = &d;
  return SMLA_OK;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

smla_status check_args(const void* q, const void* kv, int kv_dtype,
                       const float* k_scale, const int32_t* indices, int T,
                       int h, int d_qk, int d_v, int topk, int64_t num_slots,
                       const void* out) {
  if (T < 0 || h < 1 || topk < 1 || num_slots < 1) return SMLA_ERR_INVALID_ARG;
  if (h > 128) return SMLA_ERR_UNSUPPORTED;
  if (d_qk != 512 && d_qk != 576) return SMLA_ERR_UNSUPPORTED;
  if (d_v != 512) return SMLA_ERR_UNSUPPORTED;
  if (num_slots > 0x7FFFFFFFLL) return SMLA_ERR_UNSUPPORTED;
  if (kv_dtype < SMLA_KV_BF16 || kv_dtype > SMLA_KV_FP8_E4M3_GROUP4_KPE)
    return SMLA_ERR_UNSUPPORTED;
  if ((kv_dtype == SMLA_KV_FP8_DS_MLA || kv_dtype == SMLA_KV_FP8_E4M3_GROUP4_KPE) &&
      d_qk != 576)
    return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!q || !kv || !indices || !out) return SMLA_ERR_INVALID_ARG;
  if (kv_dtype != SMLA_KV_BF16 && kv_dtype != SMLA_KV_FP8_DS_MLA && !k_scale)
    return SMLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) ||
      !aligned(indices, 4) || (k_scale && !aligned(k_scale, 4)))
    return SMLA_ERR_INVALID_ARG;
  return SMLA_OK;
}

// Request-local index translation (smla_fwd_paged); table == nullptr for
// global slot ids.
struct Paged {
  const int32_t* req_id = nullptr;
  const int32_t* table = nullptr;
  int num_reqs = 0, bt_stride = 0, block_size = 0, stride_rows = 0;
};

smla_status run_fwd(const void* q, const void* kv, int kv_dtype,
                    const float* k_scale, const int32_t* indices,
                    const int32_t* valid_len, int T, int h, int d_qk, int d_v,
                    int topk, int64_t num_slots, float sm_scale, void* out,
                    float* lse, void* ws, size_t ws_bytes, bool own_ws,
                    cudaStream_t stream, const Paged& pg = Paged(),
                    float* out_f32 = nullptr, const void* q_pe = nullptr,
                    float kpe_scale = 1.0f) {
  smla_status st = check_args(q, kv, kv_dtype, k_scale, indices, T, h, d_qk,
                              d_v, topk, num_slots, out);
  if (st != SMLA_OK || T == 0) return st;
  if (d_qk == 512) q_pe = nullptr;             // NoPE: no rope part to read
  if (q_pe && !aligned(q_pe, 16)) return SMLA_ERR_INVALID_ARG;
  if (pg.table) {
    if (!pg.req_id || pg.num_reqs < 1 || pg.bt_stride < 1 || pg.block_size < 1 ||
        pg.stride_rows < 1 || !aligned(pg.req_id, 4) || !aligned(pg.table, 4) ||
        (int64_t)pg.num_reqs * pg.bt_stride > 0x7FFFFFFFLL)
      return SMLA_ERR_INVALID_ARG;
  }
  if ((valid_len && !aligned(valid_len, 4)) || (lse && !aligned(lse, 4)))
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  int stall = 0;
  uint64_t wait_limit_ns = smla::kWaitLimitNs;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    if ((st = device_info(&dev)) != SMLA_OK) return st;
    stall = dev->stall;
    if (dev->wait_limit_ns) wait_limit_ns = dev->wait_limit_ns;
  }
  smla::Plan plan =
      smla::make_plan(T, h, d_qk, d_v, topk, kv_dtype, dev->num_sms);
  if (plan.kind == smla::kKernelNone) return SMLA_ERR_UNSUPPORTED;
  if (out_f32) {
    // Partial-output mode: one range per token, written straight to the
    // caller's fp32 buffers (no workspace, no combine).  A top-k longer than
    // one range of the chosen kernel would need a split: not served.
    if (topk > smla::plan_max_range(plan.kind)) return SMLA_ERR_UNSUPPORTED;
    plan.splits = 1;
    plan.split_len = topk;
    plan.workspace_bytes = 0;
  }
  // The library-owned workspace is one buffer per device.  The lock is held
  // from taking its address until the launches that use it are queued, so a
  // call from another host thread cannot free it in between; a buffer that
  // has to grow is freed only once the device has finished the work queued
  // before (which may still read it).
  std::unique_lock<std::mutex> ws_lock(g_mutex, std::defer_lock);
  if (plan.workspace_bytes > 0) {
    if (own_ws) {
      ws_lock.lock();
      if (dev->workspace_bytes < plan.workspace_bytes) {
        if (dev->workspace) {
          if (cudaDeviceSynchronize() != cudaSuccess) return SMLA_ERR_CUDA;
          cudaFree(dev->workspace);
        }
        dev->workspace = nullptr;
        dev->workspace_bytes = 0;
        if (cudaMalloc(&dev->workspace, plan.workspace_bytes) != cudaSuccess)
          return SMLA_ERR_CUDA;
        dev->workspace_bytes = plan.workspace_bytes;
      }
      ws = dev->workspace;
    } else {
      if (!ws || ws_bytes < plan.workspace_bytes) return SMLA_ERR_WORKSPACE;
      if (!aligned(ws, 256)) return SMLA_ERR_INVALID_ARG;
    }
  }
  smla::FwdParams p{};
  p.q = q;
  p.q_pe = q_pe;
  p.kv = kv;
  p.k_scale = k_scale;
  p.kpe_scale = kpe_scale;
  p.indices = indices;
  p.valid_len = valid_len;
  p.out = out;
  p.lse = lse;
  p.status = dev->status;
  p.abort_ctr = dev->abort_ctr;
  p.wait_limit_ns = wait_limit_ns;
  p.inject_stall = stall;
  p.num_slots = num_slots;
  p.kv_format = kv_dtype;
  p.T = T;
  p.h = h;
  p.d_qk = d_qk;
  p.d_v = d_v;
  p.topk = topk;
  p.num_sms = dev->num_sms;
  p.splits = plan.splits;
  p.split_len = plan.split_len;
  p.sm_scale = sm_scale;
  p.fp32_out = plan.splits > 1 || out_f32 ? 1 : 0;
  p.lpt = plan.lpt;
  p.req_id = pg.req_id;
  p.block_table = pg.table;
  p.num_reqs = pg.num_reqs;
  p.bt_stride = pg.bt_stride;
  p.block_size = pg.block_size;
  p.block_stride_rows = pg.stride_rows;
  if (out_f32) {
    p.o_part = out_f32;
    p.lse_part = lse;
  } else if (plan.splits > 1) {
    p.o_part = static_cast<float*>(ws);
    p.lse_part = p.o_part + (size_t)plan.splits * T * h * d_v;
  }
  const cudaError_t le = plan.kind == smla::kKernelTcFp8    ? smla::launch_tc_fp8(p, stream)
                         : plan.kind == smla::kKernelTcKeys ? smla::launch_tc_keys(p, stream)
                                                            : smla::launch_tc(p, stream);
  if (le != cudaSuccess) return SMLA_ERR_CUDA;
  if (plan.splits > 1) {
    if (smla::launch_combine(p.o_part, p.lse_part, plan.splits, (int64_t)T * h,
                             d_v, out, lse, stream) != cudaSuccess)
      return SMLA_ERR_CUDA;
  }
  return SMLA_OK;
}

}  // namespace

namespace smla {

int check_fwd_args_code(const void* q, const void* kv, int kv_dtype, const float* k_scale,
                        const int32_t* indices, const int32_t* valid_len, int T, int h,
                        int d_qk, int d_v, int topk, int64_t num_slots, const void* out,
                        const float* lse) {
  const smla_status st =
      check_args(q, kv, kv_dtype, k_scale, indices, T, h, d_qk, d_v, topk, num_slots, out);
  if (st != SMLA_OK || T == 0) return st;
  if ((valid_len && !aligned(valid_len, 4)) || (lse && !aligned(lse, 4)))
    return SMLA_ERR_INVALID_ARG;
  return SMLA_OK;
}

int plan_max_range(int kind) {
  return kind == kKernelTcFp8    ? tc_fp8_max_range()
         : kind == kKernelTcKeys ? tc_keys_max_range()
                                 : tc_max_range();
}

// Split plan.  Valid counts are device data, so ranges are cut over topk; a
// range past a token's valid count yields an empty partial (0, -inf) that the
// combine ignores.
//  - kernel family: E4M3 caches with per-(slot, group) scales (every layout)
//    and per-tensor E4M3 with h <= 64 run on the E4M3-operand keys-major
//    kernel (one CTA per token, range and group of 16 heads; FP8 NoPE decode
//    at h = 64: 0.079 ms there, 0.088 ms on the heads-major kernel); bf16 with
//    h <= 16 on the bf16 keys-major kernel (one CTA per unit); bf16 and
//    per-tensor E4M3 with more heads on the heads-major kernel (a 2-SM
//    cluster per unit, up to 128 heads).
//  - tensor-core paths: split only when the units alone leave more than half
//    of the SMs (or SM pairs) idle (each split costs partial-O traffic), or
//    when topk is longer than one unit's range.
Plan make_plan(int T, int h, int d_qk, int d_v, int topk, int kv_format,
               int num_sms) {
  Plan pl{};
  int splits = 1, gran = 64;
  const bool fp8 = tc_fp8_supported(h, d_qk, kv_format) && (kv_format != kE4m3 || h <= 64);
  const bool keys = !fp8 && tc_keys_supported(h, d_qk, kv_format);
  if (!fp8 && !keys && !tc_supported(h, d_qk, kv_format)) {
    pl.kind = kKernelNone;              // (argument checks reject such shapes first)
    return pl;
  }
  {
    pl.kind = fp8 ? kKernelTcFp8 : keys ? kKernelTcKeys : kKernelTc;
    gran = fp8 ? 128 : 64;
    const int max_range = plan_max_range(pl.kind);
    // units per (token, range): head groups of 16 for the E4M3-operand kernel
    const int64_t per_token = fp8 ? (h + 15) / 16 : 1;
    const int places = (fp8 || keys) ? (num_sms > 0 ? num_sms : 1)
                                     : (num_sms > 1 ? num_sms / 2 : 1);
    if (2LL * T * per_token < places) {
      splits = (int)(places / ((T > 0 ? T : 1) * per_token));
      const int max_by_topk = (topk + 127) / 128;
      if (splits > max_by_topk) splits = max_by_topk;
      if (splits > 16) splits = 16;
      if (splits < 1) splits = 1;
    }
    const int need = (topk + max_range - 1) / max_range;
    if (splits < need) splits = need;
  }
  int len = (topk + splits - 1) / splits;
  len = (len + gran - 1) / gran * gran;
  splits = (topk + len - 1) / len;
  pl.splits = splits;
  pl.split_len = len;
  // Longest-first unit order pays only when the units do not all run at
  // once (and costs a pass over the valid counts at each CTA's start).  The
  // keys-major kernel keeps the unit order: its units are short next to a
  // launch on 152 SMs, and neighbouring tokens that select overlapping
  // slots then run together and share L2 (a 2048-token mixed batch read
  // 2.3x the DRAM bytes longest first).
  if (pl.kind == kKernelTc) {
    const int64_t n_units = (int64_t)T * splits;
    const int64_t places = num_sms / 2;
    pl.lpt = (n_units > places && n_units <= 4096) ? 1 : 0;
  }
  pl.workspace_bytes =
      splits > 1 ? sizeof(float) * (size_t)splits * T * h * (d_v + 1) : 0;
  return pl;
}

}  // namespace smla

extern "C" {

smla_status smla_fwd(const void* q, const void* kv_cache, int kv_dtype,
                     const float* k_scale, const int32_t* indices,
                     const int32_t* valid_len, int T, int h, int d_qk, int d_v,
                     int topk, int64_t num_slots, float sm_scale, void* out,
                     float* lse, cudaStream_t stream) {
  return run_fwd(q, kv_cache, kv_dtype, k_scale, indices, valid_len, T, h,
                 d_qk, d_v, topk, num_slots, sm_scale, out, lse, nullptr, 0,
                 true, stream);
}

smla_status smla_fwd_ws(const void* q, const void* kv_cache, int kv_dtype,
                        const float* k_scale, const int32_t* indices,
                        const int32_t* valid_len, int T, int h, int d_qk,
                        int d_v, int topk, int64_t num_slots, float sm_scale,
                        void* out, float* lse, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return run_fwd(q, kv_cache, kv_dtype, k_scale, indices, valid_len, T, h,
                 d_qk, d_v, topk, num_slots, sm_scale, out, lse, workspace,
                 workspace_bytes, false, stream);
}

smla_status smla_cache_write_e4m3_group(const void* kv_c, const void* k_pe,
                                       const int32_t* slot_mapping, int N, int d_qk,
                                       int64_t num_slots, void* kv_cache, float* scales,
                                       cudaStream_t stream) {
  if (N < 0 || num_slots < 1) return SMLA_ERR_INVALID_ARG;
  if (d_qk != 512 && d_qk != 576) return SMLA_ERR_UNSUPPORTED;
  if (N == 0) return SMLA_OK;
  if (!kv_c || !slot_mapping || !kv_cache || !scales || (d_qk == 576) != (k_pe != nullptr))
    return SMLA_ERR_INVALID_ARG;
  if (!aligned(kv_c, 16) || (k_pe && !aligned(k_pe, 16)) || !aligned(kv_cache, 16) ||
      !aligned(scales, 4) || !aligned(slot_mapping, 4))
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    const smla_status st = device_info(&dev);
    if (st != SMLA_OK) return st;
  }
  return smla::launch_cache_write(kv_c, k_pe, slot_mapping, N, d_qk, num_slots, kv_cache,
                                  scales, dev->status, stream) == cudaSuccess
             ? SMLA_OK
             : SMLA_ERR_CUDA;
}

smla_status smla_fwd_partial(const void* q, const void* kv_cache, int kv_dtype,
                             const float* k_scale, const int32_t* indices,
                             const int32_t* valid_len, int T, int h, int d_qk,
                             int d_v, int topk, int64_t num_slots, float sm_scale,
                             float* out_f32, float* lse, cudaStream_t stream) {
  if (T > 0 && (!out_f32 || !lse || !aligned(out_f32, 16) || !aligned(lse, 4)))
    return SMLA_ERR_INVALID_ARG;
  // check_args wants a non-NULL bf16 `out`; the fp32 buffer stands in.
  return run_fwd(q, kv_cache, kv_dtype, k_scale, indices, valid_len, T, h, d_qk,
                 d_v, topk, num_slots, sm_scale, out_f32, lse, nullptr, 0, false,
                 stream, Paged(), out_f32);
}

smla_status smla_fwd_paged(const void* q, const void* kv_cache, int kv_dtype,
                           const float* k_scale, const int32_t* token_indices,
                           const int32_t* req_id_per_token,
                           const int32_t* block_table, int num_reqs,
                           int block_table_stride, int block_size,
                           int block_stride_rows, const int32_t* valid_len,
                           int T, int h, int d_qk, int d_v, int topk,
                           int64_t num_slots, float sm_scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  if (!block_table) return SMLA_ERR_INVALID_ARG;
  Paged pg;
  pg.req_id = req_id_per_token;
  pg.table = block_table;
  pg.num_reqs = num_reqs;
  pg.bt_stride = block_table_stride;
  pg.block_size = block_size;
  pg.stride_rows = block_stride_rows == 0 ? block_size : block_stride_rows;
  return run_fwd(q, kv_cache, kv_dtype, k_scale, token_indices, valid_len, T, h,
                 d_qk, d_v, topk, num_slots, sm_scale, out, lse, workspace,
                 workspace_bytes, workspace == nullptr, stream, pg);
}

smla_status smla_fwd_split_q(const void* q_nope, const void* q_pe, const void* kv_cache,
                             int kv_dtype, const float* k_scale, float kpe_scale,
                             const int32_t* indices, const int32_t* valid_len, int T, int h,
                             int d_qk, int d_v, int topk, int64_t num_slots, float sm_scale,
                             void* out, float* lse, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  return run_fwd(q_nope, kv_cache, kv_dtype, k_scale, indices, valid_len, T, h, d_qk, d_v,
                 topk, num_slots, sm_scale, out, lse, workspace, workspace_bytes,
                 workspace == nullptr, stream, Paged(), nullptr, q_pe, kpe_scale);
}

size_t smla_workspace_size(int T, int h, int d_qk, int d_v, int topk,
                           int kv_dtype) {
  if (T <= 0 || h < 1 || topk < 1) return 0;
  DeviceInfo* dev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (device_info(&dev) != SMLA_OK) return 0;
  }
  return smla::make_plan(T, h, d_qk, d_v, topk, kv_dtype, dev->num_sms)
      .workspace_bytes;
}

smla_status smla_plan_info_for(int T, int h, int d_qk, int d_v, int topk,
                               int kv_dtype, int num_sms, int* kernel, int* splits,
                               size_t* workspace_bytes) {
  if (T < 1 || h < 1 || topk < 1 || num_sms < 1) return SMLA_ERR_INVALID_ARG;
  if (h > 128 || (d_qk != 512 && d_qk != 576) || d_v != 512 ||
      kv_dtype < SMLA_KV_BF16 || kv_dtype > SMLA_KV_FP8_E4M3_GROUP4_KPE ||
      ((kv_dtype == SMLA_KV_FP8_DS_MLA || kv_dtype == SMLA_KV_FP8_E4M3_GROUP4_KPE) &&
       d_qk != 576))
    return SMLA_ERR_UNSUPPORTED;
  const smla::Plan pl = smla::make_plan(T, h, d_qk, d_v, topk, kv_dtype, num_sms);
  if (kernel)
    *kernel = pl.kind == smla::kKernelTcFp8    ? SMLA_KERNEL_TC_KEYS_FP8
              : pl.kind == smla::kKernelTcKeys ? SMLA_KERNEL_TC_KEYS
                                               : SMLA_KERNEL_TC_HEADS;
  if (splits) *splits = pl.splits;
  if (workspace_bytes) *workspace_bytes = pl.workspace_bytes;
  return SMLA_OK;
}

smla_status smla_plan_info(int T, int h, int d_qk, int d_v, int topk,
                           int kv_dtype, int* kernel, int* splits,
                           size_t* workspace_bytes) {
  // Shape errors first, without a device query.
  smla_status st = smla_plan_info_for(T, h, d_qk, d_v, topk, kv_dtype, 1, nullptr,
                                      nullptr, nullptr);
  if (st != SMLA_OK) return st;
  DeviceInfo* dev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    if ((st = device_info(&dev)) != SMLA_OK) return st;
  }
  return smla_plan_info_for(T, h, d_qk, d_v, topk, kv_dtype, dev->num_sms, kernel, splits,
                            workspace_bytes);
}

smla_status smla_combine(const float* o_parts, const float* lse_parts,
                         int n_parts, int64_t rows, int d_v, void* out,
                         float* lse, cudaStream_t stream) {
  if (n_parts < 1 || n_parts > 64 || rows < 0) return SMLA_ERR_INVALID_ARG;
  if (d_v != 512) return SMLA_ERR_UNSUPPORTED;
  if (rows == 0) return SMLA_OK;
  if (!o_parts || !lse_parts || !out) return SMLA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(out, 8) ||
      (lse && !aligned(lse, 4)))
    return SMLA_ERR_INVALID_ARG;
  if (smla::launch_combine(o_parts, lse_parts, n_parts, rows, d_v, out, lse,
                           stream) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_test_set_stall(int stall, int wait_limit_us) {
  if (wait_limit_us < 0) return SMLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceInfo* dev = nullptr;
  const smla_status st = device_info(&dev);
  if (st != SMLA_OK) return st;
  dev->stall = stall ? 1 : 0;
  dev->wait_limit_ns = (uint64_t)wait_limit_us * 1000ull;
  return SMLA_OK;
}

smla_status smla_get_device_status(int* status_out, int clear) {
  if (!status_out) return SMLA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    smla_status st = device_info(&dev);
    if (st != SMLA_OK) return st;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return SMLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return SMLA_ERR_CUDA;
  if (clear && cudaMemset(dev->status, 0, sizeof v) != cudaSuccess)
    return SMLA_ERR_CUDA;
  *status_out = v;
  return SMLA_OK;
}

const char* smla_status_string(int status) {
  switch (status) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA";
    case SMLA_ERR_TIMEOUT: return "SMLA_ERR_TIMEOUT";
    case SMLA_ERR_BAD_INDEX: return "SMLA_ERR_BAD_INDEX";
    case SMLA_ERR_WORKSPACE: return "SMLA_ERR_WORKSPACE";
    default: return "SMLA_ERR_UNKNOWN";
  }
}

int smla_version(void) { return 100; }

}  // extern "C"

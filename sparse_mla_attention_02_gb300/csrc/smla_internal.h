// smla_internal.h — declarations shared by the CUDA translation units of
// libsmla (host API, kernels).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace smla {

// kDsMla: 656-byte rows [512 E4M3 | 4 fp32 group scales | 64 bf16 rope];
// kE4m3Group4Kpe: E4M3 [num_slots, 576] with k_scale [num_slots, 4] for the
// 512 ckv channels and one fp32 kpe_scale for the 64 rope channels.
enum KvFormat { kBf16 = 0, kE4m3 = 1, kE4m3Group = 2, kDsMla = 3, kE4m3Group4Kpe = 4 };
constexpr int kDsMlaRowBytes = 656;
constexpr int kDsMlaScaleOff = 512;   // 4 fp32 scales
constexpr int kDsMlaRopeOff = 528;    // 64 bf16 values

// Bits of the device status word (first condition wins, see smla_api.cu).
enum StatusBits { kStatusTimeout = 4, kStatusBadIndex = 5 };

// Everything a forward launch needs.  Pointers are device pointers.
struct FwdParams {
  const void* q;          // bf16 [T, h, d_qk], or q_nope [T, h, 512] if q_pe
  const void* q_pe;       // bf16 [T, h, d_qk - 512] or nullptr (q concatenated)
  const void* kv;         // [num_slots, d_qk] bf16 or E4M3 bytes, or 656-byte rows
  const float* k_scale;   // per-tensor [1], group [num_slots, G], [num_slots, 4]
  float kpe_scale;        // rope scale of kE4m3Group4Kpe
  const int32_t* indices; // [T, topk]
  const int32_t* valid_len;  // [T] or nullptr
  void* out;              // bf16 [T, h, d_v]
  float* lse;             // [T, h] or nullptr
  float* o_part;          // split partials [splits, T, h, d_v] (splits > 1)
  float* lse_part;        // [splits, T, h]
  int* status;            // device status word
  int* abort_ctr;         // device abort counter (bounded waits, see Waiter)
  uint64_t wait_limit_ns; // time limit of one bounded wait
  int inject_stall;       // tests only: the first QK batch of every unit is
                          // not issued, so the wait for its scores runs out
  int64_t num_slots;
  int kv_format;
  int T, h, d_qk, d_v, topk;
  int num_sms;            // SMs of the device (persistent launches)
  int splits;             // top-k position ranges per (token, head group)
  int split_len;          // positions per range
  int lpt;                // take the units longest first (lpt_unit): more
                          // units than run at once, at most kLptMaxUnits
  int fp32_out;           // write normalised fp32 O and LSE to o_part / lse_part
                          // (split s at s * T * h rows): splits > 1, or
                          // smla_fwd_partial (splits == 1, caller's buffers)
  float sm_scale;
  // Request-local indices (block_table != nullptr): indices hold positions
  // in the token's request; slot = block_table[req, pos / block_size] *
  // block_stride_rows + pos % block_size (see smla_fwd_paged).
  const int32_t* req_id;       // [T]
  const int32_t* block_table;  // [num_reqs, bt_stride]
  int num_reqs, bt_stride, block_size, block_stride_rows;
};

#ifdef __CUDACC__
// Channels [ch, ch + 8) of q[t, hd] (ch a multiple of 8) as one 16-byte load.
__device__ __forceinline__ const uint4* q_chunk(const FwdParams& p, int t, int hd, int ch) {
  const int64_t row = (int64_t)t * p.h + hd;
  const uint16_t* base =
      !p.q_pe    ? static_cast<const uint16_t*>(p.q) + row * p.d_qk + ch
      : ch < 512 ? static_cast<const uint16_t*>(p.q) + row * 512 + ch
                 : static_cast<const uint16_t*>(p.q_pe) + row * (p.d_qk - 512) + (ch - 512);
  return reinterpret_cast<const uint4*>(base);
}

// The global slot for top-k entry value `e` of a token whose request is
// `req` (-1 when the token's request id is out of range): e itself for
// global indices; the block-table translation for request-local ones.
// -1 when masked (e < 0, a page past the table or an unallocated page, or a
// slot >= num_slots); the out-of-range cases set *bad.
__device__ __forceinline__ int to_slot(const FwdParams& p, int req, int e, bool& bad) {
  int64_t id = e;
  if (p.block_table && e >= 0) {
    const int page = e / p.block_size;
    if (req < 0 || page >= p.bt_stride) {
      bad = true;
      return -1;
    }
    const int blk = __ldg(p.block_table + (int64_t)req * p.bt_stride + page);
    if (blk < 0) return -1;
    id = (int64_t)blk * p.block_stride_rows + (e - page * p.block_size);
  }
  if (id >= p.num_slots) {
    bad = true;
    return -1;
  }
  return id < 0 ? -1 : (int)id;
}

// The request of token t for to_slot (0 for global indices; -1 when out of
// range, which masks the token's whole row and sets *bad).
__device__ __forceinline__ int token_req(const FwdParams& p, int t, bool& bad) {
  if (!p.block_table) return 0;
  const int req = __ldg(p.req_id + t);
  if (req < 0 || req >= p.num_reqs) {
    bad = true;
    return -1;
  }
  return req;
}
#endif

// Which kernel family a plan uses.
enum KernelKind { kKernelNone = 0, kKernelTc = 1, kKernelTcKeys = 2, kKernelTcFp8 = 3 };

struct Plan {
  int kind;
  int splits;
  int split_len;
  size_t workspace_bytes;   // partial O and LSE for splits > 1, else 0
  int lpt;                  // longest-first unit order (see FwdParams::lpt)
};

// Largest top-k range one unit of a tensor-core kernel family covers.
int plan_max_range(int kind);

// Default time limit of one bounded wait in the tensor-core kernels.
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

// The host-side argument checks of smla_fwd (codes as smla_status).
int check_fwd_args_code(const void* q, const void* kv, int kv_dtype, const float* k_scale,
                        const int32_t* indices, const int32_t* valid_len, int T, int h,
                        int d_qk, int d_v, int topk, int64_t num_slots, const void* out,
                        const float* lse);

Plan make_plan(int T, int h, int d_qk, int d_v, int topk, int kv_format,
               int num_sms);

bool tc_supported(int h, int d_qk, int kv_format);
int tc_max_range();  // largest top-k range one tensor-core unit covers
cudaError_t launch_tc(const FwdParams& p, cudaStream_t stream);
// Keys-major tensor-core kernel for h <= 16 (all formats, incl. group scales).
bool tc_keys_supported(int h, int d_qk, int kv_format);
int tc_keys_max_range();
cudaError_t launch_tc_keys(const FwdParams& p, cudaStream_t stream);
// Keys-major tensor-core kernel with E4M3 operands (every E4M3 format, any
// h in groups of 16 heads).
bool tc_fp8_supported(int h, int d_qk, int kv_format);
int tc_fp8_max_range();
cudaError_t launch_tc_fp8(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_cache_write(const void* kv_c, const void* k_pe, const int32_t* slot,
                               int N, int d_qk, int64_t num_slots, void* cache,
                               float* scales, int* status, cudaStream_t stream);
cudaError_t launch_combine(const float* o_parts, const float* lse_parts,
                           int n_parts, int64_t rows, int d_v, void* out,
                           float* lse, cudaStream_t stream);

}  // namespace smla

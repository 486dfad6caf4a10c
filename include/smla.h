/*
 * smla.h — C ABI of libsmla: sparse MLA attention forward on GB300 (sm_103a).
 *
 * The operation (vLLM "Sparse MLA on Hopper: Use SGLang's kernel for the
 * sparse mla low latency runs", ops/cutlass_fa3.py, flash_attn_with_kvcache
 * docstring; vLLM API docs flashmla_sparse, FlashMLASparseImpl; and
 * flashinfer_mla_sparse_sm90.py, module docstring): for every query token t
 * and head p, attend only to the token's selected cache slots
 *
 *   J_t = { j < min(valid_len[t], topk) : 0 <= indices[t,j] < num_slots }
 *   s_j = sm_scale * < q[t,p,0:d_qk], K_j >      K_j = dequant(kv[indices[t,j]])
 *   O[t,p,:] = sum_j softmax(s)_j * K_j[0:d_v]   (V is the d_v-prefix of K)
 *   LSE[t,p] = ln sum_j exp(s_j)
 *
 * with one latent KV row shared by all heads (MQA-like).  A token with no
 * selected slot gets O = 0 and LSE = -inf (the LSE-merge identity of the
 * flashmla_sparse page, _forward_fp8_kv_mixed_batch).
 *
 * Conventions shared by every entry point:
 *  - Pointers named as device pointers must be device memory of the current
 *    device (or managed memory); host pointers are named as such.
 *  - All buffers are owned by the caller.  The library keeps no pointer past
 *    a call, except its own lazily grown workspace (smla_fwd only).
 *  - Work is enqueued on `stream` and returns without synchronising, unless
 *    a function says otherwise.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns SMLA_ERR_INVALID_ARG or SMLA_ERR_UNSUPPORTED and
 *    launches nothing.  T = 0 returns SMLA_OK and launches nothing.
 *  - Device-side conditions (an index >= num_slots, a bounded wait that ran
 *    out) never fault: the element is masked or the block exits, and a bit is
 *    set in a device status word that smla_get_device_status reads.
 *  - Accuracy: O is bf16, LSE fp32.  Against the formula above evaluated in
 *    fp64 on the same (dequantized) inputs, |dO| <= 2e-2 while |O| < 8 (the
 *    bf16 rounding of O alone takes up to 2^-8 |O| there) and
 *    |dLSE| <= 1e-3.  The softmax weights reach the PV product rounded to
 *    bf16 (bf16 caches, O divided by the sum of the rounded weights) or as
 *    three E4M3 terms that keep them to their f16 rounding (E4M3 caches), so
 *    a row that one key carries keeps that key's V row to within the output's
 *    own rounding.
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SMLA_API __attribute__((visibility("default")))
#else
#define SMLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* KV cache element formats.
 *  SMLA_KV_BF16: bf16 rows of d_qk elements (cutlass_fa3_sparse.py,
 *    get_kv_cache_shape: 576 bf16 = [kv_c_normed 512 | k_pe 64]).
 *  SMLA_KV_FP8_E4M3: E4M3 bytes, value = e4m3 * k_scale[0]
 *    (flashinfer_mla_sparse_sm90.py: per-tensor k_scale, FP8 read directly).
 *  SMLA_KV_FP8_E4M3_GROUP128: E4M3 bytes, value = e4m3 * k_scale[slot*G + c/128],
 *    G = ceil(d_qk/128) (the per-token x 128-channel-group ckv_scale_arr).
 *  SMLA_KV_FP8_DS_MLA: d_qk = 576 only; 656-byte rows (the fp8_ds_mla cache
 *    of vLLM "Sparse MLA on Hopper", cutlass_fa3_sparse.py module docstring:
 *    656 bytes per token), read as bytes [0, 512) E4M3 ckv codes, [512, 528)
 *    four little-endian fp32 scales (one per 128-channel group), [528, 656)
 *    the 64 rope values as little-endian bf16; value = e4m3 * scale[c/128]
 *    for c < 512, the bf16 rope value for c >= 512.  k_scale is unused.
 *  SMLA_KV_FP8_E4M3_GROUP4_KPE: d_qk = 576 only; E4M3 bytes [num_slots, 576],
 *    value = e4m3 * k_scale[slot*4 + c/128] for c < 512 and e4m3 * kpe_scale
 *    for the 64 rope channels (the ckv_scale / kpe_scale split of
 *    flashinfer_mla_sparse_sm90.py, forward_mqa).  Entry points without a
 *    kpe_scale argument use 1.0, the value that page passes. */
typedef enum {
  SMLA_KV_BF16 = 0,
  SMLA_KV_FP8_E4M3 = 1,
  SMLA_KV_FP8_E4M3_GROUP128 = 2,
  SMLA_KV_FP8_DS_MLA = 3,
  SMLA_KV_FP8_E4M3_GROUP4_KPE = 4
} smla_kv_dtype;

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, misaligned buffer */
  SMLA_ERR_UNSUPPORTED = 2,  /* a shape or format the library does not serve */
  SMLA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  SMLA_ERR_TIMEOUT = 4,      /* device status: a bounded wait ran out */
  SMLA_ERR_BAD_INDEX = 5,    /* device status: an index >= num_slots was masked */
  SMLA_ERR_WORKSPACE = 6     /* the caller's workspace is smaller than needed */
} smla_status;

/*
 * smla_fwd — the sparse MLA forward (the whole hot path: work setup, index
 * gather, FP8 dequant, QK^T, masked online softmax, PV, epilogue, and the
 * LSE-weighted combine when the top-k range is split across CTAs).
 *
 *  q          device, bf16 [T, h, d_qk] contiguous; d_qk = 576 ([nope 512 |
 *             rope 64]) or 512 (NoPE).  16-byte aligned.
 *  kv_cache   device, [num_slots, d_qk] contiguous rows: bf16 (2*d_qk bytes a
 *             row) or E4M3 bytes (d_qk bytes a row); SMLA_KV_FP8_DS_MLA:
 *             656-byte rows.  16-byte aligned.
 *  kv_dtype   an smla_kv_dtype value.
 *  k_scale    device fp32: NULL for SMLA_KV_BF16 and SMLA_KV_FP8_DS_MLA; [1]
 *             for SMLA_KV_FP8_E4M3; [num_slots, ceil(d_qk/128)] for
 *             SMLA_KV_FP8_E4M3_GROUP128; [num_slots, 4] for
 *             SMLA_KV_FP8_E4M3_GROUP4_KPE.
 *  indices    device int32 [T, topk]: global slot ids; entries < 0 or
 *             >= num_slots are masked wherever they sit (the -1 tail, or
 *             scattered -1 as the flashmla_sparse page's DCP path leaves them).
 *  valid_len  device int32 [T] (clamped to [0, topk]), or NULL: then every
 *             entry of the row is considered and masked entries skipped.
 *  T, h       query tokens (>= 0) and heads (1..128).
 *  d_v        must be 512.
 *  topk       index row width (>= 1).
 *  num_slots  rows in kv_cache (>= 1, < 2^31).
 *  sm_scale   multiplies the raw dot product (e.g. 1/sqrt(576)).
 *  out        device, bf16 [T, h, d_v], written in full.  16-byte aligned.
 *  lse        device fp32 [T, h] natural-log LSE, or NULL to skip it.
 *  stream     CUDA stream (0 = legacy default stream).
 *
 * Uses a library-owned device workspace for split partial results, grown
 * with cudaMalloc on first need (so the first call of a new, larger shape
 * allocates, after waiting for the device to finish the work queued before);
 * smla_fwd_ws takes a caller-owned workspace instead.  There is one such
 * workspace per device: two calls that split their top-k ranges and may run
 * at the same time on the GPU (different streams) race on it.  Keep such
 * calls on one stream, or use smla_fwd_ws with one workspace per stream.
 * Several host threads may call at once; calls that use this workspace are
 * queued one at a time.
 */
SMLA_API smla_status smla_fwd(const void* q, const void* kv_cache, int kv_dtype,
                     const float* k_scale, const int32_t* indices,
                     const int32_t* valid_len, int T, int h, int d_qk, int d_v,
                     int topk, int64_t num_slots, float sm_scale, void* out,
                     float* lse, cudaStream_t stream);

/*
 * smla_workspace_size — bytes of device workspace smla_fwd_ws needs for this
 * shape on the current device (0 when the plan does not split the top-k
 * range).  Deterministic for a given (shape, device SM count).
 */
SMLA_API size_t smla_workspace_size(int T, int h, int d_qk, int d_v, int topk,
                           int kv_dtype);

/* Kernel families a plan can choose (see smla_plan_info). */
typedef enum {
  SMLA_KERNEL_CUDA_CORE = 0,     /* (not chosen by any plan: every supported shape has a
                                    tensor-core kernel; the value stays reserved) */
  SMLA_KERNEL_TC_HEADS = 1,      /* tcgen05, heads as the MMA rows (h <= 128) */
  SMLA_KERNEL_TC_KEYS = 2,       /* tcgen05, top-k positions as the MMA rows (bf16, h <= 16) */
  SMLA_KERNEL_TC_KEYS_FP8 = 3    /* tcgen05 with E4M3 operands, top-k positions as the MMA
                                    rows, heads in groups of 16 (E4M3 caches: every layout
                                    with group scales, any h; one scale per tensor, h <= 16) */
} smla_kernel;

/*
 * smla_plan_info — how smla_fwd would run this shape on the current device:
 * the kernel family (*kernel, an smla_kernel), the number of top-k ranges
 * per token (*splits; > 1 means partial results merged by smla_combine's
 * kernel) and the workspace that needs (*workspace_bytes).  Any output
 * pointer may be NULL.  Host-only: launches nothing.  An inspection aid with
 * no counterpart in the pages.  Errors: SMLA_ERR_INVALID_ARG /
 * SMLA_ERR_UNSUPPORTED for shapes smla_fwd rejects, SMLA_ERR_CUDA when the
 * device cannot be queried.
 */
SMLA_API smla_status smla_plan_info(int T, int h, int d_qk, int d_v, int topk,
                                    int kv_dtype, int* kernel, int* splits,
                                    size_t* workspace_bytes);

/*
 * smla_plan_info_for — the same plan for a device with num_sms SMs, without
 * querying any device: the kernel family, splits and workspace smla_fwd
 * would choose there (for sizing workspaces ahead of time, on a host with
 * or without a GPU).  smla_plan_info is this call with the current
 * device's SM count.  Errors: those of smla_plan_info's shape checks, and
 * SMLA_ERR_INVALID_ARG when num_sms < 1; never SMLA_ERR_CUDA.
 */
SMLA_API smla_status smla_plan_info_for(int T, int h, int d_qk, int d_v, int topk,
                                        int kv_dtype, int num_sms, int* kernel,
                                        int* splits, size_t* workspace_bytes);

/*
 * smla_fwd_ws — smla_fwd with a caller-owned device workspace of at least
 * smla_workspace_size(...) bytes (256-byte aligned; NULL allowed when that
 * size is 0).  Returns SMLA_ERR_WORKSPACE if it is too small.  Performs no
 * allocation and no host synchronisation.  One workspace must not be shared by
 * calls that may overlap on the GPU.
 */
SMLA_API smla_status smla_fwd_ws(const void* q, const void* kv_cache, int kv_dtype,
                        const float* k_scale, const int32_t* indices,
                        const int32_t* valid_len, int T, int h, int d_qk,
                        int d_v, int topk, int64_t num_slots, float sm_scale,
                        void* out, float* lse, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/*
 * smla_cache_write_e4m3_group — write token rows into an E4M3 cache with one
 * fp32 scale per (slot, 128-channel group), the layout smla_fwd reads for
 * SMLA_KV_FP8_E4M3_GROUP128.  The flashinfer_mla_sparse_sm90.py page reads
 * that layout (ckv_scale_arr) but notes the cache-write op producing it is
 * missing; vLLM's concat_and_cache_mla (same pages) is the write for the
 * other formats: row [kv_c | k_pe] at the token's slot.  For each written
 * row and group g (channels [128 g, 128 g + 128)):
 *   scale = amax|x| / 448 in fp32 (1 for an all-zero group)
 *   code  = e4m3(x / scale), fp32 division, round to nearest even,
 *           saturating at +-448
 *  kv_c          device bf16 [N, 512], 16-byte aligned
 *  k_pe          device bf16 [N, 64] for d_qk = 576, NULL for d_qk = 512
 *  slot_mapping  device int32 [N]: the cache row of each token; < 0 = skip;
 *                >= num_slots = skip and set SMLA_ERR_BAD_INDEX (device status)
 *  kv_cache      device uint8 [num_slots, d_qk], 16-byte aligned
 *  scales        device fp32 [num_slots, ceil(d_qk / 128)]
 * Rows not written keep their bytes and scales.  Asynchronous on `stream`,
 * no allocation.  Errors: SMLA_ERR_INVALID_ARG (N < 0, num_slots < 1, NULL
 * or misaligned pointers, k_pe given for d_qk = 512 or missing for 576),
 * SMLA_ERR_UNSUPPORTED (d_qk not 512 or 576), SMLA_ERR_CUDA.  N = 0 is OK.
 */
SMLA_API smla_status smla_cache_write_e4m3_group(const void* kv_c, const void* k_pe,
                                                 const int32_t* slot_mapping, int N,
                                                 int d_qk, int64_t num_slots,
                                                 void* kv_cache, float* scales,
                                                 cudaStream_t stream);

/*
 * smla_fwd_partial — smla_fwd that writes the normalised output in fp32 and
 * its LSE, for a later LSE-weighted merge of partial results over disjoint
 * key sets (the DCP path of the vLLM API docs' flashmla_sparse page: each
 * rank attends to its shard of the top-k set, rows with no key give
 * (O = 0, LSE = -inf), and the shards are merged by LSE weights; merge them
 * with smla_combine).  Entries < 0 may sit anywhere in a row (no compaction
 * needed), exactly as for smla_fwd.
 *  out_f32  device fp32 [T, h, d_v], 16-byte aligned, written in full.
 *  lse      device fp32 [T, h], required.
 * Every other argument is that of smla_fwd.  One top-k range per token, so
 * no workspace and no allocation; SMLA_ERR_UNSUPPORTED when topk is longer
 * than one range of the tensor-core kernel the shape uses (2048 positions
 * for h <= 16, 3072 otherwise).  SMLA_ERR_INVALID_ARG when out_f32 or lse
 * is NULL or misaligned (T > 0).
 */
SMLA_API smla_status smla_fwd_partial(const void* q, const void* kv_cache, int kv_dtype,
                             const float* k_scale, const int32_t* indices,
                             const int32_t* valid_len, int T, int h, int d_qk,
                             int d_v, int topk, int64_t num_slots, float sm_scale,
                             float* out_f32, float* lse, cudaStream_t stream);

/*
 * smla_fwd_paged — smla_fwd for request-local top-k indices, translated to
 * cache slots inside the kernels' index loads (the fused form of the index
 * conversion the serving backends run as a separate kernel before the
 * attention call: vLLM "Sparse MLA on Hopper" diff, the kernel test file's
 * index-conversion tests (2.5, 2.9), which fix
 *   slot = block_table[req, e / block_size] * block_size + e % block_size
 * with -1 entries propagated).
 *  token_indices      device int32 [T, topk]: positions in the token's
 *                     request (its KV sequence); entries < 0 are masked.
 *  req_id_per_token   device int32 [T]: the token's request, in [0, num_reqs);
 *                     a token outside that range has every entry masked and
 *                     sets the SMLA_ERR_BAD_INDEX device status.
 *  block_table        device int32 [num_reqs, block_table_stride]: the cache
 *                     block of each block_size positions of a request; a
 *                     negative entry is an unallocated block (its positions
 *                     are masked).  A position whose block index is
 *                     >= block_table_stride, or whose slot is >= num_slots,
 *                     is masked and sets SMLA_ERR_BAD_INDEX.
 *  block_size         positions per block (>= 1).
 *  block_stride_rows  cache rows between consecutive blocks: slot =
 *                     block * block_stride_rows + e % block_size; 0 means
 *                     block_size (the pages' BLOCK_STRIDE_ROWS option).
 *  workspace          caller-owned workspace as for smla_fwd_ws, or NULL to
 *                     use the library-owned one as smla_fwd does.
 * Every other argument, the result and the errors are those of smla_fwd:
 * the call computes exactly what smla_fwd computes on the translated slot
 * ids (the same kernels read the same rows).  Host checks add:
 * SMLA_ERR_INVALID_ARG when block_table or req_id_per_token is NULL or
 * unaligned, or num_reqs, block_table_stride or block_size < 1.
 */
SMLA_API smla_status smla_fwd_paged(const void* q, const void* kv_cache, int kv_dtype,
                           const float* k_scale, const int32_t* token_indices,
                           const int32_t* req_id_per_token,
                           const int32_t* block_table, int num_reqs,
                           int block_table_stride, int block_size,
                           int block_stride_rows, const int32_t* valid_len,
                           int T, int h, int d_qk, int d_v, int topk,
                           int64_t num_slots, float sm_scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * smla_fwd_host_workspace_size — bytes of device workspace smla_fwd_host
 * needs for T tokens in chunks of chunk_tokens (0 = the default chunking):
 * two slots of staging buffers for a chunk's q, indices, valid_len, O and
 * LSE, plus the split workspace smla_fwd_ws needs for a chunk.  0 when
 * T <= 0.
 */
SMLA_API size_t smla_fwd_host_workspace_size(int T, int h, int d_qk, int d_v,
                                             int topk, int kv_dtype,
                                             int chunk_tokens);

/*
 * smla_fwd_host — smla_fwd for a caller whose per-step tensors live in host
 * memory: q, indices, valid_len are read from the host and O, LSE written to
 * the host, with the copies overlapped with the forward.  The pages have no
 * counterpart (their serving stacks keep these tensors on the device); it is
 * the host-memory boundary of the same computation.
 *
 * The T tokens are processed in chunks of chunk_tokens (0: about T / 16, at
 * least 256 and a multiple of 64).  While the forward of chunk i runs on
 * `stream`, a library-owned stream copies chunk i + 1 in and another copies
 * chunk i - 1 out; device staging is double-buffered in `workspace`.  Each
 * chunk runs smla_fwd_ws on its tokens, so its rows are exactly what
 * smla_fwd computes for that chunk; the split plan follows the chunk's
 * size, so where a chunk splits its top-k ranges and one call on all T
 * tokens would not (or the other way round), the rounding of those rows
 * differs within the usual bounds.
 *  q_host          bf16 [T, h, d_qk], host memory
 *  kv_cache        device, as for smla_fwd (model state stays resident)
 *  k_scale         device, as for smla_fwd
 *  indices_host    int32 [T, topk], host memory
 *  valid_len_host  int32 [T] host memory, or NULL as for smla_fwd
 *  out_host        bf16 [T, h, d_v], host memory, written
 *  lse_host        fp32 [T, h] host memory, or NULL
 *  chunk_tokens    tokens per chunk, >= 0 (0 = default)
 *  workspace       device, >= smla_fwd_host_workspace_size(...) bytes,
 *                  256-byte aligned, caller-owned
 * Host buffers should be page-locked (cudaHostAlloc / pinned): pageable
 * memory is still correct but its copies do not overlap.
 * Asynchronous on `stream`: the host buffers may be read or written until
 * `stream` has been synchronised (the call ends with `stream` waiting for
 * the last copies).  No allocation after the first call on a device, which
 * creates the two copy streams and their events.  Calls are serialised
 * inside the library (one copy pipeline per device); one workspace must not
 * be shared by calls that may overlap on the GPU.
 * Errors: those of smla_fwd for the shape and arguments (checked before
 * anything is queued), SMLA_ERR_INVALID_ARG for NULL host buffers or a
 * negative chunk_tokens, SMLA_ERR_WORKSPACE when the workspace is missing or
 * too small, SMLA_ERR_CUDA.  An error after copies were queued returns only
 * once those copies have finished (a host synchronisation of the copy
 * streams), so the host buffers are free to release.
 */
SMLA_API smla_status smla_fwd_host(const void* q_host, const void* kv_cache,
                                   int kv_dtype, const float* k_scale,
                                   const int32_t* indices_host,
                                   const int32_t* valid_len_host, int T, int h,
                                   int d_qk, int d_v, int topk, int64_t num_slots,
                                   float sm_scale, void* out_host, float* lse_host,
                                   int chunk_tokens, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/*
 * smla_combine — LSE-weighted merge of partial results computed over disjoint
 * key sets (the split-KV combine, and the cross-rank merge of the
 * flashmla_sparse page's DCP path):
 *   LSE = ln sum_p exp(LSE_p)  (-inf parts contribute nothing)
 *   O   = sum_p exp(LSE_p - LSE) * O_p,   all parts -inf -> (0, -inf)
 *  o_parts    device fp32 [n_parts, rows, d_v], each part normalised over its keys
 *  lse_parts  device fp32 [n_parts, rows]
 *  out        device bf16 [rows, d_v];  lse  device fp32 [rows] or NULL
 *  d_v        must be 512; n_parts 1..64; rows >= 0.
 */
SMLA_API smla_status smla_combine(const float* o_parts, const float* lse_parts,
                         int n_parts, int64_t rows, int d_v, void* out,
                         float* lse, cudaStream_t stream);

/* Bytes of the fixed device scratch behind smla_fwd_noalloc (16 MiB). */
#define SMLA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * smla_fwd_noalloc — the same forward as smla_fwd, for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for how the library is hosted, not for the method.
 *
 * Who needs it: code that runs inside a host which owns every byte of device
 * memory through its own pool (an inference engine's plugin, a framework
 * that forbids cudaMalloc outside its allocator so its accounting stays
 * exact), and latency-critical loops where a cudaMalloc, which may stall
 * until the device is idle, is not acceptable.  Such a caller passes its
 * inputs and outputs exactly as for smla_fwd and nothing else.
 *
 * Scratch: the split partial results go to a device array of
 * SMLA_NOALLOC_SCRATCH_BYTES that is part of the library itself; every GPU
 * on which the library is loaded holds it until the process exits.  This
 * function calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and keeps it; make that first call before any
 *    stream capture.
 *  - A shape whose split plan needs more than SMLA_NOALLOC_SCRATCH_BYTES
 *    (smla_workspace_size tells in advance) returns SMLA_ERR_WORKSPACE and
 *    launches nothing.
 *  - All calls share the one array, and it keeps whatever the last call
 *    left.  Nothing in it has to start at zero: each call writes every
 *    partial it later reads.  But two calls that may run at the same time on
 *    the GPU (different streams, or different host threads) race on the array
 *    and corrupt each other's results: keep such calls on one stream, or use
 *    smla_fwd_ws with one workspace per stream.
 * Arguments, layouts and the other error codes are those of smla_fwd.
 */
SMLA_API smla_status smla_fwd_noalloc(const void* q, const void* kv_cache,
                                      int kv_dtype, const float* k_scale,
                                      const int32_t* indices,
                                      const int32_t* valid_len, int T, int h,
                                      int d_qk, int d_v, int topk,
                                      int64_t num_slots, float sm_scale,
                                      void* out, float* lse,
                                      cudaStream_t stream);

/*
 * smla_get_device_status — read (and optionally clear) the current device's
 * status word: 0, or the SMLA_ERR_TIMEOUT / SMLA_ERR_BAD_INDEX condition
 * seen first since the last clear.  Synchronises the device; meant for tests
 * and diagnostics, not the hot path.
 */
SMLA_API smla_status smla_get_device_status(int* status_out, int clear);

/*
 * smla_test_set_stall — for tests of the timeout path only (no counterpart on
 * the pages).  Every wait inside the tensor-core kernels is bounded: a wait
 * that runs out sets SMLA_ERR_TIMEOUT in the device status word, the block
 * drains the copies and MMAs it started, frees its tensor memory and
 * returns, and the launch's outputs are undefined.  This switch lets a test
 * reach that path without a fault or a hang.
 *
 *  stall          nonzero: later tensor-core launches on the current device
 *                 leave out the first batch of score MMAs of every work
 *                 unit, so the wait for those scores cannot complete and
 *                 runs out; 0: normal launches.
 *  wait_limit_us  the time limit of one bounded wait in later launches on
 *                 the current device, in microseconds; 0 = the default
 *                 (500 ms).
 * The setting is process-wide per device and applies to launches made after
 * the call; it does not touch the status word (smla_get_device_status clears
 * it).  A timeout of one launch does not abort later launches.  Returns
 * SMLA_ERR_INVALID_ARG for wait_limit_us < 0, SMLA_ERR_CUDA when the device
 * cannot be queried.
 */
SMLA_API smla_status smla_test_set_stall(int stall, int wait_limit_us);

/* smla_status_string — a static, human-readable name for a status code. */
SMLA_API const char* smla_status_string(int status);

/* smla_version — library version as major*10000 + minor*100 + patch. */
SMLA_API int smla_version(void);

/*
 * smla_fwd_split_q — smla_fwd with the query in two tensors and an explicit
 * rope scale, as FlashInfer's run(q_nope, q_pe, ckv, kpe, ckv_scale,
 * kpe_scale) and the FA3 sparse backend take them (flashinfer_mla_sparse_sm90.py,
 * forward_mqa; vLLM "Sparse MLA on Hopper", cutlass_fa3_sparse.py module
 * docstring: the two query parts go in separately, without a concatenation
 * kernel).  The kernels read q_nope and q_pe where they sit.
 *
 *  q_nope     device, bf16 [T, h, 512] contiguous, 16-byte aligned; or, with
 *             q_pe NULL, the concatenated q [T, h, d_qk] of smla_fwd.
 *  q_pe       device, bf16 [T, h, d_qk - 512] contiguous, 16-byte aligned, or
 *             NULL.  Ignored when d_qk = 512 (NoPE; the pages hand a
 *             zero-width rope tensor through).
 *  kpe_scale  the rope channels' scale for SMLA_KV_FP8_E4M3_GROUP4_KPE;
 *             ignored by the other formats.
 *  workspace, workspace_bytes  as smla_fwd_ws; workspace NULL = the
 *             library-owned workspace of smla_fwd.
 *  Every other argument, the results and the errors are those of smla_fwd.
 */
SMLA_API smla_status smla_fwd_split_q(const void* q_nope, const void* q_pe,
                                      const void* kv_cache, int kv_dtype,
                                      const float* k_scale, float kpe_scale,
                                      const int32_t* indices, const int32_t* valid_len,
                                      int T, int h, int d_qk, int d_v, int topk,
                                      int64_t num_slots, float sm_scale, void* out,
                                      float* lse, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H_ */

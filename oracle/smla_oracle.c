/*
 * smla_oracle.c — fp64 CPU oracle for the sparse MLA attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or helper with the CUDA library under
 * sparse_mla_attention_02_gb300/csrc, and neither side includes the other.
 *
 * What it computes (one query token t, one head p), written out exactly as the
 * method defines it, with no blocking, fusion or reordering:
 *
 *   J   = { j < min(valid_len[t], topk) : 0 <= indices[t,j] < num_slots }
 *         (valid_len NULL: every entry of the row that is a real slot id)
 *   K_j = dequant(kv[indices[t,j], 0:d_qk])          V_j = K_j[0:d_v]
 *   s_j = sm_scale * sum_c q[t,p,c] * K_j[c]
 *   LSE = M + ln(sum_j exp(s_j - M)),  M = max_j s_j
 *   O   = sum_j exp(s_j - LSE) * V_j
 *   J empty  ->  O = 0, LSE = -inf
 *
 * Sources (page title, section):
 *  - vLLM "Sparse MLA on Hopper: Use SGLang's kernel for the sparse mla low
 *    latency runs", ops/cutlass_fa3.py, flash_attn_with_kvcache docstring:
 *    score = q_rope.k_rope + q_nope.c_kv, output = softmax(score*scale) @ c_kv.
 *  - same diff, cutlass_fa3_sparse.py, get_kv_cache_shape: the cache row is
 *    576 bf16 elements = [kv_c_normed(512) | k_pe(64)]; V is the 512 prefix.
 *  - same diff, tests/kernels test file: the reference gathers the selected
 *    rows and runs scaled_dot_product_attention per token (non-causal).
 *  - vLLM API docs flashmla_sparse, FlashMLASparseImpl._forward_fp8_kv_mixed_batch:
 *    a row whose selected entries are all -1 yields (O = 0, LSE = -inf), the
 *    identity of the cross-rank LSE merge; the LSE is reported per (token, head).
 *  - flashinfer_mla_sparse_sm90.py, module docstring: FP8 E4M3 cache read
 *    directly, per-tensor k_scale, per-token x 128-channel-group scales
 *    (ckv_scale_arr); the valid entries form a compacted prefix with -1 past it
 *    (forward_mqa comment on return_valid_counts).
 *  - same page, forward_mqa: the FP8 cache is handed to the kernel as ckv =
 *    row[:512] and kpe = row[512:] with ckv_scale = k_scale and a separate
 *    kpe_scale (format 4 below: four ckv group scales per slot and one
 *    per-tensor kpe scale).
 *  - same diff, cutlass_fa3_sparse.py module docstring: the FlashMLA FP8
 *    cache (fp8_ds_mla) takes 656 bytes per token (format 3 below).
 *
 * Readings where the pages are silent (listed with the others in the design
 * notes): natural-log LSE; a -1 (or out-of-range id) inside the valid prefix is
 * masked; valid_len > topk is clamped; duplicates each count once; E4M3 is the
 * "fn" variant (no Inf, S.1111.111 = NaN), as torch.float8_e4m3fn; the group
 * scale of channel c is k_scale[idx * ceil(d_qk/128) + c/128].  The 656-byte
 * fp8_ds_mla row (its layout is not printed on the pages) is read as
 * [512 E4M3 bytes | 4 fp32 scales, one per 128-channel group, little-endian |
 * 64 bf16 rope values, little-endian]: 512 + 16 + 128 = 656.
 *
 * Precision: every input value is exactly representable in fp64, so the only
 * rounding is fp64 arithmetic.  Threads (POSIX) split the token list; each
 * (token, head) result is computed by one thread in a fixed order, so results
 * do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  ORACLE_KV_BF16 = 0,
  ORACLE_KV_E4M3 = 1,
  ORACLE_KV_E4M3_GROUP128 = 2,
  ORACLE_KV_FP8_DS_MLA = 3,      /* 656-byte rows, scales and rope inside the row */
  ORACLE_KV_E4M3_GROUP4_KPE = 4  /* E4M3 [S, 576]; scales [S, 4] for ckv, one kpe scale */
};
enum { ORACLE_DS_MLA_ROW = 656 };

/* bf16 -> fp64: a bf16 value is the upper half of an IEEE binary32. */
double smla_oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 ("fn": finite only) -> fp64 from the format's definition:
 * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
 * subnormal (2^-6 * m/8); S.1111.111 is NaN; there is no infinity. */
double smla_oracle_e4m3_to_f64(uint8_t byte) {
  int s = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

typedef struct {
  const uint16_t* q;
  const void* kv;
  int kv_dtype;
  const float* k_scale;
  double kpe_scale;
  const int32_t* indices;
  const int32_t* valid_len;
  int64_t T;
  int h, d_qk, d_v, topk;
  int64_t num_slots;
  double sm_scale;
  const int64_t* tokens;
  int64_t n_tokens;
  double* out;
  double* lse;
  int64_t next; /* next position in the token list (work queue) */
  pthread_mutex_t lock;
  int status;
} oracle_job;

/* Dequantized element c of cache row `slot`. */
static double kv_value(const oracle_job* jb, int64_t slot, int c) {
  if (jb->kv_dtype == ORACLE_KV_BF16) {
    const uint16_t* row = (const uint16_t*)jb->kv + slot * (int64_t)jb->d_qk;
    return smla_oracle_bf16_to_f64(row[c]);
  } else if (jb->kv_dtype == ORACLE_KV_FP8_DS_MLA) {
    const uint8_t* row = (const uint8_t*)jb->kv + slot * (int64_t)ORACLE_DS_MLA_ROW;
    if (c < 512) {
      float sc;
      memcpy(&sc, row + 512 + 4 * (c / 128), sizeof sc);
      return smla_oracle_e4m3_to_f64(row[c]) * (double)sc;
    }
    uint16_t b = (uint16_t)(row[528 + 2 * (c - 512)] | (row[529 + 2 * (c - 512)] << 8));
    return smla_oracle_bf16_to_f64(b);
  } else {
    const uint8_t* row = (const uint8_t*)jb->kv + slot * (int64_t)jb->d_qk;
    double x = smla_oracle_e4m3_to_f64(row[c]);
    if (jb->kv_dtype == ORACLE_KV_E4M3) return x * (double)jb->k_scale[0];
    if (jb->kv_dtype == ORACLE_KV_E4M3_GROUP4_KPE)
      return c < 512 ? x * (double)jb->k_scale[slot * 4 + c / 128] : x * jb->kpe_scale;
    int G = (jb->d_qk + 127) / 128;
    return x * (double)jb->k_scale[slot * G + c / 128];
  }
}

/* One token: gather J, dequantize K_j, then every head by the definition. */
static void oracle_token(oracle_job* jb, int64_t pos, double* K, double* s,
                         int64_t* sel) {
  int64_t t = jb->tokens ? jb->tokens[pos] : pos;
  int h = jb->h, d_qk = jb->d_qk, d_v = jb->d_v, topk = jb->topk;
  const int32_t* row = jb->indices + t * (int64_t)topk;
  int64_t v = topk;
  if (jb->valid_len) {
    v = jb->valid_len[t];
    if (v > topk) v = topk;
    if (v < 0) v = 0;
  }
  /* J: positions of the valid prefix whose id is a real slot. */
  int64_t n = 0;
  for (int64_t j = 0; j < v; ++j)
    if (row[j] >= 0 && row[j] < jb->num_slots) sel[n++] = row[j];
  for (int64_t j = 0; j < n; ++j)
    for (int c = 0; c < d_qk; ++c) K[j * d_qk + c] = kv_value(jb, sel[j], c);

  for (int p = 0; p < h; ++p) {
    double* o = jb->out + (pos * h + p) * (int64_t)d_v;
    double* l = jb->lse + pos * h + p;
    const uint16_t* qp = jb->q + (t * h + p) * (int64_t)d_qk;
    if (n == 0) {
      for (int c = 0; c < d_v; ++c) o[c] = 0.0;
      *l = -INFINITY;
      continue;
    }
    double M = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int c = 0; c < d_qk; ++c)
        acc += smla_oracle_bf16_to_f64(qp[c]) * K[j * d_qk + c];
      s[j] = jb->sm_scale * acc;
      if (s[j] > M) M = s[j];
    }
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) Z += exp(s[j] - M);
    double L = M + log(Z);
    *l = L;
    for (int c = 0; c < d_v; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      double w = exp(s[j] - L);
      for (int c = 0; c < d_v; ++c) o[c] += w * K[j * d_qk + c];
    }
  }
}

static void* oracle_worker(void* arg) {
  oracle_job* jb = (oracle_job*)arg;
  double* K = (double*)malloc(sizeof(double) * (size_t)jb->topk * jb->d_qk);
  double* s = (double*)malloc(sizeof(double) * (size_t)jb->topk);
  int64_t* sel = (int64_t*)malloc(sizeof(int64_t) * (size_t)jb->topk);
  if (!K || !s || !sel) {
    pthread_mutex_lock(&jb->lock);
    jb->status = 3;
    pthread_mutex_unlock(&jb->lock);
    free(K); free(s); free(sel);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&jb->lock);
    int64_t pos = jb->next++;
    pthread_mutex_unlock(&jb->lock);
    if (pos >= jb->n_tokens) break;
    oracle_token(jb, pos, K, s, sel);
  }
  free(K); free(s); free(sel);
  return NULL;
}

/*
 * smla_oracle_fwd — the forward for a list of tokens.
 *   q        bf16 bits [T, h, d_qk]
 *   kv       bf16 bits [num_slots, d_qk] (kv_dtype 0), E4M3 bytes
 *            [num_slots, d_qk] (1, 2, 4) or 656-byte rows [num_slots, 656] (3)
 *   k_scale  kv_dtype 1: [1]; 2: [num_slots, ceil(d_qk/128)]; 4: [num_slots, 4];
 *            else unused
 *   kpe_scale  kv_dtype 4: the scale of the 64 rope channels (fp32, like every
 *            other scale); else unused
 *   indices  int32 [T, topk];  valid_len int32 [T] or NULL
 *   tokens   token ids to evaluate (NULL: 0..T-1, then n_tokens must be T)
 *   out      fp64 [n_tokens, h, d_v];  lse fp64 [n_tokens, h]
 * Returns 0 on success, 1 on a bad argument, 3 if a thread could not allocate.
 */
int smla_oracle_fwd(const uint16_t* q, const void* kv, int kv_dtype,
                    const float* k_scale, float kpe_scale, const int32_t* indices,
                    const int32_t* valid_len, int64_t T, int h, int d_qk,
                    int d_v, int topk, int64_t num_slots, double sm_scale,
                    const int64_t* tokens, int64_t n_tokens, double* out,
                    double* lse, int n_threads) {
  if (!q || !kv || !indices || !out || !lse) return 1;
  if (T < 0 || h < 1 || d_qk < 1 || d_v < 1 || d_v > d_qk || topk < 1) return 1;
  if (kv_dtype < 0 || kv_dtype > 4) return 1;
  if ((kv_dtype == ORACLE_KV_E4M3 || kv_dtype == ORACLE_KV_E4M3_GROUP128 ||
       kv_dtype == ORACLE_KV_E4M3_GROUP4_KPE) && !k_scale) return 1;
  if ((kv_dtype == ORACLE_KV_FP8_DS_MLA || kv_dtype == ORACLE_KV_E4M3_GROUP4_KPE) &&
      d_qk != 576) return 1;
  if (!tokens && n_tokens != T) return 1;
  if (tokens)
    for (int64_t i = 0; i < n_tokens; ++i)
      if (tokens[i] < 0 || tokens[i] >= T) return 1;
  if (n_threads < 1) n_threads = 1;
  oracle_job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q; jb.kv = kv; jb.kv_dtype = kv_dtype; jb.k_scale = k_scale;
  jb.kpe_scale = (double)kpe_scale;
  jb.indices = indices; jb.valid_len = valid_len; jb.T = T; jb.h = h;
  jb.d_qk = d_qk; jb.d_v = d_v; jb.topk = topk; jb.num_slots = num_slots;
  jb.sm_scale = sm_scale; jb.tokens = tokens; jb.n_tokens = n_tokens;
  jb.out = out; jb.lse = lse; jb.next = 0; jb.status = 0;
  pthread_mutex_init(&jb.lock, NULL);
  if (n_threads > n_tokens) n_threads = n_tokens > 0 ? (int)n_tokens : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  if (!th) return 3;
  int started = 0;
  for (int i = 0; i < n_threads; ++i) {
    if (pthread_create(&th[i], NULL, oracle_worker, &jb) != 0) break;
    ++started;
  }
  if (started == 0) oracle_worker(&jb);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&jb.lock);
  return jb.status;
}

/*
 * smla_oracle_merge — combine partial results over disjoint key sets.
 * Partial p holds (O_p normalised over its own keys, LSE_p); the union is
 *   LSE = ln sum_p exp(LSE_p)      (terms with LSE_p = -inf contribute 0)
 *   O   = sum_p exp(LSE_p - LSE) O_p
 * and every LSE_p = -inf gives (0, -inf): the cross-rank merge of
 * vLLM API docs flashmla_sparse, _forward_fp8_kv_mixed_batch (DCP path).
 *   o_parts [n_parts, rows, d_v], lse_parts [n_parts, rows] -> out [rows, d_v], lse [rows]
 */
void smla_oracle_merge(const double* o_parts, const double* lse_parts,
                       int n_parts, int64_t rows, int d_v, double* out,
                       double* lse) {
  for (int64_t r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int p = 0; p < n_parts; ++p)
      if (lse_parts[p * rows + r] > M) M = lse_parts[p * rows + r];
    double* o = out + r * d_v;
    for (int c = 0; c < d_v; ++c) o[c] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double Z = 0.0;
    for (int p = 0; p < n_parts; ++p) Z += exp(lse_parts[p * rows + r] - M);
    double L = M + log(Z);
    lse[r] = L;
    for (int p = 0; p < n_parts; ++p) {
      double w = exp(lse_parts[p * rows + r] - L);
      const double* op = o_parts + ((int64_t)p * rows + r) * d_v;
      for (int c = 0; c < d_v; ++c) o[c] += w * op[c];
    }
  }
}

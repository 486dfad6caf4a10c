// smla_simt.cu — portable fp32 (CUDA-core) sparse MLA forward and the
// LSE-weighted combine kernel.
//
// The forward here is the general path: any h in 1..128, any topk, every KV
// format.  One CTA owns (token, group of 16 heads, top-k position range);
// per block of 32 positions it
//   a1  reads the slot ids of the block and masks ids < 0, >= num_slots and
//       positions >= valid_len (flashinfer_mla_sparse_sm90.py, forward_mqa:
//       compacted valid prefix, -1 past it),
//   a2  gathers the selected rows into shared memory (16-byte loads),
//   a3  dequantizes E4M3 with the per-tensor or per-(slot, 128-channel group)
//       scale (same page, module docstring), the 656-byte fp8_ds_mla row
//       (scales and bf16 rope inside the row; vLLM "Sparse MLA on Hopper",
//       cutlass_fa3_sparse.py module docstring: 656 bytes per token), or four
//       ckv group scales with a separate kpe scale (flashinfer page,
//       forward_mqa: ckv_scale and kpe_scale),
//   a4  forms s = sm_scale * q . K over d_qk (vLLM "Sparse MLA on Hopper",
//       ops/cutlass_fa3.py docstring: score = q_rope.k_rope + q_nope.c_kv),
//   a5  updates the running max / sum (online softmax),
//   a6  accumulates P . V with V the first 512 channels of the same rows,
// and a7 writes O / LSE, or fp32 partials when the range is split (a8 is
// smla_combine_kernel).  Empty sets give (0, -inf) (vLLM API docs
// flashmla_sparse, _forward_fp8_kv_mixed_batch).
#include <cuda_bf16.h>
#include <math.h>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kHeads = 16;    // heads per CTA
constexpr int kBlock = 32;    // top-k positions per inner step
constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// E4M3 ("fn") byte -> float, from the format: bias 7, 3 mantissa bits,
// exponent field 0 subnormal, S.1111.111 NaN, no infinity.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t e = (b >> 3) & 0xF, m = b & 7;
  float mag;
  if (e == 0xF && m == 7) {
    mag = __uint_as_float(0x7FC00000u);
  } else if (e == 0) {
    mag = (float)m * 0.001953125f;  // m/8 * 2^-6 = m * 2^-9
  } else {
    mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
  }
  return (b & 0x80) ? -mag : mag;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int KV>
__global__ void __launch_bounds__(kThreads)
smla_simt_kernel(FwdParams p, int n_groups) {
  extern __shared__ float smem[];
  const int d_qk = p.d_qk;
  float* Qs = smem;                         // [kHeads][d_qk]
  float* Ks = Qs + kHeads * d_qk;           // [kBlock][d_qk]
  float* Ps = Ks + kBlock * d_qk;           // [kHeads][kBlock]
  float* alpha = Ps + kHeads * kBlock;      // [kHeads]
  float* m_s = alpha + kHeads;              // [kHeads]
  float* l_s = m_s + kHeads;                // [kHeads]
  int* slot = reinterpret_cast<int*>(l_s + kHeads);  // [kBlock]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int unit = blockIdx.x;
  const int split = unit % p.splits;
  unit /= p.splits;
  const int grp = unit % n_groups;
  const int t = unit / n_groups;
  const int h0 = grp * kHeads;
  const int nh = min(kHeads, p.h - h0);

  int v = p.topk;
  if (p.valid_len) v = min(max(p.valid_len[t], 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);

  // Q rows of this head group -> fp32 in shared memory (zero past nh).
  for (int i = tid; i < kHeads * (d_qk / 8); i += kThreads) {
    const int hh = i / (d_qk / 8), c = (i % (d_qk / 8)) * 8;
    float* dst = Qs + hh * d_qk + c;
    if (hh < nh) {
      const uint4 w = __ldg(q_chunk(p, t, h0 + hh, c));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dst[2 * e] = bf16_bits_to_float(ws[e] & 0xFFFFu);
        dst[2 * e + 1] = bf16_bits_to_float(ws[e] >> 16);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = 0.f;
    }
  }
  if (tid < kHeads) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  float acc[kHeads][2];
#pragma unroll
  for (int i = 0; i < kHeads; ++i) acc[i][0] = acc[i][1] = 0.f;
  const int c0 = 2 * tid;  // this thread's two output channels (d_v = 512)

  for (int kb = k0; kb < k1; kb += kBlock) {
    __syncthreads();
    if (tid < kBlock) {
      int j = kb + tid, id = -1;
      if (j < k1) {
        bool bad = false;
        const int req = token_req(p, t, bad);
        id = to_slot(p, req, p.indices[(int64_t)t * p.topk + j], bad);
        if (bad) atomicCAS(p.status, 0, kStatusBadIndex);
      }
      slot[tid] = id;
    }
    __syncthreads();
    // a2 + a3: gather (and dequantize) the rows; masked rows are zero.
    if (KV == kBf16) {
      const int chunks = d_qk / 8;  // 16-byte chunks per row
      for (int i = tid; i < kBlock * chunks; i += kThreads) {
        int r = i / chunks, c = (i % chunks) * 8;
        int id = slot[r];
        float* dst = Ks + r * d_qk + c;
        if (id < 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = 0.f;
        } else {
          const uint4 w = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint16_t*>(p.kv) + (int64_t)id * d_qk + c);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dst[2 * e] = bf16_bits_to_float(ws[e] & 0xFFFFu);
            dst[2 * e + 1] = bf16_bits_to_float(ws[e] >> 16);
          }
        }
      }
    } else {
      const int chunks = d_qk / 16;
      const int G = (d_qk + 127) / 128;
      for (int i = tid; i < kBlock * chunks; i += kThreads) {
        int r = i / chunks, c = (i % chunks) * 16;
        int id = slot[r];
        float* dst = Ks + r * d_qk + c;
        if (id < 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) dst[e] = 0.f;
        } else if (KV == kDsMla && c >= 512) {
          // rope: 16 bf16 values (32 bytes) of the 656-byte row
          const uint4* src = reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint8_t*>(p.kv) + (int64_t)id * kDsMlaRowBytes +
              kDsMlaRopeOff + 2 * (c - 512));
          const uint4 w0 = __ldg(src), w1 = __ldg(src + 1);
          const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            dst[2 * e] = bf16_bits_to_float(ws[e] & 0xFFFFu);
            dst[2 * e + 1] = bf16_bits_to_float(ws[e] >> 16);
          }
        } else {
          const uint8_t* row = reinterpret_cast<const uint8_t*>(p.kv) +
                               (int64_t)id * (KV == kDsMla ? kDsMlaRowBytes : d_qk);
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(row + c));
          float sc;
          if (KV == kE4m3) sc = p.k_scale[0];
          else if (KV == kE4m3Group) sc = p.k_scale[(int64_t)id * G + c / 128];
          else if (KV == kDsMla)
            sc = __ldg(reinterpret_cast<const float*>(row + kDsMlaScaleOff) + c / 128);
          else sc = c < 512 ? p.k_scale[(int64_t)id * 4 + c / 128] : p.kpe_scale;
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 16; ++e)
            dst[e] = e4m3_to_float((ws[e >> 2] >> (8 * (e & 3))) & 0xFF) * sc;
        }
      }
    }
    __syncthreads();
    // a4 + a5: warp w owns heads 2w and 2w+1; lane j ends up with key j.
#pragma unroll
    for (int hh2 = 0; hh2 < 2; ++hh2) {
      const int hh = warp * 2 + hh2;
      const float* qh = Qs + hh * d_qk;
      float mine = -INFINITY;
      for (int kk = 0; kk < kBlock; ++kk) {
        const float* kr = Ks + kk * d_qk;
        float part = 0.f;
        for (int c = lane; c < d_qk; c += 32) part = fmaf(qh[c], kr[c], part);
        part = warp_sum(part);
        if (lane == kk) mine = (slot[kk] >= 0) ? part * p.sm_scale : -INFINITY;
      }
      const float m_old = m_s[hh];
      const float m_new = fmaxf(m_old, warp_max(mine));
      float pj = 0.f, a = 1.f;
      if (m_new != -INFINITY) {
        pj = expf(mine - m_new);
        a = expf(m_old - m_new);
      }
      const float sum = warp_sum(pj);
      Ps[hh * kBlock + lane] = pj;
      if (lane == 0) {
        alpha[hh] = a;
        m_s[hh] = m_new;
        l_s[hh] = l_s[hh] * a + sum;
      }
    }
    __syncthreads();
    // a6: O[hh, c0..c0+1] = alpha * O + sum_kk P[hh, kk] * V[kk, c0..c0+1]
#pragma unroll
    for (int hh = 0; hh < kHeads; ++hh) {
      acc[hh][0] *= alpha[hh];
      acc[hh][1] *= alpha[hh];
    }
    for (int kk = 0; kk < kBlock; ++kk) {
      const float2 vv = *reinterpret_cast<const float2*>(Ks + kk * d_qk + c0);
#pragma unroll
      for (int hh = 0; hh < kHeads; ++hh) {
        const float pw = Ps[hh * kBlock + kk];
        acc[hh][0] = fmaf(pw, vv.x, acc[hh][0]);
        acc[hh][1] = fmaf(pw, vv.y, acc[hh][1]);
      }
    }
  }
  __syncthreads();

  // a7: epilogue.
#pragma unroll
  for (int hh = 0; hh < kHeads; ++hh) {
    if (hh >= nh) break;
    const float l = l_s[hh], m = m_s[hh];
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    const float lse_v = empty ? -INFINITY : m + logf(l);
    const int64_t row = (int64_t)t * p.h + h0 + hh;
    if (p.fp32_out) {
      const int64_t prow = (int64_t)split * p.T * p.h + row;
      float2 o = make_float2(acc[hh][0] * inv, acc[hh][1] * inv);
      *reinterpret_cast<float2*>(p.o_part + prow * p.d_v + c0) = o;
      if (tid == 0) p.lse_part[prow] = lse_v;
    } else {
      __nv_bfloat162 o = __floats2bfloat162_rn(acc[hh][0] * inv, acc[hh][1] * inv);
      *reinterpret_cast<__nv_bfloat162*>(
          reinterpret_cast<__nv_bfloat16*>(p.out) + row * p.d_v + c0) = o;
      if (tid == 0 && p.lse) p.lse[row] = lse_v;
    }
  }
}

// a8: one CTA of 128 threads per row; 4 channels a thread (d_v = 512).
__global__ void __launch_bounds__(128)
smla_combine_kernel(const float* __restrict__ o_parts,
                    const float* __restrict__ lse_parts, int n_parts,
                    int64_t rows, int d_v, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse) {
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  float M = -INFINITY;
  for (int s = 0; s < n_parts; ++s) M = fmaxf(M, lse_parts[s * rows + r]);
  const int c = threadIdx.x * 4;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (M != -INFINITY) {
    float Z = 0.f;
    for (int s = 0; s < n_parts; ++s) Z += expf(lse_parts[s * rows + r] - M);
    L = M + logf(Z);
    for (int s = 0; s < n_parts; ++s) {
      const float ls = lse_parts[s * rows + r];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - L);
      const float4 x = *reinterpret_cast<const float4*>(
          o_parts + ((int64_t)s * rows + r) * d_v + c);
      o.x = fmaf(w, x.x, o.x);
      o.y = fmaf(w, x.y, o.y);
      o.z = fmaf(w, x.z, o.z);
      o.w = fmaf(w, x.w, o.w);
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + r * d_v + c) = packed;
  if (threadIdx.x == 0 && lse) lse[r] = L;
}

}  // namespace

size_t simt_smem_bytes(int d_qk) {
  return sizeof(float) * ((size_t)(kHeads + kBlock) * d_qk + kHeads * kBlock +
                          3 * kHeads) +
         sizeof(int) * kBlock;
}

template <int KV>
cudaError_t launch_simt_fmt(const FwdParams& p, int n_groups, int64_t blocks, size_t smem,
                            cudaStream_t stream) {
  const cudaError_t e = cudaFuncSetAttribute(
      smla_simt_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  smla_simt_kernel<KV><<<(unsigned)blocks, kThreads, smem, stream>>>(p, n_groups);
  return cudaGetLastError();
}

cudaError_t launch_simt(const FwdParams& p, cudaStream_t stream) {
  const int n_groups = (p.h + kHeads - 1) / kHeads;
  const int64_t blocks = (int64_t)p.T * n_groups * p.splits;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const size_t smem = simt_smem_bytes(p.d_qk);
  switch (p.kv_format) {
    case kBf16: return launch_simt_fmt<kBf16>(p, n_groups, blocks, smem, stream);
    case kE4m3: return launch_simt_fmt<kE4m3>(p, n_groups, blocks, smem, stream);
    case kE4m3Group: return launch_simt_fmt<kE4m3Group>(p, n_groups, blocks, smem, stream);
    case kDsMla: return launch_simt_fmt<kDsMla>(p, n_groups, blocks, smem, stream);
    default: return launch_simt_fmt<kE4m3Group4Kpe>(p, n_groups, blocks, smem, stream);
  }
}

cudaError_t launch_combine(const float* o_parts, const float* lse_parts,
                           int n_parts, int64_t rows, int d_v, void* out,
                           float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  smla_combine_kernel<<<(unsigned)rows, 128, 0, stream>>>(
      o_parts, lse_parts, n_parts, rows, d_v,
      reinterpret_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace smla

// smla_combine.cu — a8, the LSE-weighted combine of partial results.
//
// A top-k range split over several units (or ranks: the DCP split of the
// vLLM API docs flashmla_sparse page, FlashMLASparseImpl, whose partial
// outputs are merged through their LSE) leaves per part a normalised O_s and
// its LSE_s; the merge is
//   LSE = ln sum_s exp(LSE_s)     (parts with LSE_s = -inf skipped;
//                                  all -inf -> -inf, O = 0)
//   O   = sum_s exp(LSE_s - LSE) * O_s
// and writes bf16 O and fp32 LSE.  HBM-bound: per row, parts * (4 d_v + 4)
// bytes read and 2 d_v + 4 written.
#include <cuda_bf16.h>
#include <math.h>

#include "smla_internal.h"

namespace smla {
namespace {

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

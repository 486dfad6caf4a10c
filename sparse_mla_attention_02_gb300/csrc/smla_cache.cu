// smla_cache.cu — group-quantizing E4M3 cache write.
//
// The flashinfer_mla_sparse_sm90.py page reads E4M3 caches with one fp32
// scale per (slot, 128-channel group) (its ckv_scale_arr layout) and notes
// that the cache-write op producing that layout is missing; vLLM's
// concat_and_cache_mla (same pages) is the write for the other formats: a
// token's row [kv_c (512) | k_pe (64)] goes to the cache row at its slot.
// This kernel is that write for the group format:
//   for each written row and group g (channels [128 g, 128 g + 128)):
//     scale = amax|x| / 448 in fp32 (1 for an all-zero group),
//     code  = e4m3(x / scale), fp32 division, round to nearest even,
//             saturating at +-448 (the satfinite conversion).
// HBM-bound: per row 2 * d_qk bytes read, d_qk + 4 * G written.
//
// One warp per token row.  The row is 64 (d_qk 512) or 72 (576) chunks of
// 8 channels; lane l converts chunks l, l + 32 and, for the rope group,
// 64 + l (l < 8).  A group's chunks sit in one half-warp (16 lanes; the rope
// group in 8), so the group max is a shuffle reduction within it.
#include <cuda_bf16.h>

#include "smla_internal.h"

namespace smla {
namespace {

struct CacheArgs {
  const uint16_t* kv_c;   // bf16 [N, 512]
  const uint16_t* k_pe;   // bf16 [N, d_qk - 512] or nullptr (d_qk 512)
  const int32_t* slot;    // [N]
  uint8_t* cache;         // [num_slots, d_qk]
  float* scales;          // [num_slots, G]
  int* status;
  int64_t num_slots;
  int N, d_qk, G;
};

// Two floats -> two E4M3 codes (RN, saturating): lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) smla_cache_write_kernel(const CacheArgs a) {
  const int lane = threadIdx.x & 31;
  const int n = (int)((blockIdx.x * 256u + threadIdx.x) >> 5);
  if (n >= a.N) return;
  const int s = __ldg(a.slot + n);
  if (s < 0) return;
  if (s >= a.num_slots) {
    if (lane == 0) atomicCAS(a.status, 0, kStatusBadIndex);
    return;
  }
  const int nchunks = a.d_qk / 8;
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int k = 32 * pass + lane;                  // this lane's chunk
    const bool live = pass < 2 ? k < nchunks : (nchunks > 64 && lane < 8);
    // channels 8k..8k+7: kv_c for k < 64, k_pe after
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (live)
      raw = k < 64 ? __ldg(reinterpret_cast<const uint4*>(a.kv_c + (int64_t)n * 512) + k)
                   : __ldg(reinterpret_cast<const uint4*>(a.k_pe + (int64_t)n * (a.d_qk - 512)) +
                           (k - 64));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    // group max: within the half-warp (passes 0, 1) or lanes 0..7 (pass 2)
    const int width = pass < 2 ? 16 : 8;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1)
      if (o < width) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (!live) continue;
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    const uint32_t c01 = e4m3x2(x[0] / scale, x[1] / scale);
    const uint32_t c23 = e4m3x2(x[2] / scale, x[3] / scale);
    const uint32_t c45 = e4m3x2(x[4] / scale, x[5] / scale);
    const uint32_t c67 = e4m3x2(x[6] / scale, x[7] / scale);
    *reinterpret_cast<uint2*>(a.cache + (int64_t)s * a.d_qk + 8 * k) =
        make_uint2(c01 | (c23 << 16), c45 | (c67 << 16));
    const int g = k >> 4;                            // 128-channel group
    if ((k & 15) == 0) a.scales[(int64_t)s * a.G + g] = scale;
  }
}

}  // namespace

cudaError_t launch_cache_write(const void* kv_c, const void* k_pe, const int32_t* slot,
                               int N, int d_qk, int64_t num_slots, void* cache,
                               float* scales, int* status, cudaStream_t stream) {
  CacheArgs a{};
  a.kv_c = static_cast<const uint16_t*>(kv_c);
  a.k_pe = static_cast<const uint16_t*>(k_pe);
  a.slot = slot;
  a.cache = static_cast<uint8_t*>(cache);
  a.scales = scales;
  a.status = status;
  a.num_slots = num_slots;
  a.N = N;
  a.d_qk = d_qk;
  a.G = (d_qk + 127) / 128;
  const unsigned blocks = (unsigned)(((int64_t)N * 32 + 255) / 256);
  smla_cache_write_kernel<<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace smla

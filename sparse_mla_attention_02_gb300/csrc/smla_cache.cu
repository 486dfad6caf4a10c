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
// Eight lanes per token row, four rows per warp.  A row is 64 (d_qk 512) or
// 72 (576) chunks of 8 channels; lane j of the row's eight converts chunks
// j + 8 i, i < 8 or 9 (all of its loads issued first), so that group g is
// chunks i = 2g, 2g + 1 of all eight lanes (the rope group, i = 8, alone):
// the group max is a shuffle reduction over the eight lanes.
//
// The kernel is bound by instruction issue as much as by HBM, so the fp32
// quotients take no division: each is the IEEE quotient x / scale, reached
// by one multiply and two fused multiply-adds (Markstein's correction of
// x * RN(1/scale)), in packed f32x2 arithmetic.
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
  int N;
};

// Two floats -> two E4M3 codes (RN, saturating): lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// RN(amax / 448) without a division: amax * RN(1/448) is within an ulp and
// one fma residual correction (Markstein) rounds it; checked against the
// IEEE quotient for every positive finite bf16 amax (amax is a bf16 value).
__device__ __forceinline__ float amax_over_448(float amax) {
  constexpr float kInv = 1.f / 448.f;
  const float q0 = amax * kInv;
  if (!(amax <= 3.0e38f)) return q0;                 // inf: inf / 448
  return fmaf(fmaf(-q0, 448.f, amax), kInv, q0);
}

// RN(1/s) for a normal s: one Newton step from the hardware approximation
// (within an ulp); checked for the scale of every bf16 amax mantissa, from
// the approximation and from both of its fp32 neighbours.
__device__ __forceinline__ float recip_rn(float s) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(s));
  return fmaf(fmaf(-s, y, 1.f), y, y);
}

// Scales whose quotients the main path does not cover: below 2^-64 (the
// residual could lose bits to underflow), inf and NaN.  The largest finite
// scale (bf16 amax / 448) is below 2^120.
__device__ __forceinline__ bool special_scale(float s) {
  return !(s >= 0x1p-64f && s <= 0x1p120f);
}

// Quotients of 8 channels given as their negations xn (two per 64-bit word)
// with ny = -RN(1/s):
//   q0 = x * y,  u = q0 * s - x (exact, one fma),  q = q0 - u * y.
// q is RN(x / s) (Markstein: y the correctly rounded reciprocal, q0 within
// an ulp), checked for every bf16 x against every bf16 amax's scale.  The
// negated inputs make the signs of zeros come out as the division's.
__device__ __forceinline__ uint2 codes8(const uint64_t (&xn)[4], uint64_t s2, uint64_t ny2) {
  uint32_t c[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint64_t q0 = mul2(xn[p], ny2);
    const uint64_t u = fma2(q0, s2, xn[p]);
    float lo, hi;
    unpack2(fma2(u, ny2, q0), lo, hi);
    c[p] = e4m3x2(lo, hi);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// A 16-byte chunk of 8 bf16 -> their negations as 4 packed fp32 pairs, and
// the largest magnitude folded into amax.
__device__ __forceinline__ void unpack_neg8(const uint4 v, uint64_t (&xn)[4], float& amax) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float lo = __uint_as_float((w[p] << 16) ^ 0x80000000u);
    const float hi = __uint_as_float((w[p] & 0xFFFF0000u) ^ 0x80000000u);
    amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
    xn[p] = pack2(lo, hi);
  }
}

// One chunk's codes for a special scale (the rare tail): a tiny scale and
// the chunk are first multiplied by 2^64 (the quotients are unchanged); inf
// and NaN scales give x * rcp(scale) (x / inf = +-0 for finite x, NaN for
// x = inf; x / NaN = NaN).
__device__ __forceinline__ uint2 special_codes8(const uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float q[8];
  if (s < 0x1p-64f) {
    const float ss = s * 0x1p64f;
    const float y = recip_rn(ss);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t b = e & 1 ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
      const float xn = -__uint_as_float(b) * 0x1p64f;
      const float q0 = xn * -y;
      q[e] = fmaf(fmaf(q0, ss, xn), -y, q0);
    }
  } else {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t b = e & 1 ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
      q[e] = __uint_as_float(b) * r;
    }
  }
  return make_uint2(e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16),
                    e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16));
}

// kChunks = d_qk / 64: 9 (kv_c + rope) or 8 (kv_c only).
template <int kChunks>
__global__ void __launch_bounds__(256) smla_cache_write_kernel(const CacheArgs a) {
  constexpr int kD = 8 * 8 * kChunks;                // d_qk
  constexpr int kG = (kChunks + 1) / 2;              // groups
  const int j = threadIdx.x & 7;                     // lane within the row's eight
  const int n = (int)((blockIdx.x * 256u + threadIdx.x) >> 3);
  int s = n < a.N ? __ldg(a.slot + n) : -1;
  if (s >= a.num_slots) {
    if (j == 0) atomicCAS(a.status, 0, kStatusBadIndex);
    s = -1;
  }
  const bool ok = s >= 0;
  // chunk i of this lane: channel 8 (j + 8 i)
  auto src = [&](int i) {
    return i < 8 ? reinterpret_cast<const uint4*>(a.kv_c + (int64_t)n * 512) + j + 8 * i
                 : reinterpret_cast<const uint4*>(a.k_pe + (int64_t)n * 64) + j;
  };
  uint4 raw[kChunks];
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    raw[i] = make_uint4(0u, 0u, 0u, 0u);
    if (ok) raw[i] = __ldg(src(i));
  }
  uint8_t* row = a.cache + (int64_t)s * kD;
  float* srow = a.scales + (int64_t)s * kG;
  uint32_t special = 0;                              // groups with a special scale
  float scale_g[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    const int i0 = 2 * g, nc = (2 * g + 1 < kChunks) ? 2 : 1;
    uint64_t xn[2][4];
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < nc; ++c) unpack_neg8(raw[i0 + c], xn[c], amax);
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? amax_over_448(amax) : 1.f;
    scale_g[g] = scale;
    special |= special_scale(scale) ? 1u << g : 0u;
    const float ny = -recip_rn(scale);
    const uint64_t s2 = pack2(scale, scale), ny2 = pack2(ny, ny);
    if (ok) {
#pragma unroll
      for (int c = 0; c < nc; ++c)
        *reinterpret_cast<uint2*>(row + 8 * (j + 8 * (i0 + c))) = codes8(xn[c], s2, ny2);
      if (j == 0) srow[g] = scale;
    }
  }
  if (ok && special) {                               // rare: redo the special groups
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      if (!(special >> g & 1u)) continue;
      for (int i = 2 * g; i < 2 * g + 2 && i < kChunks; ++i)
        *reinterpret_cast<uint2*>(row + 8 * (j + 8 * i)) = special_codes8(__ldg(src(i)), scale_g[g]);
    }
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
  const unsigned blocks = (unsigned)(((int64_t)N * 8 + 255) / 256);
  if (d_qk == 576)
    smla_cache_write_kernel<9><<<blocks, 256, 0, stream>>>(a);
  else
    smla_cache_write_kernel<8><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace smla

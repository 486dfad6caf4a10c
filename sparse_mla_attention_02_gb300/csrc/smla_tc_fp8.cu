// smla_tc_fp8.cu — tensor-core sparse MLA forward that feeds the E4M3 cache
// bytes to the tensor core as they are (tcgen05 .kind::f8f6f4), for every
// E4M3 cache format: one scale per tensor, per (slot, 128-channel group),
// the 656-byte fp8_ds_mla row, and four ckv group scales + a kpe scale.
//
// The pages read FP8 caches directly and apply the scales outside the
// product (flashinfer_mla_sparse_sm90.py, module docstring: FP8 cache read
// directly, half the bf16 HBM traffic, per-tensor k_scale or per-token x
// 128-channel-group scales).  Here the gathered rows are not converted at
// all: TMA gathers the raw E4M3 rows into shared memory, and both MMAs read
// them as E4M3 operands.  The other operand of each product is split into
// E4M3 terms (a pair for Q, three for the softmax weights):
//   * Q (bf16): per head, x = q * 2^a with a power of two a that puts
//     max|x| in [128, 256); hi = E4M3(x), lo = E4M3(16 (x - hi)), so that
//     x = hi + lo / 16 up to 2^-9 of x's binade (or 2^-14 absolute).  The
//     two are the MMA's N rows [16 heads hi | 16 heads lo]; the score is
//     2^-a (S_hi + S_lo / 16), summed in fp32.
//   * P (fp32, in [0, 2^4] by the lazy running max below): each V group g
//     gets x = p * scale_g * R_g * 2^4, R_g a power of two that keeps
//     scale_g * R_g <= 1 (one scale per tensor: x = 16 p), split into three
//     E4M3 terms, x = hi + mid / 16 + lo / 256 (mid = E4M3(16 (x - hi)), lo
//     the same of the next residual), which give back the f16 value of x
//     exactly from 2^-6 up (below, to 2^-18 absolute): a weight keeps the
//     f16 step of the split, 2^-11 of its binade.  The weight of a key that
//     carries its row can be anywhere in that range (it carries its scale,
//     and the lazy max leaves p in (1, 2^4]); with two terms (2^-9) a row
//     that one key carries with |v| near 4 came out 0.0208 from the oracle
//     (the output's own bf16 rounding takes up to 0.0156 of the 2e-2 bound
//     there).  The three are the 48 columns [hi | mid | lo] of the PV
//     operand; O = (O_hi + O_mid / 16 + O_lo / 256) / (16 R_g l).
// Keys are the MMA's M dimension (keys-major), heads its N:
//   S^T[keys, 32] = K[keys, d] . Q'^T[d, 32]      A = gathered tile, K-major
//   O^T[ch, 48]  += V^T[ch, keys] . P'^T[keys, 48] A = the same tile, MN-major
// A block is 128 keys (M = 128), full 576-byte rows in five 128-byte chunks
// (four ckv chunks and the rope chunk; for the 656-byte row the rope chunk
// holds its 64 bf16 values and its QK runs as a bf16 MMA).  With group
// scales, QK keeps one fp32 accumulator per channel group, so a key's group
// scale multiplies its partial score exactly (in fp32).
// One work unit = (token, top-k range, group of 16 heads) on one CTA.
//
// Method steps (vLLM "Sparse MLA on Hopper" diff, ops/cutlass_fa3.py
// docstring: score = q_rope.k_rope + q_nope.c_kv, output = softmax(score *
// scale) @ c_kv; flashinfer_mla_sparse_sm90.py, forward_mqa: compacted valid
// prefix with -1 past it; vLLM API docs flashmla_sparse,
// _forward_fp8_kv_mixed_batch: empty rows give (O = 0, LSE = -inf)):
//   a1 work setup: v = min(valid_len[t], topk); range [k0, k1) of the split
//   a2 gather: slot ids -> raw rows: TMA tile::gather4 for the ckv chunks,
//      cp.async for the rope (masked rows: zero fill)
//   a3 scales: per-tensor scale on the score scale and the output; group
//      scales on the group accumulators (QK) and inside P' (PV)
//   a4 QK^T, a5 masked online softmax, a6 PV, a7 O / l and LSE = m + ln l
//
// Warp roles (448 threads): warp 0 issues the QK MMAs and owns TMEM; warp 13
// issues the PV MMAs; warps 1..4 load the unit's slot ids, issue the
// gathers (each 32 tile rows) and build Q' of every unit after the first;
// warps 5..12 are two softmax warpgroups (thread <-> key <-> TMEM lane;
// warpgroup w owns heads [8w, 8w + 8)), which build the first unit's Q' and
// write O and LSE.
// Every wait is bounded; a wait that runs out records a timeout status, sets
// an abort flag that skips later waits, and the block drains its copies and
// MMAs and finishes normally.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "smla_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kBK = 128;                   // keys per block (MMA M)
constexpr int kStages = 2;                 // gathered-tile pipeline depth
constexpr int kChunkBytes = kBK * 128;     // one 128-byte column chunk of 128 rows
constexpr int kMaxChunks = 5;              // 4 ckv chunks + the rope chunk
constexpr int kStageBytes = kMaxChunks * kChunkBytes;
constexpr int kHeads = 16;                 // heads per CTA
constexpr int kNq = 32;                    // QK N: 16 heads hi | 16 heads lo
constexpr int kQChunkBytes = kNq * 128;
constexpr int kPBytes = kBK * 128;         // one P' region: a 128-byte row per key
constexpr int kNoMax = 48;                 // PV N: 16 heads hi | mid | lo
constexpr int kThreads = 448;
constexpr int kProducers = 128;            // warps 1..4
constexpr int kSoftmax = 256;              // warps 5..12
constexpr int kMaxBlocks = 16;             // ranges up to 2048 positions
constexpr float kT = 4.f;                  // lazy max threshold (log2 units)
constexpr float kPShift = 16.f;            // 2^(8 - kT): P' <= 2^8

// TMEM columns.
// O^T: 4 blocks of 128 channels x (48 or 32) from column 0, then S: 2
// buffers x 5 accumulators x 32.
constexpr uint32_t kColO = 0;
constexpr uint32_t kSBuf = 5 * kNq;
constexpr uint32_t kTmemCols = 512;
static_assert(4 * kNoMax + 2 * kSBuf <= kTmemCols, "TMEM budget");

// Shared-memory layout (offsets from a 1024-byte aligned base).  The tile
// stages carry, beside the rows, each block's valid-bit words and (group
// formats) its keys' scales, written by the producers with the gathers.
constexpr int kScaleRow = 5;                                       // floats per key
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffQ = kOffTile + kStages * kStageBytes;       // Q' chunks
// P' (one buffer, two regions: groups 0, 1 and groups 2, 3; one scale per
// tensor uses region 0 only); the bf16 O staging rows [16 heads][512] share
// region 1 (written once the unit's last PV has read P', and read by a bulk
// copy that completes before the next unit's first P' is written).
constexpr uint32_t kOffP = kOffQ + kMaxChunks * kQChunkBytes;
constexpr uint32_t kOffOst = kOffP + kPBytes;
constexpr uint32_t kOffSlot = kOffP + 2 * kPBytes;                 // [blocks*128] i32
constexpr uint32_t kOffSc = kOffSlot + kMaxBlocks * kBK * 4;       // [2][128][5] f32
constexpr uint32_t kOffMask = kOffSc + kStages * kBK * kScaleRow * 4;  // [2][4] u32
constexpr uint32_t kOffRed = kOffMask + kStages * 16;              // [2 wg][4 warps][8] f32
constexpr uint32_t kOffRedSc = kOffRed + 2 * 4 * 8 * 4;            // [2 wg][4 warps][4] f32
constexpr uint32_t kOffQf = kOffRedSc + 2 * 4 * 4 * 4;             // [2][16] f32: 2^-a per head
constexpr uint32_t kOffFac = kOffQf + 2 * kHeads * 4;             // [2 wg][8 alpha | 4 ratio] f32
constexpr uint32_t kOffBar = kOffFac + 2 * 12 * 4;
enum {
  kBarKvFull = 0,                   // [2] the tile, masks and scales of a block
  kBarKvEmpty = kBarKvFull + 2,     // [2]
  kBarSFull = kBarKvEmpty + 2,      // [2]
  kBarSEmpty = kBarSFull + 2,       // [2]
  kBarPFull = kBarSEmpty + 2,
  kBarPEmpty,
  kBarODone,
  kBarOFinal,                       // one phase per unit: its last PV is done
  kBarQReady,                       // one phase per unit: Q' written
  kBarQUsed,                        // one phase per unit: the softmax warps read qf_sh
  kBarDrain,                        // teardown: both MMA warps' MMAs are done
  kNumBars
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled operands need 1024-B alignment");
static_assert(kOffRed % 16 == 0 && kOffBar % 8 == 0, "alignment");
static_assert(kHeads * 512 * 2 <= kPBytes, "O staging fits in P' region 1");

struct Fp8Args {
  CUtensorMap kv_map;  // the cache as bytes [num_slots, row bytes], 128-byte boxes
  FwdParams p;
  int n_hg;            // head groups of 16 (units per token and range)
  int n_units;         // T * splits * n_hg
  int upc, n_big;      // CTAs [0, n_big / upc) run upc consecutive units each;
                       // the CTAs after them one unit each (see unit_range)
  int rope_x;          // byte offset of the rope box in a row (576-channel rows)
  int G;               // scales per slot (E4M3 group format)
  float scale_log2;    // sm_scale * log2(e)
};

// tcgen05 MMA with E4M3 A and B (fp32 accumulate), operands in shared memory.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor: E4M3 A and B (format code 0), fp32 D.
constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Split x0..x7 (|x| <= 448) into hi = E4M3(x) and lo = E4M3(16 (x - hi)),
// eight codes each (x0 in the lowest byte).  The pairs go through f16: x is
// rounded to f16 first (2^-11 relative, below the pair's 2^-9), and x - hi
// and its product by 16 are exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_of_h2(__half2 h) {
  return (uint32_t)__nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&h),
                                              __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ __half2 h2_of_e4m3x2(uint32_t v) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return *reinterpret_cast<const __half2*>(&r);
}
__device__ __forceinline__ void split8(const float (&x)[8], uint2& hi, uint2& lo) {
  uint32_t h[4], l[4];
  const __half2 k16 = __float2half2_rn(16.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 xh = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
    h[k] = e4m3x2_of_h2(xh);
    l[k] = e4m3x2_of_h2(__hmul2(__hsub2(xh, h2_of_e4m3x2(h[k])), k16));
  }
  hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}
// Split p[0..7] * f into kTerms E4M3 terms, x = t0 + t1 / 16 (+ t2 / 256):
// t0 = E4M3(x), each next term E4M3 of 16 times the residual left by the
// one before (each residual and its product by 16 exact in f16; |x| <= 256
// keeps every term within E4M3's range).  Term k's eight codes are stored
// (x0 in the lowest byte) at dst(k) as each term is ready, so that only one
// term's codes are live at a time.
template <int kTerms, typename Dst>
__device__ __forceinline__ void split_store8(const float (&p)[8], float f, Dst dst) {
  const __half2 k16 = __float2half2_rn(16.f);
  __half2 r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = __floats2half2_rn(p[2 * k] * f, p[2 * k + 1] * f);
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = e4m3x2_of_h2(r[k]);
    *dst(t) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    if (t + 1 < kTerms) {
#pragma unroll
      for (int k = 0; k < 4; ++k) r[k] = __hmul2(__hsub2(r[k], h2_of_e4m3x2(c[k])), k16);
    }
  }
}

// Reduce v[0..7] (one value per head) over the 32 lanes of the warp; lane l
// ends with the result for head (l >> 1) & 7.
template <bool kMax>
__device__ __forceinline__ float op2(float x, float y) {
  return kMax ? fmaxf(x, y) : x + y;
}
template <bool kMax, int kW>
__device__ __forceinline__ void xreduce_step(float (&v)[8], int lane) {
  const bool hi = (lane & (2 * kW)) != 0;
#pragma unroll
  for (int j = 0; j < kW; ++j) {
    const float send = hi ? v[j] : v[j + kW];
    const float keep = hi ? v[j + kW] : v[j];
    v[j] = op2<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, 2 * kW));
  }
}
template <bool kMax>
__device__ __forceinline__ float xreduce8(float (&v)[8], int lane) {
  xreduce_step<kMax, 4>(v, lane);
  xreduce_step<kMax, 2>(v, lane);
  xreduce_step<kMax, 1>(v, lane);
  const float x = op2<kMax>(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
  return op2<kMax>(x, __shfl_xor_sync(0xffffffffu, x, 16));
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// The smallest power of two R (as 2^e, e in [-126, 126]) with x * R <= 1,
// for x > 0.
__device__ __forceinline__ float pow2_at_most_inv(float x) {
  int e = ((__float_as_int(x) >> 23) & 255) - 127;   // x = m 2^e, m in [1, 2)
  if ((__float_as_int(x) & 0x7FFFFF) != 0) e += 1;   // x <= 2^e
  return pow2i(max(-126, min(126, -e)));
}

// The unit u of the launch: (token, range) * n_hg + head group (the head
// groups of a token select the same rows and run side by side), its valid
// range [k0, k1) and its blocks.
struct UnitInfo {
  int t, split, h0, k0, k1, nb;
};
__device__ __forceinline__ UnitInfo unit_info(const Fp8Args& a, int u) {
  const FwdParams& p = a.p;
  UnitInfo ui;
  const int hg = u % a.n_hg;
  const int ts = u / a.n_hg;
  ui.split = ts % p.splits;
  ui.t = ts / p.splits;
  ui.h0 = kHeads * hg;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + ui.t), 0), p.topk);
  ui.k0 = ui.split * p.split_len;
  ui.k1 = min(ui.k0 + p.split_len, v);
  // The host plan keeps every range within kMaxBlocks blocks.
  ui.nb = ui.k1 > ui.k0 ? min((ui.k1 - ui.k0 + kBK - 1) / kBK, kMaxBlocks) : 0;
  return ui;
}

// The units of CTA b: the first n_big units in batches of upc consecutive
// units, then one unit per CTA.  The block scheduler starts CTAs in index
// order, so the single units fill in at the end of the launch (a batch of
// units of random size would otherwise set its end), and neighbouring
// tokens, which select overlapping rows, run at the same time.
__device__ __forceinline__ void unit_range(const Fp8Args& a, int& u0, int& u1) {
  const int b = (int)blockIdx.x, nbig = a.n_big / a.upc;
  u0 = b < nbig ? b * a.upc : a.n_big + (b - nbig);
  u1 = min(b < nbig ? u0 + a.upc : u0 + 1, a.n_units);
}

// Q' = the QK B operand of unit ui: rows [0, 16) = hi codes of heads
// h0.., rows [16, 32) = lo codes, K-major, 128-byte chunks of 32 rows,
// 128-byte swizzle; per head its factor 2^-a in buffer qbuf of qf_sh.  One
// warp prepares heads hl0 and hl0 + 1 of the group.  For the 656-byte row the rope part of
// Q stays bf16, in chunk 4 (16 rows x 128 bytes).
template <bool kBf16Rope>
__device__ __forceinline__ void prepare_q_pair(const FwdParams& p, uint8_t* sm,
                                               const UnitInfo& ui, int hl0, int lane,
                                               int qbuf) {
  const bool rope = p.d_qk == 576;
  float* qf_sh = reinterpret_cast<float*>(sm + kOffQf) + kHeads * qbuf;
  const int n_fp8 = rope && !kBf16Rope ? 72 : 64;   // 8-channel pieces split to E4M3
  const int n_pc = rope ? 72 : 64;
  // both heads' loads first (one memory latency for the two)
  uint4 x[2][3];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int hd = ui.h0 + hl0 + hh;
    const bool live = hd < p.h;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int k = lane + 32 * j;
      x[hh][j] = (live && k < n_pc) ? __ldg(q_chunk(p, ui.t, hd, 8 * k))
                                    : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int hl = hl0 + hh;
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int k = lane + 32 * j;
      if (k < n_fp8) {
        const uint32_t w[4] = {x[hh][j].x, x[hh][j].y, x[hh][j].z, x[hh][j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[e] << 16)),
                               fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // x * 2^ea in [128, 256) for the largest |x| (a zero row: ea = 0)
    int ea = 0;
    if (mx > 0.f) ea = 7 - (((__float_as_int(mx) >> 23) & 255) - 127);
    ea = max(-126, min(126, ea));
    const float up = pow2i(ea);
    if (lane == 0) qf_sh[hl] = pow2i(-ea);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int k = lane + 32 * j;
      if (k < n_fp8) {
        const uint32_t w[4] = {x[hh][j].x, x[hh][j].y, x[hh][j].z, x[hh][j].w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = __uint_as_float(w[e] << 16) * up;
          f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * up;
        }
        uint2 hi, lo;
        split8(f, hi, lo);
        const int byte = 8 * k;                         // channel = byte
        const int cc = byte >> 7, u = (byte & 127) >> 4, off = byte & 8;
        uint8_t* chunk = sm + kOffQ + cc * kQChunkBytes;
        *reinterpret_cast<uint2*>(chunk + hl * 128 + (((u ^ (hl & 7)) << 4) | off)) = hi;
        const int nl = 16 + hl;
        *reinterpret_cast<uint2*>(chunk + nl * 128 + (((u ^ (nl & 7)) << 4) | off)) = lo;
      } else if (kBf16Rope && k < n_pc) {
        const int u = k - 64;                           // 16-byte unit of the bf16 row
        *reinterpret_cast<uint4*>(sm + kOffQ + 4 * kQChunkBytes + hl * 128 +
                                  ((u ^ (hl & 7)) << 4)) = x[hh][j];
      }
    }
  }
}

// Each CTA runs its units (unit_range) in order.  Every role walks the same sequence of units and skips the
// empty ones (no block), so that the CTA's running block count g (and the
// running count of non-empty units) name the same barrier phases in every
// role: block g uses stage g & 1 with phase (g >> 1) & 1, and the per-unit
// barriers (Q ready, Q used, last PV done) have one phase per non-empty
// unit.  The pipeline runs across unit boundaries: the producers load the
// next unit's slot ids right after issuing the current unit's last gathers,
// issue its first block's gathers, and then write its Q' once the current
// unit's last QK MMA has read Q' and the softmax warps have read the
// current unit's Q factors, so that the next unit's first QK runs while the
// softmax warps finish the current unit (its last block and epilogue).
template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
smla_tc_fp8_kernel(const __grid_constant__ Fp8Args a) {
  constexpr bool kGroup = kFmt != kE4m3;         // per-(slot, group) scales
  constexpr bool kBf16Rope = kFmt == kDsMla;     // rope stored as bf16 in the row
  constexpr int kTerms = 3;                      // E4M3 terms of a P' weight
  constexpr int kNo = 16 * kTerms;               // PV N
  constexpr uint32_t kColS = 4 * kNo;            // first S column
  extern __shared__ uint8_t smem_raw[];
  const FwdParams& p = a.p;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;           // shared address base
  uint8_t* sm = smem_raw + (sb - raw);                  // generic pointer base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool rope = p.d_qk == 576;
  int u_begin, u_end;
  unit_range(a, u_begin, u_end);

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W = make_waiter(abort_flag, p);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // one expect_tx per producer warp (TMA), one cp.async arrival and one
      // plain arrival (masks and scales stored) per producer thread
      mbar_init(bar(kBarKvFull + s), 4 + 2 * kProducers);
      mbar_init(bar(kBarKvEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), kSoftmax);
    }
    mbar_init(bar(kBarPFull), kSoftmax);
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarOFinal), 1);
    mbar_init(bar(kBarQReady), kProducers);
    mbar_init(bar(kBarQUsed), kSoftmax / 32);
    mbar_init(bar(kBarDrain), 2);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(sb + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kOffTmemSlot);

  if (warp == 0) {
    // ---- QK issuer ------------------------------------------------------
    const uint32_t id_qk = idesc_e4m3(128, kNq, false, false);
    const uint32_t id_rope = idesc_bf16(128, kHeads, false, false);
    const uint32_t qb = sb + kOffQ;
    int g = 0, ku = 0;
    for (int u = u_begin; u < u_end; ++u) {
      const UnitInfo ui = unit_info(a, u);
      if (ui.nb == 0) continue;
      W.wait(bar(kBarQReady), ku & 1);
      tc_fence_after();
      for (int j = 0; j < ui.nb; ++j, ++g) {
        const int s = g & 1;
        if (p.inject_stall && j == 0) continue;   // tests: block 0's scores never arrive
        W.wait(bar(kBarKvFull + s), (g >> 1) & 1);
        if (g >= 2) W.wait(bar(kBarSEmpty + s), ((g >> 1) - 1) & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kStageBytes;
        const uint32_t dS = tmem + kColS + kSBuf * s;
        if (elect_one()) {
          fence_proxy_async_smem();
          // A = 128 key rows, K-major; B = Q' rows, K-major; a step is 32
          // E4M3 channels (32 bytes of a 128-byte swizzled row).  Group c of
          // the ckv accumulates into columns [32 c, 32 c + 32).
          const uint64_t a0 = sdesc(tile, 16, 1024, kLayoutSw128);
          const uint64_t b0 = sdesc(qb, 16, 1024, kLayoutSw128);
#pragma unroll
          for (int ks = 0; ks < 16; ++ks) {
            const uint32_t oa = (uint32_t)((ks >> 2) * kChunkBytes + (ks & 3) * 32);
            const uint32_t ob = (uint32_t)((ks >> 2) * kQChunkBytes + (ks & 3) * 32);
            const uint32_t acc = kGroup ? (uint32_t)(ks >> 2) * kNq : 0u;
            const bool first = kGroup ? (ks & 3) == 0 : ks == 0;
            mma_f8(dS + acc, a0 + (oa >> 4), b0 + (ob >> 4), id_qk, first ? 0u : 1u);
          }
          if (rope) {
            const uint32_t oa = (uint32_t)(4 * kChunkBytes), ob = (uint32_t)(4 * kQChunkBytes);
            if (kBf16Rope) {
              // 64 bf16 rope channels (one 128-byte chunk) x 16 bf16 Q rows
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_ss(dS + 4 * kNq, a0 + ((oa + 32 * ks) >> 4), b0 + ((ob + 32 * ks) >> 4),
                       id_rope, ks > 0 ? 1u : 0u);
            } else {
              // 64 E4M3 rope channels: two steps (the rest of the chunk is
              // not read)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks)
                mma_f8(dS + (kGroup ? 4 * kNq : 0u), a0 + ((oa + 32 * ks) >> 4),
                       b0 + ((ob + 32 * ks) >> 4), id_qk, (kGroup && ks == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(kBarSFull + s));
        }
        __syncwarp();
      }
      ++ku;
    }
    // Every MMA this warp issued has completed (also after an abort) before
    // the TMEM is freed and the tiles are left.
    __syncwarp();
    if (elect_one()) mma_commit(bar(kBarDrain));
    __syncwarp();
    W.drain(bar(kBarDrain), 0);
  } else if (warp == 13) {
    // ---- PV issuer ------------------------------------------------------
    const uint32_t id_pv = idesc_e4m3(128, kNo, true, true);
    const uint32_t pb = sb + kOffP;
    int g = 0;
    for (int u = u_begin; u < u_end; ++u) {
      const UnitInfo ui = unit_info(a, u);
      for (int j = 0; j < ui.nb; ++j, ++g) {
        const int s = g & 1;
        W.wait(bar(kBarPFull), g & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kStageBytes;
        if (elect_one()) {
          fence_proxy_async_smem();
          // A = V^T of channel block c: chunk c (128 channels) x 32 keys,
          // MN-major; B = P'^T: 32 keys x kNo, MN-major (group scales: group
          // c's 48 bytes of each key's row, bytes 48 (c & 1) of region
          // c >> 1).  The unit's first block overwrites O (the softmax warps
          // read the previous unit's O before they handed over this P').
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int ks = 0; ks < kBK / 32; ++ks) {
              const uint64_t ad =
                  sdesc(tile + c * kChunkBytes + ks * 4096, kChunkBytes, 1024, kLayoutSw128);
              const uint32_t pc = kGroup ? (uint32_t)((c >> 1) * kPBytes + 48 * (c & 1)) : 0u;
              const uint64_t bd = sdesc(pb + pc + ks * 4096, kPBytes, 1024, kLayoutSw128);
              mma_f8(tmem + kColO + (uint32_t)(kNo * c), ad, bd, id_pv,
                     (j > 0 || ks > 0) ? 1u : 0u);
            }
          }
          mma_commit(bar(kBarODone));
          mma_commit(bar(kBarPEmpty));
          mma_commit(bar(kBarKvEmpty + s));
          if (j == ui.nb - 1) mma_commit(bar(kBarOFinal));
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (elect_one()) mma_commit(bar(kBarDrain));
    __syncwarp();
    W.drain(bar(kBarDrain), 0);
  } else if (warp <= 4) {
    // ---- producers: slot ids, then a2 gather of raw rows ------------------
    // Per unit the four warps read its index range into shared memory
    // (masked: past k1, < 0, >= num_slots); only they read it.  Per block,
    // warp wl fills tile rows [32 wl, 32 wl + 32): the four 128-byte ckv
    // chunks by TMA tile::gather4 (8 groups of 4 rows; a masked position,
    // slot id -1, reads the out-of-bounds zero fill), the rope by 16-byte
    // cp.async (zero-filled for masked rows), and the row's valid bit and
    // group scales into the stage.  (Measured on the mixed FP8 batch: the
    // four ckv chunks by TMA and the 64-byte rope by cp.async 3.06 ms; the
    // rope as a 128-byte TMA box too, 64 bytes of it fill, 3.26 ms; moving
    // ckv chunks to cp.async 3.27 ms (one), 3.62 (two), 3.81 (all four).)
    const int wl = warp - 1;
    const int pt = tid - 32;
    constexpr int kRopePieces = kBf16Rope ? 8 : 4;
    const int row_bytes = kFmt == kDsMla ? kDsMlaRowBytes : p.d_qk;
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
    int* slots = reinterpret_cast<int*>(sm + kOffSlot);
    float* scs = reinterpret_cast<float*>(sm + kOffSc);
    uint32_t* masks = reinterpret_cast<uint32_t*>(sm + kOffMask);
    const uint32_t tx_bytes = (uint32_t)(8 * 4 * 512);
    int g = 0, issued = 0, ku = 0;
    bool stop = false;
    for (int u = u_begin; u < u_end && !stop; ++u, ++ku) {
      const UnitInfo ui = unit_info(a, u);
      if (ui.nb == 0) {
        --ku;
        continue;
      }
      // (the previous unit's gathers are all issued: the ids are free)
      named_bar_sync(1, kProducers);
      if (load_unit_slots(p, ui.t, ui.k0, ui.k1, ui.nb * kBK, slots, pt, kProducers))
        atomicCAS(p.status, 0, kStatusBadIndex);
      named_bar_sync(1, kProducers);
      for (int j = 0; j < ui.nb; ++j, ++g) {
        const int s = g & 1;
        if (g >= kStages) W.wait(bar(kBarKvEmpty + s), ((g >> 1) - 1) & 1);
        if (*abort_flag) {                       // the stage may still be in use
          stop = true;
          break;
        }
        __syncwarp();
        issued = g + 1;
        const uint32_t full = bar(kBarKvFull + s);
        const uint32_t tile = sb + kOffTile + s * kStageBytes;
        const int* bs = slots + j * kBK + 32 * wl;
        if (elect_one()) mbar_arrive_expect_tx(full, tx_bytes);
        __syncwarp();
        if (elect_one()) {
          for (int q = 0; q < 8; ++q) {
            const int4 y = *reinterpret_cast<const int4*>(bs + 4 * q);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_gather4(tile + c * kChunkBytes + (32 * wl + 4 * q) * 128, &a.kv_map, 128 * c,
                          y.x, y.y, y.z, y.w, full);
          }
        }
        __syncwarp();
        if (rope) {
#pragma unroll
          for (int i = 0; i < kRopePieces; ++i) {
            const int e = lane + 32 * i;
            const int r = e / kRopePieces, k = e % kRopePieces;   // row of the warp, rope piece
            const int id = bs[r];
            const int row = 32 * wl + r;
            const uint32_t dst = tile + (uint32_t)(4 * kChunkBytes + row * 128) +
                                 ((uint32_t)(k ^ (row & 7)) << 4);
            cp_async16(dst, kv8 + (size_t)(id < 0 ? 0 : id) * row_bytes + a.rope_x + 16 * k,
                       id < 0 ? 0u : 16u);
          }
        }
        cp_async_arrive_noinc(full);
        if (j == 0 && ku > 0) {
          // Q' of this unit, once the softmax warps have read the previous
          // unit's factors and its last QK (block g - 1) has read Q'
          W.wait(bar(kBarQUsed), (ku - 1) & 1);
          W.wait(bar(kBarSFull + ((g - 1) & 1)), ((g - 1) >> 1) & 1);
          tc_fence_after();
          prepare_q_pair<kBf16Rope>(p, sm, ui, 4 * wl, lane, ku & 1);
          prepare_q_pair<kBf16Rope>(p, sm, ui, 4 * wl + 2, lane, ku & 1);
          fence_proxy_async_smem();
          mbar_arrive(bar(kBarQReady));
        }
        // This thread's row: its valid bit and (group formats) its scales.
        const int id = bs[lane];
        const uint32_t m = __ballot_sync(0xffffffffu, id >= 0);
        if (lane == 0) masks[s * 4 + wl] = m;
        if (kGroup) {
          float sc[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
          if (id >= 0) {
            if (kFmt == kDsMla) {
              const float4 s4 = __ldg(reinterpret_cast<const float4*>(
                  kv8 + (size_t)id * kDsMlaRowBytes + kDsMlaScaleOff));
              sc[0] = s4.x; sc[1] = s4.y; sc[2] = s4.z; sc[3] = s4.w; sc[4] = 1.f;
            } else if (kFmt == kE4m3Group4Kpe) {
              const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.k_scale + (int64_t)id * 4));
              sc[0] = s4.x; sc[1] = s4.y; sc[2] = s4.z; sc[3] = s4.w; sc[4] = p.kpe_scale;
            } else {
              const float* r = p.k_scale + (int64_t)id * a.G;
              sc[0] = __ldg(r); sc[1] = __ldg(r + 1); sc[2] = __ldg(r + 2); sc[3] = __ldg(r + 3);
              if (a.G > 4) sc[4] = __ldg(r + 4);
            }
          }
          float* dstf = scs + (s * kBK + pt) * kScaleRow;
#pragma unroll
          for (int q = 0; q < 5; ++q) dstf[q] = sc[q];
        }
        mbar_arrive(full);
      }
    }
    // Teardown: this thread's copies have landed; the gathers of the last
    // block issued into each stage too (earlier ones were consumed before the
    // stage was reissued).
    cp_async_wait_all();
    if (lane == 0) {
      for (int b = issued - 1; b >= 0 && b >= issued - kStages; --b)
        W.drain(bar(kBarKvFull + (b & 1)), (b >> 1) & 1);
    }
    __syncwarp();
  } else {
    // ---- softmax warpgroups (thread <-> key <-> TMEM lane) -----------------
    const int sw = warp - 5;                            // 0..7
    const int wg = sw >> 2;                             // heads [8 wg, 8 wg + 8)
    const int q4 = warp & 3;                            // TMEM lane quarter
    const int key = 32 * q4 + lane;                     // tile row == TMEM lane
    const int st = tid - 160;                           // 0..255
    const uint32_t lane_base = ((uint32_t)q4 * 32u) << 16;
    const int nbar_wg = 3 + wg;                         // warpgroup-local barrier
    float* qf_sh = reinterpret_cast<float*>(sm + kOffQf);
    const float* scs = reinterpret_cast<const float*>(sm + kOffSc);
    const uint32_t* masks = reinterpret_cast<const uint32_t*>(sm + kOffMask);
    float* red = reinterpret_cast<float*>(sm + kOffRed) + wg * 32;      // [4 warps][8]
    float* red_sc = reinterpret_cast<float*>(sm + kOffRedSc) + wg * 16; // [4 warps][4]
    float* fac_sh = reinterpret_cast<float*>(sm + kOffFac) + wg * 12;   // the O rescale factors
    // This key's 128-byte row of each P' region (MN-major, 128-byte swizzle).
    const uint32_t p_row = (uint32_t)(key >> 3) * 1024u + (uint32_t)(key & 7) * 128u;
    const uint32_t p_sw = (uint32_t)(key & 7);
    const float kscale = kFmt == kE4m3 ? __ldg(p.k_scale) : 1.f;
    const float rope_cs = a.scale_log2;                 // bf16 rope: not scaled by 2^-a

    // The next unit of this CTA with at least one block (u_end: none).
    auto next_unit = [&](int u) {
      for (++u; u < u_end; ++u)
        if (unit_info(a, u).nb > 0) break;
      return u;
    };
    // Its q rows into L2 (144 lines of 128 bytes for 16 heads of 576 channels).
    auto prefetch_q = [&](int u) {
      if (u >= u_end) return;
      const UnitInfo ui = unit_info(a, u);
      for (int i = st; i < kHeads * 9; i += kSoftmax) {
        const int hd = ui.h0 + i / 9, line = i % 9;
        if (hd < p.h && 64 * line < p.d_qk) prefetch_l2(q_chunk(p, ui.t, hd, 64 * line));
      }
    };
    auto write_empty = [&](const UnitInfo& ui) {
      // O = 0 and LSE = -inf for the unit's heads (channel `key` of each
      // 128-channel block; thread key < 8 the LSE of head 8 wg + key).
#pragma unroll 1
      for (int i = 0; i < 8; ++i) {
        const int hd = ui.h0 + 8 * wg + i;
        if (hd >= p.h) break;
        const int64_t orow = (int64_t)ui.t * p.h + hd;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = 128 * c + key;
          if (p.fp32_out)
            p.o_part[((int64_t)ui.split * p.T * p.h + orow) * p.d_v + ch] = 0.f;
          else
            reinterpret_cast<__nv_bfloat16*>(p.out)[orow * p.d_v + ch] = __float2bfloat16_rn(0.f);
        }
      }
      if (key < 8 && ui.h0 + 8 * wg + key < p.h) {
        const int64_t orow = (int64_t)ui.t * p.h + ui.h0 + 8 * wg + key;
        if (p.fp32_out)
          p.lse_part[(int64_t)ui.split * p.T * p.h + orow] = -INFINITY;
        else if (p.lse)
          p.lse[orow] = -INFINITY;
      }
    };

    int g = 0, ku = 0;
    int u = u_begin;
    while (u < u_end && unit_info(a, u).nb == 0) {   // leading empty units
      write_empty(unit_info(a, u));
      ++u;
    }
    if (u < u_end) {
      // the first unit's Q' (the producer warps write the later ones)
      prepare_q_pair<kBf16Rope>(p, sm, unit_info(a, u), 2 * sw, lane, 0);
      fence_proxy_async_smem();
      named_bar_sync(5, kSoftmax);
      if (st < kProducers) mbar_arrive(bar(kBarQReady));
    }
    while (u < u_end) {
      const UnitInfo ui = unit_info(a, u);
      const int un = next_unit(u);
      prefetch_q(un);
      W.wait(bar(kBarQReady), ku & 1);                  // qf_sh of this unit written
      // Per head of this warpgroup: Q factor 2^-a (buffer ku & 1 of qf_sh,
      // read where used), folded with the score scale (and the per-tensor
      // E4M3 scale); heads i < n_live carry data.
      const float* qf_u = qf_sh + kHeads * (ku & 1) + 8 * wg;
      const float csc = a.scale_log2 * kscale;
      const int n_live = p.h - ui.h0 - 8 * wg;
      __syncwarp();
      // (the producers write the other buffer next, then this one again
      // once this warp has started the next unit)
      if (lane == 0) mbar_arrive(bar(kBarQUsed));
      float m_run[8], l_part[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) { m_run[i] = -INFINITY; l_part[i] = 0.f; }
      float R[4] = {0.f, 0.f, 0.f, 0.f};                // PV group factors (0: not set)

      for (int j = 0; j < ui.nb; ++j, ++g) {
        const int s = g & 1;
        // the block's valid bits and scales (stage s), then its scores
        W.wait(bar(kBarKvFull + s), (g >> 1) & 1);
        float sc[5];
#pragma unroll
        for (int q = 0; q < 5; ++q) sc[q] = kGroup ? scs[(s * kBK + key) * kScaleRow + q] : 0.f;
        const bool key_ok = ((masks[s * 4 + (key >> 5)] >> (key & 31)) & 1u) != 0u;
        W.wait(bar(kBarSFull + s), (g >> 1) & 1);
        __syncwarp();
        tc_fence_after();
        // a4 result: per group, this warpgroup's 8 heads hi (columns 8 wg..)
        // and lo (16 + 8 wg..).
        float sp[8];
        {
          const uint32_t c0 = tmem + lane_base + kColS + kSBuf * s + 8u * (uint32_t)wg;
          if (kGroup) {
            // two batches of TMEM loads (register budget): groups 0, 1, then
            // groups 2, 3 and the rope
            float acc[8];
            {
              uint32_t w[2][2][8];
#pragma unroll
              for (int gg = 0; gg < 2; ++gg) {
                tmem_ld8(c0 + kNq * gg, w[gg][0]);
                tmem_ld8(c0 + kNq * gg + 16, w[gg][1]);
              }
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                acc[i] = sc[0] * fmaf(__uint_as_float(w[0][1][i]), 0.0625f, __uint_as_float(w[0][0][i]));
                acc[i] = fmaf(sc[1], fmaf(__uint_as_float(w[1][1][i]), 0.0625f,
                                          __uint_as_float(w[1][0][i])), acc[i]);
              }
            }
            {
              uint32_t w[3][2][8];
#pragma unroll
              for (int gg = 0; gg < 2; ++gg) {
                tmem_ld8(c0 + kNq * (gg + 2), w[gg][0]);
                tmem_ld8(c0 + kNq * (gg + 2) + 16, w[gg][1]);
              }
              if (rope) {
                tmem_ld8(c0 + kNq * 4, w[2][0]);
                if (!kBf16Rope) tmem_ld8(c0 + kNq * 4 + 16, w[2][1]);
              }
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int gg = 0; gg < 2; ++gg)
                  acc[i] = fmaf(sc[gg + 2], fmaf(__uint_as_float(w[gg][1][i]), 0.0625f,
                                                 __uint_as_float(w[gg][0][i])), acc[i]);
                float r = 0.f;
                if (rope && !kBf16Rope)
                  acc[i] = fmaf(sc[4], fmaf(__uint_as_float(w[2][1][i]), 0.0625f,
                                            __uint_as_float(w[2][0][i])), acc[i]);
                if (rope && kBf16Rope) r = __uint_as_float(w[2][0][i]);
                sp[i] = fmaf(acc[i], qf_u[i] * csc, r * rope_cs);
              }
            }
          } else {
            uint32_t w0[8], w1[8];
            tmem_ld8(c0, w0);
            tmem_ld8(c0 + 16, w1);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              sp[i] = fmaf(__uint_as_float(w1[i]), 0.0625f, __uint_as_float(w0[i])) *
                      (qf_u[i] * csc);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(kBarSEmpty + s));

        // a5: masked scores (log2 units) and the lazy running max; with group
        // scales also the lazy PV group factors R (scale * R <= 1).
        bool need = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          sp[i] = (key_ok && i < n_live) ? sp[i] : -INFINITY;
          need |= sp[i] > m_run[i] + kT;
        }
        if (kGroup) {
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) need |= R[gg] == 0.f || sc[gg] * R[gg] > 1.f;
        }
        float alpha[8], ratio[4] = {1.f, 1.f, 1.f, 1.f};
        bool rescale = false;                       // some factor of O is not 1
#pragma unroll
        for (int i = 0; i < 8; ++i) alpha[i] = 1.f;
        const bool voted = named_bar_or(2, kSoftmax, need);
        if (voted) {
          float bm[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) bm[i] = sp[i];
          const float wmax = xreduce8<true>(bm, lane);
          if ((lane & 17) == 0) red[q4 * 8 + ((lane >> 1) & 7)] = wmax;
          if (kGroup) {
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
              float x = sc[gg];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
              if (lane == 0) red_sc[q4 * 4 + gg] = x;
            }
          }
          named_bar_sync(nbar_wg, 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float bmax = fmaxf(fmaxf(red[i], red[8 + i]), fmaxf(red[16 + i], red[24 + i]));
            if (bmax > m_run[i] + kT) {             // also true for the first finite max
              alpha[i] = ex2_approx(m_run[i] - bmax);   // 0 when m_run = -inf
              m_run[i] = bmax;
            }
          }
          if (kGroup) {
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
              const float ms = fmaxf(fmaxf(red_sc[gg], red_sc[4 + gg]),
                                     fmaxf(red_sc[8 + gg], red_sc[12 + gg]));
              if (ms > 0.f && (R[gg] == 0.f || ms * R[gg] > 1.f)) {
                const float rn = pow2_at_most_inv(ms);
                if (R[gg] != 0.f)                   // powers of two: exact
                  ratio[gg] = rn * __uint_as_float(0x7F000000u - (__float_as_uint(R[gg]) & 0x7F800000u));
                R[gg] = rn;
              }
            }
          }
          // The warpgroup's O rescale factors (the same in all its threads)
          // go to shared memory for the rescale below, so that they need not
          // stay in registers; the barrier of the next block's vote orders
          // their next write after every read.
#pragma unroll
          for (int i = 0; i < 8; ++i) rescale |= alpha[i] != 1.f;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) rescale |= ratio[gg] != 1.f;
          if ((st & 127) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) fac_sh[i] = alpha[i];
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) fac_sh[8 + gg] = ratio[gg];
          }
          named_bar_sync(nbar_wg, 128);             // red may be rewritten
        }
        float pe[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pe[i] = m_run[i] == -INFINITY ? 0.f : ex2_approx(sp[i] - m_run[i]);
          l_part[i] = fmaf(l_part[i], alpha[i], pe[i]);
        }
        if (rescale && j >= 1) {                        // uniform in the warpgroup
          // O^T row (channel `key` of each 128-channel block): this
          // warpgroup's head columns (each term) *= alpha * ratio of the
          // block.  (Rare: a lazy max step or a new group factor.)
          W.wait(bar(kBarODone), (g - 1) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float fc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) fc[i] = fac_sh[i] * fac_sh[8 + c];
#pragma unroll 1
            for (int part = 0; part < kTerms; ++part) {
              const uint32_t col =
                  tmem + lane_base + kColO + (uint32_t)(kNo * c) + 16u * part + 8u * wg;
              uint32_t w[8];
              tmem_ld8(col, w);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * fc[i]);
              tmem_st8(col, w);
            }
          }
          tmem_wait_st();
        }
        // a6 operand: P' codes, hi / mid / lo of group gg in region gg >> 1,
        // 16-byte units 3 (gg & 1) + 0, 1, 2 (one scale per tensor: one
        // group, region 0).
        if (g >= 1) W.wait(bar(kBarPEmpty), (g - 1) & 1);   // PV(g-1) read it
        if (kGroup && j == 0 && ku > 0 && !p.fp32_out) {
          // the previous unit's O copy has read the staging rows in region 1
          if (st == 0) bulk_wait_read_all();
          named_bar_sync(5, kSoftmax);
        }
#pragma unroll
        for (int gg = 0; gg < (kGroup ? 4 : 1); ++gg) {
          uint8_t* prow = sm + kOffP + (uint32_t)(gg >> 1) * kPBytes + p_row;
          split_store8<kTerms>(pe, kGroup ? sc[gg] * R[gg] * kPShift : kPShift, [&](int k) {
            return reinterpret_cast<uint2*>(
                prow + ((((uint32_t)(kTerms * (gg & 1) + k) ^ p_sw) << 4) | (8u * wg)));
          });
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull));
      }

      // ---- a7: epilogue -------------------------------------------------------
      // Row sums: reduce the per-key partial sums over the block's keys.
      float l_tot[8];
      {
        float l8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) l8[i] = l_part[i];
        const float ws = xreduce8<false>(l8, lane);
        named_bar_sync(nbar_wg, 128);
        if ((lane & 17) == 0) red[q4 * 8 + ((lane >> 1) & 7)] = ws;
        named_bar_sync(nbar_wg, 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) l_tot[i] = (red[i] + red[8 + i]) + (red[16 + i] + red[24 + i]);
      }
      // Thread `key` < 8 writes the LSE of head 8 wg + key.
      if (key < 8 && ui.h0 + 8 * wg + key < p.h) {
        float mi = m_run[0], li = l_tot[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
          mi = key == i ? m_run[i] : mi;
          li = key == i ? l_tot[i] : li;
        }
        const bool empty = li == 0.f;         // (a NaN row sum is not empty)
        const float lse_v = empty ? -INFINITY : (mi + log2f(li)) * 0.69314718055994530942f;
        const int64_t orow = (int64_t)ui.t * p.h + ui.h0 + 8 * wg + key;
        if (p.fp32_out)
          p.lse_part[(int64_t)ui.split * p.T * p.h + orow] = lse_v;
        else if (p.lse)
          p.lse[orow] = lse_v;
      }
      W.wait(bar(kBarOFinal), ku & 1);
      __syncwarp();
      tc_fence_after();
      const float oscale = kFmt == kE4m3 ? kscale : 1.f;
      float inv[8];
#pragma unroll
      uint32_t live_l = 0u;                             // bit i: head i has a row sum
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // (fast division: the IEEE one costs ~125 cycles each here)
        inv[i] = l_tot[i] != 0.f ? __fdividef(oscale, l_tot[i] * kPShift) : 0.f;
        live_l |= l_tot[i] != 0.f ? 1u << i : 0u;
      }
      // bf16 O goes through the staging rows [16 heads][512] and leaves as
      // one bulk copy (the token's rows of these heads are contiguous).  The
      // rows are P' region 1: the unit's last PV has read it (O final); with
      // group scales the previous unit's copy was waited for before this
      // unit's first P' was written, with one scale per tensor P' does not
      // use the region and the wait is here.  fp32 partials are stored
      // directly.
      __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + kOffOst);
      if (!kGroup && !p.fp32_out) {
        if (st == 0) bulk_wait_read_all();
        named_bar_sync(5, kSoftmax);
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t wh[8], wm[8], wl8[8];
        __syncwarp();
        const uint32_t col = tmem + lane_base + kColO + (uint32_t)(kNo * c) + 8u * wg;
        tmem_ld8(col, wh);
        tmem_ld8(col + 16, wm);
        tmem_ld8(col + 32, wl8);
        tmem_wait_ld();
        const float rc = kGroup ? R[c] : 1.f;
        // 1 / R_c: R_c is a power of two (or 0: no key of the unit has a
        // nonzero scale in this group), so the reciprocal is exact from the
        // exponent field
        const float rinv =
            rc > 0.f ? __uint_as_float(0x7F000000u - (__float_as_uint(rc) & 0x7F800000u)) : 0.f;
        const int ch = 128 * c + key;                   // output channel of lane `key`
        float ov[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // (no valid key for the head, or none with a nonzero scale in this
          // group: 0 exactly)
          ov[i] = (((live_l >> i) & 1u) != 0u && rinv > 0.f)
                      ? fmaf(__uint_as_float(wl8[i]), 0.00390625f,
                             fmaf(__uint_as_float(wm[i]), 0.0625f, __uint_as_float(wh[i]))) *
                            (inv[i] * rinv)
                      : 0.f;
        }
        if (!p.fp32_out) {
          // lanes 2m and 2m + 1 hold channels ch, ch + 1: the even lane stores
          // heads 0..3 of both, the odd lane heads 4..7, as bf16 pairs
          const bool odd = (lane & 1) != 0;
          const int ch0 = ch & ~1;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float send = odd ? ov[i] : ov[i + 4];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const int hd = odd ? i + 4 : i;
            const float lo = odd ? recv : ov[i];          // channel ch0
            const float hi = odd ? ov[i + 4] : recv;      // channel ch0 + 1
            *reinterpret_cast<__nv_bfloat162*>(ost + (8 * wg + hd) * 512 + ch0) =
                __floats2bfloat162_rn(lo, hi);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < n_live) {
              const int64_t orow = (int64_t)ui.t * p.h + ui.h0 + 8 * wg + i;
              p.o_part[((int64_t)ui.split * p.T * p.h + orow) * p.d_v + ch] = ov[i];
            }
        }
      }
      // (the TMEM loads of O are complete: the next unit's first PV, which
      // waits for this thread's next P' hand-off, may overwrite it)
      tc_fence_before();
      if (!p.fp32_out) {
        fence_proxy_async_smem();
        named_bar_sync(5, kSoftmax);
        if (st == 0) {
          const int nh = min(kHeads, p.h - ui.h0);
          bulk_store(reinterpret_cast<__nv_bfloat16*>(p.out) + ((int64_t)ui.t * p.h + ui.h0) * 512,
                     sb + kOffOst, (uint32_t)(nh * 1024));
          bulk_commit_group();
        }
      }
      ++ku;
      // the empty units up to the next one with blocks
      for (++u; u < un; ++u) write_empty(unit_info(a, u));
    }
  }

  // ---- teardown -------------------------------------------------------------
  if (tid == 160) bulk_wait_all();                // the O copies have been written
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The cache as a 2-D byte tensor [num_slots, row bytes] with 128-byte x
// 1-row boxes and the 128-byte swizzle of the MMA operand tiles.
cudaError_t encode_byte_rows_map(CUtensorMap* map, const void* kv, int row_bytes,
                                 int64_t num_slots) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)num_slots};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <int kFmt>
cudaError_t launch_fmt(const Fp8Args& a, unsigned blocks, cudaStream_t stream) {
  auto kernel = smla_tc_fp8_kernel<kFmt>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<blocks, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_fp8_max_range() { return kMaxBlocks * kBK; }

bool tc_fp8_supported(int h, int d_qk, int kv_format) {
  if (h < 1 || h > 128 || (d_qk != 576 && d_qk != 512)) return false;
  if (kv_format == kDsMla || kv_format == kE4m3Group4Kpe) return d_qk == 576;
  return kv_format == kE4m3 || kv_format == kE4m3Group;
}

cudaError_t launch_tc_fp8(const FwdParams& p, cudaStream_t stream) {
  Fp8Args a{};
  a.p = p;
  const int row_bytes = p.kv_format == kDsMla ? kDsMlaRowBytes : p.d_qk;
  const cudaError_t e = encode_byte_rows_map(&a.kv_map, p.kv, row_bytes, p.num_slots);
  if (e != cudaSuccess) return e;
  a.n_hg = (p.h + kHeads - 1) / kHeads;
  a.rope_x = p.kv_format == kDsMla ? kDsMlaRopeOff : 512;
  a.G = (p.d_qk + 127) / 128;
  a.scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t units = (int64_t)p.T * p.splits * a.n_hg;
  if (units > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  a.n_units = (int)units;
  // Batches of up to 4 consecutive units per CTA (one CTA per SM at a time:
  // the shared memory allows no second), then about two waves of single
  // units at the end.  Mixed FP8 batch: 2.51 ms (batches of up to 4), 2.59
  // (8), 2.75 (16); one CTA per SM running every 152nd unit 2.78.
  const int64_t sms = p.num_sms > 0 ? p.num_sms : 1;
  const int64_t tail = 2 * sms;
  int64_t upc = units > tail ? (units - tail) / (4 * sms) : 1;
  upc = upc < 1 ? 1 : (upc > 4 ? 4 : upc);
  const int64_t n_big = units > tail ? (units - tail) / upc * upc : 0;
  a.upc = (int)upc;
  a.n_big = (int)n_big;
  const int64_t blocks = n_big / upc + (units - n_big);
  switch (p.kv_format) {
    case kE4m3: return launch_fmt<kE4m3>(a, (unsigned)blocks, stream);
    case kE4m3Group: return launch_fmt<kE4m3Group>(a, (unsigned)blocks, stream);
    case kDsMla: return launch_fmt<kDsMla>(a, (unsigned)blocks, stream);
    default: return launch_fmt<kE4m3Group4Kpe>(a, (unsigned)blocks, stream);
  }
}

}  // namespace smla

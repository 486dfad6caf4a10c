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
// them as E4M3 operands.  The other operand of each product is split into an
// E4M3 pair that carries bf16 precision:
//   * Q (bf16): per head, x = q * 2^a with a power of two a that puts
//     max|x| in [128, 256); hi = E4M3(x), lo = E4M3(16 (x - hi)), so that
//     x = hi + lo / 16 up to 2^-8 of |x| (at least 2^-14 absolute).  The
//     two are the MMA's N rows [16 heads hi | 16 heads lo]; the score is
//     2^-a (S_hi + S_lo / 16), summed in fp32.
//   * P (fp32, in [0, 2^4] by the lazy running max below): with group
//     scales, each V group g gets x = p * scale_g * R_g * 2^4, R_g a power
//     of two that keeps scale_g * R_g <= 1, split the same way into hi and
//     lo * 16 columns of the PV operand; O = (O_hi + O_lo / 16) / (16 R_g l).
// Keys are the MMA's M dimension (keys-major), heads its N:
//   S^T[keys, 32] = K[keys, d] . Q'^T[d, 32]      A = gathered tile, K-major
//   O^T[ch, 32]  += V^T[ch, keys] . P'^T[keys, 32] A = the same tile, MN-major
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
// issues the PV MMAs; warps 1..4 load the unit's slot ids, then issue the
// gathers (each 32 tile rows); warps 5..12 are two softmax warpgroups
// (thread <-> key <-> TMEM lane; warpgroup w owns heads [8w, 8w + 8)), which
// also build Q' and write O and LSE.
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
constexpr int kPBytes = kBK * 128;         // P': one 128-byte row per key
constexpr int kThreads = 448;
constexpr int kProducers = 128;            // warps 1..4
constexpr int kSoftmax = 256;              // warps 5..12
constexpr int kMaxBlocks = 16;             // ranges up to 2048 positions
// ckv chunks gathered by TMA (the rest and the rope by cp.async).  Mixed FP8
// batch: 4 -> 3.06 ms, 3 -> 3.27, 2 -> 3.62, 0 -> 3.81; the rope box by TMA
// as well (128 bytes of which 64 are real for E4M3 rows) 3.26 ms.
constexpr int kTmaChunks = 4;
constexpr float kT = 4.f;                  // lazy max threshold (log2 units)
constexpr float kPShift = 16.f;            // 2^(8 - kT): P' <= 2^8

// TMEM columns.
constexpr uint32_t kColO = 0;              // O^T: 4 blocks of 128 channels x 32
constexpr uint32_t kColS = 128;            // S: 2 buffers x 5 accumulators x 32
constexpr uint32_t kSBuf = 5 * kNq;
constexpr uint32_t kTmemCols = 512;
static_assert(kColS + 2 * kSBuf <= kTmemCols, "TMEM budget");

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffQ = kOffTile + kStages * kStageBytes;       // Q' chunks
constexpr uint32_t kOffP = kOffQ + kMaxChunks * kQChunkBytes;      // P' [2]
constexpr uint32_t kOffSlot = kOffP + 2 * kPBytes;                 // [blocks*128] i32
constexpr uint32_t kOffMask = kOffSlot + kMaxBlocks * kBK * 4;     // [blocks][4] u32
constexpr uint32_t kOffRed = kOffMask + kMaxBlocks * 16;           // [2 wg][4 warps][8] f32
constexpr uint32_t kOffRedSc = kOffRed + 2 * 4 * 8 * 4;            // [2 wg][4 warps][4] f32
constexpr uint32_t kOffQf = kOffRedSc + 2 * 4 * 4 * 4;             // [16] f32: 2^-a per head
constexpr uint32_t kOffBar = kOffQf + kHeads * 4;
enum {
  kBarKvFull = 0,                   // [2]
  kBarKvEmpty = kBarKvFull + 2,     // [2]
  kBarSFull = kBarKvEmpty + 2,      // [2]
  kBarSEmpty = kBarSFull + 2,       // [2]
  kBarPFull = kBarSEmpty + 2,       // [2]
  kBarPEmpty = kBarPFull + 2,       // [2]
  kBarODone = kBarPEmpty + 2,
  kBarOFinal,                       // one phase: the unit's last PV is done
  kBarQReady,
  kBarDrain,                        // teardown: both MMA warps' MMAs are done
  kNumBars
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled operands need 1024-B alignment");
static_assert(kOffRed % 16 == 0 && kOffBar % 8 == 0, "alignment");

struct Fp8Args {
  CUtensorMap kv_map;  // the cache as bytes [num_slots, row bytes], 128-byte boxes
  FwdParams p;
  int n_hg;            // head groups of 16 (CTAs per token and range)
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

// Two floats -> two E4M3 codes (round to nearest even, saturating), a in the
// low byte; and two E4M3 codes back to floats (exact).
__device__ __forceinline__ uint32_t e4m3x2_of(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 f2_of_e4m3x2(uint32_t v) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&r));
}
// Split x0..x7 into hi = E4M3(x) and lo = E4M3(16 (x - hi)), eight codes
// each (x0 in the lowest byte).
__device__ __forceinline__ void split8(const float (&x)[8], uint2& hi, uint2& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = e4m3x2_of(x[2 * k], x[2 * k + 1]);
    const float2 f = f2_of_e4m3x2(h[k]);
    l[k] = e4m3x2_of((x[2 * k] - f.x) * 16.f, (x[2 * k + 1] - f.y) * 16.f);
  }
  hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
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

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
smla_tc_fp8_kernel(const __grid_constant__ Fp8Args a) {
  constexpr bool kGroup = kFmt != kE4m3;         // per-(slot, group) scales
  constexpr bool kBf16Rope = kFmt == kDsMla;     // rope stored as bf16 in the row
  extern __shared__ uint8_t smem_raw[];
  const FwdParams& p = a.p;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;           // shared address base
  uint8_t* sm = smem_raw + (sb - raw);                  // generic pointer base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- a1: work unit ------------------------------------------------------
  // unit = (token, range) * n_hg + head group: the head groups of a token
  // select the same rows and run side by side.
  int unit = (int)blockIdx.x;
  const int hg = unit % a.n_hg;
  unit /= a.n_hg;
  const int split = unit % p.splits;
  const int t = unit / p.splits;
  const int h0 = kHeads * hg;                           // first head of the CTA
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);
  // The host plan keeps every range within kMaxBlocks blocks.
  const int nb = k1 > k0 ? min((k1 - k0 + kBK - 1) / kBK, kMaxBlocks) : 0;
  const bool rope = p.d_qk == 576;

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W = make_waiter(abort_flag, p);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // one expect_tx per producer warp (TMA part) + one cp.async arrival per
      // producer thread
      mbar_init(bar(kBarKvFull + s), (kTmaChunks > 0 ? 4 : 0) + kProducers);
      mbar_init(bar(kBarKvEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), kSoftmax);
      mbar_init(bar(kBarPFull + s), kSoftmax);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarOFinal), 1);
    mbar_init(bar(kBarQReady), kSoftmax);
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

  // a1/a2 setup: the producers read the unit's index range once into shared
  // memory (masked: past k1, < 0, >= num_slots), then one valid-bit word per
  // 32 keys of each block.
  int* slots = reinterpret_cast<int*>(sm + kOffSlot);
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + kOffMask);
  if (warp >= 1 && warp <= 4) {
    const int pt = tid - 32;
    if (load_unit_slots(p, t, k0, k1, nb * kBK, slots, pt, kProducers))
      atomicCAS(p.status, 0, kStatusBadIndex);
    named_bar_sync(1, kProducers);
    const int wl = warp - 1;
    for (int b = 0; b < nb; ++b) {
      const uint32_t m = __ballot_sync(0xffffffffu, slots[b * kBK + 32 * wl + lane] >= 0);
      if (lane == 0) masks[b * 4 + wl] = m;
    }
  }
  __syncthreads();

  if (warp == 0 || warp == 13) {
    // ---- MMA issuers: warp 0 issues QK, warp 13 issues PV ----------------
    if (nb > 0) {
      if (warp == 0) {
        const uint32_t id_qk = idesc_e4m3(128, kNq, false, false);
        const uint32_t id_rope = idesc_bf16(128, kHeads, false, false);
        W.wait(bar(kBarQReady), 0);
        tc_fence_after();
        const uint32_t qb = sb + kOffQ;
        for (int j = 0; j < nb; ++j) {
          const int s = j & 1;
          if (p.inject_stall && j == 0) continue;   // tests: block 0's scores never arrive
          W.wait(bar(kBarKvFull + s), (j >> 1) & 1);
          if (j >= 2) W.wait(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1);
          __syncwarp();
          tc_fence_after();
          const uint32_t tile = sb + kOffTile + s * kStageBytes;
          const uint32_t dS = tmem + kColS + kSBuf * s;
          if (elect_one()) {
            // A = 128 key rows, K-major; B = Q' rows, K-major; a step is 32
            // E4M3 channels (32 bytes of a 128-byte swizzled row).  Group c
            // of the ckv accumulates into columns [32 c, 32 c + 32).
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
                // 64 E4M3 rope channels: two steps (the chunk's other 64
                // bytes are the zero fill past the row)
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
      } else {
        const uint32_t id_pv = idesc_e4m3(128, kNq, true, true);
        for (int j = 0; j < nb; ++j) {
          const int s = j & 1;
          W.wait(bar(kBarPFull + s), (j >> 1) & 1);
          __syncwarp();
          tc_fence_after();
          const uint32_t tile = sb + kOffTile + s * kStageBytes;
          const uint32_t pb = sb + kOffP + s * kPBytes;
          if (elect_one()) {
            // A = V^T of channel block c: chunk c (128 channels) x 32 keys,
            // MN-major; B = P'^T: 32 keys x 32, MN-major (group scales:
            // group c's 32 bytes of each key's row).
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
              for (int ks = 0; ks < kBK / 32; ++ks) {
                const uint64_t ad =
                    sdesc(tile + c * kChunkBytes + ks * 4096, kChunkBytes, 1024, kLayoutSw128);
                const uint64_t bd = sdesc(pb + ks * 4096 + (kGroup ? 32 * c : 0), kPBytes, 1024,
                                          kLayoutSw128);
                mma_f8(tmem + kColO + 32u * (uint32_t)c, ad, bd, id_pv,
                       (j > 0 || ks > 0) ? 1u : 0u);
              }
            }
            mma_commit(bar(kBarODone));
            mma_commit(bar(kBarPEmpty + s));
            mma_commit(bar(kBarKvEmpty + s));
            if (j == nb - 1) mma_commit(bar(kBarOFinal));
          }
          __syncwarp();
        }
      }
    }
    // Every MMA this warp issued has completed (also after an abort) before
    // the TMEM is freed and the tiles are left.
    __syncwarp();
    if (elect_one()) mma_commit(bar(kBarDrain));
    __syncwarp();
    W.drain(bar(kBarDrain), 0);
  } else if (warp <= 4) {
    // ---- producers: a2 gather of raw rows -------------------------------------
    // Warp wl fills tile rows [32 wl, 32 wl + 32).  The first kTmaChunks
    // 128-byte ckv chunks of each row come by TMA tile::gather4 (8 groups of
    // 4 rows per warp; a masked position, slot id -1, reads the out-of-bounds
    // zero fill); the other ckv chunks and the rope by 16-byte cp.async from
    // the warp's lanes (consecutive lanes on consecutive pieces of a row;
    // masked rows are zero-filled without a read), which run beside the TMA
    // engine.  The rope piece count: 4 (64 E4M3 bytes) or 8 (64 bf16 values).
    const int wl = warp - 1;
    constexpr int kRopePieces = kBf16Rope ? 8 : 4;
    const int n_cp = (4 - kTmaChunks) * 8 + (rope ? kRopePieces : 0);   // pieces a row
    const int row_bytes = kFmt == kDsMla ? kDsMlaRowBytes : p.d_qk;
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
    const uint32_t tx_bytes = (uint32_t)(8 * kTmaChunks * 512);
    int issued = 0;
    for (int b = 0; b < nb; ++b) {
      const int s = b & 1;
      if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b >> 1) - 1) & 1);
      if (*abort_flag) break;                    // the stage may still be in use
      __syncwarp();
      issued = b + 1;
      const uint32_t full = bar(kBarKvFull + s);
      const uint32_t tile = sb + kOffTile + s * kStageBytes;
      const int* bs = slots + b * kBK + 32 * wl;
      if (kTmaChunks > 0 && elect_one()) {
        mbar_arrive_expect_tx(full, tx_bytes);
        for (int g = 0; g < 8; ++g) {
          const int y0 = bs[4 * g], y1 = bs[4 * g + 1], y2 = bs[4 * g + 2], y3 = bs[4 * g + 3];
          for (int c = 0; c < kTmaChunks; ++c)
            tma_gather4(tile + c * kChunkBytes + (32 * wl + 4 * g) * 128, &a.kv_map, 128 * c, y0,
                        y1, y2, y3, full);
        }
      }
      __syncwarp();
      for (int e = lane; e < 32 * n_cp; e += 32) {
        const int r = e / n_cp, k = e - r * n_cp;      // row of the warp, piece of the row
        const int id = bs[r];
        const int row = 32 * wl + r;
        int c, u, src_off;
        if (k < (4 - kTmaChunks) * 8) {
          c = kTmaChunks + (k >> 3);
          u = k & 7;
          src_off = 128 * c + 16 * u;
        } else {
          c = 4;
          u = k - (4 - kTmaChunks) * 8;
          src_off = a.rope_x + 16 * u;
        }
        const uint32_t dst =
            tile + (uint32_t)(c * kChunkBytes + row * 128) + ((uint32_t)(u ^ (row & 7)) << 4);
        const uint8_t* src = kv8 + (size_t)(id < 0 ? 0 : id) * row_bytes + src_off;
        cp_async16(dst, src, id < 0 ? 0u : 16u);
      }
      cp_async_arrive_noinc(full);
    }
    // Teardown: this thread's copies have landed; the gathers of the last
    // block issued into each stage too (earlier ones were consumed before the
    // stage was reissued).
    cp_async_wait_all();
    if (kTmaChunks > 0 && lane == 0) {
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
    const uint32_t lane_base = ((uint32_t)q4 * 32u) << 16;
    const int nbar_wg = 3 + wg;                         // warpgroup-local barrier
    float* qf_sh = reinterpret_cast<float*>(sm + kOffQf);

    // Q' = the QK B operand: rows [0, 16) = hi codes of heads h0.., rows
    // [16, 32) = lo codes, K-major, 128-byte chunks of 32 rows, 128-byte
    // swizzle.  Warp sw prepares heads 2 sw and 2 sw + 1.  For the 656-byte
    // row the rope part of Q stays bf16, in chunk 4 (16 rows x 128 bytes).
    if (nb > 0) {
      const int n_fp8 = rope && !kBf16Rope ? 72 : 64;   // 8-channel pieces split to E4M3
      const int n_pc = rope ? 72 : 64;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int hl = 2 * sw + hh, hd = h0 + hl;
        const bool live = hd < p.h;
        uint4 x[3];
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int k = lane + 32 * j;
          x[j] = (live && k < n_pc) ? __ldg(q_chunk(p, t, hd, 8 * k)) : make_uint4(0u, 0u, 0u, 0u);
          if (k < n_fp8) {
            const uint32_t w[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
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
            const uint32_t w[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
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
                                      ((u ^ (hl & 7)) << 4)) = x[j];
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQReady));
    }
    named_bar_sync(5, kSoftmax);                        // qf_sh written
    // Per head of this warpgroup: Q factor 2^-a, folded with the score scale
    // (and the per-tensor E4M3 scale).
    const float kscale = kFmt == kE4m3 ? __ldg(p.k_scale) : 1.f;
    float cs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = qf_sh[8 * wg + i] * a.scale_log2 * kscale;
    const float rope_cs = a.scale_log2;                 // bf16 rope: not scaled by 2^-a
    bool head_ok[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) head_ok[i] = h0 + 8 * wg + i < p.h;

    float m_run[8], l_part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { m_run[i] = -INFINITY; l_part[i] = 0.f; }
    float R[4] = {0.f, 0.f, 0.f, 0.f};                  // PV group factors (0: not set)
    float* red = reinterpret_cast<float*>(sm + kOffRed) + wg * 32;      // [4 warps][8]
    float* red_sc = reinterpret_cast<float*>(sm + kOffRedSc) + wg * 16; // [4 warps][4]
    // This key's 128-byte row of a P' buffer (MN-major, 128-byte swizzle).
    const uint32_t p_row = (uint32_t)(key >> 3) * 1024u + (uint32_t)(key & 7) * 128u;
    const uint32_t p_sw = (uint32_t)(key & 7);
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);

    // The key's group scales of block b (0 when masked): [0..3] the ckv
    // groups, [4] the rope group.
    auto load_scales = [&](int b, float (&sc)[5]) {
      const int id = b < nb ? slots[b * kBK + key] : -1;
#pragma unroll
      for (int g = 0; g < 5; ++g) sc[g] = 0.f;
      if (!kGroup || id < 0) return;
      if (kFmt == kDsMla) {
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(kv8 + (size_t)id * kDsMlaRowBytes +
                                                               kDsMlaScaleOff));
        sc[0] = s4.x; sc[1] = s4.y; sc[2] = s4.z; sc[3] = s4.w; sc[4] = 1.f;
      } else if (kFmt == kE4m3Group4Kpe) {
        const float* r = p.k_scale + (int64_t)id * 4;
        sc[0] = __ldg(r); sc[1] = __ldg(r + 1); sc[2] = __ldg(r + 2); sc[3] = __ldg(r + 3);
        sc[4] = p.kpe_scale;
      } else {
        const float* r = p.k_scale + (int64_t)id * a.G;
        sc[0] = __ldg(r); sc[1] = __ldg(r + 1); sc[2] = __ldg(r + 2); sc[3] = __ldg(r + 3);
        if (a.G > 4) sc[4] = __ldg(r + 4);
      }
    };
    float nsc[5];
    load_scales(0, nsc);

    for (int b = 0; b < nb; ++b) {
      const int s = b & 1;
      float sc[5];
#pragma unroll
      for (int g = 0; g < 5; ++g) sc[g] = nsc[g];
      load_scales(b + 1, nsc);                          // next block's, in flight
      W.wait(bar(kBarSFull + s), (b >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      // a4 result: per group, this warpgroup's 8 heads hi (columns 8 wg..)
      // and lo (16 + 8 wg..).
      float sp[8];
      {
        const uint32_t c0 = tmem + lane_base + kColS + kSBuf * s + 8u * (uint32_t)wg;
        if (kGroup) {
          uint32_t w[5][2][8];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            tmem_ld8(c0 + kNq * g, w[g][0]);
            tmem_ld8(c0 + kNq * g + 16, w[g][1]);
          }
          if (rope) {
            tmem_ld8(c0 + kNq * 4, w[4][0]);
            if (!kBf16Rope) tmem_ld8(c0 + kNq * 4 + 16, w[4][1]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              acc = fmaf(sc[g], fmaf(__uint_as_float(w[g][1][i]), 0.0625f,
                                     __uint_as_float(w[g][0][i])), acc);
            float r = 0.f;
            if (rope && !kBf16Rope)
              acc = fmaf(sc[4], fmaf(__uint_as_float(w[4][1][i]), 0.0625f,
                                     __uint_as_float(w[4][0][i])), acc);
            if (rope && kBf16Rope) r = __uint_as_float(w[4][0][i]);
            sp[i] = fmaf(acc, cs[i], r * rope_cs);
          }
        } else {
          uint32_t w0[8], w1[8];
          tmem_ld8(c0, w0);
          tmem_ld8(c0 + 16, w1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            sp[i] = fmaf(__uint_as_float(w1[i]), 0.0625f, __uint_as_float(w0[i])) * cs[i];
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty + s));

      // a5: masked scores (log2 units) and the lazy running max; with group
      // scales also the lazy PV group factors R (scale * R <= 1).
      const bool key_ok = ((masks[b * 4 + (key >> 5)] >> (key & 31)) & 1u) != 0u;
      bool need = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sp[i] = (key_ok && head_ok[i]) ? sp[i] : -INFINITY;
        need |= sp[i] > m_run[i] + kT;
      }
      if (kGroup) {
#pragma unroll
        for (int g = 0; g < 4; ++g) need |= R[g] == 0.f || sc[g] * R[g] > 1.f;
      }
      float alpha[8], ratio[4] = {1.f, 1.f, 1.f, 1.f};
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
          for (int g = 0; g < 4; ++g) {
            float x = sc[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
            if (lane == 0) red_sc[q4 * 4 + g] = x;
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
          for (int g = 0; g < 4; ++g) {
            const float ms = fmaxf(fmaxf(red_sc[g], red_sc[4 + g]),
                                   fmaxf(red_sc[8 + g], red_sc[12 + g]));
            if (ms > 0.f && (R[g] == 0.f || ms * R[g] > 1.f)) {
              const float rn = pow2_at_most_inv(ms);
              if (R[g] != 0.f) ratio[g] = rn / R[g];
              R[g] = rn;
            }
          }
        }
        named_bar_sync(nbar_wg, 128);             // red may be rewritten
      }
      float pe[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pe[i] = m_run[i] == -INFINITY ? 0.f : ex2_approx(sp[i] - m_run[i]);
        l_part[i] = fmaf(l_part[i], alpha[i], pe[i]);
      }
      // a6 operand: P' hi / lo codes into buffer s (per group with scales).
      if (b >= 2) W.wait(bar(kBarPEmpty + s), ((b >> 1) - 1) & 1);   // PV(b-2) read it
      uint8_t* prow = sm + kOffP + s * kPBytes + p_row;
#pragma unroll
      for (int g = 0; g < (kGroup ? 4 : 1); ++g) {
        const float f = kGroup ? sc[g] * R[g] * kPShift : kPShift;
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = pe[i] * f;
        uint2 hi, lo;
        split8(x, hi, lo);
        *reinterpret_cast<uint2*>(prow + ((((uint32_t)(2 * g) ^ p_sw) << 4) | (8u * wg))) = hi;
        *reinterpret_cast<uint2*>(prow + ((((uint32_t)(2 * g + 1) ^ p_sw) << 4) | (8u * wg))) = lo;
      }
      fence_proxy_async_smem();
      if (voted && b >= 1) {
        // O^T row (channel `key` of each 128-channel block): this
        // warpgroup's head columns (hi and lo) *= alpha * ratio of the block.
        bool any = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) any |= alpha[i] != 1.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) any |= ratio[g] != 1.f;
        if (any) {                                      // uniform in the warpgroup
          W.wait(bar(kBarODone), (b - 1) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const uint32_t col = tmem + lane_base + kColO + 32u * c + 16u * part + 8u * wg;
              uint32_t w[8];
              tmem_ld8(col, w);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha[i] * ratio[c]);
              tmem_st8(col, w);
            }
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + s));
    }

    // ---- a7: epilogue ---------------------------------------------------------
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
    if (nb > 0) {
      W.wait(bar(kBarOFinal), 0);
      __syncwarp();
      tc_fence_after();
    }
    const float oscale = kFmt == kE4m3 ? kscale : 1.f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t wh[8], wl8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) { wh[i] = 0u; wl8[i] = 0u; }
      __syncwarp();
      if (nb > 0) {
        const uint32_t col = tmem + lane_base + kColO + 32u * c + 8u * wg;
        tmem_ld8(col, wh);
        tmem_ld8(col + 16, wl8);
        tmem_wait_ld();
      }
      const float rc = kGroup ? R[c] : 1.f;
      const int ch = 128 * c + key;                   // output channel of lane `key`
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (head_ok[i]) {
          const bool empty = !(l_tot[i] > 0.f) || nb == 0 || !(rc > 0.f);
          const float o = empty ? 0.f
                                : fmaf(__uint_as_float(wl8[i]), 0.0625f, __uint_as_float(wh[i])) *
                                      (oscale / (l_tot[i] * kPShift * rc));
          const int64_t orow = (int64_t)t * p.h + h0 + 8 * wg + i;
          if (p.fp32_out)
            p.o_part[((int64_t)split * p.T * p.h + orow) * p.d_v + ch] = o;
          else
            reinterpret_cast<__nv_bfloat16*>(p.out)[orow * p.d_v + ch] = __float2bfloat16_rn(o);
        }
      }
    }
    // Thread `key` < 8 writes the LSE of head 8 wg + key.
    if (key < 8 && h0 + 8 * wg + key < p.h) {
      float mi = m_run[0], li = l_tot[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        mi = key == i ? m_run[i] : mi;
        li = key == i ? l_tot[i] : li;
      }
      const bool empty = !(li > 0.f) || nb == 0;
      const float lse_v = empty ? -INFINITY : (mi + log2f(li)) * 0.69314718055994530942f;
      const int64_t orow = (int64_t)t * p.h + h0 + 8 * wg + key;
      if (p.fp32_out)
        p.lse_part[(int64_t)split * p.T * p.h + orow] = lse_v;
      else if (p.lse)
        p.lse[orow] = lse_v;
    }
  }

  // ---- teardown -------------------------------------------------------------
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
  const int64_t blocks = (int64_t)p.T * p.splits * a.n_hg;   // one CTA per unit
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  switch (p.kv_format) {
    case kE4m3: return launch_fmt<kE4m3>(a, (unsigned)blocks, stream);
    case kE4m3Group: return launch_fmt<kE4m3Group>(a, (unsigned)blocks, stream);
    case kDsMla: return launch_fmt<kDsMla>(a, (unsigned)blocks, stream);
    default: return launch_fmt<kE4m3Group4Kpe>(a, (unsigned)blocks, stream);
  }
}

}  // namespace smla

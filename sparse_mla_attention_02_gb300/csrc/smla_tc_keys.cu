// smla_tc_keys.cu — tensor-core (tcgen05 / TMEM) sparse MLA forward for up
// to 16 heads, every cache format, including E4M3 with one scale per
// (slot, 128-channel group).
//
// With few heads, the heads cannot fill a 128-row MMA, so this kernel turns
// both products around: the 128 top-k positions of a block are the MMA's M
// dimension and the heads (zero-padded to 16) are N:
//   S^T[keys, heads] = K[keys, d] . Q^T[d, heads]         A = gathered tile, K-major
//   O^T[ch, heads]  += V^T[ch, keys] . P^T[keys, heads]    A = the same tile, MN-major
// One work unit = (query token, top-k range) on a cluster of two CTAs that
// split the channels: CTA r holds channels [256r, 256r + 256) (groups 2r and
// 2r + 1) and, for d_qk = 576, half of the 64-channel rope group 4,
// [512 + 32r, 544 + 32r), so both CTAs gather and multiply the same bytes.
//   * QK: with group scales each CTA keeps one fp32 accumulator per group in
//     TMEM, so a key's group scale multiplies its partial score exactly (in
//     fp32) before the groups are summed.  The CTA sends its partial scores
//     [128 keys x 16 heads] to the other with one bulk copy; both then hold
//     the full scores and run the same softmax (same inputs, same results).
//   * PV: CTA r owns output channels [256r, 256r + 256) = groups 2r, 2r + 1.
//     With group scales, P^T is stored once per group, each key's entry
//     multiplied by that key's group scale, so the tile keeps exact values.
//     A scaled entry is kept as a bf16 pair hi + lo, side by side in the N
//     dimension (N = 32: the MMA's cost is set by reading its 4 KB A slice,
//     so the wider N is free) and summed in the epilogue; a single bf16
//     rounding of p * scale would put up to 2^-9 relative error on O even
//     for one key.
// Thread i of the softmax warpgroup owns key i of the block (TMEM lane i):
// the key's group scales and valid bit are per-thread values, the per-head
// max is reduced across the warpgroup only when some score passes the
// running max by more than 2^8 (a one-barrier vote otherwise), and each
// thread keeps partial row sums for its own keys, reduced once at the end.
//
// Method steps (vLLM "Sparse MLA on Hopper" diff, ops/cutlass_fa3.py docstring:
// score = q_rope.k_rope + q_nope.c_kv, output = softmax(score*scale) @ c_kv;
// flashinfer_mla_sparse_sm90.py, module docstring: FP8 cache read directly
// with a per-tensor k_scale or per-token x 128-channel-group scales;
// forward_mqa: compacted valid prefix with -1 past it; vLLM API docs
// flashmla_sparse, _forward_fp8_kv_mixed_batch: empty rows give (O = 0,
// LSE = -inf)):
//   a1 work setup: v = min(valid_len[t], topk); range [k0, k1) of the split
//   a2 gather: slot ids -> 128-byte-swizzled bf16 tiles (TMA tile::gather4
//      for bf16; E4M3 rows converted exactly on load); masked keys are zero
//   a3 scales: per-tensor scale folded into the score scale and the output;
//      group scales applied per group accumulator (QK) and per copy of P (PV)
//   a4 QK^T, a5 masked online softmax, a6 PV, a7 O / l and LSE = m + ln l
//
// Warp roles (352 threads): warp 0 issues the QK MMAs and owns TMEM; warp 10
// issues the PV MMAs; warps 1..4 load the unit's slot ids, then gather
// (bf16: TMA; E4M3: each warp loads 32 rows cooperatively, 16 lanes a row,
// and converts and stores what it loaded);
// warp 5 tells the peer when its partial scores were consumed; warps 6..9
// (thread <-> key <-> TMEM lane) load Q, run the exchange, softmax, O
// rescale and the epilogue.  (Eleven warps leave each thread up to 168
// registers.)
// Every wait is bounded; a wait that runs out records a timeout status, sets
// an abort flag that skips later waits, and the block finishes normally.
#include <math.h>

#include "smla_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kBK = 128;                   // top-k positions per block (MMA M)
constexpr int kN = 16;                     // heads, zero-padded (MMA N)
constexpr int kStages = 2;                 // gathered-tile pipeline depth
constexpr int kChunkBytes = kBK * 128;     // 64 channels x 128 keys, bf16
constexpr int kMaxChunks = 5;              // up to 320 channels per CTA
constexpr int kStageBytes = kMaxChunks * kChunkBytes;
constexpr int kScaleBytes = kBK * 16;      // 4 group-scale slots per key
constexpr int kQChunkBytes = kN * 128;     // 64 channels x 16 heads
constexpr int kPCopyBytes = 2 * kQChunkBytes;   // P^T: 16 rows x 128 keys (2 K-atoms)
constexpr int kPAreaBytes = 4 * kPCopyBytes;    // 2 buffers x 1 copy, or 2 groups x
                                                // [hi | lo] rows (32 x 128 keys)
constexpr int kXBytes = kBK * kN * 4;      // exchanged partial scores, fp32
constexpr int kThreads = 352;
constexpr int kProducers = 128;            // warps 1..4
constexpr int kSoftmax = 128;              // warps 6..9
constexpr int kMaxBlocks = 16;             // ranges up to 2048 positions

// TMEM columns.
constexpr uint32_t kColO = 0;              // O^T: 2 blocks of 128 channels x 32
                                           // (16 heads, or hi | lo with group scales)
constexpr uint32_t kColS = 4 * kN;         // partial S: 2 buffers x 3 groups x 16
constexpr uint32_t kSBuf = 3 * kN;
constexpr uint32_t kTmemCols = 256;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffScale = kOffTile + kStages * kStageBytes;
constexpr uint32_t kOffQ = kOffScale + kStages * kScaleBytes;
constexpr uint32_t kOffP = kOffQ + kMaxChunks * kQChunkBytes;      // P^T buffers
constexpr uint32_t kOffX = kOffP + kPAreaBytes;                    // receive [2]
constexpr uint32_t kOffXs = kOffX + 2 * kXBytes;                   // send staging
constexpr uint32_t kOffSlot = kOffXs + kXBytes;                    // [blocks*128] i32
constexpr uint32_t kOffMask = kOffSlot + kMaxBlocks * kBK * 4;     // [blocks][4] u32
constexpr uint32_t kOffRed = kOffMask + kMaxBlocks * 16;           // 2 x [16][4] f32
constexpr uint32_t kOffBar = kOffRed + 2 * kN * 4 * 4;
enum {
  kBarKvFull = 0,                   // [2]
  kBarKvEmpty = kBarKvFull + 2,     // [2]
  kBarSFull = kBarKvEmpty + 2,      // [2]
  kBarSEmpty = kBarSFull + 2,       // [2]
  kBarPFull = kBarSEmpty + 2,       // [P buffers]
  kBarPEmpty = kBarPFull + 2,       // [P buffers]
  kBarXFull = kBarPEmpty + 2,       // [2]
  kBarXFree = kBarXFull + 2,        // [2]
  kBarXCons = kBarXFree + 2,        // [2]
  kBarODone = kBarXCons + 2,
  kBarOFinal,                       // one phase: the unit's last PV is done
  kBarQReady,
  kNumBars
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled operands need 1024-B alignment");
static_assert(kOffX % 16 == 0 && kOffXs % 16 == 0, "bulk copies need 16-B alignment");
static_assert(kColS + 2 * kSBuf <= kTmemCols, "TMEM budget");

struct KeysArgs {
  CUtensorMap kv_map;  // bf16 cache as a 2-D tensor, 64-channel boxes (bf16 only)
  FwdParams p;
  int ksteps;          // 16-channel QK steps per CTA: 18 (d_qk 576) or 16 (512)
  int G;               // scale groups per slot (group format)
  float scale_log2;    // sm_scale * log2(e)
};

// Reduce v[0..15] (one value per head) over the 32 lanes of the warp.  Each
// step hands half of the remaining heads to the partner lane, so lane l ends
// with the result for head l >> 1 (16 shuffles instead of 80).
template <bool kMax>
__device__ __forceinline__ float op2(float x, float y) {
  return kMax ? fmaxf(x, y) : x + y;
}
template <bool kMax, int kW>
__device__ __forceinline__ void xreduce_step(float (&v)[kN], int lane) {
  const bool hi = (lane & (2 * kW)) != 0;
#pragma unroll
  for (int j = 0; j < kW; ++j) {
    const float send = hi ? v[j] : v[j + kW];
    const float keep = hi ? v[j + kW] : v[j];
    v[j] = op2<kMax>(keep, __shfl_xor_sync(0xffffffffu, send, 2 * kW));
  }
}
template <bool kMax>
__device__ __forceinline__ float xreduce16(float (&v)[kN], int lane) {
  xreduce_step<kMax, 8>(v, lane);
  xreduce_step<kMax, 4>(v, lane);
  xreduce_step<kMax, 2>(v, lane);
  xreduce_step<kMax, 1>(v, lane);
  return op2<kMax>(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

template <int kFmt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
smla_tc_keys_kernel(const __grid_constant__ KeysArgs a) {
  // Formats with per-(slot, group) scales: one QK accumulator per group.
  constexpr bool kGroup = kFmt == kE4m3Group || kFmt == kDsMla || kFmt == kE4m3Group4Kpe;
  constexpr bool kFp8 = kFmt != kBf16;
  // P^T buffers: group scales need 4 copies (2 groups x hi/lo) in one buffer;
  // otherwise one copy, double-buffered.
  constexpr int kPBufs = kGroup ? 1 : 2;
  constexpr int kPBufBytes = kPAreaBytes / kPBufs;
  constexpr int kPAtomBytes = kGroup ? 2 * kQChunkBytes : kQChunkBytes;  // one K-atom
  constexpr int kNpv = kGroup ? 2 * kN : kN;                              // PV MMA N
  extern __shared__ uint8_t smem_raw[];
  const FwdParams& p = a.p;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;           // shared address base
  uint8_t* sm = smem_raw + (sb - raw);                  // generic pointer base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t r = cluster_ctarank();
  const uint32_t peer = r ^ 1u;

  // ---- a1: work unit ------------------------------------------------------
  const int unit = blockIdx.x >> 1;
  const int split = unit % p.splits;
  const int t = unit / p.splits;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);
  // The host plan keeps every range within kMaxBlocks blocks.
  const int nb = k1 > k0 ? min((k1 - k0 + kBK - 1) / kBK, kMaxBlocks) : 0;
  // CTA r's channels: steps 0..15 = [256r, 256r + 256); steps 16, 17 (d_qk
  // 576) = rope [512 + 32r, 544 + 32r), held in tile chunk 4.
  const int ksteps = a.ksteps;
  const int n_lg = kGroup ? (ksteps + 7) / 8 : 1;       // group accumulators
  const int g_lo = 256 * (int)r;                        // first V channel of CTA r
  const int rope_lo = 512 + 32 * (int)r;                // first rope channel

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W{abort_flag, p.status};

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // bf16: one expect_tx per TMA warp; E4M3: one arrival per loader thread
      mbar_init(bar(kBarKvFull + s), kFp8 ? kProducers : 4);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {     // (group scales use P barrier 0 only)
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), kSoftmax);
      mbar_init(bar(kBarPFull + i), kSoftmax);
      mbar_init(bar(kBarPEmpty + i), 1);
      mbar_init(bar(kBarXFull + i), 1);
      mbar_init(bar(kBarXFree + i), 1);
      mbar_init(bar(kBarXCons + i), kSoftmax);
    }
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarOFinal), 1);
    mbar_init(bar(kBarQReady), kSoftmax);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(sb + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kOffTmemSlot);

  // a1/a2 setup: the loaders read the unit's index range once into shared
  // memory, masking positions past k1, ids < 0 and ids >= num_slots; then
  // one valid-bit word per 32 keys of each block.
  int* slots = reinterpret_cast<int*>(sm + kOffSlot);
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + kOffMask);
  if (warp >= 1 && warp <= 4) {
    const int pt = tid - 32;
    const int n = nb * kBK;
    if (load_unit_slots(p, t, k0, k1, n, slots, pt, kProducers))
      atomicCAS(p.status, 0, kStatusBadIndex);
    named_bar_sync(1, kProducers);
    const int row = (warp - 1) * 32 + lane;
    for (int b = 0; b < nb; ++b) {
      const uint32_t m = __ballot_sync(0xffffffffu, slots[b * kBK + row] >= 0);
      if (lane == 0) masks[b * 4 + (warp - 1)] = m;
    }
  }
  __syncthreads();

  const bool leader = warp == 8 && lane == 0;            // softmax thread of key 0
  if (warp == 0 || warp == 10) {
    // ---- MMA issuers: warp 0 issues QK, warp 10 issues PV -------------------
    // Two warps, each blocked only on its own inputs, so neither kind of
    // batch waits behind the other.  Each warp runs its code warp-uniformly;
    // one elected lane issues a batch of MMAs and commits it (a commit
    // tracks the MMAs of the issuing thread).
    if (nb > 0) {
      const uint32_t id_qk = idesc_bf16(128, kN, false, false);
      const uint32_t id_pv = idesc_bf16(128, kNpv, true, kGroup);
      const uint32_t qb = sb + kOffQ;
      auto issue_qk = [&](int j) {
        const int s = j & 1;
        W.wait(bar(kBarKvFull + s), (j >> 1) & 1);
        if (j >= 2) W.wait(bar(kBarSEmpty + s), ((j >> 1) - 1) & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kStageBytes;
        const uint32_t dS = tmem + kColS + kSBuf * s;
        if (elect_one()) {
          fence_proxy_async_smem();
          // A descriptor's start-address field is addr >> 4 in its low bits,
          // so each step's descriptor is the base plus a constant.
          const uint64_t a0 = sdesc(tile, 16, 1024, kLayoutSw128);
          const uint64_t b0 = sdesc(qb, 16, 1024, kLayoutSw128);
#pragma unroll
          for (int ks = 0; ks < 18; ++ks) {
            if (ks < ksteps) {
              const uint32_t oa = (uint32_t)((ks >> 2) * kChunkBytes + (ks & 3) * 32);
              const uint32_t ob = (uint32_t)((ks >> 2) * kQChunkBytes + (ks & 3) * 32);
              const uint32_t acc = kGroup ? (uint32_t)(ks >> 3) * kN : 0u;
              const bool first = kGroup ? (ks & 7) == 0 : ks == 0;
              mma_ss(dS + acc, a0 + (oa >> 4), b0 + (ob >> 4), id_qk, first ? 0u : 1u);
            }
          }
          mma_commit(bar(kBarSFull + s));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int j) {
        const int s = j & 1;
        const int pbi = j % kPBufs;
        W.wait(bar(kBarPFull + pbi), (j / kPBufs) & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kStageBytes;
        const uint32_t pb = sb + kOffP + pbi * kPBufBytes;
        if (elect_one()) {
          fence_proxy_async_smem();
          // A = V^T: 128 channels (two 64-channel chunks) x 16 keys, MN-major;
          // B = P^T of this channel group: 16 keys x N.  Without group
          // scales K-major (16 head rows of 128 keys); with them MN-major,
          // one 128-byte row per key holding [g0 hi | g0 lo | g1 hi | g1 lo]
          // (16 heads each), so group mb starts 64 mb bytes into the row.
          const uint64_t a0 = sdesc(tile, kChunkBytes, 1024, kLayoutSw128);
          const uint64_t b0 = kGroup ? sdesc(pb, kPAreaBytes, 1024, kLayoutSw128)
                                     : sdesc(pb, 16, 1024, kLayoutSw128);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks) {
              const uint32_t oa = (uint32_t)(2 * mb * kChunkBytes + ks * 16 * 128);
              const uint32_t ob =
                  kGroup ? (uint32_t)(64 * mb + ks * 16 * 128)
                         : (uint32_t)((ks >> 2) * kPAtomBytes + (ks & 3) * 32);
              mma_ss(tmem + kColO + 2 * kN * mb, a0 + (oa >> 4), b0 + (ob >> 4), id_pv,
                     ks > 0 ? 1u : acc0);
            }
          }
          mma_commit(bar(kBarODone));
          mma_commit(bar(kBarPEmpty + pbi));
          mma_commit(bar(kBarKvEmpty + s));
          if (j == nb - 1) mma_commit(bar(kBarOFinal));
        }
        __syncwarp();
      };
      if (warp == 0) {
        W.wait(bar(kBarQReady), 0);
        tc_fence_after();
        for (int j = 0; j < nb; ++j) issue_qk(j);
      } else {
        for (int j = 0; j < nb; ++j) issue_pv(j);
      }
    }
  } else if (warp <= 4) {
    // ---- loaders: a2 gather (+ a3 E4M3 conversion) -------------------------
    if (kFp8) {
      // Warp-cooperative gather: loader warp w owns rows [32w, 32w + 32) of
      // every block.  A row's 256 ckv bytes are read by 16 lanes, 16 bytes
      // each, two rows per load instruction, so one instruction touches a few
      // cache lines rather than 32; the rope pieces follow, 16 (E4M3) or 8
      // (bf16) rows per instruction.  All loads of a block are in flight
      // before the stage is awaited; then each lane converts what it loaded
      // (exact E4M3 -> bf16) into the 128-byte-swizzled tile.  Masked rows
      // are zero.  656-byte rows: the rope is bf16 (copied as it is), the
      // group scales sit in the row, and the rope group's scale is 1.
      const int w0 = (warp - 1) * 32;                      // the warp's first row
      const int half = lane >> 4, pc = lane & 15;          // ckv: row of the pair, piece
      const bool rope = ksteps > 16;                       // d_qk 576
      constexpr int kRopeLanes = kFmt == kDsMla ? 4 : 2;   // 16-byte rope pieces a row
      constexpr int kRopeRows = 32 / kRopeLanes;           // rows per rope instruction
      constexpr int kRopeIns = 32 / kRopeRows;             // rope instructions per block
      const int rpc = lane % kRopeLanes, rrow = lane / kRopeLanes;
      const int row_bytes = kFmt == kDsMla ? kDsMlaRowBytes : p.d_qk;
      const uint32_t rope_off =
          kFmt == kDsMla ? (uint32_t)(kDsMlaRopeOff + 64 * (int)r) : (uint32_t)rope_lo;
      const int scale_stride = kFmt == kE4m3Group4Kpe ? 4 : a.G;
      const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
      const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
      for (int b = 0; b < nb; ++b) {
        const int s = b & 1;
        const int* bs = slots + b * kBK + w0;
        uint4 ck[16], rq[kRopeIns];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int id = bs[2 * i + half];
          ck[i] = id >= 0 ? __ldg(reinterpret_cast<const uint4*>(
                                      kv8 + (size_t)id * row_bytes + g_lo) + pc)
                          : zero4;
        }
#pragma unroll
        for (int j = 0; j < kRopeIns; ++j) {
          const int id = bs[kRopeRows * j + rrow];
          rq[j] = (rope && id >= 0) ? __ldg(reinterpret_cast<const uint4*>(
                                                kv8 + (size_t)id * row_bytes + rope_off) + rpc)
                                    : zero4;
        }
        // The lane's own row (w0 + lane): its group scales, and the row of
        // the next block into L2 while this one is converted.
        const int id = bs[lane];
        const uint8_t* rowp = kv8 + (size_t)(id < 0 ? 0 : id) * row_bytes;
        if (b + 1 < nb) {
          const int idn = slots[(b + 1) * kBK + w0 + lane];
          if (idn >= 0) {
            const uint8_t* rn = kv8 + (size_t)idn * row_bytes;
            prefetch_l2(rn + g_lo);
            prefetch_l2(rn + g_lo + 128);
            prefetch_l2(rn + g_lo + 255);
            if (rope) prefetch_l2(rn + rope_off);
            if (kFmt == kDsMla) {
              prefetch_l2(rn + kDsMlaScaleOff);
              prefetch_l2(rn + rope_off + 63);
            } else if (kGroup) {
              prefetch_l2(p.k_scale + (int64_t)idn * scale_stride);
            }
          }
        }
        float sc[3] = {0.f, 0.f, 0.f};
        if (kGroup && id >= 0) {
          const float* srow = kFmt == kDsMla
                                  ? reinterpret_cast<const float*>(rowp + kDsMlaScaleOff)
                                  : p.k_scale + (int64_t)id * scale_stride;
          sc[0] = __ldg(srow + 2 * (int)r);
          sc[1] = __ldg(srow + 2 * (int)r + 1);
          if (n_lg > 2)
            sc[2] = kFmt == kE4m3Group ? __ldg(srow + 4) : kFmt == kDsMla ? 1.f : p.kpe_scale;
        }
        if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b >> 1) - 1) & 1);
        uint8_t* tile = sm + kOffTile + s * kStageBytes;
        // 16-byte unit cj (8 bf16 channels) of `row` in the swizzled tile
        auto unit = [&](int row, uint32_t cj) -> uint4* {
          return reinterpret_cast<uint4*>(tile + row * 128 + (cj >> 3) * kChunkBytes +
                                          (((cj & 7u) ^ ((uint32_t)row & 7u)) << 4));
        };
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int row = w0 + 2 * i + half;
          uint32_t o[8];
          e4m3x4_to_bf16_sx(ck[i].x, o[0], o[1]);
          e4m3x4_to_bf16_sx(ck[i].y, o[2], o[3]);
          e4m3x4_to_bf16_sx(ck[i].z, o[4], o[5]);
          e4m3x4_to_bf16_sx(ck[i].w, o[6], o[7]);
          *unit(row, 2u * (uint32_t)pc) = make_uint4(o[0], o[1], o[2], o[3]);
          *unit(row, 2u * (uint32_t)pc + 1u) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        if (rope) {
#pragma unroll
          for (int j = 0; j < kRopeIns; ++j) {
            const int row = w0 + kRopeRows * j + rrow;
            if (kFmt == kDsMla) {
              *unit(row, 32u + (uint32_t)rpc) = rq[j];       // bf16, as is
            } else {
              uint32_t o[8];
              e4m3x4_to_bf16_sx(rq[j].x, o[0], o[1]);
              e4m3x4_to_bf16_sx(rq[j].y, o[2], o[3]);
              e4m3x4_to_bf16_sx(rq[j].z, o[4], o[5]);
              e4m3x4_to_bf16_sx(rq[j].w, o[6], o[7]);
              *unit(row, 32u + 2u * (uint32_t)rpc) = make_uint4(o[0], o[1], o[2], o[3]);
              *unit(row, 33u + 2u * (uint32_t)rpc) = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
        }
        if (kGroup)
          *reinterpret_cast<float4*>(sm + kOffScale + s * kScaleBytes + (w0 + lane) * 16) =
              make_float4(sc[0], sc[1], sc[2], 0.f);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarKvFull + s));
      }
    } else {
      // bf16: warps 1..4 each issue 8 of the 32 four-row groups per block.
      const int w = warp - 1;
      const int n_boxes = ksteps > 16 ? 5 : 4;               // + one rope box
      const uint32_t tx_bytes = (uint32_t)(8 * n_boxes * 512);
      for (int b = 0; b < nb; ++b) {
        const int s = b & 1;
        if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b >> 1) - 1) & 1);
        __syncwarp();
        if (elect_one()) {
          const uint32_t full = bar(kBarKvFull + s);
          mbar_arrive_expect_tx(full, tx_bytes);
          const uint32_t tile = sb + kOffTile + s * kStageBytes;
          const int* bs = slots + b * kBK;
          for (int g = w; g < kBK / 4; g += 4) {
            const int y0 = bs[4 * g], y1 = bs[4 * g + 1], y2 = bs[4 * g + 2], y3 = bs[4 * g + 3];
            // (the rope box of CTA 1 runs past the row end: zero fill)
            for (int c = 0; c < n_boxes; ++c)
              tma_gather4(tile + c * kChunkBytes + 4 * g * 128, &a.kv_map,
                          c < 4 ? g_lo + 64 * c : rope_lo, y0, y1, y2, y3, full);
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == 5) {
    // ---- signal warp: tell the peer when its partial scores were consumed --
    if (lane == 0) {
      const uint32_t xfree_peer = mapa(bar(kBarXFree), peer);
      for (int b = 0; b < nb; ++b) {
        W.wait(bar(kBarXCons + (b & 1)), (b >> 1) & 1);
        mbar_arrive_remote(xfree_peer + 8u * (b & 1));
      }
    }
  } else {
    // ---- softmax warpgroup (thread i <-> key i <-> TMEM lane i) -------------
    const int i = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = ((uint32_t)(warp & 3) * 32u) << 16;
    // Q (channels of this CTA, heads >= h zero) -> the QK B operand:
    // K-major, 64-channel chunks of 16 rows x 128 B, 128-byte swizzle.
    {
      const int per_head = 2 * ksteps;                   // 16-byte pieces per head
      const int total = kN * per_head;                   // <= 576
      uint4 qv[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int idx = i + kSoftmax * k;
        const int hd = idx / per_head, c16 = idx - hd * per_head;
        const int ch = c16 < 32 ? g_lo + 8 * c16 : rope_lo + 8 * (c16 - 32);
        qv[k] = (idx < total && hd < p.h) ? __ldg(q_chunk(p, t, hd, ch))
                                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int idx = i + kSoftmax * k;
        if (idx < total) {
          const int hd = idx / per_head, c16 = idx - hd * per_head;
          *reinterpret_cast<uint4*>(sm + kOffQ + (c16 >> 3) * kQChunkBytes + (hd >> 3) * 1024 +
                                    (hd & 7) * 128 + (((c16 & 7) ^ (hd & 7)) << 4)) = qv[k];
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQReady));
    }
    // Per-tensor E4M3: the scale multiplies every score and output.
    const float kscale = kFmt == kE4m3 ? __ldg(p.k_scale) : 1.f;
    const float scale_log2 = a.scale_log2 * kscale;
    float m_run[kN], l_part[kN];
#pragma unroll
    for (int hd = 0; hd < kN; ++hd) { m_run[hd] = -INFINITY; l_part[hd] = 0.f; }
    const uint32_t x_peer = mapa(sb + kOffX, peer);
    const uint32_t xfull_peer = mapa(bar(kBarXFull), peer);
    const uint32_t xrow = (uint32_t)i * kN * 4;          // this key's 64-byte row
    const uint32_t xsw = ((uint32_t)i >> 1) & 3u;        // its chunk swizzle
    float* red = reinterpret_cast<float*>(sm + kOffRed); // [16 heads][4 warps]
    // Without group scales, this key's byte offset inside the K-major P^T
    // (128-byte swizzle): K-atom (i / 64), 16-byte chunk ((i % 64) / 8) ^
    // (head % 8), element i % 8.  With them, this key's 128-byte row of the
    // MN-major P^T: atom i / 8, row i % 8, 16-byte chunk c at c ^ (i % 8).
    const uint32_t p_atom = (uint32_t)(i >> 6) * kPAtomBytes + (uint32_t)(i & 7) * 2u;
    const uint32_t p_chunk = (uint32_t)(i & 63) >> 3;
    const uint32_t p_row = (uint32_t)(i >> 3) * 1024u + (uint32_t)(i & 7) * 128u;
    const uint32_t p_sw = (uint32_t)(i & 7);

    for (int b = 0; b < nb; ++b) {
      const int s = b & 1;
      float sp[kN];
      float scp0 = 1.f, scp1 = 1.f;          // this key's PV group scales
      // a4 result: this CTA's partial scores for key i.
      if (leader) {
        mbar_arrive_expect_tx(bar(kBarXFull + s), (uint32_t)kXBytes);
        bulk_wait_read_all();                // the previous send has read the stage
      }
      if (kGroup) W.wait(bar(kBarKvFull + s), (b >> 1) & 1);   // scale rows visible
      W.wait(bar(kBarSFull + s), (b >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      {
        uint32_t w[16];
        if (kGroup) {
          const float4 sc =
              *reinterpret_cast<const float4*>(sm + kOffScale + s * kScaleBytes + i * 16);
          scp0 = sc.x;
          scp1 = sc.y;
          // The group accumulators' loads are issued together, then awaited.
          uint32_t w1[16], w2[16];
          const uint32_t sc0 = tmem + lane_base + kColS + kSBuf * s;
          tmem_ld16(sc0, w);
          tmem_ld16(sc0 + kN, w1);
          if (n_lg > 2) tmem_ld16(sc0 + 2 * kN, w2);   // same for every lane
          tmem_wait_ld();
#pragma unroll
          for (int hd = 0; hd < kN; ++hd)
            sp[hd] = fmaf(sc.y, __uint_as_float(w1[hd]), sc.x * __uint_as_float(w[hd]));
          if (n_lg > 2) {
#pragma unroll
            for (int hd = 0; hd < kN; ++hd) sp[hd] = fmaf(sc.z, __uint_as_float(w2[hd]), sp[hd]);
          }
        } else {
          tmem_ld16(tmem + lane_base + kColS + kSBuf * s, w);
          tmem_wait_ld();
#pragma unroll
          for (int hd = 0; hd < kN; ++hd) sp[hd] = __uint_as_float(w[hd]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty + s));
      // Exchange: stage the row, one bulk copy of all 128 rows to the peer.
      named_bar_sync(2, kSoftmax);           // the staging buffer is free
      {
        uint8_t* srow = sm + kOffXs + xrow;
#pragma unroll
        for (int c = 0; c < kN / 4; ++c)
          *reinterpret_cast<float4*>(srow + ((((uint32_t)c) ^ xsw) << 4)) =
              make_float4(sp[4 * c], sp[4 * c + 1], sp[4 * c + 2], sp[4 * c + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(2, kSoftmax);           // all rows staged
      if (leader) {
        if (b >= 2) W.wait(bar(kBarXFree + s), ((b >> 1) - 1) & 1);
        bulk_copy_to_peer(x_peer + s * kXBytes, sb + kOffXs, (uint32_t)kXBytes,
                          xfull_peer + 8u * s);
        bulk_commit_group();
      }
      W.wait_cluster(bar(kBarXFull + s), (b >> 1) & 1);
      {
        const uint8_t* xr = sm + kOffX + s * kXBytes + xrow;
#pragma unroll
        for (int c = 0; c < kN / 4; ++c) {
          const float4 x = *reinterpret_cast<const float4*>(xr + ((((uint32_t)c) ^ xsw) << 4));
          sp[4 * c] += x.x; sp[4 * c + 1] += x.y; sp[4 * c + 2] += x.z; sp[4 * c + 3] += x.w;
        }
      }
      mbar_arrive(bar(kBarXCons + s));       // the signal warp tells the peer

      // a5: masked scores (log2 units) and the lazy running max.
      const bool key_ok = ((masks[b * 4 + (i >> 5)] >> (i & 31)) & 1u) != 0u;
      bool need = false;
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) {
        sp[hd] = (key_ok && hd < p.h) ? sp[hd] * scale_log2 : -INFINITY;
        need |= sp[hd] > m_run[hd] + 8.f;
      }
      float alpha[kN];
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) alpha[hd] = 1.f;
      if (named_bar_or(3, kSoftmax, need)) {
        float bm[kN];
#pragma unroll
        for (int hd = 0; hd < kN; ++hd) bm[hd] = sp[hd];
        const float wmax = xreduce16<true>(bm, lane);
        if ((lane & 1) == 0) red[(lane >> 1) * 4 + (warp & 3)] = wmax;
        named_bar_sync(4, kSoftmax);
#pragma unroll
        for (int hd = 0; hd < kN; ++hd) {
          const float4 x = *reinterpret_cast<const float4*>(red + 4 * hd);
          const float bmax = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
          if (bmax > m_run[hd] + 8.f) {      // also true for the first finite max
            alpha[hd] = ex2_approx(m_run[hd] - bmax);   // 0 when m_run = -inf
            m_run[hd] = bmax;
          }
        }
      }
      float pe[kN];
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) {
        // The row sums use the unrounded values (they set the LSE); P goes to
        // the PV MMA in bf16.
        pe[hd] = m_run[hd] == -INFINITY ? 0.f : ex2_approx(sp[hd] - m_run[hd]);
        l_part[hd] = fmaf(l_part[hd], alpha[hd], pe[hd]);
      }
      // a6 operand: P^T into buffer b % kPBufs (group scales: p * scale of
      // each PV group as a bf16 pair hi + lo).
      const int pbi = b % kPBufs;
      if (b >= kPBufs) W.wait(bar(kBarPEmpty + pbi), ((b / kPBufs) - 1) & 1);  // PV read it
      if (kGroup) {
        // p * (group scale) = hi + lo, each bf16 (lo = the rounding error of
        // hi); the key's row is written as eight 16-byte chunks.
        uint8_t* prow = sm + kOffP + p_row;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const float scg = g ? scp1 : scp0;
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float v0 = pe[2 * k] * scg, v1 = pe[2 * k + 1] * scg;
            hi[k] = pack_bf16(v0, v1);
            lo[k] = pack_bf16(v0 - __uint_as_float(hi[k] << 16),
                              v1 - __uint_as_float(hi[k] & 0xFFFF0000u));
          }
          const uint32_t c0 = 4u * (uint32_t)g;
          *reinterpret_cast<uint4*>(prow + ((c0 ^ p_sw) << 4)) =
              make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(prow + (((c0 + 1u) ^ p_sw) << 4)) =
              make_uint4(hi[4], hi[5], hi[6], hi[7]);
          *reinterpret_cast<uint4*>(prow + (((c0 + 2u) ^ p_sw) << 4)) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(prow + (((c0 + 3u) ^ p_sw) << 4)) =
              make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
      } else {
        uint8_t* pb = sm + kOffP + pbi * kPBufBytes + p_atom;
#pragma unroll
        for (int hd = 0; hd < kN; ++hd) {
          const uint32_t off = (uint32_t)(hd >> 3) * 1024u + (uint32_t)(hd & 7) * 128u +
                               ((p_chunk ^ (uint32_t)(hd & 7)) << 4);
          *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(pe[hd]);
        }
      }
      fence_proxy_async_smem();
      bool rescale = false;
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) rescale |= alpha[hd] != 1.f;
      if (b >= 1 && __any_sync(0xffffffffu, rescale)) {
        // O^T row (channel i of both 128-channel blocks): column hd *= alpha[hd].
        W.wait(bar(kBarODone), (b - 1) & 1);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < (kGroup ? 4 : 2); ++c) {   // 16-column pieces (hi, lo)
          const uint32_t col = kColO + (kGroup ? kN * c : 2 * kN * c);
          uint32_t w[16];
          tmem_ld16(tmem + lane_base + col, w);
          tmem_wait_ld();
#pragma unroll
          for (int hd = 0; hd < kN; ++hd)
            w[hd] = __float_as_uint(__uint_as_float(w[hd]) * alpha[hd]);
          tmem_st16(tmem + lane_base + col, w);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + pbi));
    }

    // ---- a7: epilogue ---------------------------------------------------------
    // Row sums: reduce the per-key partial sums over the 128 keys.
    float* red2 = red + 4 * kN;
    float l[kN];
    {
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) l[hd] = l_part[hd];
      const float ws = xreduce16<false>(l, lane);
      if ((lane & 1) == 0) red2[(lane >> 1) * 4 + (warp & 3)] = ws;
      named_bar_sync(4, kSoftmax);
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) {
        const float4 x = *reinterpret_cast<const float4*>(red2 + 4 * hd);
        l[hd] = (x.x + x.y) + (x.z + x.w);
      }
    }
    if (nb > 0) {
      W.wait(bar(kBarOFinal), 0);
      tc_fence_after();
    }
    const float oscale = kFmt == kE4m3 ? kscale : 1.f;
    float inv[kN];
#pragma unroll
    for (int hd = 0; hd < kN; ++hd)
      inv[hd] = (!(l[hd] > 0.f) || nb == 0) ? 0.f : oscale / l[hd];
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      uint32_t w[16];
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) w[hd] = 0u;
      __syncwarp();
      if (nb > 0) {
        tmem_ld16(tmem + lane_base + kColO + 2 * kN * mb, w);
        if (kGroup) {                                   // O = hi part + lo part
          uint32_t w2[16];
          tmem_ld16(tmem + lane_base + kColO + 2 * kN * mb + kN, w2);
          tmem_wait_ld();
#pragma unroll
          for (int hd = 0; hd < kN; ++hd)
            w[hd] = __float_as_uint(__uint_as_float(w[hd]) + __uint_as_float(w2[hd]));
        }
        tmem_wait_ld();
      }
      const int ch = g_lo + 128 * mb + i;            // output channel of lane i
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) {
        if (hd < p.h) {
          const float o = inv[hd] == 0.f ? 0.f : __uint_as_float(w[hd]) * inv[hd];
          const int64_t orow = (int64_t)t * p.h + hd;
          if (p.fp32_out)
            p.o_part[((int64_t)split * p.T * p.h + orow) * p.d_v + ch] = o;
          else
            reinterpret_cast<__nv_bfloat16*>(p.out)[orow * p.d_v + ch] = __float2bfloat16_rn(o);
        }
      }
    }
    // Both CTAs hold the same LSE; CTA 0 writes it (thread i -> head i).
    if (r == 0 && i < p.h) {
      float mi = -INFINITY, li = 0.f;
#pragma unroll
      for (int hd = 0; hd < kN; ++hd)
        if (hd == i) { mi = m_run[hd]; li = l[hd]; }
      const bool empty = !(li > 0.f) || nb == 0;
      const float lse_v = empty ? -INFINITY : (mi + log2f(li)) * 0.69314718055994530942f;
      const int64_t orow = (int64_t)t * p.h + i;
      if (p.fp32_out)
        p.lse_part[(int64_t)split * p.T * p.h + orow] = lse_v;
      else if (p.lse)
        p.lse[orow] = lse_v;
    }
  }

  // ---- teardown: no CTA leaves while its peer may still write into it -----
  if (leader && nb > 0) {
    bulk_wait_read_all();
    if (nb >= 2) W.wait(bar(kBarXFree + ((nb - 2) & 1)), ((nb - 2) >> 1) & 1);
    W.wait(bar(kBarXFree + ((nb - 1) & 1)), ((nb - 1) >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  cluster_arrive();
  cluster_wait();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kFmt>
cudaError_t launch_keys(const KeysArgs& a, unsigned blocks, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(smla_tc_keys_kernel<kFmt>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  smla_tc_keys_kernel<kFmt><<<blocks, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_keys_max_range() { return kMaxBlocks * kBK; }

bool tc_keys_supported(int h, int d_qk, int kv_format) {
  if (h < 1 || h > kN || (d_qk != 576 && d_qk != 512)) return false;
  if (kv_format == kDsMla || kv_format == kE4m3Group4Kpe) return d_qk == 576;
  return kv_format == kBf16 || kv_format == kE4m3 || kv_format == kE4m3Group;
}

cudaError_t launch_tc_keys(const FwdParams& p, cudaStream_t stream) {
  KeysArgs a{};
  a.p = p;
  if (p.kv_format == kBf16) {
    const cudaError_t e = encode_bf16_rows_map(&a.kv_map, p.kv, p.d_qk, p.num_slots);
    if (e != cudaSuccess) return e;
  }
  a.ksteps = p.d_qk == 576 ? 18 : 16;
  a.G = (p.d_qk + 127) / 128;
  a.scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t clusters = (int64_t)p.T * p.splits;
  if (clusters * 2 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const unsigned blocks = (unsigned)(clusters * 2);
  switch (p.kv_format) {
    case kBf16: return launch_keys<kBf16>(a, blocks, stream);
    case kE4m3: return launch_keys<kE4m3>(a, blocks, stream);
    case kE4m3Group: return launch_keys<kE4m3Group>(a, blocks, stream);
    case kDsMla: return launch_keys<kDsMla>(a, blocks, stream);
    default:    return launch_keys<kE4m3Group4Kpe>(a, blocks, stream);
  }
}

}  // namespace smla

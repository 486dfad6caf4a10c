// smla_tc_keys.cu — tensor-core (tcgen05 / TMEM) sparse MLA forward for up
// to 16 heads with a bf16 cache.  (E4M3 caches run on the E4M3-operand
// kernel of smla_tc_fp8.cu.)
//
// With few heads, the heads cannot fill a 128-row MMA, so this kernel turns
// both products around: the top-k positions (keys) of a block are the MMA's
// M dimension and the heads are N:
//   S^T[keys, heads] = K[keys, d] . Q^T[d, heads]         A = gathered tile, K-major
//   O^T[ch, heads]  += V^T[ch, keys] . P^T[keys, heads]    A = the same tile, MN-major
// One work unit = (query token, top-k range) on one CTA.  A block holds 64
// keys as 128 tile rows: row r is key r % 64 restricted to channel half
// h = r / 64, i.e. ckv channels [256h, 256h + 256) and, for d_qk = 576, the
// rope channels [512 + 32h, 544 + 32h).  So one M = 128 QK MMA covers the
// whole row of 64 keys.  Q^T is the N = 32 operand [16 heads of half 0 |
// 16 heads of half 1]; lane r of the score accumulator then holds, in the 16
// columns of its own half, key r % 64's partial scores over half h (the
// other 16 columns pair a key half with the other Q half and are ignored).
// The two halves of a key are summed through shared memory by the two
// threads that own them; no score crosses an SM.  PV: O^T is four
// 128-channel blocks; block c reads V^T from tile rows [64 (c / 2),
// 64 (c / 2) + 64).
// Thread t of the softmax warpgroup owns tile row t (TMEM lane t): key
// t % 64 and heads [8 (t / 64), 8 (t / 64) + 8).  The per-head max over the
// block's keys is reduced only when some score passes the running max by
// more than 2^8 (a one-barrier vote otherwise); each thread keeps partial
// row sums for its own key, reduced once at the end.
//
// Method steps (vLLM "Sparse MLA on Hopper" diff, ops/cutlass_fa3.py docstring:
// score = q_rope.k_rope + q_nope.c_kv, output = softmax(score*scale) @ c_kv;
// flashinfer_mla_sparse_sm90.py, forward_mqa: compacted valid prefix with -1
// past it; vLLM API docs flashmla_sparse, _forward_fp8_kv_mixed_batch: empty
// rows give (O = 0, LSE = -inf)):
//   a1 work setup: v = min(valid_len[t], topk); range [k0, k1) of the split
//   a2 gather: slot ids -> 128-byte-swizzled bf16 tiles (TMA tile::gather4);
//      masked keys are zero
//   a4 QK^T, a5 masked online softmax, a6 PV, a7 O / l and LSE = m + ln l
//
// Warp roles (320 threads): warp 0 issues the QK MMAs and owns TMEM; warp 9
// issues the PV MMAs; warps 1..4 load the unit's slot ids, then gather with
// TMA; warps 5..8 (thread <-> tile row <-> TMEM lane) load Q, combine the
// halves, run the softmax, the O rescale and the epilogue.
// Every wait is bounded; a wait that runs out records a timeout status, sets
// an abort flag that skips later waits, and the block drains its copies and
// MMAs and finishes normally.
#include <math.h>

#include "smla_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kBK = 64;                    // top-k positions per block
constexpr int kRows = 128;                 // tile rows: 64 keys x 2 channel halves (MMA M)
constexpr int kN = 16;                     // heads, zero-padded
constexpr int kNq = 32;                    // QK N: 16 heads x 2 Q halves
constexpr int kStages = 2;                 // gathered-tile pipeline depth
constexpr int kChunkBytes = kRows * 128;   // 64 channels x 128 rows, bf16
constexpr int kMaxChunks = 5;              // 256 ckv + the rope chunk per row
constexpr int kStageBytes = kMaxChunks * kChunkBytes;
constexpr int kQChunkBytes = kNq * 128;    // 64 channels x 32 Q rows
constexpr int kPPlaneBytes = kBK * 128;    // P^T: 64 keys x 128 bytes
constexpr int kPAreaBytes = 2 * kPPlaneBytes;
constexpr int kCombBytes = kRows * 32;     // 8 partial scores per row
constexpr int kThreads = 320;
constexpr int kProducers = 128;            // warps 1..4
constexpr int kSoftmax = 128;              // warps 5..8
constexpr int kMaxBlocks = 32;             // ranges up to 2048 positions

// TMEM columns.
constexpr uint32_t kColO = 0;              // O^T: 4 blocks of 128 channels x 32 (16 used)
constexpr uint32_t kColS = 128;            // S: 2 buffers x 32
constexpr uint32_t kSBuf = kNq;
constexpr uint32_t kTmemCols = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffQ = kOffTile + kStages * kStageBytes;
constexpr uint32_t kOffP = kOffQ + kMaxChunks * kQChunkBytes;      // P^T
constexpr uint32_t kOffComb = kOffP + kPAreaBytes;                 // [2][128 rows][8] f32
constexpr uint32_t kOffSlot = kOffComb + 2 * kCombBytes;           // [blocks*64] i32
constexpr uint32_t kOffMask = kOffSlot + kMaxBlocks * kBK * 4;     // [blocks][2] u32
constexpr uint32_t kOffRed = kOffMask + kMaxBlocks * 8;            // [16 heads][4 warps] f32
constexpr uint32_t kOffHead = kOffRed + kN * 4 * 4;                // [4][16] f32: alpha, l, m, l~
constexpr uint32_t kOffBar = kOffHead + 4 * kN * 4;
enum {
  kBarKvFull = 0,                   // [2]
  kBarKvEmpty = kBarKvFull + 2,     // [2]
  kBarSFull = kBarKvEmpty + 2,      // [2]
  kBarSEmpty = kBarSFull + 2,       // [2]
  kBarPFull = kBarSEmpty + 2,       // [2 P buffers]
  kBarPEmpty = kBarPFull + 2,       // [2 P buffers]
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
static_assert(kOffComb % 16 == 0 && kOffBar % 8 == 0, "alignment");
static_assert(kColS + 2 * kSBuf <= kTmemCols, "TMEM budget");

struct KeysArgs {
  CUtensorMap kv_map;  // bf16 cache as a 2-D tensor, 64-channel boxes
  FwdParams p;
  int ksteps;          // 16-channel QK steps per half row: 18 (d_qk 576) or 16 (512)
  float scale_log2;    // sm_scale * log2(e)
};

// Reduce v[0..7] (one value per head) over the 32 lanes of the warp.  Each
// step hands half of the remaining heads to the partner lane, so lane l ends
// with the result for head (l >> 1) & 7 (14 shuffles instead of 40).
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

// kLpt: the units are taken longest first (lpt_unit); a separate instance,
// so that launches in unit order carry none of its code.
template <bool kLpt>
__global__ void __launch_bounds__(kThreads, 1)
smla_tc_keys_kernel(const __grid_constant__ KeysArgs a) {
  constexpr int kPBufs = 2;                 // P^T double-buffered
  constexpr int kNpv = kN;                  // PV MMA N
  extern __shared__ uint8_t smem_raw[];
  const FwdParams& p = a.p;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;           // shared address base
  uint8_t* sm = smem_raw + (sb - raw);                  // generic pointer base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- a1: work unit ------------------------------------------------------
  // (kLpt: the units are taken longest first; the slot-id area is the
  // scratch, before it is filled)
  int unit = (int)blockIdx.x;
  if (kLpt) unit = lpt_unit(p, unit, p.T * p.splits, kBK, reinterpret_cast<int*>(sm + kOffSlot));
  const int split = unit % p.splits;
  const int t = unit / p.splits;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);
  // The host plan keeps every range within kMaxBlocks blocks.
  const int nb = k1 > k0 ? min((k1 - k0 + kBK - 1) / kBK, kMaxBlocks) : 0;
  // Local channels of a half row: steps 0..15 = ckv [256h, 256h + 256);
  // steps 16, 17 (d_qk 576) = rope [512 + 32h, 544 + 32h), held in chunk 4.
  const int ksteps = a.ksteps;

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W = make_waiter(abort_flag, p);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 4);           // one expect_tx per TMA warp
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), kSoftmax);
      mbar_init(bar(kBarPFull + i), kSoftmax);
      mbar_init(bar(kBarPEmpty + i), 1);
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
    if (warp <= 2) {
      const int key = (warp - 1) * 32 + lane;
      for (int b = 0; b < nb; ++b) {
        const uint32_t m = __ballot_sync(0xffffffffu, slots[b * kBK + key] >= 0);
        if (lane == 0) masks[b * 2 + (warp - 1)] = m;
      }
    }
  }
  __syncthreads();

  if (warp == 0 || warp == 9) {
    // ---- MMA issuers: warp 0 issues QK, warp 9 issues PV --------------------
    // Two warps, each blocked only on its own inputs, so neither kind of
    // batch waits behind the other.  Each warp runs its code warp-uniformly;
    // one elected lane issues a batch of MMAs and commits it (a commit
    // tracks the MMAs of the issuing thread).
    if (nb > 0) {
      const uint32_t id_qk = idesc_bf16(128, kNq, false, false);
      const uint32_t id_pv = idesc_bf16(128, kNpv, true, true);
      if (warp == 0) {
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
            fence_proxy_async_smem();
            // A = the 128 tile rows, K-major; B = the 32 Q rows, K-major.  A
            // descriptor's start-address field is addr >> 4 in its low bits,
            // so each step's descriptor is the base plus a constant.
            const uint64_t a0 = sdesc(tile, 16, 1024, kLayoutSw128);
            const uint64_t b0 = sdesc(qb, 16, 1024, kLayoutSw128);
#pragma unroll
            for (int ks = 0; ks < 18; ++ks) {
              if (ks < ksteps) {
                const uint32_t oa = (uint32_t)((ks >> 2) * kChunkBytes + (ks & 3) * 32);
                const uint32_t ob = (uint32_t)((ks >> 2) * kQChunkBytes + (ks & 3) * 32);
                mma_ss(dS, a0 + (oa >> 4), b0 + (ob >> 4), id_qk, ks == 0 ? 0u : 1u);
              }
            }
            mma_commit(bar(kBarSFull + s));
          }
          __syncwarp();
        }
      } else {
        for (int j = 0; j < nb; ++j) {
          const int s = j & 1;
          const int pbi = j % kPBufs;
          W.wait(bar(kBarPFull + pbi), (j / kPBufs) & 1);
          __syncwarp();
          tc_fence_after();
          const uint32_t tile = sb + kOffTile + s * kStageBytes;
          const uint32_t pb = sb + kOffP + pbi * kPPlaneBytes;
          if (elect_one()) {
            fence_proxy_async_smem();
            // A = V^T of channel block c: 128 channels (two 64-channel
            // chunks) x 16 keys, MN-major, from tile rows [64 (c / 2), +64);
            // B = P^T: 16 keys x N, MN-major.
            const uint64_t a0 = sdesc(tile, kChunkBytes, 1024, kLayoutSw128);
            const uint64_t b0 = sdesc(pb, kPAreaBytes, 1024, kLayoutSw128);
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
              for (int ks = 0; ks < kBK / 16; ++ks) {
                const uint32_t oa =
                    (uint32_t)(2 * (c & 1) * kChunkBytes + (64 * (c >> 1) + 16 * ks) * 128);
                const uint32_t ob = (uint32_t)(ks * 2048);
                mma_ss(tmem + kColO + 32u * (uint32_t)c, a0 + (oa >> 4), b0 + (ob >> 4), id_pv,
                       ks > 0 ? 1u : acc0);
              }
            }
            mma_commit(bar(kBarODone));
            mma_commit(bar(kBarPEmpty + pbi));
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
    // ---- loaders: a2 gather (+ a3 E4M3 conversion) -------------------------
    // Loader warp wl = warp - 1 owns tile rows [32 wl, 32 wl + 32): keys
    // [32 (wl % 2), +32) of every block, in channel half wl / 2.
    const int wl = warp - 1;
    const int half = wl >> 1;
    const int w0 = 32 * wl;                               // the warp's first tile row
    const int kb0 = w0 & (kBK - 1);                       // and its first key
    const int g_lo = 256 * half;                          // first ckv channel of the half
    const int rope_lo = 512 + 32 * half;                  // first rope channel of the half
    {
      // bf16: warp wl issues the 8 four-row groups of its 32 tile rows.
      const int n_boxes = ksteps > 16 ? 5 : 4;               // + one rope box
      const uint32_t tx_bytes = (uint32_t)(8 * n_boxes * 512);
      int issued = 0;
      for (int b = 0; b < nb; ++b) {
        const int s = b & 1;
        if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b >> 1) - 1) & 1);
        if (*abort_flag) break;                  // the stage may still be in use
        __syncwarp();
        issued = b + 1;
        if (elect_one()) {
          const uint32_t full = bar(kBarKvFull + s);
          mbar_arrive_expect_tx(full, tx_bytes);
          const uint32_t tile = sb + kOffTile + s * kStageBytes;
          const int* bs = slots + b * kBK + kb0;
          for (int g = 0; g < 8; ++g) {
            const int y0 = bs[4 * g], y1 = bs[4 * g + 1], y2 = bs[4 * g + 2], y3 = bs[4 * g + 3];
            // (the rope box of half 1 runs past the row end: zero fill)
            for (int c = 0; c < n_boxes; ++c)
              tma_gather4(tile + c * kChunkBytes + (w0 + 4 * g) * 128, &a.kv_map,
                          c < 4 ? g_lo + 64 * c : rope_lo, y0, y1, y2, y3, full);
          }
        }
        __syncwarp();
      }
      // Teardown: the gathers of the last block issued into each stage have
      // landed (see the heads-major kernel's producers).
      if (lane == 0) {
        for (int b = issued - 1; b >= 0 && b >= issued - kStages; --b)
          W.drain(bar(kBarKvFull + (b & 1)), (b >> 1) & 1);
      }
      __syncwarp();
    }
  } else if (warp <= 8) {
    // ---- softmax warpgroup (thread <-> tile row <-> TMEM lane) ---------------
    const int q4 = warp & 3;                            // TMEM lane quarter
    const int row = 32 * q4 + lane;                     // tile row == TMEM lane
    const int hf = row >> 6;                            // channel half; heads [8 hf, 8 hf + 8)
    const int key = row & (kBK - 1);
    const int partner = row ^ 64;                       // the other half of the key
    const uint32_t lane_base = ((uint32_t)q4 * 32u) << 16;
    // Q -> the QK B operand: row n = head n % 16 with channel half n / 16
    // (heads >= h zero); K-major, 64-channel chunks of 32 rows x 128 B,
    // 128-byte swizzle.
    {
      const int per_row = 2 * ksteps;                   // 16-byte pieces per Q row
      const int total = kNq * per_row;                  // <= 1152
      uint4 qv[9];
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        const int idx = row + kSoftmax * k;
        const int n = idx / per_row, c16 = idx - n * per_row;
        const int hd = n & 15, qh = n >> 4;
        const int ch = c16 < 32 ? 256 * qh + 8 * c16 : 512 + 32 * qh + 8 * (c16 - 32);
        qv[k] = (idx < total && hd < p.h) ? __ldg(q_chunk(p, t, hd, ch))
                                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        const int idx = row + kSoftmax * k;
        if (idx < total) {
          const int n = idx / per_row, c16 = idx - n * per_row;
          *reinterpret_cast<uint4*>(sm + kOffQ + (c16 >> 3) * kQChunkBytes + (n >> 3) * 1024 +
                                    (n & 7) * 128 + (((c16 & 7) ^ (n & 7)) << 4)) = qv[k];
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQReady));
    }
    const float scale_log2 = a.scale_log2;
    // l_part: row sums of the unrounded P (they set the LSE); lr_part: of
    // the bf16-rounded P that PV multiplies (they divide O, so that where
    // one key carries a row its rounded weight cancels: the lazy running max
    // leaves that weight anywhere in (1, 2^8], where bf16 is off by up to
    // 2^-8 of it).
    float m_run[8], l_part[8], lr_part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { m_run[i] = -INFINITY; l_part[i] = 0.f; lr_part[i] = 0.f; }
    float* red = reinterpret_cast<float*>(sm + kOffRed);   // [16 heads][4 warps]
    float* hsh = reinterpret_cast<float*>(sm + kOffHead);  // [alpha | l | m | l~][16 heads]
    // This key's 128-byte row in a P^T plane (MN-major, 128-byte swizzle):
    // atom key / 8, row key % 8, 16-byte chunk c at c ^ (key % 8).
    const uint32_t p_row = (uint32_t)(key >> 3) * 1024u + (uint32_t)(key & 7) * 128u;
    const uint32_t p_sw = (uint32_t)(key & 7);

    for (int b = 0; b < nb; ++b) {
      const int s = b & 1;
      float part[16];                      // this half's partial scores, heads 0..15
      W.wait(bar(kBarSFull + s), (b >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      {
        // This lane's half: the 16 columns of each accumulator that pair it
        // with the Q rows of the same half.
        const uint32_t sc0 = tmem + lane_base + kColS + kSBuf * s + 16u * (uint32_t)hf;
        uint32_t w[16];
        tmem_ld16(sc0, w);
        tmem_wait_ld();
#pragma unroll
        for (int hd = 0; hd < kN; ++hd) part[hd] = __uint_as_float(w[hd]);
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty + s));
      // Combine the key's two halves: hand the partner its 8 heads of this
      // half's partial scores, then add the partner's share of ours.
      float sp[8];
      {
        float* cb = reinterpret_cast<float*>(sm + kOffComb + s * kCombBytes);
        float give[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          give[i] = hf ? part[i] : part[8 + i];
          sp[i] = hf ? part[8 + i] : part[i];
        }
        *reinterpret_cast<float4*>(cb + row * 8) = make_float4(give[0], give[1], give[2], give[3]);
        *reinterpret_cast<float4*>(cb + row * 8 + 4) =
            make_float4(give[4], give[5], give[6], give[7]);
        named_bar_sync(2, kSoftmax);
        const float4 x0 = *reinterpret_cast<const float4*>(cb + partner * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(cb + partner * 8 + 4);
        sp[0] += x0.x; sp[1] += x0.y; sp[2] += x0.z; sp[3] += x0.w;
        sp[4] += x1.x; sp[5] += x1.y; sp[6] += x1.z; sp[7] += x1.w;
      }

      // a5: masked scores (log2 units) and the lazy running max.
      const bool key_ok = ((masks[b * 2 + (key >> 5)] >> (key & 31)) & 1u) != 0u;
      bool need = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sp[i] = (key_ok && 8 * hf + i < p.h) ? sp[i] * scale_log2 : -INFINITY;
        need |= sp[i] > m_run[i] + 8.f;
      }
      float alpha[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) alpha[i] = 1.f;
      const bool voted = named_bar_or(3, kSoftmax, need);
      if (voted) {
        float bm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) bm[i] = sp[i];
        const float wmax = xreduce8<true>(bm, lane);
        if ((lane & 17) == 0) red[(8 * hf + ((lane >> 1) & 7)) * 4 + q4] = wmax;
        named_bar_sync(4, kSoftmax);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(red + 4 * (8 * hf + i));
          const float bmax = hf ? fmaxf(x.z, x.w) : fmaxf(x.x, x.y);
          if (bmax > m_run[i] + 8.f) {       // also true for the first finite max
            alpha[i] = ex2_approx(m_run[i] - bmax);   // 0 when m_run = -inf
            m_run[i] = bmax;
          }
        }
        // Every head's alpha, for the O rescale (O^T lanes are channels).
        if (key == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) hsh[8 * hf + i] = alpha[i];
        }
        named_bar_sync(4, kSoftmax);
      }
      float pe[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pe[i] = m_run[i] == -INFINITY ? 0.f : ex2_approx(sp[i] - m_run[i]);
        l_part[i] = fmaf(l_part[i], alpha[i], pe[i]);
      }
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pk[k] = pack_bf16(pe[2 * k], pe[2 * k + 1]);
        lr_part[2 * k] = fmaf(lr_part[2 * k], alpha[2 * k], __uint_as_float(pk[k] << 16));
        lr_part[2 * k + 1] =
            fmaf(lr_part[2 * k + 1], alpha[2 * k + 1], __uint_as_float(pk[k] & 0xFFFF0000u));
      }
      // a6 operand: P^T into buffer b % kPBufs.
      const int pbi = b % kPBufs;
      if (b >= kPBufs) W.wait(bar(kBarPEmpty + pbi), ((b / kPBufs) - 1) & 1);  // PV read it
      {
        uint8_t* prow = sm + kOffP + pbi * kPPlaneBytes + p_row;
        *reinterpret_cast<uint4*>(prow + (((uint32_t)hf ^ p_sw) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async_smem();
      if (voted && b >= 1) {
        // O^T row (channel `row` of each 128-channel block): column hd *=
        // alpha[hd].  The same decision in every thread (uniform).
        float al[kN];
        bool rescale = false;
#pragma unroll
        for (int hd = 0; hd < kN; ++hd) {
          al[hd] = hsh[hd];
          rescale |= al[hd] != 1.f;
        }
        if (rescale) {
          W.wait(bar(kBarODone), (b - 1) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {                  // the 16 head columns of block c
            const uint32_t col = kColO + 32u * (uint32_t)c;
            uint32_t w[16];
            tmem_ld16(tmem + lane_base + col, w);
            tmem_wait_ld();
#pragma unroll
            for (int hd = 0; hd < kN; ++hd)
              w[hd] = __float_as_uint(__uint_as_float(w[hd]) * al[hd]);
            tmem_st16(tmem + lane_base + col, w);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + pbi));
    }

    // ---- a7: epilogue ---------------------------------------------------------
    // Row sums: reduce the per-key partial sums over the 64 keys of each
    // half; publish l and m of every head.
    {
      float l8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) l8[i] = l_part[i];
      const float ws = xreduce8<false>(l8, lane);
      named_bar_sync(4, kSoftmax);           // (red may still be read by a vote)
      if ((lane & 17) == 0) red[(8 * hf + ((lane >> 1) & 7)) * 4 + q4] = ws;
      named_bar_sync(4, kSoftmax);
      if (key == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(red + 4 * (8 * hf + i));
          hsh[kN + 8 * hf + i] = hf ? x.z + x.w : x.x + x.y;
          hsh[2 * kN + 8 * hf + i] = m_run[i];
        }
      }
      named_bar_sync(4, kSoftmax);
      // the same for the sums of the rounded P
#pragma unroll
      for (int i = 0; i < 8; ++i) l8[i] = lr_part[i];
      const float wr = xreduce8<false>(l8, lane);
      if ((lane & 17) == 0) red[(8 * hf + ((lane >> 1) & 7)) * 4 + q4] = wr;
      named_bar_sync(4, kSoftmax);
      if (key == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(red + 4 * (8 * hf + i));
          hsh[3 * kN + 8 * hf + i] = hf ? x.z + x.w : x.x + x.y;
        }
      }
      named_bar_sync(4, kSoftmax);
    }
    if (nb > 0) {
      W.wait(bar(kBarOFinal), 0);
      tc_fence_after();
    }
    float inv[kN];
#pragma unroll
    for (int hd = 0; hd < kN; ++hd) {
      const float l = hsh[kN + hd];
      inv[hd] = (l == 0.f || nb == 0) ? 0.f : __fdividef(1.f, hsh[3 * kN + hd]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int hd = 0; hd < kN; ++hd) w[hd] = 0u;
      __syncwarp();
      if (nb > 0) {
        tmem_ld16(tmem + lane_base + kColO + 32u * (uint32_t)c, w);
        tmem_wait_ld();
      }
      const int ch = 128 * c + row;                   // output channel of lane `row`
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
    // Thread `row` < h writes head row's LSE.
    if (row < p.h) {
      const float mi = hsh[2 * kN + row], li = hsh[kN + row];
      const bool empty = li == 0.f || nb == 0;   // (a NaN row sum is not empty)
      const float lse_v = empty ? -INFINITY : (mi + log2f(li)) * 0.69314718055994530942f;
      const int64_t orow = (int64_t)t * p.h + row;
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

cudaError_t launch_keys(const KeysArgs& a, unsigned blocks, cudaStream_t stream) {
  const bool lpt = a.p.lpt && blocks <= (unsigned)kLptMaxUnits;
  auto kernel = lpt ? smla_tc_keys_kernel<true> : smla_tc_keys_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<blocks, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_keys_max_range() { return kMaxBlocks * kBK; }

bool tc_keys_supported(int h, int d_qk, int kv_format) {
  return h >= 1 && h <= kN && (d_qk == 576 || d_qk == 512) && kv_format == kBf16;
}

cudaError_t launch_tc_keys(const FwdParams& p, cudaStream_t stream) {
  KeysArgs a{};
  a.p = p;
  if (p.kv_format != kBf16) return cudaErrorInvalidValue;   // (the plan sends only bf16)
  const cudaError_t e = encode_bf16_rows_map(&a.kv_map, p.kv, p.d_qk, p.num_slots);
  if (e != cudaSuccess) return e;
  a.ksteps = p.d_qk == 576 ? 18 : 16;
  a.scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t blocks = (int64_t)p.T * p.splits;    // one CTA per unit
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  return launch_keys(a, (unsigned)blocks, stream);
}

}  // namespace smla

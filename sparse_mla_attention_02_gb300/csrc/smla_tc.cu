// smla_tc.cu — tensor-core (tcgen05 / TMEM) sparse MLA forward for sm_103a.
//
// One work unit = (query token t, top-k position range) and runs on a cluster
// of two CTAs (a pair of SMs).  Why two: for h = 128 heads the fp32 output
// accumulator O[128, 512] alone fills the 512 TMEM columns of one SM, and an
// M = 64 MMA runs at half rate.  So the pair splits the work so that every MMA
// is M = 128 (all heads):
//   * QK^T is split over d_qk: CTA r keeps Q[:, its half of d_qk] in TMEM
//     (the MMA's A operand) and computes partial scores S_r = Q_r K_r^T
//     [128 heads x 48 keys] per block of 48 top-k positions;
//   * each CTA sends its partial S to the other with bulk copies (one per
//     softmax warpgroup, counted on the receiver's mbarrier), so both hold
//     S = S_0 + S_1 and run the same softmax for all 128 heads (identical
//     inputs, identical results);
//   * PV is split over d_v: CTA r accumulates O[:, 256r : 256r+256] in TMEM
//     from its P [128 x 48] and the first 512 channels of the same gathered
//     rows (V is the prefix of K).
// Pipelining: partial S is double-buffered in TMEM; the MMA thread issues QK
// two blocks ahead of PV; the softmax warps read and send block b+1's partial
// scores before they finish block b, which hides the exchange latency.
//
// Method steps (vLLM "Sparse MLA on Hopper" diff, ops/cutlass_fa3.py docstring:
// score = q_rope.k_rope + q_nope.c_kv, output = softmax(score*scale) @ c_kv;
// flashinfer_mla_sparse_sm90.py, forward_mqa: compacted valid prefix with -1
// past it; vLLM API docs flashmla_sparse, _forward_fp8_kv_mixed_batch: empty
// rows give (O = 0, LSE = -inf)):
//   a1 work setup: v = min(valid_len[t], topk); range [k0, k1) of the split
//   a2 gather: slot ids -> rows of the cache into a 128-byte-swizzled tile
//      with TMA tile::gather4 (masked positions read the out-of-bounds
//      zero fill and get -inf scores)
//   a4 QK^T (tcgen05.mma, A = Q from TMEM, B = K tile, K-major)
//   a5 masked online softmax in registers (one thread per head row), running
//      max updated lazily (O is rescaled only when the max grows by > 2^8)
//   a6 PV (tcgen05.mma, A = P from shared memory, B = V tile, MN-major)
//   a7 epilogue: O / l -> bf16 out (or fp32 partials), LSE = m + ln l
//
// Warp roles (416 threads): warp 0 issues MMAs (warp-uniform code, one
// elected lane per batch of MMAs) and owns TMEM; warps 1..3 load the unit's
// slot ids, then gather with TMA; warps 4..7 and 8..11 are two softmax
// warpgroups (thread i <-> TMEM lane i <-> head i; positions 0..23 and 24..47
// of each block), which move Q to TMEM and run the exchange, softmax, O
// rescale and the epilogue; warp 12 signals the peer when its partial scores
// were consumed.
// Q reaches TMEM from shared memory for bf16 caches: with 128 heads and q in
// one tensor, the CTA's Q half arrives as TMA boxes issued by the thread
// that sets up the barriers; otherwise the softmax threads copy it with
// coalesced loads before the set-up.  Either way it is staged in gather
// stages 1..3, which the producers fill only after the rows were read.  With
// E4M3 caches each softmax thread loads its head's row from global memory.
// Launches with more units than clusters (and at most 4096 units) take the
// units longest first (lpt_unit, the kLpt instance).
// Every wait is bounded; a wait that runs out records a timeout status, sets
// an abort flag that skips later waits, and the block finishes normally.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "smla_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kBN = 48;                    // top-k positions per block
constexpr int kStages = 4;                 // gathered-tile pipeline depth
constexpr int kAtomBytes = kBN * 128;      // 48 rows x 128 B (64 channels)
constexpr int kTileBytes = 5 * kAtomBytes; // up to 320 channels per CTA
constexpr int kPBytes = 128 * 128;         // P: 128 rows x 64 bf16 (48 used)
// Exchanged partial scores: two halves (positions 0..23 and 24..47, one per
// softmax warpgroup), each 128 rows x 24 fp32 = 96 bytes per row; the 16-byte
// chunk c of row i sits at position c ^ ((i >> 2) & 1), which keeps a warp's
// row accesses free of bank conflicts.
constexpr int kXHalfBytes = 128 * (kBN / 2) * 4;
constexpr int kXBytes = 2 * kXHalfBytes;
constexpr int kThreads = 416;            // 12 role warps + 1 signal warp
constexpr int kProducers = 96;             // warps 1..3 (slot-id prefetch)

// TMEM columns.
constexpr uint32_t kColO = 0;              // O half: 256 columns
constexpr uint32_t kColQ = 256;            // Q half: up to 144 columns
constexpr uint32_t kColS = 400;            // partial S: 2 x 48 columns
constexpr uint32_t kTmemCols = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffP = kOffTile + kStages * kTileBytes;   // one P buffer
constexpr uint32_t kOffX = kOffP + kPBytes;                    // receive [2]
constexpr uint32_t kOffXs = kOffX + 2 * kXBytes;               // send staging
constexpr int kMaxBlocks = 64;             // covers topk <= 3072 in one range
constexpr uint32_t kOffSlot = kOffXs + kXBytes;                 // [blocks*48] i32
constexpr uint32_t kOffMask = kOffSlot + kMaxBlocks * kBN * 4;  // [blocks][2] u32
constexpr uint32_t kOffRed = kOffMask + kMaxBlocks * 8;         // [2][2][128] f32 half maxima
constexpr uint32_t kOffL = kOffRed + 2 * 2 * 128 * 4;            // [2][2][128] f32 row sums
constexpr uint32_t kOffBar = (kOffL + 2 * 2 * 128 * 4 + 7) & ~7u;
enum {
  kBarKvFull = 0,
  kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,   // [2]
  kBarSEmpty = kBarSFull + 2,          // [2]
  kBarPFull = kBarSEmpty + 2,
  kBarPEmpty,
  kBarXFull,                           // [2 buffers][2 halves]
  kBarXFree = kBarXFull + 4,           // [2]
  kBarXCons = kBarXFree + 2,           // [2]
  kBarODone = kBarXCons + 2,
  kBarOFinal,                          // one phase: the unit's last PV is done
  kBarQReady,
  kBarQStaged,                         // the staged Q rows have been read
  kBarQLoaded,                         // the Q boxes have landed (TMA staging)
  kBarDrain,                           // teardown: the MMA warp's MMAs are done
  kNumBars
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kColS + 2 * kBN <= kTmemCols, "TMEM budget");
static_assert(kAtomBytes % 1024 == 0, "swizzle atoms must stay 1024-aligned");
static_assert(kBN % 12 == 0, "three producer warps split the 4-row groups evenly");
// Q staging: the CTA's Q half as 128 rows of up to 288 channels (row stride
// 592 bytes), in gather stages 1..3, which are idle until Q is in TMEM.
constexpr uint32_t kQStageRow = 592;
constexpr uint32_t kOffQStage = kOffTile + kTileBytes;
static_assert(kOffQStage + 128 * kQStageRow <= kOffTile + kStages * kTileBytes, "Q staging");

struct TcArgs {
  CUtensorMap kv_map;  // bf16 cache as a 2-D tensor [num_slots, d_qk], 64-channel boxes
  CUtensorMap q_map;   // q as a 2-D tensor [T * 128, d_qk], 64-channel x 128-row boxes
  CUtensorMap o_map;   // out as a 2-D tensor [T * 128, 512], 64-channel x 128-row boxes
  int q_tma;           // 1: Q staged by TMA boxes (bf16 cache, h = 128, q concatenated)
  int o_tma;           // 1: O leaves by TMA boxes (h = 128, bf16 out)
  FwdParams p;
  int fp8;          // 1: E4M3 cache with a per-tensor scale (converted on load)
  int g_lo[2];      // first cache channel gathered by CTA r
  int n_boxes[2];   // 64-channel boxes gathered per row by CTA r (bf16)
  int n_chunks8[2]; // 16-byte FP8 chunks gathered per row by CTA r (fp8)
  int qk_lo[2];     // first local channel of CTA r's QK range
  int q_lo[2];      // first q channel CTA r keeps in TMEM
  int ksteps;       // 16-channel MMA steps of the QK half
  float scale_log2; // sm_scale * log2(e)
};

// kLpt: the units are taken longest first (lpt_unit); a separate instance,
// so that launches in unit order carry none of its code.
template <bool kLpt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
smla_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const FwdParams& p = a.p;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;           // shared address base
  uint8_t* sm = smem_raw + (sb - raw);                  // generic pointer base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t r = cluster_ctarank();
  const uint32_t peer = r ^ 1u;

  // ---- a1: work unit ------------------------------------------------------
  // (kLpt: the units are taken longest first; the slot-id area is the
  // scratch, before it is filled)
  int unit = (int)(blockIdx.x >> 1);
  if (kLpt) unit = lpt_unit(p, unit, p.T * p.splits, kBN, reinterpret_cast<int*>(sm + kOffSlot));
  const int split = unit % p.splits;
  const int t = unit / p.splits;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);
  // The host plan keeps every range within kMaxBlocks blocks.
  const int nb = k1 > k0 ? min((k1 - k0 + kBN - 1) / kBN, kMaxBlocks) : 0;

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W = make_waiter(abort_flag, p);

  // Q half, first step (bf16 caches): the 256 softmax threads copy the
  // CTA's Q half (128 heads x 2 * ksteps 16-byte pieces) into the staging
  // rows, consecutive threads on consecutive pieces of a head row
  // (coalesced), before the set-up below; heads >= h are zero.  The rows go
  // to TMEM after it.  (E4M3 caches load Q per head after the set-up: their
  // converters fill stages 1..3 early, and staging measured slower there.)
  if (!a.fp8 && !a.q_tma && warp >= 4 && warp <= 11) {
    const int st = tid - 128;
    const int per_row = 2 * a.ksteps;                     // 36 or 32 pieces
#pragma unroll
    for (int k0 = 0; k0 < 18; k0 += 9) {                 // two batches of 9 loads
      uint4 qv[9];
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        const int e = st + 256 * (k0 + k), hd = e / per_row, c16 = e - hd * per_row;
        qv[k] = (hd < p.h && e < 128 * per_row)
                    ? __ldg(q_chunk(p, t, hd, a.q_lo[r] + 8 * c16))
                    : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        const int e = st + 256 * (k0 + k), hd = e / per_row, c16 = e - hd * per_row;
        if (e < 128 * per_row)
          *reinterpret_cast<uint4*>(sm + kOffQStage + hd * kQStageRow + 16 * c16) = qv[k];
      }
    }
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // bf16: one expect_tx per TMA warp; fp8: one arrival per converter thread
      mbar_init(bar(kBarKvFull + s), a.fp8 ? kProducers : 3);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), 256);
      mbar_init(bar(kBarXFull + 2 * i), 1);
      mbar_init(bar(kBarXFull + 2 * i + 1), 1);
      mbar_init(bar(kBarXFree + i), 1);
      mbar_init(bar(kBarXCons + i), 256);
    }
    mbar_init(bar(kBarPFull), 256);
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarOFinal), 1);
    mbar_init(bar(kBarQReady), 256);
    mbar_init(bar(kBarQStaged), 256);
    mbar_init(bar(kBarQLoaded), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
    if (a.q_tma) {
      // The CTA's Q half as 128-row boxes of 64 channels (128-byte swizzle)
      // into the staging area; channels past d_qk read as zeros.
      const int nbox = (a.ksteps * 16 + 63) / 64;
      mbar_arrive_expect_tx(bar(kBarQLoaded), (uint32_t)(nbox * 128 * 128));
      for (int k = 0; k < nbox; ++k)
        tma_load_2d(sb + kOffQStage + (uint32_t)k * 128u * 128u, &a.q_map, a.q_lo[r] + 64 * k,
                    t * 128, bar(kBarQLoaded));
    }
  }
  // a1/a2 setup (before the TMEM allocation and the cluster barrier, which
  // it does not need, so that the loads overlap them): the producers read
  // the whole index range of the unit once
  // (coalesced, all loads in flight together) into shared memory, masking
  // positions past k1, ids < 0 and ids >= num_slots; then one valid-mask per
  // block.  Every role reads both from shared memory afterwards.
  int* slots = reinterpret_cast<int*>(sm + kOffSlot);
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + kOffMask);
  if (warp >= 1 && warp < 4) {
    const int pt = tid - 32;
    const int n = nb * kBN;
    if (load_unit_slots(p, t, k0, k1, n, slots, pt, kProducers))
      atomicCAS(p.status, 0, kStatusBadIndex);
    named_bar_sync(1, kProducers);
    // One valid-mask pair per block (rows 0..31, rows 32..47): the three
    // warps take every third block, four blocks per step (their slot-id
    // reads in flight together).
    {
      const int w = warp - 1;
      for (int b0 = 4 * w; b0 < nb; b0 += 12) {
        int id0[4], id1[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int b = min(b0 + k, nb - 1);
          id0[k] = slots[b * kBN + lane];
          id1[k] = lane < kBN - 32 ? slots[b * kBN + 32 + lane] : -1;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t m0 = __ballot_sync(0xffffffffu, id0[k] >= 0);
          const uint32_t m1 = __ballot_sync(0xffffffffu, id1[k] >= 0);
          if (lane == 0 && b0 + k < nb) {
            masks[(b0 + k) * 2] = m0;
            masks[(b0 + k) * 2 + 1] = m1;
          }
        }
      }
    }
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

  __syncthreads();

  if (warp == 0) {
    // ---- MMA issuer: QK two blocks ahead of PV ------------------------------
    // The whole warp runs this code (warp-uniform waits and descriptors); one
    // elected lane issues each batch of MMAs and its commits.
    if (nb > 0) {
      const uint32_t id_qk = idesc_bf16(128, kBN, false, false);
      const uint32_t id_pv = idesc_bf16(128, 256, false, true);
      const int qk_lo = a.qk_lo[r];
      const int ksteps = a.ksteps;
      W.wait(bar(kBarQReady), 0);
      tc_fence_after();
      auto issue_qk = [&](int j) {
        if (p.inject_stall && j == 0) return;   // tests: block 0's scores never arrive
        const int s = j % kStages;
        W.wait(bar(kBarKvFull + s), (j / kStages) & 1);
        if (j >= 2) W.wait(bar(kBarSEmpty + (j & 1)), ((j >> 1) - 1) & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kTileBytes;
        const uint32_t dS = tmem + kColS + kBN * (j & 1);
        if (elect_one()) {
          fence_proxy_async_smem();
          for (int ks = 0; ks < ksteps; ++ks) {
            const int c0 = qk_lo + 16 * ks;
            const uint32_t baddr = tile + (c0 >> 6) * kAtomBytes + (c0 & 63) * 2;
            mma_ts(dS, tmem + kColQ + 8 * ks, sdesc(baddr, 16, 1024, kLayoutSw128), id_qk,
                   ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(kBarSFull + (j & 1)));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int j) {
        W.wait(bar(kBarPFull), j & 1);
        __syncwarp();
        tc_fence_after();
        const uint32_t pa = sb + kOffP;
        const uint32_t tile = sb + kOffTile + (j % kStages) * kTileBytes;
        if (elect_one()) {
          fence_proxy_async_smem();
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            const uint64_t ad = sdesc(pa + ks * 32, 16, 1024, kLayoutSw128);
            const uint64_t bd = sdesc(tile + ks * 16 * 128, kAtomBytes, 1024, kLayoutSw128);
            mma_ss(tmem + kColO, ad, bd, id_pv, (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(bar(kBarODone));
          mma_commit(bar(kBarPEmpty));
          mma_commit(bar(kBarKvEmpty + (j % kStages)));
          if (j == nb - 1) mma_commit(bar(kBarOFinal));
        }
        __syncwarp();
      };
      issue_qk(0);
      if (nb > 1) issue_qk(1);
      for (int j = 0; j < nb; ++j) {
        if (j + 2 < nb) issue_qk(j + 2);
        issue_pv(j);
      }
    }
    // Every MMA this warp issued has completed (also after an abort) before
    // the TMEM is freed and the tiles are left.
    __syncwarp();
    if (elect_one()) mma_commit(bar(kBarDrain));
    __syncwarp();
    W.drain(bar(kBarDrain), 0);
  } else if (warp < 4) {
    // ---- producers: a2 gather with TMA (tile::gather4) ----------------------
    // Per block: 12 groups of 4 rows x n_boxes 64-channel boxes; warps 1..3
    // each issue 4 of the groups (TMA gather throughput grows with the number
    // of issuing warps).  The tensor map's 128-byte swizzle matches the MMA
    // operand layout, and a masked position (slot id -1) reads the
    // out-of-bounds fill, i.e. a zero row.
    const int g_lo = a.g_lo[r];
    if (a.fp8) {
      // a2 + a3 for an E4M3 cache: two threads per row load the row's bytes
      // with 16-byte loads (all loads of a block in flight at once, issued
      // before the stage is free), convert
      // them exactly to bf16 and store the 128-byte-swizzled tile; masked
      // rows are zero.  The per-tensor scale is applied in fp32 later (score
      // scale and output normalization), so the tile holds exact values.
      const int pt = tid - 32;
      const int row = pt >> 1, half = pt & 1;
      const uint32_t sw = (uint32_t)row & 7u;
      const int nc8 = a.n_chunks8[r];                         // <= 20
      const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
      // The row of block j into L2 (the two threads of a row cover its up to
      // four 128-byte lines); rows are prefetched two blocks ahead.
      auto prefetch_row = [&](int j) {
        const int idp = slots[j * kBN + row];
        if (idp < 0) return;
        const uint8_t* rp = kv8 + (size_t)idp * p.d_qk + g_lo;
        prefetch_l2(rp + 128 * half);
        prefetch_l2(rp + (half ? 16 * nc8 - 1 : min(256, 16 * nc8 - 1)));
      };
      if (nb > 1) prefetch_row(1);
      for (int b = 0; b < nb; ++b) {
        const int s = b % kStages;
        if (b + 2 < nb) prefetch_row(b + 2);
        const int id = slots[b * kBN + row];
        const uint4* src = reinterpret_cast<const uint4*>(
            kv8 + (size_t)(id < 0 ? 0 : id) * p.d_qk + g_lo);
        uint4 raw[10];
#pragma unroll
        for (int kk = 0; kk < 10; ++kk) {
          const int c = half + 2 * kk;
          raw[kk] = (id >= 0 && c < nc8) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        // The loads are in flight while the stage is awaited.
        if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b / kStages) - 1) & 1);
        if (*abort_flag) break;                  // the stage may still be in use
        uint8_t* rgen = sm + kOffTile + s * kTileBytes + row * 128;
#pragma unroll
        for (int kk = 0; kk < 10; ++kk) {
          const int c = half + 2 * kk;
          if (c < nc8) {
            uint32_t o[8];
            e4m3x4_to_bf16(raw[kk].x, o[0], o[1]);
            e4m3x4_to_bf16(raw[kk].y, o[2], o[3]);
            e4m3x4_to_bf16(raw[kk].z, o[4], o[5]);
            e4m3x4_to_bf16(raw[kk].w, o[6], o[7]);
            const uint32_t cj = 2u * (uint32_t)c;             // two bf16 chunks
            *reinterpret_cast<uint4*>(rgen + (cj >> 3) * kAtomBytes + (((cj & 7u) ^ sw) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
            const uint32_t cj1 = cj + 1u;
            *reinterpret_cast<uint4*>(rgen + (cj1 >> 3) * kAtomBytes + (((cj1 & 7u) ^ sw) << 4)) =
                make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarKvFull + s));
      }
    } else {
    const int n_boxes = a.n_boxes[r];
    const int w = warp - 1;                                   // 0..2
    const uint32_t tx_bytes = (uint32_t)(kBN / 4 / 3 * n_boxes * 512);
    int issued = 0;
    for (int b = 0; b < nb; ++b) {
      const int s = b % kStages;
      if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b / kStages) - 1) & 1);
      if (b >= 1 && b < kStages) W.wait(bar(kBarQStaged), 0);   // Q staging read
      if (*abort_flag) break;                    // the stage may still be in use
      __syncwarp();
      issued = b + 1;
      if (elect_one()) {
        const uint32_t full = bar(kBarKvFull + s);
        mbar_arrive_expect_tx(full, tx_bytes);
        const uint32_t tile = sb + kOffTile + s * kTileBytes;
        const int* bs = slots + b * kBN;
        for (int g = w; g < kBN / 4; g += 3) {
          const int y0 = bs[4 * g], y1 = bs[4 * g + 1], y2 = bs[4 * g + 2], y3 = bs[4 * g + 3];
          for (int bx = 0; bx < n_boxes; ++bx)
            tma_gather4(tile + bx * kAtomBytes + 4 * g * 128, &a.kv_map, g_lo + 64 * bx, y0,
                        y1, y2, y3, full);
        }
      }
      __syncwarp();
    }
    // Teardown: the gathers of the last block issued into each stage have
    // landed (earlier ones were consumed before the stage was reissued).
    // After an abort a stage's phase may lack another warp's share and wait
    // out the limit; the copies themselves land within microseconds.
    if (lane == 0) {
      for (int b = issued - 1; b >= 0 && b >= issued - kStages; --b)
        W.drain(bar(kBarKvFull + b % kStages), (b / kStages) & 1);
    }
    __syncwarp();
    }
  } else if (warp == 12) {
    // ---- signal warp: tell the peer when its partial scores were consumed --
    // (a release-ordered remote arrival; kept off the softmax warps' path)
    if (lane == 0) {
      const uint32_t xfree_peer = mapa(bar(kBarXFree), peer);
      for (int b = 0; b < nb; ++b) {
        W.wait(bar(kBarXCons + (b & 1)), (b >> 1) & 1);
        mbar_arrive_remote(xfree_peer + 8u * (b & 1));
      }
    }
  } else if (warp <= 11) {
    // ---- softmax warpgroups --------------------------------------------------
    // Warpgroup wg (warps 4..7: wg 0, warps 8..11: wg 1) owns positions
    // [24 wg, 24 wg + 24) of every block; thread i of a warpgroup owns head i
    // (TMEM lane i).  Each warpgroup exchanges its own half of the partial
    // scores with the same warpgroup of the peer CTA.  Both warpgroups keep
    // the same running max m (log2 units): once per block they meet at a
    // named barrier that also reduces "some half-block max passes m + 8"; only
    // then do they read each other's half maxima and raise m (identically).
    const int wg = (warp - 4) >> 2;
    const int i = (warp & 3) * 32 + lane;        // head row == TMEM lane
    const uint32_t lane_base = ((uint32_t)(warp & 3) * 32u) << 16;
    const int head = i;
    const bool wlead = i == 0;                   // the warpgroup's first thread
    // Q half -> TMEM (rows >= h are zero): 16-column groups [0, 5) by the
    // first warpgroup, [5, ksteps / 2) by the second.
    {
      // (staged before the set-up; the block-wide barrier since then makes
      // every thread's staging stores visible)
      const int g0 = wg == 0 ? 0 : 5, g1 = wg == 0 ? 5 : a.ksteps / 2;
      const uint8_t* qrow = sm + kOffQStage + head * kQStageRow;
      if (a.q_tma) W.wait(bar(kBarQLoaded), 0);
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        if (k < g1 - g0) {                       // same for every lane
          uint4 x0, x1, x2, x3;
          if (a.fp8) {                           // from global memory, this head's row
            const int c0 = a.q_lo[r] + 32 * (g0 + k);
            const bool live = head < p.h;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            x0 = live ? __ldg(q_chunk(p, t, head, c0)) : z;
            x1 = live ? __ldg(q_chunk(p, t, head, c0 + 8)) : z;
            x2 = live ? __ldg(q_chunk(p, t, head, c0 + 16)) : z;
            x3 = live ? __ldg(q_chunk(p, t, head, c0 + 24)) : z;
          } else if (a.q_tma) {                  // from the swizzled TMA boxes
            // channels [32 (g0 + k), +32): box (g0 + k) / 2, 16-byte chunks
            // 4 ((g0 + k) % 2) + j, stored at chunk ^ (head % 8)
            const int g = g0 + k;
            const uint8_t* brow = sm + kOffQStage + (g >> 1) * 128 * 128 + head * 128;
            const uint32_t sw = (uint32_t)head & 7u, c0 = 4u * (uint32_t)(g & 1);
            x0 = *reinterpret_cast<const uint4*>(brow + (((c0 + 0u) ^ sw) << 4));
            x1 = *reinterpret_cast<const uint4*>(brow + (((c0 + 1u) ^ sw) << 4));
            x2 = *reinterpret_cast<const uint4*>(brow + (((c0 + 2u) ^ sw) << 4));
            x3 = *reinterpret_cast<const uint4*>(brow + (((c0 + 3u) ^ sw) << 4));
          } else {                               // from the staging rows
            const uint4* q4 = reinterpret_cast<const uint4*>(qrow + 64 * (g0 + k));
            x0 = q4[0]; x1 = q4[1]; x2 = q4[2]; x3 = q4[3];
          }
          const uint32_t w[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                  x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
          __syncwarp();
          tmem_st16(tmem + lane_base + kColQ + 16 * (g0 + k), w);
        }
      }
      mbar_arrive(bar(kBarQStaged));             // the staging may be overwritten
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarQReady));
    }
    // E4M3 cache: the per-tensor scale multiplies every score and output.
    const float kscale = a.fp8 ? __ldg(p.k_scale) : 1.f;
    const float scale_log2 = a.scale_log2 * kscale;
    float m_run = -INFINITY;   // running max (log2 units), same in both warpgroups
    float l_run = 0.f;         // this warpgroup's running sum of exp2(s - m_run)
    float lr_run = 0.f;        // the same sum of the bf16-rounded P (what PV multiplies)
    const uint32_t x_half = (uint32_t)wg * kXHalfBytes;
    const uint8_t* Xr = sm + kOffX + x_half;           // receive buffers (this half)
    const uint32_t x_peer = mapa(sb + kOffX + x_half, peer);
    const uint32_t xfull_peer = mapa(bar(kBarXFull + wg), peer);
    const uint32_t xrow = (uint32_t)i * (kBN / 2) * 4; // this row's byte offset
    const uint32_t xsw = ((uint32_t)i >> 2) & 1u;      // its chunk swizzle
    float* red = reinterpret_cast<float*>(sm + kOffRed);  // [2 buf][2 wg][128]
    const int nbar = 2 + wg;                           // warpgroup-local barrier

    // O row *= alpha for this warpgroup's 128 columns.  tcgen05.ld/st are
    // warp-collective (.sync.aligned), so the whole warp takes this path when
    // any of its lanes needs it; lanes with nothing to rescale pass 1.
    auto rescale_o = [&](float alpha, int b) {
      W.wait(bar(kBarODone), (b - 1) & 1);
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int c = 128 * wg; c < 128 * wg + 128; c += 16) {
        uint32_t w[16];
        tmem_ld16(tmem + lane_base + kColO + c, w);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * alpha);
        tmem_st16(tmem + lane_base + kColO + c, w);
      }
      tmem_wait_st();
    };
    // Read this half of the row's partial scores of block j from TMEM, free
    // the S buffer, stage them in shared memory, and (the warpgroup's first
    // thread) send the 128 rows to the peer with one bulk copy counted on its
    // X-full barrier for (buffer j & 1, this half).
    auto load_and_send = [&](int j, float (&dst)[kBN / 2]) {
      const int buf = j & 1;
      if (wlead) {
        mbar_arrive_expect_tx(bar(kBarXFull + 2 * buf + wg), (uint32_t)kXHalfBytes);
        bulk_wait_read_all();                // the previous send has read the stage
      }
      W.wait(bar(kBarSFull + buf), (j >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      {
        uint32_t w16[16], w8[8];
        const uint32_t col = tmem + lane_base + kColS + kBN * buf + (kBN / 2) * wg;
        tmem_ld16(col, w16);
        tmem_ld8(col + 16, w8);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) dst[k] = __uint_as_float(w16[k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[16 + k] = __uint_as_float(w8[k]);
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty + buf));
      named_bar_sync(nbar, 128);             // staging half is free
      uint8_t* srow = sm + kOffXs + x_half + xrow;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c)
        *reinterpret_cast<float4*>(srow + ((((uint32_t)c) ^ xsw) << 4)) =
            make_float4(dst[4 * c], dst[4 * c + 1], dst[4 * c + 2], dst[4 * c + 3]);
      fence_proxy_async_smem();
      named_bar_sync(nbar, 128);             // all rows staged
      if (wlead) {
        if (j >= 2) W.wait(bar(kBarXFree + buf), ((j >> 1) - 1) & 1);
        bulk_copy_to_peer(x_peer + buf * kXBytes, sb + kOffXs + x_half, (uint32_t)kXHalfBytes,
                          xfull_peer + 16u * buf);
        bulk_commit_group();
      }
    };

    float sp[kBN / 2], nx[kBN / 2];
    if (nb > 0) load_and_send(0, nx);
    for (int b = 0; b < nb; ++b) {
      const int buf = b & 1;
#pragma unroll
      for (int j = 0; j < kBN / 2; ++j) sp[j] = nx[j];
      if (b + 1 < nb) load_and_send(b + 1, nx);
      // The peer's partial for this half-block; then let the peer reuse it.
      W.wait_cluster(bar(kBarXFull + 2 * buf + wg), (b >> 1) & 1);
      const uint8_t* xr = Xr + buf * kXBytes + xrow;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(xr + ((((uint32_t)c) ^ xsw) << 4));
        sp[4 * c] += x.x; sp[4 * c + 1] += x.y; sp[4 * c + 2] += x.z; sp[4 * c + 3] += x.w;
      }
      mbar_arrive(bar(kBarXCons + buf));   // the signal warp tells the peer
      // a5: masked online softmax (log2 domain).  When every position of
      // this half-block is valid (and the scale is positive, which keeps the
      // order), the scores stay unscaled: the row max is taken on them and
      // scaled once, and each exponent below is one fma, s * c - m.
      // Otherwise each score is masked and scaled first (c = 1 below).
      const uint64_t vm = ((uint64_t)masks[b * 2 + 1] << 32 | masks[b * 2]) >> (24 * wg);
      float cl = scale_log2;
      if ((uint32_t)(vm & 0xFFFFFFu) != 0xFFFFFFu || !(scale_log2 > 0.f)) {
#pragma unroll
        for (int j = 0; j < kBN / 2; ++j)
          sp[j] = ((vm >> j) & 1u) ? sp[j] * scale_log2 : -INFINITY;
        cl = 1.f;
      }
      float hm = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBN / 2; ++j) hm = fmaxf(hm, sp[j]);
      hm *= cl;
      float* rb = red + buf * 256;
      rb[wg * 128 + i] = hm;
      float alpha = 1.f;
      if (named_bar_or(4, 256, hm > m_run + 8.f)) {   // also true for the first finite max
        const float bm = fmaxf(hm, rb[(wg ^ 1) * 128 + i]);
        if (bm > m_run + 8.f) {
          alpha = ex2_approx(m_run - bm);             // 0 when m_run = -inf
          m_run = bm;
        }
      }
      uint32_t pk[kBN / 4];
      float lsum = 0.f, lsum_r = 0.f;
      if (m_run == -INFINITY) {
#pragma unroll
        for (int j = 0; j < kBN / 4; ++j) pk[j] = 0u;
      } else {
#pragma unroll
        for (int j = 0; j < kBN / 2; j += 2) {
          // P goes to the PV MMA in bf16; the row sum of the unrounded
          // values sets the LSE, that of the rounded ones divides O.
          const float e0 = ex2_approx(fmaf(sp[j], cl, -m_run));
          const float e1 = ex2_approx(fmaf(sp[j + 1], cl, -m_run));
          pk[j / 2] = pack_bf16(e0, e1);
          lsum += e0 + e1;
          lsum_r = add_bf16x2_f32(lsum_r, pk[j / 2]);
        }
      }
      l_run = l_run * alpha + lsum;
      lr_run = lr_run * alpha + lsum_r;
      if (b >= 1) W.wait(bar(kBarPEmpty), (b - 1) & 1);   // PV(b-1) has read P
      // This half of the P row (24 bf16 = 3 chunks of 16 B, chunks 3 wg ..
      // 3 wg + 2) into the 128-byte-swizzled buffer.
      uint8_t* prow = sm + kOffP + i * 128;
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        const uint32_t off = ((uint32_t)(3 * wg + c) ^ ((uint32_t)i & 7u)) << 4;
        *reinterpret_cast<uint4*>(prow + off) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      if (b >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o(alpha, b);
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
    }

    // ---- a7: epilogue ---------------------------------------------------------
    // l = the two warpgroups' sums.  (A parity wait on the per-PV barrier
    // could pass a phase early when two PVs are still in flight; the final
    // barrier has exactly one phase.)
    // O is divided by the sum of the rounded P that PV multiplied, so that
    // where one key carries a row its rounded weight cancels (the lazy
    // running max leaves that weight anywhere in (1, 2^8], where bf16 is off
    // by up to 2^-8 of it); the LSE takes the unrounded sum.
    float* lsh = reinterpret_cast<float*>(sm + kOffL);  // [2 sums][2][128]
    lsh[wg * 128 + i] = l_run;
    lsh[256 + wg * 128 + i] = lr_run;
    named_bar_sync(4, 256);
    const float l_tot = lsh[i] + lsh[128 + i];
    const float lr_tot = lsh[256 + i] + lsh[384 + i];
    if (nb > 0) {
      W.wait(bar(kBarOFinal), 0);
      __syncwarp();
      tc_fence_after();
    }
    // empty: no valid key (a NaN row sum, from a NaN in the cache, is not)
    const bool empty = l_tot == 0.f || nb == 0;
    const float inv = empty ? 0.f : __fdividef(kscale, lr_tot);  // (IEEE division: slow here)
    const bool live = head < p.h;          // pad rows past h are not written
    const int64_t orow = (int64_t)t * p.h + (live ? head : 0);
    // Every lane of the warpgroup runs the TMEM loads (warp-collective);
    // only the stores depend on the lane's head.  Warpgroup wg writes output
    // channels [256 r + 128 wg, 256 r + 128 wg + 128).
    if (a.o_tma) {
      // bf16 O through two 128-byte-swizzled boxes of 64 channels x 128 head
      // rows in the gather stages (idle now: every gather was consumed), then
      // two TMA stores issued by the warpgroup's first thread (one row of a
      // box per thread: the stores are whole 128-byte lines; a thread's own
      // 16-byte stores would each touch half a sector of a different row).
      uint8_t* box0 = sm + kOffTile + (uint32_t)(2 * wg) * 16384u + (uint32_t)head * 128u;
      const uint32_t hsw = (uint32_t)head & 7u;
      // (32 channels per TMEM wait)
#pragma unroll 1
      for (int c2 = 0; c2 < 128; c2 += 32) {
        uint32_t w[2][16];
        __syncwarp();
        if (nb > 0) {
          tmem_ld16(tmem + lane_base + kColO + 128 * wg + c2, w[0]);
          tmem_ld16(tmem + lane_base + kColO + 128 * wg + c2 + 16, w[1]);
          tmem_wait_ld();
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = c2 + 16 * h2;
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = empty ? 0u
                         : pack_bf16(__uint_as_float(w[h2][2 * k]) * inv,
                                     __uint_as_float(w[h2][2 * k + 1]) * inv);
          const uint32_t ck = (uint32_t)(c >> 3);           // 16-byte chunk of the 128 channels
          uint8_t* brow = box0 + (ck >> 3) * 16384u;
          *reinterpret_cast<uint4*>(brow + ((((ck & 7u) + 0u) ^ hsw) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(brow + ((((ck & 7u) + 1u) ^ hsw) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(nbar, 128);
      if (wlead) {
        for (int bx = 0; bx < 2; ++bx)
          tma_store_2d(&a.o_map, sb + kOffTile + (uint32_t)(2 * wg + bx) * 16384u,
                       256 * (int)r + 128 * wg + 64 * bx, t * 128);
        bulk_commit_group();
      }
    } else {
#pragma unroll 1
    for (int c = 128 * wg; c < 128 * wg + 128; c += 16) {
      uint32_t w[16];
      __syncwarp();
      if (nb > 0) {
        tmem_ld16(tmem + lane_base + kColO + c, w);
        tmem_wait_ld();
      }
      if (!live) {
      } else if (p.fp32_out) {
        float* dst = p.o_part + ((int64_t)split * p.T * p.h + orow) * p.d_v + 256 * r + c;
#pragma unroll
        for (int k = 0; k < 16; k += 4)
          *reinterpret_cast<float4*>(dst + k) =
              empty ? make_float4(0.f, 0.f, 0.f, 0.f)
                    : make_float4(__uint_as_float(w[k]) * inv, __uint_as_float(w[k + 1]) * inv,
                                  __uint_as_float(w[k + 2]) * inv,
                                  __uint_as_float(w[k + 3]) * inv);
      } else {
        __nv_bfloat16* dst =
            reinterpret_cast<__nv_bfloat16*>(p.out) + orow * p.d_v + 256 * r + c;
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          o[k] = empty ? 0u
                       : pack_bf16(__uint_as_float(w[2 * k]) * inv,
                                   __uint_as_float(w[2 * k + 1]) * inv);
        *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    }
    // Both CTAs hold the same LSE; the first warpgroup of CTA r writes heads
    // [64r, 64r + 64).
    if (wg == 0 && live && (uint32_t)(i >> 6) == r) {
      const float lse_v =
          empty ? -INFINITY : (m_run + log2f(l_tot)) * 0.69314718055994530942f;
      if (p.fp32_out)
        p.lse_part[(int64_t)split * p.T * p.h + orow] = lse_v;
      else if (p.lse)
        p.lse[orow] = lse_v;
    }
  }

  // ---- teardown: no CTA leaves while its peer may still write into it -----
  // Each warpgroup's sends have read their stage; the peer's last X-free
  // arrivals land asynchronously: wait for the final phases of both X-free
  // barriers first.
  // (also after an abort: the peer's shared memory stays until the cluster
  // barrier below, which this CTA passes only after its copies are complete)
  // (and the O boxes' TMA stores have read the staging: only the reads of
  // this CTA's shared memory need to be complete before it leaves; the sends
  // have landed in the peer, which consumed them before its last X-free
  // arrival waited on below)
  if (tid == 128 || tid == 256) bulk_wait_read_all();
  if (tid == 0 && a.q_tma) W.drain(bar(kBarQLoaded), 0);
  if (tid == 128 && nb > 0) {
    if (nb >= 2) W.wait(bar(kBarXFree + ((nb - 2) & 1)), ((nb - 2) >> 1) & 1);
    W.wait(bar(kBarXFree + ((nb - 1) & 1)), ((nb - 1) >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_arrive();
  cluster_wait();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int tc_max_range() { return kMaxBlocks * kBN; }

bool tc_supported(int h, int d_qk, int kv_format) {
  return h >= 1 && h <= 128 && (d_qk == 576 || d_qk == 512) &&
         (kv_format == kBf16 || kv_format == kE4m3);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

cudaError_t encode_bf16_rows_map(CUtensorMap* map, const void* kv, int d_qk,
                                 int64_t num_slots) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)d_qk, (cuuint64_t)num_slots};
  const cuuint64_t strides[1] = {(cuuint64_t)d_qk * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

cudaError_t launch_tc(const FwdParams& p, cudaStream_t stream) {
  TcArgs a{};
  a.p = p;
  a.fp8 = p.kv_format == kE4m3 ? 1 : 0;
  if (!a.fp8) {
    const cudaError_t e = encode_bf16_rows_map(&a.kv_map, p.kv, p.d_qk, p.num_slots);
    if (e != cudaSuccess) return e;
  }
  // Q by TMA boxes: bf16 cache, 128 heads (a token's rows are exactly one
  // box high), q in one tensor.
  if (!a.fp8 && p.h == 128 && !p.q_pe) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)p.d_qk, (cuuint64_t)p.T * 128};
    const cuuint64_t strides[1] = {(cuuint64_t)p.d_qk * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&a.q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.q), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    a.q_tma = 1;
  }
  // O by TMA boxes: 128 heads (a token's rows are exactly one box high),
  // bf16 output.
  if (p.h == 128 && !p.fp32_out) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)p.d_v, (cuuint64_t)p.T * 128};
    const cuuint64_t strides[1] = {(cuuint64_t)p.d_v * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&a.o_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    a.o_tma = 1;
  }
  if (p.d_qk == 576) {
    a.g_lo[0] = 0;   a.n_boxes[0] = 5; a.qk_lo[0] = 0;  a.q_lo[0] = 0;
    a.g_lo[1] = 256; a.n_boxes[1] = 5; a.qk_lo[1] = 32; a.q_lo[1] = 288;
    a.n_chunks8[0] = 18; a.n_chunks8[1] = 20;   // channels 0..287, 256..575
    a.ksteps = 18;
  } else {
    a.g_lo[0] = 0;   a.n_boxes[0] = 4; a.qk_lo[0] = 0; a.q_lo[0] = 0;
    a.g_lo[1] = 256; a.n_boxes[1] = 4; a.qk_lo[1] = 0; a.q_lo[1] = 256;
    a.n_chunks8[0] = 16; a.n_chunks8[1] = 16;   // channels 0..255, 256..511
    a.ksteps = 16;
  }
  a.scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t clusters = (int64_t)p.T * p.splits;
  if (clusters * 2 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const bool lpt = p.lpt && clusters <= kLptMaxUnits;
  auto kernel = lpt ? smla_tc_kernel<true> : smla_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)(clusters * 2), kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace smla

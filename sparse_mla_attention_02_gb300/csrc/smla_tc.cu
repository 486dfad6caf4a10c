// smla_tc.cu — tensor-core (tcgen05 / TMEM) sparse MLA forward for sm_103a.
//
// One work unit = (query token t, top-k position range) and runs on a cluster
// of two CTAs (a pair of SMs).  Why two: for h = 128 heads the fp32 output
// accumulator O[128, 512] alone fills the 512 TMEM columns of one SM, and an
// M = 64 MMA runs at half rate.  So the pair splits the work so that every MMA
// is M = 128 (all heads):
//   * QK^T is split over d_qk: CTA r holds Q[:, its half of d_qk] in TMEM
//     (the MMA's A operand) and computes the partial scores
//     S_r = Q_r K_r^T  [128 heads x 64 keys] per block of 64 positions;
//   * the pair swaps halves of S_r through distributed shared memory: CTA r
//     owns the softmax of heads [64r, 64r+64) and receives the other CTA's
//     partial for them;
//   * PV is split over d_v: CTA r accumulates O[:, 256r : 256r+256] in TMEM
//     from P [128 x 64] (both CTAs' halves, exchanged the same way) and the
//     first 512 channels of the same gathered rows (V is the prefix of K).
// Method steps (vLLM "Sparse MLA on Hopper" diff, ops/cutlass_fa3.py docstring:
// score = q_rope.k_rope + q_nope.c_kv, output = softmax(score*scale) @ c_kv;
// flashinfer_mla_sparse_sm90.py, forward_mqa: compacted valid prefix with -1
// past it; vLLM API docs flashmla_sparse, _forward_fp8_kv_mixed_batch: empty
// rows give (O = 0, LSE = -inf)):
//   a1 work setup: v = min(valid_len[t], topk); range [k0, k1) of the split
//   a2 gather: slot ids -> rows of the cache into a 128-byte-swizzled tile
//      (masked positions become zero rows)
//   a4 QK^T (tcgen05.mma, A = Q from TMEM, B = K tile, K-major)
//   a5 masked online softmax in registers (one thread per head row), with the
//      running max updated lazily (rescale O only when it grows by > 2^8)
//   a6 PV (tcgen05.mma, A = P from shared memory, B = V tile, MN-major)
//   a7 epilogue: O / l -> bf16 out (or fp32 partials), LSE = m + ln l
//
// Warp roles (256 threads): warp 0 issues MMAs (one thread) and owns TMEM;
// warps 1..3 gather with cp.async; warps 4..7 (a warpgroup; thread i <-> TMEM
// lane i <-> head i) do softmax, the exchange, O rescale and the epilogue.
// Every wait is bounded; a wait that runs out records SMLA timeout status,
// sets an abort flag that skips later waits, and the block finishes normally.
#include <cuda_bf16.h>
#include <math.h>

#include "smla_internal.h"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kBN = 64;            // top-k positions per block
constexpr int kStages = 3;         // gathered-tile pipeline depth
constexpr int kAtomBytes = 8192;   // 64 rows x 128 B (one 64-channel column)
constexpr int kTileBytes = 5 * kAtomBytes;  // up to 320 channels per CTA
constexpr int kPBytes = 128 * 128;          // P: 128 rows x 64 bf16
constexpr int kXStride = 68;                // floats per exchanged S row (padded)
constexpr int kXBytes = 64 * kXStride * 4;
constexpr int kThreads = 256;
constexpr int kProducers = 96;     // warps 1..3

// TMEM columns.
constexpr uint32_t kColO = 0;      // O half: 256 columns
constexpr uint32_t kColQ = 256;    // Q half: up to 144 columns
constexpr uint32_t kColS = 400;    // partial S: 64 columns
constexpr uint32_t kTmemCols = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffTile = 0;
constexpr uint32_t kOffP = kOffTile + kStages * kTileBytes;
constexpr uint32_t kOffX = kOffP + 2 * kPBytes;
constexpr uint32_t kOffAlpha = kOffX + 2 * kXBytes;   // [2][128] f32
constexpr uint32_t kOffL = kOffAlpha + 2 * 128 * 4;   // [2][128] f32
constexpr uint32_t kOffSlot = kOffL + 2 * 128 * 4;    // [stages][64] i32
constexpr uint32_t kOffMask = kOffSlot + kStages * 64 * 4;  // [stages][2] u32
constexpr uint32_t kOffBar = (kOffMask + kStages * 8 + 7) & ~7u;
enum {
  kBarKvFull = 0,
  kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,
  kBarSEmpty,
  kBarPFull,              // [2]
  kBarPEmpty = kBarPFull + 2,   // [2]
  kBarPxFull = kBarPEmpty + 2,  // [2]
  kBarXFull = kBarPxFull + 2,   // [2]
  kBarXFree = kBarXFull + 2,    // [2]
  kBarODone = kBarXFree + 2,
  kBarQReady,
  kNumBars
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack

struct TcArgs {
  FwdParams p;
  int g_lo[2];      // first cache channel gathered by CTA r
  int n_chunks[2];  // 16-byte chunks gathered per row by CTA r
  int qk_lo[2];     // first local channel of CTA r's QK range
  int q_lo[2];      // first q channel CTA r keeps in TMEM
  int ksteps;       // 16-channel MMA steps of the QK half
  float scale_log2; // sm_scale * log2(e)
};

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Multicast commit: one arrival on the mbarrier at this offset in every CTA
// of the cluster named by `mask`, when this thread's prior MMAs complete.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::"
      "cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Bounded waits.  A wait that runs out (or sees that another block already
// gave up) records the timeout status, sets this block's abort flag, and from
// then on every wait of the block returns at once, so the block still reaches
// its teardown.  Results of an aborted launch are undefined; no access goes
// out of bounds.
struct Waiter {
  volatile int* abort;
  int* status;
  __device__ __forceinline__ void fail() {
    if (!*abort) {
      *abort = 1;
      atomicCAS(status, 0, kStatusTimeout);
    }
  }
  __device__ __forceinline__ void wait(uint32_t bar, uint32_t parity) {
    if (*abort) return;
    if (!mbar_wait_bounded<false>(bar, parity, status, kStatusTimeout)) fail();
  }
  __device__ __forceinline__ void wait_cluster(uint32_t bar, uint32_t parity) {
    if (*abort) return;
    if (!mbar_wait_bounded<true>(bar, parity, status, kStatusTimeout)) fail();
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

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
  const int unit = blockIdx.x >> 1;
  const int split = unit % p.splits;
  const int t = unit / p.splits;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = split * p.split_len;
  const int k1 = min(k0 + p.split_len, v);
  const int nb = k1 > k0 ? (k1 - k0 + kBN - 1) / kBN : 0;

  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffAbort);
  Waiter W{abort_flag, p.status};

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 2 * kProducers);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSEmpty), 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarPFull + i), 128);
      mbar_init(bar(kBarPEmpty + i), 2);
      mbar_init(bar(kBarPxFull + i), 64);
      mbar_init(bar(kBarXFull + i), 64);
      mbar_init(bar(kBarXFree + i), 64);
    }
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarQReady), 128);
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

  if (warp == 0) {
    // ---- MMA issuer ---------------------------------------------------------
    if (lane == 0 && nb > 0) {
      const uint32_t id_qk = idesc_bf16(128, kBN, false, false);
      const uint32_t id_pv = idesc_bf16(128, 256, false, true);
      W.wait(bar(kBarQReady), 0);
      tc_fence_after();
      auto issue_pv = [&](int j) {
        const int buf = j & 1;
        W.wait(bar(kBarPFull + buf), (j >> 1) & 1);
        tc_fence_after();
        fence_proxy_async();
        const uint32_t pa = sb + kOffP + buf * kPBytes;
        const uint32_t tile = sb + kOffTile + (j % kStages) * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t ad = sdesc(pa + ks * 32, 16, 1024, kLayoutSw128);
          const uint64_t bd = sdesc(tile + ks * 16 * 128, kAtomBytes, 1024, kLayoutSw128);
          mma_ss(tmem + kColO, ad, bd, id_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarODone));
        mma_commit_mc(bar(kBarPEmpty + buf), 0x3);
        mma_commit(bar(kBarKvEmpty + (j % kStages)));
      };
      for (int b = 0; b < nb; ++b) {
        const int s = b % kStages;
        W.wait(bar(kBarKvFull + s), (b / kStages) & 1);
        fence_proxy_async();
        if (b > 0) W.wait(bar(kBarSEmpty), (b - 1) & 1);
        tc_fence_after();
        const uint32_t tile = sb + kOffTile + s * kTileBytes;
        for (int ks = 0; ks < a.ksteps; ++ks) {
          const int c0 = a.qk_lo[r] + 16 * ks;
          const uint32_t baddr = tile + (c0 >> 6) * kAtomBytes + (c0 & 63) * 2;
          mma_ts(tmem + kColS, tmem + kColQ + 8 * ks,
                 sdesc(baddr, 16, 1024, kLayoutSw128), id_qk, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(kBarSFull));
        if (b > 0) issue_pv(b - 1);
      }
      issue_pv(nb - 1);
    }
  } else if (warp < 4) {
    // ---- producers: a2 gather ---------------------------------------------
    const int pt = tid - 32;
    const int nc = a.n_chunks[r];
    const int g_lo = a.g_lo[r];
    const size_t row_bytes = (size_t)p.d_qk * 2;
    const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.kv);
    const int32_t* idx_row = p.indices + (int64_t)t * p.topk;
    int* slots = reinterpret_cast<int*>(sm + kOffSlot);
    uint32_t* masks = reinterpret_cast<uint32_t*>(sm + kOffMask);
    for (int b = 0; b < nb; ++b) {
      const int s = b % kStages;
      if (b >= kStages) W.wait(bar(kBarKvEmpty + s), ((b / kStages) - 1) & 1);
      if (pt < kBN) {
        const int pos = k0 + b * kBN + pt;
        int id = -1;
        if (pos < k1) {
          id = __ldg(idx_row + pos);
          if (id >= p.num_slots) {
            atomicCAS(p.status, 0, kStatusBadIndex);
            id = -1;
          }
        }
        id = id < 0 ? -1 : id;
        slots[s * kBN + pt] = id;
        const uint32_t m = __ballot_sync(0xffffffffu, id >= 0);
        if (lane == 0) masks[s * 2 + (pt >> 5)] = m;
      }
      named_bar_sync(1, kProducers);
      const uint32_t tile = sb + kOffTile + s * kTileBytes;
      for (int it = pt; it < kBN * nc; it += kProducers) {
        const int row = it / nc, cj = it - row * nc;
        const int id = slots[s * kBN + row];
        const uint32_t dst = tile + (cj >> 3) * kAtomBytes + row * 128 +
                             ((((uint32_t)cj & 7u) ^ ((uint32_t)row & 7u)) << 4);
        const uint8_t* src = kv + (size_t)(id < 0 ? 0 : id) * row_bytes +
                             (size_t)(g_lo + 8 * cj) * 2;
        cp_async_16(dst, src, id < 0 ? 0u : 16u);
      }
      cp_async_mbar_arrive(bar(kBarKvFull + s));
      mbar_arrive(bar(kBarKvFull + s));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ---- softmax warpgroup ---------------------------------------------------
    const int i = tid - 128;                     // head row == TMEM lane
    const uint32_t lane_base = ((uint32_t)(warp & 3) * 32u) << 16;
    const bool own = (uint32_t)(i >> 6) == r;    // this CTA owns head i
    const int head = i;
    // Q half -> TMEM (rows >= h are zero).
    {
      const int qn = a.ksteps * 16;              // channels kept
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const uint16_t*>(p.q) +
          ((int64_t)t * p.h + head) * p.d_qk + a.q_lo[r]);
      for (int c = 0; c < qn / 2; c += 16) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = head < p.h ? __ldg(qrow + c + k) : 0u;
        __syncwarp();
        tmem_st16(tmem + lane_base + kColQ + c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarQReady));
    }
    float m_run = -INFINITY;   // running max (log2 units), own heads
    float l_run = 0.f;         // running sum of P, own heads
    float l_peer = 0.f;        // sum for a peer-owned head (from the peer)
    float* Xs = reinterpret_cast<float*>(sm + kOffX);
    float* Alpha = reinterpret_cast<float*>(sm + kOffAlpha);
    float* Lx = reinterpret_cast<float*>(sm + kOffL);
    const uint32_t* masks = reinterpret_cast<const uint32_t*>(sm + kOffMask);
    const uint32_t x_peer = mapa(sb + kOffX, peer);
    const uint32_t p_peer = mapa(sb + kOffP, peer);
    const uint32_t alpha_peer = mapa(sb + kOffAlpha, peer);
    const uint32_t l_peer_addr = mapa(sb + kOffL, peer);

    // O row *= alpha.  tcgen05.ld/st are warp-collective (.sync.aligned), so
    // the whole warp takes this path when any of its lanes needs it; lanes
    // with nothing to rescale pass alpha = 1.
    auto rescale_o = [&](float alpha, int b) {
      W.wait(bar(kBarODone), (b - 1) & 1);
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 256; c += 16) {
        uint32_t w[16];
        tmem_ld16(tmem + lane_base + kColO + c, w);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * alpha);
        tmem_st16(tmem + lane_base + kColO + c, w);
      }
      tmem_wait_st();
    };

    for (int b = 0; b < nb; ++b) {
      const int s = b % kStages;
      const int buf = b & 1;
      float sp[kBN];
      W.wait(bar(kBarSFull), b & 1);
      __syncwarp();
      tc_fence_after();
      {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < kBN; c += 16) {
          tmem_ld16(tmem + lane_base + kColS + c, w);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) sp[c + k] = __uint_as_float(w[k]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty));
      if (!own) {
        // Send this partial row to the owner; get back P's scale data.
        const int prow = i - 64 * (int)peer;
        if (b >= 2) W.wait(bar(kBarXFree + buf), ((b >> 1) - 1) & 1);
        const uint32_t dst = x_peer + buf * kXBytes + prow * kXStride * 4;
#pragma unroll
        for (int c = 0; c < kBN; c += 4)
          st_cluster_v4(dst + c * 4, __float_as_uint(sp[c]), __float_as_uint(sp[c + 1]),
                        __float_as_uint(sp[c + 2]), __float_as_uint(sp[c + 3]));
        mbar_arrive_remote(mapa(bar(kBarXFull + buf), peer));
        W.wait_cluster(bar(kBarPxFull + buf), (b >> 1) & 1);
        const float alpha = Alpha[buf * 128 + i];
        l_peer = Lx[buf * 128 + i];
        if (b >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o(alpha, b);
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + buf));
      } else {
        const int prow = i - 64 * (int)r;
        W.wait_cluster(bar(kBarXFull + buf), (b >> 1) & 1);
        const float* xr = Xs + buf * (kXBytes / 4) + prow * kXStride;
#pragma unroll
        for (int c = 0; c < kBN; c += 4) {
          const float4 x = *reinterpret_cast<const float4*>(xr + c);
          sp[c] += x.x; sp[c + 1] += x.y; sp[c + 2] += x.z; sp[c + 3] += x.w;
        }
        mbar_arrive_remote(mapa(bar(kBarXFree + buf), peer));
        // a5: masked online softmax (log2 domain).  The producers' mask of
        // this block is published with their arrival on the stage barrier.
        W.wait(bar(kBarKvFull + s), (b / kStages) & 1);
        const uint32_t m_lo = masks[s * 2], m_hi = masks[s * 2 + 1];
        float bmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kBN; ++j) {
          const bool ok = ((j < 32 ? m_lo >> j : m_hi >> (j - 32)) & 1u) != 0u;
          sp[j] = ok ? sp[j] * a.scale_log2 : -INFINITY;
          bmax = fmaxf(bmax, sp[j]);
        }
        float alpha = 1.f;
        if (bmax > m_run + 8.f) {          // also true for the first finite max
          alpha = exp2f(m_run - bmax);     // 0 when m_run = -inf
          m_run = bmax;
        }
        uint32_t pk[kBN / 2];
        float lsum = 0.f;
        if (m_run == -INFINITY) {
#pragma unroll
          for (int j = 0; j < kBN / 2; ++j) pk[j] = 0u;
        } else {
#pragma unroll
          for (int j = 0; j < kBN; j += 2) {
            // The row sum uses the unrounded values (it sets the LSE); P
            // goes to the PV MMA in bf16.
            const float e0 = exp2f(sp[j] - m_run), e1 = exp2f(sp[j + 1] - m_run);
            pk[j / 2] = pack_bf16(e0, e1);
            lsum += e0 + e1;
          }
        }
        l_run = l_run * alpha + lsum;
        if (b >= 2) W.wait(bar(kBarPEmpty + buf), ((b >> 1) - 1) & 1);
        // P row (64 bf16 = 8 chunks of 16 B), swizzled, here and in the peer.
        uint8_t* prow_ptr = sm + kOffP + buf * kPBytes + i * 128;
        const uint32_t prow_peer = p_peer + buf * kPBytes + i * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = ((uint32_t)j ^ ((uint32_t)i & 7u)) << 4;
          *reinterpret_cast<uint4*>(prow_ptr + off) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          st_cluster_v4(prow_peer + off, pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                        pk[4 * j + 3]);
        }
        st_cluster_b32(alpha_peer + (buf * 128 + i) * 4, __float_as_uint(alpha));
        st_cluster_b32(l_peer_addr + (buf * 128 + i) * 4, __float_as_uint(l_run));
        fence_proxy_async();
        mbar_arrive_remote(mapa(bar(kBarPxFull + buf), peer));
        if (b >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o(alpha, b);
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + buf));
      }
    }

    // ---- a7: epilogue ---------------------------------------------------------
    if (nb > 0) {
      W.wait(bar(kBarODone), (nb - 1) & 1);
      tc_fence_after();
    }
    const float l_row = own ? l_run : l_peer;
    const bool empty = !(l_row > 0.f) || nb == 0;
    const float inv = empty ? 0.f : 1.f / l_row;
    const bool live = head < p.h;          // pad rows past h are not written
    const int64_t orow = (int64_t)t * p.h + (live ? head : 0);
    // Every lane of the warpgroup runs the TMEM loads (warp-collective);
    // only the stores depend on the lane's head.
#pragma unroll 1
    for (int c = 0; c < 256; c += 16) {
      uint32_t w[16];
      __syncwarp();
      if (nb > 0) {
        tmem_ld16(tmem + lane_base + kColO + c, w);
        tmem_wait_ld();
      }
      if (!live) {
      } else if (p.splits > 1) {
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
    if (live && own) {
      const float lse_v =
          empty ? -INFINITY : (m_run + log2f(l_row)) * 0.69314718055994530942f;
      if (p.splits > 1)
        p.lse_part[(int64_t)split * p.T * p.h + orow] = lse_v;
      else if (p.lse)
        p.lse[orow] = lse_v;
    }
  }

  // ---- teardown: no CTA leaves while its peer may still touch its memory --
  // The peer's last PV commits arrive on this CTA's P-empty barriers
  // asynchronously; wait for them before the cluster barrier.
  if (tid == 128 && nb > 0) {
    if (nb >= 2) W.wait(bar(kBarPEmpty + ((nb - 2) & 1)), ((nb - 2) >> 1) & 1);
    W.wait(bar(kBarPEmpty + ((nb - 1) & 1)), ((nb - 1) >> 1) & 1);
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

bool tc_supported(int h, int d_qk, int kv_format) {
  return h >= 1 && h <= 128 && (d_qk == 576 || d_qk == 512) && kv_format == kBf16;
}

cudaError_t launch_tc(const FwdParams& p, cudaStream_t stream) {
  TcArgs a{};
  a.p = p;
  if (p.d_qk == 576) {
    a.g_lo[0] = 0;   a.n_chunks[0] = 36; a.qk_lo[0] = 0;  a.q_lo[0] = 0;
    a.g_lo[1] = 256; a.n_chunks[1] = 40; a.qk_lo[1] = 32; a.q_lo[1] = 288;
    a.ksteps = 18;
  } else {
    a.g_lo[0] = 0;   a.n_chunks[0] = 32; a.qk_lo[0] = 0; a.q_lo[0] = 0;
    a.g_lo[1] = 256; a.n_chunks[1] = 32; a.qk_lo[1] = 0; a.q_lo[1] = 256;
    a.ksteps = 16;
  }
  a.scale_log2 = p.sm_scale * 1.4426950408889634f;
  const int64_t clusters = (int64_t)p.T * p.splits;
  if (clusters * 2 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(smla_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  smla_tc_kernel<<<(unsigned)(clusters * 2), kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace smla

// tc_common.cuh — device helpers shared by the two tensor-core kernels
// (heads-major smla_tc.cu, keys-major smla_tc_keys.cu): bounded waits with a
// per-block abort flag, exact E4M3 -> bf16 conversion, bf16 packing, named
// barriers, and the bf16 cache tensor map used by TMA gathers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "smla_internal.h"
#include "tc_ptx.cuh"

namespace smla {

// Named barriers over whole warps.  bar.sync / bar.red are the .aligned
// forms: every lane of a warp must execute them together, so the warp is
// reconverged first (lanes leave a spin-wait loop at different times, and an
// aligned barrier reached by a split warp is undefined behaviour).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// OR of `pred` over the `n` threads that meet at named barrier `id`.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
  __syncwarp();
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return out != 0u;
}

// Bounded waits.  A wait that runs out (or sees that another block of the
// same launch gave up) records the timeout status, bumps the device's abort
// counter, sets this block's abort flag, and from then on every wait of the
// block returns at once, so the block still reaches its teardown.  The
// counter's value when the thread started is the launch's reference: a
// timeout left over from an earlier launch (whose status word may still be
// set) does not stop this one.  Results of an aborted launch are undefined;
// no access goes out of bounds.
struct Waiter {
  volatile int* abort;   // this block's flag (shared memory)
  int* status;           // device status word
  int* ctr;              // device abort counter
  int ctr0;              // its value when this thread started
  uint64_t limit_ns;     // time limit of one wait
  __device__ __forceinline__ void fail() {
    if (!*abort) {
      *abort = 1;
      atomicAdd(ctr, 1);
      atomicCAS(status, 0, kStatusTimeout);
    }
  }
  __device__ __forceinline__ void wait(uint32_t bar, uint32_t parity) {
    if (*abort) return;
    if (!ptx::mbar_wait_bounded<false>(bar, parity, limit_ns, ctr, ctr0)) fail();
  }
  __device__ __forceinline__ void wait_cluster(uint32_t bar, uint32_t parity) {
    if (*abort) return;
    if (!ptx::mbar_wait_bounded<true>(bar, parity, limit_ns, ctr, ctr0)) fail();
  }
  // Teardown: wait for asynchronous work this block started itself (TMA
  // copies into its shared memory, MMAs reading it and writing its TMEM),
  // also after an abort; only the time limit ends it.
  __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    if (!ptx::mbar_wait_bounded<false>(bar, parity, limit_ns, nullptr, 0)) fail();
  }
};
__device__ __forceinline__ Waiter make_waiter(volatile int* abort_flag, const FwdParams& p) {
  return Waiter{abort_flag, p.status, p.abort_ctr, *reinterpret_cast<volatile int*>(p.abort_ctr),
                p.wait_limit_ns};
}

// Four E4M3 bytes -> four bf16 (two bf16x2 words), exactly: every E4M3 value
// is a bf16 value.  The byte's exponent and mantissa fields are placed in the
// bf16 fields (which reads the value times 2^-120, bias 7 vs 127; E4M3
// subnormals land on bf16 subnormals), then one exact bf16 multiply by 2^120
// restores it.  The NaN codes S.1111.111 (which the placement would read as
// +-480) are made bf16 NaN, as the format defines them.
__device__ __forceinline__ uint32_t e4m3x2_lanes_to_bf16x2(uint32_t x) {
  // x holds one byte in the low byte of each 16-bit lane
  uint32_t bits = ((x & 0x007F007Fu) << 4) | ((x & 0x00800080u) << 8);
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&bits);
  const uint32_t k2 = 0x7B807B80u;                 // (2^120, 2^120) in bf16
  v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&k2));
  const uint32_t nan = __vcmpeq2(x & 0x007F007Fu, 0x007F007Fu);   // 0xFFFF per NaN code
  return *reinterpret_cast<uint32_t*>(&v) | (nan & 0x7FC07FC0u);
}
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_lanes_to_bf16x2(__byte_perm(w, 0u, 0x4140u));   // bytes 0, 1
  hi = e4m3x2_lanes_to_bf16x2(__byte_perm(w, 0u, 0x4342u));   // bytes 2, 3
}

// The same conversion (the same bf16 bits) in fewer instructions.  Per bf16
// pair: one byte permute puts each E4M3 byte in the low byte of a 16-bit lane
// with copies of its sign bit above it; one shift by 4 then moves exponent
// and mantissa to bf16 bits 10..4 and a sign copy to bit 15, and one mask
// clears the rest (bits spilled into the upper lane fall on masked bits).
// The keys-major loader, whose warps are bound by instruction issue, uses
// this form; the heads-major converter measured faster with the first.
__device__ __forceinline__ uint32_t e4m3_spread_to_bf16x2(uint32_t x) {
  uint32_t bits = (x << 4) & 0x87F087F0u;
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&bits);
  const uint32_t k2 = 0x7B807B80u;                 // (2^120, 2^120) in bf16
  v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&k2));
  return *reinterpret_cast<uint32_t*>(&v);
}
// prmt with sign replication: selector nibble 8 + k yields the sign bit of
// byte k repeated over the byte (__byte_perm reads only 3 bits a nibble).
template <uint32_t kSel>
__device__ __forceinline__ uint32_t prmt_sign(uint32_t w) {
  uint32_t x;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(w), "n"(kSel));
  return x;
}
__device__ __forceinline__ void e4m3x4_to_bf16_sx(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3_spread_to_bf16x2(prmt_sign<0x9180u>(w));   // bytes 0, 1
  hi = e4m3_spread_to_bf16x2(prmt_sign<0xB3A2u>(w));   // bytes 2, 3
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// acc + the two bf16 values packed in pk (low half first), each added as an
// exact f32 value (PTX add.f32.bf16: one instruction per value).
__device__ __forceinline__ float add_bf16x2_f32(float acc, uint32_t pk) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\t"
      "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %0, h, %0;\n\t}"
      : "+f"(acc) : "r"(pk));
  return acc;
}

// The slot ids at top-k positions [k0, k0 + n) of one index row into
// slots[0, n) (n a multiple of 4), -1 where masked: at or past k1, negative,
// or >= num_slots (the last makes the return value true).  The nthr threads
// (index pt) share the row in 4-id pieces; each thread issues every load of
// a batch of 8 pieces before its first store (16-byte loads when the row
// position is 16-byte aligned), so a unit's ids arrive in about one memory
// latency instead of one latency per id.
__device__ __forceinline__ bool load_slot_ids(const int32_t* row, int k0, int k1, int topk,
                                              int n, int64_t num_slots, int* slots, int pt,
                                              int nthr) {
  bool bad = false;
  const bool vec = (reinterpret_cast<uintptr_t>(row + k0) & 15u) == 0;
  for (int base = 4 * pt; base < n; base += 4 * nthr * 8) {
    int4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 4 * nthr * u;
      const int pos = k0 + j;
      v[u] = make_int4(-1, -1, -1, -1);
      if (j < n && pos < k1) {
        if (vec && pos + 3 < topk) {
          v[u] = __ldg(reinterpret_cast<const int4*>(row + pos));
        } else {
          v[u].x = __ldg(row + pos);
          if (pos + 1 < topk) v[u].y = __ldg(row + pos + 1);
          if (pos + 2 < topk) v[u].z = __ldg(row + pos + 2);
          if (pos + 3 < topk) v[u].w = __ldg(row + pos + 3);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 4 * nthr * u;
      if (j < n) {
        const int e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          int id = k0 + j + q < k1 ? e[q] : -1;
          if (id >= num_slots) {
            bad = true;
            id = -1;
          }
          slots[j + q] = id < 0 ? -1 : id;
        }
      }
    }
  }
  return bad;
}

// The same for request-local positions (smla_fwd_paged): each loaded entry
// is translated through the block table by to_slot.  The row's table
// lookups of a batch are issued together as well (two memory latencies per
// batch).
__device__ __forceinline__ bool load_slot_ids_paged(const FwdParams& p, int t, int k0, int k1,
                                                    int n, int* slots, int pt, int nthr) {
  bool bad = false;
  const int32_t* row = p.indices + (int64_t)t * p.topk;
  const int req = token_req(p, t, bad);
  for (int base = 4 * pt; base < n; base += 4 * nthr * 8) {
    int e[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 4 * nthr * u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pos = k0 + j + q;
        e[u][q] = (j < n && pos < k1) ? __ldg(row + pos) : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 4 * nthr * u;
      if (j < n) {
#pragma unroll
        for (int q = 0; q < 4; ++q) slots[j + q] = to_slot(p, req, e[u][q], bad);
      }
    }
  }
  return bad;
}

// Either loader, by the launch's index kind.
__device__ __forceinline__ bool load_unit_slots(const FwdParams& p, int t, int k0, int k1, int n,
                                                int* slots, int pt, int nthr) {
  if (p.block_table) return load_slot_ids_paged(p, t, k0, k1, n, slots, pt, nthr);
  return load_slot_ids(p.indices + (int64_t)t * p.topk, k0, k1, p.topk, n, p.num_slots, slots,
                       pt, nthr);
}

// Longest-first unit order for launches of at most kLptMaxUnits units.  A
// unit u = (token u / splits, range u % splits) has ceil(n / bn) blocks of
// work, n = the valid positions of its range.  The block scheduler starts
// CTAs (clusters) roughly in index order, so when the unit sizes vary, a
// late large unit sets the end of the launch; taking the units in
// decreasing size instead lets the small ones fill in at the end.  Every
// thread of the CTA calls this with the same `rank` (the CTA's or cluster's
// index) and gets the unit at that rank of the order: units sorted by
// decreasing block count, ties in unit order.  The result depends only on
// (rank, valid_len, the plan), so the CTAs of a cluster agree and every unit
// is taken exactly once.  `scratch` is shared memory for (kLptMaxBlocks + 2)
// + nthr / 32 + 1 ints; the call ends with a block-wide barrier.
constexpr int kLptMaxUnits = 4096;
constexpr int kLptMaxBlocks = 64;
__device__ __forceinline__ int unit_blocks(const FwdParams& p, int u, int bn) {
  const int t = u / p.splits, sp = u - t * p.splits;
  int v = p.topk;
  if (p.valid_len) v = min(max(__ldg(p.valid_len + t), 0), p.topk);
  const int k0 = sp * p.split_len, k1 = min(k0 + p.split_len, v);
  return k1 > k0 ? min((k1 - k0 + bn - 1) / bn, kLptMaxBlocks) : 0;
}
static __device__ __noinline__ int lpt_unit(const FwdParams& p, int rank, int n_units, int bn,
                                        int* scratch) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  int* hist = scratch;                             // [kLptMaxBlocks + 1]
  int* sel = scratch + kLptMaxBlocks + 1;          // [0] bucket, [1] index in it, then the unit
  int* wsum = sel + 2;                             // [nwarps]
  for (int c = tid; c <= kLptMaxBlocks; c += nthr) hist[c] = 0;
  __syncthreads();
  for (int u = tid; u < n_units; u += nthr) atomicAdd(&hist[unit_blocks(p, u, bn)], 1);
  __syncthreads();
  if (tid == 0) {                                  // the bucket holding `rank`
    int start = 0, c = kLptMaxBlocks;
    for (; c > 0 && start + hist[c] <= rank; --c) start += hist[c];
    sel[0] = c;
    sel[1] = rank - start;
  }
  __syncthreads();
  const int cb = sel[0], k = sel[1];
  // Every unit the same size: the order is the unit order.
  if (hist[cb] == n_units) {
    __syncthreads();
    return rank;
  }
  // The k-th unit (in unit order) of bucket cb: each thread counts its chunk
  // of units, a block-wide scan places the chunks, and the thread whose
  // chunk holds it writes it.
  const int per = (n_units + nthr - 1) / nthr;
  const int u0 = tid * per, u1 = min(u0 + per, n_units);
  int cnt = 0;
  for (int u = u0; u < u1; ++u) cnt += unit_blocks(p, u, bn) == cb;
  int inc = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int before = inc - cnt;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  if (k >= before && k < before + cnt) {
    int seen = before;
    for (int u = u0; u < u1; ++u) {
      if (unit_blocks(p, u, bn) == cb) {
        if (seen == k) {
          sel[0] = u;
          break;
        }
        ++seen;
      }
    }
  }
  __syncthreads();
  const int unit = sel[0];
  __syncthreads();
  return unit;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library does not link libcuda directly); nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// A bf16 cache [num_slots, d_qk] as a 2-D tensor with 64-channel x 1-row
// boxes and the 128-byte swizzle of the MMA operand tiles (TMA tile::gather4
// reads four such rows per instruction; a row id of -1 reads zeros).
cudaError_t encode_bf16_rows_map(CUtensorMap* map, const void* kv, int d_qk,
                                 int64_t num_slots);

}  // namespace smla

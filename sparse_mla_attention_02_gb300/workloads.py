"""Seeded synthetic inputs for the sparse MLA attention forward.

This module only draws data: values, slot ids and valid counts, shaped like
the workloads the pages describe.  It holds none of the method's arithmetic,
and it is the one module that both the CUDA path's callers (tests, bench) and
the oracle's callers share.

Recipes (the readings behind them are listed in the design notes):

* Values: q and bf16 cache rows are N(0,1) float32 rounded to bf16 (RNE).
* FP8 per-tensor cache: stored byte = e4m3(clamp(N(0,1)/k_scale, +-448)).
* FP8 group cache: scales ~ U[lo, hi] per (slot, 128-channel group); stored
  byte = e4m3(clamp(N(0,1)/scale[slot, c // 128], +-448)).  The E4M3 encoder
  is torch's float -> float8_e4m3fn cast (round to nearest even).
* fp8_ds_mla 656-byte rows: the 512 ckv channels as in the group cache (four
  scales per slot), packed as [512 code bytes | 4 fp32 scales | 64 bf16 rope
  values N(0,1)], little-endian.
* E4M3 with four ckv group scales and one kpe scale: ckv codes as in the
  group cache (four scales per slot), rope codes as in the per-tensor cache
  with kpe_scale.
* Index rows: distinct slot ids in random order for the valid prefix, -1 past
  it (vLLM "Sparse MLA on Hopper" test file: randperm rows, -1 tails;
  flashinfer_mla_sparse_sm90.py, forward_mqa: compacted prefix, -1 past it).

Large value tensors are drawn directly on the requested device with a seeded
torch generator; index rows are drawn on the host with numpy and copied.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_FP8_E4M3_GROUP128 = 2
KV_FP8_DS_MLA = 3
KV_FP8_E4M3_GROUP4_KPE = 4
DS_MLA_ROW_BYTES = 656

E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    T: int
    h: int
    d_qk: int
    d_v: int
    topk: int
    num_slots: int
    kv_dtype: int
    sm_scale: float
    q: torch.Tensor            # bf16 [T, h, d_qk]
    kv: torch.Tensor           # bf16 [S, d_qk] or uint8 [S, d_qk]
    k_scale: torch.Tensor | None  # f32 [1] or [S, G] or None
    indices: torch.Tensor      # int32 [T, topk]
    valid_len: torch.Tensor    # int32 [T]
    real_heads: int = 0        # heads that carry data (pad heads excluded)
    notes: dict = field(default_factory=dict)
    kpe_scale: float = 1.0     # rope scale of KV_FP8_E4M3_GROUP4_KPE

    def to(self, device) -> "Workload":
        mv = lambda x: None if x is None else x.to(device)
        return Workload(self.name, self.T, self.h, self.d_qk, self.d_v,
                        self.topk, self.num_slots, self.kv_dtype,
                        self.sm_scale, mv(self.q), mv(self.kv),
                        mv(self.k_scale), mv(self.indices),
                        mv(self.valid_len), self.real_heads, dict(self.notes),
                        self.kpe_scale)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, device, gen, chunk=1 << 27):
    """N(0,1) float32 rounded to bf16, drawn in bounded chunks."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, device=device).to(torch.bfloat16)
    return out.view(*shape)


def e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """float32 -> E4M3 byte codes (saturating at +-448, RNE)."""
    return x.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_cache_per_tensor(S, d, k_scale, device, gen, chunk_rows=1 << 18):
    out = torch.empty((S, d), dtype=torch.uint8, device=device)
    for s in range(0, S, chunk_rows):
        e = min(S, s + chunk_rows)
        x = torch.randn((e - s, d), generator=gen, device=device) / k_scale
        out[s:e] = e4m3_bytes(x)
    return out


def fp8_cache_group(S, d, scales, device, gen, chunk_rows=1 << 18):
    G = scales.shape[1]
    assert G == (d + 127) // 128
    out = torch.empty((S, d), dtype=torch.uint8, device=device)
    grp = torch.arange(d, device=device) // 128
    for s in range(0, S, chunk_rows):
        e = min(S, s + chunk_rows)
        x = torch.randn((e - s, d), generator=gen, device=device)
        x = x / scales[s:e][:, grp]
        out[s:e] = e4m3_bytes(x)
    return out


def ds_mla_rows(codes: torch.Tensor, scales: torch.Tensor, rope: torch.Tensor) -> torch.Tensor:
    """Pack [512 E4M3 bytes | 4 fp32 scales | 64 bf16] into 656-byte rows."""
    S = codes.shape[0]
    assert codes.shape == (S, 512) and scales.shape == (S, 4) and rope.shape == (S, 64)
    return torch.cat([codes, scales.float().contiguous().view(torch.uint8),
                      rope.to(torch.bfloat16).contiguous().view(torch.uint8)], dim=1).contiguous()


def index_rows(rng: np.random.Generator, T, topk, valid, pick):
    """int32 [T, topk]: row t = shuffled pick(t, valid[t]) then -1 tail."""
    idx = np.full((T, topk), -1, dtype=np.int32)
    for t in range(T):
        v = int(valid[t])
        if v > 0:
            row = np.asarray(pick(t, v), dtype=np.int64)
            assert row.shape == (v,)
            idx[t, :v] = rng.permutation(row).astype(np.int32)
    return idx


# ---------------------------------------------------------------- configs --

def tiny(device="cpu", seed=0) -> Workload:
    """T=4, h=16, d_qk=576, 256 bf16 slots, topk=64, valid {64,40,17,1}."""
    T, h, d_qk, d_v, topk, S = 4, 16, 576, 512, 64, 256
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    kv = bf16_normal((S, d_qk), device, g)
    valid = np.array([64, 40, 17, 1], dtype=np.int32)
    idx = index_rows(rng, T, topk, valid,
                     lambda t, v: rng.choice(S, v, replace=False))
    return Workload("tiny", T, h, d_qk, d_v, topk, S, KV_BF16,
                    1.0 / math.sqrt(576), q, kv, None,
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h)


def bf16_decode(device="cpu", seed=1001, T=64, h=128, per_req=32768) -> Workload:
    """One token per request; 2048 distinct slots from its own request."""
    d_qk, d_v, topk = 576, 512, 2048
    S = T * per_req
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    kv = bf16_normal((S, d_qk), device, g)
    valid = np.full(T, topk, dtype=np.int32)
    idx = index_rows(rng, T, topk, valid, lambda t, v: t * per_req +
                     rng.choice(per_req, v, replace=False))
    return Workload("bf16_decode", T, h, d_qk, d_v, topk, S, KV_BF16,
                    1.0 / math.sqrt(576), q, kv, None,
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h)


def fp8_nope_decode(device="cpu", seed=1002, T=128, h=64, real_heads=48,
                    num_blocks=4096, block_size=64, k_scale=0.05) -> Workload:
    """NoPE (d_qk=d_v=512) E4M3 cache with a per-tensor scale; 48 real heads
    padded with zero heads to 64; valid ~ U[256, 2048]."""
    d_qk = d_v = 512
    topk = 2048
    S = num_blocks * block_size
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    q[:, real_heads:, :] = 0
    kv = fp8_cache_per_tensor(S, d_qk, k_scale, device, g)
    valid = rng.integers(256, 2049, size=T).astype(np.int32)
    idx = index_rows(rng, T, topk, valid,
                     lambda t, v: rng.choice(S, v, replace=False))
    return Workload("fp8_nope_decode", T, h, d_qk, d_v, topk, S, KV_FP8_E4M3,
                    1.0 / math.sqrt(512), q, kv,
                    torch.tensor([k_scale], dtype=torch.float32, device=device),
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), real_heads)


def _causal_pick(rng):
    def pick(t, v):
        # v distinct ids from [0, t]; v == t+1 takes all of them.
        if v == t + 1:
            return np.arange(t + 1)
        return rng.choice(t + 1, v, replace=False)
    return pick


def bf16_prefill(device="cpu", seed=1003, T=8192, h=128, topk=2048) -> Workload:
    """One T-token sequence; token i selects min(i+1, topk) distinct slots
    of [0, i] (causality by selection)."""
    d_qk, d_v = 576, 512
    S = T
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    kv = bf16_normal((S, d_qk), device, g)
    valid = np.minimum(np.arange(T) + 1, topk).astype(np.int32)
    idx = index_rows(rng, T, topk, valid, _causal_pick(rng))
    return Workload("bf16_prefill", T, h, d_qk, d_v, topk, S, KV_BF16,
                    1.0 / math.sqrt(576), q, kv, None,
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h)


def mixed_fp8_group(device="cpu", seed=1004, n_req=32, tok_per_req=512,
                    ctx=65536, h=16, recent=4096, scale_lo=0.01,
                    scale_hi=0.1) -> Workload:
    """32 requests x 512 tokens over 65536-slot contexts; E4M3 cache with
    per-token x 128-channel-group scales; valid ~ U[1, 2048]; half of each
    row from the most recent 4096 positions, the rest uniform before them."""
    d_qk, d_v, topk = 576, 512, 2048
    T = n_req * tok_per_req
    S = n_req * ctx
    G = (d_qk + 127) // 128
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    scales = (torch.rand((S, G), generator=g, device=device)
              * (scale_hi - scale_lo) + scale_lo).float()
    kv = fp8_cache_group(S, d_qk, scales, device, g)
    valid = rng.integers(1, topk + 1, size=T).astype(np.int32)

    def pick(t, v):
        r, i = divmod(t, tok_per_req)
        p = ctx - tok_per_req + i           # position of token t in its context
        a = (v + 1) // 2                    # from the recent window [p-recent+1, p]
        b = v - a                           # uniform from [0, p-recent+1)
        lo = p - recent + 1
        near = lo + rng.choice(recent, a, replace=False)
        far = rng.choice(lo, b, replace=False) if b else np.zeros(0, np.int64)
        return r * ctx + np.concatenate([near, far])

    idx = index_rows(rng, T, topk, valid, pick)
    return Workload("mixed_fp8_group", T, h, d_qk, d_v, topk, S,
                    KV_FP8_E4M3_GROUP128, 1.0 / math.sqrt(576), q, kv, scales,
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h)


def ds_mla_decode(device="cpu", seed=1005, T=128, h=128, per_req=16384,
                  scale_range=(0.01, 0.1)) -> Workload:
    """Decode on the 656-byte fp8_ds_mla cache: one token per request, 128
    heads, 2048 distinct slots from its own request's 16384; the shape of the
    pages' FP8 FlashMLA decode (heads padded to 128, fp8_ds_mla rows), with
    the rows drawn like the other FP8 caches (E4M3 of N(0,1)/scale, scales
    ~U[0.01, 0.1] per 128-channel group, bf16 N(0,1) rope)."""
    d_qk, d_v, topk = 576, 512, 2048
    S = T * per_req
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    lo, hi = scale_range
    scales = (torch.rand((S, 4), generator=g, device=device) * (hi - lo) + lo).float()
    codes = fp8_cache_group(S, 512, scales, device, g)
    kv = ds_mla_rows(codes, scales, bf16_normal((S, 64), device, g))
    del codes
    valid = np.full(T, topk, dtype=np.int32)
    idx = index_rows(rng, T, topk, valid, lambda t, v: t * per_req +
                     rng.choice(per_req, v, replace=False))
    return Workload("ds_mla_decode", T, h, d_qk, d_v, topk, S, KV_FP8_DS_MLA,
                    1.0 / math.sqrt(576), q, kv, None,
                    torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h)


CONFIGS = {
    "tiny": tiny,
    "bf16_decode": bf16_decode,
    "fp8_nope_decode": fp8_nope_decode,
    "bf16_prefill": bf16_prefill,
    "mixed_fp8_group": mixed_fp8_group,
    "ds_mla_decode": ds_mla_decode,      # secondary: not one of the five configs
}


def custom(T, h, d_qk=576, d_v=512, topk=64, num_slots=256, kv_dtype=KV_BF16,
           valid=None, seed=0, device="cpu", sm_scale=None, k_scale=0.05,
           scale_range=(0.01, 0.1), distinct=True, name="custom") -> Workload:
    """Small scenario builder for tests: random values, rows of `valid[t]`
    slot ids (distinct unless told otherwise), -1 tails."""
    g = _gen(device, seed)
    rng = np.random.default_rng(seed)
    q = bf16_normal((T, h, d_qk), device, g)
    G = (d_qk + 127) // 128
    scales = None
    kpe_scale = 1.0
    if kv_dtype == KV_BF16:
        kv = bf16_normal((num_slots, d_qk), device, g)
    elif kv_dtype in (KV_FP8_DS_MLA, KV_FP8_E4M3_GROUP4_KPE):
        assert d_qk == 576
        lo, hi = scale_range
        scales = (torch.rand((num_slots, 4), generator=g, device=device)
                  * (hi - lo) + lo).float()
        codes = fp8_cache_group(num_slots, 512, scales, device, g)
        if kv_dtype == KV_FP8_DS_MLA:
            kv = ds_mla_rows(codes, scales, bf16_normal((num_slots, 64), device, g))
            scales = None
        else:
            kpe_scale = float(k_scale)
            kv = torch.cat([codes, fp8_cache_per_tensor(num_slots, 64, kpe_scale, device, g)],
                           dim=1).contiguous()
    elif kv_dtype == KV_FP8_E4M3:
        kv = fp8_cache_per_tensor(num_slots, d_qk, k_scale, device, g)
        scales = torch.tensor([k_scale], dtype=torch.float32, device=device)
    else:
        lo, hi = scale_range
        scales = (torch.rand((num_slots, G), generator=g, device=device)
                  * (hi - lo) + lo).float()
        kv = fp8_cache_group(num_slots, d_qk, scales, device, g)
    if valid is None:
        valid = rng.integers(0, topk + 1, size=T)
    valid = np.asarray(valid, dtype=np.int32)
    if distinct:
        pick = lambda t, v: rng.choice(num_slots, v, replace=False)
    else:
        pick = lambda t, v: rng.integers(0, num_slots, size=v)
    idx = index_rows(rng, T, topk, valid, pick)
    return Workload(name, T, h, d_qk, d_v, topk, num_slots, kv_dtype,
                    (1.0 / math.sqrt(d_qk)) if sm_scale is None else sm_scale,
                    q, kv, scales, torch.from_numpy(idx).to(device),
                    torch.from_numpy(valid).to(device), h, kpe_scale=kpe_scale)


def token_subset(w: Workload, sel, device="cpu") -> Workload:
    """Tokens `sel` of `w`, with a compact copy of only the cache rows (and
    group scales) they select, ids remapped into it; -1 and out-of-range ids
    stay masked.  Lets a checker see a few tokens of a multi-GB pool."""
    sel_t = torch.as_tensor(np.asarray(sel, dtype=np.int64),
                            device=w.indices.device)
    idx = w.indices[sel_t].long()
    ok = (idx >= 0) & (idx < w.num_slots)
    rows = torch.unique(idx[ok])
    remap = torch.searchsorted(rows, idx.clamp(min=0))
    new_idx = torch.where(ok, remap, torch.full_like(remap, -1)).int()
    ks = w.k_scale
    if ks is not None and ks.dim() == 2:
        ks = ks[rows]
    mv = lambda x: None if x is None else x.to(device)
    return Workload(w.name, int(sel_t.numel()), w.h, w.d_qk, w.d_v, w.topk,
                    max(1, int(rows.numel())), w.kv_dtype, w.sm_scale,
                    mv(w.q[sel_t]), mv(w.kv[rows]), mv(ks), mv(new_idx),
                    mv(w.valid_len[sel_t]), w.real_heads, dict(w.notes))

"""The group-quantizing E4M3 cache write (smla_cache_write_e4m3_group):
bytes and scales bit-exact against the oracle's write (codes are integer
results decided in fp32 on both sides), skipped rows untouched, bad slots
flagged, and the written cache read back by smla_fwd within the forward's
parity bounds."""
import math

import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import bits16, oracle_fwd

import oracle

pytestmark = pytest.mark.gpu


def rows(N, d_qk, seed, spread=3.0):
    """bf16 rows; per-row magnitudes exp(spread * N(0,1)) for the bit-exact
    tests, unit scale (spread 0) where the forward reads them back, so that
    O stays in the range the forward's absolute bound is stated for."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((N, d_qk), generator=g)
    x *= torch.exp(torch.randn((N, 1), generator=g) * spread)
    x[::7, 128:256] = 0.0                                          # all-zero groups
    x[1::11, :64] *= 1e-6                                          # tiny values
    x[2, 5] = -0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("d_qk", [576, 512])
def test_cache_write_matches_the_oracle_bit_for_bit(cuda_lib, d_qk):
    smla = cuda_lib
    smla.smla_get_device_status(clear=True)
    N, S = 300, 1000
    x = rows(N, d_qk, seed=d_qk)
    rng = np.random.default_rng(d_qk)
    slots = rng.permutation(S)[:N].astype(np.int32)
    slots[::13] = -1
    G = (d_qk + 127) // 128
    cache = torch.full((S, d_qk), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((S, G), -2.0, dtype=torch.float32, device="cuda")
    kv_c = x[:, :512].contiguous().cuda()
    k_pe = x[:, 512:].contiguous().cuda() if d_qk == 576 else None
    smla.smla_cache_write_e4m3_group(kv_c, k_pe, torch.from_numpy(slots).cuda(), cache, scales)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 0
    ref_c = np.full((S, d_qk), 0x5A, dtype=np.uint8)
    ref_s = np.full((S, G), -2.0, dtype=np.float32)
    oracle.cache_write_e4m3_group(bits16(x[:, :512]), bits16(x[:, 512:]) if d_qk == 576 else None,
                                  slots, ref_c, ref_s)
    assert np.array_equal(cache.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def test_cache_write_flags_slots_past_the_cache(cuda_lib):
    smla = cuda_lib
    smla.smla_get_device_status(clear=True)
    x = rows(8, 576, seed=3)
    cache = torch.zeros((16, 576), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((16, 5), dtype=torch.float32, device="cuda")
    slots = torch.tensor([0, 1, 16, 3, 99, -1, 6, 7], dtype=torch.int32, device="cuda")
    smla.smla_cache_write_e4m3_group(x[:, :512].contiguous().cuda(), x[:, 512:].contiguous().cuda(),
                                     slots, cache, scales)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 5           # SMLA_ERR_BAD_INDEX
    ref_c = np.zeros((16, 576), dtype=np.uint8)
    ref_s = np.zeros((16, 5), dtype=np.float32)
    oracle.cache_write_e4m3_group(bits16(x[:, :512]), bits16(x[:, 512:]),
                                  slots.cpu().numpy(), ref_c, ref_s)
    assert np.array_equal(cache.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy(), ref_s)


@pytest.mark.parametrize("h", [16, 64])
def test_written_cache_feeds_the_forward(cuda_lib, h):
    """Write a cache with the kernel, attend over it (group format), compare
    with the oracle on the same bytes and scales."""
    smla = cuda_lib
    smla.smla_get_device_status(clear=True)
    S, d_qk, T, topk = 2048, 576, 6, 256
    x = rows(S, d_qk, seed=11 + h, spread=0.0)
    cache = torch.zeros((S, d_qk), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((S, 5), dtype=torch.float32, device="cuda")
    smla.smla_cache_write_e4m3_group(x[:, :512].contiguous().cuda(), x[:, 512:].contiguous().cuda(),
                                     torch.arange(S, dtype=torch.int32, device="cuda"), cache, scales)
    torch.cuda.synchronize()
    base = W.custom(T=T, h=h, topk=topk, num_slots=S, valid=[256, 200, 77, 1, 0, 129], seed=5)
    w = W.Workload("written", T, h, d_qk, 512, topk, S, 2, 1.0 / math.sqrt(d_qk),
                   base.q, cache.cpu(), scales.cpu(), base.indices, base.valid_len, h)
    wd = w.to("cuda")
    O, L = smla.smla_fwd(wd.q, wd.kv, 2, wd.k_scale, wd.indices, wd.valid_len, wd.sm_scale,
                         num_slots=S)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 0
    Or, Lr = oracle_fwd(w)
    Og = O.float().cpu().double().numpy()
    Lg = L.cpu().double().numpy()
    assert np.abs(Og - Or).max() <= 2e-2
    inf = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(Lg), inf)
    assert np.abs(Lg[~inf] - Lr[~inf]).max() <= 1e-3


def _exhaustive_rows(d_qk):
    """Groups whose first value is the group's amax and whose other values
    run through every bf16 magnitude from amax down to amax * 2^-24 (both
    signs), for each of the 128 bf16 mantissas of amax at several exponents,
    plus groups with a tiny amax (a subnormal fp32 scale).  These hold every
    quotient x / scale the normal range can give, the exact E4M3 rounding
    ties (amax = 1.75 * 2^k makes the scale a power of two) and the quotients
    within an ulp of a tie."""
    vals = []
    mant = np.arange(128, dtype=np.uint32)
    rng = np.random.default_rng(5)
    for i in range(128):
        e = int(rng.integers(-30, 30))
        amax_bits = np.uint32(((e + 127) << 7) | i)
        xs = []
        for de in range(0, 25):
            eb = e + 127 - de
            if eb < 1:
                break
            b = (np.uint32(eb) << 7) | mant
            xs.append(b[b <= amax_bits])
        xs = np.concatenate(xs).astype(np.uint16)
        xs = np.concatenate([xs, xs | 0x8000])
        for c in range(0, xs.size, 127):
            vals.append(np.concatenate([[amax_bits], xs[c:c + 127]]).astype(np.uint16))
    for amax_bits in (0x0001, 0x0003, 0x007F, 0x0080, 0x0105, 0x1A37):   # tiny and subnormal amax
        xs = np.arange(1, amax_bits + 1, dtype=np.uint32)[:127].astype(np.uint16)
        vals.append(np.concatenate([[amax_bits], xs]).astype(np.uint16))
    groups = np.zeros((len(vals), 128), dtype=np.uint16)
    for gi, v in enumerate(vals):
        groups[gi, :v.size] = v
    per_row = d_qk // 128
    pad = (-len(groups)) % per_row
    groups = np.concatenate([groups, np.zeros((pad, 128), dtype=np.uint16)])
    return groups.reshape(-1, d_qk)


def test_cache_write_is_exact_for_every_bf16_quotient(cuda_lib):
    """Every E4M3 code equals the code of the IEEE fp32 quotient, over the
    exhaustive quotient set of _exhaustive_rows (the fast kernel multiplies
    by an approximate reciprocal and settles the few quotients near a
    rounding midpoint with a residual test)."""
    smla = cuda_lib
    smla.smla_get_device_status(clear=True)
    d_qk = 512
    bits = _exhaustive_rows(d_qk)
    N = bits.shape[0]
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    cache = torch.zeros((N, d_qk), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((N, 4), dtype=torch.float32, device="cuda")
    smla.smla_cache_write_e4m3_group(x.cuda(), None, torch.arange(N, dtype=torch.int32, device="cuda"),
                                     cache, scales)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 0
    ref_c = np.zeros((N, d_qk), dtype=np.uint8)
    ref_s = np.zeros((N, 4), dtype=np.float32)
    oracle.cache_write_e4m3_group(bits, None, np.arange(N, dtype=np.int32), ref_c, ref_s)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref_c), f"{int((got != ref_c).sum())} codes differ"

"""Parity of smla_fwd_paged (request-local top-k positions translated to cache
slots inside the kernels' index loads) with the fp64 oracle on the converted
ids, and with smla_fwd on the same slots: the two calls must agree bit for
bit, because the same kernels read the same rows.

Covers every kernel family (heads-major bf16 and E4M3, the E4M3-operand
keys-major kernel with group scales for one and for several groups of 16
heads), a split top-k range, a block stride larger than
the block size, and the entries the translation masks (pages past the
table, unallocated blocks, a request id outside the table).
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd

import oracle

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


def paged_view(w, rng, bs, R):
    """Express w's global slot ids as request-local positions.  The cache is
    cut into blocks of bs rows; every request owns all blocks, each at a
    random page of its block table; token t belongs to a random request, and
    its global id g becomes page(g // bs) * bs + g % bs of that request."""
    nblk = (w.num_slots + bs - 1) // bs
    table = np.stack([rng.permutation(nblk) for _ in range(R)]).astype(np.int32)
    inv = np.argsort(table, axis=1)                  # inv[r, block] = page
    req = rng.integers(0, R, size=w.T).astype(np.int32)
    g = w.indices.cpu().numpy().astype(np.int64)
    local = np.where(g >= 0, inv[req[:, None], np.maximum(g, 0) // bs] * bs + g % bs, -1)
    return local.astype(np.int32), req, table


def run_both(smla, w, local, req, table, bs, stride_rows=0):
    smla.smla_get_device_status(clear=True)      # earlier tests may have set it
    wd = w.to("cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    O_p, L_p = smla.smla_fwd_paged(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, dev(local),
                                   dev(req), dev(table), bs, wd.sm_scale,
                                   valid_len=wd.valid_len, block_stride_rows=stride_rows,
                                   num_slots=wd.num_slots)
    torch.cuda.synchronize()
    st_p = smla.smla_get_device_status(clear=True)
    glob = oracle.paged_to_global(local, req, table, bs, stride_rows)
    O_g, L_g = smla.smla_fwd(wd.q, wd.kv, wd.kv_dtype, wd.k_scale,
                             dev(glob.astype(np.int32)), wd.valid_len, wd.sm_scale,
                             num_slots=wd.num_slots)
    torch.cuda.synchronize()
    st_g = smla.smla_get_device_status(clear=True)
    return (O_p, L_p, st_p), (O_g, L_g, st_g), glob


def check_oracle(w, O, L, glob):
    Or, Lr = oracle_fwd(w, indices=torch.from_numpy(glob.astype(np.int32)))
    Og = O.float().cpu().double().numpy()
    Lg = L.cpu().double().numpy()
    assert np.all(np.isfinite(Og))
    assert np.abs(Og - Or).max() <= TOL_O
    inf = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(Lg), inf)
    if (~inf).any():
        assert np.abs(Lg[~inf] - Lr[~inf]).max() <= TOL_LSE


CASES = [
    # heads-major tensor-core kernel, bf16, several blocks, empty rows
    dict(T=12, h=128, topk=256, num_slots=3000, valid=[256, 0, 5, 200, 48, 49, 1, 96, 97, 150, 256, 7]),
    # per-tensor E4M3, NoPE rows, h = 64 (the E4M3-operand kernel, four
    # groups of 16 heads)
    dict(T=6, h=64, d_qk=512, topk=300, num_slots=900, kv_dtype=1, valid=[300, 257, 33, 2, 1, 0]),
    # per-tensor E4M3 with h = 80 (the heads-major kernel, converting loaders)
    dict(T=3, h=80, topk=200, num_slots=700, kv_dtype=1, valid=[200, 64, 1]),
    # E4M3 with group scales, one group of 16 heads
    dict(T=5, h=16, topk=400, num_slots=2000, kv_dtype=2, valid=[400, 130, 1, 0, 255]),
    # E4M3 with group scales, two groups of 16 heads
    dict(T=4, h=32, topk=128, num_slots=700, kv_dtype=2, valid=[128, 64, 3, 0]),
    # split top-k ranges (few tokens, long rows): partials + combine
    dict(T=2, h=128, topk=2048, num_slots=8192, valid=[2048, 1300]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("bs", [1, 16, 64])
def test_paged_equals_global_and_oracle(cuda_lib, case, bs):
    smla = cuda_lib
    w = W.custom(seed=100 + case, **CASES[case])
    rng = np.random.default_rng(7 * case + bs)
    local, req, table = paged_view(w, rng, bs, R=3)
    (O_p, L_p, st_p), (O_g, L_g, st_g), glob = run_both(smla, w, local, req, table, bs)
    assert st_p == 0 and st_g == 0
    assert np.array_equal(glob, np.where(w.indices.cpu().numpy() >= 0,
                                         w.indices.cpu().numpy(), -1))
    assert torch.equal(O_p, O_g)
    assert torch.equal(L_p, L_g)
    check_oracle(w, O_p, L_p, glob)


def test_paged_block_stride_rows(cuda_lib):
    """slot = block * block_stride_rows + position % block_size with a stride
    larger than the block (rows between blocks are never addressed)."""
    smla = cuda_lib
    bs, stride, R = 16, 40, 2
    w = W.custom(T=6, h=128, topk=96, num_slots=4000, valid=[96, 50, 0, 17, 96, 1], seed=31)
    rng = np.random.default_rng(3)
    nblk = w.num_slots // stride
    table = np.stack([rng.permutation(nblk)[:12] for _ in range(R)]).astype(np.int32)
    req = rng.integers(0, R, size=w.T).astype(np.int32)
    local = rng.integers(0, 12 * bs, size=(w.T, w.topk)).astype(np.int32)
    (O_p, L_p, st_p), (O_g, L_g, st_g), glob = run_both(smla, w, local, req, table, bs, stride)
    assert st_p == 0 and st_g == 0
    assert torch.equal(O_p, O_g) and torch.equal(L_p, L_g)
    check_oracle(w, O_p, L_p, glob)


def test_paged_untranslatable_entries_are_masked(cuda_lib):
    """Pages past the table and a request id outside it are masked and flag
    SMLA_ERR_BAD_INDEX; unallocated (-1) blocks are masked without a flag."""
    smla = cuda_lib
    bs = 16
    w = W.custom(T=5, h=128, topk=64, num_slots=1024, valid=[64, 64, 64, 30, 64], seed=41)
    rng = np.random.default_rng(9)
    table = rng.permutation(64)[:8].reshape(2, 4).astype(np.int32)
    table[1, 2] = -1                                  # an unallocated block
    req = np.array([0, 1, 1, 0, 0], dtype=np.int32)
    local = rng.integers(0, 4 * bs, size=(w.T, w.topk)).astype(np.int32)
    # only unallocated blocks: masked, no flag
    (O_p, L_p, st_p), (O_g, L_g, st_g), glob = run_both(smla, w, local, req, table, bs)
    assert st_p == 0 and (glob[1:3] == -1).any()
    assert torch.equal(O_p, O_g) and torch.equal(L_p, L_g)
    check_oracle(w, O_p, L_p, glob)
    # pages past the table, and a token whose request is not in the table
    local2 = local.copy()
    local2[0, :5] = 4 * bs + np.arange(5)              # page 4 of a 4-page table
    req2 = req.copy()
    req2[4] = 2                                         # only requests 0, 1 exist
    (O_p, L_p, st_p), (O_g, L_g, st_g), glob = run_both(smla, w, local2, req2, table, bs)
    assert st_p == 5                                    # SMLA_ERR_BAD_INDEX
    assert np.all(glob[4] == -1) and np.all(glob[0, :5] == -1)
    assert torch.equal(O_p, O_g) and torch.equal(L_p, L_g)
    assert torch.isneginf(L_p[4]).all() and (O_p[4] == 0).all()
    check_oracle(w, O_p, L_p, glob)

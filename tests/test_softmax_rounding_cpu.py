"""Why the kernels normalize O the way they do, restated on the CPU.

The kernels' online softmax keeps a lazy running max (it moves only when a
block's max beats it by 8 in log2 units on the bf16 kernels, 4 on the
E4M3-operand kernel), so the weight of a key that arrives after the max was
set and then carries its row lies in (1, 2^8] and is rounded on its way to
the PV product.  These tests restate that online softmax in numpy (scores
in fp64 from the dequantized rows; blocks, thresholds and the weights'
rounding as the kernels have them) on seeded inputs where one key carries
a row (tests/_late_key.py) and compare with the fp64 oracle:

* bf16 weights (the bf16 kernels), a key that arrives after the max was
  set: O divided by the sum of the unrounded weights misses the 2e-2 bound;
  divided by the sum of the rounded weights that PV multiplies (what the
  kernels do) it keeps it;
* E4M3 weights with group scales (the E4M3-operand kernel: per channel
  group g, x = p * scale_g * R_g * 16 rounded to f16 and split), rows of
  one key whose scale puts x where the pair is furthest from it: two E4M3
  terms miss the bound, three keep it.
"""
import math

import numpy as np
import pytest
import torch

from tests._helpers import dequant_rows_torch, oracle_fwd
from tests._late_key import build, build_one_key

TOL_O = 2e-2


def bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).double().numpy()


def e4m3_terms(x, n):
    """x (f16 values, |x| <= 256) as n E4M3 terms: t0 + t1/16 + t2/256."""
    out, r, scale = np.zeros_like(x), x.copy(), 1.0
    for _ in range(n):
        t = e4m3(r)
        out += t * scale
        r, scale = (r - t) * 16, scale / 16
    return out


def online_softmax(w, blk, thr, weights, rounded_sum):
    """O (bf16) as the kernels form it: per block, a lazy max update, the
    block's weights p (the kernel's form of them: weights(p)), O and the
    row sum rescaled by alpha; O / l at the end, l the sum of p or of the
    rounded weights."""
    K = dequant_rows_torch(w).numpy()
    V = K[:, :512]
    c = w.sm_scale * math.log2(math.e)
    q = w.q.double().numpy()
    out = np.zeros((w.T, w.h, 512))
    for t in range(w.T):
        s = (q[t] @ K[w.indices[t].numpy()].T) * c          # [h, topk], log2 units
        m = np.full(w.h, -np.inf)
        l = np.zeros(w.h)
        O = np.zeros((w.h, 512))
        for b0 in range(0, w.topk, blk):
            sb = s[:, b0:b0 + blk]
            bm = sb.max(1)
            up = bm > m + thr
            alpha = np.where(up, np.exp2(np.where(np.isinf(m), -np.inf, m - bm)), 1.0)
            m = np.where(up, bm, m)
            p = np.exp2(sb - m[:, None])
            pr = weights(p)
            l = l * alpha + (pr if rounded_sum else p).sum(1)
            O = O * alpha[:, None] + pr @ V[w.indices[t, b0:b0 + blk].numpy()]
        out[t] = bf16(O / l[:, None])
    return out


@pytest.mark.parametrize("blk", [48, 128])     # the heads-major and keys-major blocks
def test_bf16_weights_need_the_rounded_row_sum(blk):
    w = build(0, 32, 32)
    Or, _ = oracle_fwd(w)
    assert np.abs(Or).max() > 4.0
    err_plain = np.abs(online_softmax(w, blk, 8.0, bf16, False) - Or).max()
    err_kernel = np.abs(online_softmax(w, blk, 8.0, bf16, True) - Or).max()
    assert err_plain > TOL_O, err_plain
    assert err_kernel <= TOL_O, err_kernel


def pow2_at_most_inv(x):
    """The largest power of two R with x R <= 1 (x > 0)."""
    return 2.0 ** -np.ceil(np.log2(x))


def online_softmax_groups(w, terms):
    """O (bf16) as the E4M3-operand kernel forms it for group scales: lazy
    max (threshold 4, blocks of 128), per group the weights
    x = p * scale * R * 16 in f16 split into `terms` E4M3 terms, multiplied
    by the cache codes, O_g = sum / (16 R_g l)."""
    K = dequant_rows_torch(w).numpy()
    c = w.sm_scale * math.log2(math.e)
    q = w.q.double().numpy()
    ks = w.k_scale.double().numpy()
    codes = torch.from_numpy(w.kv.numpy().copy()).view(torch.float8_e4m3fn).double().numpy()
    out = np.zeros((w.T, w.h, 512))
    for t in range(w.T):
        idx = w.indices[t, :int(w.valid_len[t])].numpy()
        R = pow2_at_most_inv(ks[idx, :4].max(0))          # per group, from the unit's keys
        s = (q[t] @ K[idx].T) * c
        m = np.full(w.h, -np.inf)
        l = np.zeros(w.h)
        O = np.zeros((w.h, 512))
        for b0 in range(0, len(idx), 128):
            rows = idx[b0:b0 + 128]
            sb = s[:, b0:b0 + 128]
            bm = sb.max(1)
            up = bm > m + 4.0
            alpha = np.where(up, np.exp2(np.where(np.isinf(m), -np.inf, m - bm)), 1.0)
            m = np.where(up, bm, m)
            p = np.exp2(sb - m[:, None])
            l = l * alpha + p.sum(1)
            O *= alpha[:, None]
            for g in range(4):
                x = e4m3_terms(f16(p * (ks[rows, g] * R[g] * 16)[None, :]), terms)
                O[:, 128 * g:128 * (g + 1)] += x @ codes[rows, 128 * g:128 * (g + 1)] / (16 * R[g])
        out[t] = bf16(O / l[:, None])
    return out


def test_group_scaled_e4m3_weights_need_three_terms():
    w = build_one_key(2, 16, 24)
    Or, _ = oracle_fwd(w)
    assert np.abs(Or).max() > 4.0
    err_two = np.abs(online_softmax_groups(w, 2) - Or).max()
    err_three = np.abs(online_softmax_groups(w, 3) - Or).max()
    assert err_two > TOL_O, err_two
    assert err_three <= TOL_O, err_three

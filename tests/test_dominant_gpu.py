"""A key that carries its row, arriving after the row's running max was set.

The kernels keep a lazy running max: it moves only when a block's max
exceeds it by a threshold, so a later, larger score gets a softmax weight
above 1 (up to the threshold's power of two) before it is rounded for the
PV product.  Where that key carries the row, O is its V row times the
relative error of its rounded weight, and with |v| near 4.4 the output's
own bf16 rounding (up to 0.0156 at |O| in [4, 8)) leaves 0.0044 of the
2e-2 bound for that error.

Construction (per token t, head h): q = a_{t,h} on channel 0, zero
elsewhere; cache rows hold channel 0 = 1 at position 3 of every 48-key
block (a moderate score that sets the running max), 2 at position 200 (the
late key), -4 elsewhere.  The late key's score then exceeds the running max
by g = a sm_scale log2(e) (log2 units), and a_{t,h} spreads g over
(0.5, 7.9); its V row holds values of magnitude near 4.4 with mixed signs.
Enough tokens that the plan does not split the rows (each 256-key row is one
range), which is asserted; and few tokens with 512-key rows, which the plan
splits in two ranges whose partial outputs the combine merges (the late
key at 400, in a later block of the second range).
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import Guarded, oracle_fwd
from tests._late_key import build, build_one_key
from tests.test_parity_gpu import compare, gpu_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_dtype,h,T", [
    (W.KV_BF16, 128, 256),            # heads-major
    (W.KV_BF16, 16, 512),             # keys-major (bf16)
    (W.KV_FP8_E4M3, 128, 256),        # heads-major, converted E4M3
    (W.KV_FP8_E4M3, 16, 512),         # E4M3 operands, one scale
    (W.KV_FP8_E4M3_GROUP128, 16, 512),  # E4M3 operands, group scales
    (W.KV_FP8_E4M3_GROUP128, 128, 64),
])
def test_late_dominant_key(cuda_lib, kv_dtype, h, T):
    w = build(kv_dtype, h, T)
    plan = cuda_lib.smla_plan_info(T, h, w.d_qk, w.topk, kv_dtype)
    assert plan["splits"] == 1, plan
    O, L = gpu_fwd(cuda_lib, w.to("cuda"))
    Or, Lr = oracle_fwd(w)
    assert np.abs(Or).max() > 4.0                    # the case the test is about
    compare(O, L, Or, Lr, f"{w.name} ({plan['kernel']})")


@pytest.mark.parametrize("kv_dtype,h,T", [
    (W.KV_BF16, 128, 30),
    (W.KV_BF16, 16, 60),
    (W.KV_FP8_E4M3, 128, 30),
    (W.KV_FP8_E4M3, 16, 60),
    (W.KV_FP8_E4M3_GROUP128, 16, 60),
    (W.KV_FP8_E4M3_GROUP128, 128, 8),
])
def test_late_dominant_key_split_rows(cuda_lib, kv_dtype, h, T):
    w = build(kv_dtype, h, T, topk=512, late=400)
    plan = cuda_lib.smla_plan_info(T, h, w.d_qk, w.topk, kv_dtype)
    assert plan["splits"] == 2, plan               # ranges [0, 256) and [256, 512)
    O, L = gpu_fwd(cuda_lib, w.to("cuda"))
    Or, Lr = oracle_fwd(w)
    assert np.abs(Or).max() > 4.0
    compare(O, L, Or, Lr, f"{w.name} ({plan['kernel']}, 2 ranges)")


@pytest.mark.parametrize("kv_dtype,h", [
    (W.KV_FP8_E4M3_GROUP128, 16),
    (W.KV_FP8_E4M3_GROUP128, 128),
    (W.KV_FP8_E4M3_GROUP4_KPE, 16),
])
def test_one_key_rows_at_the_worst_pair_scales(cuda_lib, kv_dtype, h):
    """Rows of one key whose group scale puts its E4M3 weight where a pair of
    E4M3 terms is furthest from it (2^-9), with V in [4, 8): two terms miss
    the bound there (tests/test_softmax_rounding_cpu.py), the kernel's three
    keep it."""
    w = build_one_key(kv_dtype, h, 24)
    wd = w.to("cuda")
    if kv_dtype == W.KV_FP8_E4M3_GROUP4_KPE:
        go = Guarded((w.T, w.h, w.d_v), torch.bfloat16)
        gl = Guarded((w.T, w.h), torch.float32)
        O, L = cuda_lib.smla_fwd_split_q(wd.q, None, wd.kv, wd.kv_dtype, wd.k_scale, wd.indices,
                                         wd.valid_len, wd.sm_scale, kpe_scale=w.kpe_scale,
                                         out=go.t, lse=gl.t, num_slots=w.num_slots)
        torch.cuda.synchronize()
        go.check(w.name)
        gl.check(w.name)
    else:
        O, L = gpu_fwd(cuda_lib, wd)
    Or, Lr = oracle_fwd(w)
    assert np.abs(Or).max() > 4.0
    compare(O, L, Or, Lr, w.name)

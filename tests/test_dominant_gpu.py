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
import math

import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd
from tests.test_parity_gpu import compare, gpu_fwd

pytestmark = pytest.mark.gpu


def build(kv_dtype, h, T, topk=256, late=200):
    d_qk, S = 576, topk
    sm_scale = 1.0 / math.sqrt(d_qk)
    rng = np.random.default_rng(700 + 10 * kv_dtype + h)
    g = np.linspace(0.5, 7.9, T * h).reshape(T, h)
    rng.shuffle(g.reshape(-1))
    a = g / (sm_scale * math.log2(math.e))
    q = torch.zeros(T, h, d_qk, dtype=torch.bfloat16)
    q[:, :, 0] = torch.from_numpy(a).to(torch.bfloat16)
    # cache values (before quantization): channel 0 is the score channel
    x = np.clip(rng.standard_normal((S, d_qk)), -3.0, 3.0)
    x[:, 0] = -4.0
    x[3::48, 0] = 1.0
    x[late, 0] = 2.0
    mags = np.array([4.375, 4.25, 4.125, 4.0])
    x[late, 1:] = mags[rng.integers(0, 4, d_qk - 1)] * rng.choice([-1.0, 1.0], d_qk - 1)
    xt = torch.from_numpy(x).float()
    k_scale = None
    if kv_dtype == W.KV_BF16:
        kv = xt.to(torch.bfloat16)
    elif kv_dtype == W.KV_FP8_E4M3:
        kv = W.e4m3_bytes(xt / 0.05)
        k_scale = torch.tensor([0.05], dtype=torch.float32)
    else:
        G = d_qk // 128 + (1 if d_qk % 128 else 0)
        k_scale = torch.full((S, G), 0.05, dtype=torch.float32)
        k_scale[late] = 0.0371                       # a scale that is not a power of two
        kv = W.e4m3_bytes(xt / k_scale[:, torch.arange(d_qk) // 128])
    idx = torch.arange(topk, dtype=torch.int32).repeat(T, 1)
    valid = torch.full((T,), topk, dtype=torch.int32)
    return W.Workload(f"dominant_kv{kv_dtype}_h{h}_T{T}", T, h, d_qk, 512, topk, S, kv_dtype,
                      sm_scale, q, kv, k_scale, idx, valid, h)


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

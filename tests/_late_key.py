"""A key that carries its row, arriving after the row's lazy running max was
set: the seeded input of the late-key tests (the GPU test of every kernel
family and the CPU emulation of the softmax weights' rounding).

Per token t and head h: q = a_{t,h} on channel 0, zero elsewhere; cache
rows hold channel 0 = 1 at position 3 of every 48-key block (a moderate
score that sets the running max), 2 at position `late` (the late key), -4
elsewhere.  The late key's score then exceeds the running max by
g = a sm_scale log2(e) (log2 units), and a_{t,h} spreads g over
(0.5, 7.9); its V row holds values of magnitude near 4.4 with mixed signs.
"""
import math

import numpy as np
import torch

from sparse_mla_attention_02_gb300 import workloads as W


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


def build_one_key(kv_dtype, h, T):
    """Rows of one valid key each (its softmax weight is 1, so the E4M3
    kernel's weight is x = scale * R * 16 with R = 16 here), with group
    scales at which the E4M3 pair of x is furthest from x (about 2^-9 of
    it: x just above 8) and V values in [4, 8) (codes 128 .. 240), where the
    bf16 rounding of O alone takes up to 0.0156 of the 2e-2 bound."""
    assert kv_dtype in (W.KV_FP8_E4M3_GROUP128, W.KV_FP8_E4M3_GROUP4_KPE)
    d_qk, S = 576, T
    rng = np.random.default_rng(900 + kv_dtype + h)
    xs = np.array([8.265625, 8.296875, 8.328125, 8.359375, 8.390625, 8.421875])
    sigma = (xs / 256.0)[np.arange(S) % len(xs)]               # exact in fp32
    codes = rng.choice([128.0, 144.0, 160.0, 176.0, 192.0, 208.0, 224.0, 240.0], (S, d_qk))
    codes *= rng.choice([-1.0, 1.0], (S, d_qk))
    q = torch.from_numpy(rng.standard_normal((T, h, d_qk))).to(torch.bfloat16)
    kv = W.e4m3_bytes(torch.from_numpy(codes).float())          # the codes themselves
    if kv_dtype == W.KV_FP8_E4M3_GROUP128:
        k_scale = torch.from_numpy(np.repeat(sigma[:, None], 5, axis=1)).float()
        kpe = 1.0
    else:
        k_scale = torch.from_numpy(np.repeat(sigma[:, None], 4, axis=1)).float()
        kpe = float(sigma[0])
    idx = torch.full((T, 4), -1, dtype=torch.int32)
    idx[:, 0] = torch.arange(T, dtype=torch.int32)
    valid = torch.ones(T, dtype=torch.int32)
    return W.Workload(f"one_key_kv{kv_dtype}_h{h}", T, h, d_qk, 512, 4, S, kv_dtype,
                      1.0 / math.sqrt(d_qk), q, kv, k_scale, idx, valid, h, kpe_scale=kpe)

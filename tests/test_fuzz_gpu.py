"""Seeded random shapes through smla_fwd against the fp64 oracle.

Each case draws a cache format (bf16, E4M3 with one scale, E4M3 with
per-(slot, 128-channel group) scales, the 656-byte fp8_ds_mla row, E4M3 with
four ckv group scales and a kpe scale), a head count from both sides of
every boundary of the plan (1..16 keys-major, 17..64, 65..128), d_qk 576 or
512 where the format allows it, a top-k length from one position to a full
2048 (partial blocks of both kernel families' block sizes), valid counts
from 0 to topk, scattered -1 and out-of-range ids inside the valid prefix,
duplicate ids, and either softmax scale the pages use.  Every case must
match the oracle within the parity bounds, with empty rows exactly (0,
-inf), write nothing outside its output buffers (sentinel bands), and
report a masked out-of-range id in the device status exactly when it holds
one; a failure names the kernel family the plan picked.  The four-scale
format with its own rope scale goes through the split-query entry point,
the one that takes that scale.
"""
import math

import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import Guarded, oracle_fwd
from tests.test_parity_gpu import compare, gpu_fwd

pytestmark = pytest.mark.gpu

N_CASES = 160
HEADS = [1, 2, 3, 8, 16, 17, 24, 31, 48, 64, 65, 80, 100, 127, 128]
TOPKS = [1, 5, 47, 48, 49, 64, 127, 128, 129, 200, 300, 640, 1000, 2048]
FORMATS = [W.KV_BF16, W.KV_FP8_E4M3, W.KV_FP8_E4M3_GROUP128, W.KV_FP8_DS_MLA,
           W.KV_FP8_E4M3_GROUP4_KPE]


def draw(i):
    rng = np.random.default_rng(9000 + i)
    kv = int(rng.choice(FORMATS))
    h = int(rng.choice(HEADS))
    d_qk = 576 if kv in (W.KV_FP8_DS_MLA, W.KV_FP8_E4M3_GROUP4_KPE) \
        else int(rng.choice([576, 512]))
    topk = int(rng.choice(TOPKS))
    T = int(rng.integers(1, 6))
    num_slots = int(max(2 * topk, 256) + rng.integers(0, 200))
    valid = rng.integers(0, topk + 1, size=T)
    valid[rng.integers(0, T)] = topk                    # at least one full row
    sm_scale = float(rng.choice([1.0 / math.sqrt(d_qk), 192 ** -0.5]))
    return dict(T=T, h=h, d_qk=d_qk, topk=topk, num_slots=num_slots, kv_dtype=kv,
                valid=valid.tolist(), sm_scale=sm_scale, seed=9000 + i,
                k_scale=float(rng.choice([0.05, 0.07])),
                distinct=bool(rng.integers(0, 4) > 0)), rng


CASES = [draw(i)[0] for i in range(N_CASES)]


def case_id(c):
    return f"kv{c['kv_dtype']}_h{c['h']}_d{c['d_qk']}_k{c['topk']}_T{c['T']}"


@pytest.mark.parametrize("i", range(N_CASES), ids=[case_id(c) for c in CASES])
def test_random_shape_matches_the_oracle(cuda_lib, i):
    smla = cuda_lib
    kw, rng = draw(i)
    w = W.custom(name=f"fuzz{i}", **kw)
    # a few masked entries inside the valid prefixes: -1 and ids past the cache
    oor = False
    for t in range(w.T):
        v = int(w.valid_len[t])
        if v >= 3 and rng.integers(0, 2):
            j = int(rng.integers(0, v))
            if rng.integers(0, 2):
                w.indices[t, j] = -1
            else:
                w.indices[t, j] = w.num_slots + int(rng.integers(0, 50))
                oor = True
    kind = smla.smla_plan_info(w.T, w.h, w.d_qk, w.topk, w.kv_dtype)["kernel"]
    smla.smla_get_device_status(clear=True)
    wd = w.to("cuda")
    if w.kv_dtype == W.KV_FP8_E4M3_GROUP4_KPE:
        # the rope scale goes in through the split-query entry point (the
        # others read it as 1.0)
        go = Guarded((w.T, w.h, w.d_v), torch.bfloat16)
        gl = Guarded((w.T, w.h), torch.float32)
        O, L = smla.smla_fwd_split_q(wd.q[..., :512].contiguous(), wd.q[..., 512:].contiguous(),
                                     wd.kv, wd.kv_dtype, wd.k_scale, wd.indices, wd.valid_len,
                                     wd.sm_scale, kpe_scale=w.kpe_scale, out=go.t, lse=gl.t,
                                     num_slots=w.num_slots)
        torch.cuda.synchronize()
        go.check(f"{w.name} out")
        gl.check(f"{w.name} lse")
    else:
        O, L = gpu_fwd(smla, wd)                        # guarded out, lse, workspace
    status = smla.smla_get_device_status(clear=True)
    assert status == (5 if oor else 0), (kind, status)  # 5: an id past the cache was masked
    Or, Lr = oracle_fwd(w)
    compare(O, L, Or, Lr, f"{w.name} ({kind})")

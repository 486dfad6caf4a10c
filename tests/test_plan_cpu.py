"""The split plan without a GPU (smla_plan_info_for with a given SM count):
the kernel family each shape gets, when the top-k range is split, and the
workspace that needs.  These are the host-side rules the header states;
the GPU tests run the same plans through the kernels."""
import math
import random

import pytest

import sparse_mla_attention_02_gb300 as smla
from sparse_mla_attention_02_gb300 import build

SMS = 152                       # GB300
KEYS_RANGE, HEADS_RANGE = 2048, 3072   # top-k positions one unit covers


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return smla.load()


def plan(T, h, topk, kv=0, d_qk=576, sms=SMS):
    return smla.smla_plan_info_for(T, h, d_qk, topk, kv, num_sms=sms)


def family(h, kv):
    """E4M3 caches with group scales (every layout, any h) and per-tensor
    E4M3 with h <= 64: the E4M3-operand keys-major kernel; bf16 with h <= 16:
    the bf16 keys-major kernel; the rest: the heads-major kernel."""
    if kv in (2, 3, 4) or (kv == 1 and h <= 64):
        return "tc_keys_fp8"
    return "tc_keys" if h <= 16 else "tc_heads"


def test_benchmark_workloads_run_unsplit():
    """Each benchmark workload has enough tokens to fill the GPU by itself."""
    assert plan(8192, 128, 2048) == {"kernel": "tc_heads", "splits": 1, "workspace_bytes": 0}
    assert plan(64, 128, 2048) == {"kernel": "tc_heads", "splits": 1, "workspace_bytes": 0}
    assert plan(128, 64, 2048, kv=1, d_qk=512)["splits"] == 1
    assert plan(16384, 16, 2048, kv=2) == {"kernel": "tc_keys_fp8", "splits": 1,
                                           "workspace_bytes": 0}
    assert plan(128, 128, 2048, kv=3)["splits"] == 1


def test_few_tokens_split_to_fill_the_gpu():
    p = plan(2, 16, 2048, kv=2)                 # one CTA per unit, 152 SMs
    assert p["kernel"] == "tc_keys_fp8" and p["splits"] == 16
    p = plan(2, 16, 2048, kv=0)
    assert p["kernel"] == "tc_keys" and p["splits"] == 16
    p = plan(2, 64, 2048, kv=3)                 # 4 head groups per token
    assert p["kernel"] == "tc_keys_fp8" and p["splits"] == 16
    assert plan(8, 128, 2048, kv=2)["splits"] == 2   # 8 tokens x 8 head groups
    p = plan(4, 128, 2048)                      # a cluster of two SMs per unit
    assert p["kernel"] == "tc_heads" and 2 <= p["splits"] <= 16
    assert plan(1, 128, 64)["splits"] == 1      # 64 positions: nothing to split


def test_topk_longer_than_one_range_always_splits():
    assert plan(4096, 16, 3000, kv=2)["splits"] == 2
    assert plan(4096, 128, 4000)["splits"] == 2
    assert plan(4096, 128, 3072)["splits"] == 1


def test_argument_errors():
    with pytest.raises(smla.SmlaError, match="INVALID_ARG"):
        plan(4, 16, 64, sms=0)
    with pytest.raises(smla.SmlaError, match="INVALID_ARG"):
        plan(0, 16, 64)
    with pytest.raises(smla.SmlaError, match="UNSUPPORTED"):
        plan(4, 129, 64)
    with pytest.raises(smla.SmlaError, match="UNSUPPORTED"):
        plan(4, 16, 64, kv=3, d_qk=512)


def test_plan_invariants_over_random_shapes():
    rng = random.Random(7)
    for _ in range(3000):
        T = rng.choice([1, 2, 3, 7, 31, 64, 75, 76, 77, 151, 152, 500, 4096])
        h = rng.choice([1, 5, 16, 17, 32, 64, 100, 128])
        kv = rng.choice([0, 1, 2, 3, 4])
        d_qk = 576 if kv in (3, 4) else rng.choice([512, 576])
        topk = rng.choice([1, 47, 48, 64, 100, 2047, 2048, 2049, 3000, 3072, 3073, 5000])
        sms = rng.choice([2, 20, 148, 152])
        p = plan(T, h, topk, kv=kv, d_qk=d_qk, sms=sms)
        sp, ws = p["splits"], p["workspace_bytes"]
        assert p["kernel"] == family(h, kv), (T, h, kv)
        assert sp >= 1
        assert ws == (4 * sp * T * h * 513 if sp > 1 else 0), (T, h, topk, sp, ws)
        if p["kernel"] != "cuda_core":
            rng_len = HEADS_RANGE if p["kernel"] == "tc_heads" else KEYS_RANGE
            need = math.ceil(topk / rng_len)
            assert sp >= need, (T, h, topk, sp)
            assert sp <= max(16, need), (T, h, topk, sp)
            places = max(sms // 2, 1) if p["kernel"] == "tc_heads" else sms
            per_token = math.ceil(h / 16) if p["kernel"] == "tc_keys_fp8" else 1
            if 2 * T * per_token >= places:     # the tokens fill the GPU
                assert sp == need, (T, h, topk, sms, sp)
        # more tokens never split more
        assert plan(2 * T, h, topk, kv=kv, d_qk=d_qk, sms=sms)["splits"] <= sp

"""The cache layouts the pages print (tests/golden/cache_row_formats.json,
each entry with its page and section) against the seeded generator, the
binding's constants, the ABI's shape checks and the oracle.

The pages print no worked example with output values; the row sizes, head
sizes and scale groups are the numbers they do print that the rest of the
path depends on."""
import ctypes
import json
import math
import os

import numpy as np
import pytest
import torch

import sparse_mla_attention_02_gb300 as smla
from sparse_mla_attention_02_gb300 import build
from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "cache_row_formats.json")))


def _row_bytes(kv):
    return kv.shape[1] * kv.element_size()


def test_bf16_row_size_and_parts():
    g = GOLDEN["bf16_row"]
    assert sum(n for _, n in g["parts"]) == g["elements"]
    w = W.custom(T=2, h=4, d_qk=g["elements"], topk=8, num_slots=16, kv_dtype=W.KV_BF16,
                 valid=[8, 3], seed=1)
    assert w.kv.dtype == torch.bfloat16 and _row_bytes(w.kv) == g["bytes"]


def test_bf16_row_value_part_is_the_kv_c_prefix():
    """V is the kv_c part (the first 512 channels): with equal kv_c in every
    row and a query on the k_pe part only, O is that kv_c whatever k_pe is."""
    g = GOLDEN["bf16_row"]
    n_c = dict(g["parts"])["kv_c_normed"]
    w = W.custom(T=1, h=2, d_qk=g["elements"], topk=6, num_slots=6, kv_dtype=W.KV_BF16,
                 valid=[6], seed=2)
    kv = w.kv.float()
    kv[:, :n_c] = kv[0, :n_c]
    w.kv = kv.to(torch.bfloat16)
    w.q[:, :, :n_c] = 0
    O, _ = oracle_fwd(w)
    np.testing.assert_allclose(O[0], np.broadcast_to(w.kv[0, :n_c].double().numpy(), O[0].shape),
                               rtol=0, atol=1e-12)


def test_fp8_ds_mla_row_size():
    g = GOLDEN["fp8_ds_mla_row"]
    assert smla.DS_MLA_ROW_BYTES == g["bytes"] == W.DS_MLA_ROW_BYTES
    w = W.custom(T=2, h=4, d_qk=576, topk=8, num_slots=16, kv_dtype=W.KV_FP8_DS_MLA,
                 valid=[8, 3], seed=3)
    assert w.kv.dtype == torch.uint8 and _row_bytes(w.kv) == g["bytes"]


def test_e4m3_nope_row_and_per_tensor_scale():
    g = GOLDEN["e4m3_nope_row"]
    w = W.custom(T=2, h=4, d_qk=512, topk=8, num_slots=16, kv_dtype=W.KV_FP8_E4M3,
                 valid=[8, 3], seed=4)
    assert w.kv.dtype == getattr(torch, g["storage"]) and _row_bytes(w.kv) == g["bytes"]
    assert tuple(w.k_scale.shape) == (1,)


@pytest.mark.parametrize("d_qk", GOLDEN["head_sizes"]["values"])
def test_group_scales_per_token_and_128_channels(d_qk):
    g = GOLDEN["group_scales"]
    w = W.custom(T=2, h=4, d_qk=d_qk, topk=8, num_slots=16, kv_dtype=W.KV_FP8_E4M3_GROUP128,
                 valid=[8, 3], seed=5)
    assert tuple(w.k_scale.shape) == (16, math.ceil(d_qk / g["channels_per_group"]))


def test_head_sizes_accepted_by_the_abi():
    """d_qk in the printed head sizes passes the shape checks (on a machine
    without a GPU the call then stops at the device query, code 3); any
    other width is SMLA_ERR_UNSUPPORTED (2)."""
    g = GOLDEN["head_sizes"]
    assert sorted(g["ckv"] + k for k in g["kpe"]) == g["values"]
    build.build()
    lib = smla.load()
    k, s, n = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_size_t(0)
    info = lambda d: lib.smla_plan_info(4, 16, d, 512, 64, 0, ctypes.byref(k),
                                        ctypes.byref(s), ctypes.byref(n))
    for d in g["values"]:
        assert info(d) not in (1, 2), d
    for d in (448, 511, 513, 575, 577, 640):
        assert info(d) == 2, d

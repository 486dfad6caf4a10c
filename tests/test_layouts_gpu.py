"""Input-layout variants through the C ABI, against the fp64 oracle.

* The 656-byte fp8_ds_mla row (512 E4M3 ckv bytes, four fp32 group scales,
  64 bf16 rope values in one row) and E4M3 with four ckv group scales plus a
  separate kpe scale, on the kernel that serves them (the E4M3-operand
  keys-major kernel, in groups of 16 heads: one group, several groups with
  a partial last one, and a split top-k range).  Bar: max|dO| <= 2e-2,
  max|dLSE| <= 1e-3.
* The split query (q_nope, q_pe): smla_fwd_split_q must give exactly what
  smla_fwd gives on the concatenated q, on every kernel family, because the
  kernels read the same values from two places.
* Four group scales + kpe scale s must equal, bit for bit, the five-group
  layout whose rope scale is s for every slot (same values, same kernel).
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd
from tests.test_parity_gpu import compare

pytestmark = pytest.mark.gpu

CASES = [
    # one group of 16 heads: several 128-key blocks, a partial block, empty rows
    dict(T=6, h=16, topk=400, num_slots=2000, valid=[400, 257, 128, 1, 0, 129]),
    dict(T=3, h=5, topk=128, num_slots=300, valid=[128, 60, 2]),
    # a split top-k range (few tokens, long rows)
    dict(T=2, h=16, topk=2048, num_slots=6000, valid=[2048, 1500]),
    # several groups of 16 heads, the last one partial (h = 17, 32, 64, 128)
    dict(T=3, h=17, topk=160, num_slots=600, valid=[160, 129, 0]),
    dict(T=4, h=32, topk=96, num_slots=500, valid=[96, 40, 1, 0]),
    dict(T=3, h=64, topk=256, num_slots=900, valid=[256, 100, 3]),
    dict(T=2, h=128, topk=64, num_slots=300, valid=[64, 33]),
]


def run_split(smla, wd, q_nope, q_pe, kpe_scale):
    smla.smla_get_device_status(clear=True)
    O, L = smla.smla_fwd_split_q(q_nope, q_pe, wd.kv, wd.kv_dtype, wd.k_scale,
                                 wd.indices, wd.valid_len, wd.sm_scale,
                                 kpe_scale=kpe_scale, num_slots=wd.num_slots)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 0
    return O, L


def run_concat(smla, wd):
    smla.smla_get_device_status(clear=True)
    O, L = smla.smla_fwd(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, wd.indices,
                         wd.valid_len, wd.sm_scale, num_slots=wd.num_slots)
    torch.cuda.synchronize()
    assert smla.smla_get_device_status(clear=True) == 0
    return O, L


@pytest.mark.parametrize("kv_dtype", [W.KV_FP8_DS_MLA, W.KV_FP8_E4M3_GROUP4_KPE])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_layout_formats_match_the_oracle(cuda_lib, kv_dtype, case):
    w = W.custom(kv_dtype=kv_dtype, seed=300 + 10 * case + kv_dtype, k_scale=0.07,
                 name=f"case{case}_kv{kv_dtype}", **CASES[case])
    w.indices[0, 3] = -1                       # a masked entry inside the prefix
    wd = w.to("cuda")
    q = wd.q
    O, L = run_split(cuda_lib, wd, q[..., :512].contiguous(), q[..., 512:].contiguous(),
                     w.kpe_scale)
    Or, Lr = oracle_fwd(w)
    compare(O, L, Or, Lr, w.name)


@pytest.mark.parametrize("h", [16, 32])
def test_group4_kpe_through_smla_fwd_takes_kpe_scale_one(cuda_lib, h):
    """Entry points without a kpe argument read the rope scale as 1.0."""
    w = W.custom(T=4, h=h, topk=200, num_slots=900, kv_dtype=W.KV_FP8_E4M3_GROUP4_KPE,
                 k_scale=1.0, valid=[200, 129, 7, 0], seed=41 + h)
    assert w.kpe_scale == 1.0
    O, L = run_concat(cuda_lib, w.to("cuda"))
    Or, Lr = oracle_fwd(w)
    compare(O, L, Or, Lr, f"group4 kpe=1 h={h}")


@pytest.mark.parametrize("h", [16, 32])
def test_group4_kpe_equals_five_groups_with_the_kpe_scale(cuda_lib, h):
    w4 = W.custom(T=5, h=h, topk=300, num_slots=1200, kv_dtype=W.KV_FP8_E4M3_GROUP4_KPE,
                  k_scale=0.11, valid=[300, 256, 255, 1, 0], seed=52 + h)
    wd = w4.to("cuda")
    O4, L4 = run_split(cuda_lib, wd, wd.q, None, w4.kpe_scale)
    k5 = torch.cat([wd.k_scale, torch.full((w4.num_slots, 1), np.float32(0.11),
                                           device="cuda")], dim=1).contiguous()
    smla = cuda_lib
    O2, L2 = smla.smla_fwd(wd.q, wd.kv, W.KV_FP8_E4M3_GROUP128, k5, wd.indices,
                           wd.valid_len, wd.sm_scale, num_slots=w4.num_slots)
    torch.cuda.synchronize()
    assert torch.equal(O4, O2) and torch.equal(L4, L2)


SPLIT_Q = [
    # (h, kv_dtype, d_qk, T, topk, valid): one per kernel family and format
    (128, W.KV_BF16, 576, 8, 256, [256, 200, 97, 96, 48, 1, 0, 130]),        # heads-major
    (64, W.KV_FP8_E4M3, 576, 5, 300, [300, 257, 33, 1, 0]),                  # heads-major E4M3
    (64, W.KV_FP8_E4M3, 512, 4, 128, [128, 64, 1, 0]),                       # NoPE
    (128, W.KV_BF16, 576, 2, 2048, [2048, 1300]),                            # split range
    (16, W.KV_BF16, 576, 4, 256, [256, 129, 1, 0]),                          # keys-major bf16
    (16, W.KV_FP8_E4M3_GROUP128, 576, 4, 256, [256, 129, 1, 0]),             # keys-major group
    (16, W.KV_FP8_DS_MLA, 576, 4, 256, [256, 129, 1, 0]),                    # keys-major 656-B
    (32, W.KV_FP8_E4M3_GROUP128, 576, 3, 96, [96, 33, 0]),                   # CUDA cores
]


@pytest.mark.parametrize("case", range(len(SPLIT_Q)))
def test_split_q_equals_concatenated_q(cuda_lib, case):
    h, kv_dtype, d_qk, T, topk, valid = SPLIT_Q[case]
    w = W.custom(T=T, h=h, d_qk=d_qk, topk=topk, num_slots=3000, kv_dtype=kv_dtype,
                 valid=valid, seed=600 + case)
    wd = w.to("cuda")
    O1, L1 = run_concat(cuda_lib, wd)
    q_nope = wd.q[..., :512].contiguous()
    q_pe = wd.q[..., 512:].contiguous() if d_qk == 576 else None
    O2, L2 = run_split(cuda_lib, wd, q_nope, q_pe, 1.0)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    Or, Lr = oracle_fwd(w)
    compare(O2, L2, Or, Lr, f"split q case {case}")

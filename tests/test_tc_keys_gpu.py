"""Parity of the keys-major tensor-core kernel (h <= 16 heads) with the fp64
oracle, through the C ABI.

This kernel puts a block's 64 keys on the MMA's 128 rows (each key once per
channel half), keeps one fp32 score accumulator per 128-channel scale group,
and sums the two halves of a key's scores inside the CTA; the cases below aim
at what that design can get wrong: every cache format at both row widths,
head counts that are not 16 (or not 8, the heads a thread owns), ragged last
blocks (1, 63, 64, 65, 127, 128, 129 valid keys), top-k ranges longer than
one unit (split + merge), many units per SM, scores that keep growing across
blocks (the lazy running max must rescale O), and group scales over four
decades.  Same bar as the other parity tests: max|dO| <= 2e-2,
max|dLSE| <= 1e-3, empty rows exactly (0, -inf).
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd
from tests.test_parity_gpu import check, compare, gpu_fwd

pytestmark = pytest.mark.gpu


def test_dispatch_uses_keys_kernels_up_to_16_heads(cuda_lib):
    for kv in (0, 1, 2):
        for h in (1, 7, 16):
            for d in (512, 576):
                info = cuda_lib.smla_plan_info(512, h, d, 2048, kv)
                want = "tc_keys" if kv == 0 else "tc_keys_fp8"
                assert info["kernel"] == want, (kv, h, d, info)
    assert cuda_lib.smla_plan_info(512, 17, 576, 2048, 0)["kernel"] == "tc_heads"
    assert cuda_lib.smla_plan_info(512, 64, 576, 2048, 1)["kernel"] == "tc_keys_fp8"
    assert cuda_lib.smla_plan_info(512, 65, 576, 2048, 1)["kernel"] == "tc_heads"
    for kv in (2, 3, 4):
        assert cuda_lib.smla_plan_info(512, 128, 576, 2048, kv)["kernel"] == "tc_keys_fp8"
    assert cuda_lib.smla_plan_info(512, 16, 576, 4096, 2)["splits"] >= 2


def test_device_plan_is_the_plan_for_its_sm_count(cuda_lib):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for shape in [(8192, 128, 576, 2048, 0), (64, 128, 576, 2048, 0), (2, 16, 576, 2048, 2),
                  (80, 16, 576, 3000, 2), (4, 32, 576, 2048, 2), (128, 64, 512, 2048, 1)]:
        assert cuda_lib.smla_plan_info(*shape) == cuda_lib.smla_plan_info_for(*shape, num_sms=sms)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("d_qk", [576, 512])
@pytest.mark.parametrize("h", [1, 5, 16])
def test_formats_widths_heads(cuda_lib, kv_dtype, d_qk, h):
    w = W.custom(T=5, h=h, d_qk=d_qk, topk=300, num_slots=900,
                 kv_dtype=kv_dtype, valid=[300, 129, 128, 127, 1],
                 seed=200 + 10 * kv_dtype + h + d_qk)
    check(cuda_lib, w)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("h", [9, 16])
def test_block_edges(cuda_lib, kv_dtype, h):
    """Valid counts at and around the 64-key block edge."""
    w = W.custom(T=6, h=h, topk=200, num_slots=700, kv_dtype=kv_dtype,
                 valid=[63, 64, 65, 191, 192, 2], seed=260 + kv_dtype + h)
    check(cuda_lib, w)


@pytest.mark.parametrize("kv_dtype", [0, 2])
def test_topk_longer_than_one_unit_splits(cuda_lib, kv_dtype):
    """topk 3000 > 2048 positions per unit: at least two ranges per token,
    merged by the combine kernel, at a T that fills the GPU on its own."""
    T = 80
    rng = np.random.default_rng(5)
    valid = rng.integers(1, 3001, size=T)
    valid[:4] = [3000, 2049, 2048, 0]
    w = W.custom(T=T, h=16, topk=3000, num_slots=4096, kv_dtype=kv_dtype,
                 valid=valid, seed=210 + kv_dtype)
    assert cuda_lib.smla_plan_info(T, 16, 576, 3000, kv_dtype)["splits"] >= 2
    check(cuda_lib, w)


def test_many_units_per_sm_group_scales(cuda_lib):
    """400 units of 1..256 keys on the SMs: every SM runs several units back to
    back (barrier phases, TMEM and the shared buffers restart)."""
    T = 400
    rng = np.random.default_rng(6)
    w = W.custom(T=T, h=16, topk=256, num_slots=3000, kv_dtype=2,
                 valid=rng.integers(0, 257, size=T), seed=220)
    check(cuda_lib, w)


def test_wide_group_scale_range(cuda_lib):
    """Group scales from 1e-3 to 10 (per slot and channel group)."""
    w = W.custom(T=6, h=16, topk=512, num_slots=2000, kv_dtype=2,
                 valid=[512, 400, 257, 256, 100, 3], scale_range=(1e-3, 10.0),
                 seed=230)
    check(cuda_lib, w)


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_growing_scores_force_rescales(cuda_lib, kv_dtype):
    """Keys visited in an order where each block scores several log2 units
    above the last: the running max moves many times, so O must be rescaled
    correctly between PV products.  The growth is put in the 64 rope channels
    (part of K, not of V), so O stays O(1) and the 2e-2 bar is meaningful
    next to bf16 output rounding."""
    T, h, S, d = 2, 16, 2048, 576
    w = W.custom(T=T, h=h, topk=S, num_slots=S, kv_dtype=0, valid=[S, 1500],
                 seed=240)
    g = torch.Generator().manual_seed(241)
    rope_dir = w.q[0, :, 512:].float().mean(0)               # [64]
    ramp = torch.linspace(0.0, 1.0, S)[:, None]
    kv = 0.5 * torch.randn((S, d), generator=g)
    kv[:, 512:] += 400.0 * ramp * rope_dir[None, :]
    idx = torch.arange(S, dtype=torch.int32)
    w.indices = torch.stack([idx, idx])
    w.indices[1, 1500:] = -1
    if kv_dtype == 0:
        w.kv = kv.to(torch.bfloat16)
    else:
        w.kv_dtype = 1
        w.k_scale = torch.tensor([1.0])
        w.kv = W.e4m3_bytes(kv)
    Or, Lr = oracle_fwd(w)
    assert Lr[0].max() > 30.0                   # scores really grow
    O, L = gpu_fwd(cuda_lib, w.to("cuda"))
    compare(O, L, Or, Lr, "growing scores")


def test_all_masked_and_empty_rows(cuda_lib):
    """valid = 0, all ids -1, all ids out of range: (0, -inf) exactly."""
    w = W.custom(T=4, h=16, topk=200, num_slots=500, kv_dtype=2,
                 valid=[0, 200, 200, 150], seed=250)
    w.indices[1, :] = -1
    w.indices[2, :] = 500 + torch.arange(200, dtype=torch.int32)
    cuda_lib.smla_get_device_status(clear=True)
    O, L = gpu_fwd(cuda_lib, w.to("cuda"))
    assert cuda_lib.smla_get_device_status(clear=True) == 5   # ids >= num_slots
    Or, Lr = oracle_fwd(w)
    compare(O, L, Or, Lr, "masked rows")
    Lc = L.cpu()
    assert torch.all(torch.isneginf(Lc[:3])) and torch.all(O[:3].cpu() == 0)

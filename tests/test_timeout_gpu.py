"""The timeout contract of the bounded waits, on the GPU without a fault.

Every wait inside the tensor-core kernels gives up after a time limit: the
block records SMLA_ERR_TIMEOUT in the device status word, drains the copies
and MMAs it started, frees its tensor memory and returns.  The test switch
smla_test_set_stall makes a wait that cannot complete (each unit's first
batch of score MMAs is left out) with a short limit, so the call must:
return normally, report SMLA_ERR_TIMEOUT, and leave the device usable; the
next launch (stall off) must match the oracle even while the old timeout is
still in the status word, i.e. a stale timeout does not stop a new launch.
"""

import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd
from tests.test_parity_gpu import compare

pytestmark = pytest.mark.gpu

SMLA_ERR_TIMEOUT = 4


def _run(smla, wd):
    out, lse = smla.smla_fwd(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, wd.indices,
                             wd.valid_len, wd.sm_scale, num_slots=wd.num_slots)
    torch.cuda.synchronize()
    return out, lse


# (kernel family, workload): the heads-major kernel with a bf16 cache (TMA
# gathers, DSMEM exchange) and an E4M3 cache (converting loaders), and the
# keys-major kernels for h <= 16 (bf16 and grouped E4M3).
CASES = [
    ("heads_bf16", dict(T=3, h=32, topk=256, num_slots=700, kv_dtype=0,
                        valid=[256, 100, 1], seed=71)),
    ("heads_e4m3", dict(T=3, h=64, topk=256, num_slots=700, kv_dtype=1,
                        valid=[256, 200, 5], seed=72)),
    ("keys_bf16", dict(T=3, h=16, topk=256, num_slots=700, kv_dtype=0,
                       valid=[256, 70, 2], seed=73)),
    ("keys_e4m3_group", dict(T=3, h=16, topk=256, num_slots=700, kv_dtype=2,
                             valid=[256, 129, 3], seed=74)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_stalled_wait_reports_timeout_and_the_next_launch_is_clean(cuda_lib, name, kw):
    smla = cuda_lib
    w = W.custom(name=name, **kw)
    wd = w.to("cuda")
    Or, Lr = oracle_fwd(w)
    smla.smla_get_device_status(clear=True)       # earlier tests may leave bits set
    smla.smla_test_set_stall(True, 2000)          # 2 ms per wait
    try:
        _run(smla, wd)                            # returns; outputs undefined
    finally:
        smla.smla_test_set_stall(False, 0)
    # A launch after the timeout, with the status word not yet cleared, runs
    # to completion and is correct.
    O, L = _run(smla, wd)
    compare(O, L, Or, Lr, name + " after a timeout")
    assert smla.smla_get_device_status(clear=True) == SMLA_ERR_TIMEOUT
    O, L = _run(smla, wd)
    compare(O, L, Or, Lr, name + " after clearing")
    assert smla.smla_get_device_status(clear=True) == 0
    assert np.isfinite(L.cpu().numpy()[L.cpu().numpy() > -np.inf]).all()

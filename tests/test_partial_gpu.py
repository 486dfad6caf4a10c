"""smla_fwd_partial (fp32 normalised O + LSE for a cross-shard merge): the
DCP path of the flashmla_sparse page, emulated on one GPU.  Each index row
is split into two shards by a random mask (masked entries left as -1 in
place, no compaction); each shard runs through smla_fwd_partial; the shards
are merged by smla_combine.  Checked against the oracle per shard and merged,
and against one smla_fwd over the whole rows, for every kernel family.
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3

CASES = [
    dict(T=8, h=128, topk=512, num_slots=3000, valid=[512, 400, 77, 1, 0, 256, 49, 48]),
    dict(T=6, h=64, d_qk=512, topk=300, num_slots=900, kv_dtype=1, valid=[300, 257, 33, 2, 1, 0]),
    dict(T=5, h=16, topk=400, num_slots=2000, kv_dtype=2, valid=[400, 130, 1, 0, 255]),
    dict(T=4, h=32, topk=128, num_slots=700, kv_dtype=2, valid=[128, 64, 3, 0]),
    dict(T=2, h=128, topk=2048, num_slots=8192, valid=[2048, 1300]),   # split-sized rows
]


def assert_close(O, L, Or, Lr, what):
    O = O.double().cpu().numpy()
    L = L.double().cpu().numpy()
    assert np.all(np.isfinite(O)), what
    assert np.abs(O - Or).max() <= TOL_O, what
    inf = np.isneginf(Lr)
    assert np.array_equal(np.isneginf(L), inf), what
    assert np.all(O[inf] == 0.0), what
    if (~inf).any():
        assert np.abs(L[~inf] - Lr[~inf]).max() <= TOL_LSE, what


@pytest.mark.parametrize("case", range(len(CASES)))
def test_shards_merge_to_the_whole(cuda_lib, case):
    smla = cuda_lib
    smla.smla_get_device_status(clear=True)      # earlier tests may have set it
    w = W.custom(seed=200 + case, **CASES[case])
    wd = w.to("cuda")
    rng = np.random.default_rng(case)
    keep = torch.from_numpy(rng.random(tuple(w.indices.shape)) < 0.5).to("cuda")
    shards = [torch.where(keep, wd.indices, -1).contiguous(),
              torch.where(~keep, wd.indices, -1).contiguous()]
    parts = []
    for sh in shards:
        O, L = smla.smla_fwd_partial(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, sh,
                                     wd.valid_len, wd.sm_scale, num_slots=wd.num_slots)
        torch.cuda.synchronize()
        assert smla.smla_get_device_status(clear=True) == 0
        Or, Lr = oracle_fwd(w, indices=sh.cpu())
        assert_close(O, L, Or, Lr, "shard")
        parts.append((O, L))
    Om, Lm = smla.smla_combine(
        torch.stack([parts[0][0], parts[1][0]]).reshape(2, -1, 512).contiguous(),
        torch.stack([parts[0][1], parts[1][1]]).reshape(2, -1).contiguous())
    Of, Lf = smla.smla_fwd(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, wd.indices, wd.valid_len,
                           wd.sm_scale, num_slots=wd.num_slots)
    torch.cuda.synchronize()
    Or, Lr = oracle_fwd(w)
    assert_close(Om.float().reshape(w.T, w.h, 512), Lm.reshape(w.T, w.h), Or, Lr, "merged")
    assert_close(Of.float(), Lf, Or, Lr, "whole")


def test_partial_output_rejects_a_topk_longer_than_one_range(cuda_lib):
    smla = cuda_lib
    w = W.custom(T=2, h=128, topk=4096, num_slots=8192, valid=[10, 20], seed=3).to("cuda")
    with pytest.raises(smla.SmlaError, match="UNSUPPORTED"):
        smla.smla_fwd_partial(w.q, w.kv, w.kv_dtype, w.k_scale, w.indices, w.valid_len,
                              w.sm_scale, num_slots=w.num_slots)

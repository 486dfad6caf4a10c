"""smla_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some hosts own all device memory through their own pool and forbid a library
from calling cudaMalloc on its own (an inference engine's plugin, a framework
that keeps exact accounting of device memory), and some latency-critical loops
cannot afford the stall a cudaMalloc may cause.  For them the library keeps
the split scratch in a fixed device array of its own.  This test calls that
entry point through the C ABI, twice in a row on different inputs, and checks
each result against the regular smla_fwd with the parity tolerances.  It also
checks that a shape needing more scratch than the array holds is refused.

The file name makes pytest collect it last, so a failure here comes after
every other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
SCRATCH_BYTES = 16 * 1024 * 1024   # SMLA_NOALLOC_SCRATCH_BYTES in smla.h


def _noalloc(lib):
    f = lib.smla_fwd_noalloc
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, I, P, P, P, I, I, I, I, I, I64, F, P, P, P]
    f.restype = I
    return f


def _call_noalloc(lib, w, out, lse):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _noalloc(lib)(p(w.q), p(w.kv), w.kv_dtype, p(w.k_scale),
                         p(w.indices), p(w.valid_len), w.T, w.h, w.d_qk,
                         w.d_v, w.topk, w.num_slots, w.sm_scale, p(out),
                         p(lse), stream)


def _check_same(O_a, L_a, O_b, L_b):
    dO = (O_a.float() - O_b.float()).abs().max().item()
    assert dO <= TOL_O, dO
    inf_a, inf_b = torch.isneginf(L_a), torch.isneginf(L_b)
    assert torch.equal(inf_a, inf_b)
    fin = ~inf_a
    if fin.any():
        dL = (L_a[fin] - L_b[fin]).abs().max().item()
        assert dL <= TOL_LSE, dL


def test_noalloc_matches_smla_fwd_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib.load()
    cases = [
        W.custom(T=3, h=128, topk=2048, num_slots=8192,
                 valid=[2048, 1000, 1], seed=901, name="noalloc_a"),
        W.custom(T=5, h=64, topk=1024, num_slots=4096, kv_dtype=2,
                 valid=[1024, 0, 77, 512, 3], seed=902, name="noalloc_b"),
    ]
    refs, dev = [], []
    for w in cases:
        w = w.to("cuda")
        need = cuda_lib.smla_workspace_size(w.T, w.h, w.d_qk, w.topk,
                                            w.kv_dtype)
        assert 0 < need <= SCRATCH_BYTES  # the split path (scratch) is used
        refs.append(cuda_lib.smla_fwd(w.q, w.kv, w.kv_dtype, w.k_scale,
                                      w.indices, w.valid_len, w.sm_scale,
                                      num_slots=w.num_slots))
        dev.append(w)
    torch.cuda.synchronize()
    outs = []
    for w in dev:                      # two calls in a row, sharing the scratch
        out = torch.empty((w.T, w.h, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.T, w.h), dtype=torch.float32, device="cuda")
        assert _call_noalloc(lib, w, out, lse) == 0
        outs.append((out, lse))
    torch.cuda.synchronize()
    for (out, lse), (O_ref, L_ref) in zip(outs, refs):
        _check_same(out, lse, O_ref, L_ref)


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load()
    big = None
    for T, h in [(300, 16), (296, 16), (37, 128), (150, 32), (18, 128)]:
        need = cuda_lib.smla_workspace_size(T, h, 576, 2048, 0)
        if need > SCRATCH_BYTES:
            big = (T, h)
            break
    if big is None:
        pytest.skip("no candidate shape needs more than the fixed scratch "
                    "on this device's split plan")
    T, h = big
    w = W.custom(T=T, h=h, topk=2048, num_slots=2048, seed=903,
                 valid=np.full(T, 16)).to("cuda")
    out = torch.empty((T, h, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, h), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, w, out, lse) == 6   # SMLA_ERR_WORKSPACE

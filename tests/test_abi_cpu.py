"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import sparse_mla_attention_02_gb300 as smla
from sparse_mla_attention_02_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return smla.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SMLA_API\s+[\w\s\*]+?\b(smla_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ["smla_fwd", "smla_fwd_ws", "smla_workspace_size", "smla_combine",
              "smla_get_device_status", "smla_status_string", "smla_version",
              "smla_plan_info"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in smla.STATUS_NAMES.items():
        assert smla.smla_status_string(code) == name
    assert smla.smla_status_string(99) == "SMLA_ERR_UNKNOWN"
    assert lib.smla_version() >= 100


def _fwd(lib, **kw):
    a = dict(q=1 << 12, kv=1 << 12, kv_dtype=0, k_scale=None, idx=1 << 12,
             valid=None, T=4, h=16, d_qk=576, d_v=512, topk=64, S=256,
             scale=0.04, out=1 << 12, lse=None)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.smla_fwd(P(a["q"]), P(a["kv"]), a["kv_dtype"], P(a["k_scale"]),
                        P(a["idx"]), P(a["valid"]), a["T"], a["h"], a["d_qk"],
                        a["d_v"], a["topk"], a["S"], a["scale"], P(a["out"]),
                        P(a["lse"]), None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), 1), (dict(h=0), 1), (dict(topk=0), 1), (dict(S=0), 1),
    (dict(h=129), 2), (dict(d_qk=128), 2), (dict(d_v=256), 2),
    (dict(kv_dtype=5), 2), (dict(kv_dtype=-1), 2), (dict(S=1 << 31), 2),
    (dict(kv_dtype=3, d_qk=512), 2), (dict(kv_dtype=4, d_qk=512), 2),
    (dict(kv_dtype=4), 1),
    (dict(q=None), 1), (dict(kv=None), 1), (dict(idx=None), 1),
    (dict(out=None), 1), (dict(kv_dtype=1), 1), (dict(kv_dtype=2), 1),
    (dict(q=(1 << 12) + 8), 1), (dict(out=(1 << 12) + 4), 1),
    (dict(idx=(1 << 12) + 2), 1),
])
def test_bad_arguments_are_rejected_on_the_host(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _fwd_noalloc(lib, **kw):
    a = dict(q=1 << 12, kv=1 << 12, kv_dtype=0, k_scale=None, idx=1 << 12,
             valid=None, T=4, h=16, d_qk=576, d_v=512, topk=64, S=256,
             scale=0.04, out=1 << 12, lse=None)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    f = lib.smla_fwd_noalloc
    VP, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.argtypes = [VP, VP, I, VP, VP, VP, I, I, I, I, I, I64, F, VP, VP, VP]
    f.restype = I
    return lib.smla_fwd_noalloc(P(a["q"]), P(a["kv"]), a["kv_dtype"], P(a["k_scale"]),
                                P(a["idx"]), P(a["valid"]), a["T"], a["h"], a["d_qk"],
                                a["d_v"], a["topk"], a["S"], a["scale"], P(a["out"]),
                                P(a["lse"]), None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), 1), (dict(h=0), 1), (dict(topk=0), 1), (dict(S=0), 1),
    (dict(h=200), 2), (dict(d_qk=128), 2), (dict(d_v=256), 2), (dict(kv_dtype=5), 2),
    (dict(q=None), 1), (dict(out=(1 << 12) + 4), 1), (dict(valid=(1 << 12) + 2), 1),
    # oversized shapes with a bad argument: the argument's code, not the
    # scratch limit's
    (dict(h=200, T=1 << 20, topk=1 << 16), 2), (dict(q=None, T=1 << 20, topk=1 << 16), 1),
])
def test_noalloc_rejects_what_smla_fwd_rejects(lib, kw, code):
    """smla_fwd_noalloc runs smla_fwd's own checks before its scratch-size
    check, so a call that smla_fwd would reject gets the same code."""
    assert _fwd_noalloc(lib, **kw) == code
    if "T" not in kw or kw["T"] >= 0:
        assert _fwd(lib, **{k: v for k, v in kw.items()}) == code


def test_stall_switch_argument_check(lib):
    assert lib.smla_test_set_stall(1, -1) == 1


def test_zero_tokens_is_ok_and_launches_nothing(lib):
    assert _fwd(lib, T=0, q=None, kv=None, idx=None, out=None) == 0


def test_combine_argument_checks(lib):
    P = ctypes.c_void_p
    c = lib.smla_combine
    assert c(P(4096), P(4096), 0, 10, 512, P(4096), None, None) == 1
    assert c(P(4096), P(4096), 65, 10, 512, P(4096), None, None) == 1
    assert c(P(4096), P(4096), 2, 10, 256, P(4096), None, None) == 2
    assert c(None, P(4096), 2, 10, 512, P(4096), None, None) == 1
    assert c(P(4100), P(4096), 2, 10, 512, P(4096), None, None) == 1
    assert c(None, None, 2, 0, 512, None, None, None) == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(smla, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        smla.load()


def test_plan_info_argument_checks(lib):
    """Shape errors are reported before any device query."""
    k, n = ctypes.c_int(-1), ctypes.c_size_t(0)
    q = lambda *a: lib.smla_plan_info(*a, ctypes.byref(k), None, ctypes.byref(n))
    assert q(0, 16, 576, 512, 64, 0) == 1
    assert q(4, 0, 576, 512, 64, 0) == 1
    assert q(4, 16, 576, 512, 0, 0) == 1
    assert q(4, 129, 576, 512, 64, 0) == 2
    assert q(4, 16, 640, 512, 64, 0) == 2
    assert q(4, 16, 576, 256, 64, 0) == 2
    assert q(4, 16, 576, 512, 64, 5) == 2
    assert q(4, 16, 512, 512, 64, 3) == 2     # the 656-byte row is 576 channels
    assert q(4, 16, 512, 512, 64, 4) == 2
    assert k.value == -1                      # outputs untouched on error


def _fwd_paged(lib, **kw):
    a = dict(q=1 << 12, kv=1 << 12, kv_dtype=0, k_scale=None, idx=1 << 12,
             req=1 << 12, bt=1 << 12, nreq=2, bts=8, bs=64, bsr=0,
             valid=None, T=4, h=16, d_qk=576, d_v=512, topk=64, S=256,
             scale=0.04, out=1 << 12, lse=None)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.smla_fwd_paged(
        P(a["q"]), P(a["kv"]), a["kv_dtype"], P(a["k_scale"]), P(a["idx"]),
        P(a["req"]), P(a["bt"]), a["nreq"], a["bts"], a["bs"], a["bsr"],
        P(a["valid"]), a["T"], a["h"], a["d_qk"], a["d_v"], a["topk"], a["S"],
        a["scale"], P(a["out"]), P(a["lse"]), None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=None), 1), (dict(req=None), 1), (dict(nreq=0), 1),
    (dict(bts=0), 1), (dict(bs=0), 1), (dict(bsr=-1), 1),
    (dict(req=(1 << 12) + 2), 1), (dict(bt=(1 << 12) + 1), 1),
    (dict(nreq=1 << 20, bts=1 << 12), 1),
    (dict(h=0), 1), (dict(idx=None), 1), (dict(d_qk=128), 2),
])
def test_paged_bad_arguments_are_rejected_on_the_host(lib, kw, code):
    assert _fwd_paged(lib, **kw) == code


def test_paged_zero_tokens_is_ok(lib):
    assert _fwd_paged(lib, T=0, q=None, kv=None, idx=None, out=None) == 0


def test_partial_argument_checks(lib):
    P = ctypes.c_void_p
    f = lambda out, lse, T=4, h=16: lib.smla_fwd_partial(
        P(4096), P(4096), 0, None, P(4096), None, T, h, 576, 512, 64, 256, 0.04,
        None if out is None else P(out), None if lse is None else P(lse), None)
    assert f(None, 4096) == 1
    assert f(4096, None) == 1
    assert f(4104, 4096) == 1            # fp32 output not 16-byte aligned
    assert f(4096, 4098) == 1
    assert f(4096, 4096, h=0) == 1
    assert f(None, None, T=0) == 0


def test_cache_write_argument_checks(lib):
    P = ctypes.c_void_p
    f = lambda kv=4096, pe=4096, sl=4096, N=4, d=576, S=64, c=4096, sc=4096: \
        lib.smla_cache_write_e4m3_group(
            None if kv is None else P(kv), None if pe is None else P(pe),
            None if sl is None else P(sl), N, d, S, None if c is None else P(c),
            None if sc is None else P(sc), None)
    assert f(N=-1) == 1
    assert f(S=0) == 1
    assert f(d=640) == 2
    assert f(N=0, kv=None, pe=None, sl=None, c=None, sc=None) == 0
    assert f(kv=None) == 1
    assert f(sl=None) == 1
    assert f(c=None) == 1
    assert f(sc=None) == 1
    assert f(pe=None) == 1               # 576-channel rows need k_pe
    assert f(d=512) == 1                 # 512-channel rows take no k_pe
    assert f(kv=4104) == 1               # misaligned
    assert f(c=4104) == 1


def test_split_q_argument_checks(lib):
    P = ctypes.c_void_p
    f = lambda qn=4096, qp=4096, kv_dtype=0, ks=None, d_qk=576, T=4: lib.smla_fwd_split_q(
        None if qn is None else P(qn), None if qp is None else P(qp), P(4096), kv_dtype,
        None if ks is None else P(ks), 0.5, P(4096), None, T, 16, d_qk, 512, 64, 256, 0.04,
        P(4096), None, None, 0, None)
    assert f(qn=None) == 1
    assert f(qp=4104) == 1                    # q_pe not 16-byte aligned
    assert f(qn=4104) == 1
    assert f(kv_dtype=4) == 1                 # four group scales needed
    assert f(kv_dtype=3, d_qk=512) == 2
    assert f(kv_dtype=5) == 2
    assert f(T=0, qn=None, qp=None) == 0


def _fwd_host(lib, **kw):
    a = dict(q=1 << 12, kv=1 << 12, kv_dtype=0, k_scale=None, idx=1 << 12,
             valid=None, T=4, h=16, d_qk=576, d_v=512, topk=64, S=256,
             scale=0.04, out=1 << 12, lse=None, chunk=0, ws=1 << 12,
             ws_bytes=1 << 30)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.smla_fwd_host(
        P(a["q"]), P(a["kv"]), a["kv_dtype"], P(a["k_scale"]), P(a["idx"]),
        P(a["valid"]), a["T"], a["h"], a["d_qk"], a["d_v"], a["topk"], a["S"],
        a["scale"], P(a["out"]), P(a["lse"]), a["chunk"], P(a["ws"]),
        a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), 1), (dict(h=0), 1), (dict(topk=0), 1), (dict(S=0), 1),
    (dict(chunk=-1), 1), (dict(h=129), 2), (dict(d_qk=128), 2),
    (dict(d_v=256), 2), (dict(kv_dtype=5), 2), (dict(kv_dtype=3, d_qk=512), 2),
])
def test_host_entry_shape_errors_come_before_any_device_call(lib, kw, code):
    assert _fwd_host(lib, **kw) == code


def test_host_workspace_size_covers_two_staging_slots(lib):
    """Whatever the split plan adds, the workspace holds two chunks' worth of
    q, indices, valid counts, O and LSE (the copy of one chunk overlaps the
    forward of the other)."""
    f = lib.smla_fwd_host_workspace_size
    assert f(0, 16, 576, 512, 64, 0, 0) == 0
    assert f(4, 0, 576, 512, 64, 0, 0) == 0
    for T, h, topk, chunk in [(4, 16, 64, 0), (1000, 16, 2048, 64),
                              (1000, 128, 2048, 0), (8192, 128, 2048, 512)]:
        cdiv = lambda a, b: -(-a // b)
        C = min(chunk, T) if chunk else min(T, max(256, cdiv(cdiv(T, 16), 64) * 64))
        per_token = h * 576 * 2 + topk * 4 + 4 + h * 512 * 2 + h * 4
        assert f(T, h, 576, 512, topk, 0, chunk) >= 2 * C * per_token, (T, h, chunk)
    assert f(1000, 16, 576, 512, 2048, 0, 64) < f(1000, 16, 576, 512, 2048, 0, 512)


def test_host_binding_rejects_bad_tensors_before_any_device_call(lib):
    import torch
    T, h, topk = 3, 16, 64
    q = torch.zeros((T, h, 576), dtype=torch.bfloat16)
    idx = torch.zeros((T, topk), dtype=torch.int32)
    vl = torch.full((T,), topk, dtype=torch.int32)
    kv = torch.zeros((256, 576), dtype=torch.bfloat16)
    call = lambda **kw: smla.smla_fwd_host(
        kw.get("q", q), kv, 0, None, kw.get("idx", idx), kw.get("vl", vl), 0.04)
    with pytest.raises(ValueError, match="bf16"):
        call(q=q.float())
    with pytest.raises(ValueError, match="bf16"):
        call(q=q.transpose(0, 1))
    with pytest.raises(ValueError, match="int32"):
        call(idx=idx.long())
    with pytest.raises(ValueError, match="int32"):
        call(idx=idx[:2])
    with pytest.raises(ValueError, match="valid_len"):
        call(vl=vl[:2])
    with pytest.raises(ValueError, match="valid_len"):
        call(vl=vl.long())


def test_device_entry_points_refuse_host_tensors(lib):
    """Host tensors given to a device entry point are refused by the binding
    (a ValueError naming the argument) before any pointer reaches the
    library; the checks survive ``python -O``."""
    import torch
    T, h, topk = 2, 16, 64
    q = torch.zeros((T, h, 576), dtype=torch.bfloat16)
    kv = torch.zeros((256, 576), dtype=torch.bfloat16)
    idx = torch.zeros((T, topk), dtype=torch.int32)
    with pytest.raises(ValueError, match="q must be"):
        smla.smla_fwd(q, kv, 0, None, idx, None, 0.04)
    with pytest.raises(ValueError, match="q must be"):
        smla.smla_fwd_partial(q, kv, 0, None, idx, None, 0.04)
    with pytest.raises(ValueError, match="q_nope must be"):
        smla.smla_fwd_split_q(q, None, kv, 0, None, idx, None, 0.04)
    with pytest.raises(ValueError, match="o_parts must be"):
        smla.smla_combine(torch.zeros((2, 4, 512), dtype=torch.float64),
                          torch.zeros((2, 4)))
    with pytest.raises(ValueError, match="kv_c and k_pe"):
        smla.smla_cache_write_e4m3_group(
            torch.zeros((4, 512), dtype=torch.bfloat16), None,
            torch.zeros(4, dtype=torch.int32), torch.zeros((8, 512), dtype=torch.uint8),
            torch.zeros((8, 4)))

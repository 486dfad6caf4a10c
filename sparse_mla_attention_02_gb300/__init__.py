"""GB300-native sparse MLA attention forward.

A thin Python binding over the C ABI of libsmla (include/smla.h): the
functions below carry the C names, take torch tensors that already live on the
GPU, check dtypes and shapes, and pass raw pointers and sizes through ctypes.
Every step of the computation runs in the library's CUDA kernels; there is no
fallback of any kind.  If libsmla.so has not been built (``build.build()``,
or ``__graft_entry__.build()``), every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lib = None
_lock = threading.Lock()

SMLA_KV_BF16 = 0
SMLA_KV_FP8_E4M3 = 1
SMLA_KV_FP8_E4M3_GROUP128 = 2
SMLA_KV_FP8_DS_MLA = 3            # 656-byte rows: 512 E4M3 | 4 fp32 scales | 64 bf16
SMLA_KV_FP8_E4M3_GROUP4_KPE = 4   # E4M3 [S, 576], k_scale [S, 4], one kpe scale
DS_MLA_ROW_BYTES = 656

SMLA_OK = 0
STATUS_NAMES = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG",
                2: "SMLA_ERR_UNSUPPORTED", 3: "SMLA_ERR_CUDA",
                4: "SMLA_ERR_TIMEOUT", 5: "SMLA_ERR_BAD_INDEX",
                6: "SMLA_ERR_WORKSPACE"}


class SmlaError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load():
    """Load libsmla.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"libsmla.so not built at {path}; run "
                "python -m sparse_mla_attention_02_gb300.build")
        lib = ctypes.CDLL(path)
        P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                            ctypes.c_float, ctypes.c_size_t)
        fwd_args = [P, P, I, P, P, P, I, I, I, I, I, I64, F, P, P]
        lib.smla_fwd.argtypes = fwd_args + [P]
        lib.smla_fwd.restype = I
        lib.smla_fwd_ws.argtypes = fwd_args + [P, SZ, P]
        lib.smla_fwd_ws.restype = I
        lib.smla_cache_write_e4m3_group.argtypes = [P, P, P, I, I, I64, P, P, P]
        lib.smla_cache_write_e4m3_group.restype = I
        lib.smla_fwd_partial.argtypes = fwd_args + [P]
        lib.smla_fwd_partial.restype = I
        lib.smla_fwd_paged.argtypes = [P, P, I, P, P, P, P, I, I, I, I, P, I, I, I,
                                       I, I, I64, F, P, P, P, SZ, P]
        lib.smla_fwd_paged.restype = I
        lib.smla_fwd_split_q.argtypes = [P, P, P, I, P, F, P, P, I, I, I, I, I, I64, F,
                                         P, P, P, SZ, P]
        lib.smla_fwd_split_q.restype = I
        lib.smla_fwd_host.argtypes = fwd_args + [I, P, SZ, P]
        lib.smla_fwd_host.restype = I
        lib.smla_fwd_host_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.smla_fwd_host_workspace_size.restype = SZ
        lib.smla_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.smla_workspace_size.restype = SZ
        lib.smla_plan_info.argtypes = [I, I, I, I, I, I, ctypes.POINTER(I),
                                       ctypes.POINTER(I), ctypes.POINTER(SZ)]
        lib.smla_plan_info.restype = I
        lib.smla_plan_info_for.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(I),
                                           ctypes.POINTER(I), ctypes.POINTER(SZ)]
        lib.smla_plan_info_for.restype = I
        lib.smla_combine.argtypes = [P, P, I, I64, I, P, P, P]
        lib.smla_combine.restype = I
        lib.smla_get_device_status.argtypes = [ctypes.POINTER(I), I]
        lib.smla_get_device_status.restype = I
        lib.smla_test_set_stall.argtypes = [I, I]
        lib.smla_test_set_stall.restype = I
        lib.smla_status_string.argtypes = [I]
        lib.smla_status_string.restype = ctypes.c_char_p
        lib.smla_version.argtypes = []
        lib.smla_version.restype = I
        _lib = lib
        return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, what):
    if code != SMLA_OK:
        raise SmlaError(code, what)


def _require(cond, what):
    """Argument check of the binding (kept under ``python -O``)."""
    if not cond:
        raise ValueError(what)


def _kv_slots(kv_cache, kv_dtype, k_scale, d_qk, num_slots):
    """Check the cache and its scales; return the slot count."""
    import torch
    _require(kv_cache.is_cuda and kv_cache.is_contiguous(),
             "kv_cache must be a contiguous device tensor")
    if kv_dtype == SMLA_KV_BF16:
        _require(kv_cache.dtype == torch.bfloat16, "a bf16 cache must be torch.bfloat16")
    else:
        _require(kv_cache.dtype == torch.uint8, "an E4M3 cache must be torch.uint8 bytes")
    if kv_dtype in (SMLA_KV_FP8_E4M3, SMLA_KV_FP8_E4M3_GROUP128, SMLA_KV_FP8_E4M3_GROUP4_KPE):
        _require(k_scale is not None and k_scale.dtype == torch.float32 and
                 k_scale.is_cuda and k_scale.is_contiguous(),
                 "this cache format needs k_scale, a contiguous fp32 device tensor")
    row = DS_MLA_ROW_BYTES if kv_dtype == SMLA_KV_FP8_DS_MLA else d_qk
    return kv_cache.numel() // row if num_slots is None else int(num_slots)


def _idx_checks(indices, valid_len, T):
    import torch
    _require(indices.is_cuda and indices.dtype == torch.int32 and indices.is_contiguous()
             and indices.dim() == 2 and indices.shape[0] == T,
             "indices must be a contiguous int32 device tensor [T, topk]")
    if valid_len is not None:
        _require(valid_len.is_cuda and valid_len.dtype == torch.int32 and
                 valid_len.is_contiguous() and valid_len.shape == (T,),
                 "valid_len must be a contiguous int32 device tensor [T]")


def _in_args(q, kv_cache, kv_dtype, k_scale, indices, valid_len, sm_scale,
             num_slots):
    """The input arguments of the forward entry points, checked."""
    import torch
    _require(q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3,
             "q must be a contiguous bf16 device tensor [T, h, d_qk]")
    T, h, d_qk = q.shape
    S = _kv_slots(kv_cache, kv_dtype, k_scale, d_qk, num_slots)
    _idx_checks(indices, valid_len, T)
    return [_p(q), _p(kv_cache), int(kv_dtype), _p(k_scale), _p(indices),
            _p(valid_len), T, h, d_qk, 512, indices.shape[1], S, float(sm_scale)]


def _fwd_args(q, kv_cache, kv_dtype, k_scale, indices, valid_len, sm_scale,
              out, lse, num_slots):
    import torch
    _require(q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3,
             "q must be a contiguous bf16 device tensor [T, h, d_qk]")
    T, h, d_qk = q.shape
    S = _kv_slots(kv_cache, kv_dtype, k_scale, d_qk, num_slots)
    _idx_checks(indices, valid_len, T)
    topk = indices.shape[1]
    d_v = 512
    if out is None:
        out = torch.empty((T, h, d_v), dtype=torch.bfloat16, device=q.device)
    _require(out.dtype == torch.bfloat16 and out.is_contiguous() and out.shape == (T, h, d_v),
             "out must be contiguous bf16 [T, h, 512]")
    if lse is not None:
        _require(lse.dtype == torch.float32 and lse.is_contiguous() and lse.shape == (T, h),
                 "lse must be contiguous fp32 [T, h]")
    args = [_p(q), _p(kv_cache), int(kv_dtype), _p(k_scale), _p(indices),
            _p(valid_len), T, h, d_qk, d_v, topk, S, float(sm_scale),
            _p(out), _p(lse)]
    return args, out, lse


def smla_fwd(q, kv_cache, kv_dtype, k_scale, indices, valid_len, sm_scale,
             out=None, lse=None, want_lse=True, num_slots=None, stream=None):
    """Sparse MLA forward through ``smla_fwd`` (library-owned workspace).

    q bf16 [T,h,d_qk]; kv_cache bf16 or uint8 [S,d_qk]; k_scale f32 or None;
    indices int32 [T,topk]; valid_len int32 [T] or None.
    Returns (out bf16 [T,h,512], lse f32 [T,h] or None)."""
    import torch
    lib = load()
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args, out, lse = _fwd_args(q, kv_cache, kv_dtype, k_scale, indices,
                               valid_len, sm_scale, out, lse, num_slots)
    _check(lib.smla_fwd(*args, _stream(stream)), "smla_fwd")
    return out, lse


def smla_fwd_split_q(q_nope, q_pe, kv_cache, kv_dtype, k_scale, indices, valid_len,
                     sm_scale, kpe_scale=1.0, out=None, lse=None, want_lse=True,
                     num_slots=None, workspace=None, stream=None):
    """``smla_fwd_split_q``: the forward on q_nope bf16 [T,h,512] and q_pe
    bf16 [T,h,d_qk-512] (or None: q_nope is the concatenated q), with the
    rope scale kpe_scale for SMLA_KV_FP8_E4M3_GROUP4_KPE.
    Returns (out bf16 [T,h,512], lse f32 [T,h] or None)."""
    import torch
    lib = load()
    _require(q_nope.is_cuda and q_nope.dtype == torch.bfloat16 and q_nope.is_contiguous(),
             "q_nope must be a contiguous bf16 device tensor")
    if q_pe is None:
        T, h, d_qk = q_nope.shape
    else:
        T, h, d_nope = q_nope.shape
        _require(d_nope == 512 and q_pe.shape[:2] == (T, h),
                 "q_nope must be [T, h, 512] and q_pe [T, h, d_qk - 512]")
        _require(q_pe.is_cuda and q_pe.dtype == torch.bfloat16 and q_pe.is_contiguous(),
                 "q_pe must be a contiguous bf16 device tensor")
        d_qk = 512 + q_pe.shape[2]
    S = _kv_slots(kv_cache, kv_dtype, k_scale, d_qk, num_slots)
    _idx_checks(indices, valid_len, T)
    if out is None:
        out = torch.empty((T, h, 512), dtype=torch.bfloat16, device=q_nope.device)
    _require(out.dtype == torch.bfloat16 and out.is_contiguous() and out.shape == (T, h, 512),
             "out must be contiguous bf16 [T, h, 512]")
    if lse is None and want_lse:
        lse = torch.empty((T, h), dtype=torch.float32, device=q_nope.device)
    if lse is not None:
        _require(lse.dtype == torch.float32 and lse.is_contiguous() and lse.shape == (T, h),
                 "lse must be contiguous fp32 [T, h]")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.smla_fwd_split_q(_p(q_nope), _p(q_pe), _p(kv_cache), int(kv_dtype),
                                _p(k_scale), float(kpe_scale), _p(indices), _p(valid_len),
                                T, h, d_qk, 512, indices.shape[1], S, float(sm_scale),
                                _p(out), _p(lse), _p(workspace), nbytes, _stream(stream)),
           "smla_fwd_split_q")
    return out, lse


def smla_cache_write_e4m3_group(kv_c, k_pe, slot_mapping, kv_cache, scales,
                                stream=None):
    """``smla_cache_write_e4m3_group``: quantize token rows [kv_c | k_pe]
    (bf16 [N,512] and [N,64], or k_pe None for 512-channel rows) into the
    E4M3 cache (uint8 [S, d_qk]) with one fp32 scale per (slot, 128-channel
    group) (scales [S, ceil(d_qk/128)]) at rows slot_mapping (int32 [N];
    negative = skip)."""
    import torch
    lib = load()
    N = kv_c.shape[0]
    for x in (kv_c, k_pe):
        if x is not None:
            _require(x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous(),
                     "kv_c and k_pe must be contiguous bf16 device tensors")
    _require(kv_c.shape == (N, 512), "kv_c must be [N, 512]")
    d_qk = 512 if k_pe is None else 512 + k_pe.shape[1]
    _require(slot_mapping.dtype == torch.int32 and slot_mapping.shape == (N,),
             "slot_mapping must be int32 [N]")
    _require(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 2 and kv_cache.shape[1] == d_qk,
             "kv_cache must be uint8 [S, d_qk]")
    _require(scales.dtype == torch.float32 and
             scales.shape == (kv_cache.shape[0], (d_qk + 127) // 128),
             "scales must be fp32 [S, ceil(d_qk / 128)]")
    _check(lib.smla_cache_write_e4m3_group(_p(kv_c), _p(k_pe), _p(slot_mapping), N, d_qk,
                                           kv_cache.shape[0], _p(kv_cache), _p(scales),
                                           _stream(stream)), "smla_cache_write_e4m3_group")
    return kv_cache, scales


def smla_fwd_partial(q, kv_cache, kv_dtype, k_scale, indices, valid_len,
                     sm_scale, out=None, lse=None, num_slots=None, stream=None):
    """``smla_fwd_partial``: normalised fp32 O [T,h,512] and LSE [T,h] for an
    LSE-weighted merge (smla_combine).  Returns (out, lse)."""
    import torch
    lib = load()
    T, h, _ = q.shape
    if out is None:
        out = torch.empty((T, h, 512), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((T, h), dtype=torch.float32, device=q.device)
    _require(out.dtype == torch.float32 and out.is_contiguous() and out.shape == (T, h, 512),
             "out must be contiguous fp32 [T, h, 512]")
    _require(lse.dtype == torch.float32 and lse.is_contiguous() and lse.shape == (T, h),
             "lse must be contiguous fp32 [T, h]")
    args = _in_args(q, kv_cache, kv_dtype, k_scale, indices, valid_len,
                    sm_scale, num_slots) + [_p(out), _p(lse)]
    _check(lib.smla_fwd_partial(*args, _stream(stream)), "smla_fwd_partial")
    return out, lse


def smla_fwd_paged(q, kv_cache, kv_dtype, k_scale, token_indices, req_id,
                   block_table, block_size, sm_scale, valid_len=None,
                   block_stride_rows=0, out=None, lse=None, want_lse=True,
                   num_slots=None, workspace=None, stream=None):
    """``smla_fwd_paged``: the forward on request-local top-k indices.

    token_indices int32 [T,topk] (positions in the token's request, -1 =
    none); req_id int32 [T]; block_table int32 [num_reqs, stride]; the slot
    of position e is block_table[req, e // block_size] * block_stride_rows +
    e % block_size (block_stride_rows 0 = block_size).  workspace: a uint8
    device tensor (caller-owned, as smla_fwd_ws) or None (library-owned).
    Returns (out, lse) as smla_fwd."""
    import torch
    lib = load()
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args, out, lse = _fwd_args(q, kv_cache, kv_dtype, k_scale, token_indices,
                               valid_len, sm_scale, out, lse, num_slots)
    for x in (req_id, block_table):
        _require(x.is_cuda and x.dtype == torch.int32 and x.is_contiguous(),
                 "req_id and block_table must be contiguous int32 device tensors")
    _require(req_id.shape == (args[6],) and block_table.dim() == 2,
             "req_id must be [T] and block_table [num_reqs, stride]")
    ws_p = None if workspace is None else _p(workspace)
    ws_n = 0 if workspace is None else workspace.numel()
    pargs = args[:4] + [args[4], _p(req_id), _p(block_table),
                        int(block_table.shape[0]), int(block_table.shape[1]),
                        int(block_size), int(block_stride_rows), args[5]] + args[6:]
    _check(lib.smla_fwd_paged(*pargs, ws_p, ws_n, _stream(stream)),
           "smla_fwd_paged")
    return out, lse


def smla_workspace_size(T, h, d_qk, topk, kv_dtype, d_v=512) -> int:
    return int(load().smla_workspace_size(T, h, d_qk, d_v, topk, kv_dtype))


KERNEL_NAMES = {0: "cuda_core", 1: "tc_heads", 2: "tc_keys", 3: "tc_keys_fp8"}


def smla_plan_info(T, h, d_qk, topk, kv_dtype, d_v=512) -> dict:
    """``smla_plan_info``: the kernel family, top-k splits and workspace a
    forward of this shape uses on the current device."""
    lib = load()
    k, s, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    _check(lib.smla_plan_info(T, h, d_qk, d_v, topk, kv_dtype, ctypes.byref(k),
                              ctypes.byref(s), ctypes.byref(n)), "smla_plan_info")
    return {"kernel": KERNEL_NAMES[k.value], "splits": s.value,
            "workspace_bytes": n.value}


def smla_plan_info_for(T, h, d_qk, topk, kv_dtype, num_sms, d_v=512) -> dict:
    """``smla_plan_info_for``: the same plan for a device with ``num_sms``
    SMs, without a device query (works on a host without a GPU)."""
    lib = load()
    k, s, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_size_t(0)
    _check(lib.smla_plan_info_for(T, h, d_qk, d_v, topk, kv_dtype, num_sms, ctypes.byref(k),
                                  ctypes.byref(s), ctypes.byref(n)), "smla_plan_info_for")
    return {"kernel": KERNEL_NAMES[k.value], "splits": s.value,
            "workspace_bytes": n.value}


def smla_fwd_ws(q, kv_cache, kv_dtype, k_scale, indices, valid_len, sm_scale,
                workspace, out=None, lse=None, want_lse=True, num_slots=None,
                stream=None):
    """``smla_fwd_ws``: as smla_fwd with a caller-owned workspace tensor
    (uint8 on the device, at least smla_workspace_size bytes)."""
    import torch
    lib = load()
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    args, out, lse = _fwd_args(q, kv_cache, kv_dtype, k_scale, indices,
                               valid_len, sm_scale, out, lse, num_slots)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.smla_fwd_ws(*args, _p(workspace), nbytes, _stream(stream)),
           "smla_fwd_ws")
    return out, lse


def smla_fwd_host_workspace_size(T, h, d_qk, topk, kv_dtype, d_v=512,
                                 chunk_tokens=0) -> int:
    return int(load().smla_fwd_host_workspace_size(T, h, d_qk, d_v, topk,
                                                   kv_dtype, chunk_tokens))


def smla_fwd_host(q, kv_cache, kv_dtype, k_scale, indices, valid_len, sm_scale,
                  out=None, lse=None, want_lse=True, num_slots=None,
                  chunk_tokens=0, workspace=None, stream=None):
    """``smla_fwd_host``: q, indices, valid_len, out and lse are CPU tensors
    (pin them for overlap); kv_cache and k_scale are device tensors.  The
    copies and the forward are queued on ``stream`` (and the library's copy
    streams); synchronise the stream before reading ``out``/``lse``.
    ``workspace``: a device uint8 tensor of at least
    smla_fwd_host_workspace_size(...) bytes, or None to allocate one."""
    import torch
    lib = load()
    T, h, d_qk = q.shape
    d_v = 512
    if q.device.type != "cpu" or indices.device.type != "cpu" or \
            (valid_len is not None and valid_len.device.type != "cpu"):
        raise ValueError("smla_fwd_host: q, indices, valid_len live in host memory")
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be contiguous bf16 [T, h, d_qk]")
    if indices.dtype != torch.int32 or not indices.is_contiguous() or \
            indices.dim() != 2 or indices.shape[0] != T:
        raise ValueError("indices must be contiguous int32 [T, topk]")
    if valid_len is not None and (valid_len.dtype != torch.int32 or
                                  valid_len.shape != (T,) or
                                  not valid_len.is_contiguous()):
        raise ValueError("valid_len must be contiguous int32 [T]")
    topk = indices.shape[1]
    S = _kv_slots(kv_cache, kv_dtype, k_scale, d_qk, num_slots)
    if out is None:
        out = torch.empty((T, h, d_v), dtype=torch.bfloat16, pin_memory=True)
    if lse is None and want_lse:
        lse = torch.empty((T, h), dtype=torch.float32, pin_memory=True)
    for t in (out, lse):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError("out / lse must be contiguous host tensors")
    nbytes = smla_fwd_host_workspace_size(T, h, d_qk, topk, kv_dtype, d_v,
                                          chunk_tokens)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8,
                                device=kv_cache.device)
    _check(lib.smla_fwd_host(_p(q), _p(kv_cache), kv_dtype, _p(k_scale),
                             _p(indices), _p(valid_len), T, h, d_qk, d_v, topk,
                             S, float(sm_scale), _p(out), _p(lse),
                             int(chunk_tokens), _p(workspace),
                             workspace.numel(), _stream(stream)),
           "smla_fwd_host")
    return out, lse


def smla_combine(o_parts, lse_parts, out=None, lse=None, stream=None):
    """``smla_combine``: o_parts f32 [P, rows, 512], lse_parts f32 [P, rows]."""
    import torch
    lib = load()
    P, rows, d_v = o_parts.shape
    _require(o_parts.dtype == torch.float32 and o_parts.is_contiguous(),
             "o_parts must be contiguous fp32 [P, rows, 512]")
    _require(lse_parts.dtype == torch.float32 and lse_parts.is_contiguous() and
             lse_parts.shape == (P, rows), "lse_parts must be contiguous fp32 [P, rows]")
    if out is None:
        out = torch.empty((rows, d_v), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    _check(lib.smla_combine(_p(o_parts), _p(lse_parts), P, rows, d_v, _p(out),
                            _p(lse), _stream(stream)), "smla_combine")
    return out, lse


def smla_get_device_status(clear=True) -> int:
    v = ctypes.c_int(0)
    _check(load().smla_get_device_status(ctypes.byref(v), int(clear)),
           "smla_get_device_status")
    return v.value


def smla_test_set_stall(stall: bool, wait_limit_us: int = 0) -> None:
    """Tests of the timeout path only: while ``stall`` is set, tensor-core
    launches on the current device leave out each unit's first batch of
    score MMAs, so a bounded wait runs out after ``wait_limit_us`` (0 = the
    default limit) and the launch reports SMLA_ERR_TIMEOUT."""
    _check(load().smla_test_set_stall(int(bool(stall)), int(wait_limit_us)),
           "smla_test_set_stall")


def smla_status_string(code: int) -> str:
    return load().smla_status_string(int(code)).decode()

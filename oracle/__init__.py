"""fp64 CPU oracle for the sparse MLA attention forward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never does, and this package imports nothing from the product.

The arithmetic lives in ``smla_oracle.c`` (plain C, fp64); this module builds
it with gcc and marshals numpy arrays to it.  The C file's header gives the
definition it follows and the pages it cites.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsmla_oracle.so")
_lib = None
_lock = threading.Lock()

KV_BF16 = 0
KV_E4M3 = 1
KV_E4M3_GROUP128 = 2
KV_FP8_DS_MLA = 3          # 656-byte rows: 512 E4M3 | 4 fp32 scales | 64 bf16
KV_E4M3_GROUP4_KPE = 4     # E4M3 [S, 576], scales [S, 4] (ckv), one kpe scale
DS_MLA_ROW_BYTES = 656


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (no fast-math, no FMA
    contraction, so the arithmetic is the C source's)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.smla_oracle_fwd.restype = ctypes.c_int
        lib.smla_oracle_fwd.argtypes = [
            P, P, ctypes.c_int, P, ctypes.c_float, P, P, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
            ctypes.c_double, P, ctypes.c_int64, P, P, ctypes.c_int]
        lib.smla_oracle_merge.restype = None
        lib.smla_oracle_merge.argtypes = [P, P, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, P, P]
        lib.smla_oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.smla_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.smla_oracle_bf16_to_f64.restype = ctypes.c_double
        lib.smla_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3_to_f64(byte: int) -> float:
    return _load().smla_oracle_e4m3_to_f64(int(byte))


def bf16_to_f64(bits: int) -> float:
    return _load().smla_oracle_bf16_to_f64(int(bits))


def default_threads() -> int:
    return os.cpu_count() or 1


def sparse_mla_fwd(q_bits, kv, kv_dtype, k_scale, indices, valid_len,
                   sm_scale, d_v=512, num_slots=None, tokens=None,
                   n_threads=None, kpe_scale=1.0):
    """Oracle forward.

    q_bits    uint16 [T, h, d_qk]  (bf16 bit patterns)
    kv        uint16 [S, d_qk] (bf16 bits), uint8 [S, d_qk] (E4M3 bytes) or
              uint8 [S, 656] (KV_FP8_DS_MLA rows)
    kv_dtype  KV_BF16 / KV_E4M3 / KV_E4M3_GROUP128 / KV_FP8_DS_MLA /
              KV_E4M3_GROUP4_KPE
    k_scale   float32 [1], [S, ceil(d_qk/128)], [S, 4] (KV_E4M3_GROUP4_KPE) or None
    kpe_scale the rope channels' scale (KV_E4M3_GROUP4_KPE only)
    indices   int32 [T, topk];  valid_len int32 [T] or None
    tokens    optional int64 list of token ids (rows of the result follow it)
    Returns (O float64 [n, h, d_v], LSE float64 [n, h]).
    """
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    T, h, d_qk = q_bits.shape
    want = np.uint16 if kv_dtype == KV_BF16 else np.uint8
    row = DS_MLA_ROW_BYTES if kv_dtype == KV_FP8_DS_MLA else d_qk
    kv = np.ascontiguousarray(kv, dtype=want).reshape(-1, row)
    S = kv.shape[0] if num_slots is None else int(num_slots)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    assert indices.shape[0] == T
    topk = indices.shape[1]
    if valid_len is not None:
        valid_len = np.ascontiguousarray(valid_len, dtype=np.int32)
        assert valid_len.shape == (T,)
    if k_scale is not None:
        k_scale = np.ascontiguousarray(k_scale, dtype=np.float32)
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        n = tokens.shape[0]
    else:
        n = T
    out = np.zeros((n, h, d_v), dtype=np.float64)
    lse = np.zeros((n, h), dtype=np.float64)
    rc = lib.smla_oracle_fwd(
        _ptr(q_bits), _ptr(kv), int(kv_dtype), _ptr(k_scale), float(kpe_scale),
        _ptr(indices),
        _ptr(valid_len), T, h, d_qk, int(d_v), topk, S, float(sm_scale),
        _ptr(tokens), n, _ptr(out), _ptr(lse),
        int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"smla_oracle_fwd failed with code {rc}")
    return out, lse


def merge(o_parts, lse_parts):
    """LSE-weighted merge of partial results over disjoint key sets.

    o_parts float64 [P, rows, d_v] (each normalised over its keys),
    lse_parts float64 [P, rows].  Returns (O [rows, d_v], LSE [rows])."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    P, rows, d_v = o_parts.shape
    assert lse_parts.shape == (P, rows)
    out = np.zeros((rows, d_v), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    lib.smla_oracle_merge(_ptr(o_parts), _ptr(lse_parts), P, rows, d_v,
                          _ptr(out), _ptr(lse))
    return out, lse


def paged_to_global(token_indices, req_id, block_table, block_size,
                    block_stride_rows=0):
    """Request-local top-k positions -> global cache slots, entry by entry.

    Follows the index conversion the serving backends run before the
    attention call (vLLM "Sparse MLA on Hopper" diff, kernel test file,
    index-conversion tests 2.5 and 2.9): for a position e >= 0 of token t in
    request r = req_id[t],
        slot = block_table[r, e // block_size] * stride + e % block_size,
    stride = block_stride_rows or block_size (the BLOCK_STRIDE_ROWS option);
    entries < 0 stay -1.  Readings where the pages are silent: a request id
    outside [0, num_reqs), a block index past the table's width, and a
    negative (unallocated) table entry all give -1.  Returns int64 [T, topk]
    with -1 for masked entries; slots past the cache are left for the
    forward to mask.
    """
    idx = np.asarray(token_indices, dtype=np.int64)
    req = np.asarray(req_id, dtype=np.int64)
    table = np.asarray(block_table, dtype=np.int64)
    stride = int(block_stride_rows) or int(block_size)
    T, K = idx.shape
    out = np.full((T, K), -1, dtype=np.int64)
    for t in range(T):
        r = int(req[t])
        if r < 0 or r >= table.shape[0]:
            continue
        for j in range(K):
            e = int(idx[t, j])
            if e < 0:
                continue
            page = e // block_size
            if page >= table.shape[1]:
                continue
            blk = int(table[r, page])
            if blk < 0:
                continue
            out[t, j] = blk * stride + e % block_size
    return out


def _e4m3_positive_values():
    """Values of the codes 0x00..0x7E (0x7F is NaN), ascending."""
    return np.array([e4m3_to_f64(c) for c in range(0x7F)], dtype=np.float64)


def e4m3_encode(v):
    """float32 values -> E4M3 ("fn") codes, round to nearest with ties to the
    even code, saturating at +-448 (the satfinite conversion); the sign is
    kept for values that round to zero.  Written from the format's value
    list, not from a conversion routine."""
    vals = _e4m3_positive_values()
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    i = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, len(vals) - 1)
    j = np.minimum(i + 1, len(vals) - 1)
    lo, hi = vals[i], vals[j]
    d_lo, d_hi = a - lo, hi - a
    code = np.where(d_lo < d_hi, i, j)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(i % 2 == 0, i, j), code)
    code = np.where(a >= vals[-1], len(vals) - 1, code).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def cache_write_e4m3_group(kv_c_bits, k_pe_bits, slot_mapping, cache, scales):
    """The group-quantizing E4M3 cache write (test infrastructure).

    The flashinfer_mla_sparse_sm90.py page reads the per-token x
    128-channel-group scale layout (``ckv_scale_arr``) but notes that the
    cache-write op producing it is missing; vLLM's concat_and_cache_mla
    (same pages) writes a token's [kv_c | k_pe] row at its slot.  Reading:
    for each written row and group g (channels [128 g, 128 g + 128)),
    scale = amax|x| / 448 in fp32 (1 for an all-zero group) and
    code = e4m3(x / scale) (fp32 division, round to nearest even,
    saturating).  Rows with slot < 0 or >= num_slots are not written.
    kv_c_bits: uint16 bf16 bits [N, 512]; k_pe_bits: [N, d_qk - 512] or
    None; cache: uint8 [S, d_qk] (updated in place); scales: fp32 [S, G].
    """
    kv = np.asarray(kv_c_bits, dtype=np.uint16)
    rows = kv if k_pe_bits is None else np.concatenate(
        [kv, np.asarray(k_pe_bits, dtype=np.uint16)], axis=1)
    x_all = (rows.astype(np.uint32) << 16).view(np.float32)
    S, d_qk = cache.shape
    G = (d_qk + 127) // 128
    for n, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0 or s >= S:
            continue
        for g in range(G):
            x = x_all[n, 128 * g: min(128 * g + 128, d_qk)]
            amax = np.float32(np.max(np.abs(x)))
            scale = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
            cache[s, 128 * g: 128 * g + x.size] = e4m3_encode(x / scale)
            scales[s, g] = scale
    return cache, scales

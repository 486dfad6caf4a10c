"""Test-side glue: hand a generated workload to the oracle as numpy arrays."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def kv_numpy(w) -> np.ndarray:
    if w.kv.dtype == torch.bfloat16:
        return bits16(w.kv)
    return w.kv.detach().contiguous().cpu().numpy()


def oracle_fwd(w, tokens=None, valid=True, n_threads=None, indices=None):
    """Run the oracle on workload `w` (optionally a token subset)."""
    ks = None if w.k_scale is None else w.k_scale.detach().cpu().numpy()
    idx = (w.indices if indices is None else indices).detach().cpu().numpy()
    vl = w.valid_len.detach().cpu().numpy() if valid else None
    return oracle.sparse_mla_fwd(bits16(w.q), kv_numpy(w), w.kv_dtype, ks, idx,
                                 vl, w.sm_scale, d_v=w.d_v,
                                 num_slots=w.num_slots, tokens=tokens,
                                 n_threads=n_threads, kpe_scale=w.kpe_scale)


def dequant_rows_torch(w) -> torch.Tensor:
    """float64 [S, d_qk] dequantized cache via torch's own dtype casts (a
    library route independent of the oracle's decoder)."""
    if w.kv.dtype == torch.bfloat16:
        return w.kv.cpu().to(torch.float64)
    if w.kv_dtype == 3:                       # 656-byte rows
        rows = w.kv.cpu()
        codes = rows[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        sc = rows[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
        rope = rows[:, 528:656].contiguous().view(torch.bfloat16).to(torch.float64)
        return torch.cat([codes * sc[:, torch.arange(512) // 128], rope], dim=1)
    x = w.kv.cpu().view(torch.float8_e4m3fn).to(torch.float64)
    if w.kv_dtype == 4:                       # 4 ckv group scales + kpe scale
        sc = w.k_scale.cpu().to(torch.float64)
        return torch.cat([x[:, :512] * sc[:, torch.arange(512) // 128],
                          x[:, 512:] * w.kpe_scale], dim=1)
    if w.kv_dtype == 1:
        return x * float(w.k_scale.cpu()[0])
    grp = torch.arange(w.d_qk) // 128
    return x * w.k_scale.cpu().to(torch.float64)[:, grp]


# Out-of-bounds write check (compute-sanitizer is closed on this machine): output
# and workspace buffers are carved out of a larger allocation whose first and
# last GUARD bytes hold a sentinel; after the launch every sentinel byte must
# be intact.  The buffer itself starts filled with the sentinel too, so a
# value the kernel never wrote shows up as a mismatch against the oracle.
GUARD = 4096
SENTINEL = 0x5A


class Guarded:
    def __init__(self, shape, dtype, device="cuda"):
        n = 1
        for s in shape:
            n *= int(s)
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), SENTINEL,
                              dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def check(self, what=""):
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.nbytes:]
        bad_lo = int((lo != SENTINEL).sum().item())
        bad_hi = int((hi != SENTINEL).sum().item())
        assert bad_lo == 0 and bad_hi == 0, \
            f"{what}: {bad_lo} bytes written below and {bad_hi} above the buffer"

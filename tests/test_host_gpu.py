"""smla_fwd_host: the forward on host-resident q / indices / valid_len / O /
LSE, chunked with the copies overlapped, through the C ABI.

Each chunk runs smla_fwd_ws on its tokens.  Where a chunk's split plan is
the whole batch's (no top-k split in either), the result must equal the
device entry point's bit for bit; every case is also checked against the
fp64 oracle.  The cases cover several chunks with a ragged last one, the
default chunking, both kernel families, NULL valid_len and LSE, a single
chunk, and the argument errors."""
import pytest
import torch

from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import oracle_fwd
from tests.test_parity_gpu import compare

pytestmark = pytest.mark.gpu


def _host_run(smla, w, chunk_tokens, valid=True, want_lse=True):
    q = w.q.cpu().pin_memory()
    idx = w.indices.cpu().pin_memory()
    vl = w.valid_len.cpu().pin_memory() if valid else None
    kv = w.kv.cuda()
    ks = None if w.k_scale is None else w.k_scale.cuda()
    out, lse = smla.smla_fwd_host(q, kv, w.kv_dtype, ks, idx, vl, w.sm_scale,
                                  want_lse=want_lse, num_slots=w.num_slots,
                                  chunk_tokens=chunk_tokens)
    torch.cuda.current_stream().synchronize()
    return out, lse


def _device_run(smla, w, valid=True, want_lse=True):
    wd = w.to("cuda")
    out, lse = smla.smla_fwd(wd.q, wd.kv, wd.kv_dtype, wd.k_scale, wd.indices,
                             wd.valid_len if valid else None, wd.sm_scale,
                             want_lse=want_lse, num_slots=wd.num_slots)
    torch.cuda.synchronize()
    return out.cpu(), None if lse is None else lse.cpu()


@pytest.mark.parametrize("kv_dtype,h", [(0, 128), (2, 16), (1, 64)])
def test_chunks_equal_device_path(cuda_lib, kv_dtype, h):
    """300 tokens in chunks of 64 (five chunks, the last of 44)."""
    w = W.custom(T=300, h=h, topk=256, num_slots=1500, kv_dtype=kv_dtype,
                 valid=list(range(1, 257)) + [256] * 44, seed=300 + kv_dtype)
    Oh, Lh = _host_run(cuda_lib, w, 64)
    Or, Lr = oracle_fwd(w)
    compare(Oh, Lh, Or, Lr, "host path, chunks of 64")
    same_plan = all(cuda_lib.smla_plan_info(n, h, 576, 256, kv_dtype)["splits"] == 1
                    for n in (64, 44, 300))
    if same_plan:
        Od, Ld = _device_run(cuda_lib, w)
        assert torch.equal(Oh, Od) and torch.equal(Lh, Ld)


def test_default_chunking_matches_oracle(cuda_lib):
    """1000 tokens with the default chunking (256: four chunks, the last of
    232), bit-exact against the device path and within the bar of the
    oracle on a sample of tokens."""
    w = W.custom(T=1000, h=16, topk=128, num_slots=800, kv_dtype=2,
                 valid=[(7 * t) % 129 for t in range(1000)], seed=310)
    assert cuda_lib.smla_fwd_host_workspace_size(1000, 16, 576, 128, 2) > 0
    Oh, Lh = _host_run(cuda_lib, w, 0)
    Od, Ld = _device_run(cuda_lib, w)
    assert torch.equal(Oh, Od) and torch.equal(Lh, Ld)
    sel = list(range(0, 1000, 37))
    Or, Lr = oracle_fwd(w, tokens=sel)
    compare(Oh[sel], Lh[sel], Or, Lr, "host path vs oracle")


def test_null_valid_len_and_lse_one_chunk(cuda_lib):
    w = W.custom(T=40, h=32, topk=96, num_slots=400, kv_dtype=0,
                 valid=[96] * 40, seed=320)
    w.indices[::3, 50:] = -1
    Oh, Lh = _host_run(cuda_lib, w, 0, valid=False, want_lse=False)
    Od, _ = _device_run(cuda_lib, w, valid=False, want_lse=False)
    assert Lh is None and torch.equal(Oh, Od)


def test_argument_errors(cuda_lib):
    w = W.custom(T=100, h=16, topk=64, num_slots=300, kv_dtype=0,
                 valid=[64] * 100, seed=330)
    q, idx = w.q.pin_memory(), w.indices.pin_memory()
    kv = w.kv.cuda()
    need = cuda_lib.smla_fwd_host_workspace_size(100, 16, 576, 64, 0, 512, 32)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.SmlaError) as e:
        cuda_lib.smla_fwd_host(q, kv, 0, None, idx, None, w.sm_scale,
                               chunk_tokens=32, workspace=small)
    assert e.value.code == 6                          # SMLA_ERR_WORKSPACE
    with pytest.raises(cuda_lib.SmlaError) as e:
        cuda_lib.smla_fwd_host(q, kv, 0, None, idx, None, w.sm_scale,
                               chunk_tokens=-1)
    assert e.value.code == 1                          # SMLA_ERR_INVALID_ARG

"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a closed
form, an invariant, a library routine (torch's dtype casts, torch's
scaled_dot_product_attention in float64) or an independently written brute
force.  A dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sparse_mla_attention_02_gb300 import workloads as W
from tests._helpers import dequant_rows_torch, oracle_fwd

RTOL = 1e-12


def _close(a, b, rtol=RTOL, atol=1e-12):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


# ---------------------------------------------------------------- decoders --

def test_e4m3_decode_all_256_codes():
    """E4M3 ('fn') decoding equals torch.float8_e4m3fn for every byte."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(5)
    bits = np.concatenate([rng.integers(0, 1 << 16, 4000),
                           [0, 0x8000, 0x0001, 0x7F7F, 0x3F80, 0xBF80]])
    ref = torch.from_numpy(bits.astype(np.int32)).to(torch.int16).view(
        torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


# ------------------------------------------------------------ closed forms --

@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3,
                                      W.KV_FP8_E4M3_GROUP128])
def test_single_key_gives_that_row(kv_dtype):
    """topk=1, one valid entry: O = V_idx exactly, LSE = its scaled score."""
    w = W.custom(T=6, h=5, topk=1, num_slots=40, kv_dtype=kv_dtype,
                 valid=[1] * 6, seed=11)
    O, L = oracle_fwd(w)
    K = dequant_rows_torch(w).numpy()
    q = w.q.to(torch.float64).numpy()
    idx = w.indices.numpy()[:, 0]
    for t in range(w.T):
        for p in range(w.h):
            assert np.array_equal(O[t, p], K[idx[t], :512])
            s = w.sm_scale * float(np.dot(q[t, p], K[idx[t]]))
            _close(L[t, p], s)


def test_zero_query_gives_mean_and_log_count():
    """q = 0: every score is 0, so LSE = ln v and O = mean of the V rows."""
    w = W.custom(T=4, h=3, topk=16, num_slots=64, valid=[16, 7, 1, 3], seed=3)
    w.q.zero_()
    O, L = oracle_fwd(w)
    K = dequant_rows_torch(w).numpy()
    for t in range(w.T):
        v = int(w.valid_len[t])
        rows = K[w.indices.numpy()[t, :v], :512]
        for p in range(w.h):
            _close(L[t, p], math.log(v))
            _close(O[t, p], rows.mean(axis=0))


def test_identical_rows_give_lse_log_count_plus_score():
    """All selected rows equal to r: O = r[:512], LSE = ln v + s(r)."""
    w = W.custom(T=3, h=4, topk=12, num_slots=32, valid=[12, 5, 2], seed=4)
    w.kv[:] = w.kv[7]
    O, L = oracle_fwd(w)
    r = w.kv[7].to(torch.float64).numpy()
    q = w.q.to(torch.float64).numpy()
    for t in range(w.T):
        v = int(w.valid_len[t])
        for p in range(w.h):
            _close(O[t, p], r[:512])
            _close(L[t, p], math.log(v) + w.sm_scale * float(np.dot(q[t, p], r)))


def test_equal_values_give_that_value_for_any_scores():
    """V rows all equal u (rope parts differ, so scores differ): O = u."""
    w = W.custom(T=3, h=4, topk=10, num_slots=30, valid=[10, 4, 9], seed=6)
    w.kv[:, :512] = w.kv[0, :512]
    O, L = oracle_fwd(w)
    u = w.kv[0, :512].to(torch.float64).numpy()
    for t in range(w.T):
        for p in range(w.h):
            _close(O[t, p], u, rtol=1e-12, atol=1e-13)
    assert np.all(np.isfinite(L))


@pytest.mark.parametrize("kv_dtype", [W.KV_FP8_E4M3, W.KV_FP8_E4M3_GROUP128])
def test_scale_applies_to_the_right_channels(kv_dtype):
    """One-hot q at channel c, one key: LSE = sm_scale * e4m3(b_c) * scale,
    where the scale is k_scale[0] (per tensor) or k_scale[idx, c // 128]
    (per token x 128-channel group, the rope channels in group 4)."""
    w = W.custom(T=1, h=1, topk=1, num_slots=9, kv_dtype=kv_dtype, valid=[1],
                 seed=8)
    idx = int(w.indices[0, 0])
    codes = w.kv[idx].view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in [0, 5, 127, 128, 300, 511, 512, 575]:
        w.q.zero_()
        w.q[0, 0, c] = 1.0
        O, L = oracle_fwd(w)
        if kv_dtype == W.KV_FP8_E4M3:
            sc = float(w.k_scale[0])
        else:
            sc = float(w.k_scale[idx, c // 128])
        _close(L[0, 0], w.sm_scale * codes[c] * sc)
    ch = np.arange(512)
    if kv_dtype == W.KV_FP8_E4M3:
        expect = codes[:512] * float(w.k_scale[0])
    else:
        expect = codes[:512] * w.k_scale[idx].to(torch.float64).numpy()[ch // 128]
    _close(O[0, 0], expect)


# -------------------------------------------------------------- invariants --

def test_permutation_of_prefix_leaves_result_unchanged():
    w = W.custom(T=5, h=4, topk=32, num_slots=128, valid=[32, 20, 9, 31, 2],
                 seed=9)
    O1, L1 = oracle_fwd(w)
    rng = np.random.default_rng(1)
    idx = w.indices.clone()
    for t in range(w.T):
        v = int(w.valid_len[t])
        idx[t, :v] = idx[t, :v][torch.from_numpy(rng.permutation(v))]
    O2, L2 = oracle_fwd(w, indices=idx)
    _close(O1, O2, rtol=1e-11, atol=1e-12)
    _close(L1, L2, rtol=1e-12, atol=1e-12)


def test_all_slots_equals_dense_sdpa():
    """topk covering every slot = dense non-causal attention (torch SDPA,
    float64, CPU) — the reference the pages' kernel tests use."""
    S, T, h = 48, 3, 4
    w = W.custom(T=T, h=h, topk=S, num_slots=S, valid=[S] * T, seed=12,
                 sm_scale=192 ** -0.5)
    O, L = oracle_fwd(w)
    K = w.kv.to(torch.float64)
    q = w.q.to(torch.float64)
    for t in range(T):
        ref = F.scaled_dot_product_attention(
            q[t].unsqueeze(0).unsqueeze(2),                  # [1, h, 1, 576]
            K.unsqueeze(0).unsqueeze(0).expand(1, h, S, 576),
            K[:, :512].unsqueeze(0).unsqueeze(0).expand(1, h, S, 512),
            scale=w.sm_scale).squeeze(0).squeeze(1)
        _close(O[t], ref.numpy(), rtol=1e-10, atol=1e-12)
        lse = torch.logsumexp(w.sm_scale * (q[t] @ K.T), dim=-1)
        _close(L[t], lse.numpy(), rtol=1e-12, atol=1e-12)


def test_split_union_equals_merge_of_parts():
    """Oracle over J equals the LSE-merge of the oracle over J1 and J2,
    J = J1 + J2 disjoint; an empty part is the merge identity."""
    w = W.custom(T=4, h=3, topk=40, num_slots=200, valid=[40, 23, 1, 0],
                 seed=13)
    O, L = oracle_fwd(w)
    idx = w.indices.clone()
    cut = [17, 5, 1, 0]
    a = idx.clone()
    b = idx.clone()
    for t in range(w.T):
        a[t, cut[t]:] = -1          # first part keeps positions < cut
        b[t, :cut[t]] = -1          # second part keeps the rest (scattered -1)
    Oa, La = oracle_fwd(w, indices=a)
    Ob, Lb = oracle_fwd(w, indices=b)
    Om, Lm = oracle.merge(np.stack([Oa, Ob]).reshape(2, -1, 512),
                          np.stack([La, Lb]).reshape(2, -1))
    Om = Om.reshape(O.shape)
    Lm = Lm.reshape(L.shape)
    _close(Om, O, rtol=1e-11, atol=1e-12)
    fin = np.isfinite(L)
    _close(Lm[fin], L[fin])
    assert np.all(np.isneginf(Lm[~fin]))
    assert (~fin).sum() == w.h  # token 3 has valid 0
    # token 2 (valid 1) has an empty second part: the merge is exact there
    assert np.array_equal(Om[2], O[2]) and np.array_equal(Lm[2], L[2])


# ---------------------------------------------------------- masking rules --

def test_empty_and_masked_rows_are_zero_and_neg_inf():
    """valid = 0, an all -1 prefix, and all ids out of range give (0, -inf)."""
    w = W.custom(T=4, h=2, topk=8, num_slots=16, valid=[0, 8, 8, 3], seed=14)
    w.indices[1, :] = -1
    w.indices[2, :] = 16          # == num_slots: out of range
    O, L = oracle_fwd(w)
    for t in range(3):
        assert np.all(O[t] == 0.0) and np.all(np.isneginf(L[t]))
    assert np.all(np.isfinite(L[3]))


def test_scattered_minus_one_equals_compacted_row():
    w = W.custom(T=2, h=3, topk=16, num_slots=64, valid=[16, 10], seed=15)
    idx = w.indices.clone()
    keep = [0, 2, 3, 7, 9, 12, 15]
    holes = torch.full((2, 16), -1, dtype=torch.int32)
    holes[0, keep] = idx[0, keep]
    comp = torch.full((2, 16), -1, dtype=torch.int32)
    comp[0, :len(keep)] = idx[0, keep]
    holes[1] = idx[1]
    comp[1] = idx[1]
    Oh, Lh = oracle_fwd(w, indices=holes)     # -1 inside the valid prefix
    w.valid_len = torch.tensor([len(keep), 10], dtype=torch.int32)
    Oc, Lc = oracle_fwd(w, indices=comp)
    _close(Oh, Oc, rtol=1e-11, atol=1e-12)
    _close(Lh, Lc)


def test_entries_past_valid_are_ignored_and_valid_is_clamped():
    w = W.custom(T=3, h=2, topk=12, num_slots=50, valid=[12, 6, 12], seed=16)
    O1, L1 = oracle_fwd(w)
    rng = np.random.default_rng(2)
    w.indices[1, 6:] = torch.from_numpy(rng.integers(0, 50, 6).astype(np.int32))
    w.valid_len = torch.tensor([99, 6, 12], dtype=torch.int32)  # 99 > topk
    O2, L2 = oracle_fwd(w)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_null_valid_len_takes_every_non_negative_id():
    w = W.custom(T=3, h=2, topk=12, num_slots=50, valid=[12, 6, 0], seed=17)
    O1, L1 = oracle_fwd(w)
    O2, L2 = oracle_fwd(w, valid=False)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    assert np.all(np.isneginf(L2[2]))


# ------------------------------------------------ independent brute force --

def _brute(q, K, idx, v, sm_scale, S):
    """Direct float64 Python: exp without max subtraction, LSE as defined."""
    T, h, d = q.shape
    O = np.zeros((T, h, 512))
    L = np.zeros((T, h))
    for t in range(T):
        J = [int(i) for i in idx[t, :v[t]] if 0 <= i < S]
        for p in range(h):
            if not J:
                L[t, p] = -math.inf
                continue
            e = []
            for j in J:
                s = 0.0
                for c in range(d):
                    s += float(q[t, p, c]) * float(K[j, c])
                e.append(math.exp(sm_scale * s))
            Z = sum(e)
            L[t, p] = math.log(Z)
            for k, j in enumerate(J):
                for c in range(512):
                    O[t, p, c] += e[k] / Z * float(K[j, c])
    return O, L


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3,
                                      W.KV_FP8_E4M3_GROUP128, W.KV_FP8_DS_MLA,
                                      W.KV_FP8_E4M3_GROUP4_KPE])
def test_brute_force_tiny(kv_dtype):
    w = W.custom(T=2, h=2, topk=8, num_slots=24, kv_dtype=kv_dtype,
                 valid=[8, 3], seed=21, sm_scale=0.02, k_scale=0.5,
                 scale_range=(0.2, 0.6))
    w.indices[0, 2] = -1
    w.indices[0, 5] = 24   # out of range inside the prefix
    O, L = oracle_fwd(w)
    Ob, Lb = _brute(w.q.to(torch.float64).numpy(),
                    dequant_rows_torch(w).numpy(), w.indices.numpy(),
                    w.valid_len.numpy(), w.sm_scale, w.num_slots)
    _close(O, Ob, rtol=1e-12, atol=1e-13)
    _close(L, Lb, rtol=1e-12, atol=1e-13)


def test_thread_count_does_not_change_result():
    w = W.custom(T=9, h=3, topk=20, num_slots=60, seed=22)
    O1, L1 = oracle_fwd(w, n_threads=1)
    O2, L2 = oracle_fwd(w, n_threads=7)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_token_subset_matches_full_run():
    w = W.custom(T=10, h=2, topk=16, num_slots=64, seed=23)
    O, L = oracle_fwd(w)
    sel = np.array([7, 0, 9, 3])
    Os, Ls = oracle_fwd(w, tokens=sel)
    assert np.array_equal(Os, O[sel]) and np.array_equal(Ls, L[sel])


# ------------------------------------------------- generator structure --

def test_config_inputs_have_the_stated_structure():
    w = W.tiny()
    assert list(w.valid_len.numpy()) == [64, 40, 17, 1]
    for t in range(w.T):
        v = int(w.valid_len[t])
        row = w.indices[t].numpy()
        assert np.all(row[v:] == -1) and len(set(row[:v])) == v
        assert np.all((row[:v] >= 0) & (row[:v] < 256))
    p = W.bf16_prefill(T=300, topk=64)
    for t in range(p.T):
        v = int(p.valid_len[t])
        assert v == min(t + 1, 64)
        row = p.indices[t].numpy()
        assert np.all(row[:v] <= t) and len(set(row[:v])) == v
        assert np.all(row[v:] == -1)


# ---- request-local index conversion (paged_to_global) ----------------------
# Pinned against the pages' worked cases and an independent construction, not
# against a retyping of the formula.


def test_paged_identity_table_gives_positions():
    """Kernel test file, test 2.9: with block_table = arange(num_blocks) and
    positions 0..nv-1 the converted ids equal the positions; -1 tails stay
    -1 and the valid counts (non -1 entries, test 2.5) are [1, 10, 50, 100]."""
    T, topk, nblk, bs = 4, 128, 16, 64
    valid = [1, 10, 50, 100]
    idx = np.full((T, topk), -1, dtype=np.int64)
    for t, nv in enumerate(valid):
        idx[t, :nv] = np.arange(nv)
    out = oracle.paged_to_global(idx, np.zeros(T), np.arange(nblk)[None, :], bs)
    for t, nv in enumerate(valid):
        assert np.array_equal(out[t, :nv], np.arange(nv))
        assert np.all(out[t, nv:] == -1)
        assert int((out[t] >= 0).sum()) == nv


def test_paged_inverts_a_random_block_assignment():
    """Build the global slots first (block b, offset o), place each block at
    a random page of a random request, derive the request-local position
    page * bs + o, and check the conversion recovers b * stride + o."""
    rng = np.random.default_rng(5)
    R, pages, bs, stride = 3, 6, 16, 24
    nblocks = R * pages
    perm = rng.permutation(nblocks).reshape(R, pages)   # table[r, page] = block
    T, K = 7, 20
    req = rng.integers(0, R, size=T)
    page = rng.integers(0, pages, size=(T, K))
    off = rng.integers(0, bs, size=(T, K))
    blk = perm[req[:, None], page]
    local = page * bs + off
    local[:, -3:] = -1
    out = oracle.paged_to_global(local, req, perm, bs, block_stride_rows=stride)
    want = blk * stride + off
    want[:, -3:] = -1
    assert np.array_equal(out, want)


def test_paged_masks_what_cannot_be_translated():
    """Readings: a page past the table, an unallocated (-1) block and a
    request id outside the table all give -1."""
    table = np.array([[4, -1, 7]])
    idx = np.array([[0, 5, 15, 16, 40, 47, 48, 100]])
    out = oracle.paged_to_global(idx, [0], table, 16)
    assert out.tolist() == [[64, 69, 79, -1, 120, 127, -1, -1]]
    assert oracle.paged_to_global(idx, [1], table, 16).tolist() == [[-1] * 8]
    assert oracle.paged_to_global(idx, [-1], table, 16).tolist() == [[-1] * 8]


# ---- E4M3 encoding and the group-quantizing cache write ---------------------


def test_e4m3_encode_round_trips_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), codes)


def test_e4m3_encode_midpoints_go_to_the_even_code():
    vals = np.array([oracle.e4m3_to_f64(c) for c in range(0x7F)])
    mid = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (vals[:-1] + vals[1:]) / 2)  # exact in fp32
    got = oracle.e4m3_encode(mid)
    want = np.where(np.arange(126) % 2 == 0, np.arange(126), np.arange(1, 127))
    assert np.array_equal(got, want.astype(np.uint8))


def test_e4m3_encode_agrees_with_torch_and_saturates():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 0.01, 5000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)
    big = np.array([448.0, 470.0, 1e6, -1e30, np.inf], dtype=np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def test_cache_write_quantizes_within_the_format_bound():
    rng = np.random.default_rng(1)
    N, S = 40, 64
    kv = rng.normal(0, 1, (N, 512)).astype(np.float32)
    pe = rng.normal(0, 3, (N, 64)).astype(np.float32)
    kv[3, 128:256] = 0.0                                      # an all-zero group
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)   # exact: truncate to bf16 below
    kv = (bits(kv).astype(np.uint32) << 16).view(np.float32)
    pe = (bits(pe).astype(np.uint32) << 16).view(np.float32)
    slots = rng.permutation(S)[:N].astype(np.int64)
    slots[5] = -1
    cache = np.full((S, 576), 0xAA, dtype=np.uint8)
    scales = np.full((S, 5), -1.0, dtype=np.float32)
    oracle.cache_write_e4m3_group(bits(kv), bits(pe), slots, cache, scales)
    rows = np.concatenate([kv, pe], axis=1).astype(np.float64)
    for n, s in enumerate(slots):
        if s < 0:
            continue
        for g in range(5):
            sl = slice(128 * g, min(128 * g + 128, 576))
            x = rows[n, sl]
            sc = float(scales[s, g])
            dq = np.array([oracle.e4m3_to_f64(int(b)) for b in cache[s, sl]]) * sc
            amax = np.abs(x).max()
            if amax == 0:
                assert sc == 1.0 and np.all(cache[s, sl] == 0)
                continue
            assert sc == np.float32(amax) / np.float32(448)
            # relative E4M3 spacing is at most 2^-3: error <= half of it at |x|,
            # or half the subnormal step 2^-9 * scale
            bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sc) * (1 + 1e-6)
            assert np.all(np.abs(dq - x) <= bound)
            assert np.max(np.abs(dq)) == pytest.approx(448 * sc, rel=1e-6)
    untouched = np.setdiff1d(np.arange(S), slots[slots >= 0])
    assert np.all(cache[untouched] == 0xAA) and np.all(scales[untouched] == -1.0)


# ------------------------------------------------------- layout variants --

def _e4m3_torch(b: int) -> float:
    return float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))


@pytest.mark.parametrize("kv_dtype", [W.KV_FP8_DS_MLA, W.KV_FP8_E4M3_GROUP4_KPE])
def test_layout_variant_channels_read_the_right_bytes(kv_dtype):
    """One-hot q at channel c, one key: LSE = sm_scale * K[c], K[c] decoded
    here from the row's own bytes with struct and torch's E4M3 cast.
    656-byte row: c < 512 -> e4m3(byte c) * fp32 at bytes 512 + 4 (c // 128);
    c >= 512 -> bf16 at bytes 528 + 2 (c - 512).  Four group scales + kpe
    scale: c < 512 -> e4m3 * k_scale[idx, c // 128]; c >= 512 -> e4m3 * kpe."""
    import struct
    w = W.custom(T=1, h=1, topk=1, num_slots=7, kv_dtype=kv_dtype, valid=[1],
                 seed=18, k_scale=0.37)
    idx = int(w.indices[0, 0])
    row = bytes(w.kv[idx].numpy().tobytes())
    for c in [0, 5, 127, 128, 255, 256, 300, 383, 384, 511, 512, 513, 543, 575]:
        if kv_dtype == W.KV_FP8_DS_MLA:
            if c < 512:
                sc = struct.unpack("<f", row[512 + 4 * (c // 128): 516 + 4 * (c // 128)])[0]
                val = _e4m3_torch(row[c]) * sc
            else:
                lo = 528 + 2 * (c - 512)
                val = struct.unpack("<f", b"\x00\x00" + row[lo: lo + 2])[0]
        else:
            sc = float(w.k_scale[idx, c // 128]) if c < 512 else float(np.float32(0.37))
            val = _e4m3_torch(row[c]) * sc
        w.q.zero_()
        w.q[0, 0, c] = 1.0
        O, L = oracle_fwd(w)
        _close(L[0, 0], w.sm_scale * val)
        if c < 512:
            _close(O[0, 0, c], val)


def test_ds_mla_rows_equal_the_bf16_rows_they_encode():
    """With power-of-two group scales every dequantized ckv value is a bf16
    value, so a bf16 cache holding the same rows must give the same result
    (both computed in fp64 from identical values)."""
    S, T, h = 40, 3, 4
    g = torch.Generator().manual_seed(5)
    scales = 2.0 ** -torch.randint(2, 7, (S, 4), generator=g).float()
    codes = W.fp8_cache_group(S, 512, scales, "cpu", g)
    rope = W.bf16_normal((S, 64), "cpu", g)
    ds = W.custom(T=T, h=h, topk=16, num_slots=S, kv_dtype=W.KV_FP8_DS_MLA,
                  valid=[16, 9, 1], seed=6)
    ds.kv = W.ds_mla_rows(codes, scales, rope)
    bf = W.custom(T=T, h=h, topk=16, num_slots=S, valid=[16, 9, 1], seed=6)
    ckv = codes.view(torch.float8_e4m3fn).to(torch.float32) * scales[:, torch.arange(512) // 128]
    bf.kv = torch.cat([ckv.to(torch.bfloat16), rope], dim=1).contiguous()
    assert torch.equal(bf.kv[:, :512].float(), ckv)          # the encoding is exact
    bf.q, bf.indices, bf.valid_len = ds.q, ds.indices, ds.valid_len
    O1, L1 = oracle_fwd(ds)
    O2, L2 = oracle_fwd(bf)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_group4_kpe_equals_group128_with_the_kpe_scale_as_group_4():
    """Four ckv group scales and a per-tensor kpe scale are the 5-group
    layout whose fifth (rope) scale is that kpe scale for every slot."""
    w4 = W.custom(T=3, h=3, topk=20, num_slots=50, kv_dtype=W.KV_FP8_E4M3_GROUP4_KPE,
                  valid=[20, 7, 0], seed=9, k_scale=0.21)
    w2 = W.custom(T=3, h=3, topk=20, num_slots=50, kv_dtype=W.KV_FP8_E4M3_GROUP128,
                  valid=[20, 7, 0], seed=9)
    w2.q, w2.kv, w2.indices, w2.valid_len = w4.q, w4.kv, w4.indices, w4.valid_len
    w2.k_scale = torch.cat([w4.k_scale, torch.full((50, 1), 0.21)], dim=1).contiguous()
    O1, L1 = oracle_fwd(w4)
    O2, L2 = oracle_fwd(w2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    assert np.isneginf(L1[2]).all()

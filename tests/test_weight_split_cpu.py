"""The E4M3 operand splits of the E4M3-operand kernel, by brute force.

That kernel multiplies the raw E4M3 cache bytes by a second operand that it
splits into E4M3 terms in f16 arithmetic: Q as a pair x = hi + lo/16 with
lo = E4M3(16 (x - hi)), the softmax weights as three terms
x = hi + mid/16 + lo/256 (each next term E4M3 of 16 times the residual),
with round-to-nearest-even E4M3 conversions.  These tests restate the
split with torch's own float8_e4m3fn casts (RNE) and check, over every
positive f16 value, the facts the kernel's error budget rests on:

* each residual and its product by 16 is exact in f16 (the kernel forms
  them with f16x2 subtractions and multiplications);
* the pair is within max(2^-9 of x's binade, 2^-14) of x, and 2^-9 is
  reached;
* the three terms give back every f16 value from 2^-6 up exactly, and
  smaller values to 2^-18 absolute; so a weight keeps only the f16
  rounding on the way in, 2^-11 of its binade.
"""
import numpy as np
import pytest
import torch

F16_MAX_SPLIT = 256.0     # the kernel keeps |x| <= 256 (2^4 from the lazy max, 2^4 shift)


def all_f16(lo=0.0, hi=F16_MAX_SPLIT):
    bits = np.arange(0x0001, 0x7C00, dtype=np.uint16)
    x = bits.view(np.float16).astype(np.float64)
    return x[(x > lo) & (x <= hi)]


def e4m3(v):
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def exact_in_f16(v):
    return np.array_equal(v.astype(np.float16).astype(np.float64), v)


def binade(x):
    return 2.0 ** np.floor(np.log2(x))


def test_residuals_are_exact_in_f16():
    x = all_f16()
    hi = e4m3(x)
    r1 = (x - hi) * 16
    assert exact_in_f16(x - hi) and exact_in_f16(r1)
    mid = e4m3(r1)
    r2 = (r1 - mid) * 16
    assert exact_in_f16(r1 - mid) and exact_in_f16(r2)
    assert np.abs(r1).max() <= F16_MAX_SPLIT and np.abs(r2).max() <= F16_MAX_SPLIT


def test_pair_bound():
    x = all_f16()
    hi = e4m3(x)
    lo = e4m3((x - hi) * 16)
    err = np.abs(x - (hi + lo / 16))
    assert np.all(err <= np.maximum(2.0 ** -9 * binade(x), 2.0 ** -14))
    big = x >= 0.25
    assert (err[big] / binade(x[big])).max() == 2.0 ** -9      # the bound is reached


def test_three_terms_give_back_f16():
    x = all_f16()
    hi = e4m3(x)
    r1 = (x - hi) * 16
    mid = e4m3(r1)
    lo = e4m3((r1 - mid) * 16)
    err = np.abs(x - (hi + mid / 16 + lo / 256))
    assert np.all(err[x >= 2.0 ** -6] == 0.0)
    assert err.max() <= 2.0 ** -18


@pytest.mark.parametrize("seed", [0, 1])
def test_f16_step(seed):
    y = np.random.default_rng(seed).uniform(2.0 ** -6, F16_MAX_SPLIT, 100000)
    err = np.abs(y.astype(np.float16).astype(np.float64) - y)
    assert (err / binade(y)).max() <= 2.0 ** -11

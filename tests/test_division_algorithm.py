"""The division form's quotient, emulated exactly on the CPU.

The logits kernel's sampler-parity form computes z = x / t for bf16 x and
fp32 t as Markstein's correction of a reciprocal product (P. Markstein,
"Computation of elementary functions on the IBM RISC System/6000 processor",
IBM J. Res. Dev. 34(1), 1990):

    r = RN(1 / t);  q0 = RN(x * r);  rem = RN(x - q0 * t) (one FMA, exact);
    z = RN(q0 + rem * r) (one FMA)

Where every intermediate is a normal number the steps scale exactly with the
exponents of x and t, so the significands decide everything: x in [1, 2)
(the 128 bf16 significands) against t in [1, 2). This test replays the steps
with exact float64 products and an error-free sum, and compares the result
with numpy's IEEE float32 division. The default run samples temperature
significands; LMH_EXHAUSTIVE_DIVISION=1 runs all 2^23 of them (about a
minute and a half). The GPU test of the same quotient against CUDA's IEEE
division is in test_gpu_parity.py.
"""

import os

import numpy as np

M = 1.0 + np.arange(128) / 128.0  # bf16 significands in [1, 2)


def _rn32_sum(a, b):
    """fp32 round-to-nearest of the exact sum a + b (float64 inputs)."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)  # a + b == s + err exactly
    f = s.astype(np.float32)
    f64 = f.astype(np.float64)
    up = np.nextafter(f, np.float32(np.inf))
    dn = np.nextafter(f, np.float32(-np.inf))
    at_up = s == (f64 + up.astype(np.float64)) / 2  # s on a midpoint: err decides
    at_dn = s == (f64 + dn.astype(np.float64)) / 2
    f = np.where(at_up & (err > 0), up, f)
    return np.where(at_dn & (err < 0), dn, f)


def _markstein(t32):
    """The kernel's quotient for every significand in M and each t (fp32 [n])."""
    t64 = t32.astype(np.float64)[:, None]
    r = (np.float32(1.0) / t32).astype(np.float64)[:, None]  # RN(1/t)
    m = M[None, :]
    q0 = (m * r).astype(np.float32)  # the product is exact in float64: one rounding
    rem = (m - q0.astype(np.float64) * t64).astype(np.float32)  # exact difference
    return _rn32_sum(q0.astype(np.float64), rem.astype(np.float64) * r)


def _count_bad(t32):
    ref = M[None, :].astype(np.float32) / t32[:, None]
    return int((_markstein(t32) != ref).sum())


def test_markstein_quotient_is_correctly_rounded():
    if os.environ.get("LMH_EXHAUSTIVE_DIVISION") == "1":
        sig = np.arange(1 << 23, dtype=np.int64)
    else:
        sig = np.random.default_rng(0).integers(0, 1 << 23, size=40000)
        sig = np.concatenate([sig, [0, 1, (1 << 23) - 1, (1 << 22), 0x36db6e]])  # 1/0.7 ~ 1.4286
    bad = 0
    for c in range(0, len(sig), 1 << 15):
        t32 = (sig[c:c + (1 << 15)] | (127 << 23)).astype(np.uint32).view(np.float32)
        bad += _count_bad(t32)
    assert bad == 0


def test_plain_reciprocal_product_is_not():
    """Without the correction (z = RN(x * RN(1/t))) many quotients are off by
    one ulp: the check above would see a skipped step."""
    t32 = (np.random.default_rng(1).integers(0, 1 << 23, size=2000) | (127 << 23)).astype(
        np.uint32).view(np.float32)
    r = (np.float32(1.0) / t32).astype(np.float64)[:, None]
    q0 = (M[None, :] * r).astype(np.float32)
    ref = M[None, :].astype(np.float32) / t32[:, None]
    assert int((q0 != ref).sum()) > 1000


def test_every_bf16_input_of_the_fast_range():
    """All bf16 x with |x| in [2^-100, 2^100] at temperatures across
    [2^-20, 2^20] (the kernel sends zeros and every other input to IEEE
    division)."""
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    with np.errstate(invalid="ignore"):
        ax = np.abs(bits.astype(np.float64))
    x32 = bits[np.isfinite(bits) & (ax >= 2.0 ** -100) & (ax <= 2.0 ** 100)]
    x64 = x32.astype(np.float64)
    rng = np.random.default_rng(2)
    ex = rng.integers(-20, 20, size=150)
    sig = rng.integers(0, 1 << 23, size=150)
    ts = ((sig | ((127 + ex) << 23)).astype(np.uint32)).view(np.float32)
    ts = np.concatenate([ts, np.array([2.0 ** -20, 2.0 ** 20, 0.7, 1.0], np.float32)])
    for t32 in ts:
        r = np.float64(np.float32(1.0) / t32)
        q0 = (x64 * r).astype(np.float32)
        rem = (x64 - q0.astype(np.float64) * np.float64(t32)).astype(np.float32)
        z = _rn32_sum(q0.astype(np.float64), rem.astype(np.float64) * r)
        ref = x32 / t32
        assert np.array_equal(z.view(np.uint32), ref.view(np.uint32)), t32

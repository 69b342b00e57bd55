"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each check is written as a function of the oracle entry points it tests, so
that the planted-mistake tests at the end can run the same check on a mutated
copy and show that it fails.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle
from oracle import loops
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
S07 = oracle.fp32_scalar(1.0 / 0.7)


def _bf(x):
    """Round to bf16 and widen back, as the library's inputs are stored."""
    return W.bf16_bits_to_f32(W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _tiny(seed, T=3, H=8, V=16, oov_row=None):
    rng = np.random.default_rng(seed)
    hidden = _bf(rng.standard_normal((T, H)))
    weight = _bf(0.7 * rng.standard_normal((V, H)))
    labels = rng.integers(0, V, size=T).astype(np.int32)
    if oov_row is not None:
        labels[oov_row] = -100
    grad = rng.standard_normal(T).astype(np.float32)
    return hidden, weight, labels, grad


# ---------------------------------------------------------------------------
# checks (each returns the worst error it saw)
# ---------------------------------------------------------------------------

def check_loops_forward(fwd, seed, s):
    h, w, lab, _ = _tiny(seed, oov_row=1)
    got = fwd(h, w, lab, s)
    ref = loops.forward(h.tolist(), w.tolist(), lab.tolist(), s)
    return max(float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) for a, b in zip(got, ref))


def check_torch_log_softmax(sampler, seed):
    """The sampler formula as a torch call on CPU in float64."""
    rng = np.random.default_rng(seed)
    z = 3.0 * rng.standard_normal((17, 301))
    lab = rng.integers(0, 301, size=17)
    lp, _, _ = sampler(z, lab)
    ref = torch.log_softmax(torch.from_numpy(z), dim=-1).gather(
        -1, torch.from_numpy(lab).unsqueeze(-1)).squeeze(-1).numpy()
    return float(np.max(np.abs(lp - ref)))


def check_scipy_lse_entropy(sampler, seed):
    rng = np.random.default_rng(seed)
    z = 2.0 * rng.standard_normal((9, 257)) + 750.0  # exp() of these overflows fp64
    lab = rng.integers(0, 257, size=9)
    _, ent, lse = sampler(z, lab)
    ref_lse = scipy.special.logsumexp(z, axis=1)
    ref_ent = scipy.stats.entropy(scipy.special.softmax(z, axis=1), axis=1)
    return max(float(np.max(np.abs(lse - ref_lse))), float(np.max(np.abs(ent - ref_ent))))


def check_two_value(sampler, V, k, a, b):
    """k logits equal a, V - k equal b: closed-form lse, log-probs and entropy."""
    z = np.full((2, V), b, dtype=np.float64)
    z[:, :k] = a
    lab = np.array([0, V - 1])
    lp, ent, lse = sampler(z, lab)
    m = max(a, b)
    zsum = k * math.exp(a - m) + (V - k) * math.exp(b - m)
    ref_lse = m + math.log(zsum)
    pa = math.exp(a - ref_lse)
    pb = math.exp(b - ref_lse)
    ref_ent = -(k * pa * math.log(pa) + (V - k) * pb * math.log(pb))
    errs = [abs(lse[0] - ref_lse), abs(lp[0] - (a - ref_lse)), abs(lp[1] - (b - ref_lse)),
            abs(ent[0] - ref_ent)]
    return max(errs)


def _fd_objective(h, w, lab, g, s, fwd):
    """sum_t g_t * logprob_t for labels inside the vocab and -g_t * lse_t outside.

    The second term is what the out-of-vocab convention differentiates: the
    forward value is masked to 0, and the backward keeps only -softmax * g.
    """
    lp, _, lse = fwd(h, w, lab, s)
    V = w.shape[0]
    inside = (lab >= 0) & (lab < V)
    return float(np.sum(np.where(inside, g * lp, -g * lse)))


def check_finite_differences(fwd, bwd, seed, s, oov_row=None, eps=1e-6):
    h, w, lab, g = _tiny(seed, oov_row=oov_row)
    h = h.astype(np.float64)
    w = w.astype(np.float64)
    g = g.astype(np.float64)
    gh, gw = bwd(h, w, lab, g, s)
    worst = 0.0
    for arr, grad in ((h, gh), (w, gw)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            fp = _fd_objective(h, w, lab, g, s, fwd)
            arr[idx] = old - eps
            fm = _fd_objective(h, w, lab, g, s, fwd)
            arr[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        worst = max(worst, float(np.max(np.abs(num - grad)) / (np.max(np.abs(num)) + 1e-300)))
    return worst


def _fd_objective_entropy(h, w, lab, g, gh, s, fwd):
    """The log-prob objective plus sum_t gH[t] * entropy[t]."""
    _, ent, _ = fwd(h, w, lab, s)
    return _fd_objective(h, w, lab, g, s, fwd) + float(np.sum(gh * ent))


def check_finite_differences_entropy(fwd, bwd, seed, s, oov_row=None, eps=1e-6):
    h, w, lab, g = _tiny(seed, oov_row=oov_row)
    h = h.astype(np.float64)
    w = w.astype(np.float64)
    g = g.astype(np.float64)
    gh = np.random.default_rng(seed + 100).standard_normal(len(g))
    dh, dw = bwd(h, w, lab, g, s, gh)
    worst = 0.0
    for arr, grad in ((h, dh), (w, dw)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            fp = _fd_objective_entropy(h, w, lab, g, gh, s, fwd)
            arr[idx] = old - eps
            fm = _fd_objective_entropy(h, w, lab, g, gh, s, fwd)
            arr[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        worst = max(worst, float(np.max(np.abs(num - grad)) / (np.max(np.abs(num)) + 1e-300)))
    return worst


def check_torch_autograd(bwd, seed, s):
    h, w, lab, g = _tiny(seed, T=5, H=16, V=24)
    th = torch.from_numpy(h.astype(np.float64)).requires_grad_(True)
    tw = torch.from_numpy(w.astype(np.float64)).requires_grad_(True)
    z = s * (th @ tw.T)
    lp = torch.log_softmax(z, dim=-1).gather(-1, torch.from_numpy(lab.astype(np.int64)).unsqueeze(-1)).squeeze(-1)
    (lp * torch.from_numpy(g.astype(np.float64))).sum().backward()
    gh, gw = bwd(h, w, lab, g, s)
    return max(float(np.max(np.abs(gh - th.grad.numpy()))), float(np.max(np.abs(gw - tw.grad.numpy()))))


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("s", [1.0, S07])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_blas_form_matches_loop_form(seed, s):
    assert check_loops_forward(oracle.fused_forward, seed, s) < 1e-12
    h, w, lab, g = _tiny(seed, oov_row=2)
    gh, gw = oracle.fused_backward(h, w, lab, g, s)
    rgh, rgw = loops.backward(h.tolist(), w.tolist(), lab.tolist(), g.tolist(), s)
    assert np.max(np.abs(gh - np.array(rgh))) < 1e-12
    assert np.max(np.abs(gw - np.array(rgw))) < 1e-12


@pytest.mark.parametrize("seed", [0, 1])
def test_sampler_formula_matches_torch_log_softmax_gather(seed):
    assert check_torch_log_softmax(oracle.sampler_logprob, seed) < 1e-12


@pytest.mark.parametrize("seed", [0, 1])
def test_lse_and_entropy_match_scipy(seed):
    assert check_scipy_lse_entropy(oracle.sampler_logprob, seed) < 1e-11


def test_uniform_rows_closed_form():
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        cases = json.load(f)["uniform"]
    for c in cases:
        V = c["V"]
        h = np.ones((2, 8), dtype=np.float32)
        w = np.zeros((V, 8), dtype=np.float32)  # weight 0 => every logit 0
        lp, ent, _ = oracle.fused_forward(h, w, np.array([0, V - 1]), 1.0)
        assert np.allclose(lp, c["logprob"], atol=1e-12, rtol=0)
        assert np.allclose(ent, c["entropy"], atol=1e-12, rtol=0)


@pytest.mark.parametrize("V,k,a,b", [(16, 1, 3.0, -1.0), (4096, 7, 5.5, 0.25),
                                     (32000, 31999, -2.0, 9.0), (1000, 500, 0.0, 0.0)])
def test_two_value_rows_closed_form(V, k, a, b):
    assert check_two_value(oracle.sampler_logprob, V, k, a, b) < 1e-11


def test_one_hot_dominant_row():
    rng = np.random.default_rng(5)
    T, H, V = 4, 64, 4096
    hidden = rng.standard_normal((T, H))
    weight = 1e-3 * rng.standard_normal((V, H))
    labels = rng.integers(0, V, size=T)
    for t in range(T):
        weight[labels[t]] = 50.0 * hidden[t] / np.dot(hidden[t], hidden[t])
    # rows share W, so make each label row dominant only for its own token
    for t in range(T):
        lp, ent, _ = oracle.fused_forward(hidden[t:t + 1], weight, labels[t:t + 1], 1.0)
        assert -1e-6 < lp[0] <= 0.0
        assert 0.0 <= ent[0] < 1e-6 + 1e-3  # other label rows give at most a small tail
    # a single dominant row alone: both vanish
    w1 = 1e-3 * rng.standard_normal((V, H))
    w1[3] = 50.0 * hidden[0] / np.dot(hidden[0], hidden[0])
    lp, ent, _ = oracle.fused_forward(hidden[:1], w1, np.array([3]), 1.0)
    assert abs(lp[0]) < 1e-6 and 0.0 <= ent[0] < 1e-6


def test_probabilities_sum_to_one_and_bounds():
    rng = np.random.default_rng(7)
    V = 2000
    z = 2.0 * rng.standard_normal((3, V)) + rng.standard_normal((3, 1))
    for r in range(3):
        zz = np.repeat(z[r:r + 1], V, axis=0)
        lp, ent, _ = oracle.sampler_logprob(zz, np.arange(V))
        assert abs(np.sum(np.exp(lp)) - 1.0) < 1e-12
        assert np.all(lp <= 0.0)
        assert 0.0 <= ent[0] <= math.log(V)


@pytest.mark.parametrize("s", [1.0, S07])
def test_finite_differences_in_vocab(s):
    assert check_finite_differences(oracle.fused_forward, oracle.fused_backward, 11, s) < 1e-6


@pytest.mark.parametrize("s", [1.0, S07])
def test_finite_differences_out_of_vocab(s):
    assert check_finite_differences(oracle.fused_forward, oracle.fused_backward, 12, s, oov_row=0) < 1e-6


@pytest.mark.parametrize("s", [1.0, S07])
def test_torch_autograd_of_sampler_formula(s):
    assert check_torch_autograd(oracle.fused_backward, 13, s) < 1e-12


@pytest.mark.parametrize("s", [1.0, S07])
def test_entropy_gradient_finite_differences(s):
    bwd = lambda h, w, lab, g, s_, gh: oracle.fused_backward(h, w, lab, g, s_, grad_entropy=gh)
    assert check_finite_differences_entropy(oracle.fused_forward, bwd, 14, s, oov_row=1) < 1e-6


def test_entropy_gradient_torch_autograd_and_loops():
    h, w, lab, g = _tiny(15, T=5, H=16, V=24)
    gh = np.random.default_rng(3).standard_normal(5)
    th = torch.from_numpy(h.astype(np.float64)).requires_grad_(True)
    tw = torch.from_numpy(w.astype(np.float64)).requires_grad_(True)
    z = S07 * (th @ tw.T)
    logp = torch.log_softmax(z, dim=-1)
    ent = -(logp.exp() * logp).sum(-1)
    lp = logp.gather(-1, torch.from_numpy(lab.astype(np.int64)).unsqueeze(-1)).squeeze(-1)
    (lp * torch.from_numpy(g.astype(np.float64)) + ent * torch.from_numpy(gh)).sum().backward()
    dh, dw = oracle.fused_backward(h, w, lab, g, S07, grad_entropy=gh)
    assert np.max(np.abs(dh - th.grad.numpy())) < 1e-12
    assert np.max(np.abs(dw - tw.grad.numpy())) < 1e-12
    rdh, rdw = loops.backward(h.tolist(), w.tolist(), lab.tolist(), g.tolist(), S07, gh.tolist())
    assert np.max(np.abs(dh - np.array(rdh))) < 1e-12
    assert np.max(np.abs(dw - np.array(rdw))) < 1e-12


def test_entropy_gradient_row_sums_vanish():
    h, w, lab, _ = _tiny(16, T=4, H=8, V=32)
    z = oracle.scaled_logits(h, w, S07)
    d = oracle.dlogits_entropy(z, np.array([1.0, -2.0, 0.5, 3.0]), S07)
    assert np.all(np.abs(d.sum(axis=1)) < 1e-12)  # sum_j p_j (z_j - lse + H) = 0


def test_sum_p2_closed_forms_library_and_bounds():
    # uniform row: 1/V; two-value row: k pa^2 + (V-k) pb^2; dominant row: ~1
    for V in (16, 4096):
        assert abs(oracle.row_sum_p2(np.zeros((1, V)))[0] - 1.0 / V) < 1e-15
    V, k, a, b = 4096, 7, 5.5, 0.25
    z = np.full((1, V), b)
    z[0, :k] = a
    zs = k * math.exp(a) + (V - k) * math.exp(b)
    ref = k * (math.exp(a) / zs) ** 2 + (V - k) * (math.exp(b) / zs) ** 2
    assert abs(oracle.row_sum_p2(z)[0] - ref) < 1e-14
    z = np.zeros((1, 100))
    z[0, 3] = 60.0
    assert abs(oracle.row_sum_p2(z)[0] - 1.0) < 1e-20 + 1e-12
    rng = np.random.default_rng(17)
    z = 3.0 * rng.standard_normal((12, 777)) + 500.0
    sp = scipy.special.softmax(z, axis=1)
    got = oracle.row_sum_p2(z)
    assert np.max(np.abs(got - (sp ** 2).sum(axis=1))) < 1e-12
    _, ent, _ = oracle.sampler_logprob(z, np.zeros(12, dtype=np.int64))
    assert np.all(got <= sp.max(axis=1) + 1e-15) and np.all(got >= 1.0 / 777)
    assert np.all(got >= np.exp(-ent) - 1e-15)  # Renyi-2 entropy <= Shannon entropy
    h, w, _, _ = _tiny(18)
    ref = loops.sum_p2(h.tolist(), w.tolist(), S07)
    assert np.max(np.abs(oracle.fused_sum_p2(h, w, S07) - np.array(ref))) < 1e-14


def test_dlogit_row_sums():
    h, w, lab, g = _tiny(21, T=4, H=8, V=32, oov_row=3)
    z = oracle.scaled_logits(h, w, S07)
    dl = oracle.dlogits(z, lab, g, S07)
    sums = dl.sum(axis=1)
    assert np.all(np.abs(sums[:3]) < 1e-12)
    assert abs(sums[3] - (-S07 * float(g[3]))) < 1e-12


def test_row_independence_and_sampled_forms():
    h, w, lab, g = _tiny(31, T=40, H=16, V=64, oov_row=5)
    lp, ent, lse = oracle.fused_forward(h, w, lab, S07)
    rows = np.array([39, 0, 5, 17])
    slp, sent, slse = oracle.fused_forward_rows(h, w, lab, S07, rows)
    assert np.max(np.abs(slp - lp[rows])) < 1e-12
    assert np.max(np.abs(sent - ent[rows])) < 1e-12
    for t in rows:  # one row alone gives the value it had inside the batch
        a, b, c = oracle.fused_forward(h[t:t + 1], w, lab[t:t + 1], S07)
        assert abs(a[0] - lp[t]) < 1e-12 and abs(b[0] - ent[t]) < 1e-12
    gh, gw = oracle.fused_backward(h, w, lab, g, S07)
    sgh = oracle.fused_grad_hidden_rows(h, w, lab, g, S07, rows)
    assert np.max(np.abs(sgh - gh[rows])) < 1e-12
    g0 = np.zeros_like(g)
    g0[rows] = g[rows]
    _, gw0 = oracle.fused_backward(h, w, lab, g0, S07)
    assert np.max(np.abs(oracle.grad_weight_from_rows(h, w, lab, g0, S07, rows) - gw0)) < 1e-12
    vr = np.array([3, 0, 63])
    assert np.max(np.abs(oracle.grad_weight_from_rows(h, w, lab, g0, S07, rows, vr) - gw0[vr])) < 1e-12


def test_logits_path_equals_fused_with_identity_weight():
    rng = np.random.default_rng(41)
    T, V = 6, 48
    logits = _bf(2.0 * rng.standard_normal((T, V)))
    lab = rng.integers(0, V, size=T)
    a = oracle.logprob_from_logits(logits, lab, S07)
    b = oracle.fused_forward(logits, np.eye(V), lab, S07)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) < 1e-12


def test_frobenius_identity():
    """<grad_weight, weight> = <grad_hidden, hidden>: both equal sum dlogit * logits."""
    h, w, lab, g = _tiny(51, T=9, H=16, V=40, oov_row=4)
    gh, gw = oracle.fused_backward(h, w, lab, g, S07)
    lhs = float(np.sum(gw * w))
    rhs = float(np.sum(gh * h))
    assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(lhs))


def test_temperature_order_policy():
    """Mirror of the page's temperature experiment on a smaller grid."""
    with open(os.path.join(GOLDEN, "temperature_order.json")) as f:
        gold = json.load(f)
    rng = np.random.default_rng(61)
    rows, V = 64, 32000
    logits = _bf(2.0 * rng.standard_normal((rows, V)) + rng.standard_normal((rows, 1)))
    lab = rng.integers(0, V, size=rows)
    for c in gold["cases"]:
        T = c["temperature"]
        tb = float(W.bf16_bits_to_f32(W.f32_to_bf16_bits(np.array([T], np.float32)))[0])
        assert tb == c["bf16_temperature"]
        # bf16 path: divide bf16 logits by the bf16 temperature, result rounded to bf16
        z_bf16 = _bf(logits.astype(np.float32) / np.float32(tb))
        lp_bf16, _, _ = oracle.logprob_from_logits(z_bf16, lab, 1.0)
        # policy: fp32 logits scaled by the fp32 factor
        lp_fp32, _, _ = oracle.logprob_from_logits(logits, lab, 1.0 / T)
        lp_fp32_again, _, _ = oracle.logprob_from_logits(logits, lab, 1.0 / T)
        mism = int(np.sum(lp_bf16 != lp_fp32))
        expected = rows if c["mismatched_rows"] == gold["rows"] else 0
        assert mism == expected, (T, mism)
        assert np.array_equal(lp_fp32, lp_fp32_again)


# ---------------------------------------------------------------------------
# sampler-parity form: z = fp32(logits) / fp32(t)
# ---------------------------------------------------------------------------

def check_division_rounding(divide, seed, n=300):
    """Number of quotients that are not the round-to-nearest fp32 value of x / t.

    Exact rational arithmetic: z is the nearest fp32 value to the rational
    x / t when neither fp32 neighbour of z is strictly closer to it.
    """
    rng = np.random.default_rng(seed)
    x = _bf(4.0 * rng.standard_normal((1, n)))
    t = np.float32(rng.uniform(0.3, 1.7))
    z = np.asarray(divide(x, t), dtype=np.float64)[0]
    bad = 0
    for xi, zi in zip(x[0], z):
        zf = np.float32(zi)
        if float(zf) != zi:
            bad += 1
            continue
        exact = Fraction(float(xi)) / Fraction(float(t))
        d = abs(Fraction(float(zf)) - exact)
        for nb in (np.nextafter(zf, np.float32(-np.inf)), np.nextafter(zf, np.float32(np.inf))):
            if abs(Fraction(float(nb)) - exact) < d:
                bad += 1
                break
    return bad


def test_division_is_round_to_nearest_fp32():
    for seed in range(3):
        assert check_division_rounding(oracle.divided_logits, seed) == 0


def test_division_form_matches_torch_fp32_division_and_log_softmax():
    rng = np.random.default_rng(71)
    rows, V = 6, 3000
    logits = _bf(2.0 * rng.standard_normal((rows, V)))
    lab = rng.integers(0, V, size=rows)
    lab[2] = -100
    temps = rng.uniform(0.5, 1.5, size=rows).astype(np.float32)
    # torch's fp32 tensor division, then the sampler formula in float64
    zt = torch.from_numpy(logits.astype(np.float32)) / torch.from_numpy(temps)[:, None]
    assert np.array_equal(zt.numpy().astype(np.float64), oracle.divided_logits(logits, temps))
    lsm = torch.log_softmax(zt.double(), dim=-1)
    want = lsm.gather(1, torch.from_numpy(np.where(lab < 0, 0, lab))[:, None])[:, 0].numpy()
    want[2] = 0.0
    lp, ent, lse = oracle.logprob_from_logits_div(logits, lab, temps)
    assert np.max(np.abs(lp - want)) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(zt.double(), dim=-1).numpy())) < 1e-12
    # per-row temperatures are row-by-row scalar calls
    for r in range(rows):
        lp_r, ent_r, _ = oracle.logprob_from_logits_div(logits[r:r + 1], lab[r:r + 1], temps[r])
        assert lp_r[0] == lp[r] and ent_r[0] == ent[r]
    # t = 1 divides exactly: the same as the multiplied form with s = 1
    lp1, ent1, _ = oracle.logprob_from_logits_div(logits, lab, 1.0)
    lp1m, ent1m, _ = oracle.logprob_from_logits(logits, lab, 1.0)
    assert np.array_equal(lp1, lp1m) and np.array_equal(ent1, ent1m)
    # the two forms differ only by the last-bit rounding of z
    lpm, _, _ = oracle.logprob_from_logits(logits, lab, 1.0 / 0.7)
    lpd, _, _ = oracle.logprob_from_logits_div(logits, lab, 0.7)
    assert 0 < np.max(np.abs(lpm - lpd)) < 1e-5


def test_temperature_order_policy_division_form():
    """The table's claim for the fp32 division inside a chunk: a row's value
    does not depend on the chunk it is taken in, and the bf16-temperature path
    mismatches every row unless t = 1."""
    with open(os.path.join(GOLDEN, "temperature_order.json")) as f:
        gold = json.load(f)
    rng = np.random.default_rng(62)
    rows, V = 64, 32000
    logits = _bf(2.0 * rng.standard_normal((rows, V)) + rng.standard_normal((rows, 1)))
    lab = rng.integers(0, V, size=rows)
    for c in gold["cases"]:
        T = c["temperature"]
        tb = c["bf16_temperature"]
        z_bf16 = _bf(logits.astype(np.float32) / np.float32(tb))
        lp_bf16, _, _ = oracle.logprob_from_logits(z_bf16, lab, 1.0)
        lp_div, _, _ = oracle.logprob_from_logits_div(logits, lab, T)
        chunks = [oracle.logprob_from_logits_div(logits[i:i + 8], lab[i:i + 8], T)[0]
                  for i in range(0, rows, 8)]
        assert np.array_equal(np.concatenate(chunks), lp_div)
        expected = rows if c["mismatched_rows"] == gold["rows"] else 0
        assert int(np.sum(lp_bf16 != lp_div)) == expected, T


# ---------------------------------------------------------------------------
# planted mistakes: each pin must reject a plausible error in the oracle
# ---------------------------------------------------------------------------

def _sampler_entropy_missing_lse(z, labels):
    lp, _, lse = oracle.sampler_logprob(z, labels)
    z = np.asarray(z, np.float64)
    p = np.exp(z - lse[:, None])
    return lp, -(p * z).sum(axis=1), lse  # dropped "+ lse" term


def _sampler_no_max_shift(z, labels):
    z = np.asarray(z, np.float64)
    lse = np.log(np.exp(z).sum(axis=1))  # overflows for large logits
    lp = z[np.arange(len(z)), labels] - lse
    p = np.exp(z - lse[:, None])
    return lp, -(p * (z - lse[:, None])).sum(axis=1), lse


def _backward_sign_flip(h, w, lab, g, s):
    gh, gw = oracle.fused_backward(h, w, lab, g, s)
    return -gh, -gw


def _backward_missing_temperature(h, w, lab, g, s):
    gh, gw = oracle.fused_backward(h, w, lab, g, s)
    return gh / oracle.fp32_scalar(s), gw / oracle.fp32_scalar(s)


def _backward_oov_zeroed(h, w, lab, g, s):
    g = np.where((lab >= 0) & (lab < w.shape[0]), g, 0.0)  # the bug the page fixed
    return oracle.fused_backward(h, w, lab, g, s)


def _forward_transposed_index(h, w, lab, s):
    z = oracle.scaled_logits(h, w, s)
    V = z.shape[1]
    lab2 = (V - 1) - np.asarray(lab)  # wrong label index
    lp, ent, lse = oracle.sampler_logprob(z, np.where((lab >= 0) & (lab < V), lab2, lab))
    return lp, ent, lse


def _backward_entropy_sign_flip(h, w, lab, g, s, gh):
    z = oracle.scaled_logits(h, w, s)
    dl = oracle.dlogits(z, lab, g, s) - oracle.dlogits_entropy(z, gh, s)
    return dl @ np.asarray(w, np.float64), dl.T @ np.asarray(h, np.float64)


def _backward_entropy_missing_h(h, w, lab, g, s, gh):
    z = oracle.scaled_logits(h, w, s)
    lse, _ = oracle.row_lse_entropy(z)
    p = np.exp(z - lse[:, None])
    dz = -np.asarray(gh)[:, None] * p * (z - lse[:, None])  # dropped "+ H"
    dl = oracle.dlogits(z, lab, g, s) + oracle.fp32_scalar(s) * dz
    return dl @ np.asarray(w, np.float64), dl.T @ np.asarray(h, np.float64)


def _sum_p2_unnormalised(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return (e * e).sum(axis=1) / e.sum(axis=1)  # divides by s instead of s^2


def _divide_by_reciprocal(x, t):
    return np.asarray(x, np.float32) * np.float32(1.0 / np.float32(t))  # x * RN(1/t)


def _divide_in_bf16(x, t):
    tb = W.bf16_bits_to_f32(W.f32_to_bf16_bits(np.array([t], np.float32)))[0]
    return np.asarray(x, np.float32) / tb


def test_planted_mistakes_are_caught():
    assert check_division_rounding(_divide_by_reciprocal, 0) > 0
    assert check_division_rounding(_divide_in_bf16, 0) > 0
    assert check_scipy_lse_entropy(_sampler_entropy_missing_lse, 0) > 1e-3
    assert check_two_value(_sampler_entropy_missing_lse, 4096, 7, 5.5, 0.25) > 1e-3
    with np.errstate(over="ignore", invalid="ignore"):
        err = check_scipy_lse_entropy(_sampler_no_max_shift, 0)
    assert not (err < 1e-11)
    assert check_finite_differences(oracle.fused_forward, _backward_sign_flip, 11, 1.0) > 1e-3
    assert check_finite_differences(oracle.fused_forward, _backward_missing_temperature, 11, S07) > 1e-3
    assert check_finite_differences(oracle.fused_forward, _backward_oov_zeroed, 12, 1.0, oov_row=0) > 1e-3
    assert check_loops_forward(_forward_transposed_index, 0, 1.0) > 1e-3
    assert abs(_sum_p2_unnormalised(np.zeros((1, 4096)))[0] - 1.0 / 4096) > 1e-3
    assert check_finite_differences_entropy(oracle.fused_forward, _backward_entropy_sign_flip, 14,
                                            1.0) > 1e-3
    assert check_finite_differences_entropy(oracle.fused_forward, _backward_entropy_missing_h, 14,
                                            S07) > 1e-3

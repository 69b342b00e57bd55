"""GPU parity: the CUDA path through the C ABI against the fp64 oracle,
element by element, on shapes that span several tiles and ragged tails."""

import math

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (ATOL_LOGPROB, RTOL_FROB_GRAD, f64, fused_case, max_abs, rel_frob, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu

S07 = W.f32(1.0 / 0.7)


@pytest.fixture(scope="module")
def lmh():
    import torch

    import invariant_lm_head_gb300 as m

    m.build()
    m.library()
    torch.cuda.set_device(0)
    return m


def _fwd(lmh, hidden, weight, labels, s):
    import torch

    lp, ent, lse = lmh.lmhead_logprob_fwd(to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels),
                                          s, want_lse=True)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    return lp.cpu().numpy(), ent.cpu().numpy(), lse.cpu().numpy()


# ----------------------------------------------------------------- engine
@pytest.mark.parametrize("layout", [0, 1, 2, 3])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (304, 520, 200), (8, 8, 4096), (1000, 264, 72)])
def test_engine_gemm_matches_fp64(lmh, M, N, K, layout):
    """D = A B^T with A [M,K] or [K,M] (bit 0) and B [N,K] or [K,N] (bit 1)."""
    import torch

    a = W.random_bf16(11, (M, K))
    b = W.random_bf16(12, (N, K))
    a_k, b_k = not (layout & 1), not (layout & 2)
    A = to_dev_bf16(a if a_k else np.ascontiguousarray(a.T))
    B = to_dev_bf16(b if b_k else np.ascontiguousarray(b.T))
    d = lmh.lmhead_engine_gemm(A, B, a_kmajor=a_k, b_kmajor=b_k)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    ref = f64(a) @ f64(b).T
    err = np.abs(d.cpu().numpy() - ref) / (np.abs(f64(a)) @ np.abs(f64(b)).T + 1e-30)
    assert float(err.max()) < 1e-5


# ----------------------------------------------------------------- forward
@pytest.mark.parametrize("s", [1.0, S07])
@pytest.mark.parametrize("T,H,V", [(300, 264, 5000), (64, 256, 4096), (1, 8, 16), (129, 512, 1025)])
def test_fused_forward_matches_oracle(lmh, T, H, V, s):
    hidden, weight, labels, _ = fused_case(21, T, H, V, w_std=0.05,
                                           oov=[(0, -100)] if T > 1 else [])
    if T > 3:
        labels[1] = V - 1
        labels[2] = 0
        labels[3] = V + 5
    lp, ent, lse = _fwd(lmh, hidden, weight, labels, s)
    rlp, rent, rlse = oracle.fused_forward(f64(hidden), f64(weight), labels, s)
    assert max_abs(lp, rlp) < ATOL_LOGPROB
    assert max_abs(ent, rent) < ATOL_LOGPROB
    assert max_abs(lse, rlse) < ATOL_LOGPROB
    oov = (labels < 0) | (labels >= V)
    assert np.all(lp[oov] == 0.0)


def test_fused_forward_uniform_closed_form(lmh):
    T, H = 130, 64
    for V in (4096, 32000):
        hidden = W.random_bf16(5, (T, H))
        weight = np.zeros((V, H), dtype=np.uint16)  # bf16 zeros: every logit is 0
        labels = W.random_labels(5, T, V)
        lp, ent, _ = _fwd(lmh, hidden, weight, labels, 1.0)
        assert np.allclose(lp, -math.log(V), atol=ATOL_LOGPROB, rtol=0)
        assert np.allclose(ent, math.log(V), atol=ATOL_LOGPROB, rtol=0)


def test_fused_forward_vocab_of_one(lmh):
    hidden, weight, labels, _ = fused_case(3, 5, 16, 1)
    labels[:] = 0
    labels[4] = 1  # out of vocab
    lp, ent, lse = _fwd(lmh, hidden, weight, labels, 1.0)
    assert np.all(lp == 0.0)
    assert np.allclose(ent, 0.0, atol=1e-6)
    rl = oracle.fused_forward(f64(hidden), f64(weight), labels, 1.0)[2]
    assert max_abs(lse, rl) < ATOL_LOGPROB


def test_fused_forward_large_logits_are_stable(lmh):
    T, H, V = 200, 128, 3000
    hidden, weight, labels, _ = fused_case(9, T, H, V, w_std=0.5)
    s = 40.0  # logits up to about 1000 in magnitude: any missing max shift overflows fp32
    lp, ent, lse = _fwd(lmh, hidden, weight, labels, s)
    rlp, rent, rlse = oracle.fused_forward(f64(hidden), f64(weight), labels, s)
    assert np.max(np.abs(rlse)) > 500.0  # the case does reach the overflow range
    assert np.all(np.isfinite(lp)) and np.all(np.isfinite(ent))
    assert max_abs(lp, rlp) < ATOL_LOGPROB
    assert max_abs(ent, rent) < ATOL_LOGPROB
    assert max_abs(lse, rlse) < ATOL_LOGPROB


def test_nan_row_stays_in_its_row(lmh):
    T, H, V = 40, 64, 2048
    hidden, weight, labels, _ = fused_case(4, T, H, V)
    hidden[17, 3] = 0x7FC0  # bf16 NaN
    lp, ent, _ = _fwd(lmh, hidden, weight, labels, 1.0)
    assert np.isnan(lp[17]) and np.isnan(ent[17])
    keep = np.arange(T) != 17
    assert np.all(np.isfinite(lp[keep]))


def test_empty_batch_is_a_noop(lmh):
    import torch

    d = torch.device("cuda:0")
    h = torch.zeros(0, 64, dtype=torch.bfloat16, device=d)
    w = torch.zeros(100, 64, dtype=torch.bfloat16, device=d)
    lab = torch.zeros(0, dtype=torch.int32, device=d)
    lp, ent, _ = lmh.lmhead_logprob_fwd(h, w, lab, 1.0)
    assert lp.numel() == 0
    gw = torch.full((100, 64), 7.0, device=d)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, torch.zeros(0, device=d), 1.0, grad_weight=gw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(gw).item() == 0


# ----------------------------------------------------------------- backward
def _bwd(lmh, hidden, weight, labels, grad, s, pass_lse=True):
    import torch

    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    lse = None
    if pass_lse:
        _, _, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True, want_entropy=False)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, g, s, lse=lse)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    return gh.float().cpu().numpy(), gw.cpu().numpy()


@pytest.mark.parametrize("pass_lse", [True, False])
@pytest.mark.parametrize("s", [1.0, S07])
@pytest.mark.parametrize("T,H,V", [(300, 264, 5000), (64, 256, 4096), (3, 8, 16), (5, 8, 1),
                                   (9, 16, 7), (130, 24, 1031)])
def test_fused_backward_matches_oracle(lmh, T, H, V, s, pass_lse):
    hidden, weight, labels, grad = fused_case(31, T, H, V, w_std=0.05, oov=[(T - 1, -100)])
    gh, gw = _bwd(lmh, hidden, weight, labels, grad, s, pass_lse)
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, s)
    assert rel_frob(gh, rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw, rgw) < RTOL_FROB_GRAD
    # per-row check of grad_hidden (each row is its own reduction)
    for t in range(T):
        assert rel_frob(gh[t], rgh[t]) < RTOL_FROB_GRAD


def test_fused_backward_several_row_chunks(lmh):
    T, H, V = 16384 + 300, 136, 1500  # two row chunks, ragged second one
    hidden, weight, labels, grad = fused_case(41, T, H, V, w_std=0.1, oov=[(16383, 5000)])
    gh, gw = _bwd(lmh, hidden, weight, labels, grad, S07)
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, S07)
    assert rel_frob(gh, rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw, rgw) < RTOL_FROB_GRAD


def test_fused_backward_all_out_of_vocab(lmh):
    T, H, V = 50, 64, 700
    hidden, weight, labels, grad = fused_case(43, T, H, V)
    labels[:] = -100
    gh, gw = _bwd(lmh, hidden, weight, labels, grad, 1.0)
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, 1.0)
    assert rel_frob(gh, rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw, rgw) < RTOL_FROB_GRAD


@pytest.mark.parametrize("s", [1.0, S07])
@pytest.mark.parametrize("T,H,V", [(300, 264, 5000), (3, 8, 16), (16384 + 40, 72, 700)])
def test_entropy_backward_matches_oracle(lmh, T, H, V, s):
    import torch

    hidden, weight, labels, grad = fused_case(33, T, H, V, w_std=0.2, oov=[(1, -100)])
    gent = W.random_f32(34, T)
    h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
    g, ge = to_dev(grad), to_dev(gent)
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_entropy_bwd(h, w, lab, g, ge, s, lse=lse, entropy=ent)
    gh2, gw2 = lmh.lmhead_logprob_entropy_bwd(h, w, lab, g, ge, s)  # statistics recomputed
    gh3, gw3 = lmh.lmhead_logprob_entropy_bwd(h, w, lab, None, ge, s)  # entropy term alone
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    assert torch.equal(gh, gh2) and torch.equal(gw, gw2)
    h64, w64 = f64(hidden), f64(weight)
    rgh, rgw = oracle.fused_backward(h64, w64, labels, grad, s, grad_entropy=gent)
    assert rel_frob(gh.float().cpu().numpy(), rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw.cpu().numpy(), rgw) < RTOL_FROB_GRAD
    rgh3, rgw3 = oracle.fused_backward(h64, w64, labels, np.zeros(T), s, grad_entropy=gent)
    assert rel_frob(gh3.float().cpu().numpy(), rgh3) < RTOL_FROB_GRAD
    assert rel_frob(gw3.cpu().numpy(), rgw3) < RTOL_FROB_GRAD


def test_entropy_backward_without_entropy_grad_equals_plain_backward(lmh):
    import torch

    T, H, V = 200, 128, 3000
    hidden, weight, labels, grad = fused_case(35, T, H, V)
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    a = lmh.lmhead_logprob_bwd(h, w, lab, g, S07)
    b = lmh.lmhead_logprob_entropy_bwd(h, w, lab, g, None, S07)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# (2048, 1024, 40000): grad_weight runs on wide CTA pairs over 316 units, more
# than four waves, so the odd waves' downward K walk is exercised too.
@pytest.mark.parametrize("T,H,V", [(400, 128, 3000), (2048, 1024, 40000)])
def test_backward_deterministic_run_to_run(lmh, T, H, V):
    import torch

    hidden, weight, labels, grad = fused_case(51, T, H, V)
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    a = lmh.lmhead_logprob_bwd(h, w, lab, g, S07)
    b = lmh.lmhead_logprob_bwd(h, w, lab, g, S07)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ----------------------------------------------------------------- logits path
@pytest.mark.parametrize("s", [1.0, S07])
@pytest.mark.parametrize("T,V", [(300, 5000), (64, 152064), (5, 4999), (3, 1), (130, 8)])
def test_logits_path_matches_oracle(lmh, T, V, s):
    import torch

    wl = W.LOGITS
    inp = W.logits_inputs(wl, T=T, V=V)
    logits, labels = inp["logits"], inp["labels"]
    if T > 2:
        labels[0] = -100
        labels[1] = V - 1
    lp, ent, lse = lmh.logprob_from_logits(to_dev_bf16(logits), to_dev(labels), s, want_lse=True)
    torch.cuda.synchronize()
    rlp, rent, rlse = oracle.logprob_from_logits(f64(logits), labels, s)
    assert max_abs(lp.cpu().numpy(), rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy(), rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy(), rlse) < ATOL_LOGPROB


def test_logits_path_equals_fused_path_on_same_logits(lmh):
    """Fused path with weight = identity sees the same logits as the logits path."""
    import torch

    T, V = 40, 512
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    eye = W.f32_to_bf16_bits(np.eye(V, dtype=np.float32))
    lp1, ent1, _ = lmh.logprob_from_logits(to_dev_bf16(inp["logits"]), to_dev(inp["labels"]), S07)
    lp2, ent2, _ = lmh.lmhead_logprob_fwd(to_dev_bf16(inp["logits"]), to_dev_bf16(eye),
                                          to_dev(inp["labels"]), S07)
    torch.cuda.synchronize()
    assert max_abs(lp1.cpu().numpy(), lp2.cpu().numpy()) < 1e-4
    assert max_abs(ent1.cpu().numpy(), ent2.cpu().numpy()) < 1e-4


# ----------------------------------------------------------------- sum_pi_squared
@pytest.mark.parametrize("s", [1.0, S07])
def test_sum_p2_fused_and_logits_match_oracle(lmh, s):
    import torch

    T, H, V = 300, 264, 5000
    hidden, weight, labels, _ = fused_case(37, T, H, V, w_std=0.2)
    h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
    lp, ent, lse, q = lmh.lmhead_logprob_fwd_stats(h, w, lab, s, want_lse=True)
    lp0, ent0, lse0 = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    torch.cuda.synchronize()
    for a, b in ((lp, lp0), (ent, ent0), (lse, lse0)):  # the extra output changes nothing else
        assert torch.equal(a, b)
    ref = oracle.fused_sum_p2(f64(hidden), f64(weight), s)
    assert max_abs(q.cpu().numpy(), ref) < 1e-5
    inp = W.logits_inputs(W.LOGITS, T=130, V=4999)  # scalar path
    for V_, x in ((4999, inp["logits"]), (5000, W.logits_inputs(W.LOGITS, T=130, V=5000)["logits"])):
        lab2 = to_dev(W.random_labels(3, 130, V_))
        out = lmh.logprob_from_logits_stats(to_dev_bf16(x), lab2, s, want_lse=True)
        base = lmh.logprob_from_logits(to_dev_bf16(x), lab2, s, want_lse=True)
        torch.cuda.synchronize()
        for a, b in zip(out[:3], base):
            assert torch.equal(a, b)
        ref = oracle.row_sum_p2(oracle.fp32_scalar(s) * f64(x))
        assert max_abs(out[3].cpu().numpy(), ref) < 1e-5


def test_sum_p2_uniform_and_dominant_rows(lmh):
    import torch

    T, H, V = 20, 64, 4096
    hidden = W.random_bf16(8, (T, H))
    weight = np.zeros((V, H), dtype=np.uint16)
    q = lmh.lmhead_logprob_fwd_stats(to_dev_bf16(hidden), to_dev_bf16(weight),
                                     to_dev(W.random_labels(8, T, V)), 1.0)[3]
    torch.cuda.synchronize()
    assert np.allclose(q.cpu().numpy(), 1.0 / V, rtol=1e-4, atol=0)


# ----------------------------------------------------------------- status
def test_bounded_wait_selftest_reports_timeout(lmh):
    assert lmh.lmhead_selftest_wait_timeout(2_000_000) == lmh.LMH_ERR_DEVICE_TIMEOUT
    with pytest.raises(lmh.LMHeadError) as e:
        lmh.lmhead_device_status()
    assert e.value.code == lmh.LMH_ERR_DEVICE_TIMEOUT
    assert lmh.lmhead_device_status() == 0  # cleared by the read
    # the context is still usable
    test_engine_gemm_matches_fp64(lmh, 128, 256, 64, 3)


# ----------------------------------------------------------------- sampler-parity (division) form
@pytest.mark.parametrize("T,V", [(300, 5000), (64, 152064), (5, 4999), (3, 1), (130, 8)])
def test_logits_division_form_matches_oracle(lmh, T, V):
    import torch

    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    logits, labels = inp["logits"], inp["labels"]
    if T > 2:
        labels[0] = -100
        labels[1] = V - 1
    temps = np.random.default_rng(T + V).uniform(0.4, 1.6, size=T).astype(np.float32)
    for t in (0.7, temps):
        t_dev = to_dev(temps) if isinstance(t, np.ndarray) else t
        lp, ent, lse, q = lmh.logprob_from_logits_div(to_dev_bf16(logits), to_dev(labels), t_dev,
                                                      want_lse=True, want_sum_p2=True)
        torch.cuda.synchronize()
        rlp, rent, rlse = oracle.logprob_from_logits_div(f64(logits), labels, t)
        assert max_abs(lp.cpu().numpy(), rlp) < ATOL_LOGPROB
        assert max_abs(ent.cpu().numpy(), rent) < ATOL_LOGPROB
        assert max_abs(lse.cpu().numpy(), rlse) < ATOL_LOGPROB
        rq = oracle.row_sum_p2(oracle.divided_logits(f64(logits), t))
        assert max_abs(q.cpu().numpy(), rq) < 1e-5


def test_logits_division_per_row_temperature_equals_scalar_calls(lmh):
    """A row's outputs with a per-row temperature array are bit-identical to a
    call with that row's temperature as the scalar, and the optional outputs
    change nothing else."""
    import torch

    T, V = 12, 5000
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    temps = np.random.default_rng(5).uniform(0.3, 2.0, size=T).astype(np.float32)
    full = lmh.logprob_from_logits_div(x, lab, to_dev(temps), want_lse=True, want_sum_p2=True)
    plain = lmh.logprob_from_logits_div(x, lab, to_dev(temps), want_lse=True)
    for r in range(T):
        one = lmh.logprob_from_logits_div(x[r:r + 1], lab[r:r + 1], float(temps[r]), want_lse=True,
                                          want_sum_p2=True)
        for a, b in zip(one, full):
            assert torch.equal(a.view(torch.int32), b[r:r + 1].view(torch.int32))
    for a, b in zip(plain[:3], full[:3]):
        assert torch.equal(a, b)
    torch.cuda.synchronize()


def test_logits_division_bad_row_temperature_is_nan_in_that_row_only(lmh):
    import torch

    T, V = 6, 4096
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    temps = np.array([0.7, 0.0, 0.9, -1.0, float("inf"), 1.1], dtype=np.float32)
    lp, ent, _, _ = lmh.logprob_from_logits_div(x, lab, to_dev(temps))
    torch.cuda.synchronize()
    lp, ent = lp.cpu().numpy(), ent.cpu().numpy()
    bad = np.array([False, True, False, True, True, False])
    assert np.all(np.isnan(lp[bad])) and np.all(np.isnan(ent[bad]))
    assert np.all(np.isfinite(lp[~bad])) and np.all(np.isfinite(ent[~bad]))
    rlp, _, _ = oracle.logprob_from_logits_div(f64(inp["logits"][~bad]), inp["labels"][~bad],
                                               temps[~bad])
    assert max_abs(lp[~bad], rlp) < ATOL_LOGPROB


@pytest.mark.parametrize("V", [5000, 4999])
def test_logits_division_by_a_power_of_two_is_the_multiplied_form_bit_for_bit(lmh, V):
    """For t = 2^k, z = x / t is exact and z * log2(e) is the same real number
    as x * (log2(e) / t), so every shifted value, and every output, must carry
    the bits of the multiplied form with s = 1/t. The rows mix in what the
    division's fast path treats apart: exact zeros of both signs, bf16
    subnormals, tiny normals (|x| < 2^-100), huge values (2^110), a row of
    tiny values only (its maximum is tiny too), a row of zeros, rows with -inf
    entries (a masked sampler's logits), a row of huge negative values only,
    and a row holding +inf. NaN outputs (entropy where a -inf logit makes
    p * log p = 0 * -inf, every output of the +inf row) must be NaN in both."""
    import torch

    T = 11
    rng = np.random.default_rng(V)
    x = rng.normal(0.0, 2.0, size=(T, V)).astype(np.float32)
    x[0, rng.choice(V, V // 3, replace=False)] = 0.0
    x[0, rng.choice(V, V // 8, replace=False)] = -0.0
    sub = rng.choice(V, V // 8, replace=False)
    x[1, sub] = np.float32(2.0 ** -130) * rng.integers(1, 100, size=sub.size)  # bf16 subnormals
    tiny = rng.choice(V, V // 4, replace=False)
    x[1, tiny] = np.float32(2.0 ** -110) * rng.normal(size=tiny.size).astype(np.float32)
    x[2] = np.float32(2.0 ** -105) * rng.normal(size=V).astype(np.float32)  # tiny maximum
    x[3] = 0.0
    x[4, rng.choice(V, 5, replace=False)] = np.float32(2.0 ** 110)
    x[5, :3] = -np.float32(2.0 ** 110)
    x[6, rng.choice(V, V // 3, replace=False)] = -np.inf
    x[7] = -np.float32(2.0 ** 101) * (1.0 + rng.random(V).astype(np.float32))  # all huge negative
    x[8, 7] = np.inf
    x[9, :40] = -np.inf
    bits = W.f32_to_bf16_bits(x)
    labels = W.random_labels(3, T, V)
    xd, lab = to_dev_bf16(bits), to_dev(labels)
    for t in (2.0, 0.5, 0.25, 1.0):
        div = lmh.logprob_from_logits_div(xd, lab, t, want_lse=True, want_sum_p2=True)
        mul = lmh.logprob_from_logits_stats(xd, lab, 1.0 / t, want_lse=True)
        torch.cuda.synchronize()
        for a, b, name in zip(div, mul, ("logprob", "entropy", "lse", "sum_p2")):
            same = (a.view(torch.int32) == b.view(torch.int32)) | (torch.isnan(a) & torch.isnan(b))
            assert bool(same.all()), f"{name} at t={t}: division and multiplication differ"
        # -inf logits (a masked sampler's) leave logprob finite. The huge rows
        # (|z| >= 2^100) are outside the range the statistics hold finite
        # (|z| < 2^30, include/lmhead.h); only their bits are compared above.
        assert torch.isfinite(div[0][[0, 1, 2, 3, 6, 9, 10]]).all()


def test_logits_division_against_torch_sampler_formula(lmh):
    """Against torch's own fp32 sampler formula on the GPU (log_softmax of the
    fp32 logits divided by a per-row temperature tensor, then gather): the
    same z, reduced in another order, so equal to within a few fp32 ulps of
    the log-probs, not bit for bit."""
    import torch

    T, V = 64, 152064
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    temps = torch.full((T,), 0.7, dtype=torch.float32, device=x.device)
    lp, _, _, _ = lmh.logprob_from_logits_div(x, lab, temps)
    ref = torch.log_softmax(x.float() / temps[:, None], dim=-1).gather(1, lab.long()[:, None])[:, 0]
    torch.cuda.synchronize()
    assert float((lp - ref).abs().max()) < 1e-4


# ----------------------------------------------------------------- forward from host memory
@pytest.mark.parametrize("T,H,V", [(300, 264, 5000), (64, 128, 152064), (7, 64, 1000), (5, 8, 1)])
def test_forward_from_host_is_bitwise_the_device_forward(lmh, T, H, V):
    """The staged forward (host copies overlapped with per-slice launches)
    fills the device inputs and gives the device forward's exact bits."""
    import torch

    hidden, weight, labels, _ = fused_case(41, T, H, V, w_std=0.2, oov=((0, -100),) if T > 1 else ())
    h_host = W.as_torch_bf16(hidden).pin_memory()
    w_host = W.as_torch_bf16(weight).pin_memory()
    l_host = torch.from_numpy(labels).pin_memory()
    dev = torch.device("cuda:0")
    h = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    w = torch.empty(V, H, dtype=torch.bfloat16, device=dev)
    lab = torch.empty(T, dtype=torch.int32, device=dev)
    lp_host = torch.empty(T, dtype=torch.float32).pin_memory()
    ent_host = torch.empty(T, dtype=torch.float32).pin_memory()
    for copy_stream in (None, torch.cuda.Stream()):
        lp, ent, lse = lmh.lmhead_logprob_fwd_host(h_host, w_host, l_host, S07, hidden=h, weight=w,
                                                   labels=lab, out_logprob_host=lp_host,
                                                   out_entropy_host=ent_host,
                                                   copy_stream=copy_stream)
        torch.cuda.synchronize()
        assert torch.equal(h.cpu(), h_host) and torch.equal(w.cpu(), w_host)
        assert torch.equal(lab.cpu(), l_host)
        rlp, rent, rlse = lmh.lmhead_logprob_fwd(to_dev_bf16(hidden), to_dev_bf16(weight),
                                                 to_dev(labels), S07, want_lse=True)
        torch.cuda.synchronize()
        for a, b in ((lp, rlp), (ent, rent), (lse, rlse)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(lp_host, lp.cpu()) and torch.equal(ent_host, ent.cpu())
        lmh.lmhead_device_status()
        h.zero_(), w.zero_(), lab.zero_()


def test_division_form_is_ieee_division_for_every_bf16_input(lmh):
    """The quotient the division form uses, for all 65536 bf16 inputs, equals
    IEEE fp32 division bit for bit: at the pages' temperatures, at temperatures
    whose significand is all ones or a power of two, at random ones across
    the fast path's range, and at extreme or invalid ones (IEEE path)."""
    rng = np.random.default_rng(123)
    ts = [0.7, 0.9, 0.6, 1.0, 0.8984375, 0.69921875, 0.6015625, 2.0, 0.5,
          float(np.nextafter(np.float32(1.0), np.float32(2.0))),
          float(np.nextafter(np.float32(2.0), np.float32(1.0))),
          float(np.nextafter(np.float32(1.0), np.float32(0.0))),
          2.0 ** -20, 2.0 ** 20, 2.0 ** -21, 3.0e6, 1e-30, 1e30, 0.0, -1.0,
          float("inf"), float("nan")]
    ts += [float(np.float32(v)) for v in np.exp(rng.uniform(np.log(2.0 ** -20), np.log(2.0 ** 20),
                                                            size=300))]
    ts += [float(np.uint32((127 << 23) | int(m)).view(np.float32)) for m in
           rng.integers(0, 1 << 23, size=300)]
    bad = {t: n for t in ts if (n := lmh.lmhead_selftest_division(t)) != 0}
    assert not bad, bad


# ----------------------------------------------------------------- autograd wrapper
@pytest.mark.parametrize("use_entropy", [False, True])
def test_autograd_wrapper_matches_the_direct_calls(lmh, use_entropy):
    """loss.backward() through lmhead_logprob runs the library's backward:
    the same bits as calling it directly, and within tolerance of the oracle."""
    import torch

    T, H, V = 300, 264, 5000
    hidden, weight, labels, grad = fused_case(61, T, H, V, w_std=0.2, oov=((2, -100),))
    g_ent = W.random_f32(62, T)
    h = to_dev_bf16(hidden).requires_grad_(True)
    w = to_dev_bf16(weight).requires_grad_(True)
    lab, g, ge = to_dev(labels), to_dev(grad), to_dev(g_ent)
    lp, ent = lmh.lmhead_logprob(h, w, lab, S07)
    loss = (lp * g).sum() + ((ent * ge).sum() if use_entropy else 0.0)
    loss.backward()
    torch.cuda.synchronize()
    with torch.no_grad():
        lp0, ent0, lse0 = lmh.lmhead_logprob_fwd(h.detach(), w.detach(), lab, S07, want_lse=True)
        if use_entropy:
            gh0, gw0 = lmh.lmhead_logprob_entropy_bwd(h.detach(), w.detach(), lab, g, ge, S07,
                                                      lse=lse0, entropy=ent0)
        else:
            gh0, gw0 = lmh.lmhead_logprob_bwd(h.detach(), w.detach(), lab, g, S07, lse=lse0)
    torch.cuda.synchronize()
    assert torch.equal(lp.detach(), lp0) and torch.equal(ent.detach(), ent0)
    assert torch.equal(h.grad, gh0)
    assert torch.equal(w.grad, gw0.to(torch.bfloat16))
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, S07,
                                     grad_entropy=g_ent if use_entropy else None)
    assert rel_frob(h.grad.float().cpu().numpy(), rgh) < RTOL_FROB_GRAD
    assert rel_frob(w.grad.float().cpu().numpy(), rgw) < RTOL_FROB_GRAD


# ----------------------------------------------------------------- chunk coverage, poisoned outputs
@pytest.mark.parametrize("T", [127, 128, 129, 257, 16383, 16385])
def test_every_output_element_is_written(lmh, T):
    """Output buffers filled with NaN beforehand: every element of every output
    must be written (finite) and match the oracle, for T at and around
    multiples of the 128-row tile and the 16384-row backward chunk, and prime T."""
    import torch

    H, V = 64, 1000
    hidden, weight, labels, grad = fused_case(71, T, H, V, w_std=0.2, oov=((T // 2, -100),))
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    dev = h.device
    nan = float("nan")
    lp, ent, lse, q = (torch.full((T,), nan, device=dev) for _ in range(4))
    gh = torch.full((T, H), nan, dtype=torch.bfloat16, device=dev)
    gw = torch.full((V, H), nan, device=dev)
    lmh.lmhead_logprob_fwd_stats(h, w, lab, S07, out_logprob=lp, out_entropy=ent, out_lse=lse,
                                 out_sum_p2=q)
    lmh.lmhead_logprob_bwd(h, w, lab, g, S07, lse=lse, grad_hidden=gh, grad_weight=gw)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    for t in (lp, ent, lse, q, gh.float(), gw):
        assert bool(torch.isfinite(t).all())
    rlp, rent, rlse = oracle.fused_forward(f64(hidden), f64(weight), labels, S07)
    assert max_abs(lp.cpu().numpy(), rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy(), rent) < ATOL_LOGPROB
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, S07)
    assert rel_frob(gh.float().cpu().numpy(), rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw.cpu().numpy(), rgw) < RTOL_FROB_GRAD
    # the logits path and its division form into poisoned buffers
    x = to_dev_bf16(W.f32_to_bf16_bits((f64(hidden) @ f64(weight).T).astype(np.float32)))
    for fill in (lp, ent, lse, q):
        fill.fill_(nan)
    lmh.logprob_from_logits_stats(x, lab, S07, out_logprob=lp, out_entropy=ent, out_lse=lse,
                                  out_sum_p2=q)
    torch.cuda.synchronize()
    for t in (lp, ent, lse, q):
        assert bool(torch.isfinite(t).all())
    for fill in (lp, ent, lse, q):
        fill.fill_(nan)
    lmh.logprob_from_logits_div(x, lab, 0.7, out_logprob=lp, out_entropy=ent, out_lse=lse,
                                out_sum_p2=q)
    torch.cuda.synchronize()
    for t in (lp, ent, lse, q):
        assert bool(torch.isfinite(t).all())


# ----------------------------------------------------------------- vocab shards
@pytest.mark.parametrize("T,H,V,cuts", [(300, 264, 5000, (2048, 4096)), (64, 128, 152064, (65536,)),
                                        (7, 64, 3072, (1024, 2048)), (130, 8, 1025, (1024,))])
def test_vocab_shards_merge_to_the_whole_forward(lmh, T, H, V, cuts):
    """Shards of the weight (cut at 1024-column boundaries) computed separately,
    their label logits summed as ranks would all-reduce them, and merged: the
    whole forward's bits."""
    import torch

    hidden, weight, labels, _ = fused_case(81, T, H, V, w_std=0.2, oov=((0, -100),))
    h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
    dev = h.device
    n = -(-V // 1024)
    pm, ps, pu = (torch.full((n, T), float("nan"), device=dev) for _ in range(3))
    zl = torch.zeros(T, device=dev)
    bounds = [0, *cuts, V]
    for a, b in zip(bounds[:-1], bounds[1:]):
        c0, c1 = a // 1024, -(-b // 1024)
        part = torch.full((T,), float("nan"), device=dev)
        lmh.lmhead_logprob_fwd_partials(h, w[a:b].contiguous(), lab, a, S07, part_m=pm[c0:c1],
                                        part_s=ps[c0:c1], part_u=pu[c0:c1], label_logit=part)
        zl += part  # one shard holds each row's label; the others contribute 0
    lp, ent, lse = lmh.lmhead_logprob_merge(pm, ps, pu, zl, lab, V)
    ref = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    torch.cuda.synchronize()
    for x, y in zip((lp, ent, lse), ref):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))

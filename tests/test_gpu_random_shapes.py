"""Seeded random shapes through every entry point, against the oracle: ragged
T, H and V (tails of every tile size), random out-of-vocab labels and
temperatures, and a sub-batch of each case checked for bit-identity. A second
set spans 700 to 2600 rows, across the 1024-row chunks up to which the
backward runs grad_hidden beside grad_weight (and picks other engines)."""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import ATOL_LOGPROB, RTOL_FROB_GRAD, f64, fused_case, max_abs, rel_frob, to_dev, \
    to_dev_bf16

pytestmark = pytest.mark.gpu


def _shapes(n=16, seed=77, t_lo=1, t_hi=700):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        T = int(rng.integers(t_lo, t_hi))
        H = 8 * int(rng.integers(1, 80))
        V = int(rng.integers(1, 6000))
        s = float(np.float32(rng.uniform(0.5, 2.0)))
        out.append((T, H, V, s))
    return out


@pytest.fixture(scope="module")
def lmh():
    import torch

    import invariant_lm_head_gb300 as m

    m.build()
    m.library()
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("T,H,V,s", _shapes() + _shapes(n=8, seed=78, t_lo=700, t_hi=2600))
def test_random_shape_all_paths(lmh, T, H, V, s):
    import torch

    seed = T * 7919 + H * 31 + V
    rng = np.random.default_rng(seed)
    oov = [(int(i), -100) for i in rng.choice(T, size=min(T, 3), replace=False)]
    hidden, weight, labels, grad = fused_case(seed % 100000, T, H, V, w_std=0.1, oov=oov)
    g_ent = W.random_f32(seed % 100000 + 1, T)
    h, w, lab, g, ge = (to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad),
                        to_dev(g_ent))
    h64, w64 = f64(hidden), f64(weight)

    # fused forward and both backward forms
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, g, s, lse=lse)
    ghe, gwe = lmh.lmhead_logprob_entropy_bwd(h, w, lab, g, ge, s, lse=lse, entropy=ent)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    rlp, rent, rlse = oracle.fused_forward(h64, w64, labels, s)
    assert max_abs(lp.cpu().numpy(), rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy(), rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy(), rlse) < ATOL_LOGPROB
    rgh, rgw = oracle.fused_backward(h64, w64, labels, grad, s)
    assert rel_frob(gh.float().cpu().numpy(), rgh) < RTOL_FROB_GRAD
    assert rel_frob(gw.cpu().numpy(), rgw) < RTOL_FROB_GRAD
    rghe, rgwe = oracle.fused_backward(h64, w64, labels, grad, s, grad_entropy=g_ent)
    assert rel_frob(ghe.float().cpu().numpy(), rghe) < RTOL_FROB_GRAD
    assert rel_frob(gwe.cpu().numpy(), rgwe) < RTOL_FROB_GRAD

    # a sub-batch gives the same bits
    a = int(rng.integers(0, T))
    b = int(rng.integers(a + 1, T + 1))
    part = lmh.lmhead_logprob_fwd(h[a:b], w, lab[a:b], s, want_lse=True)
    for x, y in zip(part, (lp, ent, lse)):
        assert torch.equal(x.view(torch.int32), y[a:b].view(torch.int32))

    # the same logits materialised: multiplied and divided forms
    logits_bits = W.f32_to_bf16_bits((h64 @ w64.T).astype(np.float32))
    x = to_dev_bf16(logits_bits)
    llp, lent, _ = lmh.logprob_from_logits(x, lab, s)
    temps = rng.uniform(0.5, 1.5, size=T).astype(np.float32)
    dlp, dent, _, _ = lmh.logprob_from_logits_div(x, lab, to_dev(temps))
    torch.cuda.synchronize()
    xl = f64(logits_bits)
    rllp, rlent, _ = oracle.logprob_from_logits(xl, labels, s)
    rdlp, rdent, _ = oracle.logprob_from_logits_div(xl, labels, temps)
    assert max_abs(llp.cpu().numpy(), rllp) < ATOL_LOGPROB
    assert max_abs(lent.cpu().numpy(), rlent) < ATOL_LOGPROB
    assert max_abs(dlp.cpu().numpy(), rdlp) < ATOL_LOGPROB
    assert max_abs(dent.cpu().numpy(), rdent) < ATOL_LOGPROB

    # the staged forward from host memory gives the device forward's bits
    hh = W.as_torch_bf16(hidden).pin_memory()
    wh = W.as_torch_bf16(weight).pin_memory()
    lh = torch.from_numpy(labels).pin_memory()
    hd, wd, ld = torch.empty_like(h), torch.empty_like(w), torch.empty_like(lab)
    sp, se, sl = lmh.lmhead_logprob_fwd_host(hh, wh, lh, s, hidden=hd, weight=wd, labels=ld)
    torch.cuda.synchronize()
    for x_, y_ in zip((sp, se, sl), (lp, ent, lse)):
        assert torch.equal(x_.view(torch.int32), y_.view(torch.int32))

"""The backward with a caller-chosen row chunk (lmhead_logprob_bwd_chunked).

The SkyRL page's streaming backward tests compare chunked and single-shot
gradients over several chunk sizes, ragged last chunks included. Here each row's
dlogits and its K = V walk do not depend on the chunk, so grad_hidden must keep
its bits for every chunk; grad_weight sums the chunks in ascending order, so it
must be run-to-run identical for a given chunk and within the suite's 1e-2 of
the fp64 oracle for every chunk. Output buffers are NaN-poisoned first, so an
element that no chunk writes shows up.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import RTOL_FROB_GRAD, f64, fused_case, rel_frob, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

S07 = W.f32(1.0 / 0.7)


@pytest.fixture(scope="module")
def lmh():
    import torch

    import invariant_lm_head_gb300 as m

    m.build()
    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("use_entropy", [False, True])
@pytest.mark.parametrize("T,H,V", [(1000, 264, 3001), (257, 128, 1025)])
def test_row_chunk_keeps_grad_hidden_bits(lmh, T, H, V, use_entropy):
    import torch

    hidden, weight, labels, grad = fused_case(81, T, H, V, w_std=0.1, oov=((3, -100),))
    g_ent = W.random_f32(82, T)
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    ge = to_dev(g_ent) if use_entropy else None
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    rgh, rgw = oracle.fused_backward(f64(hidden), f64(weight), labels, grad, S07,
                                     grad_entropy=g_ent if use_entropy else None)
    ref_gh = None
    for chunk in (16384, 128, 384, 4096):
        gws = []
        for _ in range(2):  # run to run
            gh = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=h.device)
            gw = torch.full((V, H), float("nan"), dtype=torch.float32, device=h.device)
            lmh.lmhead_logprob_bwd_chunked(h, w, lab, g, S07, row_chunk=chunk, grad_entropy=ge,
                                           lse=lse, entropy=ent if use_entropy else None,
                                           grad_hidden=gh, grad_weight=gw)
            torch.cuda.synchronize()
            assert lmh.lmhead_device_status() == 0
            assert bool(torch.isfinite(gh.float()).all()) and bool(torch.isfinite(gw).all())
            gws.append(gw.clone())
            if ref_gh is None:
                ref_gh = gh.clone()
            assert torch.equal(gh.view(torch.int16), ref_gh.view(torch.int16)), \
                f"grad_hidden changed its bits with row_chunk={chunk}"
        assert torch.equal(gws[0].view(torch.int32), gws[1].view(torch.int32)), \
            f"grad_weight differs run to run with row_chunk={chunk}"
        assert rel_frob(gws[0].cpu().numpy(), rgw) < RTOL_FROB_GRAD
    assert rel_frob(ref_gh.float().cpu().numpy(), rgh) < RTOL_FROB_GRAD


def test_row_chunk_equal_to_the_default_backward(lmh):
    """row_chunk = 16384 is the plain backward, bit for bit."""
    import torch

    T, H, V = 700, 136, 2000
    hidden, weight, labels, grad = fused_case(83, T, H, V, w_std=0.1)
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    _, _, lse = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    a = lmh.lmhead_logprob_bwd(h, w, lab, g, S07, lse=lse)
    b = lmh.lmhead_logprob_bwd_chunked(h, w, lab, g, S07, row_chunk=16384, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    ws_small = lmh.lmhead_workspace_size_bwd(T, H, V, 128)
    ws_full = lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, T, H, V)
    assert ws_small < ws_full

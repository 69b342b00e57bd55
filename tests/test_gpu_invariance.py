"""Batch invariance on the GPU: a row's log-prob, entropy, lse and grad_hidden
row are bit-identical whatever batch size, offset, chunk or packing it comes
in. The oracle plays no part here; the comparison is GPU against GPU, in the
fp32 (or bf16) bits of the outputs."""

import pytest

import workloads as W
from helpers import fused_case, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

S07 = W.f32(1.0 / 0.7)


@pytest.fixture(scope="module")
def lmh():
    import torch

    import invariant_lm_head_gb300 as m

    m.build()
    torch.cuda.set_device(0)
    return m


def _fwd_all(lmh, h, w, lab, s):
    import torch

    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    torch.cuda.synchronize()
    return lp, ent, lse


def _mismatch(a, b):
    """Number of fp32 outputs whose bits differ."""
    import torch

    return int((a.view(torch.int32) != b.view(torch.int32)).sum().item())


@pytest.mark.parametrize("T,H,V,s", [(64, 256, 4096, 1.0), (300, 264, 5000, S07)])
def test_forward_sub_batches_offsets_and_shuffles(lmh, T, H, V, s):
    import torch

    hidden, weight, labels, _ = fused_case(61, T, H, V, oov=[(2, -100)])
    h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
    full = _fwd_all(lmh, h, w, lab, s)
    # sub-batches of 1, 7, 256 and T rows, in order
    for bs in sorted({1, 7, min(256, T), T}):
        for r0 in range(0, T, bs):
            r1 = min(T, r0 + bs)
            part = _fwd_all(lmh, h[r0:r1], w, lab[r0:r1], s)
            for a, b in zip(part, full):
                assert _mismatch(a, b[r0:r1]) == 0, (bs, r0)
    # every row at every position of a 128-row tile: shift by 1..127
    for shift in range(1, 128):
        if shift >= T:
            continue
        part = _fwd_all(lmh, h[shift:], w, lab[shift:], s)
        for a, b in zip(part, full):
            assert _mismatch(a, b[shift:]) == 0, shift
    # three shuffled packings
    g = torch.Generator().manual_seed(7)
    for _ in range(3):
        perm = torch.randperm(T, generator=g).to(h.device)
        part = _fwd_all(lmh, h[perm].contiguous(), w, lab[perm].contiguous(), s)
        inv = torch.argsort(perm)
        for a, b in zip(part, full):
            assert _mismatch(a[inv], b) == 0


def test_sum_p2_invariant_across_batches(lmh):
    import torch

    T, H, V = 300, 264, 5000
    hidden, weight, labels, _ = fused_case(63, T, H, V)
    h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
    full = lmh.lmhead_logprob_fwd_stats(h, w, lab, S07)[3]
    for r0, r1 in [(0, 1), (1, 8), (8, 264), (131, 300)]:
        part = lmh.lmhead_logprob_fwd_stats(h[r0:r1], w, lab[r0:r1], S07)[3]
        assert _mismatch(part, full[r0:r1]) == 0
    torch.cuda.synchronize()


def test_logits_path_sub_batches_and_shuffles(lmh):
    import torch

    T, V = 300, 5000
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    full = lmh.logprob_from_logits(x, lab, S07, want_lse=True)
    for bs in (1, 7, 256):
        for r0 in range(0, T, bs):
            r1 = min(T, r0 + bs)
            part = lmh.logprob_from_logits(x[r0:r1], lab[r0:r1], S07, want_lse=True)
            for a, b in zip(part, full):
                assert _mismatch(a, b[r0:r1]) == 0
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3)).to(x.device)
    part = lmh.logprob_from_logits(x[perm].contiguous(), lab[perm].contiguous(), S07, want_lse=True)
    for a, b in zip(part, full):
        assert _mismatch(a, b[perm]) == 0
    torch.cuda.synchronize()


def test_grad_hidden_rows_invariant_across_batches(lmh):
    import torch

    T, H, V = 300, 136, 3000
    hidden, weight, labels, grad = fused_case(71, T, H, V, oov=[(5, V)])
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    gh_full, _ = lmh.lmhead_logprob_bwd(h, w, lab, g, S07)
    for bs in (1, 7, 256):
        for r0 in range(0, T, bs):
            r1 = min(T, r0 + bs)
            gh, _ = lmh.lmhead_logprob_bwd(h[r0:r1], w, lab[r0:r1], g[r0:r1], S07)
            assert torch.equal(gh, gh_full[r0:r1]), (bs, r0)
    # shifts that move rows between the two 128-row halves of a CTA pair's tile
    for shift in (1, 127, 128, 129, 255):
        gh, _ = lmh.lmhead_logprob_bwd(h[shift:], w, lab[shift:], g[shift:], S07)
        assert torch.equal(gh, gh_full[shift:]), shift
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(5)).to(h.device)
    gh, _ = lmh.lmhead_logprob_bwd(h[perm].contiguous(), w, lab[perm].contiguous(),
                                   g[perm].contiguous(), S07)
    assert torch.equal(gh, gh_full[perm])
    # with and without a precomputed lse
    _, _, lse = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    gh2, _ = lmh.lmhead_logprob_bwd(h, w, lab, g, S07, lse=lse)
    assert torch.equal(gh2, gh_full)
    torch.cuda.synchronize()


def test_entropy_grad_hidden_rows_invariant_across_batches(lmh):
    import torch

    T, H, V = 300, 136, 3000
    hidden, weight, labels, grad = fused_case(73, T, H, V)
    gent = W.random_f32(74, T)
    h, w, lab, g, ge = (to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad),
                        to_dev(gent))
    full, _ = lmh.lmhead_logprob_entropy_bwd(h, w, lab, g, ge, S07)
    for r0, r1 in [(0, 1), (1, 8), (8, 264), (17, 300)]:
        part, _ = lmh.lmhead_logprob_entropy_bwd(h[r0:r1], w, lab[r0:r1], g[r0:r1], ge[r0:r1], S07)
        assert torch.equal(part, full[r0:r1]), (r0, r1)
    torch.cuda.synchronize()


def test_grad_hidden_rows_invariant_across_row_chunk_boundary(lmh):
    import torch

    T, H, V = 16384 + 130, 64, 600
    hidden, weight, labels, grad = fused_case(81, T, H, V)
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    gh_full, _ = lmh.lmhead_logprob_bwd(h, w, lab, g, 1.0)
    for r0, r1 in [(16300, 16500), (16383, 16385), (0, 1), (16384, T)]:
        gh, _ = lmh.lmhead_logprob_bwd(h[r0:r1], w, lab[r0:r1], g[r0:r1], 1.0)
        assert torch.equal(gh, gh_full[r0:r1]), (r0, r1)
    torch.cuda.synchronize()


def test_logits_division_form_sub_batches_and_shuffles(lmh):
    import torch

    T, V = 300, 5000
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    full = lmh.logprob_from_logits_div(x, lab, 0.7, want_lse=True, want_sum_p2=True)
    for bs in (1, 7, 256):
        for r0 in range(0, T, bs):
            r1 = min(T, r0 + bs)
            part = lmh.logprob_from_logits_div(x[r0:r1], lab[r0:r1], 0.7, want_lse=True,
                                               want_sum_p2=True)
            for a, b in zip(part, full):
                assert _mismatch(a, b[r0:r1]) == 0
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(4)).to(x.device)
    part = lmh.logprob_from_logits_div(x[perm].contiguous(), lab[perm].contiguous(), 0.7,
                                       want_lse=True, want_sum_p2=True)
    for a, b in zip(part, full):
        assert _mismatch(a, b[perm]) == 0
    torch.cuda.synchronize()

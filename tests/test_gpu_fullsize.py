"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: outputs the oracle can compute one by one (sampled rows,
sampled vocabulary rows of grad_weight) and properties that hold at any size.

Workloads (seeded inputs from workloads.py):
  tiny fused forward      T=64    H=256  V=4096   (whole output, plus 1/7-row batches)
  logits path             T=8192         V=152064 (also its division form)
  Llama-like forward      T=4096  H=4096 V=32000
  Qwen-like fwd+bwd       T=16384 H=3584 V=152064 inv_T=1/0.7 (also from host memory)
  packed varlen fwd+bwd   32 sequences, lengths U[128, 4096], H=5120 V=152064
"""

import math

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import ATOL_LOGPROB, RTOL_FROB_GRAD, f64, max_abs, rel_frob, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lmh():
    import torch

    import invariant_lm_head_gb300 as m

    m.build()
    torch.cuda.set_device(0)
    return m


def _sample_rows(T, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    base = [0, 1, 127, 128, T - 129, T - 1] + [x for x in extra if 0 <= x < T]
    rest = rng.choice(T, size=max(0, n - len(base)), replace=False)
    return np.unique(np.concatenate([np.array(base), rest]))


def _bits_equal(a, b):
    import torch

    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_tiny_config_whole_output_and_small_batches(lmh):
    import torch

    wl = W.TINY
    inp = W.fused_inputs(wl)
    h, w = to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"])
    lab = to_dev(inp["labels"])
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, wl.inv_temperature, want_lse=True)
    torch.cuda.synchronize()
    rlp, rent, rlse = oracle.fused_forward(f64(inp["hidden"]), f64(inp["weight"]), inp["labels"],
                                           wl.inv_temperature)
    assert max_abs(lp.cpu().numpy(), rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy(), rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy(), rlse) < ATOL_LOGPROB
    for bs in (1, 7):
        for r0 in range(0, wl.T, bs):
            r1 = min(wl.T, r0 + bs)
            p = lmh.lmhead_logprob_fwd(h[r0:r1], w, lab[r0:r1], wl.inv_temperature, want_lse=True)
            for a, b in zip(p, (lp, ent, lse)):
                assert _bits_equal(a, b[r0:r1])


def test_logits_config_sampled_rows_and_properties(lmh):
    import torch

    wl = W.LOGITS
    inp = W.logits_inputs(wl)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    lp, ent, lse = lmh.logprob_from_logits(x, lab, wl.inv_temperature, want_lse=True)
    torch.cuda.synchronize()
    lp, ent, lse = lp.cpu().numpy(), ent.cpu().numpy(), lse.cpu().numpy()
    rows = _sample_rows(wl.T, 256, 1)
    rlp, rent, rlse = oracle.logprob_from_logits(f64(inp["logits"][rows]), inp["labels"][rows],
                                                 wl.inv_temperature)
    assert max_abs(lp[rows], rlp) < ATOL_LOGPROB
    assert max_abs(ent[rows], rent) < ATOL_LOGPROB
    assert max_abs(lse[rows], rlse) < ATOL_LOGPROB
    # any size: log-probs are <= 0, entropy in [0, ln V], lse >= the largest logit
    assert np.all(lp <= 1e-6)
    assert np.all(ent >= -1e-6) and np.all(ent <= math.log(wl.V) + 1e-4)
    row_max = x.float().max(dim=1).values.cpu().numpy()
    assert np.all(lse >= row_max - 1e-4)


def test_logits_config_division_form_sampled_rows(lmh):
    """The sampler-parity form on the full logits workload, per-row
    temperatures, against the oracle's fp32-division form on sampled rows."""
    import torch

    wl = W.LOGITS
    inp = W.logits_inputs(wl)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    temps = np.random.default_rng(8).uniform(0.5, 1.5, size=wl.T).astype(np.float32)
    lp, ent, lse, q = lmh.logprob_from_logits_div(x, lab, to_dev(temps), want_lse=True,
                                                  want_sum_p2=True)
    torch.cuda.synchronize()
    rows = _sample_rows(wl.T, 128, 9)
    rlp, rent, rlse = oracle.logprob_from_logits_div(f64(inp["logits"][rows]), inp["labels"][rows],
                                                     temps[rows])
    assert max_abs(lp.cpu().numpy()[rows], rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy()[rows], rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy()[rows], rlse) < ATOL_LOGPROB
    rq = oracle.row_sum_p2(oracle.divided_logits(f64(inp["logits"][rows]), temps[rows]))
    assert max_abs(q.cpu().numpy()[rows], rq) < 1e-5


def test_llama_config_forward_sampled_rows(lmh):
    import torch

    wl = W.LLAMA
    inp = W.fused_inputs(wl)
    lp, ent, lse = lmh.lmhead_logprob_fwd(to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"]),
                                          to_dev(inp["labels"]), wl.inv_temperature, want_lse=True)
    torch.cuda.synchronize()
    rows = _sample_rows(wl.T, 128, 2)
    rlp, rent, rlse = oracle.fused_forward_rows(f64(inp["hidden"]), f64(inp["weight"]),
                                                inp["labels"], wl.inv_temperature, rows)
    assert max_abs(lp.cpu().numpy()[rows], rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy()[rows], rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy()[rows], rlse) < ATOL_LOGPROB


@pytest.fixture(scope="module")
def qwen(lmh):
    wl = W.QWEN
    inp = W.fused_inputs(wl)
    return wl, inp, f64(inp["weight"])


def test_qwen_config_forward_backward_sampled(lmh, qwen):
    import torch

    wl, inp, w64 = qwen
    s = wl.inv_temperature
    h, w = to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"])
    lab, g = to_dev(inp["labels"]), to_dev(inp["grad"])
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, g, s, lse=lse)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    rows = _sample_rows(wl.T, 64, 3, extra=(8191, 8192, 16383))
    h64 = f64(inp["hidden"][rows])
    rlp, rent, rlse = oracle.fused_forward_rows(h64, w64, inp["labels"][rows], s,
                                                np.arange(len(rows)))
    assert max_abs(lp.cpu().numpy()[rows], rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy()[rows], rent) < ATOL_LOGPROB
    assert max_abs(lse.cpu().numpy()[rows], rlse) < ATOL_LOGPROB
    rgh = oracle.fused_grad_hidden_rows(h64, w64, inp["labels"][rows], inp["grad"][rows], s,
                                        np.arange(len(rows)))
    ghs = gh.float().cpu().numpy()[rows]
    assert rel_frob(ghs, rgh) < RTOL_FROB_GRAD
    # any size: <grad_weight, weight> = <grad_hidden, hidden> (both = sum dlogit * logit)
    lhs = float(torch.sum(gw.double() * w.double()).item())
    rhs = float(torch.sum(gh.double() * h.double()).item())
    assert abs(lhs - rhs) < RTOL_FROB_GRAD * max(abs(lhs), abs(rhs))


def test_qwen_config_forward_from_host_is_bitwise_the_device_forward(lmh, qwen):
    """The host-staged forward (the benchmark's end-to-end path: weight copied
    in vocab slices, one launch per slice) gives the device forward's bits."""
    import torch

    wl, inp, _ = qwen
    s = wl.inv_temperature
    h_host = W.as_torch_bf16(inp["hidden"]).pin_memory()
    w_host = W.as_torch_bf16(inp["weight"]).pin_memory()
    l_host = torch.from_numpy(inp["labels"]).pin_memory()
    dev = torch.device("cuda:0")
    h = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    w = torch.empty(wl.V, wl.H, dtype=torch.bfloat16, device=dev)
    lab = torch.empty(wl.T, dtype=torch.int32, device=dev)
    lp_host = torch.empty(wl.T, dtype=torch.float32).pin_memory()
    lp, ent, lse = lmh.lmhead_logprob_fwd_host(h_host, w_host, l_host, s, hidden=h, weight=w,
                                               labels=lab, out_logprob_host=lp_host)
    ref = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    assert torch.equal(w.cpu(), w_host) and torch.equal(h.cpu(), h_host)
    for a, b in zip((lp, ent, lse), ref):
        assert _bits_equal(a, b)
    assert torch.equal(lp_host, lp.cpu())


def test_qwen_config_grad_weight_with_sparse_upstream_grad(lmh, qwen):
    """Same shapes and launch configuration; g is zero outside 48 rows, so the
    oracle can form the exact grad_weight (sampled vocabulary rows)."""
    import torch

    wl, inp, w64 = qwen
    s = wl.inv_temperature
    active = _sample_rows(wl.T, 48, 4, extra=(8191, 8192, 16383))
    g = np.zeros(wl.T, dtype=np.float32)
    g[active] = inp["grad"][active]
    h, w = to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"])
    lab = to_dev(inp["labels"])
    _, gw = lmh.lmhead_logprob_bwd(h, w, lab, to_dev(g), s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    vrows = np.unique(np.concatenate([inp["labels"][active], [0, wl.V - 1],
                                      rng.choice(wl.V, 200, replace=False)]))
    ref = oracle.grad_weight_from_rows(f64(inp["hidden"][active]), w64, inp["labels"][active],
                                       g[active], s, np.arange(len(active)), vocab_rows=vrows)
    got = gw[to_dev(vrows.astype(np.int64))].cpu().numpy()
    assert rel_frob(got, ref) < RTOL_FROB_GRAD
    # label rows carry the one-hot term; check them on their own as well
    lab_rows = np.searchsorted(vrows, np.unique(inp["labels"][active]))
    assert rel_frob(got[lab_rows], ref[lab_rows]) < RTOL_FROB_GRAD


def test_qwen_config_entropy_backward_sampled(lmh, qwen):
    """The backward with an entropy gradient (the next row after the hot
    path) at the full workload: grad_hidden on sampled rows, and grad_weight
    on sampled vocabulary rows with both upstream grads zero outside 32 rows."""
    import torch

    wl, inp, w64 = qwen
    s = wl.inv_temperature
    h, w = to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"])
    lab = to_dev(inp["labels"])
    g_ent = np.random.default_rng(12).standard_normal(wl.T).astype(np.float32)
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, _ = lmh.lmhead_logprob_entropy_bwd(h, w, lab, to_dev(inp["grad"]), to_dev(g_ent), s,
                                           lse=lse, entropy=ent)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    rows = _sample_rows(wl.T, 32, 13, extra=(8191, 8192))
    rgh = oracle.fused_grad_hidden_rows(f64(inp["hidden"][rows]), w64, inp["labels"][rows],
                                        inp["grad"][rows], s, np.arange(len(rows)),
                                        grad_entropy=g_ent[rows])
    assert rel_frob(gh.float().cpu().numpy()[rows], rgh) < RTOL_FROB_GRAD
    active = _sample_rows(wl.T, 32, 14)
    g = np.zeros(wl.T, dtype=np.float32)
    ge = np.zeros(wl.T, dtype=np.float32)
    g[active] = inp["grad"][active]
    ge[active] = g_ent[active]
    _, gw = lmh.lmhead_logprob_entropy_bwd(h, w, lab, to_dev(g), to_dev(ge), s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(15)
    vrows = np.unique(np.concatenate([inp["labels"][active], rng.choice(wl.V, 100, replace=False)]))
    ref = oracle.grad_weight_from_rows(f64(inp["hidden"][active]), w64, inp["labels"][active],
                                       g[active], s, np.arange(len(active)), vocab_rows=vrows,
                                       grad_entropy=ge[active])
    got = gw[to_dev(vrows.astype(np.int64))].cpu().numpy()
    assert rel_frob(got, ref) < RTOL_FROB_GRAD


def test_packed_varlen_rows_identical_alone_and_shuffled(lmh):
    import torch

    wl = W.PACKED
    inp = W.fused_inputs(wl)
    s = wl.inv_temperature
    h, w = to_dev_bf16(inp["hidden"]), to_dev_bf16(inp["weight"])
    lab, g = to_dev(inp["labels"]), to_dev(inp["grad"])
    lp, ent, lse = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_bwd(h, w, lab, g, s, lse=lse)
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    offs = np.concatenate([[0], np.cumsum(wl.seq_lens)])
    # every sequence alone
    for i in range(len(wl.seq_lens)):
        a, b = int(offs[i]), int(offs[i + 1])
        p = lmh.lmhead_logprob_fwd(h[a:b], w, lab[a:b], s, want_lse=True)
        for x, y in zip(p, (lp, ent, lse)):
            assert _bits_equal(x, y[a:b]), i
        ghi, _ = lmh.lmhead_logprob_bwd(h[a:b], w, lab[a:b], g[a:b], s, lse=p[2])
        assert torch.equal(ghi, gh[a:b]), i
    # two shuffled packings of the sequences
    rng = np.random.default_rng(6)
    for _ in range(2):
        order = rng.permutation(len(wl.seq_lens))
        idx = np.concatenate([np.arange(offs[i], offs[i + 1]) for i in order])
        ti = to_dev(idx.astype(np.int64))
        hp, lp_, gp = h[ti].contiguous(), lab[ti].contiguous(), g[ti].contiguous()
        p = lmh.lmhead_logprob_fwd(hp, w, lp_, s, want_lse=True)
        ghp, _ = lmh.lmhead_logprob_bwd(hp, w, lp_, gp, s, lse=p[2])
        for x, y in zip(p, (lp, ent, lse)):
            assert _bits_equal(x, y[ti])
        assert torch.equal(ghp, gh[ti])
    torch.cuda.synchronize()
    # sampled rows against the oracle
    rows = _sample_rows(wl.T, 24, 7, extra=tuple(int(o) for o in offs[1:-1][:4]))
    w64 = f64(inp["weight"])
    h64 = f64(inp["hidden"][rows])
    rlp, rent, _ = oracle.fused_forward_rows(h64, w64, inp["labels"][rows], s, np.arange(len(rows)))
    assert max_abs(lp.cpu().numpy()[rows], rlp) < ATOL_LOGPROB
    assert max_abs(ent.cpu().numpy()[rows], rent) < ATOL_LOGPROB
    rgh = oracle.fused_grad_hidden_rows(h64, w64, inp["labels"][rows], inp["grad"][rows], s,
                                        np.arange(len(rows)))
    assert rel_frob(gh.float().cpu().numpy()[rows], rgh) < RTOL_FROB_GRAD

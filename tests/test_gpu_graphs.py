"""CUDA-graph capture of the library's calls: the entry points allocate
nothing and never synchronise, so a whole step can be captured once and
replayed; a replay gives the eager call's bits."""

import numpy as np
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
    m.library()
    torch.cuda.set_device(0)
    return m


def _bits(t):
    import torch

    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def test_forward_backward_step_replays_from_a_graph(lmh):
    import torch

    T, H, V = 300, 264, 5000
    hidden, weight, labels, grad = fused_case(51, T, H, V, w_std=0.2, oov=((3, -100),))
    h, w, lab, g = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), to_dev(grad)
    dev = h.device
    lp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    lse = torch.empty(T, device=dev)
    gh = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    gw = torch.empty(V, H, device=dev)
    ws_f = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, T, H, V), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, T, H, V), dtype=torch.uint8,
                       device=dev)

    def step():
        lmh.lmhead_logprob_fwd(h, w, lab, S07, out_logprob=lp, out_entropy=ent, out_lse=lse,
                               workspace=ws_f)
        lmh.lmhead_logprob_bwd(h, w, lab, g, S07, lse=lse, grad_hidden=gh, grad_weight=gw,
                               workspace=ws_b)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager, also the warm-up before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (lp, ent, lse, gh, gw)]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for x in (lp, ent, lse, gh, gw):
        x.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    lmh.lmhead_device_status()
    for a, b in zip((lp, ent, lse, gh, gw), eager):
        assert torch.equal(_bits(a), _bits(b))

    # new inputs copied into the captured buffers are picked up by the replay
    hidden2 = W.random_bf16(52, (T, H), 1.0)
    h.copy_(to_dev_bf16(hidden2))
    graph.replay()
    torch.cuda.synchronize()
    ref = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    for a, b in zip((lp, ent, lse), ref):
        assert torch.equal(_bits(a), _bits(b))


def test_logits_paths_replay_from_a_graph(lmh):
    import torch

    T, V = 64, 5000
    inp = W.logits_inputs(W.LOGITS, T=T, V=V)
    x, lab = to_dev_bf16(inp["logits"]), to_dev(inp["labels"])
    temps = to_dev(np.random.default_rng(3).uniform(0.5, 1.5, size=T).astype(np.float32))
    out = [torch.empty(T, device=x.device) for _ in range(4)]

    def run():
        lmh.logprob_from_logits(x, lab, S07, out_logprob=out[0], out_entropy=out[1])
        lmh.logprob_from_logits_div(x, lab, temps, out_logprob=out[2], out_entropy=out[3])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [o.clone() for o in out]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for o in out:
        o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(out, eager):
        assert torch.equal(_bits(a), _bits(b))


def test_forward_from_host_replays_from_a_graph(lmh):
    """The staged forward forks its copies onto a second stream through
    events; captured, the fork and join become graph edges and a replay
    copies the current host inputs."""
    import torch

    T, H, V = 200, 128, 5000
    hidden, weight, labels, _ = fused_case(53, T, H, V, w_std=0.2)
    h_host = W.as_torch_bf16(hidden).pin_memory()
    w_host = W.as_torch_bf16(weight).pin_memory()
    l_host = torch.from_numpy(labels).pin_memory()
    dev = torch.device("cuda:0")
    h = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    w = torch.empty(V, H, dtype=torch.bfloat16, device=dev)
    lab = torch.empty(T, dtype=torch.int32, device=dev)
    lp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    lse = torch.empty(T, device=dev)
    ws = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_FWD, T, H, V), dtype=torch.uint8,
                     device=dev)
    copy_stream = torch.cuda.Stream()

    def run():
        lmh.lmhead_logprob_fwd_host(h_host, w_host, l_host, S07, hidden=h, weight=w, labels=lab,
                                    out_logprob=lp, out_entropy=ent, out_lse=lse, workspace=ws,
                                    copy_stream=copy_stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (lp, ent, lse)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    h.zero_(), w.zero_(), lp.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(w.cpu(), w_host)
    for a, b in zip((lp, ent, lse), eager):
        assert torch.equal(_bits(a), _bits(b))
    # new host contents are copied by the next replay
    h_host.copy_(W.as_torch_bf16(W.random_bf16(54, (T, H), 1.0)))
    graph.replay()
    torch.cuda.synchronize()
    ref = lmh.lmhead_logprob_fwd(h, w, lab, S07, want_lse=True)
    assert torch.equal(h.cpu(), h_host)
    for a, b in zip((lp, ent, lse), ref):
        assert torch.equal(_bits(a), _bits(b))

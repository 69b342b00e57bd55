"""The vocab-parallel (tensor-parallel) LM head end to end: two gloo ranks,
each a child process holding one vocabulary shard of the weight, run the
forward and backward of invariant_lm_head_gb300.vocab_parallel on the one GPU.
No kernel waits on another rank: the exchange is torch.distributed's all-gather
and all-reduce through host memory, between the ranks' launches.

Checked, as the SkyRL page's tensor-parallel tests check its distributed
log-prob against the single-rank one:
  - logprob, entropy and lse are the same bits on both ranks, and the same
    bits as lmhead_logprob_fwd on the whole weight;
  - grad_hidden is the same bits on both ranks, and within 1e-2 relative
    Frobenius error of the fp64 oracle, with and without an entropy gradient;
  - each rank's grad_weight rows, put together, are within 1e-2 of the oracle's.
"""

import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import RTOL_FROB_GRAD, f64, fused_case, rel_frob, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os, sys
sys.path.insert(0, sys.argv[2])
sys.path.insert(0, os.path.join(sys.argv[2], "tests"))
import numpy as np
import torch
import torch.distributed as dist
import invariant_lm_head_gb300 as lmh
from invariant_lm_head_gb300 import vocab_parallel as vp
from helpers import fused_case, to_dev, to_dev_bf16

rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
torch.cuda.set_device(0)
lmh.build()
dist.init_process_group("gloo", rank=rank, world_size=world)
out = {}
for (seed, T, H, V, s) in [(31, 300, 264, 5000, float(np.float32(1 / 0.7))),
                           (32, 777, 512, 4099, 1.0)]:
    hidden, weight, labels, grad = fused_case(seed, T, H, V, oov=[(0, -100)])
    labels[1], labels[2], labels[3] = 0, V - 1, 3071
    g_ent = np.random.default_rng(seed).standard_normal(T).astype(np.float32)
    b0, b1 = vp.shard_bounds(V, world, rank)
    h, lab = to_dev_bf16(hidden), to_dev(labels)
    w = to_dev_bf16(weight[b0:b1])
    lp, ent, lse = vp.vocab_parallel_logprob_fwd(h, w, lab, b0, V, s)
    gh, gw = vp.vocab_parallel_logprob_bwd(h, w, lab, to_dev(grad), lse, b0, s)
    gh2, gw2 = vp.vocab_parallel_logprob_bwd(h, w, lab, to_dev(grad), lse, b0, s,
                                             grad_entropy=to_dev(g_ent), entropy=ent)
    torch.cuda.synchronize()
    assert lmh.lmhead_device_status() == 0
    for k, v in dict(lp=lp, ent=ent, lse=lse, gh=gh, gw=gw, gh2=gh2, gw2=gw2).items():
        out[f"{seed}_{k}"] = v.cpu()
    out[f"{seed}_bounds"] = (b0, b1)
dist.destroy_process_group()
torch.save(out, sys.argv[1])
'''


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _i32(t):
    import torch

    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def test_two_vocab_shards_on_gloo_ranks(tmp_path):
    import torch

    import invariant_lm_head_gb300 as lmh

    child = tmp_path / "child.py"
    child.write_text(CHILD)
    world, port = 2, _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(child), str(tmp_path / f"r{r}.pt"),
                                       ROOT], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    logs = [p.communicate(timeout=900)[0] for p in procs]
    for p, log in zip(procs, logs):
        assert p.returncode == 0, log[-3000:]
    res = [torch.load(tmp_path / f"r{r}.pt") for r in range(world)]

    lmh.build()
    torch.cuda.set_device(0)
    for (seed, T, H, V, s) in [(31, 300, 264, 5000, W.f32(1 / 0.7)), (32, 777, 512, 4099, 1.0)]:
        hidden, weight, labels, grad = fused_case(seed, T, H, V, oov=[(0, -100)])
        labels[1], labels[2], labels[3] = 0, V - 1, 3071
        g_ent = np.random.default_rng(seed).standard_normal(T).astype(np.float32)
        whole = lmh.lmhead_logprob_fwd(to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels), s,
                                       want_lse=True)
        torch.cuda.synchronize()
        for k, want in zip(("lp", "ent", "lse"), whole):
            for r in range(world):
                assert torch.equal(_i32(res[r][f"{seed}_{k}"]), _i32(want.cpu())), \
                    f"{k} on rank {r} differs in its bits from the whole-weight forward"
        for k in ("gh", "gh2"):
            assert torch.equal(_i32(res[0][f"{seed}_{k}"]), _i32(res[1][f"{seed}_{k}"])), k
        h64, w64 = f64(hidden), f64(weight)
        rgh, rgw = oracle.fused_backward(h64, w64, labels, grad, s)
        rgh2, rgw2 = oracle.fused_backward(h64, w64, labels, grad, s, grad_entropy=g_ent)
        for k, rgh_, rgw_ in (("", rgh, rgw), ("2", rgh2, rgw2)):
            gh = res[0][f"{seed}_gh{k}"].float().numpy()
            assert rel_frob(gh, rgh_) < RTOL_FROB_GRAD
            gw = np.concatenate([res[r][f"{seed}_gw{k}"].numpy() for r in range(world)])
            assert gw.shape == rgw_.shape
            assert rel_frob(gw, rgw_) < RTOL_FROB_GRAD
            for r in range(world):
                b0, b1 = res[r][f"{seed}_bounds"]
                assert rel_frob(res[r][f"{seed}_gw{k}"].numpy(), rgw_[b0:b1]) < RTOL_FROB_GRAD


def test_shard_backward_without_lse_is_refused():
    import torch

    import invariant_lm_head_gb300 as lmh

    lmh.build()
    lib = lmh.library()
    d = torch.device("cuda:0")
    T, H, V = 8, 64, 2048
    h = torch.zeros(T, H, dtype=torch.bfloat16, device=d)
    w = torch.zeros(V, H, dtype=torch.bfloat16, device=d)
    lab = torch.zeros(T, dtype=torch.int32, device=d)
    g = torch.zeros(T, device=d)
    gh = torch.empty(T, H, device=d)
    gw = torch.empty(V, H, device=d)
    ws = torch.empty(lmh.lmhead_workspace_size(lmh.LMH_OP_BWD, T, H, V), dtype=torch.uint8,
                     device=d)
    before = lmh.lmhead_kernel_launches()
    rc = lib.lmhead_logprob_bwd_shard(h.data_ptr(), w.data_ptr(), lab.data_ptr(), g.data_ptr(),
                                      None, None, None, T, H, V, 1024, 1.0, gh.data_ptr(),
                                      gw.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert rc == lmh.LMH_ERR_INVALID_ARG
    assert b"lse" in lib.lmhead_last_error_string()
    assert lmh.lmhead_kernel_launches() == before

"""The tensor-core engine runs a contraction on single CTAs (128 x 256
tiles), on CTA pairs that share each MMA (256 x 256), or on wide pairs
(256 x 512). Which one runs must not change a bit of the log-probs, entropy,
lse or grad_hidden: each output element's dot product walks K in the same
order on every engine. Child processes force each engine (the choice is read
once per process) on ragged shapes, including pairs whose second half lies
wholly past the last row, and every output is compared bit for bit.

Store contractions also run on narrower tiles (64, 128 or 192 columns on
single CTAs, 128 on pairs) when a short launch would leave SMs idle; every
width is forced in turn and compared too.

grad_weight walks K downwards on a CTA's odd waves, so its summation order
follows the engine's wave structure. The shapes here fit each grad_weight
launch in one wave on the single and paired engines, where that order is the
same, so grad_weight and the bare engine GEMM are compared bit for bit there.

The schedule (a fixed stride over the units, or units claimed from a counter
in ascending order) must not change a bit either, grad_weight included: its K
direction follows the unit's wave index, not the CTA that runs it. A grid cap
of a few CTAs (or pairs) makes each walk dozens of units long, so the dynamic
schedule's 16-slot unit ring wraps several times."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import torch
sys.path.insert(0, sys.argv[2])
import workloads as W
import invariant_lm_head_gb300 as lmh

lmh.build()
dev = torch.device("cuda:0")
out = {}
for (T, H, V, s) in [(777, 520, 3001, 1 / 0.7), (129, 1024, 4099, 1.0), (300, 264, 517, 2.0)]:
    hidden = W.as_torch_bf16(W.random_bf16(T, (T, H), 1.0)).to(dev)
    weight = W.as_torch_bf16(W.random_bf16(T + 1, (V, H), 0.05)).to(dev)
    labels = torch.from_numpy(W.random_labels(T, T, V)).to(dev)
    grad = torch.from_numpy(W.random_f32(T, T)).to(dev)
    grad_e = torch.from_numpy(W.random_f32(T + 2, T)).to(dev)
    lp, ent, lse = lmh.lmhead_logprob_fwd(hidden, weight, labels, s, want_lse=True)
    gh, gw = lmh.lmhead_logprob_bwd(hidden, weight, labels, grad, s, lse=lse)
    gh2, gw2 = lmh.lmhead_logprob_entropy_bwd(hidden, weight, labels, grad, grad_e, s)
    for k, v in dict(lp=lp, ent=ent, lse=lse, gh=gh, gw=gw, gh2=gh2, gw2=gw2).items():
        out[f"{T}_{k}"] = v.cpu()
M, N, K = 296, 264, 136
A = W.as_torch_bf16(W.random_bf16(5, (M, K), 1.0)).to(dev)
B = W.as_torch_bf16(W.random_bf16(6, (N, K), 1.0)).to(dev)
for ak in (True, False):
    for bk in (True, False):
        a = A if ak else A.t().contiguous()
        b = B if bk else B.t().contiguous()
        out[f"gemm_{int(ak)}{int(bk)}"] = lmh.lmhead_engine_gemm(a, b, a_kmajor=ak, b_kmajor=bk).cpu()
torch.cuda.synchronize()
assert lmh.lmhead_device_status() == 0
torch.save(out, sys.argv[1])
'''


def _run(tmp_path, name, env_extra):
    import torch

    child = tmp_path / "child.py"
    if not child.exists():
        child.write_text(CHILD)
    path = tmp_path / f"out_{name}.pt"
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, str(child), str(path), ROOT], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    return torch.load(path)


def _same(a, b):
    import torch

    return a.shape == b.shape and torch.equal(
        a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
        b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


@pytest.fixture(scope="module")
def single(tmp_path_factory):
    return _run(tmp_path_factory.mktemp("single"), "single", {"LMH_GEMM_CTA_PAIRS": "0"})


# "1": every contraction on wide pairs; "2": every contraction on 256-wide pairs.
@pytest.mark.parametrize("pairs", ["1", "2"])
def test_pair_and_single_engines_give_identical_bits(tmp_path, single, pairs):
    pair = _run(tmp_path, f"pair{pairs}", {"LMH_GEMM_CTA_PAIRS": pairs})
    assert single.keys() == pair.keys()
    for k in single:
        assert _same(single[k], pair[k]), f"{k}: the single-CTA and CTA-pair engines differ"


# Every engine and tile width the store contractions can take (forced with
# LMH_GEMM_STORE_ENGINE): grad_hidden (gh, gh2) and the bare engine GEMM must
# keep their bits, and so must the forward outputs. grad_weight is left out
# here: narrow tiles spread it over several waves, whose K direction differs.
@pytest.mark.parametrize("engine", ["s64", "s128", "s192", "p128", "p256", "w"])
def test_every_store_engine_and_width_gives_identical_bits(tmp_path, single, engine):
    forced = _run(tmp_path, engine, {"LMH_GEMM_STORE_ENGINE": engine})
    assert single.keys() == forced.keys()
    for k in single:
        if k.endswith("_gw") or k.endswith("_gw2"):
            continue
        assert _same(single[k], forced[k]), f"{k}: engine {engine} differs from single CTAs"


@pytest.mark.parametrize("pairs,cap", [("0", "2"), ("1", "3"), ("2", "3")])
def test_dynamic_schedule_gives_identical_bits(tmp_path, single, pairs, cap):
    env = {"LMH_GEMM_CTA_PAIRS": pairs, "LMH_GEMM_GRID_CAP": cap}
    fixed = _run(tmp_path, f"static_{pairs}", dict(env, LMH_GEMM_SCHEDULE="static"))
    claimed = _run(tmp_path, f"dynamic_{pairs}", dict(env, LMH_GEMM_SCHEDULE="dynamic"))
    assert fixed.keys() == claimed.keys() == single.keys()
    for k in fixed:
        assert _same(fixed[k], claimed[k]), f"{k}: the dynamic schedule changed bits"
        if not (k.endswith("_gw") or k.endswith("_gw2")):
            assert _same(single[k], claimed[k]), f"{k}: capped grid differs from single CTAs"


# A ragged batch on CTA pairs: with 7 row tiles the last pair's second half
# lies wholly past the last row and stores nothing. On a one-pair grid every
# such half follows a live tile of the same CTA, whose last TMA store may
# still be reading its staging buffer; the backward is repeated and must keep
# its bits (and match single CTAs) every time.
CHILD_REPEAT = r'''
import sys
import torch
sys.path.insert(0, sys.argv[2])
import workloads as W
import invariant_lm_head_gb300 as lmh

lmh.build()
dev = torch.device("cuda:0")
T, H, V, s = 777, 520, 3001, 1 / 0.7
hidden = W.as_torch_bf16(W.random_bf16(T, (T, H), 1.0)).to(dev)
weight = W.as_torch_bf16(W.random_bf16(T + 1, (V, H), 0.05)).to(dev)
labels = torch.from_numpy(W.random_labels(T, T, V)).to(dev)
grad = torch.from_numpy(W.random_f32(T, T)).to(dev)
_, _, lse = lmh.lmhead_logprob_fwd(hidden, weight, labels, s, want_lse=True)
out = {}
for rep in range(int(sys.argv[3])):
    gh, gw = lmh.lmhead_logprob_bwd(hidden, weight, labels, grad, s, lse=lse)
    out[f"gh{rep}"] = gh.cpu()
    out[f"gw{rep}"] = gw.cpu()
torch.cuda.synchronize()
assert lmh.lmhead_device_status() == 0
torch.save(out, sys.argv[1])
'''


@pytest.mark.parametrize("pairs", ["1", "2"])
@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_pair_halves_past_the_last_row_keep_live_stores_intact(tmp_path, single, schedule, pairs):
    import torch

    reps = 12
    child = tmp_path / "repeat.py"
    child.write_text(CHILD_REPEAT)
    path = tmp_path / "rep.pt"
    env = dict(os.environ, LMH_GEMM_CTA_PAIRS=pairs, LMH_GEMM_GRID_CAP="1",
               LMH_GEMM_SCHEDULE=schedule)
    r = subprocess.run([sys.executable, str(child), str(path), ROOT, str(reps)], env=env,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    out = torch.load(path)
    for rep in range(reps):
        assert _same(out[f"gh{rep}"], single["777_gh"]), f"grad_hidden differs on repeat {rep}"
        assert _same(out[f"gw{rep}"], out["gw0"]), f"grad_weight differs on repeat {rep}"


# On single CTAs and 256-wide pairs the forward and dlogits overlap
# consecutive tiles' K loops (the operand ring then alternates between two
# tiles); each tile's own MMAs keep their order, so turning the overlap off
# must change no bit on either engine.
@pytest.mark.parametrize("pairs", ["0", "2"])
def test_overlapped_tiles_give_identical_bits(tmp_path, single, pairs):
    on = single if pairs == "0" else _run(tmp_path, "pairs_on", {"LMH_GEMM_CTA_PAIRS": pairs})
    off = _run(tmp_path, f"off_{pairs}", {"LMH_GEMM_CTA_PAIRS": pairs, "LMH_GEMM_INTERLEAVE": "0"})
    assert on.keys() == off.keys()
    for k in on:
        assert _same(on[k], off[k]), f"{k}: overlapping the tiles changed bits"


# grad_hidden and grad_weight of a row chunk may run side by side, grad_hidden
# on a second stream of the library's own (LMH_BWD_OVERLAP forces it off or
# on), over one chunk and over seven 128-row chunks, where the next chunk's
# dlogits must wait for the side stream before it overwrites dl and
# grad_weight's reduce-adds must keep chunk order. grad_hidden keeps its bits.
# Side by side, grad_weight runs on wide pairs, whose summation order differs
# from the 256-wide pairs it takes alone: with every store contraction forced
# onto wide pairs the two modes must agree bit for bit, and by default each
# mode must repeat its own bits and agree with the other to fp32 rounding. A
# grid cap makes grad_weight claim several units per CTA meanwhile.
CHILD_CHUNKS = r'''
import sys
import torch
sys.path.insert(0, sys.argv[2])
import workloads as W
import invariant_lm_head_gb300 as lmh

lmh.build()
dev = torch.device("cuda:0")
out = {}
for (T, H, V, s) in [(777, 520, 3001, 1 / 0.7), (300, 264, 517, 2.0)]:
    hidden = W.as_torch_bf16(W.random_bf16(T, (T, H), 1.0)).to(dev)
    weight = W.as_torch_bf16(W.random_bf16(T + 1, (V, H), 0.05)).to(dev)
    labels = torch.from_numpy(W.random_labels(T, T, V)).to(dev)
    grad = torch.from_numpy(W.random_f32(T, T)).to(dev)
    grad_e = torch.from_numpy(W.random_f32(T + 2, T)).to(dev)
    _, ent, lse = lmh.lmhead_logprob_fwd(hidden, weight, labels, s, want_lse=True)
    for rep in range(3):
        gh, gw = lmh.lmhead_logprob_bwd(hidden, weight, labels, grad, s, lse=lse)
        gh_c, gw_c = lmh.lmhead_logprob_bwd_chunked(hidden, weight, labels, grad, s, row_chunk=128,
                                                    grad_entropy=grad_e, lse=lse, entropy=ent)
        for k, v in dict(gh=gh, gw=gw, gh_c=gh_c, gw_c=gw_c).items():
            out[f"{T}_{k}_{rep}"] = v.cpu()
torch.cuda.synchronize()
assert lmh.lmhead_device_status() == 0
torch.save(out, sys.argv[1])
'''


@pytest.mark.parametrize("engine", ["", "w"])
@pytest.mark.parametrize("cap", ["", "4"])
def test_grad_hidden_beside_grad_weight(tmp_path, engine, cap):
    import torch

    child = tmp_path / "chunks.py"
    child.write_text(CHILD_CHUNKS)
    res = {}
    for mode in ("0", "1"):
        path = tmp_path / f"ov{mode}.pt"
        env = dict(os.environ, LMH_BWD_OVERLAP=mode)
        if cap:
            env["LMH_GEMM_GRID_CAP"] = cap
        if engine:
            env["LMH_GEMM_STORE_ENGINE"] = engine
        r = subprocess.run([sys.executable, str(child), str(path), ROOT], env=env, cwd=ROOT,
                           capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, r.stderr[-2000:]
        res[mode] = torch.load(path)
    assert res["0"].keys() == res["1"].keys()
    for k in res["0"]:
        base = k.rsplit("_", 1)[0] + "_0"
        for mode in ("0", "1"):
            assert _same(res[mode][k], res[mode][base]), f"{k}: repeats differ (mode {mode})"
        a, b = res["0"][k], res["1"][k]
        if engine or "_gh" in k:
            assert _same(a, b), f"{k}: running grad_hidden beside grad_weight changed bits"
        else:
            err = (a.double() - b.double()).norm() / a.double().norm()
            assert err < 1e-5, f"{k}: side by side, grad_weight moved by {float(err):.2e}"


# A wide tile's last K blocks run its first 256 columns ahead of the second
# (LMH_GEMM_WIDE_SKEW; 0 runs the two together to the end). Each chain keeps
# its K order, so with every contraction on wide pairs no output may change a
# bit, grad_weight included (same engine, same waves).
def test_skewed_tile_ends_give_identical_bits(tmp_path):
    on = _run(tmp_path, "skew_on", {"LMH_GEMM_CTA_PAIRS": "1"})
    off = _run(tmp_path, "skew_off", {"LMH_GEMM_CTA_PAIRS": "1", "LMH_GEMM_WIDE_SKEW": "0"})
    assert on.keys() == off.keys()
    for k in on:
        assert _same(on[k], off[k]), f"{k}: the skewed tile ends changed bits"

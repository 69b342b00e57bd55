"""The forward entry point that allocates nothing, checked on the GPU.

lmhead_logprob_fwd_noalloc serves callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory, or code that
must not call cudaMalloc because it may block and synchronise the device). It
keeps its scratch in a fixed array inside the library, shared by every call and
never cleared between calls.

It runs the same kernels on the same tiles as the workspace-taking
lmhead_logprob_fwd, so its outputs must be bit-identical to that entry point's,
and within the suite's 1e-3 tolerance of the fp64 oracle. The calls here run
through the C ABI in a sequence that leaves the previous call's values in the
array: a large call followed by a smaller one with another vocabulary size, and
the same shape twice with different inputs. A merge that read a stale partial
would then differ in its bits. A call too large for the array is refused.

The file name makes pytest collect it last.
"""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import ATOL_LOGPROB, f64, fused_case, max_abs, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

# (seed, T, H, V): largest first, so each later call runs over an array that
# still holds the earlier calls' partials; the last two share a shape.
CALLS = [(101, 4000, 512, 32000), (102, 300, 264, 5000), (103, 777, 256, 4099),
         (104, 777, 256, 4099)]
ORACLE_ROWS = 96  # rows checked against the oracle per call (all of them when fewer)


def _noalloc(lib, h, w, lab, s):
    import torch

    T, H = h.shape
    V = w.shape[0]
    d = h.device
    lp = torch.full((T,), float("nan"), device=d)
    ent = torch.full((T,), float("nan"), device=d)
    lse = torch.full((T,), float("nan"), device=d)
    rc = lib.lmhead_logprob_fwd_noalloc(h.data_ptr(), w.data_ptr(), lab.data_ptr(), T, H, V, s,
                                        lp.data_ptr(), ent.data_ptr(), lse.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    return rc, lp, ent, lse


def _bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.int32)


def test_noalloc_forward_matches_workspace_forward_and_oracle_over_successive_calls():
    import torch

    import invariant_lm_head_gb300 as lmh

    lmh.build()
    lib = lmh.library()
    torch.cuda.set_device(0)
    s = W.f32(1.0 / 0.7)
    for seed, T, H, V in CALLS:
        hidden, weight, labels, _ = fused_case(seed, T, H, V, oov=[(0, -100)])
        labels[1] = V - 1
        h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
        rc, lp, ent, lse = _noalloc(lib, h, w, lab, s)
        assert rc == lmh.LMH_OK, lib.lmhead_last_error_string()
        torch.cuda.synchronize()
        assert lmh.lmhead_device_status() == 0
        got = [t.cpu().numpy() for t in (lp, ent, lse)]
        ref = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
        torch.cuda.synchronize()
        for g, r, name in zip(got, ref, ("logprob", "entropy", "lse")):
            assert np.array_equal(_bits(g), _bits(r.cpu().numpy())), \
                f"{name} differs in its bits from lmhead_logprob_fwd (T={T}, V={V})"
        rng = np.random.default_rng(seed)
        rows = np.arange(T) if T <= ORACLE_ROWS else np.unique(np.concatenate(
            [[0, 1, 127, 128, T - 1], rng.choice(T, ORACLE_ROWS - 5, replace=False)]))
        rlp, rent, rlse = oracle.fused_forward_rows(f64(hidden), f64(weight), labels, s, rows)
        assert max_abs(got[0][rows], rlp) < ATOL_LOGPROB
        assert max_abs(got[1][rows], rent) < ATOL_LOGPROB
        assert max_abs(got[2][rows], rlse) < ATOL_LOGPROB
        assert got[0][0] == 0.0  # the out-of-vocab row


def test_noalloc_forward_refuses_calls_beyond_its_scratch():
    import torch

    import invariant_lm_head_gb300 as lmh

    lmh.build()
    lib = lmh.library()
    d = torch.device("cuda:0")
    T, H, V = 16384, 64, 152064  # partials need ~29 MB > 16 MiB
    h = torch.zeros(T, H, dtype=torch.bfloat16, device=d)
    w = torch.zeros(V, H, dtype=torch.bfloat16, device=d)
    lab = torch.zeros(T, dtype=torch.int32, device=d)
    before = lmh.lmhead_kernel_launches()
    rc, *_ = _noalloc(lib, h, w, lab, 1.0)
    assert rc == lmh.LMH_ERR_WORKSPACE
    assert b"scratch" in lib.lmhead_last_error_string()
    assert lmh.lmhead_kernel_launches() == before

"""The forward entry point that allocates nothing, checked on the GPU.

lmhead_logprob_fwd_noalloc serves callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory, or code that
must not call cudaMalloc because it may block and synchronise the device). It
keeps its scratch in a fixed array inside the library. This test calls it
through the C ABI twice in a row, on different inputs, and compares each result
with the workspace-taking lmhead_logprob_fwd within the suite's tolerance. It
also checks that a call too large for the fixed scratch is refused.

The file name makes pytest collect it last.
"""

import numpy as np
import pytest

import workloads as W
from helpers import ATOL_LOGPROB, fused_case, max_abs, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


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


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    import torch

    import invariant_lm_head_gb300 as lmh

    lmh.build()
    lib = lmh.library()
    torch.cuda.set_device(0)
    s = W.f32(1.0 / 0.7)
    for seed, (T, H, V) in [(101, (300, 264, 5000)), (102, (1000, 512, 32000))]:
        hidden, weight, labels, _ = fused_case(seed, T, H, V, oov=[(0, -100)])
        h, w, lab = to_dev_bf16(hidden), to_dev_bf16(weight), to_dev(labels)
        rc, lp, ent, lse = _noalloc(lib, h, w, lab, s)
        assert rc == lmh.LMH_OK, lib.lmhead_last_error_string()
        ref = lmh.lmhead_logprob_fwd(h, w, lab, s, want_lse=True)
        torch.cuda.synchronize()
        assert lmh.lmhead_device_status() == 0
        for got, want in zip((lp, ent, lse), ref):
            g, r = got.cpu().numpy(), want.cpu().numpy()
            assert np.all(np.isfinite(g))
            assert max_abs(g, r) < ATOL_LOGPROB


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

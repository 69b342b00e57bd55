"""Host-side checks of the C ABI: the library loads without a GPU, exports every
symbol include/lmhead.h declares, sizes workspaces and rejects bad arguments
before touching a device."""

import ctypes
import os
import re

import pytest

import invariant_lm_head_gb300 as lmh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmhead.h")


@pytest.fixture(scope="module")
def lib():
    lmh.build()
    return lmh.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w \t*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["lmhead_logprob_fwd", "lmhead_logprob_bwd", "logprob_from_logits",
              "lmhead_workspace_size", "lmhead_last_error_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(lmh.SIGNATURES)


def test_abi_version(lib):
    assert lib.lmhead_abi_version() == 1


def test_workspace_sizes(lib):
    f = lmh.lmhead_workspace_size
    assert f(lmh.LMH_OP_LOGITS, 8192, 0, 152064) == 0
    # forward: 4 planes of ceil(V / 1024) floats per row + the label logit
    n_chunks = -(-152064 // 1024)
    fwd = f(lmh.LMH_OP_FWD, 16384, 3584, 152064)
    assert fwd >= (4 * n_chunks + 1) * 16384 * 4
    assert fwd < (4 * n_chunks + 1) * 16384 * 4 + 8 * 256
    # backward: forward partials + lse, logprob, entropy per row + bf16 dlogits [min(T,16384), V]
    b1 = f(lmh.LMH_OP_BWD, 16384, 3584, 152064)
    b2 = f(lmh.LMH_OP_BWD, 32768, 3584, 152064)
    extra = (4 * n_chunks + 4) * 16384 * 4
    assert 0 <= (b2 - b1) - extra < 64 * 256
    assert b1 > 16384 * 152064 * 2
    assert f(lmh.LMH_OP_FWD, 0, 256, 4096) > 0
    for bad in [(lmh.LMH_OP_FWD, -1, 256, 4096), (lmh.LMH_OP_FWD, 4, 12, 4096),
                (lmh.LMH_OP_FWD, 4, 256, 0), (7, 4, 256, 4096)]:
        with pytest.raises(lmh.LMHeadError):
            f(*bad)


def _call_fwd(lib, **kw):
    a = dict(hidden=16, weight=16, labels=16, T=4, H=256, V=4096, s=1.0, lp=16, ent=None, lse=None,
             ws=256, wsb=1 << 30)
    a.update(kw)
    return lib.lmhead_logprob_fwd(a["hidden"], a["weight"], a["labels"], a["T"], a["H"], a["V"],
                                  a["s"], a["lp"], a["ent"], a["lse"], a["ws"], a["wsb"], None)


def test_argument_errors_are_reported_without_a_launch(lib):
    # Fake, never dereferenced addresses: every case fails validation first.
    assert _call_fwd(lib, hidden=None) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, hidden=24) == lmh.LMH_ERR_ALIGNMENT
    assert _call_fwd(lib, H=12) == lmh.LMH_ERR_ALIGNMENT
    assert _call_fwd(lib, T=-1) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, V=0) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, s=0.0) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, s=float("inf")) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, s=float("nan")) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, lp=None) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, ent=18) == lmh.LMH_ERR_ALIGNMENT
    assert _call_fwd(lib, wsb=16) == lmh.LMH_ERR_WORKSPACE
    assert _call_fwd(lib, ws=None) == lmh.LMH_ERR_WORKSPACE
    assert b"workspace" in lib.lmhead_last_error_string()
    big = 2147483392 + 1  # one past LMH_MAX_DIM
    assert _call_fwd(lib, T=big) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, V=big) == lmh.LMH_ERR_INVALID_ARG
    assert _call_fwd(lib, H=big + 7) == lmh.LMH_ERR_INVALID_ARG  # a multiple of 8 past the limit
    assert lmh.library().lmhead_workspace_size(lmh.LMH_OP_FWD, big, 256, 4096) == ctypes.c_size_t(-1).value
    assert _call_fwd(lib, T=0) == lmh.LMH_OK  # empty batch: nothing to do
    assert _call_fwd(lib, T=0, hidden=None, labels=None, lp=None, ws=None) == lmh.LMH_OK
    rc = lib.logprob_from_logits(24, 16, 4, 4096, 1.0, 16, None, None, None)
    assert rc == lmh.LMH_ERR_ALIGNMENT
    rc = lib.logprob_from_logits(18, 16, 4, 4095, 1.0, 16, None, None, None)
    assert rc != lmh.LMH_ERR_ALIGNMENT  # odd V only needs 2-byte alignment
    rc = lib.lmhead_logprob_bwd(16, 16, 16, None, None, 4, 256, 4096, 1.0, 16, 16, 256, 1 << 30,
                                None)
    assert rc == lmh.LMH_ERR_INVALID_ARG
    rc = lib.lmhead_logprob_entropy_bwd(16, 16, 16, None, None, None, None, 4, 256, 4096, 1.0, 16,
                                        16, 256, 1 << 30, None)
    assert rc == lmh.LMH_ERR_INVALID_ARG  # both upstream grads missing
    div = lib.logprob_from_logits_div
    assert div(16, 16, 4, 4096, 0.0, None, 16, None, None, None, None) == lmh.LMH_ERR_INVALID_ARG
    assert div(16, 16, 4, 4096, float("nan"), None, 16, None, None, None, None) == \
        lmh.LMH_ERR_INVALID_ARG
    assert b"temperature" in lib.lmhead_last_error_string()
    assert div(16, 16, 4, 4096, 0.7, 18, 16, None, None, None, None) == lmh.LMH_ERR_ALIGNMENT
    assert div(24, 16, 4, 4096, 0.7, None, 16, None, None, None, None) == lmh.LMH_ERR_ALIGNMENT
    assert div(None, None, 0, 4096, 0.7, None, None, None, None, None, None) == lmh.LMH_OK
    fh = lib.lmhead_logprob_fwd_host
    args = [16, 16, 16, 4, 256, 4096, 1.0, 16, 16, 16, 16, None, None, None, None, 256, 1 << 30,
            None, None]
    assert fh(*args[:2], None, *args[3:]) == lmh.LMH_ERR_INVALID_ARG  # host labels missing
    assert fh(*args[:7], 24, *args[8:]) == lmh.LMH_ERR_ALIGNMENT  # device hidden
    assert fh(*args[:14], 16, *args[15:]) == lmh.LMH_ERR_INVALID_ARG  # entropy host w/o device
    assert fh(*args[:15], None, *args[16:]) == lmh.LMH_ERR_WORKSPACE
    assert fh(*args[:6], 0.0, *args[7:]) == lmh.LMH_ERR_INVALID_ARG
    assert fh(None, None, None, 0, 256, 4096, 1.0, *([None] * 9), 0, None, None) == lmh.LMH_OK
    fp = lib.lmhead_logprob_fwd_partials
    pa = [16, 16, 16, 4, 256, 4096, 0, 1.0, 16, 16, 16, 16, None]
    assert fp(*pa[:6], 512, *pa[7:]) == lmh.LMH_ERR_ALIGNMENT  # v_offset not a chunk start
    assert fp(*pa[:6], -1024, *pa[7:]) == lmh.LMH_ERR_INVALID_ARG
    assert fp(*pa[:11], None, None) == lmh.LMH_ERR_INVALID_ARG  # label_logit missing
    assert fp(None, None, None, 0, 256, 4096, 2048, 1.0, None, None, None, None, None) == lmh.LMH_OK
    assert lib.lmhead_logprob_merge(16, 16, 16, 16, 16, 4, 4096, None, None, None, None) == \
        lmh.LMH_ERR_INVALID_ARG  # out_logprob missing
    assert lib.lmhead_logprob_merge(None, None, None, None, None, 0, 4096, None, None, None,
                                    None) == lmh.LMH_OK
    assert lib.lmhead_engine_gemm(16, 16, 8, 8, 8, 4, 16, None) == lmh.LMH_ERR_INVALID_ARG
    assert lib.lmhead_selftest_wait_timeout(10, None) == lmh.LMH_ERR_INVALID_ARG


def test_noalloc_argument_errors_are_reported_without_a_launch(lib):
    # lmhead_logprob_fwd_noalloc checks its arguments before any CUDA call;
    # fake, never dereferenced addresses.
    def call(**kw):
        a = dict(hidden=16, weight=16, labels=16, T=4, H=256, V=4096, s=1.0, lp=16, ent=None,
                 lse=None)
        a.update(kw)
        return lib.lmhead_logprob_fwd_noalloc(a["hidden"], a["weight"], a["labels"], a["T"],
                                              a["H"], a["V"], a["s"], a["lp"], a["ent"], a["lse"],
                                              None)

    before = lib.lmhead_kernel_launches()
    big = 2147483392 + 1  # one past LMH_MAX_DIM
    assert call(T=-1) == lmh.LMH_ERR_INVALID_ARG
    assert call(T=big) == lmh.LMH_ERR_INVALID_ARG
    assert call(V=0) == lmh.LMH_ERR_INVALID_ARG
    assert call(V=big) == lmh.LMH_ERR_INVALID_ARG
    assert call(H=0) == lmh.LMH_ERR_INVALID_ARG
    assert call(H=big + 7) == lmh.LMH_ERR_INVALID_ARG
    assert call(H=12) == lmh.LMH_ERR_ALIGNMENT
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert call(s=bad) == lmh.LMH_ERR_INVALID_ARG
    for name in ("hidden", "weight", "labels", "lp"):
        assert call(**{name: None}) == lmh.LMH_ERR_INVALID_ARG
    assert call(hidden=24) == lmh.LMH_ERR_ALIGNMENT
    assert call(weight=8) == lmh.LMH_ERR_ALIGNMENT
    assert call(labels=18) == lmh.LMH_ERR_ALIGNMENT
    assert call(lp=18) == lmh.LMH_ERR_ALIGNMENT
    assert call(ent=18) == lmh.LMH_ERR_ALIGNMENT
    assert call(lse=18) == lmh.LMH_ERR_ALIGNMENT
    # partials beyond the fixed 16 MiB scratch are refused before any device use
    assert call(T=16384, V=152064) == lmh.LMH_ERR_WORKSPACE
    assert b"scratch" in lib.lmhead_last_error_string()
    assert call(T=0, hidden=None, weight=None, labels=None, lp=None) == lmh.LMH_OK
    assert lib.lmhead_kernel_launches() == before


def test_chunked_shard_and_sum_argument_errors(lib):
    # fake, never dereferenced addresses: each case fails validation first
    before = lib.lmhead_kernel_launches()
    big = (1 << 64) - 1
    ws = lib.lmhead_workspace_size_bwd
    for bad in (0, 100, 129, -128, (1 << 20) + 128):
        assert ws(16384, 3584, 152064, bad) == big
    # a smaller row chunk needs a smaller workspace; 16384 rows match the plain backward
    assert ws(16384, 3584, 152064, 4096) < ws(16384, 3584, 152064, 16384)
    assert ws(16384, 3584, 152064, 16384) == lib.lmhead_workspace_size(lmh.LMH_OP_BWD, 16384,
                                                                      3584, 152064)
    ch = lib.lmhead_logprob_bwd_chunked
    args = [16, 16, 16, 16, None, 16, None, 4, 256, 4096, 1.0, 128, 16, 16, 256, 1 << 30, None]
    assert ch(*args[:11], 100, *args[12:]) == lmh.LMH_ERR_INVALID_ARG
    assert ch(*args[:11], 0, *args[12:]) == lmh.LMH_ERR_INVALID_ARG
    assert b"row_chunk" in lib.lmhead_last_error_string()
    assert ch(*args[:3], None, None, *args[5:]) == lmh.LMH_ERR_INVALID_ARG  # no upstream grad
    assert ch(*args[:15], 16, None) == lmh.LMH_ERR_WORKSPACE
    sh = lib.lmhead_logprob_bwd_shard
    sargs = [16, 16, 16, 16, None, 16, None, 4, 256, 4096, 1024, 1.0, 16, 16, 256, 1 << 30, None]
    assert sh(*sargs[:5], None, *sargs[6:]) == lmh.LMH_ERR_INVALID_ARG  # no whole-vocab lse
    assert sh(*sargs[:4], 16, 16, None, *sargs[7:]) == lmh.LMH_ERR_INVALID_ARG  # gH w/o entropy
    assert sh(*sargs[:10], -1, *sargs[11:]) == lmh.LMH_ERR_INVALID_ARG
    assert sh(*sargs[:12], 24, *sargs[13:]) == lmh.LMH_ERR_ALIGNMENT  # grad_hidden_part
    sr = lib.lmhead_sum_ranks_bf16
    assert sr(16, 0, 10, 16, None) == lmh.LMH_ERR_INVALID_ARG
    assert sr(16, 2, -1, 16, None) == lmh.LMH_ERR_INVALID_ARG
    assert sr(None, 2, 10, 16, None) == lmh.LMH_ERR_INVALID_ARG
    assert sr(None, 2, 0, None, None) == lmh.LMH_OK
    assert lib.lmhead_kernel_launches() == before


def test_binding_refuses_a_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        lmh.library(str(tmp_path / "nope.so"))

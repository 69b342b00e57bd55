"""Batch-invariant LM-head token log-probabilities on GB300 (sm_103a).

A thin ctypes binding over ``liblmhead.so`` (C ABI declared in
``include/lmhead.h``). The functions keep the C names; they take torch
tensors, check dtypes/devices, allocate outputs and workspace with torch when
they are not given, and pass raw device pointers and the current CUDA stream
to the library. Every step of the computation runs in the library's CUDA
kernels: there is no Python, PyTorch or CPU path for any of them, and a
missing library raises instead of falling back.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from ._build import LIB_PATH, build  # noqa: F401

LMH_OK = 0
LMH_ERR_INVALID_ARG = 1
LMH_ERR_ALIGNMENT = 2
LMH_ERR_WORKSPACE = 3
LMH_ERR_UNSUPPORTED_DEVICE = 4
LMH_ERR_LAUNCH = 5
LMH_ERR_DEVICE_TIMEOUT = 6
ERROR_NAMES = {
    0: "LMH_OK",
    1: "LMH_ERR_INVALID_ARG",
    2: "LMH_ERR_ALIGNMENT",
    3: "LMH_ERR_WORKSPACE",
    4: "LMH_ERR_UNSUPPORTED_DEVICE",
    5: "LMH_ERR_LAUNCH",
    6: "LMH_ERR_DEVICE_TIMEOUT",
}

LMH_OP_FWD = 0
LMH_OP_BWD = 1
LMH_OP_LOGITS = 2

# Exported C symbols and their signatures (argtypes, restype).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
SIGNATURES = {
    "lmhead_workspace_size": ([ctypes.c_int, _I64, _I64, _I64], ctypes.c_size_t),
    "lmhead_logprob_fwd": ([_P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P, _P, ctypes.c_size_t, _P],
                           ctypes.c_int),
    "lmhead_logprob_bwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P, ctypes.c_size_t,
                            _P], ctypes.c_int),
    "logprob_from_logits": ([_P, _P, _I64, _I64, _F, _P, _P, _P, _P], ctypes.c_int),
    "lmhead_logprob_fwd_stats": ([_P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P, _P, _P,
                                  ctypes.c_size_t, _P], ctypes.c_int),
    "logprob_from_logits_stats": ([_P, _P, _I64, _I64, _F, _P, _P, _P, _P, _P], ctypes.c_int),
    "logprob_from_logits_div": ([_P, _P, _I64, _I64, _F, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "lmhead_logprob_fwd_partials": ([_P, _P, _P, _I64, _I64, _I64, _I64, _F, _P, _P, _P, _P, _P],
                                    ctypes.c_int),
    "lmhead_logprob_merge": ([_P, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P], ctypes.c_int),
    "lmhead_logprob_fwd_host": ([_P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _P, ctypes.c_size_t, _P, _P], ctypes.c_int),
    "lmhead_last_error_string": ([], ctypes.c_char_p),
    "lmhead_abi_version": ([], ctypes.c_int),
    "lmhead_kernel_launches": ([], ctypes.c_ulonglong),
    "lmhead_timing_enable": ([ctypes.c_int], ctypes.c_int),
    "lmhead_timing_read": ([ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                            ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "lmhead_timing_kind_name": ([ctypes.c_int], ctypes.c_char_p),
    "lmhead_device_status": ([_P, ctypes.POINTER(ctypes.c_uint)], ctypes.c_int),
    "lmhead_selftest_wait_timeout": ([ctypes.c_uint64, _P], ctypes.c_int),
    "lmhead_selftest_division": ([_F, ctypes.POINTER(ctypes.c_int), _P], ctypes.c_int),
    "lmhead_engine_gemm": ([_P, _P, _I64, _I64, _I64, ctypes.c_int, _P, _P], ctypes.c_int),
    "lmhead_logprob_entropy_bwd": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P,
                                    ctypes.c_size_t, _P], ctypes.c_int),
    "lmhead_logprob_fwd_noalloc": ([_P, _P, _P, _I64, _I64, _I64, _F, _P, _P, _P, _P],
                                   ctypes.c_int),
    "lmhead_logprob_bwd_chunked": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _I64, _P, _P,
                                    _P, ctypes.c_size_t, _P], ctypes.c_int),
    "lmhead_workspace_size_bwd": ([_I64, _I64, _I64, _I64], ctypes.c_size_t),
    "lmhead_logprob_bwd_shard": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, _P, _P,
                                  _P, ctypes.c_size_t, _P], ctypes.c_int),
    "lmhead_sum_ranks_bf16": ([_P, _I64, _I64, _P, _P], ctypes.c_int),
}

_lib_handle: Optional[ctypes.CDLL] = None


class LMHeadError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


def library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblmhead.so (built by ``build()``); raises if it is missing."""
    global _lib_handle
    if _lib_handle is not None and path is None:
        return _lib_handle
    p = path or os.environ.get("LMHEAD_LIB") or str(LIB_PATH)
    if not os.path.exists(p):
        raise RuntimeError(f"liblmhead.so not found at {p}; run invariant_lm_head_gb300.build()")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib_handle = lib
    return lib


def _check(fn: str, rc: int) -> None:
    if rc != LMH_OK:
        msg = library().lmhead_last_error_string().decode(errors="replace")
        raise LMHeadError(fn, rc, msg)


def _torch():
    import torch

    return torch


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, name: str, dtype, device, ndim: int):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def lmhead_workspace_size(op: int, T: int, H: int, V: int) -> int:
    n = library().lmhead_workspace_size(op, T, H, V)
    if n == ctypes.c_size_t(-1).value:
        _check("lmhead_workspace_size", LMH_ERR_INVALID_ARG)
    return n


def _workspace(op, T, H, V, workspace, device):
    torch = _torch()
    need = lmhead_workspace_size(op, T, H, V)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def lmhead_logprob_fwd(hidden, weight, labels, inv_temperature: float = 1.0, *, out_logprob=None,
                       out_entropy=None, out_lse=None, want_entropy: bool = True,
                       want_lse: bool = False, workspace=None, stream=None):
    """Fused LM-head forward. Returns (logprob, entropy or None, lse or None), f32 [T]."""
    return _fwd("lmhead_logprob_fwd", hidden, weight, labels, inv_temperature, out_logprob,
                out_entropy, out_lse, None, want_entropy, want_lse, False, workspace, stream)[:3]


def lmhead_logprob_fwd_stats(hidden, weight, labels, inv_temperature: float = 1.0, *,
                             out_logprob=None, out_entropy=None, out_lse=None, out_sum_p2=None,
                             want_entropy: bool = True, want_lse: bool = False, workspace=None,
                             stream=None):
    """Fused forward with sum_pi_squared. Returns (logprob, entropy, lse, sum_p2)."""
    return _fwd("lmhead_logprob_fwd_stats", hidden, weight, labels, inv_temperature, out_logprob,
                out_entropy, out_lse, out_sum_p2, want_entropy, want_lse, True, workspace, stream)


def lmhead_logprob_fwd_host(hidden_host, weight_host, labels_host, inv_temperature: float = 1.0,
                            *, hidden, weight, labels, out_logprob=None, out_entropy=None,
                            out_lse=None, out_logprob_host=None, out_entropy_host=None,
                            want_entropy: bool = True, want_lse: bool = True, workspace=None,
                            stream=None, copy_stream=None):
    """Fused forward from host inputs, copies overlapped with the forward.

    hidden_host, weight_host, labels_host are CPU tensors (page-locked for the
    copies to overlap); hidden, weight, labels are device tensors of the same
    shapes that the call fills. out_logprob_host / out_entropy_host (CPU f32
    [T] or None) receive the results in stream order. copy_stream is a
    torch.cuda.Stream or None (the library's own). Returns (logprob, entropy
    or None, lse or None) on the device.
    """
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight, "weight", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    cpu = torch.device("cpu")
    _need(hidden_host, "hidden_host", torch.bfloat16, cpu, 2)
    _need(weight_host, "weight_host", torch.bfloat16, cpu, 2)
    _need(labels_host, "labels_host", torch.int32, cpu, 1)
    T, H = hidden.shape
    V = weight.shape[0]
    if (tuple(hidden_host.shape) != (T, H) or tuple(weight_host.shape) != (V, H)
            or weight.shape[1] != H or labels.shape[0] != T or labels_host.shape[0] != T):
        raise ValueError("shape mismatch between the host and device inputs")
    for t, n in ((out_logprob_host, "out_logprob_host"), (out_entropy_host, "out_entropy_host")):
        if t is not None:
            _need(t, n, torch.float32, cpu, 1)
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_entropy is None and (want_entropy or out_entropy_host is not None):
        out_entropy = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    ws, ws_bytes = _workspace(LMH_OP_FWD, T, H, V, workspace, dev)
    cs = None if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    rc = library().lmhead_logprob_fwd_host(
        _ptr(hidden_host), _ptr(weight_host), _ptr(labels_host), T, H, V, float(inv_temperature),
        _ptr(hidden), _ptr(weight), _ptr(labels), _ptr(out_logprob), _ptr(out_entropy),
        _ptr(out_lse), _ptr(out_logprob_host), _ptr(out_entropy_host), _ptr(ws), ws_bytes,
        _stream_ptr(stream), cs)
    _check("lmhead_logprob_fwd_host", rc)
    return out_logprob, out_entropy, out_lse


def _fwd(name, hidden, weight, labels, inv_temperature, out_logprob, out_entropy, out_lse,
         out_sum_p2, want_entropy, want_lse, want_sum_p2, workspace, stream):
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight, "weight", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    T, H = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != H or labels.shape[0] != T:
        raise ValueError("shape mismatch between hidden, weight and labels")
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_entropy is None and want_entropy:
        out_entropy = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if out_sum_p2 is None and want_sum_p2:
        out_sum_p2 = torch.empty(T, dtype=torch.float32, device=dev)
    ws, ws_bytes = _workspace(LMH_OP_FWD, T, H, V, workspace, dev)
    lib = library()
    args = [_ptr(hidden), _ptr(weight), _ptr(labels), T, H, V, float(inv_temperature),
            _ptr(out_logprob), _ptr(out_entropy), _ptr(out_lse)]
    if name == "lmhead_logprob_fwd_stats":
        args.append(_ptr(out_sum_p2))
    rc = getattr(lib, name)(*args, _ptr(ws), ws_bytes, _stream_ptr(stream))
    _check(name, rc)
    return out_logprob, out_entropy, out_lse, out_sum_p2


def lmhead_logprob_bwd(hidden, weight, labels, grad_logprob, inv_temperature: float = 1.0, *,
                       lse=None, grad_hidden=None, grad_weight=None, workspace=None, stream=None):
    """Fused backward. Returns (grad_hidden bf16 [T, H], grad_weight f32 [V, H])."""
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight, "weight", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    _need(grad_logprob, "grad_logprob", torch.float32, dev, 1)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev, 1)
    T, H = hidden.shape
    V = weight.shape[0]
    if grad_hidden is None:
        grad_hidden = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if grad_weight is None:
        grad_weight = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws, ws_bytes = _workspace(LMH_OP_BWD, T, H, V, workspace, dev)
    rc = library().lmhead_logprob_bwd(_ptr(hidden), _ptr(weight), _ptr(labels), _ptr(grad_logprob),
                                      _ptr(lse), T, H, V, float(inv_temperature), _ptr(grad_hidden),
                                      _ptr(grad_weight), _ptr(ws), ws_bytes, _stream_ptr(stream))
    _check("lmhead_logprob_bwd", rc)
    return grad_hidden, grad_weight


def lmhead_logprob_entropy_bwd(hidden, weight, labels, grad_logprob, grad_entropy,
                               inv_temperature: float = 1.0, *, lse=None, entropy=None,
                               grad_hidden=None, grad_weight=None, workspace=None, stream=None):
    """Backward of sum g*logprob + gH*entropy. Returns (grad_hidden bf16, grad_weight f32)."""
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight, "weight", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    for t, n in ((grad_logprob, "grad_logprob"), (grad_entropy, "grad_entropy"), (lse, "lse"),
                 (entropy, "entropy")):
        if t is not None:
            _need(t, n, torch.float32, dev, 1)
    T, H = hidden.shape
    V = weight.shape[0]
    if grad_hidden is None:
        grad_hidden = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if grad_weight is None:
        grad_weight = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws, ws_bytes = _workspace(LMH_OP_BWD, T, H, V, workspace, dev)
    rc = library().lmhead_logprob_entropy_bwd(
        _ptr(hidden), _ptr(weight), _ptr(labels), _ptr(grad_logprob), _ptr(grad_entropy),
        _ptr(lse), _ptr(entropy), T, H, V, float(inv_temperature), _ptr(grad_hidden),
        _ptr(grad_weight), _ptr(ws), ws_bytes, _stream_ptr(stream))
    _check("lmhead_logprob_entropy_bwd", rc)
    return grad_hidden, grad_weight


def lmhead_workspace_size_bwd(T: int, H: int, V: int, row_chunk: int) -> int:
    """Workspace bytes of lmhead_logprob_bwd_chunked."""
    n = library().lmhead_workspace_size_bwd(T, H, V, row_chunk)
    if n == ctypes.c_size_t(-1).value:
        _check("lmhead_workspace_size_bwd", LMH_ERR_INVALID_ARG)
    return n


def lmhead_logprob_bwd_chunked(hidden, weight, labels, grad_logprob, inv_temperature: float = 1.0,
                               *, row_chunk: int, grad_entropy=None, lse=None, entropy=None,
                               grad_hidden=None, grad_weight=None, workspace=None, stream=None):
    """Backward with a chosen row chunk (bounded workspace). Returns (grad_hidden, grad_weight)."""
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight, "weight", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    for t, n in ((grad_logprob, "grad_logprob"), (grad_entropy, "grad_entropy"), (lse, "lse"),
                 (entropy, "entropy")):
        if t is not None:
            _need(t, n, torch.float32, dev, 1)
    T, H = hidden.shape
    V = weight.shape[0]
    if grad_hidden is None:
        grad_hidden = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if grad_weight is None:
        grad_weight = torch.empty(V, H, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(lmhead_workspace_size_bwd(T, H, V, row_chunk), 16),
                                dtype=torch.uint8, device=dev)
    rc = library().lmhead_logprob_bwd_chunked(
        _ptr(hidden), _ptr(weight), _ptr(labels), _ptr(grad_logprob), _ptr(grad_entropy),
        _ptr(lse), _ptr(entropy), T, H, V, float(inv_temperature), int(row_chunk),
        _ptr(grad_hidden), _ptr(grad_weight), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("lmhead_logprob_bwd_chunked", rc)
    return grad_hidden, grad_weight


def lmhead_logprob_bwd_shard(hidden, weight_shard, labels, grad_logprob, lse, v_offset: int,
                             inv_temperature: float = 1.0, *, grad_entropy=None, entropy=None,
                             grad_hidden_part=None, grad_weight=None, workspace=None, stream=None):
    """One vocab shard's backward (see include/lmhead.h).

    lse (and entropy, with grad_entropy) are the whole vocabulary's, f32 [T].
    Returns (grad_hidden_part f32 [T, H], grad_weight f32 [V_shard, H]).
    """
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight_shard, "weight_shard", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    for t, n in ((grad_logprob, "grad_logprob"), (grad_entropy, "grad_entropy"), (lse, "lse"),
                 (entropy, "entropy")):
        if t is not None:
            _need(t, n, torch.float32, dev, 1)
    T, H = hidden.shape
    V = weight_shard.shape[0]
    if grad_hidden_part is None:
        grad_hidden_part = torch.empty(T, H, dtype=torch.float32, device=dev)
    if grad_weight is None:
        grad_weight = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws, ws_bytes = _workspace(LMH_OP_BWD, T, H, V, workspace, dev)
    rc = library().lmhead_logprob_bwd_shard(
        _ptr(hidden), _ptr(weight_shard), _ptr(labels), _ptr(grad_logprob), _ptr(grad_entropy),
        _ptr(lse), _ptr(entropy), T, H, V, int(v_offset), float(inv_temperature),
        _ptr(grad_hidden_part), _ptr(grad_weight), _ptr(ws), ws_bytes, _stream_ptr(stream))
    _check("lmhead_logprob_bwd_shard", rc)
    return grad_hidden_part, grad_weight


def lmhead_sum_ranks_bf16(parts, *, out=None, stream=None):
    """bf16 of the rank-ordered sum of parts [n, ...] (f32) over its first axis."""
    torch = _torch()
    dev = parts.device
    if not isinstance(parts, torch.Tensor) or parts.dtype != torch.float32:
        raise TypeError("parts must be a float32 tensor")
    if parts.device != dev or not parts.is_contiguous() or parts.dim() < 2:
        raise ValueError("parts must be a contiguous tensor [n, ...]")
    n = parts.shape[0]
    count = parts[0].numel()
    if out is None:
        out = torch.empty(parts.shape[1:], dtype=torch.bfloat16, device=dev)
    if out.dtype != torch.bfloat16 or out.numel() != count or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of parts[0]'s size")
    rc = library().lmhead_sum_ranks_bf16(_ptr(parts), n, count, _ptr(out), _stream_ptr(stream))
    _check("lmhead_sum_ranks_bf16", rc)
    return out


def logprob_from_logits(logits, labels, inv_temperature: float = 1.0, *, out_logprob=None,
                        out_entropy=None, out_lse=None, want_entropy: bool = True,
                        want_lse: bool = False, stream=None):
    """Sampler formula on bf16 logits [T, V]. Returns (logprob, entropy or None, lse or None)."""
    return _logits("logprob_from_logits", logits, labels, inv_temperature, out_logprob,
                   out_entropy, out_lse, None, want_entropy, want_lse, False, stream)[:3]


def logprob_from_logits_stats(logits, labels, inv_temperature: float = 1.0, *, out_logprob=None,
                              out_entropy=None, out_lse=None, out_sum_p2=None,
                              want_entropy: bool = True, want_lse: bool = False, stream=None):
    """Sampler formula with sum_pi_squared. Returns (logprob, entropy, lse, sum_p2)."""
    return _logits("logprob_from_logits_stats", logits, labels, inv_temperature, out_logprob,
                   out_entropy, out_lse, out_sum_p2, want_entropy, want_lse, True, stream)


def logprob_from_logits_div(logits, labels, temperature=1.0, *, out_logprob=None,
                            out_entropy=None, out_lse=None, out_sum_p2=None,
                            want_entropy: bool = True, want_lse: bool = False,
                            want_sum_p2: bool = False, stream=None):
    """Sampler formula with the temperature as an fp32 division, z = logits / t.

    temperature is a float (one t for every row) or an f32 tensor [T] of
    per-row temperatures on the logits' device. Returns (logprob, entropy,
    lse, sum_p2), the ones not asked for None.
    """
    torch = _torch()
    row_t = None
    t = 1.0
    if isinstance(temperature, torch.Tensor):
        _need(temperature, "temperature", torch.float32, logits.device, 1)
        if temperature.shape[0] != logits.shape[0]:
            raise ValueError("temperature must have one value per row")
        row_t = temperature
    else:
        t = float(temperature)
    return _logits("logprob_from_logits_div", logits, labels, t, out_logprob, out_entropy,
                   out_lse, out_sum_p2, want_entropy, want_lse, want_sum_p2, stream, row_t=row_t)


def _logits(name, logits, labels, inv_temperature, out_logprob, out_entropy, out_lse, out_sum_p2,
            want_entropy, want_lse, want_sum_p2, stream, row_t=None):
    torch = _torch()
    dev = logits.device
    _need(logits, "logits", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    T, V = logits.shape
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_entropy is None and want_entropy:
        out_entropy = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None and want_lse:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if out_sum_p2 is None and want_sum_p2:
        out_sum_p2 = torch.empty(T, dtype=torch.float32, device=dev)
    args = [_ptr(logits), _ptr(labels), T, V, float(inv_temperature)]
    if name == "logprob_from_logits_div":
        args.append(_ptr(row_t))
    args += [_ptr(out_logprob), _ptr(out_entropy), _ptr(out_lse)]
    if name in ("logprob_from_logits_stats", "logprob_from_logits_div"):
        args.append(_ptr(out_sum_p2))
    rc = getattr(library(), name)(*args, _stream_ptr(stream))
    _check(name, rc)
    return out_logprob, out_entropy, out_lse, out_sum_p2


def lmhead_logprob_fwd_partials(hidden, weight_shard, labels, v_offset: int,
                                inv_temperature: float = 1.0, *, part_m, part_s, part_u,
                                label_logit, stream=None):
    """One vocab shard's forward statistics (see include/lmhead.h).

    part_m, part_s, part_u: f32 [ceil(V_shard / 1024), T] views into the
    whole-vocabulary planes at chunk v_offset / 1024; label_logit f32 [T].
    """
    torch = _torch()
    dev = hidden.device
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(weight_shard, "weight_shard", torch.bfloat16, dev, 2)
    _need(labels, "labels", torch.int32, dev, 1)
    T, H = hidden.shape
    V = weight_shard.shape[0]
    n = -(-V // 1024)
    for t, nm in ((part_m, "part_m"), (part_s, "part_s"), (part_u, "part_u")):
        _need(t, nm, torch.float32, dev, 2)
        if tuple(t.shape) != (n, T):
            raise ValueError(f"{nm} must be [{n}, {T}]")
    _need(label_logit, "label_logit", torch.float32, dev, 1)
    rc = library().lmhead_logprob_fwd_partials(
        _ptr(hidden), _ptr(weight_shard), _ptr(labels), T, H, V, int(v_offset),
        float(inv_temperature), _ptr(part_m), _ptr(part_s), _ptr(part_u), _ptr(label_logit),
        _stream_ptr(stream))
    _check("lmhead_logprob_fwd_partials", rc)


def lmhead_logprob_merge(part_m, part_s, part_u, label_logit, labels, V: int, *,
                         out_logprob=None, out_entropy=None, out_lse=None, stream=None):
    """Merge whole-vocabulary planes into (logprob, entropy, lse), f32 [T]."""
    torch = _torch()
    dev = labels.device
    T = labels.shape[0]
    out_logprob = torch.empty(T, device=dev) if out_logprob is None else out_logprob
    out_entropy = torch.empty(T, device=dev) if out_entropy is None else out_entropy
    out_lse = torch.empty(T, device=dev) if out_lse is None else out_lse
    n = -(-int(V) // 1024)
    for t, nm in ((part_m, "part_m"), (part_s, "part_s"), (part_u, "part_u")):
        _need(t, nm, torch.float32, dev, 2)
        if tuple(t.shape) != (n, T):
            raise ValueError(f"{nm} must be [{n}, {T}]")
    rc = library().lmhead_logprob_merge(
        _ptr(part_m), _ptr(part_s), _ptr(part_u), _ptr(label_logit), _ptr(labels), T, int(V),
        _ptr(out_logprob), _ptr(out_entropy), _ptr(out_lse), _stream_ptr(stream))
    _check("lmhead_logprob_merge", rc)
    return out_logprob, out_entropy, out_lse


_LOGPROB_FN = None
# Row chunk of the autograd backward (lmhead_logprob_bwd_chunked): at H = 3584,
# V = 152064 its workspace is 1.4 GB instead of 5.6 GB for 16384 rows.
AUTOGRAD_ROW_CHUNK = 4096


def _logprob_function():
    """The autograd Function behind lmhead_logprob, built on first use (torch
    is imported lazily so that the module loads without it)."""
    global _LOGPROB_FN
    if _LOGPROB_FN is not None:
        return _LOGPROB_FN
    torch = _torch()

    class _LMHeadLogprob(torch.autograd.Function):
        @staticmethod
        def forward(ctx, hidden, weight, labels, inv_temperature):
            lp, ent, lse = lmhead_logprob_fwd(hidden, weight, labels, inv_temperature,
                                              want_lse=True)
            ctx.save_for_backward(hidden, weight, labels, lse, ent)
            ctx.inv_temperature = inv_temperature
            ctx.set_materialize_grads(False)
            return lp, ent

        @staticmethod
        def backward(ctx, grad_logprob, grad_entropy):
            hidden, weight, labels, lse, ent = ctx.saved_tensors
            if grad_logprob is None and grad_entropy is None:
                return None, None, None, None
            s = ctx.inv_temperature
            g = None if grad_logprob is None else grad_logprob.float().contiguous()
            ge = None if grad_entropy is None else grad_entropy.float().contiguous()
            # rows in chunks of AUTOGRAD_ROW_CHUNK: a quarter of the default
            # backward's workspace, at no measurable cost in time
            gh, gw = lmhead_logprob_bwd_chunked(hidden, weight, labels, g, s,
                                                row_chunk=AUTOGRAD_ROW_CHUNK, grad_entropy=ge,
                                                lse=lse, entropy=ent if ge is not None else None)
            gw_out = None
            if ctx.needs_input_grad[1]:
                # the fp32 sum rounded once to the weight's bf16 by the library
                gw_out = lmhead_sum_ranks_bf16(gw.view(1, *gw.shape))
            del gw
            return (gh if ctx.needs_input_grad[0] else None, gw_out, None, None)

    _LOGPROB_FN = _LMHeadLogprob
    return _LOGPROB_FN


def lmhead_logprob(hidden, weight, labels, inv_temperature: float = 1.0):
    """Differentiable fused LM-head log-probs: (logprob, entropy), f32 [T].

    Forward is lmhead_logprob_fwd; backward is lmhead_logprob_bwd, or
    lmhead_logprob_entropy_bwd when the entropy output also receives a
    gradient. hidden bf16 [T, H] and weight bf16 [V, H] get bf16 gradients
    (grad_weight is accumulated in fp32 by the library and rounded once to
    bf16 by it; call lmhead_logprob_bwd directly to keep it in fp32). The
    backward runs in row chunks of AUTOGRAD_ROW_CHUNK. labels int32 [T] get
    none.
    """
    return _logprob_function().apply(hidden, weight, labels, float(inv_temperature))


def lmhead_kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(library().lmhead_kernel_launches())


def lmhead_timing_enable(on: bool = True) -> None:
    """Start (and clear) or stop per-launch event timing inside the library."""
    _check("lmhead_timing_enable", library().lmhead_timing_enable(1 if on else 0))


def lmhead_timing_read(capacity: int = 1 << 16):
    """[(kernel kind name, milliseconds)] for the launches recorded since enabling."""
    kinds = (ctypes.c_int * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = ctypes.c_int(0)
    lib = library()
    _check("lmhead_timing_read", lib.lmhead_timing_read(kinds, ms, capacity, ctypes.byref(n)))
    return [(lib.lmhead_timing_kind_name(kinds[i]).decode(), float(ms[i])) for i in range(n.value)]


def lmhead_device_status(stream=None) -> int:
    """Synchronise the stream; return the device status word (raises on a timeout bit)."""
    bits = ctypes.c_uint(0)
    rc = library().lmhead_device_status(_stream_ptr(stream), ctypes.byref(bits))
    _check("lmhead_device_status", rc)
    return bits.value


def lmhead_selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> int:
    """Run the bounded-wait self-test; returns the library's status code (6 expected)."""
    return library().lmhead_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream))


def lmhead_selftest_division(temperature: float, stream=None) -> int:
    """Number of bf16 inputs whose quotient in the division form differs from
    IEEE fp32 division by ``temperature`` (0 = bit-exact)."""
    n = ctypes.c_int(-1)
    _check("lmhead_selftest_division",
           library().lmhead_selftest_division(float(temperature), ctypes.byref(n),
                                              _stream_ptr(stream)))
    return int(n.value)


def lmhead_engine_gemm(A, B, out=None, a_kmajor: bool = True, b_kmajor: bool = True,
                       stream=None):
    """D = sum_k A[m,k] B[n,k] through the tensor-core engine; D f32 [M, N].

    A is [M, K] when a_kmajor else [K, M]; B is [N, K] when b_kmajor else [K, N].
    """
    torch = _torch()
    dev = A.device
    _need(A, "A", torch.bfloat16, dev, 2)
    _need(B, "B", torch.bfloat16, dev, 2)
    M, K = A.shape if a_kmajor else (A.shape[1], A.shape[0])
    N = B.shape[0] if b_kmajor else B.shape[1]
    layout = (0 if a_kmajor else 1) | (0 if b_kmajor else 2)
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=dev)
    rc = library().lmhead_engine_gemm(_ptr(A), _ptr(B), M, N, K, layout, _ptr(out),
                                      _stream_ptr(stream))
    _check("lmhead_engine_gemm", rc)
    return out

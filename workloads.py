"""Seeded synthetic inputs for the LM-head log-prob workloads.

This module is shared by the tests, the benchmark and the oracle's self-tests.
It holds no part of the log-prob arithmetic: it only draws random numbers,
rounds them to bf16 and describes the workload shapes.

Every array is drawn with numpy's PCG64 generator, whose streams are the same
on every platform, in fixed row blocks that each get their own child seed.
The result therefore depends only on the seed and the shape, never on the
number of threads that fill the blocks.

bf16 values are returned as numpy ``uint16`` bit patterns (round to nearest,
ties to even, from the fp32 draw); ``as_torch_bf16`` views them as a
``torch.bfloat16`` tensor without copying.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_BLOCK_ELEMS = 1 << 22  # elements per independently seeded block


# --------------------------------------------------------------------------
# bf16 helpers (storage format only)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits.

    Inputs here are finite draws, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_torch_bf16(bits: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16)).view(torch.bfloat16)


# --------------------------------------------------------------------------
# block-parallel seeded draws
# --------------------------------------------------------------------------

def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def _normal_bf16(seed: int, stream: int, shape: tuple[int, ...], std: float,
                 row_offset_std: float = 0.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws; optional per-row N(0, row_offset_std^2)
    offset added in fp32 before rounding."""
    rows = shape[0]
    cols = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((rows, cols), dtype=np.uint16)
    rows_per_block = max(1, _BLOCK_ELEMS // max(cols, 1))
    nblocks = (rows + rows_per_block - 1) // rows_per_block
    seeds = np.random.SeedSequence([seed, stream]).spawn(nblocks + 1)
    offsets = None
    if row_offset_std:
        offsets = np.random.Generator(np.random.PCG64(seeds[-1])).standard_normal(rows).astype(np.float32)
        offsets *= np.float32(row_offset_std)

    def fill(b: int) -> None:
        r0 = b * rows_per_block
        r1 = min(rows, r0 + rows_per_block)
        g = np.random.Generator(np.random.PCG64(seeds[b]))
        x = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        x *= np.float32(std)
        if offsets is not None:
            x += offsets[r0:r1, None]
        out[r0:r1] = f32_to_bf16_bits(x)

    if nblocks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nblocks)))
    return out.reshape(shape)


def _uniform_labels(seed: int, stream: int, n: int, V: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return g.integers(0, V, size=n, dtype=np.int64).astype(np.int32)


def _normal_f32(seed: int, stream: int, n: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return g.standard_normal(n, dtype=np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class FusedWorkload:
    """hidden bf16[T,H] ~ N(0,1), weight bf16[V,H] ~ N(0, w_std^2), labels U[0,V),
    upstream grad f32[T] ~ N(0,1); inv_temperature is an fp32 scalar."""

    name: str
    T: int
    H: int
    V: int
    inv_temperature: float
    seed: int
    w_std: float = 0.02
    seq_lens: tuple[int, ...] | None = None  # packed variable-length batch


@dataclasses.dataclass(frozen=True)
class LogitsWorkload:
    """logits bf16[T,V] ~ N(0, std^2) plus a per-row N(0, 1) offset; labels U[0,V)."""

    name: str
    T: int
    V: int
    inv_temperature: float
    seed: int
    std: float = 2.0
    row_offset_std: float = 1.0


def packed_lengths(seed: int = 5, n: int = 32, lo: int = 128, hi: int = 4096) -> tuple[int, ...]:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))
    return tuple(int(x) for x in g.integers(lo, hi + 1, size=n))


def f32(x: float) -> float:
    """Round a Python float to the nearest fp32 value."""
    return float(np.float32(x))


TINY = FusedWorkload("tiny fused forward T=64 H=256 V=4096", 64, 256, 4096, 1.0, seed=1)
LOGITS = LogitsWorkload("sampler formula on bf16 logits T=8192 V=152064", 8192, 152064, 1.0, seed=2)
LLAMA = FusedWorkload("fused forward T=4096 H=4096 V=32000", 4096, 4096, 32000, 1.0, seed=3)
QWEN = FusedWorkload("fused forward+backward T=16384 H=3584 V=152064 inv_T=1/0.7",
                     16384, 3584, 152064, f32(1.0 / 0.7), seed=4)
_PACKED_LENS = packed_lengths()
PACKED = FusedWorkload("packed varlen forward+backward 32 seqs H=5120 V=152064",
                       int(sum(_PACKED_LENS)), 5120, 152064, 1.0, seed=5, seq_lens=_PACKED_LENS)


def fused_inputs(w: FusedWorkload, T: int | None = None, H: int | None = None, V: int | None = None):
    """Return dict(hidden=uint16[T,H], weight=uint16[V,H], labels=int32[T], grad=f32[T]).

    ``T``, ``H``, ``V`` override the workload's sizes (same distributions, same
    seed) for reduced-size parity cases.
    """
    T = w.T if T is None else T
    H = w.H if H is None else H
    V = w.V if V is None else V
    return dict(
        hidden=_normal_bf16(w.seed, 1, (T, H), 1.0),
        weight=_normal_bf16(w.seed, 2, (V, H), w.w_std),
        labels=_uniform_labels(w.seed, 3, T, V),
        grad=_normal_f32(w.seed, 4, T),
    )


def logits_inputs(w: LogitsWorkload, T: int | None = None, V: int | None = None):
    """Return dict(logits=uint16[T,V], labels=int32[T])."""
    T = w.T if T is None else T
    V = w.V if V is None else V
    return dict(
        logits=_normal_bf16(w.seed, 1, (T, V), w.std, row_offset_std=w.row_offset_std),
        labels=_uniform_labels(w.seed, 3, T, V),
    )


def random_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    return _normal_bf16(seed, 7, tuple(shape), std)


def random_labels(seed: int, n: int, V: int) -> np.ndarray:
    return _uniform_labels(seed, 8, n, V)


def random_f32(seed: int, n: int) -> np.ndarray:
    return _normal_f32(seed, 9, n)

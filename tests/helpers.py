"""Shared helpers for the GPU tests: device copies of seeded inputs, oracle
calls on the same bits, and the tolerances.

Tolerances (stated by the method's accuracy target): log-probs, entropy and
lse within 1e-3 absolute of the fp64 oracle; grad_hidden and grad_weight
within 1e-2 relative Frobenius error. Batch invariance is bitwise.
"""

import numpy as np

import workloads as W

ATOL_LOGPROB = 1e-3
RTOL_FROB_GRAD = 1e-2


def dev():
    import torch

    return torch.device("cuda:0")


def to_dev_bf16(bits):
    return W.as_torch_bf16(bits).to(dev())


def to_dev(arr):
    import torch

    return torch.from_numpy(np.ascontiguousarray(arr)).to(dev())


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def rel_frob(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_abs(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)))


def fused_case(seed, T, H, V, w_std=0.02, oov=()):
    """Seeded fused inputs (uint16 bits / int32 / f32) with chosen rows made out-of-vocab."""
    hidden = W.random_bf16(seed, (T, H), 1.0)
    weight = W.random_bf16(seed + 1000, (V, H), w_std)
    labels = W.random_labels(seed, T, V)
    grad = W.random_f32(seed, T)
    for i, lab in oov:
        labels[i] = lab
    return hidden, weight, labels, grad


def bitwise_equal(a, b):
    import torch

    return torch.equal(a.view(torch.int32), b.view(torch.int32))

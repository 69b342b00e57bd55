"""Pure-Python loop restatement of the oracle, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (see ``oracle/lmhead_oracle.py``). Every sum is an
explicit loop with ``math.fsum`` so that the BLAS-backed float64 oracle can be
checked against a second, independently written form on small inputs.

Definitions followed: the sampler formula (verl pull request "batch-invariant
actor forward and sampler log-prob formula", the ``logprobs_from_logits_sampler``
diff), the out-of-vocab convention and fused projection (SkyRL pull request
"Triton backend for fused LM-head log-prob", summary and the out-of-vocab
gradient fix), temperature applied as an fp32 factor (verl page, temperature
comment).
"""

from __future__ import annotations

import math

import numpy as np


def _s(inv_temperature: float) -> float:
    return float(np.float32(inv_temperature))


def forward(hidden, weight, labels, inv_temperature):
    """Lists (logprob, entropy, lse) for each row, from explicit loops."""
    s = _s(inv_temperature)
    T, H = len(hidden), len(hidden[0])
    V = len(weight)
    lp_out, ent_out, lse_out = [], [], []
    for t in range(T):
        z = [s * math.fsum(float(hidden[t][h]) * float(weight[v][h]) for h in range(H))
             for v in range(V)]
        m = max(z)
        lse = m + math.log(math.fsum(math.exp(zv - m) for zv in z))
        ent = -math.fsum(math.exp(zv - lse) * (zv - lse) for zv in z)
        lab = int(labels[t])
        lp = z[lab] - lse if 0 <= lab < V else 0.0
        lp_out.append(lp)
        ent_out.append(ent)
        lse_out.append(lse)
    return lp_out, ent_out, lse_out


def sum_p2(hidden, weight, inv_temperature):
    """List of sum_v p_v^2 per row, from explicit loops."""
    s = _s(inv_temperature)
    T, H = len(hidden), len(hidden[0])
    V = len(weight)
    out = []
    for t in range(T):
        z = [s * math.fsum(float(hidden[t][h]) * float(weight[v][h]) for h in range(H))
             for v in range(V)]
        m = max(z)
        lse = m + math.log(math.fsum(math.exp(zv - m) for zv in z))
        out.append(math.fsum(math.exp(2.0 * (zv - lse)) for zv in z))
    return out


def backward(hidden, weight, labels, grad, inv_temperature, grad_entropy=None):
    """Nested lists (grad_hidden [T][H], grad_weight [V][H]) from explicit loops.

    With grad_entropy, d(gH * entropy)/dz_v = -gH * p_v * (z_v - lse + entropy)
    is added to each row's logit gradient.
    """
    s = _s(inv_temperature)
    T, H = len(hidden), len(hidden[0])
    V = len(weight)
    dl = []
    for t in range(T):
        z = [s * math.fsum(float(hidden[t][h]) * float(weight[v][h]) for h in range(H))
             for v in range(V)]
        m = max(z)
        lse = m + math.log(math.fsum(math.exp(zv - m) for zv in z))
        g = float(grad[t])
        ge = 0.0 if grad_entropy is None else float(grad_entropy[t])
        ent = -math.fsum(math.exp(zv - lse) * (zv - lse) for zv in z)
        lab = int(labels[t])
        row = []
        for v in range(V):
            onehot = 1.0 if v == lab else 0.0
            p = math.exp(z[v] - lse)
            row.append(s * (g * (onehot - p) - ge * p * (z[v] - lse + ent)))
        dl.append(row)
    gh = [[math.fsum(dl[t][v] * float(weight[v][h]) for v in range(V)) for h in range(H)]
          for t in range(T)]
    gw = [[math.fsum(dl[t][v] * float(hidden[t][h]) for t in range(T)) for h in range(H)]
          for v in range(V)]
    return gh, gw

"""fp64 CPU oracle for batch-invariant LM-head token log-probabilities.

TEST INFRASTRUCTURE ONLY. This module is the independent reference that the
CUDA library is checked against. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never does, and it
shares no code with the library.

What it computes (all arithmetic in float64 over the bf16 values exactly as
stored, each step written out as the pages define it):

* The sampler formula, from the verl pull request "batch-invariant actor
  forward and sampler log-prob formula" (the ``logprobs_from_logits_sampler``
  diff): log-probabilities are an fp32 ``log_softmax`` over the full
  vocabulary followed by a gather of the label. Here the log-softmax is taken
  in float64: ``logprob[t] = z[t, label[t]] - lse[t]`` with
  ``lse[t] = M + log(sum_v exp(z[t, v] - M))`` and ``M = max_v z[t, v]``.
* Row chunking does not change a row's value (same page, the review note that
  a per-row or chunked log-softmax plus gather equals one large one): every
  function below works row by row; no quantity mixes rows.
* Temperature (same page, the temperature-order comment and its table): the
  logits are scaled in fp32 precision by the fp32 temperature, never by a
  bf16-rounded one. Most entry points take ``inv_temperature`` as an fp32
  scalar, so ``z = s * logits`` with ``s`` the fp32 value widened to float64.
  The sampler-parity form divides instead: ``z = fp32(logits) / fp32(t)``,
  the quotient rounded to fp32 as the table's "cast first, then divide" fixes.
* The fused projection, from the SkyRL pull request "Triton backend for fused
  LM-head log-prob" (summary: the vocab projection folded into the chunked
  log-prob, fp32 softmax math): ``logits[t, v] = sum_h hidden[t, h] *
  weight[v, h]`` (an ``nn.Linear`` weight of shape ``[V, H]``).
* Out-of-vocabulary labels (same SkyRL page, the out-of-vocab gradient fix):
  the forward log-prob of a position whose label is outside ``[0, V)`` is 0;
  its backward keeps the ``-softmax * g`` term and drops the one-hot term.
* Entropy of the same temperature-scaled distribution whose log-probs are
  returned (verl page, review note that an entropy taken elsewhere is not the
  entropy of the fp32 log-softmax): ``entropy[t] = -sum_v p log p`` with
  ``p = exp(z - lse)``, natural log.
* ``sum_pi_squared`` (verl page, the review note listing entropy and
  sum_pi_squared as the per-token statistics still taken from the logits):
  ``sum_p2[t] = sum_v p[t, v]^2`` of the same distribution.
* Backward of ``sum_t g[t] * logprob[t]`` with respect to the projection:
  ``dz = g * (onehot - p)``, ``dlogit = s * dz``, ``grad_hidden = dlogit @
  weight``, ``grad_weight = dlogit^T @ hidden``.
* Optional entropy term (the SkyRL page notes entropy under the fused head is
  metric-only until its gradient is wired): for ``sum_t gH[t] * entropy[t]``,
  ``dH/dz_j = -p_j * (log p_j + H) = -p_j * (z_j - lse + H)``, added to ``dz``
  before the temperature factor.

Pins (tests/test_oracle_pins.py): closed forms (uniform rows, two-value rows,
one-hot-dominant rows), invariants (sum of probabilities, sign, entropy
bounds, gradient row sums), library routines on CPU (``torch.log_softmax`` in
float64, ``scipy.special.logsumexp``, ``scipy.stats.entropy``, torch autograd),
central finite differences, and a pure-Python loop restatement
(``oracle/loops.py``) on tiny shapes.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "fp32_scalar",
    "scaled_logits",
    "row_lse_entropy",
    "sampler_logprob",
    "row_sum_p2",
    "fused_sum_p2",
    "fused_forward",
    "logprob_from_logits",
    "divided_logits",
    "logprob_from_logits_div",
    "dlogits",
    "dlogits_entropy",
    "fused_backward",
    "fused_forward_rows",
    "fused_grad_hidden_rows",
    "grad_weight_from_rows",
]


def fp32_scalar(x: float) -> float:
    """The fp32 value of a temperature factor, widened to float64."""
    return float(np.float32(x))


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def scaled_logits(hidden, weight, inv_temperature: float) -> np.ndarray:
    """z[t, v] = s * sum_h hidden[t, h] * weight[v, h]   (float64, [T, V])."""
    h = _f64(hidden)
    w = _f64(weight)
    return fp32_scalar(inv_temperature) * (h @ w.T)


def row_lse_entropy(z) -> tuple[np.ndarray, np.ndarray]:
    """Per row: log-sum-exp and the entropy of softmax(z), natural log."""
    z = _f64(z)
    m = z.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z - m).sum(axis=1))
    logp = z - lse[:, None]
    p = np.exp(logp)
    entropy = -(p * logp).sum(axis=1)
    return lse, entropy


def row_sum_p2(z) -> np.ndarray:
    """Per row: sum_v p_v^2 with p = softmax(z)."""
    z = _f64(z)
    lse, _ = row_lse_entropy(z)
    p = np.exp(z - lse[:, None])
    return (p * p).sum(axis=1)


def sampler_logprob(z, labels) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """log_softmax over the full row, then gather of the label.

    Returns (logprob, entropy, lse), each float64 [T]. A label outside [0, V)
    gives logprob 0; entropy and lse are still those of the full row.
    """
    z = _f64(z)
    labels = np.asarray(labels, dtype=np.int64)
    T, V = z.shape
    lse, entropy = row_lse_entropy(z)
    inside = (labels >= 0) & (labels < V)
    logprob = np.zeros(T, dtype=np.float64)
    rows = np.nonzero(inside)[0]
    logprob[rows] = z[rows, labels[rows]] - lse[rows]
    return logprob, entropy, lse


def fused_forward(hidden, weight, labels, inv_temperature: float):
    """(logprob, entropy, lse) of the fused LM head: z = s * hidden @ weight^T."""
    return sampler_logprob(scaled_logits(hidden, weight, inv_temperature), labels)


def fused_sum_p2(hidden, weight, inv_temperature: float) -> np.ndarray:
    """sum_v p[t, v]^2 of the fused LM head's distribution, per row."""
    return row_sum_p2(scaled_logits(hidden, weight, inv_temperature))


def logprob_from_logits(logits, labels, inv_temperature: float = 1.0):
    """(logprob, entropy, lse) of the sampler formula on given logits, z = s * logits."""
    return sampler_logprob(fp32_scalar(inv_temperature) * _f64(logits), labels)


def divided_logits(logits, temperature) -> np.ndarray:
    """z = fp32(logits) / fp32(t), the quotient rounded to fp32, as float64 [T, V].

    The verl page's temperature-order table fixes this step's precision: the
    logits are cast to fp32 first and then divided by the fp32 temperature.
    numpy's float32 division is the IEEE round-to-nearest quotient, so ``z``
    holds exactly the fp32 values a sampler that divides by the temperature
    sees. ``temperature`` is a scalar or one value per row.
    """
    x = np.asarray(logits, dtype=np.float32)
    t = np.asarray(temperature, dtype=np.float32)
    if t.ndim == 1:
        t = t[:, None]
    return (x / t).astype(np.float64)


def logprob_from_logits_div(logits, labels, temperature):
    """(logprob, entropy, lse) of the sampler formula on z = fp32(logits) / fp32(t).

    The log-softmax and everything after it are float64, as in
    ``sampler_logprob``; only the division is taken at the fp32 precision the
    pages fix for it.
    """
    return sampler_logprob(divided_logits(logits, temperature), labels)


def dlogits(z, labels, grad, inv_temperature: float, lse=None) -> np.ndarray:
    """Gradient of sum_t g[t] * logprob[t] with respect to the unscaled logits.

    dz[t, v] = g[t] * (onehot[t, v] - p[t, v]); the one-hot term is absent for
    a label outside [0, V). The result is s * dz (chain rule through z = s * logits).
    """
    z = _f64(z)
    T, V = z.shape
    g = _f64(grad)
    labels = np.asarray(labels, dtype=np.int64)
    if lse is None:
        lse, _ = row_lse_entropy(z)
    p = np.exp(z - _f64(lse)[:, None])
    dz = -g[:, None] * p
    inside = (labels >= 0) & (labels < V)
    rows = np.nonzero(inside)[0]
    dz[rows, labels[rows]] += g[rows]
    return fp32_scalar(inv_temperature) * dz


def dlogits_entropy(z, grad_entropy, inv_temperature: float) -> np.ndarray:
    """Gradient of sum_t gH[t] * entropy[t] with respect to the unscaled logits.

    d entropy / d z_j = -p_j * (z_j - lse + entropy); times s (z = s * logits).
    """
    z = _f64(z)
    gh = _f64(grad_entropy)
    lse, ent = row_lse_entropy(z)
    p = np.exp(z - lse[:, None])
    dz = -gh[:, None] * p * (z - lse[:, None] + ent[:, None])
    return fp32_scalar(inv_temperature) * dz


def fused_backward(hidden, weight, labels, grad, inv_temperature: float, grad_entropy=None):
    """(grad_hidden [T, H], grad_weight [V, H]) in float64.

    Differentiates sum_t grad[t] * logprob[t] (+ sum_t grad_entropy[t] * entropy[t]
    when grad_entropy is given).
    """
    h = _f64(hidden)
    w = _f64(weight)
    z = scaled_logits(h, w, inv_temperature)
    dl = dlogits(z, labels, grad, inv_temperature)
    if grad_entropy is not None:
        dl = dl + dlogits_entropy(z, grad_entropy, inv_temperature)
    return dl @ w, dl.T @ h


# ---------------------------------------------------------------------------
# Row-sampled forms for shapes too large for the full computation. Rows are
# independent, so each sampled row is computed exactly as in the full form.
# ---------------------------------------------------------------------------

def _row_blocks(rows, block: int = 32):
    rows = np.asarray(rows, dtype=np.int64)
    for i in range(0, len(rows), block):
        yield rows[i:i + block]


def fused_forward_rows(hidden, weight, labels, inv_temperature: float, rows):
    """(logprob, entropy, lse) for the listed rows only."""
    w = _f64(weight)
    labels = np.asarray(labels, dtype=np.int64)
    out = [[], [], []]
    for r in _row_blocks(rows):
        z = fp32_scalar(inv_temperature) * (_f64(hidden[r]) @ w.T)
        for k, x in enumerate(sampler_logprob(z, labels[r])):
            out[k].append(x)
    return tuple(np.concatenate(x) if x else np.zeros(0) for x in out)


def fused_grad_hidden_rows(hidden, weight, labels, grad, inv_temperature: float, rows,
                           grad_entropy=None):
    """grad_hidden for the listed rows only, [len(rows), H]."""
    w = _f64(weight)
    labels = np.asarray(labels, dtype=np.int64)
    g = _f64(grad)
    out = []
    for r in _row_blocks(rows):
        z = fp32_scalar(inv_temperature) * (_f64(hidden[r]) @ w.T)
        dl = dlogits(z, labels[r], g[r], inv_temperature)
        if grad_entropy is not None:
            dl = dl + dlogits_entropy(z, _f64(grad_entropy)[r], inv_temperature)
        out.append(dl @ w)
    return np.concatenate(out) if out else np.zeros((0, w.shape[1]))


def grad_weight_from_rows(hidden, weight, labels, grad, inv_temperature: float, rows,
                          vocab_rows=None, grad_entropy=None):
    """sum over the listed rows t of dlogit[t, :]^T hidden[t, :], [V, H].

    Equals the full grad_weight when grad[t] = 0 for every row not listed.
    With ``vocab_rows`` only those rows of the result are formed
    ([len(vocab_rows), H]); the softmax still runs over the full vocabulary.
    """
    w = _f64(weight)
    labels = np.asarray(labels, dtype=np.int64)
    g = _f64(grad)
    out_rows = w.shape[0] if vocab_rows is None else len(vocab_rows)
    acc = np.zeros((out_rows, w.shape[1]), dtype=np.float64)
    for r in _row_blocks(rows):
        h = _f64(hidden[r])
        z = fp32_scalar(inv_temperature) * (h @ w.T)
        dl = dlogits(z, labels[r], g[r], inv_temperature)
        if grad_entropy is not None:
            dl = dl + dlogits_entropy(z, _f64(grad_entropy)[r], inv_temperature)
        if vocab_rows is not None:
            dl = dl[:, np.asarray(vocab_rows, dtype=np.int64)]
        acc += dl.T @ h
    return acc

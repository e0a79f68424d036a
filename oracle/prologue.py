"""Maps around the recurrence, fp64 numpy (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs use
this module; it shares no code with the CUDA library.

Written from the first page ("Scrivere meglio nella memoria: gate e delta
rule"):

* keys and queries: DeltaNet absorbs the feature map into the projections and
  applies a SiLU followed by an L2 normalisation, per token (opening section);
* the write strength of the delta rule is a sigmoid of the input,
  beta_t = sigmoid(w^T x_t), which keeps it between 0 and 1 (section
  "Correggere: la delta rule");
* the read-out of DeltaNet is stabilised by an RMSNorm on the output (same
  section);
* the scalar decay alpha_t is produced from the input in Mamba-2 (section
  "Dimenticare: i gate"); the page leaves its parametrisation open, so the two
  used by the workloads are provided: sigmoid(a) and exp(-c softplus(a));
* the diagonal gate of GLA (same section) is a sigmoid raised to 1/tau with
  tau = 16 (a temperature that pushes the gates towards 1): sigmoid(a)^c,
  c = 1/tau, applied per key channel.

Each map takes the pre-activation values (after the projection, which is not
part of this library) and returns the values the recurrence consumes.
"""
from __future__ import annotations

import numpy as np

from . import recurrent

# flags, the same bits as the library's lr_fuse_flags
QK_SILU_L2 = 1
BETA_SIGMOID = 2
ALPHA_SIGMOID = 4
ALPHA_SOFTPLUS = 8
O_RMSNORM = 16
ALPHA_SIGMOID_POW = 32

L2_EPS = 1e-12   # x / max(||x||, eps): the pages give no epsilon
RMS_EPS = 1e-6   # o / sqrt(mean(o^2) + eps): the pages give no epsilon


def silu(x):
    """x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def sigmoid(x):
    """1 / (1 + e^-x), evaluated without overflow for either sign."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softplus(x):
    """ln(1 + e^x), evaluated without overflow."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def l2_normalise(x, eps=L2_EPS):
    """Each vector along the last axis divided by max(its L2 norm, eps)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, eps)


def silu_l2(x):
    """The key/query map: SiLU, then L2 normalisation per token."""
    return l2_normalise(silu(x))


def _per_head(c, ndim):
    c = np.asarray(c, dtype=np.float64)
    if c.ndim == 1:
        c = c.reshape((1, -1) + (1,) * (ndim - 2))
    return c


def sigmoid_pow_gate(a, c):
    """alpha = sigmoid(a)^c (GLA: c = 1/tau).  `a` is [B, H, T(, dk)] or
    [N, H(, dk)]; `c` a scalar or one value per head [H]."""
    a = np.asarray(a, dtype=np.float64)
    return np.exp(-_per_head(c, a.ndim) * softplus(-a))


def softplus_gate(a, c):
    """alpha = exp(-c softplus(a)), in (0, 1) for c > 0.  `a` is [B, H, T]
    (prefill) or [N, H] (decode); `c` a scalar or one value per head [H]."""
    a = np.asarray(a, dtype=np.float64)
    return np.exp(-_per_head(c, a.ndim) * softplus(a))


def rmsnorm(o, weight=None, eps=RMS_EPS):
    """Each vector along the last axis divided by sqrt(mean of squares + eps),
    then multiplied channel-wise by `weight` (ones when None)."""
    o = np.asarray(o, dtype=np.float64)
    r = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    if weight is not None:
        r = r * np.asarray(weight, dtype=np.float64)
    return r


def apply_prologue(flags, q, k, alpha, beta, alpha_scale=1.0):
    """The values the recurrence consumes, from the pre-activation inputs.
    ALPHA_SIGMOID takes precedence over ALPHA_SOFTPLUS (the library rejects
    both together)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if flags & QK_SILU_L2:
        q, k = silu_l2(q), silu_l2(k)
    if alpha is not None:
        alpha = np.asarray(alpha, dtype=np.float64)
        if flags & ALPHA_SIGMOID:
            alpha = sigmoid(alpha)
        elif flags & ALPHA_SOFTPLUS:
            alpha = softplus_gate(alpha, alpha_scale)
        elif flags & ALPHA_SIGMOID_POW:
            alpha = sigmoid_pow_gate(alpha, alpha_scale)
    if beta is not None:
        beta = np.asarray(beta, dtype=np.float64)
        if flags & BETA_SIGMOID:
            beta = sigmoid(beta)
    return q, k, alpha, beta


def fused(mode, flags, q, k, v, alpha=None, beta=None, S0=None, alpha_scale=1.0,
          norm_weight=None, norm_eps=RMS_EPS, threads: int = 0):
    """Prologue, the recurrence (:func:`oracle.recurrent`), then the output
    RMSNorm when ``flags & O_RMSNORM``.  Returns (o, S_T) like the recurrence."""
    q, k, alpha, beta = apply_prologue(flags, q, k, alpha, beta, alpha_scale)
    o, st = recurrent(mode, q, k, v, alpha, beta, S0, threads=threads)
    if flags & O_RMSNORM:
        o = rmsnorm(o, norm_weight, norm_eps)
    return o, st

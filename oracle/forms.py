"""The parallel and chunkwise forms of the recurrence, fp64 numpy (test infrastructure).

Only ``tests/`` use these.  They exist to pin the recurrent oracle and the
chunk algebra: the pages state that the three forms give exactly the same
result ("Le architetture lineari: RetNet, RWKV, xLSTM", section "RetNet: la
retention e le sue tre forme", Fig. 16.5 and the text around it).

Notation per sequence (tokens t = 0..T-1, all products empty -> 1):

* decay weight  D[t, i] = prod_{j=i+1..t} alpha_j  for i <= t, else 0
  (contribution written at step i and seen at step t, first page section
  "Dimenticare: i gate");
* initial-state weight  g[t] = prod_{j=0..t} alpha_j;
* pseudo-values u_t (first page, section "Correggere: la delta rule", the WY
  representation S_t = sum_i u_i k_i^T): for the delta rows
      u_t = beta_t (v_t - g[t] S_0 k_t - sum_{i<t} D[t,i] (k_i . k_t) u_i),
  a lower-triangular system in the u's; for the rows without delta u_t = v_t.
  (The gated version is the same WY representation with the decay weights
  carried on every coupling, as the Gated DeltaNet section says it extends.)
* output  o_t = g[t] S_0 q_t + sum_{i<=t} D[t,i] (k_i . q_t) u_i
  i.e. O = diag(g) Q S_0^T + (Q K^T (.) D) U;
* final state  S_T = g[T-1] S_0 + sum_i D[T-1,i] u_i k_i^T.

The decay weights are formed as explicit running products of alpha, not in
log space.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from . import USES_ALPHA, USES_BETA


def _decay_weights(alpha_seq):
    """D[t,i] and g[t] from the per-token gates of one sequence."""
    T = alpha_seq.shape[0]
    D = np.zeros((T, T))
    g = np.empty(T)
    for t in range(T):
        w = 1.0
        D[t, t] = 1.0
        for i in range(t - 1, -1, -1):
            w *= alpha_seq[i + 1]
            D[t, i] = w
        g[t] = (g[t - 1] if t > 0 else 1.0) * alpha_seq[t]
    return D, g


def _parallel_one(mode, q, k, v, a, b, S0):
    T, dk = q.shape
    dv = v.shape[1]
    if T == 0:
        return np.zeros((0, dv)), S0.copy()
    alpha_seq = a if USES_ALPHA[mode] else np.ones(T)
    D, g = _decay_weights(alpha_seq)
    if USES_BETA[mode]:
        KK = k @ k.T                               # k_i . k_t
        A = np.tril(b[:, None] * D * KK.T, -1)     # A[t,i] = beta_t D[t,i] (k_i.k_t), i < t
        rhs = b[:, None] * (v - g[:, None] * (k @ S0.T))
        U = solve_triangular(np.eye(T) + A, rhs, lower=True, unit_diagonal=True)
    else:
        U = v.copy()
    O = g[:, None] * (q @ S0.T) + ((q @ k.T) * D) @ U
    ST = g[T - 1] * S0 + U.T @ (D[T - 1][:, None] * k)
    return O, ST


def _as_f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def parallel_form(mode, q, k, v, alpha=None, beta=None, S0=None):
    """Masked quadratic form over whole sequences.  Shapes as in ``oracle.recurrent``."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    alpha, beta, S0 = _as_f64(alpha), _as_f64(beta), _as_f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    O = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dv, dk))
    for bb in range(B):
        for hh in range(H):
            s0 = S0[bb, hh] if S0 is not None else np.zeros((dv, dk))
            a = alpha[bb, hh] if alpha is not None else None
            b = beta[bb, hh] if beta is not None else None
            O[bb, hh], ST[bb, hh] = _parallel_one(mode, q[bb, hh], k[bb, hh], v[bb, hh], a, b, s0)
    return O, ST


def chunked_form(mode, q, k, v, alpha=None, beta=None, S0=None, chunk=64):
    """Chunkwise form: the parallel form inside blocks of ``chunk`` tokens,
    only the end-of-block state carried from one block to the next; the last
    block may be shorter."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    alpha, beta, S0 = _as_f64(alpha), _as_f64(beta), _as_f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    O = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dv, dk))
    for bb in range(B):
        for hh in range(H):
            S = S0[bb, hh].copy() if S0 is not None else np.zeros((dv, dk))
            for s in range(0, T, chunk):
                e = min(T, s + chunk)
                a = alpha[bb, hh, s:e] if alpha is not None else None
                b = beta[bb, hh, s:e] if beta is not None else None
                O[bb, hh, s:e], S = _parallel_one(mode, q[bb, hh, s:e], k[bb, hh, s:e],
                                                  v[bb, hh, s:e], a, b, S)
            ST[bb, hh] = S
    return O, ST

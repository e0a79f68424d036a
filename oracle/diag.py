"""Diagonal gate (GLA row), fp64 numpy forms (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs use
this module; it shares no code with the CUDA library.

The recurrence (page "Scrivere meglio nella memoria: gate e delta rule",
section "Dimenticare: i gate", the GLA equation, and the summary table):

    S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T,   alpha_t in (0,1)^{d_k},
    o_t = S_t q_t,

the diagonal multiplying from the right so that column c (key channel c)
decays by alpha_t[c].  The definition itself is ``oracle.recurrent`` with
mode DIAG_DECAY (plain C, one token at a time).  The two forms here exist to
pin the algebra the kernels use:

* :func:`parallel_form` -- unrolling the recurrence: what token i wrote
  reaches token t with channel c weighted by the product of alpha_j[c] for
  j = i+1..t (the gates section states this for the scalar gate; per channel
  it is the same product taken channel by channel).
* :func:`chunked_form` -- blocks of C tokens, the end-of-block state handed on
  (page "Le architetture lineari", RetNet section, chunkwise form), with the
  second level of blocks that the summary of the first page says GLA needs
  for numerical stability: inside a block the scores of the rows of
  sub-block I are formed relative to the cumulative gate b_I at the last
  token before sub-block I, so every exponent of a query factor is <= 0 and
  every exponent of a key factor that precedes the sub-block is <= 0.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def parallel_form(q, k, v, alpha, S0=None):
    """Brute force over all pairs (tiny T): returns (o, S_T).

    o_t = S0 (q_t * prod_{j<=t} alpha_j) + sum_{i<=t} v_i sum_c q_t[c] k_i[c] prod_{j=i+1..t} alpha_j[c]
    """
    q, k, v, alpha, S0 = _f64(q), _f64(k), _f64(v), _f64(alpha), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    st = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            a = alpha[b, h]
            s0 = np.zeros((dv, dk)) if S0 is None else S0[b, h]
            for t in range(T):
                acc = s0 @ (q[b, h, t] * np.prod(a[: t + 1], axis=0))
                for i in range(t + 1):
                    w = np.prod(a[i + 1: t + 1], axis=0)  # empty product = 1
                    acc = acc + v[b, h, i] * np.sum(q[b, h, t] * k[b, h, i] * w)
                o[b, h, t] = acc
            s = s0 * np.prod(a, axis=0)[None, :]
            for i in range(T):
                s = s + np.outer(v[b, h, i], k[b, h, i] * np.prod(a[i + 1:], axis=0))
            st[b, h] = s
    return o, st


def chunked_form(q, k, v, alpha, S0=None, chunk=64, sub=16):
    """Blocks of ``chunk`` tokens with sub-blocks of ``sub`` tokens: returns
    (o, S_T).  Per block, with G_r the cumulative log-gate from the block start
    (one value per key channel), g_C = e^{G_last}:

      output     O = (Q * e^G) S^T + P V
      scores     P_ri = sum_c q_r[c] k_i[c] e^{G_r[c] - G_i[c]},  i <= r,
                 evaluated per sub-block I as (Q_I * e^{G_r - b_I}) (K * e^{b_I - G_i})^T
      carry      S <- S Diag(g_C) + V^T (K * e^{G_last - G})
    """
    q, k, v, alpha, S0 = _f64(q), _f64(k), _f64(v), _f64(alpha), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    st = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else S0[b, h].copy()
            for t0 in range(0, T, chunk):
                n = min(chunk, T - t0)
                Q, K, V = q[b, h, t0:t0 + n], k[b, h, t0:t0 + n], v[b, h, t0:t0 + n]
                G = np.cumsum(np.log(alpha[b, h, t0:t0 + n]), axis=0)   # [n, dk]
                P = np.zeros((n, n))
                for r0 in range(0, n, sub):
                    r1 = min(n, r0 + sub)
                    ref = G[r0 - 1] if r0 > 0 else np.zeros(dk)         # b_I
                    Qh = Q[r0:r1] * np.exp(G[r0:r1] - ref)               # exponents <= 0
                    Kh = K[:r1] * np.exp(ref - G[:r1])                   # <= 0 before the sub-block
                    Pi = Qh @ Kh.T
                    rows = np.arange(r0, r1)[:, None]
                    cols = np.arange(r1)[None, :]
                    P[r0:r1, :r1] = np.where(cols <= rows, Pi, 0.0)
                O = (Q * np.exp(G)) @ S.T + P @ V
                o[b, h, t0:t0 + n] = O
                S = S * np.exp(G[-1])[None, :] + V.T @ (K * np.exp(G[-1] - G))
            st[b, h] = S
    return o, st

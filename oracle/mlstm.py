"""mLSTM memory, fp64 (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs use
this module; it shares no code with the CUDA library.

Page "Le architetture lineari: RetNet, RWKV, xLSTM", section on xLSTM (the
matrix-memory cell, mLSTM): the scalar-gate row of the summary table with an
exponential write factor and a normaliser,

    C_t = f_t C_{t-1} + i_t v_t k_t^T,   n_t = f_t n_{t-1} + i_t k_t,   i_t = e^{igate_t},
    h_t = C_t q_t / max(|n_t^T q_t|, 1),

and its stabilised form (same section, after the authors' appendix): a
log-space state m_t = max(log f_t + m_{t-1}, igate_t), memory kept as
C~ = e^{-m} C and n~ = e^{-m} n, and the threshold rescaled with them,
h_t = C~ q / max(|n~^T q|, e^{-m_t}), which the page shows is the same output.

* :func:`stabilized` -- the stabilised recurrence in plain C (one token at a
  time, the library's state convention: (C~, n~, m)).
* :func:`plain` -- the definition above in numpy, without the stabiliser
  (the initial memory C_0 = e^{m_0} C~_0, n_0 = e^{m_0} n~_0).
* :func:`chunked_form` -- blocks of C tokens as the kernels compute them: the
  stabiliser of every token first (it depends on the gates only), then per
  block the decay-masked scores weighted by e^{F_t - F_s + igate_s - m_t}, the
  inter-block part weighted by e^{F_t + m_prev - m_t}, and the state and
  normaliser carried with e^{F_C + m_prev - m_C} and e^{F_C - F_s + igate_s - m_C}
  (F the cumulative log forget gate inside the block).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _f64, _load, _ptr


def _lib():
    L = _load()
    if not getattr(L, "_mlstm_ready", False):
        dp = ctypes.POINTER(ctypes.c_double)
        L.gdr_oracle_mlstm.restype = ctypes.c_int
        L.gdr_oracle_mlstm.argtypes = [ctypes.c_int] * 5 + [dp] * 12 + [ctypes.c_int]
        L._mlstm_ready = True
    return L


def stabilized(q, k, v, logf, igate, C0=None, n0=None, m0=None, threads: int = 0):
    """Returns (h [B,H,T,dv], C~_T [B,H,dv,dk], n~_T [B,H,dk], m_T [B,H])."""
    q, k, v, logf, igate = _f64(q), _f64(k), _f64(v), _f64(logf), _f64(igate)
    C0, n0, m0 = _f64(C0), _f64(n0), _f64(m0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    h = np.empty((B, H, T, dv))
    CT = np.empty((B, H, dv, dk))
    nT = np.empty((B, H, dk))
    mT = np.empty((B, H))
    rc = _lib().gdr_oracle_mlstm(B, H, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(logf),
                                 _ptr(igate), _ptr(C0), _ptr(n0), _ptr(m0), _ptr(h), _ptr(CT),
                                 _ptr(nT), _ptr(mT), int(threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_mlstm failed with code {rc}")
    return h, CT, nT, mT


def plain(q, k, v, logf, igate, C0=None, n0=None, m0=None):
    """The definition without the stabiliser: returns (h, C_T, n_T) with the
    unscaled memory C, n."""
    q, k, v, logf, igate = (np.asarray(x, dtype=np.float64) for x in (q, k, v, logf, igate))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    h = np.zeros((B, H, T, dv))
    CT = np.zeros((B, H, dv, dk))
    nT = np.zeros((B, H, dk))
    for b in range(B):
        for hh in range(H):
            if C0 is None:
                C, n = np.zeros((dv, dk)), np.zeros(dk)
            else:
                s = np.exp(float(m0[b, hh]))
                C, n = s * np.asarray(C0[b, hh], float), s * np.asarray(n0[b, hh], float)
            for t in range(T):
                f, i = np.exp(logf[b, hh, t]), np.exp(igate[b, hh, t])
                C = f * C + i * np.outer(v[b, hh, t], k[b, hh, t])
                n = f * n + i * k[b, hh, t]
                h[b, hh, t] = C @ q[b, hh, t] / max(abs(n @ q[b, hh, t]), 1.0)
            CT[b, hh], nT[b, hh] = C, n
    return h, CT, nT


def stabilizer(logf, igate, m0=None):
    """m_t for every token: m_t = max(log f_t + m_{t-1}, igate_t) from m_0
    (-inf for the empty memory)."""
    logf, igate = np.asarray(logf, dtype=np.float64), np.asarray(igate, dtype=np.float64)
    B, H, T = logf.shape
    m = np.empty((B, H, T))
    prev = np.full((B, H), -np.inf) if m0 is None else np.asarray(m0, dtype=np.float64).copy()
    for t in range(T):
        prev = np.maximum(logf[:, :, t] + prev, igate[:, :, t])
        m[:, :, t] = prev
    return m


def chunked_form(q, k, v, logf, igate, C0=None, n0=None, m0=None, chunk=64):
    """Blocks of ``chunk`` tokens (the kernels' algebra); returns the same
    quantities as :func:`stabilized`."""
    q, k, v, logf, igate = (np.asarray(x, dtype=np.float64) for x in (q, k, v, logf, igate))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    m_all = stabilizer(logf, igate, m0)
    h = np.zeros((B, H, T, dv))
    CT = np.zeros((B, H, dv, dk))
    nT = np.zeros((B, H, dk))
    mT = np.zeros((B, H))
    for b in range(B):
        for hh in range(H):
            if C0 is None:
                C, n, m_prev = np.zeros((dv, dk)), np.zeros(dk), -np.inf
            else:
                C, n = np.array(C0[b, hh], float), np.array(n0[b, hh], float)
                m_prev = float(m0[b, hh])
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                Q, K, V = q[b, hh, t0:t1], k[b, hh, t0:t1], v[b, hh, t0:t1]
                F = np.cumsum(logf[b, hh, t0:t1])
                ig = igate[b, hh, t0:t1]
                m = m_all[b, hh, t0:t1]
                with np.errstate(invalid="ignore"):
                    g = np.exp(F + m_prev - m)                     # inter-block weight per row
                W = np.exp((F - m)[:, None] + (ig - F)[None, :])    # e^{F_t - F_s + ig_s - m_t}
                W = np.tril(W)
                P = (Q @ K.T) * W
                num = g[:, None] * (Q @ C.T) + P @ V
                den = g * (Q @ n) + P.sum(axis=1)
                h[b, hh, t0:t1] = num / np.maximum(np.abs(den), np.exp(-m))[:, None]
                kd = np.exp(F[-1] - F + ig - m[-1])
                gC = np.exp(F[-1] + m_prev - m[-1])
                C = gC * C + V.T @ (K * kd[:, None])
                n = gC * n + K.T @ kd
                m_prev = m[-1]
            CT[b, hh], nT[b, hh], mT[b, hh] = C, n, m_prev
    return h, CT, nT, mT

"""Generalised delta rule of RWKV-7 (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s oracle legs use
this module; it shares no code with the CUDA library.

Page "Le architetture lineari: RetNet, RWKV, xLSTM", RWKV section: RWKV-7
adopts a generalised delta rule whose transition is a per-channel decay plus a
rank-one correction, with a normalised removal key decoupled from the write
key and a per-channel in-context learning rate; its eigenvalues can fall
anywhere in [-1, 1].  The extracted page lost the equation itself.  Reading,
in the chapter's convention (S is d_v x d_k, o = S q, transitions multiply
from the right):

    S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) + v_t kw_t^T.

* :func:`recurrent` -- the C recurrence, one value row at a time.
* :func:`matrix_form` -- the same with the transition built as a matrix and
  multiplied (tiny sizes): a second evaluation order of the definition.
* :func:`chunked_form` -- blocks of C tokens as the kernels compute them: with
  u_t = S_{t-1} kappa_t and per-channel cumulative log decays L inside a
  block, u solves (I + A) U = Kdec S0^T + Bk V, and
  O = Qdec S0^T + Qk V - Qb U,  S_C = S0 Diag(e^{L_C}) + V^T Kc - U^T Bc,
  where every decay factor e^{L_t - L_s} (s <= t) is at most 1.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _f64, _load, _ptr


def _lib():
    L = _load()
    if not getattr(L, "_gd_ready", False):
        dp = ctypes.POINTER(ctypes.c_double)
        L.gdr_oracle_gen_delta.restype = ctypes.c_int
        L.gdr_oracle_gen_delta.argtypes = [ctypes.c_int] * 5 + [dp] * 9 + [ctypes.c_int]
        L._gd_ready = True
    return L


def recurrent(q, kw, v, w, kappa, a, S0=None, threads: int = 0):
    """Returns (o [B,H,T,dv], S_T [B,H,dv,dk])."""
    q, kw, v, w, kappa, a, S0 = (_f64(x) for x in (q, kw, v, w, kappa, a, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.empty((B, H, T, dv))
    st = np.empty((B, H, dv, dk))
    rc = _lib().gdr_oracle_gen_delta(B, H, T, dk, dv, _ptr(q), _ptr(kw), _ptr(v), _ptr(w),
                                     _ptr(kappa), _ptr(a), _ptr(S0), _ptr(o), _ptr(st),
                                     int(threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_gen_delta failed with code {rc}")
    return o, st


def matrix_form(q, kw, v, w, kappa, a, S0=None):
    q, kw, v, w, kappa, a = (np.asarray(x, dtype=np.float64) for x in (q, kw, v, w, kappa, a))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    st = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for t in range(T):
                G = np.diag(w[b, h, t]) - np.outer(kappa[b, h, t], a[b, h, t] * kappa[b, h, t])
                S = S @ G + np.outer(v[b, h, t], kw[b, h, t])
                o[b, h, t] = S @ q[b, h, t]
            st[b, h] = S
    return o, st


def chunked_form(q, kw, v, w, kappa, a, S0=None, chunk=32):
    q, kw, v, w, kappa, a = (np.asarray(x, dtype=np.float64) for x in (q, kw, v, w, kappa, a))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    st = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                n = t1 - t0
                Q, K, V = q[b, h, t0:t1], kw[b, h, t0:t1], v[b, h, t0:t1]
                Kp = kappa[b, h, t0:t1]
                Bv = a[b, h, t0:t1] * Kp
                L = np.cumsum(np.log(w[b, h, t0:t1]), axis=0)          # [n, dk]
                Lm = np.vstack([np.zeros((1, dk)), L[:-1]])              # L_{t-1}
                # D[t, s, c] = e^{L_t - L_s}, D0[t, s, c] = e^{L_{t-1} - L_s}, s <= t
                D = np.exp(L[:, None, :] - L[None, :, :])
                D0 = np.exp(Lm[:, None, :] - L[None, :, :])
                lower = np.tril(np.ones((n, n)))
                strict = np.tril(np.ones((n, n)), -1)
                Qk = np.einsum("tc,sc,tsc->ts", Q, K, D) * lower
                Qb = np.einsum("tc,sc,tsc->ts", Q, Bv, D) * lower
                Bk = np.einsum("tc,sc,tsc->ts", Kp, K, D0) * strict
                A = np.einsum("tc,sc,tsc->ts", Kp, Bv, D0) * strict
                Kdec = Kp * np.exp(Lm)
                U = np.linalg.solve(np.eye(n) + A, Kdec @ S.T + Bk @ V)
                O = (Q * np.exp(L)) @ S.T + Qk @ V - Qb @ U
                o[b, h, t0:t1] = O
                dec = np.exp(L[-1][None, :] - L)                         # e^{L_C - L_s}
                S = S * np.exp(L[-1])[None, :] + V.T @ (K * dec) - U.T @ (Bv * dec)
            st[b, h] = S
    return o, st

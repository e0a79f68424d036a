"""Pins of the generalised-delta (RWKV-7) oracle (CPU only).

The page (RWKV section of "Le architetture lineari") gives the ingredients but
its extracted text lost the equation, so the reading
S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) + v_t kw_t^T is pinned
to what the page and the other rows fix: with w = 1, a = beta and kappa = k,
kw = beta k it is the delta rule; with a = 0 it is the diagonal gate (the
page: RWKV-7 keeps the per-channel gate and adds the correction); with a unit
removal key and a uniform rate a, a memory along that key is scaled by 1 - a,
so the eigenvalues cover [-1, 1] (a = 2 reflects, which is what lets the
state keep count); and the blocked algebra of the kernels equals the
recurrence.  Checks take ``rec(q, kw, v, w, kappa, a, S0) -> (o, S_T)`` so
planted mistakes can be run through them.
"""
import numpy as np
import pytest

import oracle
from oracle import DELTA, DIAG_DECAY
from oracle.gen_delta import chunked_form, matrix_form, recurrent

RNG = np.random.default_rng(4)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def pin_delta_rule(rec):
    B, H, T, d, dv = 1, 2, 11, 6, 5
    q, k = RNG.standard_normal((2, B, H, T, d))
    k = _unit(k)
    v = RNG.standard_normal((B, H, T, dv))
    beta = RNG.uniform(0, 1, (B, H, T))
    S0 = RNG.standard_normal((B, H, dv, d))
    bd = np.repeat(beta[..., None], d, axis=-1)
    o1, s1 = rec(q, bd * k, v, np.ones((B, H, T, d)), k, bd, S0)
    o2, s2 = oracle.recurrent(DELTA, q, k, v, None, beta, S0)
    return bool(np.allclose(o1, o2, rtol=1e-11, atol=1e-11) and np.allclose(s1, s2, rtol=1e-11, atol=1e-11))


def pin_diagonal_gate(rec):
    B, H, T, d, dv = 1, 2, 9, 5, 4
    q, k, kap = RNG.standard_normal((3, B, H, T, d))
    v = RNG.standard_normal((B, H, T, dv))
    w = RNG.uniform(0.2, 1, (B, H, T, d))
    S0 = RNG.standard_normal((B, H, dv, d))
    o1, s1 = rec(q, k, v, w, _unit(kap), np.zeros((B, H, T, d)), S0)
    o2, s2 = oracle.recurrent(DIAG_DECAY, q, k, v, w, None, S0)
    return bool(np.allclose(o1, o2, rtol=1e-11, atol=1e-11) and np.allclose(s1, s2, rtol=1e-11, atol=1e-11))


def pin_eigenvalues(rec):
    """A memory u kappa^T with a unit removal key, w = 1, uniform rate a and
    nothing written becomes (1 - a) u kappa^T: eigenvalue 1 - a, -1 for a = 2;
    two reflections with the same key restore any memory."""
    d, dv = 6, 4
    kap = _unit(RNG.standard_normal(d))
    u = RNG.standard_normal(dv)
    S0 = np.outer(u, kap)[None, None]
    z = np.zeros((1, 1, 1, d))
    ok = True
    for av in (0.0, 0.5, 1.0, 1.5, 2.0):
        _, s = rec(z, z, np.zeros((1, 1, 1, dv)), np.ones((1, 1, 1, d)), kap.reshape(1, 1, 1, d),
                   np.full((1, 1, 1, d), av), S0)
        ok &= np.allclose(s[0, 0], (1 - av) * S0[0, 0], rtol=0, atol=1e-13)
    S1 = RNG.standard_normal((1, 1, dv, d))
    z2 = np.zeros((1, 1, 2, d))
    _, s = rec(z2, z2, np.zeros((1, 1, 2, dv)), np.ones((1, 1, 2, d)),
               np.broadcast_to(kap, (1, 1, 2, d)).copy(), np.full((1, 1, 2, d), 2.0), S1)
    ok &= np.allclose(s, S1, rtol=0, atol=1e-12)
    return bool(ok)


def pin_forms(rec):
    B, H, T, dk, dv = 1, 2, 37, 5, 4
    q, kw, kap = RNG.standard_normal((3, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    w = RNG.uniform(0.3, 1, (B, H, T, dk))
    a = RNG.uniform(0, 2, (B, H, T, dk))
    S0 = RNG.standard_normal((B, H, dv, dk))
    args = (q, kw, v, w, _unit(kap), a, S0)
    o, s = rec(*args)
    om, sm = matrix_form(*args)
    ok = np.allclose(o, om, rtol=1e-10, atol=1e-10) and np.allclose(s, sm, rtol=1e-10, atol=1e-10)
    for chunk in (32, 8, 5, 1):
        oc, sc = chunked_form(*args, chunk=chunk)
        ok &= np.allclose(o, oc, rtol=1e-9, atol=1e-9) and np.allclose(s, sc, rtol=1e-9, atol=1e-9)
    return bool(ok)


PINS = (pin_delta_rule, pin_diagonal_gate, pin_eigenvalues, pin_forms)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_gen_delta_pin(pin):
    assert pin(recurrent)


def _rec_np(kind):
    def rec(q, kw, v, w, kappa, a, S0):
        B, H, T, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((B, H, T, dv))
        st = np.zeros((B, H, dv, dk))
        for b in range(B):
            for h in range(H):
                S = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
                for t in range(T):
                    kp, at, wt = kappa[b, h, t], a[b, h, t], w[b, h, t]
                    if kind == "rate_side":      # rate on the removal key instead of the update
                        G = np.diag(wt) - np.outer(at * kp, kp)
                    elif kind == "no_rate":
                        G = np.diag(wt) - np.outer(kp, kp)
                    else:
                        G = np.diag(wt) - np.outer(kp, at * kp)
                    Sp = S
                    if kind == "decay_after":
                        S = (S + np.outer(v[b, h, t], kw[b, h, t])) @ G
                    elif kind == "write_key":    # write with the removal key
                        S = S @ G + np.outer(v[b, h, t], kp)
                    else:
                        S = S @ G + np.outer(v[b, h, t], kw[b, h, t])
                    o[b, h, t] = (Sp if kind == "read_before" else S) @ q[b, h, t]
                st[b, h] = S
        return o, st
    return rec


@pytest.mark.parametrize("kind", ["none", "rate_side", "no_rate", "decay_after", "write_key",
                                  "read_before"])
def test_gen_delta_pins_catch_planted_mistake(kind):
    failed = [p.__name__ for p in PINS if not p(_rec_np(kind))]
    if kind == "none":
        assert not failed, failed
    else:
        assert failed, f"planted mistake {kind} passed every pin"

"""Pins of the mLSTM oracle (CPU only).

Page "Le architetture lineari: RetNet, RWKV, xLSTM", xLSTM section: the matrix
memory C_t = f_t C_{t-1} + i_t v_t k_t^T with i_t = exp(igate_t), the
normaliser n_t = f_t n_{t-1} + i_t k_t, the read h_t = C_t q_t /
max(|n_t^T q_t|, 1); the log-space stabiliser m_t = max(log f_t + m_{t-1},
igate_t) with the threshold rescaled to e^{-m_t} gives the same output, while
keeping the threshold at 1 with the rescaled memory does not.

Checks take ``rec(q, k, v, logf, igate, C0, n0, m0) -> (h, C~_T, n~_T, m_T)``
so that planted mistakes in a numpy copy of the stabilised recurrence can be
run through them too.
"""
import numpy as np
import pytest

import oracle
from oracle import DECAY
from oracle.mlstm import chunked_form, plain, stabilized, stabilizer

RNG = np.random.default_rng(77)


def _inputs(B=1, H=2, T=13, dk=5, dv=4, ig_std=3.0, state=True):
    q, k = RNG.standard_normal((2, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    logf = np.log(1.0 / (1.0 + np.exp(-(3.0 + RNG.standard_normal((B, H, T))))))
    ig = RNG.standard_normal((B, H, T)) * ig_std
    if state:
        C0 = RNG.standard_normal((B, H, dv, dk))
        n0 = RNG.standard_normal((B, H, dk))
        m0 = RNG.standard_normal((B, H))
        return q, k, v, logf, ig, C0, n0, m0
    return q, k, v, logf, ig, None, None, None


def pin_stabilised_equals_plain(rec):
    """The stabilised form returns the plain definition's output, and its
    memory times e^m is the plain memory (page: the factor cancels)."""
    ok = True
    for state in (True, False):
        x = _inputs(state=state)
        h, C, n, m = rec(*x)
        hp, Cp, np_ = plain(*x)
        ok &= np.allclose(h, hp, rtol=1e-10, atol=1e-10)
        s = np.exp(m)[..., None]
        ok &= np.allclose(C * s[..., None], Cp, rtol=1e-10, atol=1e-10)
        ok &= np.allclose(n * s, np_, rtol=1e-10, atol=1e-10)
    return bool(ok)


def pin_one_write(rec):
    """One write with a unit key, read with the same key: n.q = i, so
    h = i v / max(i, 1): v when i >= 1, i v when the threshold is active."""
    ok = True
    k = RNG.standard_normal(6)
    k /= np.linalg.norm(k)
    v = RNG.standard_normal((1, 1, 1, 3))
    for i, want in ((4.0, 1.0), (0.25, 0.25)):
        h, _, _, _ = rec(k.reshape(1, 1, 1, 6), k.reshape(1, 1, 1, 6), v, np.zeros((1, 1, 1)),
                         np.full((1, 1, 1), np.log(i)), None, None, None)
        ok &= np.allclose(h, want * v, rtol=1e-12, atol=1e-14)
    return bool(ok)


def pin_scalar_gate_numerator(rec):
    """With large input gates the threshold never acts and h = (C q)/|n q|,
    where C q is the scalar-gate row with the write scaled by i and n q the
    same row with a single value channel equal to i."""
    x = _inputs(T=9, ig_std=0.5, state=False)
    q, k, v, logf, ig = x[:5]
    ig = ig + 6.0
    h, _, _, _ = rec(q, k, v, logf, ig, None, None, None)
    i = np.exp(ig)
    o, _ = oracle.recurrent(DECAY, q, k, v * i[..., None], np.exp(logf), None, None)
    nq, _ = oracle.recurrent(DECAY, q, k, i[..., None], np.exp(logf), None, None)
    assert np.all(np.abs(nq) > 1.0)
    return bool(np.allclose(h, o / np.abs(nq), rtol=1e-10, atol=1e-12))


def pin_stabiliser(rec):
    """m_t = max(log f_t + m_{t-1}, igate_t): from the empty memory the first
    m is igate_0; with igate = 0 and f = 1 it stays 0; the final m matches."""
    x = _inputs(state=False)
    _, _, _, m = rec(*x)
    ms = stabilizer(x[3], x[4])
    ok = np.allclose(m, ms[:, :, -1], rtol=0, atol=1e-12)
    ok &= np.allclose(ms[:, :, 0], x[4][:, :, 0], rtol=0, atol=0)
    z = np.zeros((1, 1, 5))
    ok &= np.allclose(stabilizer(z, z), 0.0)
    return bool(ok)


def pin_chunked(rec):
    """The kernels' blocked algebra equals the recurrence."""
    ok = True
    x = _inputs(B=1, H=2, T=37, dk=6, dv=5)
    h, C, n, m = rec(*x)
    for chunk in (64, 16, 5, 1):
        hc, Cc, nc, mc = chunked_form(*x, chunk=chunk)
        ok &= np.allclose(h, hc, rtol=1e-9, atol=1e-10) and np.allclose(C, Cc, rtol=1e-9, atol=1e-10)
        ok &= np.allclose(n, nc, rtol=1e-9, atol=1e-10) and np.allclose(m, mc, rtol=0, atol=1e-10)
    return bool(ok)


PINS = (pin_stabilised_equals_plain, pin_one_write, pin_scalar_gate_numerator, pin_stabiliser,
        pin_chunked)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_mlstm_pin(pin):
    assert pin(stabilized)


# ------------------------------------------------------------- planted mistakes

def _rec_np(kind):
    def rec(q, k, v, logf, ig, C0, n0, m0):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, T, dk = q.shape
        dv = v.shape[-1]
        h = np.zeros((B, H, T, dv))
        CT, nT, mT = np.zeros((B, H, dv, dk)), np.zeros((B, H, dk)), np.zeros((B, H))
        for b in range(B):
            for hh in range(H):
                if C0 is None:
                    C, n, m = np.zeros((dv, dk)), np.zeros(dk), -np.inf
                else:
                    C, n, m = np.array(C0[b, hh]), np.array(n0[b, hh]), float(m0[b, hh])
                for t in range(T):
                    lf, g = logf[b, hh, t], ig[b, hh, t]
                    mn = max(lf + m, g)
                    a = np.exp(lf + m - mn) if kind != "drop_m" else np.exp(lf - mn)
                    bb = np.exp(g - mn) if kind != "b_unscaled" else np.exp(g)
                    Cn = a * C + bb * np.outer(v[b, hh, t], k[b, hh, t])
                    nn = (a * n if kind != "n_no_decay" else n) + bb * k[b, hh, t]
                    Cr, nr = (C, n) if kind == "read_before" else (Cn, nn)
                    nq = nr @ q[b, hh, t]
                    thr = 1.0 if kind == "threshold_one" else np.exp(-mn)
                    den = max(nq if kind == "no_abs" else abs(nq), thr)
                    h[b, hh, t] = Cr @ q[b, hh, t] / den
                    C, n, m = Cn, nn, mn
                CT[b, hh], nT[b, hh], mT[b, hh] = C, n, m
        return h, CT, nT, mT
    return rec


@pytest.mark.parametrize("kind", ["none", "threshold_one", "drop_m", "b_unscaled", "n_no_decay",
                                  "read_before", "no_abs"])
def test_mlstm_pins_catch_planted_mistake(kind):
    rec = _rec_np(kind)
    failed = []
    for p in PINS:
        with np.errstate(all="ignore"):
            try:
                if not p(rec):
                    failed.append(p.__name__)
            except (AssertionError, FloatingPointError, ValueError):
                failed.append(p.__name__ + " (raised)")
    if kind == "none":
        assert not failed, failed
    else:
        assert failed, f"planted mistake {kind} passed every pin"

"""Pins of the diagonal-gate (GLA) oracle to what the pages fix (CPU only).

Page "Scrivere meglio nella memoria: gate e delta rule", section "Dimenticare:
i gate": S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T with one gate per key
channel, multiplying from the right so that key-channel columns decay;
alpha -> 1 keeps a channel (pure accumulation in the limit), alpha -> 0 clears
it; the scalar gate is the special case of equal channels.

Each check is a function of ``rec(q, k, v, alpha, S0) -> (o, S_T)`` so the
same checks run against the oracle (all must pass) and against planted
mistakes in a numpy copy of the recurrence (each must fail at least one).
"""
import numpy as np
import pytest

import oracle
from oracle import DECAY, DIAG_DECAY, LINEAR
from oracle.diag import chunked_form, parallel_form

RNG = np.random.default_rng(31)


def ref(q, k, v, alpha, S0):
    return oracle.recurrent(DIAG_DECAY, q, k, v, alpha, None, S0)


def pin_scalar_reduction(rec):
    """Equal gates on every channel are the scalar-gate row."""
    B, H, T, dk, dv = 2, 2, 9, 5, 3
    q, k = RNG.standard_normal((2, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    a = RNG.uniform(0.3, 1.0, (B, H, T))
    S0 = RNG.standard_normal((B, H, dv, dk))
    o1, s1 = rec(q, k, v, np.repeat(a[..., None], dk, axis=-1), S0)
    o2, s2 = oracle.recurrent(DECAY, q, k, v, a, None, S0)
    return np.allclose(o1, o2, rtol=1e-12, atol=1e-12) and np.allclose(s1, s2, rtol=1e-12, atol=1e-12)


def pin_unit_gate(rec):
    """alpha = 1 on every channel is pure accumulation."""
    B, H, T, dk, dv = 1, 2, 7, 4, 6
    q, k = RNG.standard_normal((2, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    o1, s1 = rec(q, k, v, np.ones((B, H, T, dk)), None)
    o2, s2 = oracle.recurrent(LINEAR, q, k, v, None, None, None)
    return np.allclose(o1, o2, rtol=1e-12, atol=1e-12) and np.allclose(s1, s2, rtol=1e-12, atol=1e-12)


def pin_zero_gate_clears_channel(rec):
    """alpha[t, c] = 0 clears column c before token t writes: afterwards the
    column holds exactly v_t k_t[c]; the other columns are untouched by it."""
    dk = dv = 4
    T = 3
    q = RNG.standard_normal((1, 1, T, dk))
    k = RNG.standard_normal((1, 1, T, dk))
    v = RNG.standard_normal((1, 1, T, dv))
    a = np.ones((1, 1, T, dk))
    a[0, 0, 2, 1] = 0.0
    S0 = RNG.standard_normal((1, 1, dv, dk))
    _, s = rec(q, k, v, a, S0)
    _, s_lin = oracle.recurrent(LINEAR, q, k, v, None, None, S0)
    col_ok = np.allclose(s[0, 0, :, 1], v[0, 0, 2] * k[0, 0, 2, 1], rtol=0, atol=1e-14)
    others = [0, 2, 3]
    return bool(col_ok and np.allclose(s[0, 0][:, others], s_lin[0, 0][:, others], rtol=0, atol=1e-13))


def pin_columns_decay(rec):
    """With nothing written, S_t = S0 Diag(prod alpha): column c (key channel
    c) decays by its own product, so reading with q = e_c returns column c of
    S0 times that product (value channels are not decayed differently)."""
    dk = dv = 4
    T = 4
    a = RNG.uniform(0.2, 0.9, (1, 1, T, dk))
    S0 = RNG.standard_normal((1, 1, dv, dk))
    z = np.zeros((1, 1, T, dk))
    ok = True
    for c in range(dk):
        q = np.zeros((1, 1, T, dk))
        q[..., c] = 1.0
        o, s = rec(q, z, np.zeros((1, 1, T, dv)), a, S0)
        want = S0[0, 0, :, c][None, :] * np.cumprod(a[0, 0, :, c])[:, None]
        ok &= np.allclose(o[0, 0], want, rtol=1e-13, atol=1e-15)
    ok &= np.allclose(s[0, 0], S0[0, 0] * np.prod(a[0, 0], axis=0)[None, :], rtol=1e-13, atol=1e-15)
    return bool(ok)


def pin_decay_weight(rec):
    """What token 0 wrote reaches token t weighted, channel by channel, by the
    gates of tokens 1..t (not its own gate): o_t = v_0 (q_t . (k_0 * prod_{j=1..t} alpha_j))."""
    dk, dv, T = 5, 3, 6
    k = np.zeros((1, 1, T, dk))
    v = np.zeros((1, 1, T, dv))
    k[0, 0, 0] = RNG.standard_normal(dk)
    v[0, 0, 0] = RNG.standard_normal(dv)
    q = RNG.standard_normal((1, 1, T, dk))
    a = RNG.uniform(0.3, 0.95, (1, 1, T, dk))
    o, _ = rec(q, k, v, a, None)
    ok = True
    for t in range(T):
        w = np.prod(a[0, 0, 1:t + 1], axis=0)
        ok &= np.allclose(o[0, 0, t], v[0, 0, 0] * np.dot(q[0, 0, t], k[0, 0, 0] * w), rtol=1e-12,
                          atol=1e-14)
    return bool(ok)


def pin_forms_agree(rec):
    """Parallel and chunkwise forms (with sub-blocks, ragged tails, strong
    decays) equal the recurrence."""
    B, H, T, dk, dv = 1, 2, 37, 6, 5
    q, k = RNG.standard_normal((2, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    a = RNG.uniform(0.2, 1.0, (B, H, T, dk))
    S0 = RNG.standard_normal((B, H, dv, dk))
    o, s = rec(q, k, v, a, S0)
    ok = True
    op, sp = parallel_form(q, k, v, a, S0)
    ok &= np.allclose(o, op, rtol=1e-10, atol=1e-10) and np.allclose(s, sp, rtol=1e-10, atol=1e-10)
    for chunk, sub in ((64, 16), (16, 4), (8, 8), (5, 2)):
        oc, sc = chunked_form(q, k, v, a, S0, chunk=chunk, sub=sub)
        ok &= np.allclose(o, oc, rtol=1e-10, atol=1e-10) and np.allclose(s, sc, rtol=1e-10, atol=1e-10)
    return bool(ok)


PINS = (pin_scalar_reduction, pin_unit_gate, pin_zero_gate_clears_channel, pin_columns_decay,
        pin_decay_weight, pin_forms_agree)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_diag_pin(pin):
    assert pin(ref)


def test_chunked_form_stable_under_strong_decay():
    """Sub-blocks keep every exponential finite where a single reference point
    per 64-token block would overflow: per-channel decay of e^-3 per token
    (e^-192 over a block) still gives the recurrence's result."""
    B, H, T, dk, dv = 1, 1, 64, 4, 3
    q, k = RNG.standard_normal((2, B, H, T, dk))
    v = RNG.standard_normal((B, H, T, dv))
    a = np.full((B, H, T, dk), np.exp(-3.0))
    o, s = ref(q, k, v, a, None)
    with np.errstate(over="raise", invalid="raise"):
        oc, sc = chunked_form(q, k, v, a, None, chunk=64, sub=16)
    assert np.allclose(o, oc, rtol=1e-9, atol=1e-12) and np.allclose(s, sc, rtol=1e-9, atol=1e-12)


# ------------------------------------------------------------- planted mistakes

def _rec_np(kind):
    def rec(q, k, v, alpha, S0):
        q, k, v, alpha = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha))
        B, H, T, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((B, H, T, dv))
        st = np.zeros((B, H, dv, dk))
        for b in range(B):
            for h in range(H):
                S = np.zeros((dv, dk)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
                for t in range(T):
                    a = alpha[b, h, t]
                    if kind == "shift":
                        a = alpha[b, h, t - 1] if t > 0 else np.ones(dk)
                    if kind == "mean":
                        a = np.full(dk, a.mean())
                    if kind == "reversed":
                        a = a[::-1]
                    w = np.outer(v[b, h, t], k[b, h, t])
                    if kind == "left":
                        S = a[:dv, None] * S + w
                    elif kind == "after_write":
                        S = (S + w) * a[None, :]
                    else:
                        S_prev = S
                        S = S * a[None, :] + w
                    o[b, h, t] = (S_prev if kind == "read_before" else S) @ q[b, h, t]
                st[b, h] = S
        return o, st
    return rec


@pytest.mark.parametrize("kind", ["none", "left", "after_write", "shift", "mean", "reversed",
                                  "read_before"])
def test_diag_pins_catch_planted_mistake(kind):
    rec = _rec_np(kind)
    failed = []
    for p in PINS:
        try:
            if not p(rec):
                failed.append(p.__name__)
        except ValueError:   # e.g. a row-side gate with d_v != d_k does not even broadcast
            failed.append(p.__name__ + " (raised)")
    if kind == "none":
        assert not failed, failed   # the unmutated copy passes every pin
    else:
        assert failed, f"planted mistake {kind} passed every pin"

"""Pins of the oracle's maps around the recurrence (CPU only).

The maps (page "Scrivere meglio nella memoria: gate e delta rule"): SiLU then
L2 normalisation of keys and queries (opening section), beta = sigmoid(.)
(section "Correggere: la delta rule"), an RMSNorm on the output (same
section), and a data-dependent scalar decay (section "Dimenticare: i gate").

Each pin checks a closed form or a property the pages give, not a retyped
formula; a planted-mistake test swaps one map of ``oracle.prologue`` for a
plausible wrong version and requires some pin to fail.
"""
import math

import numpy as np
import pytest

from oracle import DECAY, DELTA, GATED_DELTA
from oracle import prologue as P

RNG = np.random.default_rng(20261202)


# --------------------------------------------------------------------------- pins

def pin_silu():
    """SiLU(0) = 0, SiLU(1) = e / (1 + e), SiLU(x) - SiLU(-x) = x, SiLU ~ relu far out."""
    x = RNG.standard_normal(64) * 3
    ok = P.silu(0.0) == 0.0
    ok &= abs(P.silu(1.0) - math.e / (1.0 + math.e)) < 1e-15
    ok &= np.allclose(P.silu(x) - P.silu(-x), x, rtol=0, atol=1e-13)
    ok &= abs(P.silu(50.0) - 50.0) < 1e-12 and abs(P.silu(-50.0)) < 1e-18
    return bool(ok)


def pin_sigmoid():
    """sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(x) + sigmoid(-x) = 1, no overflow."""
    x = RNG.standard_normal(64) * 5
    ok = P.sigmoid(0.0) == 0.5
    ok &= abs(P.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    ok &= np.allclose(P.sigmoid(x) + P.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    with np.errstate(over="raise"):
        ok &= P.sigmoid(-1000.0) == 0.0 and P.sigmoid(1000.0) == 1.0
    return bool(ok)


def pin_softplus_gate():
    """softplus(0) = ln 2 so the gate is 2^-c at 0; softplus(ln(e - 1)) = 1;
    softplus(x) - softplus(-x) = x; exp(-c softplus(a)) = sigmoid(-a)^c."""
    a = RNG.standard_normal(64) * 3
    ok = abs(P.softplus(0.0) - math.log(2.0)) < 1e-15
    ok &= abs(P.softplus(math.log(math.e - 1.0)) - 1.0) < 1e-15
    ok &= np.allclose(P.softplus(a) - P.softplus(-a), a, rtol=0, atol=1e-13)
    for c in (0.1, 1.0, 3.0):
        ok &= abs(P.softplus_gate(0.0, c) - 2.0 ** -c) < 1e-15
        ok &= np.allclose(P.softplus_gate(a, c), P.sigmoid(-a) ** c, rtol=1e-13, atol=0)
    # one value of c per head: [B, H, T] gates, c of shape [H]
    g = P.softplus_gate(np.zeros((1, 3, 2)), np.array([1.0, 2.0, 3.0]))
    ok &= np.allclose(g[0, :, 0], [0.5, 0.25, 0.125], rtol=0, atol=1e-15)
    # GLA's gate sigmoid(a)^(1/tau): at a = 0 it is 2^(-1/tau); at a = ln 3 it is (3/4)^(1/tau);
    # per key channel ([B, H, T, dk]) with c per head
    tau = 16.0
    ok &= abs(P.sigmoid_pow_gate(0.0, 1 / tau) - 2.0 ** (-1 / tau)) < 1e-15
    ok &= abs(P.sigmoid_pow_gate(math.log(3.0), 1 / tau) - 0.75 ** (1 / tau)) < 1e-15
    gd = P.sigmoid_pow_gate(np.zeros((1, 2, 3, 4)), np.array([1.0, 0.5]))
    ok &= np.allclose(gd[0, 0], 0.5, rtol=0, atol=1e-15) and np.allclose(gd[0, 1], 0.5 ** 0.5, rtol=0,
                                                                            atol=1e-15)
    return bool(ok)


def pin_l2():
    """(3, 4) -> (0.6, 0.8); unit norm along the last axis; direction kept; 0 -> 0."""
    ok = np.allclose(P.l2_normalise(np.array([3.0, 4.0])), [0.6, 0.8], rtol=0, atol=1e-16)
    x = RNG.standard_normal((5, 7, 33))
    y = P.l2_normalise(x)
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    ok &= np.allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=0, atol=1e-14)
    ok &= np.allclose(y * n, x, rtol=0, atol=1e-13)
    ok &= np.all(P.l2_normalise(np.zeros((2, 8))) == 0.0)
    # the key map is SiLU first, then the norm: for (1, -1) the SiLU values are
    # e/(1+e) and -1/(1+e), whose norm is sqrt(e^2 + 1)/(1 + e)
    s = P.silu_l2(np.array([1.0, -1.0]))
    ok &= np.allclose(s, np.array([math.e, -1.0]) / math.sqrt(math.e ** 2 + 1.0), rtol=0, atol=1e-15)
    return bool(ok)


def pin_rmsnorm():
    """(3, 4) -> (3, 4) / sqrt(12.5 + eps); a constant row -> the weight (times
    the sign); the output's root mean square is 1 before the weight; the norm
    runs over channels (the last axis); scale invariance as eps -> 0."""
    eps = 1e-6
    ok = np.allclose(P.rmsnorm(np.array([3.0, 4.0]), None, eps),
                     np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=0, atol=1e-15)
    w = RNG.uniform(0.5, 2.0, 16)
    ok &= np.allclose(P.rmsnorm(np.full(16, -7.0), w, 0.0), -w, rtol=0, atol=1e-14)
    x = RNG.standard_normal((3, 4, 16)) * RNG.uniform(0.1, 10.0, (3, 4, 1))
    y = P.rmsnorm(x, None, 0.0)
    ok &= np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=0, atol=1e-13)
    ok &= np.allclose(P.rmsnorm(x, w, 0.0), y * w, rtol=0, atol=1e-13)
    ok &= np.allclose(P.rmsnorm(123.0 * x, w, 0.0), P.rmsnorm(x, w, 0.0), rtol=0, atol=1e-12)
    return bool(ok)


def _run(mode, flags, q, k, v, alpha, beta, S0, **kw):
    return P.fused(mode, flags, q, k, v, alpha, beta, S0, **kw)


def pin_normalised_delta_overwrites():
    """With keys (and queries) normalised and beta = sigmoid(40) = 1, the delta
    rule replaces what a key holds (first page, delta-rule section: eigenvalues
    of I - beta k k^T in [0, 1], 0 for beta = 1), so reading with the same key
    returns the new value whatever the memory held."""
    B, H, T, d = 1, 2, 6, 16
    x = RNG.standard_normal((B, H, T, d)) * 2
    v = RNG.standard_normal((B, H, T, d))
    S0 = RNG.standard_normal((B, H, d, d)) * 3
    beta = np.full((B, H, T), 40.0)
    ok = True
    for mode in (DELTA, GATED_DELTA):
        alpha = np.full((B, H, T), -3.0)  # any decay: the erase follows it
        o, _ = _run(mode, P.QK_SILU_L2 | P.BETA_SIGMOID | P.ALPHA_SIGMOID, x, x, v, alpha, beta, S0)
        ok &= np.allclose(o, v, rtol=0, atol=1e-12)
    return bool(ok)


def pin_gates_route():
    """DECAY with nothing written after the first token: the state decays by
    alpha per token, so o_t = alpha^t S0 q with alpha = 2^-c per head
    (softplus gate at 0) or 3/4 (sigmoid gate at ln 3)."""
    B, H, T, d = 1, 2, 5, 8
    q = np.zeros((B, H, T, d))
    q[..., 0] = 1.0
    k = np.zeros((B, H, T, d))
    v = np.zeros((B, H, T, d))
    S0 = RNG.standard_normal((B, H, d, d))
    base = S0[:, :, None, :, 0]  # S0 q for q = e_0
    c = np.array([0.5, 2.0])
    o, _ = _run(DECAY, P.ALPHA_SOFTPLUS, q, k, v, np.zeros((B, H, T)), None, S0, alpha_scale=c)
    t = np.arange(1, T + 1)
    want = base * (2.0 ** -(c[None, :, None] * t[None, None, :]))[..., None]
    ok = np.allclose(o, want, rtol=1e-13, atol=1e-15)
    o, _ = _run(DECAY, P.ALPHA_SIGMOID, q, k, v, np.full((B, H, T), math.log(3.0)), None, S0)
    ok &= np.allclose(o, base * (0.75 ** t)[None, None, :, None], rtol=1e-13, atol=1e-15)
    return bool(ok)


def pin_output_norm():
    """With O_RMSNORM the root mean square of every output row equals the
    weight's (a constant weight w gives rms w), independent of the scale of v."""
    B, H, T, d = 1, 2, 7, 16
    q = RNG.standard_normal((B, H, T, d))
    k = RNG.standard_normal((B, H, T, d))
    v = RNG.standard_normal((B, H, T, d))
    beta = RNG.standard_normal((B, H, T))
    alpha = RNG.standard_normal((B, H, T))
    fl = P.QK_SILU_L2 | P.BETA_SIGMOID | P.ALPHA_SIGMOID | P.O_RMSNORM
    w = np.full(d, 2.5)
    o, st = _run(GATED_DELTA, fl, q, k, v, alpha, beta, None, norm_weight=w, norm_eps=0.0)
    ok = np.allclose(np.sqrt(np.mean(o * o, axis=-1)), 2.5, rtol=1e-12, atol=0)
    o2, st2 = _run(GATED_DELTA, fl, q, k, 1000.0 * v, alpha, beta, None, norm_weight=w, norm_eps=0.0)
    ok &= np.allclose(o2, o, rtol=1e-10, atol=1e-12)
    ok &= np.allclose(st2, 1000.0 * st, rtol=1e-10, atol=1e-12)  # the state is not normalised
    return bool(ok)


PINS = (pin_silu, pin_sigmoid, pin_softplus_gate, pin_l2, pin_rmsnorm,
        pin_normalised_delta_overwrites, pin_gates_route, pin_output_norm)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_prologue_pin(pin):
    assert pin()


# ------------------------------------------------------------- planted mistakes

def _sig(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


MISTAKES = {
    # SiLU with the wrong sign inside the sigmoid
    "silu_sign": ("silu", lambda x: np.asarray(x, float) * _sig(-np.asarray(x, float))),
    # plain sigmoid with a dropped minus
    "sigmoid_sign": ("sigmoid", lambda x: 1.0 / (1.0 + np.exp(np.asarray(x, float)))),
    # softplus without the max term
    "softplus_drop": ("softplus", lambda x: np.log1p(np.exp(-np.abs(np.asarray(x, float))))),
    # L2 norm over the wrong axis
    "l2_axis": ("l2_normalise", lambda x, eps=P.L2_EPS: np.asarray(x, float) / np.maximum(
        np.sqrt(np.sum(np.asarray(x, float) ** 2, axis=0, keepdims=True)), eps)),
    # L2 normalisation left out of the key map
    "l2_missing": ("silu_l2", lambda x: P.silu(x)),
    # RMSNorm dividing by the root of the sum instead of the mean
    "rms_sum": ("rmsnorm", lambda o, weight=None, eps=P.RMS_EPS: (
        np.asarray(o, float) / np.sqrt(np.sum(np.asarray(o, float) ** 2, axis=-1, keepdims=True) + eps)
        * (1.0 if weight is None else np.asarray(weight, float)))),
    # GLA gate with the power applied outside the wrong way
    "pow_inverse": ("sigmoid_pow_gate", lambda a, c: P.sigmoid(a) ** (1.0 / np.asarray(c, float))
                    if np.ndim(c) == 0 else P.sigmoid(a)),
    # softplus gate with the sign of c flipped
    "gate_sign": ("softplus_gate", lambda a, c: np.exp(np.asarray(c, float).reshape(
        (1, -1) + (1,) * (np.ndim(a) - 2)) * P.softplus(a) if np.ndim(c) == 1 else c * P.softplus(a))),
    # beta left as its pre-activation
    "beta_raw": ("apply_prologue", None),
}


def _beta_raw_prologue(orig):
    def f(flags, q, k, alpha, beta, alpha_scale=1.0):
        return orig(flags & ~P.BETA_SIGMOID, q, k, alpha, beta, alpha_scale)
    return f


@pytest.mark.parametrize("kind", sorted(MISTAKES))
def test_prologue_pins_catch_planted_mistake(kind, monkeypatch):
    name, fn = MISTAKES[kind]
    if kind == "beta_raw":
        fn = _beta_raw_prologue(P.apply_prologue)
    monkeypatch.setattr(P, name, fn)
    failed = []
    for pin in PINS:
        try:
            if not pin():
                failed.append(pin.__name__)
        except (FloatingPointError, ValueError, AssertionError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {kind} passed every pin"

"""Pins of the fp64 oracle to facts the pages fix (CPU only).

Each check below is written as a function of an oracle callable
``rec(mode, q, k, v, alpha, beta, S0) -> (o, S_T)`` so that the same checks
run against the real oracle (all must pass) and against planted mistakes in
a numpy copy of the recurrence (each mistake must fail at least one check).
"""
import numpy as np
import pytest

import oracle
from oracle import DECAY, DELTA, GATED_DELTA, LINEAR
from oracle.forms import chunked_form, parallel_form

ALL_MODES = (LINEAR, DECAY, DELTA, GATED_DELTA)


def _col(x):
    """[T] scalars -> [1,1,T,1] (one sequence, d = 1)."""
    return np.asarray(x, dtype=np.float64).reshape(1, 1, -1, 1)


def _seq(x):
    return np.asarray(x, dtype=np.float64).reshape(1, 1, -1)


# --------------------------------------------------------------------------- pins

def pin_three_votes(rec, fx):
    """Three forms of retention give 6, 10, 13 (second page, RetNet section)."""
    T = len(fx["votes"])
    one = _col(np.ones(T))
    v = _col(fx["votes"])
    a = _seq(np.full(T, fx["decay"]))
    o, _ = rec(DECAY, one, one, v, a, None, None)
    return np.allclose(o.ravel(), fx["totals"], rtol=0, atol=1e-12)


def pin_mario(rec, fx):
    """One delta write from a memory reading 7 towards 10 (first page, delta rule)."""
    ok = True
    for dose, expect in fx["after_by_dose"].items():
        for mode in (DELTA, GATED_DELTA):
            one = _col([1.0])
            o, st = rec(mode, one, one, _col([fx["target"]]), _seq([1.0]), _seq([float(dose)]),
                        np.full((1, 1, 1, 1), fx["read_before"]))
            ok &= abs(o.ravel()[0] - expect) < 1e-12 and abs(st.ravel()[0] - expect) < 1e-12
    # the erase-then-write order: (1 - beta) * old + beta * new, beta = 1/2
    e = fx["erase_then_write_half"]
    ok &= abs(0.5 * fx["read_before"] - e["erased_part"]) < 1e-12
    ok &= abs(0.5 * fx["target"] - e["written_part"]) < 1e-12
    o, _ = rec(DELTA, _col([1.0]), _col([1.0]), _col([fx["target"]]), None, _seq([0.5]),
               np.full((1, 1, 1, 1), fx["read_before"]))
    ok &= abs(o.ravel()[0] - e["total"]) < 1e-12
    return bool(ok)


def pin_marker(rec, fx):
    """A key with squared norm 2 at full dose oscillates 13, 7, 13, ... (first page)."""
    reads = fx["reads_after_each_write"]
    T = len(reads)
    kn = np.sqrt(fx["key_squared_norm"])
    k = _col(np.full(T, kn))
    s0 = np.full((1, 1, 1, 1), fx["read_before"] / kn)    # S0 k = 7
    o, _ = rec(DELTA, k, k, _col(np.full(T, fx["target"])), None, _seq(np.full(T, fx["dose"])), s0)
    return np.allclose(o.ravel(), reads, rtol=0, atol=1e-9)


def recall_experiment(rec, N, d, trials, seed):
    """The page's recall/rewrite experiment, run through the oracle's own update."""
    rng = np.random.default_rng(seed)
    K = np.empty((trials, N, d))
    V = np.empty((trials, N, d))
    vn = np.empty((trials, d))
    for i in range(trials):                       # the page's draw order
        kk = rng.standard_normal((N, d))
        K[i] = kk / np.linalg.norm(kk, axis=1, keepdims=True)
        V[i] = rng.standard_normal((N, d))
        vn[i] = rng.standard_normal(d)
    out = {}
    for name, mode in (("sum", LINEAR), ("delta", DELTA)):
        ones = np.ones((trials, 1, N))
        _, S = rec(mode, K[:, None], K[:, None], V[:, None], None, ones, None)
        read = np.einsum("bvk,bnk->bnv", S[:, 0], K)
        recall = (np.linalg.norm(read - V, axis=2) / np.linalg.norm(V, axis=2)).mean(axis=1).mean()
        k0 = K[:, None, :1, :]
        o, _ = rec(mode, k0, k0, vn[:, None, None, :], None, np.ones((trials, 1, 1)), S)
        rew = (np.linalg.norm(o[:, 0, 0] - vn, axis=1) / np.linalg.norm(vn, axis=1)).mean()
        out["recall_" + name] = recall
        out["rewrite_" + name] = rew
    return out


def pin_recall_table(rec, fx, rows=None):
    ok = True
    for row in fx["rows"] if rows is None else rows:
        got = recall_experiment(rec, row["N"], fx["d"], fx["trials"], fx["seed"])
        for key in ("recall_sum", "recall_delta", "rewrite_sum", "rewrite_delta"):
            ok &= round(got[key], fx["decimals"]) == pytest.approx(row[key], abs=1e-9)
    return bool(ok)


def pin_overwrite(rec):
    """beta = 1 and a unit key: S_t k_t = v_t whatever came before (first page)."""
    rng = np.random.default_rng(11)
    d, T = 8, 6
    k = rng.standard_normal((1, 1, T, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, 1, T, d))
    a = rng.uniform(0.3, 1.0, (1, 1, T))
    s0 = rng.standard_normal((1, 1, d, d))
    ok = True
    for mode in (DELTA, GATED_DELTA):
        o, _ = rec(mode, k, k, v, a, np.ones((1, 1, T)), s0)
        ok &= np.allclose(o, v, rtol=0, atol=1e-12)
    return bool(ok)


def pin_orthonormal_keys(rec):
    """Orthonormal keys, S0 = 0: every write lands whole, so
    S_T = sum_t w_t v_t k_t^T with w_t = beta_t * prod_{s>t} alpha_s for the
    gated delta row, the same without beta for the decay row, and without
    alpha for the plain delta row (first page, online-regression section and
    the decay-weight remark of the gates section)."""
    rng = np.random.default_rng(12)
    d, T = 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm[:T].reshape(1, 1, T, d)
    v = rng.standard_normal((1, 1, T, 6))
    a = rng.uniform(0.5, 1.0, T)
    b = rng.uniform(0.1, 1.0, T)
    ok = True
    for mode in ALL_MODES:
        w = np.ones(T)
        for t in range(T):
            if mode in (DECAY, GATED_DELTA):
                w[t] *= np.prod(a[t + 1:])
            if mode in (DELTA, GATED_DELTA):
                w[t] *= b[t]
        expect = sum(w[t] * np.outer(v[0, 0, t], k[0, 0, t]) for t in range(T))
        _, st = rec(mode, k, k, v, _seq(a), _seq(b), None)
        ok &= np.allclose(st[0, 0], expect, rtol=0, atol=1e-12)
    # first token at half dose: delta writes half of what accumulation writes
    _, s_lin = rec(LINEAR, k[:, :, :1], k[:, :, :1], v[:, :, :1], None, None, None)
    _, s_del = rec(DELTA, k[:, :, :1], k[:, :, :1], v[:, :, :1], None, _seq([0.5]), None)
    ok &= np.allclose(s_lin, 2.0 * s_del, rtol=0, atol=1e-14)
    return bool(ok)


def pin_zero_dose(rec):
    """Gated delta with beta = 0: S_t = alpha_t S_{t-1}, nothing written (first page)."""
    rng = np.random.default_rng(13)
    d, T = 6, 7
    q = rng.standard_normal((1, 1, T, d))
    k = rng.standard_normal((1, 1, T, d))
    v = rng.standard_normal((1, 1, T, d))
    a = rng.uniform(0.5, 1.0, T)
    s0 = rng.standard_normal((1, 1, d, d))
    o, st = rec(GATED_DELTA, q, k, v, _seq(a), np.zeros((1, 1, T)), s0)
    g = np.cumprod(a)
    ok = np.allclose(st[0, 0], g[-1] * s0[0, 0], rtol=0, atol=1e-12)
    ok &= np.allclose(o[0, 0], g[:, None] * (q[0, 0] @ s0[0, 0].T), rtol=0, atol=1e-12)
    return bool(ok)


def pin_gradient_step(rec):
    """The delta update is one gradient step of l(S) = 1/2 |S k - v|^2 with
    learning rate beta; the gated update is that step taken from alpha*S
    (online-regression section).  The gradient here is by central differences."""
    rng = np.random.default_rng(14)
    dk, dv = 5, 4
    S = rng.standard_normal((dv, dk))
    k = rng.standard_normal(dk)
    v = rng.standard_normal(dv)
    beta, alpha = 0.37, 0.81

    def loss(M):
        r = M @ k - v
        return 0.5 * float(r @ r)

    def grad(M):
        G = np.zeros_like(M)
        h = 1e-5
        for i in range(dv):
            for j in range(dk):
                E = np.zeros_like(M)
                E[i, j] = h
                G[i, j] = (loss(M + E) - loss(M - E)) / (2 * h)
        return G

    one = lambda x: x.reshape(1, 1, 1, -1)
    _, s_delta = rec(DELTA, one(k), one(k), one(v), None, _seq([beta]), S.reshape(1, 1, dv, dk))
    _, s_gated = rec(GATED_DELTA, one(k), one(k), one(v), _seq([alpha]), _seq([beta]),
                     S.reshape(1, 1, dv, dk))
    ok = np.allclose(s_delta[0, 0], S - beta * grad(S), rtol=0, atol=1e-8)
    ok &= np.allclose(s_gated[0, 0], alpha * S - beta * grad(alpha * S), rtol=0, atol=1e-8)
    return bool(ok)


def pin_transition_spectrum(rec):
    """The state transition alpha (I - beta k k^T): all eigenvalues alpha except
    one, alpha (1 - beta |k|^2); for the plain delta rule with beta |k|^2 <= 1 the
    spectral norm is exactly 1 (first page, Householder form).  The transition
    is read off the oracle by feeding S0 = I and v = 0."""
    rng = np.random.default_rng(15)
    d = 6
    k = rng.standard_normal(d)
    k *= 0.9 / np.linalg.norm(k)
    ok = True
    for mode, alpha, beta in ((DELTA, 1.0, 0.8), (GATED_DELTA, 0.7, 0.8), (GATED_DELTA, 0.9, 1.0)):
        _, st = rec(mode, k.reshape(1, 1, 1, d), k.reshape(1, 1, 1, d), np.zeros((1, 1, 1, d)),
                    _seq([alpha]), _seq([beta]), np.eye(d).reshape(1, 1, d, d))
        M = st[0, 0]
        ev = np.sort(np.linalg.eigvals(M).real)
        expect = np.sort(np.r_[alpha * (1 - beta * (k @ k)), np.full(d - 1, alpha)])
        ok &= np.allclose(ev, expect, rtol=0, atol=1e-12)
        ok &= abs(np.linalg.norm(M, 2) - alpha) < 1e-12
    return bool(ok)


def pin_decay_weight(rec, fx):
    """A write at step j reaches step t weighted by prod_{i=j+1..t} alpha_i
    (first page, gates section); with 0.9 for ten steps that is about 0.35."""
    rng = np.random.default_rng(16)
    T, j = 9, 2
    a = rng.uniform(0.5, 1.0, T)
    v = np.zeros(T)
    v[j] = 1.0
    one = _col(np.ones(T))
    o, st = rec(DECAY, one, one, _col(v), _seq(a), None, None)
    ok = np.allclose(o.ravel()[j:], np.cumprod(np.r_[1.0, a[j + 1:]]), rtol=0, atol=1e-14)
    n = fx["steps"]
    a9 = np.full(n + 1, fx["factor"])
    v9 = np.zeros(n + 1)
    v9[0] = 1.0
    o9, _ = rec(DECAY, _col(np.ones(n + 1)), _col(np.ones(n + 1)), _col(v9), _seq(a9), None, None)
    ok &= round(o9.ravel()[-1], fx["decimals"]) == fx["weight_approx"]
    return bool(ok)


def pin_forms_agree(rec):
    """Parallel, chunkwise and recurrent forms agree on random tiny inputs, in
    every mode, for several block sizes and ragged lengths (second page: the
    three forms give exactly the same result)."""
    rng = np.random.default_rng(17)
    ok = True
    for T in (1, 3, 37):
        dk, dv = 4, 3
        q = rng.standard_normal((1, 2, T, dk))
        k = rng.standard_normal((1, 2, T, dk)) * 0.5
        v = rng.standard_normal((1, 2, T, dv))
        a = rng.uniform(0.6, 1.0, (1, 2, T))
        b = rng.uniform(0.0, 1.0, (1, 2, T))
        s0 = rng.standard_normal((1, 2, dv, dk))
        for mode in ALL_MODES:
            o_r, s_r = rec(mode, q, k, v, a, b, s0)
            o_p, s_p = parallel_form(mode, q, k, v, a, b, s0)
            ok &= np.allclose(o_r, o_p, rtol=0, atol=1e-11) and np.allclose(s_r, s_p, rtol=0, atol=1e-11)
            for C in (1, 2, 16):
                o_c, s_c = chunked_form(mode, q, k, v, a, b, s0, chunk=C)
                ok &= np.allclose(o_r, o_c, rtol=0, atol=1e-11) and np.allclose(s_r, s_c, rtol=0, atol=1e-11)
    return bool(ok)


def _real(mode, q, k, v, a, b, s0):
    return oracle.recurrent(mode, q, k, v, a, b, s0)


# --------------------------------------------------------------- real oracle

def test_three_votes_all_forms(golden):
    fx = golden("retention_three_votes.json")
    assert pin_three_votes(_real, fx)
    T = len(fx["votes"])
    one = _col(np.ones(T))
    v = _col(fx["votes"])
    a = _seq(np.full(T, fx["decay"]))
    o_p, _ = parallel_form(DECAY, one, one, v, a)
    o_c, _ = chunked_form(DECAY, one, one, v, a, chunk=fx["block"])
    assert np.allclose(o_p.ravel(), fx["totals"], atol=1e-12)
    assert np.allclose(o_c.ravel(), fx["totals"], atol=1e-12)


def test_mario(golden):
    assert pin_mario(_real, golden("delta_rule_mario.json"))


def test_marker_overshoot(golden):
    assert pin_marker(_real, golden("delta_rule_marker_overshoot.json"))


def test_recall_table(golden):
    assert pin_recall_table(_real, golden("recall_experiment_d32.json"))


def test_overwrite():
    assert pin_overwrite(_real)


def test_orthonormal_keys():
    assert pin_orthonormal_keys(_real)


def test_zero_dose():
    assert pin_zero_dose(_real)


def test_gradient_step():
    assert pin_gradient_step(_real)


def test_transition_spectrum():
    assert pin_transition_spectrum(_real)


def test_decay_weight(golden):
    assert pin_decay_weight(_real, golden("decay_point_nine.json"))


def test_forms_agree():
    assert pin_forms_agree(_real)


@pytest.mark.parametrize("T,C", [(130, 64), (64, 64), (65, 64), (130, 2)])
def test_chunk_algebra_larger(T, C):
    """Chunked fp64 form equals the recurrence with d = 16 at the block size the
    GPU uses, with a ragged tail."""
    rng = np.random.default_rng(T * 7 + C)
    dk, dv = 16, 12
    q = rng.standard_normal((1, 1, T, dk))
    k = rng.standard_normal((1, 1, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, 1, T, dv))
    a = 1.0 / (1.0 + np.exp(-(3.0 + rng.standard_normal((1, 1, T)))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, 1, T))))
    s0 = 0.1 * rng.standard_normal((1, 1, dv, dk))
    for mode in ALL_MODES:
        o_r, s_r = oracle.recurrent(mode, q, k, v, a, b, s0)
        o_c, s_c = chunked_form(mode, q, k, v, a, b, s0, chunk=C)
        assert np.allclose(o_r, o_c, rtol=0, atol=1e-10)
        assert np.allclose(s_r, s_c, rtol=0, atol=1e-10)


def test_empty_sequence_keeps_state():
    rng = np.random.default_rng(3)
    s0 = rng.standard_normal((2, 3, 4, 5))
    z = np.zeros((2, 3, 0, 5))
    o, st = oracle.recurrent(GATED_DELTA, z, z, np.zeros((2, 3, 0, 4)), np.zeros((2, 3, 0)),
                             np.zeros((2, 3, 0)), s0)
    assert o.shape == (2, 3, 0, 4)
    assert np.array_equal(st, s0)


def test_threads_do_not_change_result():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((2, 3, 20, 8)), rng.standard_normal((2, 3, 20, 8)) * 0.3
    v = rng.standard_normal((2, 3, 20, 8))
    a, b = rng.uniform(0.5, 1, (2, 3, 20)), rng.uniform(0, 1, (2, 3, 20))
    o1, s1 = oracle.recurrent(GATED_DELTA, q, k, v, a, b, threads=1)
    o4, s4 = oracle.recurrent(GATED_DELTA, q, k, v, a, b, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)


# ------------------------------------------------------ planted mistakes

def _mutant(kind):
    """A numpy copy of the recurrence with one planted mistake."""
    def rec(mode, q, k, v, alpha, beta, S0):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, T, dk = q.shape
        dv = v.shape[-1]
        o = np.zeros((B, H, T, dv))
        st = np.zeros((B, H, dv, dk))
        for bb in range(B):
            for hh in range(H):
                S = np.zeros((dv, dk)) if S0 is None else np.array(S0[bb, hh], dtype=np.float64)
                for t in range(T):
                    kt, qt, vt = k[bb, hh, t], q[bb, hh, t], v[bb, hh, t]
                    a = alpha[bb, hh, t] if mode in (DECAY, GATED_DELTA) else 1.0
                    b = beta[bb, hh, t] if mode in (DELTA, GATED_DELTA) else 1.0
                    if kind == "alpha_ignored":
                        a = 1.0
                    if kind == "beta_ignored":
                        b = 1.0
                    w = (S.T @ kt) if kind == "transposed_read" and dv == dk else S @ kt
                    prev = S.copy()
                    if mode == LINEAR:
                        S = S + np.outer(vt, kt)
                    elif mode == DECAY:
                        S = a * S + np.outer(vt, kt)
                    elif mode == DELTA:
                        sign = -1.0 if kind == "wrong_sign" else 1.0
                        S = S + sign * b * np.outer(vt - w, kt)
                    else:
                        if kind == "decay_after_read":      # v - S k instead of v - alpha S k
                            S = a * S + b * np.outer(vt - w, kt)
                        elif kind == "decay_after_write":   # alpha (S + beta (v - S k) k^T)
                            S = a * (S + b * np.outer(vt - w, kt))
                        elif kind == "beta_only_on_erase":  # S[a(I - b k k^T)] + v k^T
                            S = a * S - a * b * np.outer(w, kt) + np.outer(vt, kt)
                        else:
                            S = a * S - a * b * np.outer(w, kt) + b * np.outer(vt, kt)
                    if kind == "preupdate_readout":
                        o[bb, hh, t] = prev @ qt
                    elif kind == "transposed_readout" and dv == dk:
                        o[bb, hh, t] = S.T @ qt
                    else:
                        o[bb, hh, t] = S @ qt
                st[bb, hh] = S
        return o, st
    return rec


MUTANTS = ["alpha_ignored", "beta_ignored", "transposed_read", "wrong_sign", "decay_after_read",
           "decay_after_write", "beta_only_on_erase", "preupdate_readout", "transposed_readout"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind, golden):
    rec = _mutant(kind)
    short_table = golden("recall_experiment_d32.json")
    short_table = dict(short_table, trials=200)
    checks = [
        lambda: pin_three_votes(rec, golden("retention_three_votes.json")),
        lambda: pin_mario(rec, golden("delta_rule_mario.json")),
        lambda: pin_marker(rec, golden("delta_rule_marker_overshoot.json")),
        lambda: pin_overwrite(rec),
        lambda: pin_orthonormal_keys(rec),
        lambda: pin_zero_dose(rec),
        lambda: pin_gradient_step(rec),
        lambda: pin_transition_spectrum(rec),
        lambda: pin_decay_weight(rec, golden("decay_point_nine.json")),
        lambda: pin_forms_agree(rec),
    ]
    results = [c() for c in checks]
    # the unmutated copy passes every check, so a failure is the planted mistake
    assert not all(results), f"planted mistake '{kind}' passed every pin"


def test_unmutated_copy_passes_all_pins(golden):
    rec = _mutant("none")
    assert pin_three_votes(rec, golden("retention_three_votes.json"))
    assert pin_mario(rec, golden("delta_rule_mario.json"))
    assert pin_marker(rec, golden("delta_rule_marker_overshoot.json"))
    assert pin_overwrite(rec)
    assert pin_orthonormal_keys(rec)
    assert pin_zero_dose(rec)
    assert pin_gradient_step(rec)
    assert pin_transition_spectrum(rec)
    assert pin_decay_weight(rec, golden("decay_point_nine.json"))
    assert pin_forms_agree(rec)
    fx = golden("recall_experiment_d32.json")
    assert pin_recall_table(rec, dict(fx, trials=2000), rows=fx["rows"][:1])

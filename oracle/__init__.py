"""fp64 CPU oracle for the gated delta rule family (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
in ``gated_delta_rule_fwd_gb300`` and never imports it.

Three forms of the same result, each written from the pages:

* :func:`recurrent` -- the definition: the sequential recurrence in plain C,
  one token at a time ("Scrivere meglio nella memoria: gate e delta rule",
  the update equations of each section and the summary table).
* :func:`oracle.forms.parallel_form` -- the masked quadratic form
  ("Le architetture lineari: RetNet, RWKV, xLSTM", section "RetNet: la
  retention e le sue tre forme", parallel form), extended to the delta rows by
  the pseudo-value triangular system (first page, section "Correggere: la
  delta rule", WY representation).
* :func:`oracle.forms.chunked_form` -- the chunkwise form: the parallel form
  inside each block, the recurrent hand-off of the end-of-block state between
  blocks (second page, same section, chunkwise form).

Mode numbers: 0 LINEAR, 1 DECAY, 2 DELTA, 3 GATED_DELTA, 4 DIAG_DECAY (the
diagonal gate of GLA, first page, section "Dimenticare: i gate": alpha has one
value per key channel, [B,H,T,dk]; :mod:`oracle.diag` holds its parallel and
chunkwise forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

LINEAR, DECAY, DELTA, GATED_DELTA, DIAG_DECAY = 0, 1, 2, 3, 4
MODE_NAMES = {LINEAR: "linear", DECAY: "decay", DELTA: "delta", GATED_DELTA: "gated_delta",
              DIAG_DECAY: "diag_decay"}
USES_ALPHA = {LINEAR: False, DECAY: True, DELTA: False, GATED_DELTA: True, DIAG_DECAY: True}
USES_BETA = {LINEAR: False, DECAY: False, DELTA: True, GATED_DELTA: True, DIAG_DECAY: False}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "libgdr_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libgdr_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdr_oracle_recurrent.restype = ctypes.c_int
        lib.gdr_oracle_recurrent.argtypes = [ctypes.c_int] * 6 + [dp] * 7 + [dp, ctypes.c_int]
        lib.gdr_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads an OpenMP region of the oracle uses by default."""
    return int(_load().gdr_oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrent(mode, q, k, v, alpha=None, beta=None, S0=None, threads: int = 0):
    """Sequential definition of the recurrence, fp64.

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; alpha, beta: [B,H,T] (only where the mode
    uses them; alpha is [B,H,T,dk] for DIAG_DECAY); S0: [B,H,dv,dk] or None
    for zeros.  Inputs of any float dtype are widened exactly to float64.
    Returns (o [B,H,T,dv], S_T [B,H,dv,dk]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv)
    a = _f64(alpha) if USES_ALPHA[mode] else None
    b = _f64(beta) if USES_BETA[mode] else None
    if a is not None:
        assert a.shape == ((B, H, T, dk) if mode == DIAG_DECAY else (B, H, T))
    if b is not None:
        assert b.shape == (B, H, T)
    s0 = _f64(S0)
    if s0 is not None:
        assert s0.shape == (B, H, dv, dk)
    o = np.empty((B, H, T, dv), dtype=np.float64)
    st = np.empty((B, H, dv, dk), dtype=np.float64)
    rc = _load().gdr_oracle_recurrent(int(mode), B, H, T, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(a), _ptr(b), _ptr(s0), _ptr(o), _ptr(st), int(threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_recurrent failed with code {rc}")
    return o, st

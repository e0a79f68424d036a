"""CPU-side checks of liblr: it builds, loads, exports every symbol the header
declares, and rejects invalid arguments before any launch.

Calls that pass deliberately invalid arguments run in a child process with no
GPU visible, so that even a validation bug could not launch a kernel on fake
pointers.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lr.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_fwd_gb300.build import build
    build()
    import gated_delta_rule_fwd_gb300 as lr
    return lr.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lr_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert set(_declared_functions()) == {"lr_fwd_chunked", "lr_fwd_chunked_workspace_size",
                                          "lr_fwd_chunked_noalloc", "lr_step", "lr_device_status",
                                          "lr_fwd_chunked_fused",
                                          "lr_fwd_chunked_fused_workspace_size", "lr_step_fused",
                                          "lr_fwd_chunked_mlstm",
                                          "lr_fwd_chunked_mlstm_workspace_size", "lr_step_mlstm",
                                          "lr_fwd_chunked_gen_delta",
                                          "lr_fwd_chunked_gen_delta_workspace_size",
                                          "lr_step_gen_delta", "lr_status_string",
                                          "lr_debug_inject_scan_timeout", "lr_abi_version"}


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(\w+)", out))
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    import gated_delta_rule_fwd_gb300 as lr
    assert lib.lr_abi_version() == 3
    for code in range(13):
        s = lr.status_string(code)
        assert s and s != "unknown status"
    assert lr.status_string(99) == "unknown status"


def test_python_binding_matches_header_names():
    import gated_delta_rule_fwd_gb300 as lr
    assert callable(lr.lr_fwd_chunked) and callable(lr.lr_step)
    assert callable(lr.lr_fwd_chunked_fused) and callable(lr.lr_step_fused)
    assert tuple(sorted(lr.SYMBOLS)) == tuple(_declared_functions())


_VALIDATION_CHILD = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
import gated_delta_rule_fwd_gb300 as lr
L = lr.lib()
P = lambda a: ctypes.c_void_p(a)
A = [0x10000000 + i * 0x10000000 for i in range(9)]   # distinct, aligned, never dereferenced
q, k, v, al, be, s0, o, st, ws = (P(a) for a in A)
S = None
def chunk(**kw):
    args = dict(q=q, k=k, v=v, al=al, be=be, s0=s0, o=o, st=st, B=1, H=1, T=8, dk=32, dv=32,
                chunk=64, dt=0, mode=3, ws=ws, wsb=1 << 24)
    args.update(kw)
    a = args
    return L.lr_fwd_chunked(a['q'], a['k'], a['v'], a['al'], a['be'], a['s0'], a['o'], a['st'],
                            a['B'], a['H'], a['T'], a['dk'], a['dv'], a['chunk'], a['dt'],
                            a['mode'], a['ws'], a['wsb'], None)
need = L.lr_fwd_chunked_workspace_size(1, 1, 8, 32, 32, 64, 1, 3)
def step(**kw):
    args = dict(q=q, k=k, v=v, al=al, be=be, s=s0, o=o, N=1, H=1, dk=32, dv=32, dt=1, mode=3)
    args.update(kw)
    a = args
    return L.lr_step(a['q'], a['k'], a['v'], a['al'], a['be'], a['s'], a['o'], a['N'], a['H'],
                     a['dk'], a['dv'], a['dt'], a['mode'], None)
cases = [
    ("mode", chunk(mode=6), 5), ("mode-neg", chunk(mode=-1), 5), ("dtype", chunk(dt=2), 3),
    ("B0", chunk(B=0), 2), ("Hneg", chunk(H=-1), 2), ("Tneg", chunk(T=-1), 2),
    ("huge", chunk(B=1 << 20, H=1 << 10, T=1 << 20), 2),
    ("dk48", chunk(dk=48), 6), ("dv256", chunk(dv=256), 6), ("chunk32", chunk(chunk=32), 6),
    ("nullq", chunk(q=None), 1), ("nullo", chunk(o=None), 1), ("nullST", chunk(st=None), 1),
    ("nullalpha", chunk(al=None), 1), ("nullbeta", chunk(be=None), 1),
    ("decay-nullbeta-ok-but-nullalpha", chunk(mode=1, be=None, al=None), 1),
    ("misaligned", chunk(k=P(A[1] + 8)), 4),
    ("alias-o-q", chunk(o=q), 8), ("alias-st-k", chunk(st=k), 8),
    ("alias-st-partial-s0", chunk(st=P(A[5] + 16)), 8),
    ("ws-null", chunk(dt=1, ws=None), 10), ("ws-small", chunk(dt=1, wsb=need - 16), 10),
    ("ws-misaligned", chunk(dt=1, ws=P(A[8] + 8)), 4), ("ws-alias-o", chunk(dt=1, ws=o), 8),
    ("ws-size-f32", L.lr_fwd_chunked_workspace_size(1, 1, 8, 32, 32, 64, 0, 3), 0),
    ("ws-size-T0", L.lr_fwd_chunked_workspace_size(1, 1, 0, 32, 32, 64, 1, 3), 0),
    ("ws-size-bad", L.lr_fwd_chunked_workspace_size(1, 1, 8, 48, 32, 64, 1, 3), 0),
    ("ws-size-bf16-positive", int(need > 0), 1),
    ("step-mode", step(mode=9), 5), ("step-dtype", step(dt=3), 3), ("step-N0", step(N=0), 2),
    ("step-dk16", step(dk=16), 6), ("step-nullS", step(s=None), 1),
    ("step-nullalpha", step(al=None), 1), ("step-misaligned", step(v=P(A[2] + 4)), 4),
    ("step-alias-o-S", step(o=s0), 8),
]
def fz(flags=0, ascale=A[6] + 0x100000, w=A[6] + 0x200000, eps=1e-6):
    return ctypes.byref(lr.Fuse(flags, ascale, w, eps))
def fchunk(flags=0, ascale=A[6] + 0x100000, w=A[6] + 0x200000, eps=1e-6, **kw):
    args = dict(q=q, k=k, v=v, al=al, be=be, s0=s0, o=P(A[7] + 0x4000000), st=st, B=1, H=1, T=8,
                dk=32, dv=32, chunk=64, dt=1, mode=3, ws=ws, wsb=1 << 24)
    args.update(kw)
    a = args
    return L.lr_fwd_chunked_fused(a['q'], a['k'], a['v'], a['al'], a['be'], a['s0'], a['o'],
                                  a['st'], a['B'], a['H'], a['T'], a['dk'], a['dv'], a['chunk'],
                                  a['dt'], a['mode'], fz(flags, ascale, w, eps), a['ws'], a['wsb'],
                                  None)
def fstep(flags=0, ascale=A[6] + 0x100000, w=A[6] + 0x200000, eps=1e-6, **kw):
    args = dict(q=q, k=k, v=v, al=al, be=be, s=s0, o=o, N=1, H=1, dk=32, dv=32, dt=1, mode=3)
    args.update(kw)
    a = args
    return L.lr_step_fused(a['q'], a['k'], a['v'], a['al'], a['be'], a['s'], a['o'], a['N'],
                           a['H'], a['dk'], a['dv'], a['dt'], a['mode'], fz(flags, ascale, w, eps),
                           None)
ws_plain = L.lr_fwd_chunked_fused_workspace_size(1, 1, 8, 32, 32, 64, 1, 3, 0)
ws_qk = L.lr_fwd_chunked_fused_workspace_size(1, 1, 8, 32, 32, 64, 1, 3, 1)
cases += [
    ("fused-unknown-flag", fchunk(flags=0x40), 12),
    ("fused-both-alpha-maps", fchunk(flags=0x4 | 0x8), 12),
    ("fused-negative-eps", fchunk(flags=0x10, eps=-1.0), 12),
    ("fused-nan-eps", fchunk(flags=0x10, eps=float("nan")), 12),
    ("fused-softplus-null-scale", fchunk(flags=0x8, ascale=None), 1),
    ("fused-misaligned-weight", fchunk(flags=0x10, w=A[6] + 0x200004), 4),
    ("fused-misaligned-scale", fchunk(flags=0x8, ascale=A[6] + 0x100008), 4),
    ("fused-alias-o-weight", fchunk(flags=0x10, w=A[7] + 0x4000000), 8),
    ("fused-alias-st-scale", fchunk(flags=0x8, ascale=A[7]), 8),
    ("fused-ws-small-with-qk", fchunk(flags=0x1, wsb=ws_plain), 10),
    ("fused-shape-first", fchunk(flags=0x40, dk=48), 6),
    # a map of a gate the mode does not use is dropped: validation passes, and
    # with no GPU visible the launch then fails
    ("fused-softplus-ignored-in-delta", fchunk(flags=0x8, ascale=None, mode=2), 7),
    ("ws-size-qk", ws_qk - ws_plain, 2 * 8 * 32 * 2),
    ("ws-size-bad-flags", L.lr_fwd_chunked_fused_workspace_size(1, 1, 8, 32, 32, 64, 1, 3, 0x40), 0),
    ("ws-size-plain-same", ws_plain, need),
    ("step-fused-unknown-flag", fstep(flags=0x80), 12),
    ("step-fused-null-scale", fstep(flags=0x8, ascale=None), 1),
    ("step-fused-alias-S-weight", fstep(flags=0x10, w=A[5]), 8),
    ("step-fused-misaligned-weight", fstep(flags=0x10, w=A[6] + 0x200004), 4),
    ("fused-two-alpha-maps-pow", fchunk(flags=0x20 | 0x8), 12),
    ("fused-pow-null-scale", fchunk(flags=0x20, ascale=None), 1),
    # the diagonal gate: alpha [B, H, T, dk] (here 8 x 32 floats = 1 KB)
    ("diag-null-alpha", chunk(mode=4, al=None), 1),
    ("diag-mode-range", chunk(mode=5), 5),
    ("diag-alias-o-alpha", chunk(mode=4, o=P(A[3] + 512)), 8),
    ("scalar-alpha-span-is-short", chunk(mode=1, o=P(A[3] + 512)), 7),  # passes validation
    ("diag-step-alias-o-alpha", step(mode=4, o=P(A[3] + 64)), 8),
    ("diag-ws-larger", int(L.lr_fwd_chunked_workspace_size(1, 1, 8, 32, 32, 64, 1, 4) - need), 2 * 8 * 32 * 2),
]
# mLSTM: q k v fgate igate C0 n0 m0 h C_T n_T m_T
M = [P(0x10000000 + i * 0x10000000) for i in range(12)]
def ml(**kw):
    a = dict(zip("q k v f i C0 n0 m0 h CT nT mT".split(), M))
    a.update(dict(B=1, H=1, T=8, dk=32, dv=32, chunk=64, dt=0, ws=None, wsb=0))
    a.update(kw)
    return L.lr_fwd_chunked_mlstm(a["q"], a["k"], a["v"], a["f"], a["i"], a["C0"], a["n0"],
                                  a["m0"], a["h"], a["CT"], a["nT"], a["mT"], a["B"], a["H"],
                                  a["T"], a["dk"], a["dv"], a["chunk"], a["dt"], a["ws"],
                                  a["wsb"], None)
def mls(**kw):
    a = dict(zip("q k v f i C n m h".split(), M))
    a.update(dict(N=1, H=1, dk=32, dv=32, dt=1))
    a.update(kw)
    return L.lr_step_mlstm(a["q"], a["k"], a["v"], a["f"], a["i"], a["C"], a["n"], a["m"], a["h"],
                           a["N"], a["H"], a["dk"], a["dv"], a["dt"], None)
mneed = L.lr_fwd_chunked_mlstm_workspace_size(1, 1, 8, 32, 32, 64, 1)
cases += [
    ("mlstm-null-fgate", ml(f=None), 1), ("mlstm-null-mT", ml(mT=None), 1),
    ("mlstm-partial-state", ml(n0=None), 1), ("mlstm-dtype", ml(dt=2), 3),
    ("mlstm-dk48", ml(dk=48), 6), ("mlstm-misaligned", ml(v=P(0x30000008)), 4),
    ("mlstm-alias-h-q", ml(h=M[0]), 8), ("mlstm-alias-CT-n0", ml(CT=M[6]), 8),
    ("mlstm-ws-null-bf16", ml(dt=1), 10),
    ("mlstm-in-place-ok", ml(CT=M[5], nT=M[6], mT=M[7]), 7),   # passes validation, no GPU
    ("mlstm-ws-positive", int(mneed > 0), 1),
    ("mlstm-ws-f32", L.lr_fwd_chunked_mlstm_workspace_size(1, 1, 8, 32, 32, 64, 0), 0),
    ("mlstm-step-null", mls(n=None), 1), ("mlstm-step-alias-h-C", mls(h=M[5]), 8),
    ("mlstm-step-dk16", mls(dk=16), 6),
]
def gd(**kw):
    a = dict(zip("q kw v w kap a S0 o ST".split(), M[:9]))
    a.update(dict(B=1, H=1, T=8, dk=32, dv=32, chunk=64, dt=0, ws=None, wsb=0))
    a.update(kw)
    return L.lr_fwd_chunked_gen_delta(a["q"], a["kw"], a["v"], a["w"], a["kap"], a["a"], a["S0"],
                                      a["o"], a["ST"], a["B"], a["H"], a["T"], a["dk"], a["dv"],
                                      a["chunk"], a["dt"], a["ws"], a["wsb"], None)
gneed = L.lr_fwd_chunked_gen_delta_workspace_size(1, 1, 8, 32, 32, 64, 1)
cases += [
    ("gd-null-kappa", gd(kap=None), 1), ("gd-dk48", gd(dk=48), 6), ("gd-chunk32", gd(chunk=32), 6),
    ("gd-alias-o-w", gd(o=P(0x40000000 + 512)), 8), ("gd-misaligned", gd(a=P(0x60000004)), 4),
    ("gd-valid", gd(), 7),   # passes validation, no GPU
    ("gd-ws-null-bf16", gd(dt=1), 10), ("gd-ws-short", gd(dt=1, ws=P(0xD0000000), wsb=gneed - 16), 10),
    ("gd-ws-alias-q", gd(dt=1, ws=M[0], wsb=gneed), 8),
    ("gd-ws-misaligned", gd(dt=1, ws=P(0xD0000008), wsb=gneed), 4),
    ("gd-ws-valid-bf16", gd(dt=1, ws=P(0xD0000000), wsb=gneed), 7),
    ("gd-ws-positive", int(gneed > 0), 1),
    ("gd-ws-f32", L.lr_fwd_chunked_gen_delta_workspace_size(1, 1, 8, 32, 32, 64, 0), 0),
    ("gd-step-null", L.lr_step_gen_delta(M[0], M[1], M[2], M[3], M[4], None, M[6], M[7], 1, 1, 32,
                                         32, 1, None), 1),
]
bad = [(n, got, want) for n, got, want in cases if got != want]
print("BAD", bad)
sys.exit(1 if bad else 0)
"""


def test_invalid_arguments_rejected_before_launch(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _VALIDATION_CHILD, ROOT], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import gated_delta_rule_fwd_gb300 as lr
    monkeypatch.setattr(lr, "_lib", None)
    monkeypatch.setattr(lr, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        lr.lib()


class _NoLaunch:
    """Stands in for the loaded library: any attribute access (a call into the
    C ABI) fails the test."""

    def __getattr__(self, name):
        raise AssertionError(f"the binding reached the library ({name}) with invalid arguments")


@pytest.mark.parametrize("which", ["o", "S_T"])
@pytest.mark.parametrize("bad", ["shape", "dtype", "strided"])
def test_noalloc_binding_checks_outputs_before_any_call(monkeypatch, which, bad):
    """lr_fwd_chunked_noalloc's binding checks a caller-given o or S_T the way
    lr_fwd_chunked's does: a wrong shape, dtype or layout raises before the
    library is reached (the C ABI cannot see a buffer's size, so a short
    buffer would be written past its end)."""
    import torch
    import gated_delta_rule_fwd_gb300 as lr
    monkeypatch.setattr(lr, "_require_cuda", lambda dev: None)   # CPU tensors stand in
    monkeypatch.setattr(lr, "lib", lambda: _NoLaunch())
    B, H, T, dk, dv = 1, 2, 10, 32, 32
    q = torch.zeros(B, H, T, dk, dtype=torch.bfloat16)
    v = torch.zeros(B, H, T, dv, dtype=torch.bfloat16)
    a = torch.ones(B, H, T)
    o = torch.zeros(B, H, T, dv, dtype=torch.bfloat16)
    st = torch.zeros(B, H, dv, dk)
    good = {"o": o, "S_T": st}
    t = good[which]
    if bad == "shape":
        t = t[..., :-1].contiguous()
    elif bad == "dtype":
        t = t.to(torch.float16)
    else:
        t = t.transpose(-1, -2).contiguous().transpose(-1, -2)
    kw = dict(good)
    kw[which] = t
    with pytest.raises((ValueError, TypeError)):
        lr.lr_fwd_chunked_noalloc(q, q.clone(), v, a, a.clone(), None, **kw)

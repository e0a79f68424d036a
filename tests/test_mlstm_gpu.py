"""Parity of the mLSTM entry points (lr_fwd_chunked_mlstm, lr_step_mlstm) with
the fp64 oracle of the stabilised recurrence (``oracle.mlstm.stabilized``),
through the C ABI.  Metric as for the other modes, per output tensor:
max|gpu - oracle| / max|oracle|, 1e-4 for fp32 inputs, 2e-2 for bf16; the
final stabiliser m is compared in absolute terms (it is a log-weight).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import workloads
from oracle.mlstm import stabilized

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gated_delta_rule_fwd_gb300.build import build
    build()
    yield torch.device("cuda:0")
    assert lr.device_status() == 0


def rel_err(gpu, ref):
    g = gpu.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def to_dev(x, dev):
    return {n: (t.to(dev) if t is not None else None) for n, t in x.items()}


def ref(x):
    return stabilized(x["q"], x["k"], x["v"], np.log(x["fgate"].double().numpy()), x["igate"],
                      x["C0"], x["n0"], x["m0"])


def check(out, x, tol):
    h, C, n, m = out
    hr, Cr, nr, mr = ref(x)
    e = (rel_err(h, hr), rel_err(C, Cr), rel_err(n, nr),
         float(np.max(np.abs(m.cpu().double().numpy() - mr))))
    print(f"rel err h={e[0]:.3e} C={e[1]:.3e} n={e[2]:.3e} |dm|={e[3]:.2e}")
    assert e[0] <= tol and e[1] <= tol and e[2] <= tol and e[3] <= 1e-4


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_mlstm_chunked_small(dev, dtype, dk, dv, T):
    x = workloads.draw_mlstm(2, 3, T, dk, dv, seed=800 + T + dk + 3 * dv, dtype=dtype,
                             state=bool(T % 2))
    d = to_dev(x, dev)
    out = lr.lr_fwd_chunked_mlstm(d["q"], d["k"], d["v"], d["fgate"], d["igate"], d["C0"],
                                  d["n0"], d["m0"])
    torch.cuda.synchronize()
    check(out, x, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_mlstm_large_input_gates(dev, dtype):
    """igate ~ N(0, 8^2): write factors from e^-30 to e^30, which only the
    stabiliser keeps in range.  The outputs reach 1.6e3 here (|n.q| near its
    threshold), so the read's division amplifies the fp32 rounding of exponents
    up to ~30 (about 30 * 2^-24 each) by the normaliser's conditioning: the fp32
    bar of this case is 1e-3 (measured 3.8e-4; the state C, n, m stays at ~3e-7)."""
    x = workloads.draw_mlstm(1, 4, 64 * 3 + 11, 128, 128, seed=5, dtype=dtype, state=True,
                             igate_std=8.0)
    d = to_dev(x, dev)
    out = lr.lr_fwd_chunked_mlstm(d["q"], d["k"], d["v"], d["fgate"], d["igate"], d["C0"],
                                  d["n0"], d["m0"])
    torch.cuda.synchronize()
    assert np.all(np.isfinite(out[0].float().cpu().numpy()))
    check(out, x, 1e-3 if dtype == torch.float32 else TOL[dtype])


def test_mlstm_workload_full_size(dev):
    """B=8, H=16, T=4096, d=128, bf16: every output and the whole final state."""
    w = workloads.WORKLOADS["mlstm_bf16"]
    x = workloads.draw_mlstm(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=torch.bfloat16)
    d = to_dev(x, dev)
    out = lr.lr_fwd_chunked_mlstm(d["q"], d["k"], d["v"], d["fgate"], d["igate"])
    torch.cuda.synchronize()
    check(out, x, 2e-2)


def test_mlstm_resume_equals_one_call(dev):
    """The stabilised triple (C~, n~, m) is the checkpoint: two calls equal one."""
    x = workloads.draw_mlstm(1, 3, 300, 128, 128, seed=9, dtype=torch.bfloat16, state=True)
    d = to_dev(x, dev)
    h1, C1, n1, m1 = lr.lr_fwd_chunked_mlstm(*(d[n][:, :, :150].contiguous() for n in
                                               ("q", "k", "v", "fgate", "igate")),
                                             d["C0"], d["n0"], d["m0"])
    h2, C2, n2, m2 = lr.lr_fwd_chunked_mlstm(*(d[n][:, :, 150:].contiguous() for n in
                                               ("q", "k", "v", "fgate", "igate")), C1, n1, m1)
    torch.cuda.synchronize()
    check((torch.cat([h1, h2], 2), C2, n2, m2), x, 2e-2)


def test_mlstm_empty_sequence(dev):
    x = workloads.draw_mlstm(1, 2, 0, 64, 64, seed=2, dtype=torch.bfloat16, state=True)
    d = to_dev(x, dev)
    h, C, n, m = lr.lr_fwd_chunked_mlstm(d["q"], d["k"], d["v"], d["fgate"], d["igate"], d["C0"],
                                         d["n0"], d["m0"])
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), x["C0"]) and torch.equal(n.cpu(), x["n0"])
    assert torch.equal(m.cpu(), x["m0"])
    x2 = {**d, "C0": None, "n0": None, "m0": None}
    h, C, n, m = lr.lr_fwd_chunked_mlstm(x2["q"], x2["k"], x2["v"], x2["fgate"], x2["igate"])
    torch.cuda.synchronize()
    assert torch.count_nonzero(C) == 0 and torch.all(torch.isinf(m)) and bool((m < 0).all())


def test_mlstm_repeated_calls_bit_identical(dev):
    x = to_dev(workloads.draw_mlstm(4, 16, 2048, 128, 128, seed=3, dtype=torch.bfloat16), dev)
    outs0 = lr.lr_fwd_chunked_mlstm(x["q"], x["k"], x["v"], x["fgate"], x["igate"])
    bad = 0
    for _ in range(30):
        outs = lr.lr_fwd_chunked_mlstm(x["q"], x["k"], x["v"], x["fgate"], x["igate"])
        bad += int(not all(torch.equal(a, b) for a, b in zip(outs, outs0)))
    torch.cuda.synchronize()
    assert bad == 0, f"{bad} of 30 calls differ from the first"


def test_mlstm_workload_repeated_calls_bit_identical(dev):
    """The bench workload (B=8 H=16 T=4096, a given state, 64-channel scan CTAs):
    40 calls on the same inputs give the same bits.  A form of the scan that
    read the per-token factor from a global array inside its output loop
    failed this in about one call in five."""
    w = workloads.WORKLOADS["mlstm_bf16"]
    x = to_dev(workloads.draw_mlstm(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=torch.bfloat16,
                                    state=True), dev)
    args = (x["q"], x["k"], x["v"], x["fgate"], x["igate"], x["C0"], x["n0"], x["m0"])
    outs0 = [t.clone() for t in lr.lr_fwd_chunked_mlstm(*args)]
    bad = 0
    for _ in range(40):
        outs = lr.lr_fwd_chunked_mlstm(*args)
        bad += int(not all(torch.equal(a, b) for a, b in zip(outs, outs0)))
    torch.cuda.synchronize()
    assert bad == 0, f"{bad} of 40 calls differ from the first"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
@pytest.mark.parametrize("state", [True, False], ids=["state", "empty"])
def test_mlstm_step(dev, dtype, dk, dv, state):
    N, H, T = 5, 3, 4
    x = workloads.draw_mlstm(N, H, T, dk, dv, seed=31 + dk + dv, dtype=dtype, state=state)
    d = to_dev(x, dev)
    if state:
        C, n, m = d["C0"].clone(), d["n0"].clone(), d["m0"].clone()
    else:
        C = torch.zeros((N, H, dv, dk), device=dev)
        n = torch.zeros((N, H, dk), device=dev)
        m = torch.full((N, H), -float("inf"), device=dev)
    hs = []
    for t in range(T):
        c = lambda nm: d[nm][:, :, t].contiguous()
        hs.append(lr.lr_step_mlstm(c("q"), c("k"), c("v"), c("fgate"), c("igate"), C, n, m))
    torch.cuda.synchronize()
    check((torch.stack(hs, 2), C, n, m), x, TOL[dtype])

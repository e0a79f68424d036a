"""Parity of the sequential pass with 64 value channels per CTA.

The library runs each (batch, head) of the bf16 chunked forward on dv / NV scan
CTAs, NV = 32 or 64: 64 when 32-channel CTAs would need more waves over the
SMs than 64-channel ones (many heads).  These cases have enough heads for the
wide scan on this device (checked with the same rule), at small, ragged T, in
every mode that runs the 32/64-channel scan: the four lr modes, the diagonal
gate (one score product per block and the sub-block form), the fused maps and
the mLSTM numerator.  Metric and bar as for the other parity tests:
max|gpu - oracle| / max|oracle| per tensor, 2e-2 for bf16 inputs.
"""
import math

import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import oracle
import workloads
from oracle import prologue as P
from oracle.mlstm import stabilized

pytestmark = pytest.mark.gpu

TOL = 2e-2


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
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def wide(dev, B, H, dv):
    """The library's choice: 64 channels when that takes fewer waves."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n32 = B * H * (dv // 32)
    return dv >= 64 and math.ceil(n32 // 2 / sms) < math.ceil(n32 / sms)


def sizes(dev, dv):
    """(B, H) with enough heads for the 64-channel scan on this device."""
    for B, H in ((5, 8), (7, 11), (8, 12), (8, 16), (16, 16)):
        if wide(dev, B, H, dv):
            return B, H
    pytest.skip("this device's SM count selects the 32-channel scan for these sizes")


def to_dev(x, dev):
    return {n: (t.to(dev) if t is not None else None) for n, t in x.items()}


@pytest.mark.parametrize("mode", [lr.LINEAR, lr.DECAY, lr.DELTA, lr.GATED_DELTA],
                         ids=["linear", "decay", "delta", "gated_delta"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64)])
def test_wide_scan_lr_modes(dev, mode, dk, dv):
    B, H = sizes(dev, dv)
    gen = "mamba2" if mode == lr.DECAY else "gdn"
    x = workloads.draw(gen, B, H, 130, dk, dv, seed=5100 + mode + dk, dtype=torch.bfloat16,
                       s0_std=0.1)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], mode=mode)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrent(mode, x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"B={B} H={H}: rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= TOL and es <= TOL


@pytest.mark.parametrize("gen", ["gla", "gla_strong"])
def test_wide_scan_diagonal_gate(dev, gen):
    B, H = sizes(dev, 128)
    x = workloads.draw(gen, B, H, 200, 128, 128, seed=5200, dtype=torch.bfloat16, s0_std=0.2)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], None, d["S0"],
                              mode=lr.DIAG_DECAY)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrent(oracle.DIAG_DECAY, x["q"], x["k"], x["v"], x["alpha"], None,
                                    x["S0"])
    assert rel_err(o, o_ref) <= TOL and rel_err(st, s_ref) <= TOL


def test_wide_scan_fused_maps(dev):
    B, H = sizes(dev, 128)
    flags = lr.FUSE_QK_SILU_L2 | lr.FUSE_BETA_SIGMOID | lr.FUSE_ALPHA_SIGMOID | lr.FUSE_O_RMSNORM
    x = workloads.draw_pre("gdn", B, H, 130, 128, 128, seed=5300, dtype=torch.bfloat16,
                           s0_std=0.3)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                    mode=lr.GATED_DELTA, flags=flags,
                                    alpha_scale=d["alpha_scale"], norm_weight=d["norm_weight"])
    torch.cuda.synchronize()
    f64 = lambda t: t.double().numpy()
    o_ref, s_ref = P.fused(lr.GATED_DELTA, flags, f64(x["q"]), f64(x["k"]), f64(x["v"]),
                           f64(x["alpha"]), f64(x["beta"]), f64(x["S0"]),
                           alpha_scale=f64(x["alpha_scale"]), norm_weight=f64(x["norm_weight"]))
    assert rel_err(o, o_ref) <= TOL and rel_err(st, s_ref) <= TOL


def test_wide_scan_mlstm(dev):
    B, H = sizes(dev, 128)
    x = workloads.draw_mlstm(B, H, 200, 128, 128, seed=5400, dtype=torch.bfloat16, state=True)
    d = to_dev(x, dev)
    h, C, n, m = lr.lr_fwd_chunked_mlstm(d["q"], d["k"], d["v"], d["fgate"], d["igate"], d["C0"],
                                         d["n0"], d["m0"])
    torch.cuda.synchronize()
    hr, Cr, nr, mr = stabilized(x["q"], x["k"], x["v"], np.log(x["fgate"].double().numpy()),
                                x["igate"], x["C0"], x["n0"], x["m0"])
    assert rel_err(h, hr) <= TOL and rel_err(C, Cr) <= TOL and rel_err(n, nr) <= TOL
    assert float(np.max(np.abs(m.cpu().double().numpy() - mr))) <= 1e-4


def test_wide_scan_repeated_calls_bit_identical(dev):
    """The wide scan's hand-offs hold: 50 calls on the same inputs, same bits."""
    B, H = sizes(dev, 128)
    x = to_dev(workloads.draw("gdn", B, H, 1024, 128, 128, seed=5500, dtype=torch.bfloat16,
                              s0_std=0.1), dev)
    o0, s0 = lr.lr_fwd_chunked(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    bad = 0
    for _ in range(50):
        o, s = lr.lr_fwd_chunked(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
        bad += int(not (torch.equal(o, o0) and torch.equal(s, s0)))
    torch.cuda.synchronize()
    assert bad == 0

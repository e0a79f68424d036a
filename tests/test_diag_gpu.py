"""Parity of the diagonal gate (GLA row, LR_MODE_DIAG_DECAY) with the fp64
oracle, through the C ABI: chunked fp32 (CUDA cores) and bf16 (tensor cores),
the decode step, the fused gate map and output norm, strong decays, ragged
tails and repeatability.  Metric and bars as for the other modes:
max|gpu - oracle| / max|oracle| per tensor, 1e-4 (fp32) and 2e-2 (bf16).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import oracle
import workloads
from oracle import prologue as P

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
    g = gpu.detach().float().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def to_dev(x, dev):
    return {n: (t.to(dev) if t is not None else None) for n, t in x.items()}


def run(x, dev, **kw):
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], None, d["S0"],
                              mode=lr.DIAG_DECAY, **kw)
    torch.cuda.synchronize()
    return o, st


def ref(x):
    return oracle.recurrent(oracle.DIAG_DECAY, x["q"], x["k"], x["v"], x["alpha"], None, x["S0"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 17, 64, 65, 200])
def test_diag_chunked_small(dev, dtype, dk, dv, T):
    x = workloads.draw("gla", 2, 3, T, dk, dv, seed=700 + T + dk + 3 * dv, dtype=dtype,
                       s0_std=0.2 if T % 2 else 0.0)
    o, st = run(x, dev)
    o_ref, s_ref = ref(x)
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= TOL[dtype] and es <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk", [64, 128])
def test_diag_strong_decay(dev, dtype, dk):
    """Gates of about sigmoid(-2): per-channel decays near e^-136 over a block,
    beyond what one reference point per block could hold in fp32."""
    x = workloads.draw("gla_strong", 1, 4, 64 * 4 + 9, dk, 64, seed=41 + dk, dtype=dtype,
                       s0_std=0.5)
    o, st = run(x, dev)
    o_ref, s_ref = ref(x)
    assert np.all(np.isfinite(o.float().cpu().numpy()))
    assert rel_err(o, o_ref) <= TOL[dtype] and rel_err(st, s_ref) <= TOL[dtype]


def test_diag_equal_channels_match_scalar_gate(dev):
    """Equal gates on every channel give the scalar-gate (DECAY) result."""
    x = workloads.draw("mamba2", 2, 2, 150, 128, 128, seed=9, dtype=torch.bfloat16, s0_std=0.1)
    d = to_dev(x, dev)
    a_diag = d["alpha"][..., None].expand(2, 2, 150, 128).contiguous()
    o1, s1 = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], a_diag, None, d["S0"], mode=lr.DIAG_DECAY)
    o2, s2 = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], None, d["S0"], mode=lr.DECAY)
    torch.cuda.synchronize()
    assert rel_err(o1, o2.float().cpu().numpy()) <= 2e-2 and rel_err(s1, s2.cpu().numpy()) <= 2e-2


def test_diag_workload_full_size(dev):
    """The GLA workload (B=8, H=16, T=4096, d=128, bf16): every output and the
    whole final state."""
    w = workloads.WORKLOADS["gla_bf16"]
    x = workloads.draw_workload(w)
    o, st = run(x, dev)
    o_ref, s_ref = ref(x)
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"gla_bf16: rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= 2e-2 and es <= 2e-2


def test_diag_repeated_calls_bit_identical(dev):
    x = to_dev(workloads.draw("gla", 4, 16, 2048, 128, 128, seed=5, dtype=torch.bfloat16,
                              s0_std=0.1), dev)
    ws = torch.empty(lr.workspace_size(4, 16, 2048, 128, 128, torch.bfloat16, lr.DIAG_DECAY),
                     dtype=torch.uint8, device=dev)
    o0, s0 = lr.lr_fwd_chunked(x["q"], x["k"], x["v"], x["alpha"], None, x["S0"],
                               mode=lr.DIAG_DECAY, workspace=ws)
    o, st = torch.empty_like(o0), torch.empty_like(s0)
    bad = 0
    for _ in range(50):
        lr.lr_fwd_chunked(x["q"], x["k"], x["v"], x["alpha"], None, x["S0"], mode=lr.DIAG_DECAY,
                          o=o, S_T=st, workspace=ws)
        bad += int(not (torch.equal(o, o0) and torch.equal(st, s0)))
    torch.cuda.synchronize()
    assert bad == 0, f"{bad} of 50 calls differ from the first"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", ["gate_norm", "gate_norm_qk"])
def test_diag_fused(dev, dtype, flags):
    """GLA's gate sigmoid(a)^(1/16) per channel, the output RMSNorm, and (second
    case) SiLU + L2 of q and k, in the kernels."""
    fl = workloads.FUSED_FLAGS["gla"] | (lr.FUSE_QK_SILU_L2 if flags == "gate_norm_qk" else 0)
    x = workloads.draw_pre("gla", 2, 3, 64 * 3 + 5, 128, 64, seed=17, dtype=dtype, s0_std=0.3)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], d["alpha"], None, d["S0"],
                                    mode=lr.DIAG_DECAY, flags=fl, alpha_scale=d["alpha_scale"],
                                    norm_weight=d["norm_weight"])
    torch.cuda.synchronize()
    f = {n: (t.double().numpy() if t is not None else None) for n, t in x.items()}
    o_ref, s_ref = P.fused(oracle.DIAG_DECAY, fl, f["q"], f["k"], f["v"], f["alpha"], None, f["S0"],
                           alpha_scale=f["alpha_scale"], norm_weight=f["norm_weight"])
    assert rel_err(o, o_ref) <= TOL[dtype] and rel_err(st, s_ref) <= TOL[dtype]


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
def test_diag_step(dev, dtype, dk, dv):
    N, H, T = 5, 3, 4
    x = workloads.draw("gla_strong", N, H, T, dk, dv, seed=13 + dk + dv, dtype=dtype, s0_std=0.3)
    S = x["S0"].to(dev)
    outs = []
    for t in range(T):
        c = lambda n: x[n][:, :, t].contiguous().to(dev)
        outs.append(lr.lr_step(c("q"), c("k"), c("v"), c("alpha"), None, S, mode=lr.DIAG_DECAY))
    torch.cuda.synchronize()
    o_ref, s_ref = ref(x)
    assert rel_err(torch.stack(outs, 2), o_ref) <= TOL[dtype]
    assert rel_err(S, s_ref) <= TOL[dtype]


def test_diag_step_fused(dev):
    N, H, T, d = 4, 2, 3, 128
    fl = workloads.FUSED_FLAGS["gla"] | lr.FUSE_QK_SILU_L2
    x = workloads.draw_pre("gla", N, H, T, d, d, seed=23, dtype=torch.bfloat16, s0_std=0.3)
    dd = to_dev(x, dev)
    S = dd["S0"].clone()
    outs = []
    for t in range(T):
        c = lambda n: dd[n][:, :, t].contiguous()
        outs.append(lr.lr_step_fused(c("q"), c("k"), c("v"), c("alpha"), None, S,
                                     mode=lr.DIAG_DECAY, flags=fl, alpha_scale=dd["alpha_scale"],
                                     norm_weight=dd["norm_weight"]))
    torch.cuda.synchronize()
    f = {n: (t.double().numpy() if t is not None else None) for n, t in x.items()}
    o_ref, s_ref = P.fused(oracle.DIAG_DECAY, fl, f["q"], f["k"], f["v"], f["alpha"], None, f["S0"],
                           alpha_scale=f["alpha_scale"], norm_weight=f["norm_weight"])
    assert rel_err(torch.stack(outs, 2), o_ref) <= 2e-2
    assert rel_err(S, s_ref) <= 2e-2

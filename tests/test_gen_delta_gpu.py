"""Parity of the generalised delta rule (RWKV-7 reading; lr_fwd_chunked_gen_delta,
lr_step_gen_delta) with the fp64 oracle, through the C ABI.  Bars as for the
other rows: max|gpu - oracle| / max|oracle| per tensor, 1e-4 for fp32 inputs
(the CUDA-core kernel) and 2e-2 for bf16 inputs (the tensor-core path: bf16
operands, fp32 accumulation and state; the decode step widens to fp32)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import workloads
from oracle.gen_delta import recurrent

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
NAMES = ("q", "kw", "v", "w", "kappa", "a")


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
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30)) if ref.size else 0.0


def to_dev(x, dev):
    return {n: (t.to(dev) if t is not None else None) for n, t in x.items()}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 31, 32, 33, 100, 257])
def test_gen_delta_chunked(dev, dtype, dk, dv, T):
    x = workloads.draw_gen_delta(2, 3, T, dk, dv, seed=60 + T + dk + dv, dtype=dtype,
                                 state=bool(T % 2))
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_gen_delta(*(d[n] for n in NAMES), d["S0"])
    torch.cuda.synchronize()
    o_ref, s_ref = recurrent(*(x[n] for n in NAMES), x["S0"])
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= TOL[dtype] and es <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gen_delta_reflection_keeps_count(dev, dtype):
    """Rate 2 with w = 1 reflects the memory along the removal key (eigenvalue
    -1): after an even number of reflections and nothing written, the memory
    is back where it started (bf16: the pseudo-values u = S kappa are rounded
    once per block, so within the bf16 bar)."""
    B, H, T, d = 1, 2, 6, 64
    kap = torch.randn((B, H, 1, d))
    kap = (kap / kap.norm(dim=-1, keepdim=True)).expand(B, H, T, d).contiguous()
    z = torch.zeros((B, H, T, d))
    S0 = torch.randn((B, H, d, d)) * 0.1
    o, st = lr.lr_fwd_chunked_gen_delta(z.to(dtype).to(dev), z.to(dtype).to(dev),
                                        z.to(dtype).to(dev), torch.ones_like(z).to(dev),
                                        kap.to(dev), torch.full_like(z, 2.0).to(dev), S0.to(dev))
    torch.cuda.synchronize()
    assert rel_err(st, S0.numpy()) <= (1e-5 if dtype == torch.float32 else TOL[dtype])


def test_gen_delta_strong_decay(dev):
    """Decays down to w = 0.01 per token (a factor e^-74 across 16 tokens, near
    the e^-80 limit of the bf16 path's split of the decay) against the oracle."""
    x = workloads.draw_gen_delta(1, 4, 200, 128, 128, seed=31, dtype=torch.bfloat16, state=True)
    g = torch.Generator().manual_seed(5)
    x["w"] = (0.01 + 0.99 * torch.rand(x["w"].shape, generator=g)).contiguous()
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_gen_delta(*(d[n] for n in NAMES), d["S0"])
    torch.cuda.synchronize()
    o_ref, s_ref = recurrent(*(x[n] for n in NAMES), x["S0"])
    assert np.all(np.isfinite(o.float().cpu().numpy()))
    assert rel_err(o, o_ref) <= 2e-2 and rel_err(st, s_ref) <= 2e-2


def test_gen_delta_workload_full_size(dev):
    """B=2, H=16, T=4096, d=128, bf16 with an initial state: every output and
    the whole final state against the oracle."""
    w = workloads.WORKLOADS["rwkv7_bf16"]
    x = workloads.draw_gen_delta(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=torch.bfloat16,
                                 state=True)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_gen_delta(*(d[n] for n in NAMES), d["S0"])
    torch.cuda.synchronize()
    o_ref, s_ref = recurrent(*(x[n] for n in NAMES), x["S0"])
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"full size: rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= 2e-2 and es <= 2e-2


def test_gen_delta_resume_equals_one_call(dev):
    """The final state is the checkpoint: two calls (split inside a block)
    give the one-call result within the bar."""
    x = workloads.draw_gen_delta(1, 3, 300, 128, 128, seed=19, dtype=torch.bfloat16, state=True)
    d = to_dev(x, dev)
    o1, s1 = lr.lr_fwd_chunked_gen_delta(*(d[n][:, :, :150].contiguous() for n in NAMES), d["S0"])
    o2, s2 = lr.lr_fwd_chunked_gen_delta(*(d[n][:, :, 150:].contiguous() for n in NAMES), s1)
    torch.cuda.synchronize()
    o_ref, s_ref = recurrent(*(x[n] for n in NAMES), x["S0"])
    assert rel_err(torch.cat([o1, o2], 2), o_ref) <= 2e-2 and rel_err(s2, s_ref) <= 2e-2


def test_gen_delta_empty_sequence(dev):
    x = workloads.draw_gen_delta(1, 2, 0, 64, 64, seed=2, dtype=torch.bfloat16, state=True)
    d = to_dev(x, dev)
    o, st = lr.lr_fwd_chunked_gen_delta(*(d[n] for n in NAMES), d["S0"])
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.equal(st.cpu(), x["S0"])


def test_gen_delta_matches_delta_rule_path(dev):
    """w = 1, kappa = k, a = beta, kw = beta k gives the delta rule: the result
    matches lr_fwd_chunked in DELTA mode (the tensor-core path) on the same
    bf16 inputs, up to the two paths' rounding."""
    x = workloads.draw("gdn", 1, 4, 200, 128, 128, seed=12, dtype=torch.bfloat16, s0_std=0.1)
    d = to_dev(x, dev)
    bd = d["beta"][..., None].expand(1, 4, 200, 128).contiguous()
    kf = d["k"].float()
    o1, s1 = lr.lr_fwd_chunked_gen_delta(d["q"], (bd * kf).to(torch.bfloat16), d["v"],
                                         torch.ones_like(bd), kf.contiguous(), bd, d["S0"])
    o2, s2 = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], None, d["beta"], d["S0"], mode=lr.DELTA)
    torch.cuda.synchronize()
    assert rel_err(o1, o2.float().cpu().numpy()) <= 2e-2 and rel_err(s1, s2.cpu().numpy()) <= 2e-2


def test_gen_delta_repeated_calls_bit_identical(dev):
    x = to_dev(workloads.draw_gen_delta(2, 16, 1024, 128, 128, seed=2, dtype=torch.bfloat16), dev)
    ws = torch.empty(lr.gen_delta_workspace_size(2, 16, 1024, 128, 128, torch.bfloat16),
                     dtype=torch.uint8, device=dev)
    o0, s0 = lr.lr_fwd_chunked_gen_delta(*(x[n] for n in NAMES), workspace=ws)
    bad = 0
    for _ in range(20):
        o, st = lr.lr_fwd_chunked_gen_delta(*(x[n] for n in NAMES), workspace=ws)
        bad += int(not (torch.equal(o, o0) and torch.equal(st, s0)))
    torch.cuda.synchronize()
    assert bad == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
def test_gen_delta_step(dev, dtype, dk, dv):
    N, H, T = 5, 3, 4
    x = workloads.draw_gen_delta(N, H, T, dk, dv, seed=90 + dk + dv, dtype=dtype, state=True)
    d = to_dev(x, dev)
    S = d["S0"].clone()
    outs = []
    for t in range(T):
        outs.append(lr.lr_step_gen_delta(*(d[n][:, :, t].contiguous() for n in NAMES), S))
    torch.cuda.synchronize()
    o_ref, s_ref = recurrent(*(x[n] for n in NAMES), x["S0"])
    assert rel_err(torch.stack(outs, 2), o_ref) <= TOL[dtype]
    assert rel_err(S, s_ref) <= TOL[dtype]

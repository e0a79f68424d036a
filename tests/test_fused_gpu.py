"""Parity of the fused entry points (the maps around the recurrence applied in
the library's kernels) with the fp64 oracle of those maps followed by the
recurrence (``oracle.prologue.fused``).

The oracle receives the same pre-activation inputs as the library (q, k, v
rounded once to the input dtype) and keeps everything after that in fp64,
including the normalised q and k that the bf16 path rounds to bf16.  Metric
and bars as for the plain entry points: max|gpu - oracle| / max|oracle| per
tensor, 1e-4 for fp32 inputs and 2e-2 for bf16.  Inputs that use the output
RMSNorm start from a nonzero state, so that no read-out row is a near-zero
difference whose normalisation would magnify rounding (the RMSNorm of a row
is only as accurate, relative to the row, as the row itself).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import workloads
from oracle import prologue as P

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
ALL = lr.FUSE_QK_SILU_L2 | lr.FUSE_BETA_SIGMOID | lr.FUSE_ALPHA_SIGMOID | lr.FUSE_O_RMSNORM


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


def inputs(gen, B, H, T, dk, dv, seed, dtype, s0_std, flags):
    """Pre-activation values for the mapped inputs, already-mapped values (the
    plain generator's, same seed) for the others."""
    pre = workloads.draw_pre(gen, B, H, T, dk, dv, seed=seed, dtype=dtype, s0_std=s0_std)
    if gen == "gdn":
        post = workloads.draw("gdn", B, H, T, dk, dv, seed=seed, dtype=dtype, s0_std=s0_std)
        x = dict(pre)
        if not flags & lr.FUSE_QK_SILU_L2:
            x["q"], x["k"] = post["q"], post["k"]
        if not flags & lr.FUSE_BETA_SIGMOID:
            x["beta"] = post["beta"]
        if not flags & (lr.FUSE_ALPHA_SIGMOID | lr.FUSE_ALPHA_SOFTPLUS):
            x["alpha"] = post["alpha"]
        if flags & lr.FUSE_ALPHA_SOFTPLUS:
            x["alpha"] = pre["alpha"] - 3.0       # pre-activations ~ N(0, 1)
            x["alpha_scale"] = 0.1 * torch.arange(1, H + 1, dtype=torch.float32)
        return x
    pre["q"] = (pre["q"].float() / np.sqrt(dk)).to(dtype)
    pre["k"] = (pre["k"].float() / np.sqrt(dk)).to(dtype)
    return pre


def run_fused(x, mode, flags, dev, eps=1e-6):
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, st = lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                    mode=mode, flags=flags, alpha_scale=d["alpha_scale"],
                                    norm_weight=d["norm_weight"], norm_eps=eps)
    torch.cuda.synchronize()
    return o, st


def ref_fused(x, mode, flags, eps=1e-6):
    return P.fused(mode, flags, x["q"].double().numpy(), x["k"].double().numpy(),
                   x["v"].double().numpy(), x["alpha"].double().numpy(),
                   x["beta"].double().numpy(), None if x["S0"] is None else x["S0"].double().numpy(),
                   alpha_scale=x["alpha_scale"].double().numpy(),
                   norm_weight=x["norm_weight"].double().numpy(), norm_eps=eps)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 64, 65, 200])
def test_fused_gated_delta_all_maps(dev, dtype, dk, dv, T):
    x = inputs("gdn", 2, 3, T, dk, dv, seed=500 + T + dk + dv, dtype=dtype, s0_std=0.3,
               flags=ALL)
    o, st = run_fused(x, lr.GATED_DELTA, ALL, dev)
    o_ref, s_ref = ref_fused(x, lr.GATED_DELTA, ALL)
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= TOL[dtype] and es <= TOL[dtype]


FLAG_SETS = {
    "qk": lr.FUSE_QK_SILU_L2,
    "beta": lr.FUSE_BETA_SIGMOID,
    "alpha_sigmoid": lr.FUSE_ALPHA_SIGMOID,
    "alpha_softplus": lr.FUSE_ALPHA_SOFTPLUS,
    "rmsnorm": lr.FUSE_O_RMSNORM,
    "gates": lr.FUSE_BETA_SIGMOID | lr.FUSE_ALPHA_SOFTPLUS,
}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode", [lr.LINEAR, lr.DECAY, lr.DELTA, lr.GATED_DELTA],
                         ids=["linear", "decay", "delta", "gated_delta"])
@pytest.mark.parametrize("fs", sorted(FLAG_SETS))
def test_fused_each_map(dev, dtype, mode, fs):
    """Each map on its own, in every mode (maps of gates a mode does not use
    are ignored)."""
    flags = FLAG_SETS[fs]
    x = inputs("gdn", 1, 3, 130, 64, 64, seed=900 + mode, dtype=dtype, s0_std=0.3, flags=flags)
    o, st = run_fused(x, mode, flags, dev)
    o_ref, s_ref = ref_fused(x, mode, flags)
    assert rel_err(o, o_ref) <= TOL[dtype] and rel_err(st, s_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_fused_mamba2_softplus_gate(dev, dtype):
    flags = workloads.FUSED_FLAGS["mamba2"]
    x = inputs("mamba2", 2, 4, 64 * 3 + 9, 128, 128, seed=41, dtype=dtype, s0_std=0.3, flags=flags)
    o, st = run_fused(x, lr.DECAY, flags, dev)
    o_ref, s_ref = ref_fused(x, lr.DECAY, flags)
    assert rel_err(o, o_ref) <= TOL[dtype] and rel_err(st, s_ref) <= TOL[dtype]


def test_fused_no_flags_equals_plain(dev):
    """flags 0 is the plain call, bit for bit."""
    x = {n: (t.to(dev) if t is not None else None) for n, t in
         workloads.draw("gdn", 2, 2, 150, 128, 128, seed=3, dtype=torch.bfloat16, s0_std=0.1).items()}
    o1, s1 = lr.lr_fwd_chunked(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"])
    o2, s2 = lr.lr_fwd_chunked_fused(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["S0"], flags=0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_fused_qk_matches_pre_normalised_inputs(dev):
    """The bf16 path with SiLU + L2 in the kernel gives the result of the plain
    path on q, k normalised in fp32 and rounded to bf16 beforehand, up to
    rounding ties: the normalised rows it stores are what the scan reads."""
    x = workloads.draw_pre("gdn", 1, 4, 64 * 4 + 5, 128, 128, seed=12, dtype=torch.bfloat16,
                           s0_std=0.1)
    post = workloads.draw("gdn", 1, 4, 64 * 4 + 5, 128, 128, seed=12, dtype=torch.bfloat16,
                          s0_std=0.1)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    a, b = post["alpha"].to(dev), post["beta"].to(dev)
    o1, s1 = lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], a, b, d["S0"],
                                     flags=lr.FUSE_QK_SILU_L2)

    def silu_l2_f32(t):
        t = t.float()
        t = t * torch.sigmoid(t)
        return (t / torch.clamp(t.norm(dim=-1, keepdim=True), min=1e-12)).to(torch.bfloat16)
    o2, s2 = lr.lr_fwd_chunked(silu_l2_f32(d["q"]), silu_l2_f32(d["k"]), d["v"], a, b, d["S0"])
    torch.cuda.synchronize()
    assert rel_err(o1, o2.float().cpu().numpy()) <= 1e-2
    assert rel_err(s1, s2.cpu().numpy()) <= 1e-2


def test_fused_empty_sequence(dev):
    x = inputs("gdn", 1, 2, 0, 64, 64, seed=4, dtype=torch.bfloat16, s0_std=0.3, flags=ALL)
    o, st = run_fused(x, lr.GATED_DELTA, ALL, dev)
    assert o.shape == (1, 2, 0, 64)
    assert torch.equal(st.cpu(), x["S0"])


def test_fused_workspace_size(dev):
    plain = lr.fused_workspace_size(2, 3, 100, 128, 64, torch.bfloat16, flags=0)
    qk = lr.fused_workspace_size(2, 3, 100, 128, 64, torch.bfloat16, flags=lr.FUSE_QK_SILU_L2)
    assert plain == lr.workspace_size(2, 3, 100, 128, 64, torch.bfloat16)
    assert qk - plain == 2 * 2 * 3 * 100 * 128 * 2
    assert lr.fused_workspace_size(2, 3, 100, 128, 64, torch.float32, flags=ALL) == 0


def test_fused_gdn_prefill_full_size(dev):
    """The full-size gated-delta prefill (B=2, H=16, T=16384, d=128, bf16) with
    every map: every output and the whole final state."""
    w = workloads.WORKLOADS["gdn_prefill_bf16"]
    flags = workloads.FUSED_FLAGS["gdn"]
    x = workloads.draw_pre("gdn", w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=w.torch_dtype,
                           s0_std=w.s0_std)
    o, st = run_fused(x, w.mode, flags, dev)
    o_ref, s_ref = ref_fused(x, w.mode, flags)
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"fused gdn prefill: rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= 2e-2 and es <= 2e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("case", ["strong_decay", "full_dose", "zero_dose", "alpha_one"])
def test_fused_gates_at_domain_ends(dev, dtype, case):
    """The maps driven to the ends of the gates' ranges (page "Scrivere meglio
    nella memoria": sigmoid write strength, sigmoid or softplus forget gate):
    sigmoid(-3 + N(0,1)) forgets a 64-token block far below e^-80; beta
    pre-activations of +40 and -40 give a full dose (1.0 in fp32) and a dose of
    about 4e-18; a softplus gate of -100 gives alpha = 1 to fp32 precision."""
    flags = ALL
    x = inputs("gdn", 2, 3, 200, 128, 128, seed=4600, dtype=dtype, s0_std=0.3, flags=flags)
    if case == "strong_decay":
        x["alpha"] = (x["alpha"] - 6.0).contiguous()          # N(-3, 1) before the sigmoid
        # without the output norm: once the state is forgotten within a few
        # tokens some read-out rows are 2000x smaller than others, and the
        # per-row norm lifts their rounding to the scale of the largest row
        # (the bf16 rounding of the normalised q and k alone gives 3.4e-2
        # after the norm and 1.7e-3 before it, in the fp64 oracle)
        flags = ALL & ~lr.FUSE_O_RMSNORM
    elif case == "full_dose":
        x["beta"] = torch.full_like(x["beta"], 40.0)
    elif case == "zero_dose":
        x["beta"] = torch.full_like(x["beta"], -40.0)
        flags = ALL & ~lr.FUSE_O_RMSNORM
    else:
        flags = (ALL & ~lr.FUSE_ALPHA_SIGMOID) | lr.FUSE_ALPHA_SOFTPLUS
        x["alpha"] = torch.full_like(x["alpha"], -100.0)
        x["alpha_scale"] = torch.ones(3)
    o, st = run_fused(x, lr.GATED_DELTA, flags, dev)
    o_ref, s_ref = ref_fused(x, lr.GATED_DELTA, flags)
    eo, es = rel_err(o, o_ref), rel_err(st, s_ref)
    print(f"{case}: rel err o={eo:.3e} S_T={es:.3e}")
    assert eo <= TOL[dtype] and es <= TOL[dtype]


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode", [lr.DECAY, lr.DELTA, lr.GATED_DELTA],
                         ids=["decay", "delta", "gated_delta"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
@pytest.mark.parametrize("fs", ["all", "softplus"])
def test_step_fused(dev, dtype, mode, dk, dv, fs):
    N, H, T = 5, 3, 4
    flags = ALL if fs == "all" else (lr.FUSE_QK_SILU_L2 | lr.FUSE_ALPHA_SOFTPLUS |
                                     lr.FUSE_BETA_SIGMOID)
    x = inputs("gdn", N, H, T, dk, dv, seed=77 + dk + dv + mode, dtype=dtype, s0_std=0.3,
               flags=flags)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    S = d["S0"].clone()
    outs = []
    for t in range(T):
        c = lambda n: d[n][:, :, t].contiguous()
        outs.append(lr.lr_step_fused(c("q"), c("k"), c("v"), c("alpha"), c("beta"), S, mode=mode,
                                     flags=flags, alpha_scale=d["alpha_scale"],
                                     norm_weight=d["norm_weight"]))
    torch.cuda.synchronize()
    o_ref, s_ref = ref_fused(x, mode, flags)
    assert rel_err(torch.stack(outs, 2), o_ref) <= TOL[dtype]
    assert rel_err(S, s_ref) <= TOL[dtype]


def test_step_fused_decode_workload_sampled(dev):
    """The decode workload's shape (512 x 32 states, d = 128, bf16) with every
    map, 20 consecutive steps: all heads after the first step, 64 sampled
    (sequence, head) pairs over all 20."""
    w = workloads.WORKLOADS["gdn_decode_bf16"]
    flags = workloads.FUSED_FLAGS["gdn"]
    g = torch.Generator(dev)
    S = workloads.draw_decode_state(w, dev, g)
    wn = (0.5 + torch.rand((w.dv,), generator=g, device=dev)).float()
    rng = np.random.default_rng(7)
    pick = rng.choice(w.B * w.H, size=64, replace=False)
    pn = torch.tensor(pick // w.H, device=dev)
    ph = torch.tensor(pick % w.H, device=dev)
    S_all0 = S.cpu().double().numpy()
    S0_pick = S[pn, ph].cpu()
    seq = {n: [] for n in ("q", "k", "v", "alpha", "beta", "o")}
    for step in range(20):
        inp = workloads.draw_decode_step_pre(w, step, dev, g)
        o = lr.lr_step_fused(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], S,
                             mode=w.mode, flags=flags, norm_weight=wn)
        if step == 0:
            torch.cuda.synchronize()
            c = {n: t.cpu().double().numpy()[:, :, None] for n, t in inp.items()}
            o_ref, s_ref = P.fused(w.mode, flags, c["q"], c["k"], c["v"], c["alpha"], c["beta"],
                                   S_all0, norm_weight=wn.cpu().double().numpy())
            assert rel_err(o, o_ref[:, :, 0]) <= 2e-2
            assert rel_err(S, s_ref) <= 2e-2
            del S_all0, c, o_ref, s_ref
        for n in ("q", "k", "v", "alpha", "beta"):
            seq[n].append(inp[n][pn, ph].cpu())
        seq["o"].append(o[pn, ph].cpu())
    torch.cuda.synchronize()
    st = lambda n: torch.stack(seq[n], dim=1).unsqueeze(1).double().numpy()
    o_ref, s_ref = P.fused(w.mode, flags, st("q"), st("k"), st("v"), st("alpha"), st("beta"),
                           S0_pick.unsqueeze(1).double().numpy(),
                           norm_weight=wn.cpu().double().numpy())
    eo = rel_err(torch.from_numpy(st("o")), o_ref)
    es = rel_err(S[pn, ph].unsqueeze(1), s_ref)
    print(f"fused decode 20 steps, 64 sampled heads: rel err o={eo:.3e} S={es:.3e}")
    assert eo <= 2e-2 and es <= 2e-2


def test_fused_folded_norm_repeated_calls_bit_identical(dev):
    """The scan that applies the output norm (2-CTA clusters exchanging row sums
    through distributed shared memory, on the Mamba-2 workload's 64-channel
    CTAs): 30 calls on the same inputs give the same bits."""
    w = workloads.WORKLOADS["mamba2_gate_bf16"]
    flags = workloads.FUSED_FLAGS["mamba2"]
    x = workloads.draw_pre("mamba2", w.B, w.H, w.T, w.dk, w.dv, w.seed, torch.bfloat16, w.s0_std)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}

    def call():
        return lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                       mode=w.mode, flags=flags, alpha_scale=d["alpha_scale"],
                                       norm_weight=d["norm_weight"])

    o0, s0 = [t.clone() for t in call()]
    bad = 0
    for _ in range(30):
        o, s = call()
        bad += int(not (torch.equal(o, o0) and torch.equal(s, s0)))
    torch.cuda.synchronize()
    assert bad == 0, f"{bad} of 30 calls differ from the first"

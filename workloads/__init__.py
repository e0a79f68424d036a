"""Seeded synthetic inputs for the gated delta rule family.

This module only draws and shapes random inputs; it holds none of the
method's arithmetic.  Tests, the smoke check and the benchmark use it to give
the CUDA library and the fp64 oracle the same inputs.

The feature maps applied here belong to the model layer around the memory,
not to the memory itself (page "Scrivere meglio nella memoria: gate e delta
rule", opening section: the feature map is absorbed in the projections that
produce q and k -- DeltaNet puts a SiLU followed by an L2 normalisation
there -- and beta comes from a sigmoid):

* ``gdn`` inputs: q, k = L2norm(SiLU(N(0,1))) per token; v ~ N(0,1);
  beta = sigmoid(N(0,1)); alpha = sigmoid(N(3,1)); S0 = 0 or N(0, 0.1^2).
* ``gdn_strong``: as ``gdn`` with alpha = sigmoid(N(-3,1)) (about 0.05 per
  token): a 64-token block decays near e^-190, far beyond fp32's range for
  one reference point per block, so the kernels' direct-difference form of
  the decay mask is the one that runs.
* ``retnet``: q, k, v ~ N(0,1)/sqrt(dk); alpha = gamma_h = 1 - 2^(-5-h) for
  head h = 0..H-1, the same at every token.
* ``mamba2``: q, k ~ N(0,1)/sqrt(dk); v ~ N(0,1);
  alpha = exp(-0.1 softplus(N(0,1))).
* ``gla`` (diagonal gate, alpha [B,H,T,dk]): q, k ~ N(0,1)/sqrt(dk); v ~ N(0,1);
  alpha = sigmoid(N(0,1))^(1/16) per key channel (GLA's gate with tau = 16,
  first page, gates section).
* ``gla_strong``: as ``gla`` with alpha = sigmoid(N(-2,1)): decays near e^-136
  over a 64-token block (beyond fp32's range for one reference point per
  block) and near e^-34 over 16 tokens, which the kernels' 16-token
  sub-blocks must absorb.

Draw order with one ``torch.Generator('cpu')``: q, k, v, beta, alpha, S0.
Values are drawn in fp32 and, for bf16 workloads, rounded to bf16 once; the
oracle consumes the rounded values.
"""
from __future__ import annotations

import dataclasses
import math

import torch

LINEAR, DECAY, DELTA, GATED_DELTA, DIAG_DECAY = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: int
    dtype: str          # "f32" or "bf16": element type of q, k, v, o
    B: int
    H: int
    T: int
    dk: int
    dv: int
    chunk: int
    seed: int
    gen: str            # "gdn", "retnet" or "mamba2"
    s0_std: float       # 0 -> S0 = None (zeros)
    steps: int = 0      # decode workloads: number of consecutive steps (T unused)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def describe(self):
        return dataclasses.asdict(self)


# The five workloads: (1) gated delta fp32 small; (2) RetNet retention;
# (3) Mamba-2-style scalar gate; (4) gated delta long prefill; (5) gated delta
# decode, 1000 consecutive steps over 512 sequences x 32 heads.
WORKLOADS = {
    "gdn_fp32_small": Workload("gdn_fp32_small", GATED_DELTA, "f32", 1, 2, 256, 32, 32, 64, 0,
                               "gdn", 0.0),
    "retnet_bf16": Workload("retnet_bf16", DECAY, "bf16", 4, 8, 2048, 128, 128, 64, 2,
                            "retnet", 0.0),
    "mamba2_gate_bf16": Workload("mamba2_gate_bf16", DECAY, "bf16", 8, 16, 4096, 128, 128, 64, 3,
                                 "mamba2", 0.0),
    "gdn_prefill_bf16": Workload("gdn_prefill_bf16", GATED_DELTA, "bf16", 2, 16, 16384, 128, 128,
                                 64, 4, "gdn", 0.1),
    "gdn_decode_bf16": Workload("gdn_decode_bf16", GATED_DELTA, "bf16", 512, 32, 1, 128, 128, 64,
                                5, "gdn", 0.1, steps=1000),
    # the diagonal gate (GLA row), at the Mamba-2-style workload's size
    "gla_bf16": Workload("gla_bf16", DIAG_DECAY, "bf16", 8, 16, 4096, 128, 128, 64, 6, "gla", 0.0),
    # the mLSTM memory, same size (mode: the scalar-gate engine; inputs from draw_mlstm)
    "mlstm_bf16": Workload("mlstm_bf16", DECAY, "bf16", 8, 16, 4096, 128, 128, 64, 7, "mlstm", 0.0),
    # the generalised delta rule of RWKV-7 (inputs from draw_gen_delta; CUDA-core path)
    "rwkv7_bf16": Workload("rwkv7_bf16", DELTA, "bf16", 2, 16, 4096, 128, 128, 64, 8, "gd", 0.1),
}


def _silu_l2(x):
    x = x * torch.sigmoid(x)
    return x / torch.clamp(torch.linalg.vector_norm(x, dim=-1, keepdim=True), min=1e-12)


def retnet_gamma(H: int) -> torch.Tensor:
    """Per-head fixed decay 1 - 2^(-5-h), h = 0..H-1 (multi-scale retention)."""
    return 1.0 - torch.pow(2.0, -5.0 - torch.arange(H, dtype=torch.float64)).float()


def draw(gen: str, B, H, T, dk, dv, seed, dtype=torch.float32, s0_std=0.0, device="cpu"):
    """Draw one input set.  Returns dict q, k, v, alpha, beta, S0 (S0 may be None).

    Shapes: q, k [B,H,T,dk]; v [B,H,T,dv]; alpha, beta [B,H,T] fp32 (alpha
    [B,H,T,dk] for the diagonal-gate generators); S0 [B,H,dv,dk] fp32.  q, k, v are rounded once to ``dtype``.  Drawn on
    the CPU generator and then moved to ``device``.
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    shp_k, shp_v, shp_t = (B, H, T, dk), (B, H, T, dv), (B, H, T)
    if gen in ("gdn", "gdn_strong"):
        q = _silu_l2(torch.randn(shp_k, generator=g))
        k = _silu_l2(torch.randn(shp_k, generator=g))
        v = torch.randn(shp_v, generator=g)
        beta = torch.sigmoid(torch.randn(shp_t, generator=g))
        mu = 3.0 if gen == "gdn" else -3.0
        alpha = torch.sigmoid(mu + torch.randn(shp_t, generator=g))
    elif gen == "retnet":
        s = 1.0 / math.sqrt(dk)
        q = torch.randn(shp_k, generator=g) * s
        k = torch.randn(shp_k, generator=g) * s
        v = torch.randn(shp_v, generator=g) * s
        beta = torch.zeros(shp_t)
        alpha = retnet_gamma(H).view(1, H, 1).expand(B, H, T).contiguous()
    elif gen == "mamba2":
        s = 1.0 / math.sqrt(dk)
        q = torch.randn(shp_k, generator=g) * s
        k = torch.randn(shp_k, generator=g) * s
        v = torch.randn(shp_v, generator=g)
        beta = torch.zeros(shp_t)
        alpha = torch.exp(-0.1 * torch.nn.functional.softplus(torch.randn(shp_t, generator=g)))
    elif gen in ("gla", "gla_strong"):
        s = 1.0 / math.sqrt(dk)
        q = torch.randn(shp_k, generator=g) * s
        k = torch.randn(shp_k, generator=g) * s
        v = torch.randn(shp_v, generator=g)
        beta = torch.zeros(shp_t)
        if gen == "gla":
            alpha = torch.sigmoid(torch.randn(shp_k, generator=g)) ** (1.0 / 16.0)
        else:
            alpha = torch.sigmoid(torch.randn(shp_k, generator=g) - 2.0)
    elif gen == "uniform":
        # generic small-case inputs: keys of norm <= 1, gates in (0.5, 1)
        q = torch.randn(shp_k, generator=g) / math.sqrt(dk)
        k = _silu_l2(torch.randn(shp_k, generator=g))
        v = torch.randn(shp_v, generator=g)
        beta = torch.rand(shp_t, generator=g)
        alpha = 0.5 + 0.5 * torch.rand(shp_t, generator=g)
    else:
        raise ValueError(gen)
    S0 = torch.randn((B, H, dv, dk), generator=g) * s0_std if s0_std > 0 else None
    out = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), alpha=alpha.float().contiguous(),
               beta=beta.float().contiguous(), S0=S0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


# lr_fuse flags (the library's LR_FUSE_* bits) of the pre-activation inputs
# of each generator: the gated-delta layer maps q, k, beta and alpha and
# normalises o; the Mamba-2-style layer maps alpha by the softplus gate.
FUSE_QK_SILU_L2, FUSE_BETA_SIGMOID, FUSE_ALPHA_SIGMOID, FUSE_ALPHA_SOFTPLUS, FUSE_O_RMSNORM = (
    0x1, 0x2, 0x4, 0x8, 0x10)
FUSE_ALPHA_SIGMOID_POW = 0x20
FUSED_FLAGS = {
    "gdn": FUSE_QK_SILU_L2 | FUSE_BETA_SIGMOID | FUSE_ALPHA_SIGMOID | FUSE_O_RMSNORM,
    "mamba2": FUSE_ALPHA_SOFTPLUS | FUSE_O_RMSNORM,
    "gla": FUSE_ALPHA_SIGMOID_POW | FUSE_O_RMSNORM,
}
MAMBA2_ALPHA_SCALE = 0.1
GLA_ALPHA_POWER = 1.0 / 16.0   # GLA's gate sigmoid(.)^(1/tau), tau = 16


def draw_pre(gen: str, B, H, T, dk, dv, seed, dtype=torch.float32, s0_std=0.0, device="cpu"):
    """Pre-activation inputs for the fused entry points (the same distributions
    as :func:`draw` before its maps): q, k, v ~ N(0,1) rounded once to
    ``dtype``; for "gdn" beta ~ N(0,1) and alpha ~ N(3,1) (sigmoid gates), for
    "mamba2" alpha ~ N(0,1) (softplus gate, alpha_scale 0.1 for every head)
    and beta = 0, for "gla" alpha ~ N(0,1) per key channel [B,H,T,dk]
    (sigmoid gate raised to alpha_scale = 1/16) and beta = 0;
    norm_weight ~ U(0.5, 1.5) [dv]; S0 ~ N(0, s0_std^2) or None.

    Returns dict q, k, v, alpha, beta, S0, alpha_scale [H], norm_weight [dv].
    Draw order: q, k, v, beta, alpha, S0, norm_weight.
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    shp_k, shp_v, shp_t = (B, H, T, dk), (B, H, T, dv), (B, H, T)
    q = torch.randn(shp_k, generator=g)
    k = torch.randn(shp_k, generator=g)
    v = torch.randn(shp_v, generator=g)
    if gen == "gdn":
        beta = torch.randn(shp_t, generator=g)
        alpha = 3.0 + torch.randn(shp_t, generator=g)
    elif gen == "mamba2":
        beta = torch.zeros(shp_t)
        alpha = torch.randn(shp_t, generator=g)
    elif gen == "gla":
        beta = torch.zeros(shp_t)
        alpha = torch.randn(shp_k, generator=g)
    else:
        raise ValueError(gen)
    S0 = torch.randn((B, H, dv, dk), generator=g) * s0_std if s0_std > 0 else None
    w = 0.5 + torch.rand((dv,), generator=g)
    scale = GLA_ALPHA_POWER if gen == "gla" else MAMBA2_ALPHA_SCALE
    out = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), alpha=alpha.float().contiguous(),
               beta=beta.float().contiguous(), S0=S0,
               alpha_scale=torch.full((H,), scale), norm_weight=w.float())
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def draw_decode_step_pre(w: Workload, step: int, device, generator=None):
    """Pre-activation inputs of decode step ``step`` (the fused decode entry
    point): q, k, v ~ N(0,1) in the workload dtype; beta ~ N(0,1), alpha ~
    N(3,1) [N,H]."""
    g = generator if generator is not None else torch.Generator(device)
    g.manual_seed(int(w.seed) * 1000003 + int(step))
    N, H, dk, dv = w.B, w.H, w.dk, w.dv
    q = torch.randn((N, H, dk), generator=g, device=device)
    k = torch.randn((N, H, dk), generator=g, device=device)
    v = torch.randn((N, H, dv), generator=g, device=device)
    beta = torch.randn((N, H), generator=g, device=device)
    alpha = 3.0 + torch.randn((N, H), generator=g, device=device)
    dt = w.torch_dtype
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), alpha=alpha.float(), beta=beta.float())


def draw_mlstm(B, H, T, dk, dv, seed, dtype=torch.float32, state=False, igate_std=2.0,
               device="cpu"):
    """mLSTM inputs (page "Le architetture lineari", xLSTM section): q, k ~
    N(0,1)/sqrt(dk), v ~ N(0,1) rounded once to ``dtype``; forget gate
    f = sigmoid(N(3,1)); input-gate pre-activation igate ~ N(0, igate_std^2)
    (the exponential gate e^igate spans several orders of magnitude); with
    ``state`` a stabilised initial state C0 ~ N(0, 0.1^2), n0 ~ N(0, 0.1^2),
    m0 ~ N(0, 1).  Draw order: q, k, v, f, igate, C0, n0, m0.
    Returns dict q, k, v, fgate, igate, C0, n0, m0 (the last three may be None).
    """
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    s = 1.0 / math.sqrt(dk)
    q = torch.randn((B, H, T, dk), generator=g) * s
    k = torch.randn((B, H, T, dk), generator=g) * s
    v = torch.randn((B, H, T, dv), generator=g)
    f = torch.sigmoid(3.0 + torch.randn((B, H, T), generator=g))
    ig = torch.randn((B, H, T), generator=g) * igate_std
    C0 = n0 = m0 = None
    if state:
        C0 = torch.randn((B, H, dv, dk), generator=g) * 0.1
        n0 = torch.randn((B, H, dk), generator=g) * 0.1
        m0 = torch.randn((B, H), generator=g)
    out = dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), fgate=f.float().contiguous(),
               igate=ig.float().contiguous(), C0=C0, n0=n0, m0=m0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def draw_gen_delta(B, H, T, dk, dv, seed, dtype=torch.float32, state=False, device="cpu"):
    """Generalised-delta (RWKV-7) inputs: q, kw ~ N(0,1)/sqrt(dk), v ~ N(0,1)
    rounded once to ``dtype``; decay w = exp(-e^{-1/2} sigmoid(N(0,1))) in
    (0.54, 1); removal key kappa = N(0,1) normalised per token; rate
    a = sigmoid(N(0,1)) per channel; with ``state`` S0 ~ N(0, 0.1^2).
    Draw order: q, kw, v, w, kappa, a, S0."""
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    s = 1.0 / math.sqrt(dk)
    shp = (B, H, T, dk)
    q = torch.randn(shp, generator=g) * s
    kw = torch.randn(shp, generator=g) * s
    v = torch.randn((B, H, T, dv), generator=g)
    w = torch.exp(-math.exp(-0.5) * torch.sigmoid(torch.randn(shp, generator=g)))
    kap = torch.randn(shp, generator=g)
    kap = kap / torch.linalg.vector_norm(kap, dim=-1, keepdim=True)
    a = torch.sigmoid(torch.randn(shp, generator=g))
    S0 = torch.randn((B, H, dv, dk), generator=g) * 0.1 if state else None
    out = dict(q=q.to(dtype), kw=kw.to(dtype), v=v.to(dtype), w=w.float().contiguous(),
               kappa=kap.float().contiguous(), a=a.float().contiguous(), S0=S0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def draw_workload(w: Workload, device="cpu"):
    return draw(w.gen, w.B, w.H, w.T, w.dk, w.dv, w.seed, w.torch_dtype, w.s0_std, device)


def draw_decode_step(w: Workload, step: int, device, generator=None):
    """Inputs of decode step ``step`` for workload ``w`` (fresh per step), drawn
    on ``device`` with a generator seeded from (seed, step).

    Returns q, k [N,H,dk]; v [N,H,dv] in the workload dtype; alpha, beta [N,H].
    """
    g = generator if generator is not None else torch.Generator(device)
    g.manual_seed(int(w.seed) * 1000003 + int(step))
    N, H, dk, dv = w.B, w.H, w.dk, w.dv
    q = _silu_l2(torch.randn((N, H, dk), generator=g, device=device))
    k = _silu_l2(torch.randn((N, H, dk), generator=g, device=device))
    v = torch.randn((N, H, dv), generator=g, device=device)
    beta = torch.sigmoid(torch.randn((N, H), generator=g, device=device))
    alpha = torch.sigmoid(3.0 + torch.randn((N, H), generator=g, device=device))
    dt = w.torch_dtype
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), alpha=alpha.float(), beta=beta.float())


def draw_decode_state(w: Workload, device, generator=None):
    """Initial decode state S ~ N(0, s0_std^2), [N,H,dv,dk] fp32, on ``device``."""
    g = generator if generator is not None else torch.Generator(device)
    g.manual_seed(int(w.seed) * 1000003 - 1)
    return torch.randn((w.B, w.H, w.dv, w.dk), generator=g, device=device) * w.s0_std

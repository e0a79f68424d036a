"""lr_fwd_chunked_noalloc: the chunked forward for callers that cannot
allocate device memory (a host framework that owns all device memory and
gives its plug-ins no allocator, or a path where cudaMalloc must not run).

It takes its scratch from a fixed array inside the library instead of a
caller workspace, so it must give the same results as lr_fwd_chunked with a
workspace.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process (the first call sets up the static scratch on the device).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 bar of the parity tests


def _rel(a, b):
    a = a.detach().float().cpu().double().numpy()
    b = b.detach().float().cpu().double().numpy()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gated_delta_rule_fwd_gb300.build import build
    build()
    return torch.device("cuda:0")


def test_noalloc_matches_workspace_entry_point_twice(dev):
    """Two calls in a row (different modes, sizes and inputs, the second
    reusing the scratch the first left behind) give the same bits as
    lr_fwd_chunked with a workspace: the same kernels run on the same inputs,
    and the kernels are deterministic.  The diagonal gate also keeps its
    transformed q and k in the scratch, after the records."""
    cases = [(lr.GATED_DELTA, "gdn", 2, 4, 1000, 0.1, 11), (lr.DECAY, "mamba2", 2, 3, 333, 0.0, 12),
             (lr.DIAG_DECAY, "gla", 1, 3, 700, 0.1, 13)]
    for mode, gen, B, H, T, s0, seed in cases:
        x = workloads.draw(gen, B, H, T, 128, 128, seed=seed, dtype=torch.bfloat16, s0_std=s0)
        d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
        need = lr.workspace_size(B, H, T, 128, 128, torch.bfloat16, mode)
        assert need <= lr.STATIC_WORKSPACE_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        o_ref, s_ref = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                         mode=mode, workspace=ws)
        o_na, s_na = lr.lr_fwd_chunked_noalloc(d["q"], d["k"], d["v"], d["alpha"], d["beta"],
                                               d["S0"], mode=mode)
        torch.cuda.synchronize()
        assert torch.equal(o_na, o_ref) and torch.equal(s_na, s_ref)
        assert _rel(o_na, o_ref) <= TOL   # (implied by the above; the parity tests' bar)
    assert lr.device_status() == 0


def test_noalloc_allocates_no_device_memory(dev):
    """With o and S_T given, a call takes no device memory: neither the
    caching allocator's count nor the device's free memory changes."""
    B, H, T = 2, 4, 1000
    x = workloads.draw("gdn", B, H, T, 128, 128, seed=14, dtype=torch.bfloat16, s0_std=0.1)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((B, H, T, 128), dtype=torch.bfloat16, device=dev)
    st = torch.empty((B, H, 128, 128), dtype=torch.float32, device=dev)

    def call():
        lr.lr_fwd_chunked_noalloc(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                  mode=lr.GATED_DELTA, o=o, S_T=st)
    call()                      # first call: the scratch address is looked up
    torch.cuda.synchronize()
    used0 = torch.cuda.memory_allocated(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(dev) == used0
    assert torch.cuda.mem_get_info(dev)[0] == free0


def test_noalloc_rejects_problems_beyond_static_scratch(dev):
    w = workloads.WORKLOADS["gdn_prefill_bf16"]   # 32 heads x 256 blocks: ~270 MB of scratch
    assert lr.workspace_size(w.B, w.H, w.T, w.dk, w.dv, torch.bfloat16) > lr.STATIC_WORKSPACE_BYTES
    q = torch.zeros((w.B, w.H, w.T, w.dk), dtype=torch.bfloat16, device=dev)
    a = torch.ones((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    o = torch.full((w.B, w.H, w.T, w.dv), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(lr.LrError) as e:
        lr.lr_fwd_chunked_noalloc(q, q.clone(), q.clone(), a, a.clone(), None, o=o)
    assert e.value.status == 11
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())   # nothing was launched

"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait in the tensor-core kernels gives up after a bounded number
of polls; the kernel then waits for its own copies and products in flight,
frees its tensor memory, sets the library's error word and returns, and
lr_device_status() reports LR_ERR_TIMEOUT.  The test hook
lr_debug_inject_scan_timeout makes that happen on purpose in the chunked
forward's sequential pass: a short poll limit, and stage 1's tiles never
loaded, so every role's wait for stage 1 runs out.  Nothing faults and
nothing waits without a limit; the context stays usable, which the normal
call afterwards checks against the oracle.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_fwd_gb300 as lr
import oracle
import workloads

pytestmark = pytest.mark.gpu

LR_ERR_TIMEOUT = 9


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gated_delta_rule_fwd_gb300.build import build
    build()
    yield torch.device("cuda:0")
    lr.debug_inject_scan_timeout(False)


def _rel(a, ref):
    a = a.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(a - ref)) / max(np.max(np.abs(ref)), 1e-30))


def test_scan_wait_runs_out_and_reports_timeout(dev):
    x = workloads.draw("gdn", 1, 1, 128, 128, 128, seed=21, dtype=torch.bfloat16, s0_std=0.1)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    assert lr.device_status() == 0          # nothing pending from earlier tests
    lr.debug_inject_scan_timeout(True)
    try:
        lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                          mode=lr.GATED_DELTA)
        torch.cuda.synchronize()            # the call returns: every wait was bounded
        assert lr.device_status() == LR_ERR_TIMEOUT
        assert lr.device_status() == 0      # reading the word clears it
    finally:
        lr.debug_inject_scan_timeout(False)
    # the context is intact: a normal call on the same inputs matches the oracle
    o, st = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                              mode=lr.GATED_DELTA)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrent(lr.GATED_DELTA, x["q"], x["k"], x["v"], x["alpha"],
                                    x["beta"], x["S0"])
    assert _rel(o, o_ref) <= 2e-2 and _rel(st, s_ref) <= 2e-2
    assert lr.device_status() == 0


def test_scan_timeout_hook_without_delta(dev):
    """The same exit path in the instantiation without the delta term (its
    roles hand off differently: the state warps release the late group)."""
    x = workloads.draw("mamba2", 1, 2, 200, 128, 128, seed=22, dtype=torch.bfloat16)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    lr.debug_inject_scan_timeout(True)
    try:
        lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], None, None, mode=lr.DECAY)
        torch.cuda.synchronize()
        assert lr.device_status() == LR_ERR_TIMEOUT
    finally:
        lr.debug_inject_scan_timeout(False)
    o, st = lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], None, None, mode=lr.DECAY)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrent(lr.DECAY, x["q"], x["k"], x["v"], x["alpha"], x["beta"], None)
    assert _rel(o, o_ref) <= 2e-2 and _rel(st, s_ref) <= 2e-2
    assert lr.device_status() == 0


def test_scan_timeout_hook_with_folded_norm(dev):
    """The same exit path in the scan that applies the output RMSNorm, where the
    dv / NV CTAs of a head run as one cluster and exchange the rows' partial
    sums through each other's shared memory: the CTAs that gave up still meet
    at the cluster barrier before any of them leaves."""
    from oracle import prologue as P
    flags = lr.FUSE_QK_SILU_L2 | lr.FUSE_BETA_SIGMOID | lr.FUSE_ALPHA_SIGMOID | lr.FUSE_O_RMSNORM
    # d_v = 64: two 32-channel CTAs per head, the scan applies the norm
    x = workloads.draw_pre("gdn", 1, 2, 200, 128, 64, seed=23, dtype=torch.bfloat16, s0_std=0.3)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}

    def call():
        return lr.lr_fwd_chunked_fused(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"],
                                       mode=lr.GATED_DELTA, flags=flags,
                                       alpha_scale=d["alpha_scale"], norm_weight=d["norm_weight"])

    lr.debug_inject_scan_timeout(True)
    try:
        call()
        torch.cuda.synchronize()
        assert lr.device_status() == LR_ERR_TIMEOUT
    finally:
        lr.debug_inject_scan_timeout(False)
    o, st = call()
    torch.cuda.synchronize()
    f64 = lambda t: t.double().numpy()
    o_ref, s_ref = P.fused(lr.GATED_DELTA, flags, f64(x["q"]), f64(x["k"]), f64(x["v"]),
                           f64(x["alpha"]), f64(x["beta"]), f64(x["S0"]),
                           alpha_scale=f64(x["alpha_scale"]), norm_weight=f64(x["norm_weight"]))
    assert _rel(o, o_ref) <= 2e-2 and _rel(st, s_ref) <= 2e-2
    assert lr.device_status() == 0

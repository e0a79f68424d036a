"""Gated delta rule forward on GB300 (sm_103a): Python binding of liblr.

The library's C ABI is declared in ``include/lr.h``; this module only
marshals arguments (tensor pointers, sizes, the current CUDA stream) into it.
Every step of the computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  There is no fallback: if ``liblr.so`` is
missing or cannot be loaded, every call raises.

    lr_fwd_chunked(q, k, v, alpha, beta, S0, mode=...) -> (o, S_T)
        chunkwise prefill over whole sequences (q, k: [B,H,T,dk], v: [B,H,T,dv])
    lr_step(q, k, v, alpha, beta, S, mode=...) -> o
        one decode step for N sequences, S: [N,H,dv,dk] updated in place
    lr_fwd_chunked_mlstm / lr_step_mlstm(q, k, v, fgate, igate, ...)
        the mLSTM memory (exponential write gate, normaliser, stabiliser)
    lr_fwd_chunked_gen_delta / lr_step_gen_delta(q, kw, v, w, kappa, a, ...)
        the generalised delta rule of RWKV-7 (per-channel decay plus a rank-one
        correction)
    lr_fwd_chunked_fused / lr_step_fused(..., flags=..., ...)
        the same with the maps around the recurrence (SiLU + L2 of q and k,
        sigmoid beta, sigmoid or softplus alpha, output RMSNorm) applied inside
        the kernels; flags are the FUSE_* constants
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

LINEAR, DECAY, DELTA, GATED_DELTA, DIAG_DECAY = 0, 1, 2, 3, 4
MODES = {"linear": LINEAR, "decay": DECAY, "delta": DELTA, "gated_delta": GATED_DELTA,
         "diag_decay": DIAG_DECAY}
F32, BF16 = 0, 1
SYMBOLS = ("lr_fwd_chunked", "lr_fwd_chunked_workspace_size", "lr_fwd_chunked_noalloc", "lr_step",
           "lr_fwd_chunked_fused", "lr_fwd_chunked_fused_workspace_size", "lr_step_fused",
           "lr_fwd_chunked_mlstm", "lr_fwd_chunked_mlstm_workspace_size", "lr_step_mlstm",
           "lr_fwd_chunked_gen_delta", "lr_fwd_chunked_gen_delta_workspace_size",
           "lr_step_gen_delta",
           "lr_device_status", "lr_debug_inject_scan_timeout", "lr_status_string",
           "lr_abi_version")
# lr_fuse flags (include/lr.h)
FUSE_QK_SILU_L2 = 0x1
FUSE_BETA_SIGMOID = 0x2
FUSE_ALPHA_SIGMOID = 0x4
FUSE_ALPHA_SOFTPLUS = 0x8
FUSE_O_RMSNORM = 0x10
FUSE_ALPHA_SIGMOID_POW = 0x20
STATIC_WORKSPACE_BYTES = 64 << 20   # LR_STATIC_WORKSPACE_BYTES
STATUS = {0: "LR_OK", 1: "LR_ERR_NULL", 2: "LR_ERR_SHAPE", 3: "LR_ERR_DTYPE", 4: "LR_ERR_ALIGN",
          5: "LR_ERR_MODE", 6: "LR_ERR_UNSUPPORTED", 7: "LR_ERR_CUDA", 8: "LR_ERR_ALIAS",
          9: "LR_ERR_TIMEOUT", 10: "LR_ERR_WORKSPACE", 11: "LR_ERR_TOO_LARGE", 12: "LR_ERR_FUSE"}
_USES_ALPHA = {LINEAR: False, DECAY: True, DELTA: False, GATED_DELTA: True, DIAG_DECAY: True}
_USES_BETA = {LINEAR: False, DECAY: False, DELTA: True, GATED_DELTA: True, DIAG_DECAY: False}


def _alpha_shape(mode, lead, dk):
    """alpha has one value per token, or one per key channel for DIAG_DECAY."""
    return tuple(lead) + ((dk,) if mode == DIAG_DECAY else ())


class Fuse(ctypes.Structure):
    """lr_fuse (include/lr.h)."""
    _fields_ = [("flags", ctypes.c_uint), ("alpha_scale", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float)]


class LrError(RuntimeError):
    """A non-OK lr_status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded liblr.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "or `python -m gated_delta_rule_fwd_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, fp, i = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
        L.lr_fwd_chunked.restype = i
        L.lr_fwd_chunked.argtypes = ([vp, vp, vp, fp, fp, fp, vp, fp] + [i] * 6 +
                                     [i, i, vp, ctypes.c_size_t, vp])
        L.lr_fwd_chunked_noalloc.restype = i
        L.lr_fwd_chunked_noalloc.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp] + [i] * 6 + [i, i, vp]
        L.lr_fwd_chunked_workspace_size.restype = ctypes.c_size_t
        L.lr_fwd_chunked_workspace_size.argtypes = [i] * 8
        L.lr_step.restype = i
        L.lr_step.argtypes = [vp, vp, vp, fp, fp, fp, vp] + [i] * 4 + [i, i, vp]
        fz = ctypes.POINTER(Fuse)
        L.lr_fwd_chunked_fused.restype = i
        L.lr_fwd_chunked_fused.argtypes = ([vp, vp, vp, fp, fp, fp, vp, fp] + [i] * 6 +
                                           [i, i, fz, vp, ctypes.c_size_t, vp])
        L.lr_fwd_chunked_fused_workspace_size.restype = ctypes.c_size_t
        L.lr_fwd_chunked_fused_workspace_size.argtypes = [i] * 8 + [ctypes.c_uint]
        L.lr_step_fused.restype = i
        L.lr_step_fused.argtypes = [vp, vp, vp, fp, fp, fp, vp] + [i] * 4 + [i, i, fz, vp]
        L.lr_fwd_chunked_mlstm.restype = i
        L.lr_fwd_chunked_mlstm.argtypes = ([vp] * 12 + [i] * 6 + [i, vp, ctypes.c_size_t, vp])
        L.lr_fwd_chunked_mlstm_workspace_size.restype = ctypes.c_size_t
        L.lr_fwd_chunked_mlstm_workspace_size.argtypes = [i] * 7
        L.lr_step_mlstm.restype = i
        L.lr_step_mlstm.argtypes = [vp] * 9 + [i] * 4 + [i, vp]
        L.lr_fwd_chunked_gen_delta.restype = i
        L.lr_fwd_chunked_gen_delta.argtypes = [vp] * 9 + [i] * 6 + [i, vp, ctypes.c_size_t, vp]
        L.lr_fwd_chunked_gen_delta_workspace_size.restype = ctypes.c_size_t
        L.lr_fwd_chunked_gen_delta_workspace_size.argtypes = [i] * 7
        L.lr_step_gen_delta.restype = i
        L.lr_step_gen_delta.argtypes = [vp] * 8 + [i] * 4 + [i, vp]
        L.lr_status_string.restype = ctypes.c_char_p
        L.lr_status_string.argtypes = [i]
        L.lr_abi_version.restype = i
        L.lr_abi_version.argtypes = []
        L.lr_device_status.restype = i
        L.lr_device_status.argtypes = []
        L.lr_debug_inject_scan_timeout.restype = i
        L.lr_debug_inject_scan_timeout.argtypes = [i]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().lr_status_string(int(status)).decode()


def device_status() -> int:
    """lr_device_status(): synchronises the current device and returns (and
    clears) the library's bounded-wait error word as a status code."""
    return int(lib().lr_device_status())


def debug_inject_scan_timeout(on: bool) -> None:
    """lr_debug_inject_scan_timeout: the failure-detection test hook.  While
    on, the chunked forward's bf16 sequential pass gives up a bounded wait on
    purpose (short poll limit, stage 1 never loaded) and takes its exit path;
    ``device_status()`` then reports LR_ERR_TIMEOUT.  Synchronises the device."""
    st = lib().lr_debug_inject_scan_timeout(1 if on else 0)
    if st != 0:
        raise LrError(st, "lr_debug_inject_scan_timeout")


def _require_cuda(device):
    if device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"q, k, v must be float32 or bfloat16, got {t.dtype}")


def _check(t, name, shape, dtype, device):
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(B, H, T, dk, dv, dtype, mode=GATED_DELTA, chunk=64) -> int:
    """lr_fwd_chunked_workspace_size for these sizes (dtype: torch dtype)."""
    import torch
    dt = F32 if dtype == torch.float32 else BF16
    return int(lib().lr_fwd_chunked_workspace_size(B, H, T, dk, dv, int(chunk), dt,
                                                   int(MODES.get(mode, mode))))


def lr_fwd_chunked(q, k, v, alpha=None, beta=None, S0=None, *, mode=GATED_DELTA, chunk=64,
                   o=None, S_T=None, workspace=None, stream=None):
    """Chunkwise forward (see ``lr_fwd_chunked`` in include/lr.h).

    q, k: [B,H,T,dk]; v: [B,H,T,dv] (float32 or bfloat16, same dtype);
    alpha, beta: [B,H,T] float32 where the mode uses them (alpha [B,H,T,dk]
    for DIAG_DECAY); S0: [B,H,dv,dk]
    float32 or None.  ``o`` and ``S_T`` may be given to write into (``S_T``
    may be ``S0``).  ``workspace`` is a uint8 CUDA tensor of at least
    ``workspace_size(...)`` bytes; when None one is allocated through the
    PyTorch caching allocator.  Returns (o, S_T).
    """
    import torch
    mode = MODES.get(mode, mode)
    dev = q.device
    _require_cuda(dev)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (B, H, T, dk), q.dtype, dev)
    _check(k, "k", (B, H, T, dk), q.dtype, dev)
    _check(v, "v", (B, H, T, dv), q.dtype, dev)
    if _USES_ALPHA[mode]:
        _check(alpha, "alpha", _alpha_shape(mode, (B, H, T), dk), torch.float32, dev)
    else:
        alpha = None
    if _USES_BETA[mode]:
        _check(beta, "beta", (B, H, T), torch.float32, dev)
    else:
        beta = None
    if S0 is not None:
        _check(S0, "S0", (B, H, dv, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", (B, H, T, dv), q.dtype, dev)
    if S_T is None:
        S_T = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    else:
        _check(S_T, "S_T", (B, H, dv, dk), torch.float32, dev)
    need = int(lib().lr_fwd_chunked_workspace_size(B, H, T, dk, dv, int(chunk), dt, int(mode)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().lr_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                              _ptr(o), _ptr(S_T), B, H, T, dk, dv, int(chunk), dt, int(mode),
                              _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_fwd_chunked")
    return o, S_T


def lr_fwd_chunked_noalloc(q, k, v, alpha=None, beta=None, S0=None, *, mode=GATED_DELTA,
                           chunk=64, o=None, S_T=None, stream=None):
    """Chunkwise forward through ``lr_fwd_chunked_noalloc`` (include/lr.h):
    the same result as :func:`lr_fwd_chunked`, with the scratch taken from
    the library's fixed static device array instead of a workspace, for
    callers that cannot allocate device memory.  Raises LrError with
    LR_ERR_TOO_LARGE when the problem needs more than STATIC_WORKSPACE_BYTES
    of scratch.  Outputs ``o`` and ``S_T`` are allocated here only when not
    given.  Returns (o, S_T).
    """
    import torch
    mode = MODES.get(mode, mode)
    dev = q.device
    _require_cuda(dev)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (B, H, T, dk), q.dtype, dev)
    _check(k, "k", (B, H, T, dk), q.dtype, dev)
    _check(v, "v", (B, H, T, dv), q.dtype, dev)
    alpha = alpha if _USES_ALPHA[mode] else None
    beta = beta if _USES_BETA[mode] else None
    if alpha is not None:
        _check(alpha, "alpha", _alpha_shape(mode, (B, H, T), dk), torch.float32, dev)
    if beta is not None:
        _check(beta, "beta", (B, H, T), torch.float32, dev)
    if S0 is not None:
        _check(S0, "S0", (B, H, dv, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", (B, H, T, dv), q.dtype, dev)
    if S_T is None:
        S_T = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    else:
        _check(S_T, "S_T", (B, H, dv, dk), torch.float32, dev)
    st = lib().lr_fwd_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                      _ptr(S0), _ptr(o), _ptr(S_T), B, H, T, dk, dv, int(chunk),
                                      dt, int(mode), _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_fwd_chunked_noalloc")
    return o, S_T


def lr_step(q, k, v, alpha, beta, S, *, mode=GATED_DELTA, o=None, stream=None):
    """One decode step (see ``lr_step`` in include/lr.h); S is updated in place.

    q, k: [N,H,dk]; v: [N,H,dv]; alpha, beta: [N,H] float32 where the mode
    uses them (alpha [N,H,dk] for DIAG_DECAY); S: [N,H,dv,dk] float32.  Returns o: [N,H,dv].
    """
    import torch
    mode = MODES.get(mode, mode)
    dev = q.device
    _require_cuda(dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (N, H, dk), q.dtype, dev)
    _check(k, "k", (N, H, dk), q.dtype, dev)
    _check(v, "v", (N, H, dv), q.dtype, dev)
    if _USES_ALPHA[mode]:
        _check(alpha, "alpha", _alpha_shape(mode, (N, H), dk), torch.float32, dev)
    else:
        alpha = None
    if _USES_BETA[mode]:
        _check(beta, "beta", (N, H), torch.float32, dev)
    else:
        beta = None
    _check(S, "S", (N, H, dv, dk), torch.float32, dev)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", (N, H, dv), q.dtype, dev)
    st = lib().lr_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S), _ptr(o),
                       N, H, dk, dv, dt, int(mode), _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_step")
    return o


def _fuse(flags, alpha_scale, norm_weight, norm_eps, H, dv, dev):
    import torch
    if alpha_scale is not None:
        _check(alpha_scale, "alpha_scale", (H,), torch.float32, dev)
    if norm_weight is not None:
        _check(norm_weight, "norm_weight", (dv,), torch.float32, dev)
    return Fuse(int(flags), None if alpha_scale is None else alpha_scale.data_ptr(),
                None if norm_weight is None else norm_weight.data_ptr(), float(norm_eps))


def fused_workspace_size(B, H, T, dk, dv, dtype, mode=GATED_DELTA, flags=0, chunk=64) -> int:
    """lr_fwd_chunked_fused_workspace_size for these sizes and flags."""
    import torch
    dt = F32 if dtype == torch.float32 else BF16
    return int(lib().lr_fwd_chunked_fused_workspace_size(B, H, T, dk, dv, int(chunk), dt,
                                                         int(MODES.get(mode, mode)), int(flags)))


def lr_fwd_chunked_fused(q, k, v, alpha=None, beta=None, S0=None, *, mode=GATED_DELTA, flags=0,
                         alpha_scale=None, norm_weight=None, norm_eps=1e-6, chunk=64, o=None,
                         S_T=None, workspace=None, stream=None):
    """Chunkwise forward with the maps around the recurrence
    (``lr_fwd_chunked_fused`` in include/lr.h).

    As :func:`lr_fwd_chunked`, with q, k, alpha and beta holding the
    pre-activation values of the maps that ``flags`` selects (FUSE_*);
    ``alpha_scale``: [H] float32 (the c_h of FUSE_ALPHA_SOFTPLUS);
    ``norm_weight``: [dv] float32 or None (FUSE_O_RMSNORM).  Returns (o, S_T).
    """
    import torch
    mode = MODES.get(mode, mode)
    dev = q.device
    _require_cuda(dev)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (B, H, T, dk), q.dtype, dev)
    _check(k, "k", (B, H, T, dk), q.dtype, dev)
    _check(v, "v", (B, H, T, dv), q.dtype, dev)
    alpha = alpha if _USES_ALPHA[mode] else None
    beta = beta if _USES_BETA[mode] else None
    if alpha is not None:
        _check(alpha, "alpha", _alpha_shape(mode, (B, H, T), dk), torch.float32, dev)
    if beta is not None:
        _check(beta, "beta", (B, H, T), torch.float32, dev)
    if S0 is not None:
        _check(S0, "S0", (B, H, dv, dk), torch.float32, dev)
    fz = _fuse(flags, alpha_scale, norm_weight, norm_eps, H, dv, dev)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", (B, H, T, dv), q.dtype, dev)
    if S_T is None:
        S_T = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    else:
        _check(S_T, "S_T", (B, H, dv, dk), torch.float32, dev)
    need = int(lib().lr_fwd_chunked_fused_workspace_size(B, H, T, dk, dv, int(chunk), dt,
                                                         int(mode), int(flags)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().lr_fwd_chunked_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                    _ptr(S0), _ptr(o), _ptr(S_T), B, H, T, dk, dv, int(chunk),
                                    dt, int(mode), ctypes.byref(fz), _ptr(workspace), ws_bytes,
                                    _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_fwd_chunked_fused")
    return o, S_T


def lr_step_fused(q, k, v, alpha, beta, S, *, mode=GATED_DELTA, flags=0, alpha_scale=None,
                  norm_weight=None, norm_eps=1e-6, o=None, stream=None):
    """One decode step with the maps around the recurrence
    (``lr_step_fused`` in include/lr.h); S is updated in place.  Arguments as
    :func:`lr_step` plus those of :func:`lr_fwd_chunked_fused`.  Returns o."""
    import torch
    mode = MODES.get(mode, mode)
    dev = q.device
    _require_cuda(dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (N, H, dk), q.dtype, dev)
    _check(k, "k", (N, H, dk), q.dtype, dev)
    _check(v, "v", (N, H, dv), q.dtype, dev)
    alpha = alpha if _USES_ALPHA[mode] else None
    beta = beta if _USES_BETA[mode] else None
    if alpha is not None:
        _check(alpha, "alpha", _alpha_shape(mode, (N, H), dk), torch.float32, dev)
    if beta is not None:
        _check(beta, "beta", (N, H), torch.float32, dev)
    _check(S, "S", (N, H, dv, dk), torch.float32, dev)
    fz = _fuse(flags, alpha_scale, norm_weight, norm_eps, H, dv, dev)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", (N, H, dv), q.dtype, dev)
    st = lib().lr_step_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S), _ptr(o),
                             N, H, dk, dv, dt, int(mode), ctypes.byref(fz),
                             _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_step_fused")
    return o


def mlstm_workspace_size(B, H, T, dk, dv, dtype, chunk=64) -> int:
    """lr_fwd_chunked_mlstm_workspace_size for these sizes."""
    import torch
    dt = F32 if dtype == torch.float32 else BF16
    return int(lib().lr_fwd_chunked_mlstm_workspace_size(B, H, T, dk, dv, int(chunk), dt))


def lr_fwd_chunked_mlstm(q, k, v, fgate, igate, C0=None, n0=None, m0=None, *, chunk=64, h=None,
                         C_T=None, n_T=None, m_T=None, workspace=None, stream=None):
    """mLSTM memory over whole sequences (``lr_fwd_chunked_mlstm`` in include/lr.h).

    q, k: [B,H,T,dk]; v: [B,H,T,dv] (float32 or bfloat16); fgate, igate:
    [B,H,T] float32 (forget gate in (0,1], input-gate pre-activation); the
    stabilised state (C0 [B,H,dv,dk], n0 [B,H,dk], m0 [B,H]) float32 or all
    None for the empty memory.  Returns (h, C_T, n_T, m_T).
    """
    import torch
    dev = q.device
    _require_cuda(dev)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q", (B, H, T, dk), q.dtype, dev)
    _check(k, "k", (B, H, T, dk), q.dtype, dev)
    _check(v, "v", (B, H, T, dv), q.dtype, dev)
    _check(fgate, "fgate", (B, H, T), torch.float32, dev)
    _check(igate, "igate", (B, H, T), torch.float32, dev)
    if C0 is not None:
        _check(C0, "C0", (B, H, dv, dk), torch.float32, dev)
        _check(n0, "n0", (B, H, dk), torch.float32, dev)
        _check(m0, "m0", (B, H), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    h = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev) if h is None else h
    C_T = torch.empty((B, H, dv, dk), **f32) if C_T is None else C_T
    n_T = torch.empty((B, H, dk), **f32) if n_T is None else n_T
    m_T = torch.empty((B, H), **f32) if m_T is None else m_T
    need = int(lib().lr_fwd_chunked_mlstm_workspace_size(B, H, T, dk, dv, int(chunk), dt))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().lr_fwd_chunked_mlstm(_ptr(q), _ptr(k), _ptr(v), _ptr(fgate), _ptr(igate), _ptr(C0),
                                    _ptr(n0), _ptr(m0), _ptr(h), _ptr(C_T), _ptr(n_T), _ptr(m_T),
                                    B, H, T, dk, dv, int(chunk), dt, _ptr(workspace), ws_bytes,
                                    _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_fwd_chunked_mlstm")
    return h, C_T, n_T, m_T


def lr_step_mlstm(q, k, v, fgate, igate, C, n, m, *, h=None, stream=None):
    """One mLSTM step (``lr_step_mlstm``); (C, n, m) updated in place.
    q, k: [N,H,dk]; v: [N,H,dv]; fgate, igate: [N,H]; C [N,H,dv,dk], n [N,H,dk],
    m [N,H] float32.  Returns h: [N,H,dv]."""
    import torch
    dev = q.device
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(k, "k", (N, H, dk), q.dtype, dev)
    _check(v, "v", (N, H, dv), q.dtype, dev)
    _check(fgate, "fgate", (N, H), torch.float32, dev)
    _check(igate, "igate", (N, H), torch.float32, dev)
    _check(C, "C", (N, H, dv, dk), torch.float32, dev)
    _check(n, "n", (N, H, dk), torch.float32, dev)
    _check(m, "m", (N, H), torch.float32, dev)
    h = torch.empty((N, H, dv), dtype=q.dtype, device=dev) if h is None else h
    st = lib().lr_step_mlstm(_ptr(q), _ptr(k), _ptr(v), _ptr(fgate), _ptr(igate), _ptr(C), _ptr(n),
                             _ptr(m), _ptr(h), N, H, dk, dv, dt, _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_step_mlstm")
    return h


def gen_delta_workspace_size(B, H, T, dk, dv, dtype, chunk=64) -> int:
    """lr_fwd_chunked_gen_delta_workspace_size for these sizes."""
    import torch
    dt = F32 if dtype == torch.float32 else BF16
    return int(lib().lr_fwd_chunked_gen_delta_workspace_size(B, H, T, dk, dv, int(chunk), dt))


def lr_fwd_chunked_gen_delta(q, kw, v, w, kappa, a, S0=None, *, chunk=64, o=None, S_T=None,
                             workspace=None, stream=None):
    """Generalised delta rule over whole sequences (``lr_fwd_chunked_gen_delta``).
    q, kw: [B,H,T,dk]; v: [B,H,T,dv] (float32 or bfloat16); w, kappa, a:
    [B,H,T,dk] float32; S0: [B,H,dv,dk] float32 or None.  The bfloat16 path
    needs a workspace (allocated here when none is given).  Returns (o, S_T)."""
    import torch
    dev = q.device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(kw, "kw", (B, H, T, dk), q.dtype, dev)
    _check(v, "v", (B, H, T, dv), q.dtype, dev)
    for t, nm in ((w, "w"), (kappa, "kappa"), (a, "a")):
        _check(t, nm, (B, H, T, dk), torch.float32, dev)
    if S0 is not None:
        _check(S0, "S0", (B, H, dv, dk), torch.float32, dev)
    o = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev) if o is None else o
    S_T = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev) if S_T is None else S_T
    need = int(lib().lr_fwd_chunked_gen_delta_workspace_size(B, H, T, dk, dv, int(chunk), dt))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().lr_fwd_chunked_gen_delta(_ptr(q), _ptr(kw), _ptr(v), _ptr(w), _ptr(kappa), _ptr(a),
                                        _ptr(S0), _ptr(o), _ptr(S_T), B, H, T, dk, dv, int(chunk),
                                        dt, _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_fwd_chunked_gen_delta")
    return o, S_T


def lr_step_gen_delta(q, kw, v, w, kappa, a, S, *, o=None, stream=None):
    """One generalised-delta step (``lr_step_gen_delta``); S updated in place."""
    import torch
    dev = q.device
    N, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(kw, "kw", (N, H, dk), q.dtype, dev)
    _check(v, "v", (N, H, dv), q.dtype, dev)
    for t, nm in ((w, "w"), (kappa, "kappa"), (a, "a")):
        _check(t, nm, (N, H, dk), torch.float32, dev)
    _check(S, "S", (N, H, dv, dk), torch.float32, dev)
    o = torch.empty((N, H, dv), dtype=q.dtype, device=dev) if o is None else o
    st = lib().lr_step_gen_delta(_ptr(q), _ptr(kw), _ptr(v), _ptr(w), _ptr(kappa), _ptr(a), _ptr(S),
                                 _ptr(o), N, H, dk, dv, dt, _stream_handle(stream, dev))
    if st != 0:
        raise LrError(st, "lr_step_gen_delta")
    return o

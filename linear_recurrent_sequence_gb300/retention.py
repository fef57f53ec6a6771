"""Python binding of the retention C ABI (``include/retention.h``).

Argument marshalling only: every step of retention runs in the CUDA kernels
of ``libretention.so``.  PyTorch supplies device memory and the stream.  If
the library has not been built this module raises at import; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

F32, BF16 = 0, 1
NORM_SCALE, NORM_DROW, NORM_RSUM = 1, 2, 4
NORM_ALL = NORM_SCALE | NORM_DROW | NORM_RSUM
STATUS = {0: "RET_OK", 1: "RET_EINVAL", 2: "RET_EUNSUPPORTED", 3: "RET_EWORKSPACE",
          4: "RET_ECUDA", 5: "RET_ETIMEOUT"}
MAX_HEADS = 256

_I64x3 = ctypes.c_int64 * 3


class RetDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("chunk", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("gamma", ctypes.POINTER(ctypes.c_double)),
                ("theta_base", ctypes.c_double), ("norm_flags", ctypes.c_int),
                ("gn_eps", ctypes.c_float), ("pos0", ctypes.c_int64),
                ("rotate", ctypes.c_int),
                ("sq", _I64x3), ("sk", _I64x3), ("sv", _I64x3), ("so", _I64x3)]


class MsrDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("d_model", ctypes.c_int),
                ("H", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("chunk", ctypes.c_int), ("gamma", ctypes.POINTER(ctypes.c_double)),
                ("theta_base", ctypes.c_double), ("norm_flags", ctypes.c_int),
                ("gn_eps", ctypes.c_float), ("pos0", ctypes.c_int64)]


class BlockDesc(ctypes.Structure):
    _fields_ = [("msr", MsrDesc), ("d_ffn", ctypes.c_int), ("ln_eps", ctypes.c_float)]


class StackDesc(ctypes.Structure):
    _fields_ = [("block", BlockDesc), ("n_layers", ctypes.c_int)]


LAYER_KEYS = ("ln1_w", "ln1_b", "WQ", "WK", "WV", "WG", "WO", "ln2_w", "ln2_b", "W1", "W2")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_KEYS]


# Every symbol include/retention.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_SIGS = {
    "retention_desc_init": (None, [ctypes.POINTER(RetDesc), ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_double)]),
    "retention_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(RetDesc)]),
    "retention_rotate": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P,
                                        ctypes.POINTER(ctypes.c_int64), ctypes.c_int, _P,
                                        ctypes.c_int, _P, _P]),
    "retention_parallel_fwd": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P, _P,
                                              ctypes.c_size_t, _P]),
    "retention_chunkwise_fwd": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "retention_recurrent_step": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P, _P,
                                                _P, _P, ctypes.c_size_t, _P]),
    "retention_chunkwise_fwd_noalloc": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P,
                                                       _P, _P, _P, _P, _P]),
    "retention_state_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(RetDesc)]),
    "retention_chunkwise_state": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P, _P,
                                                 _P, _P, ctypes.c_size_t, _P]),
    "retention_state_combine": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                               ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_int64), _P, _P, _P]),
    "retention_backward_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(RetDesc)]),
    "retention_chunkwise_bwd": (ctypes.c_int, [ctypes.POINTER(RetDesc), _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "msr_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(MsrDesc)]),
    "retention_gemm_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int,
                                                        ctypes.c_int]),
    "retention_gemm_bf16": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _P, ctypes.c_size_t, _P]),
    "msr_layer_fwd": (ctypes.c_int, [ctypes.POINTER(MsrDesc), _P, _P, _P, _P, _P, _P, _P, _P,
                                     ctypes.c_size_t, _P]),
    "retnet_block_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(BlockDesc)]),
    "retnet_block_fwd": (ctypes.c_int, [ctypes.POINTER(BlockDesc)] + [_P] * 14 +
                         [ctypes.c_size_t, _P]),
    "retnet_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(StackDesc)]),
    "retnet_decode_step": (ctypes.c_int, [ctypes.POINTER(StackDesc), ctypes.POINTER(LayerWeights),
                                          ctypes.POINTER(ctypes.c_void_p),
                                          ctypes.POINTER(ctypes.c_void_p), _P, _P,
                                          ctypes.c_size_t, _P]),
    "retention_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "retention_last_cuda_error": (ctypes.c_int, []),
    "retention_poll_status": (ctypes.c_int, [_P, _P]),
    "retention_kernel_timer_enable": (None, [ctypes.c_int]),
    "retention_set_report_wait_budget": (None, [ctypes.c_uint]),
    "retention_kernel_timer_reset": (None, []),
    "retention_kernel_count": (ctypes.c_int, []),
    "retention_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
    "retention_launch_count": (ctypes.c_longlong, []),
    "retention_tc_probe": (ctypes.c_int, [ctypes.c_int] * 9 + [_P, _P, _P, _P, _P]),
    "retention_tc_probe_scale_d": (ctypes.c_int, [ctypes.c_int, _P, _P, _P, _P, _P]),
    "retention_tc_probe_pair": (ctypes.c_int, [ctypes.c_int, ctypes.c_int] + [_P] * 6),
    "retention_kernel_timer_read": (ctypes.c_int, [ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_double),
                                                   ctypes.POINTER(ctypes.c_longlong),
                                                   ctypes.POINTER(ctypes.c_int)]),
}


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} is missing "
                          "(run __graft_entry__.build() or linear_recurrent_sequence_gb300/build.py)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


lib = _load()


class RetentionError(RuntimeError):
    def __init__(self, status, where):
        msg = lib.retention_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib.retention_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def _check(status, where):
    if status != 0:
        raise RetentionError(status, where)


def _ptr(t):
    """Device address of a tensor for the C ABI.  Only CUDA tensors on the
    current device are accepted: any other address would reach a kernel."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dt}")


def _bhnd_strides(t, name):
    """Element strides (b, h, n) of a [B, H, N, d] tensor with unit feature stride."""
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B,H,N,d], got {tuple(t.shape)}")
    if t.stride(3) != 1 and t.shape[3] > 1:
        raise ValueError(f"{name}: the feature dimension must be contiguous")
    return (t.stride(0), t.stride(1), t.stride(2))


class _Gamma:
    """Keeps a float64 host copy of the decays alive for the call."""

    def __init__(self, gamma, H):
        import numpy as np
        g = np.ascontiguousarray(np.broadcast_to(np.asarray(gamma, dtype=np.float64), (H,)))
        self.arr = g
        self.ptr = g.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def make_desc(q, k, v, o, gamma, *, chunk=64, norm_flags=0, gn_eps=1e-6, pos0=0,
              rotate=True, theta_base=10000.0):
    B, H, N, dk = q.shape
    dv = v.shape[3]
    g = _Gamma(gamma, H)
    d = RetDesc()
    d.B, d.H, d.N, d.d_k, d.d_v, d.chunk = B, H, N, dk, dv, int(chunk)
    d.in_dtype = _dtype_code(q.dtype)
    d.out_dtype = _dtype_code(o.dtype)
    d.gamma = g.ptr
    d.theta_base = float(theta_base)
    d.norm_flags = int(norm_flags)
    d.gn_eps = float(-1.0 if gn_eps is None else gn_eps)
    d.pos0 = int(pos0)
    d.rotate = int(bool(rotate))
    d.sq = _I64x3(*_bhnd_strides(q, "q"))
    d.sk = _I64x3(*_bhnd_strides(k, "k"))
    d.sv = _I64x3(*_bhnd_strides(v, "v"))
    d.so = _I64x3(*_bhnd_strides(o, "o"))
    return d, g


def workspace_size(desc):
    return int(lib.retention_workspace_size(ctypes.byref(desc)))


def new_workspace(nbytes, device):
    # zeroed once: its first bytes hold the device status word
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _prep(q, k, v, out, out_dtype):
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        B, H, N, _ = q.shape
        out = torch.empty((B, H, N, v.shape[3]), dtype=out_dtype or q.dtype, device=q.device)
    return out


def chunkwise_fwd(q, k, v, gamma, *, chunk=64, norm_flags=0, gn_eps=1e-6, pos0=0,
                  rotate=True, theta_base=10000.0, S_in=None, z_in=None, S_out=None,
                  z_out=None, out=None, out_dtype=None, workspace=None, stream=None):
    """Chunkwise retention forward; q,k [B,H,N,d_k], v [B,H,N,d_v] (any strides
    with a contiguous feature dimension).  Returns the output tensor."""
    out = _prep(q, k, v, out, out_dtype)
    d, g = make_desc(q, k, v, out, gamma, chunk=chunk, norm_flags=norm_flags, gn_eps=gn_eps,
                     pos0=pos0, rotate=rotate, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(workspace_size(d), q.device)
    st = lib.retention_chunkwise_fwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(S_in),
                                     _ptr(z_in), _ptr(S_out), _ptr(z_out), _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "retention_chunkwise_fwd")
    return out


def state_workspace_size(desc):
    return int(lib.retention_state_workspace_size(ctypes.byref(desc)))


def chunkwise_state(k, v, gamma, *, pos0=0, rotate=True, theta_base=10000.0, S_in=None,
                    z_in=None, S_out=None, z_out=None, with_z=True, workspace=None,
                    stream=None):
    """The recurrent state after the tokens of k [B,H,N,d_k], v [B,H,N,d_v]
    (no outputs): S = gamma^N S_in + sum_m gamma^(N-1-m) K'_m^T V_m and z
    likewise.  Returns (S_out, z_out); z_out is None when with_z is False."""
    B, H, N, dk = k.shape
    dv = v.shape[3]
    if S_out is None:
        S_out = torch.empty(B, H, dk, dv, dtype=torch.float32, device=k.device)
    if with_z and z_out is None:
        z_out = torch.empty(B, H, dk, dtype=torch.float32, device=k.device)
    d, g = make_desc(k, k, v, v, gamma, pos0=pos0, rotate=rotate, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(state_workspace_size(d), k.device)
    st = lib.retention_chunkwise_state(ctypes.byref(d), _ptr(k), _ptr(v), _ptr(S_in),
                                       _ptr(z_in), _ptr(S_out), _ptr(z_out), _ptr(workspace),
                                       workspace.numel(), _stream(stream))
    _check(st, "retention_chunkwise_state")
    return S_out, (z_out if with_z else None)


def state_combine(parts, tokens, gamma, *, S_out, z_out=None, stream=None):
    """S_out = sum_i gamma_h^(tokens[i]) S_i (z likewise) over parts, a list of
    (S_i, z_i) pairs of fp32 device tensors (None for a zero state)."""
    B, H, dk, dv = S_out.shape
    n = len(parts)
    Sp = (ctypes.c_void_p * max(n, 1))(*[_ptr(S) for S, _ in parts])
    zp = (ctypes.c_void_p * max(n, 1))(*[_ptr(z) for _, z in parts])
    tk = (ctypes.c_int64 * max(n, 1))(*[int(t) for t in tokens])
    g = (ctypes.c_double * H)(*[float(x) for x in gamma])
    st = lib.retention_state_combine(B, H, dk, dv, g, n, Sp, zp, tk, _ptr(S_out), _ptr(z_out),
                                     _stream(stream))
    _check(st, "retention_state_combine")
    return S_out, z_out


def backward_workspace_size(desc):
    return int(lib.retention_backward_workspace_size(ctypes.byref(desc)))


def chunkwise_bwd(q, k, v, dO, gamma, *, norm_flags=0, pos0=0, rotate=True,
                  theta_base=10000.0, S_in=None, dS_out=None, dS_in=None, dq=None, dk=None,
                  dv=None, workspace=None, stream=None):
    """Gradients of retention without GroupNorm (gn_eps < 0) and without the
    third normalisation: returns (dq, dk, dv, dS_in).  dq, dk, dv take the
    layouts and dtype of q, k, v; dS_in (fp32 [B,H,d_k,d_v]) is returned only
    when passed in (it may be dS_out itself)."""
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")

    def like(x, given, name):
        if given is None:
            return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)
        if given.shape != x.shape or given.stride() != x.stride() or given.dtype != x.dtype:
            raise ValueError(f"{name} must have the shape, strides and dtype of its input")
        return given

    dq, dk, dv = like(q, dq, "dq"), like(k, dk, "dk"), like(v, dv, "dv")
    d, g = make_desc(q, k, v, dO, gamma, norm_flags=norm_flags, gn_eps=None, pos0=pos0,
                     rotate=rotate, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(backward_workspace_size(d), q.device)
    st = lib.retention_chunkwise_bwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(S_in),
                                     _ptr(dO), _ptr(dS_out), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(dS_in), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    _check(st, "retention_chunkwise_bwd")
    return dq, dk, dv, dS_in


def chunkwise_fwd_noalloc(q, k, v, gamma, *, chunk=64, norm_flags=0, gn_eps=1e-6, pos0=0,
                          rotate=True, theta_base=10000.0, S_in=None, z_in=None, S_out=None,
                          z_out=None, out=None, out_dtype=None, stream=None):
    """Chunkwise forward whose workspace is the library's own fixed device
    array (for callers that cannot allocate); see retention.h."""
    out = _prep(q, k, v, out, out_dtype)
    d, g = make_desc(q, k, v, out, gamma, chunk=chunk, norm_flags=norm_flags, gn_eps=gn_eps,
                     pos0=pos0, rotate=rotate, theta_base=theta_base)
    st = lib.retention_chunkwise_fwd_noalloc(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(S_in), _ptr(z_in), _ptr(S_out), _ptr(z_out),
                                             _ptr(out), _stream(stream))
    _check(st, "retention_chunkwise_fwd_noalloc")
    return out


def parallel_fwd(q, k, v, gamma, *, norm_flags=0, gn_eps=1e-6, pos0=0, rotate=True,
                 theta_base=10000.0, out=None, out_dtype=None, workspace=None, stream=None):
    out = _prep(q, k, v, out, out_dtype)
    d, g = make_desc(q, k, v, out, gamma, norm_flags=norm_flags, gn_eps=gn_eps, pos0=pos0,
                     rotate=rotate, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(workspace_size(d), q.device)
    st = lib.retention_parallel_fwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "retention_parallel_fwd")
    return out


def recurrent_step(q, k, v, S, gamma, *, z=None, pos, norm_flags=0, gn_eps=1e-6,
                   rotate=True, theta_base=10000.0, out=None, out_dtype=None,
                   workspace=None, stream=None):
    """One decode step at absolute position ``pos``.  q,k [B,H,d_k], v [B,H,d_v]
    (or with a length-1 token axis); S fp32 [B,H,d_k,d_v] updated in place."""
    q4 = q if q.dim() == 4 else q.unsqueeze(2)
    k4 = k if k.dim() == 4 else k.unsqueeze(2)
    v4 = v if v.dim() == 4 else v.unsqueeze(2)
    out = _prep(q4, k4, v4, out if out is None or out.dim() == 4 else out.unsqueeze(2), out_dtype)
    d, g = make_desc(q4, k4, v4, out, gamma, norm_flags=norm_flags, gn_eps=gn_eps, pos0=pos,
                     rotate=rotate, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(256, q.device)
    st = lib.retention_recurrent_step(ctypes.byref(d), _ptr(q4), _ptr(k4), _ptr(v4), _ptr(S),
                                      _ptr(z), _ptr(out), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    _check(st, "retention_recurrent_step")
    return out


def rotate(x, *, pos0=0, theta_base=10000.0, scale=None, out_dtype=None, stream=None):
    """Theta applied to x [B,H,N,d]; returns a contiguous tensor."""
    B, H, N, dd = x.shape
    out = torch.empty((B, H, N, dd), dtype=out_dtype or x.dtype, device=x.device)
    d, g = make_desc(x, x, x[..., :2], out[..., :2], [1.0] * H, pos0=pos0,
                     theta_base=theta_base)
    sx = _I64x3(*_bhnd_strides(x, "x"))
    st = lib.retention_rotate(ctypes.byref(d), _ptr(x), sx, dd, _ptr(out),
                              _dtype_code(out.dtype), _ptr(scale), _stream(stream))
    _check(st, "retention_rotate")
    return out


def msr_desc(B, N, d_model, H, d_k, d_v, gamma, *, chunk=128, norm_flags=0, gn_eps=1e-6,
             pos0=0, theta_base=10000.0):
    g = _Gamma(gamma, H)
    m = MsrDesc()
    m.B, m.N, m.d_model, m.H, m.d_k, m.d_v, m.chunk = B, N, d_model, H, d_k, d_v, chunk
    m.gamma = g.ptr
    m.theta_base = float(theta_base)
    m.norm_flags = int(norm_flags)
    m.gn_eps = float(-1.0 if gn_eps is None else gn_eps)
    m.pos0 = int(pos0)
    return m, g


def msr_layer_fwd(X, WQ, WK, WV, WG, WO, *, H, d_k, d_v, gamma, chunk=128, norm_flags=0,
                  gn_eps=1e-6, pos0=0, theta_base=10000.0, out=None, workspace=None,
                  stream=None):
    B, N, dm = X.shape
    m, g = msr_desc(B, N, dm, H, d_k, d_v, gamma, chunk=chunk, norm_flags=norm_flags,
                    gn_eps=gn_eps, pos0=pos0, theta_base=theta_base)
    if out is None:
        out = torch.empty((B, N, dm), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = new_workspace(int(lib.msr_workspace_size(ctypes.byref(m))), X.device)
    for name, t in (("X", X), ("WQ", WQ), ("WK", WK), ("WV", WV), ("WG", WG), ("WO", WO)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    st = lib.msr_layer_fwd(ctypes.byref(m), _ptr(X), _ptr(WQ), _ptr(WK), _ptr(WV), _ptr(WG),
                           _ptr(WO), _ptr(out), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check(st, "msr_layer_fwd")
    return out


def block_desc(B, N, d_model, H, d_k, d_v, d_ffn, gamma, *, chunk=128, norm_flags=0,
               gn_eps=1e-6, ln_eps=1e-5, pos0=0, theta_base=10000.0):
    m, g = msr_desc(B, N, d_model, H, d_k, d_v, gamma, chunk=chunk, norm_flags=norm_flags,
                    gn_eps=gn_eps, pos0=pos0, theta_base=theta_base)
    d = BlockDesc()
    d.msr = m
    d.d_ffn = int(d_ffn)
    d.ln_eps = float(ln_eps)
    return d, g


def retnet_block_fwd(X, ln1_w, ln1_b, WQ, WK, WV, WG, WO, ln2_w, ln2_b, W1, W2, *, H, d_k, d_v,
                     gamma, chunk=128, norm_flags=0, gn_eps=1e-6, ln_eps=1e-5, pos0=0,
                     theta_base=10000.0, out=None, workspace=None, stream=None):
    """One RetNet block: Y = MSR(LN1(X)) + X, X' = gelu(LN2(Y) W1) W2 + Y.
    bf16 activations and weights, fp32 LayerNorm gains and biases."""
    B, N, dm = X.shape
    d, g = block_desc(B, N, dm, H, d_k, d_v, W1.shape[1], gamma, chunk=chunk,
                      norm_flags=norm_flags, gn_eps=gn_eps, ln_eps=ln_eps, pos0=pos0,
                      theta_base=theta_base)
    if out is None:
        out = torch.empty((B, N, dm), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = new_workspace(int(lib.retnet_block_workspace_size(ctypes.byref(d))),
                                  X.device)
    for name, t in (("X", X), ("WQ", WQ), ("WK", WK), ("WV", WV), ("WG", WG), ("WO", WO),
                    ("W1", W1), ("W2", W2)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    for name, t in (("ln1_w", ln1_w), ("ln1_b", ln1_b), ("ln2_w", ln2_w), ("ln2_b", ln2_b)):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != dm:
            raise ValueError(f"{name} must be a contiguous fp32 tensor of d_model values")
    st = lib.retnet_block_fwd(ctypes.byref(d), _ptr(X), _ptr(ln1_w), _ptr(ln1_b), _ptr(WQ),
                              _ptr(WK), _ptr(WV), _ptr(WG), _ptr(WO), _ptr(ln2_w), _ptr(ln2_b),
                              _ptr(W1), _ptr(W2), _ptr(out), _ptr(workspace), workspace.numel(),
                              _stream(stream))
    _check(st, "retnet_block_fwd")
    return out


def stack_desc(B, d_model, H, d_k, d_v, d_ffn, n_layers, gamma, *, pos, norm_flags=0,
               gn_eps=1e-6, ln_eps=1e-5, theta_base=10000.0):
    b, g = block_desc(B, 1, d_model, H, d_k, d_v, d_ffn, gamma, norm_flags=norm_flags,
                      gn_eps=gn_eps, ln_eps=ln_eps, pos0=pos, theta_base=theta_base)
    d = StackDesc()
    d.block = b
    d.n_layers = int(n_layers)
    return d, g


def retnet_decode_step(X, layers, S, z=None, *, H, d_k, d_v, gamma, pos, norm_flags=0,
                       gn_eps=1e-6, ln_eps=1e-5, theta_base=10000.0, workspace=None,
                       stream=None):
    """One decode step of a stack of RetNet blocks: X [B, d_model] bf16 is the
    token's input and is overwritten with the stack's output; `layers` is a
    list of dicts with the keys LAYER_KEYS (bf16 weights, fp32 LayerNorm
    gains and biases); S (and z, with the third normalisation) lists of the
    layers' fp32 states, updated in place."""
    if X.dim() != 2 or X.dtype != torch.bfloat16 or not X.is_contiguous():
        raise ValueError("X must be a contiguous bf16 [B, d_model] tensor")
    B, dm = X.shape
    n = len(layers)
    if len(S) != n or (z is not None and len(z) != n):
        raise ValueError("one state per layer")
    d_ffn = layers[0]["W1"].shape[1] if n else 1
    d, g = stack_desc(B, dm, H, d_k, d_v, d_ffn, n, gamma, pos=pos, norm_flags=norm_flags,
                      gn_eps=gn_eps, ln_eps=ln_eps, theta_base=theta_base)
    if workspace is None:
        workspace = new_workspace(int(lib.retnet_decode_workspace_size(ctypes.byref(d))),
                                  X.device)
    recs = (LayerWeights * max(n, 1))()
    for i, L in enumerate(layers):
        for k in LAYER_KEYS:
            t = L[k]
            want = torch.float32 if k.startswith("ln") else torch.bfloat16
            if t.dtype != want or not t.is_contiguous():
                raise ValueError(f"layer {i} {k}: contiguous {want} expected")
            setattr(recs[i], k, t.data_ptr())
    Sp = (ctypes.c_void_p * max(n, 1))(*[s.data_ptr() for s in S])
    zp = None if z is None else (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in z])
    st = lib.retnet_decode_step(ctypes.byref(d), recs, Sp, zp, _ptr(X), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(st, "retnet_decode_step")
    return X


def gemm_bf16(A, B, out=None, workspace=None, stream=None):
    """C = A @ B for bf16 row-major matrices (the MSR projections' GEMM)."""
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if workspace is None:
        workspace = new_workspace(int(lib.retention_gemm_workspace_size(M, N, K)), A.device)
    _check(lib.retention_gemm_bf16(_ptr(A), _ptr(B), _ptr(out), M, N, K, _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "retention_gemm_bf16")
    return out


def poll_status(workspace, stream=None):
    """Reads and clears the device status word (synchronises the stream)."""
    return int(lib.retention_poll_status(_ptr(workspace), _stream(stream)))


def kernel_times():
    """{kernel name: (total ms of timed launches, launches, timed launches)}
    since the last reset; call after synchronising the streams."""
    out = {}
    for i in range(lib.retention_kernel_count()):
        ms, n, t = ctypes.c_double(), ctypes.c_longlong(), ctypes.c_int()
        _check(lib.retention_kernel_timer_read(i, ctypes.byref(ms), ctypes.byref(n),
                                               ctypes.byref(t)), "kernel_timer_read")
        if n.value:
            out[lib.retention_kernel_name(i).decode()] = (ms.value, n.value, t.value)
    return out

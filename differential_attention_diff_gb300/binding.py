"""ctypes binding of libdiffattn.so (the C ABI in include/diffattn.h).

Argument marshalling only: each function takes torch CUDA tensors, fills the
C parameter struct with their device pointers, sizes and element strides,
calls the entry point of the same name on the current torch stream and
raises ``DiffAttnError`` on a non-OK status.  Output and workspace buffers
that the caller does not pass are allocated here with torch (device-memory
plumbing); every computation runs in the library's kernels.  There is no
fallback: if the shared library is missing or cannot be loaded, every call
raises.
"""

from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdiffattn.so")

DA_OK, DA_ERR_INVALID_ARG, DA_ERR_UNSUPPORTED, DA_ERR_CUDA, DA_ERR_TIMEOUT, DA_ERR_BOUNDS, \
    DA_ERR_WORKSPACE = range(7)
DA_F32, DA_BF16 = 0, 1

# Every symbol the header declares (checked by the ABI tests).
EXPORTS = (
    "diffattn_lambda_init",
    "diffattn_v1_fwd",
    "diffattn_v1_fwd_workspace_size",
    "diffattn_v1_bwd",
    "diffattn_v1_bwd_workspace_size",
    "diffattn_v1_decode",
    "diffattn_v1_decode_num_splits",
    "diffattn_v1_decode_workspace_size",
    "diffattn_v2_bwd",
    "diffattn_v2_bwd_workspace_size",
    "diffattn_grouped_fwd",
    "diffattn_grouped_fwd_workspace_size",
    "diffattn_grouped_bwd",
    "diffattn_grouped_bwd_workspace_size",
    "diffattn_v2_gate",
    "diffattn_v2_fwd",
    "diffattn_v2_fwd_workspace_size",
    "diffattn_v2_decode",
    "diffattn_v2_decode_noalloc",
    "diffattn_v2_decode_num_splits",
    "diffattn_v2_decode_workspace_size",
    "diffattn_get_device_status",
    "diffattn_debug_inject_fault",
    "diffattn_get_device_status_detail",
    "diffattn_status_string",
)


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_str(status)} (status {status})")


class da_t4(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("sb", C.c_int64), ("sn", C.c_int64), ("sh", C.c_int64)]


_fp = C.POINTER(C.c_float)


class da_v1_fwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("H", C.c_int), ("d_qk", C.c_int), ("d_v", C.c_int),
                ("dtype", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("lambda_init", C.c_float), ("rms_eps", C.c_float),
                ("q1", da_t4), ("q2", da_t4), ("k1", da_t4), ("k2", da_t4), ("v", da_t4),
                ("lq1", C.c_void_p), ("lk1", C.c_void_p), ("lq2", C.c_void_p), ("lk2", C.c_void_p),
                ("out", da_t4), ("lse1", C.c_void_p), ("lse2", C.c_void_p), ("rstd", C.c_void_p),
                ("o2", da_t4), ("lambda_out", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("rms_weight", C.c_void_p)]


class da_v1_bwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("H", C.c_int), ("d_qk", C.c_int), ("d_v", C.c_int),
                ("dtype", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("lambda_init", C.c_float), ("rms_eps", C.c_float),
                ("q1", da_t4), ("q2", da_t4), ("k1", da_t4), ("k2", da_t4), ("v", da_t4),
                ("lq1", C.c_void_p), ("lk1", C.c_void_p), ("lq2", C.c_void_p), ("lk2", C.c_void_p),
                ("out", da_t4), ("dout", da_t4),
                ("lse1", C.c_void_p), ("lse2", C.c_void_p), ("rstd", C.c_void_p), ("o2", da_t4),
                ("dq1", da_t4), ("dq2", da_t4), ("dk1", da_t4), ("dk2", da_t4), ("dv", da_t4),
                ("dlq1", C.c_void_p), ("dlk1", C.c_void_p), ("dlq2", C.c_void_p), ("dlk2", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("deterministic", C.c_int),
                ("rms_weight", C.c_void_p)]


class da_v1_decode_params(C.Structure):
    _fields_ = [("B", C.c_int), ("H", C.c_int), ("d_qk", C.c_int), ("d_v", C.c_int), ("L_max", C.c_int),
                ("softmax_scale", C.c_float), ("lambda_init", C.c_float), ("rms_eps", C.c_float),
                ("q1", C.c_void_p), ("q2", C.c_void_p), ("k1_cache", da_t4), ("k2_cache", da_t4),
                ("v_cache", da_t4), ("seqlens", C.c_void_p), ("lq1", C.c_void_p), ("lk1", C.c_void_p),
                ("lq2", C.c_void_p), ("lk2", C.c_void_p), ("out", C.c_void_p), ("num_splits", C.c_int),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("rms_weight", C.c_void_p)]


class da_v2_gate_params(C.Structure):
    _fields_ = [("T", C.c_int), ("d_model", C.c_int), ("h", C.c_int), ("x", C.c_void_p),
                ("x_stride", C.c_int64), ("w_lambda", C.c_void_p), ("gate", C.c_void_p)]


class da_v2_fwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("h", C.c_int), ("h_kv", C.c_int), ("d", C.c_int),
                ("d_model", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("q", da_t4), ("k", da_t4), ("v", da_t4), ("gate", C.c_void_p), ("x", C.c_void_p),
                ("w_lambda", C.c_void_p), ("out", da_t4), ("lse", C.c_void_p), ("o_heads", da_t4),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class da_grouped_fwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("h", C.c_int), ("ratio", C.c_int), ("h_kv", C.c_int),
                ("d", C.c_int), ("d_model", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("q", da_t4), ("k", da_t4), ("v", da_t4), ("gate", C.c_void_p), ("x", C.c_void_p),
                ("w_lambda", C.c_void_p), ("out", da_t4), ("lse", C.c_void_p), ("o_heads", da_t4),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class da_v2_bwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("h", C.c_int), ("h_kv", C.c_int), ("d", C.c_int),
                ("d_model", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("q", da_t4), ("k", da_t4), ("v", da_t4), ("gate", C.c_void_p), ("x", C.c_void_p),
                ("w_lambda", C.c_void_p), ("o_heads", da_t4), ("lse", C.c_void_p), ("dout", da_t4),
                ("dq", da_t4), ("dk", da_t4), ("dv", da_t4), ("dgate_logit", C.c_void_p),
                ("dx", C.c_void_p), ("dw_lambda", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class da_grouped_bwd_params(C.Structure):
    _fields_ = [("B", C.c_int), ("N", C.c_int), ("h", C.c_int), ("ratio", C.c_int), ("h_kv", C.c_int),
                ("d", C.c_int), ("d_model", C.c_int), ("causal", C.c_int), ("softmax_scale", C.c_float),
                ("q", da_t4), ("k", da_t4), ("v", da_t4), ("gate", C.c_void_p), ("x", C.c_void_p),
                ("w_lambda", C.c_void_p), ("o_heads", da_t4), ("lse", C.c_void_p), ("dout", da_t4),
                ("dq", da_t4), ("dk", da_t4), ("dv", da_t4), ("dgate_logit", C.c_void_p),
                ("dx", C.c_void_p), ("dw_lambda", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class da_v2_decode_params(C.Structure):
    _fields_ = [("B", C.c_int), ("h", C.c_int), ("h_kv", C.c_int), ("d", C.c_int),
                ("L_max", C.c_int), ("d_model", C.c_int), ("softmax_scale", C.c_float),
                ("q", C.c_void_p), ("k_cache", da_t4), ("v_cache", da_t4), ("seqlens", C.c_void_p),
                ("gate", C.c_void_p), ("x", C.c_void_p), ("w_lambda", C.c_void_p),
                ("out", C.c_void_p), ("num_splits", C.c_int), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load the shared library once and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m differential_attention_diff_gb300.build` "
                "(there is no fallback implementation)")
        lib = C.CDLL(path)
        vp = C.c_void_p
        lib.diffattn_lambda_init.restype = C.c_float
        lib.diffattn_lambda_init.argtypes = [C.c_int]
        lib.diffattn_status_string.restype = C.c_char_p
        lib.diffattn_status_string.argtypes = [C.c_int]
        for name, st in (("diffattn_v1_fwd", da_v1_fwd_params), ("diffattn_v1_bwd", da_v1_bwd_params),
                         ("diffattn_v2_gate", da_v2_gate_params), ("diffattn_v2_fwd", da_v2_fwd_params),
                         ("diffattn_v2_bwd", da_v2_bwd_params), ("diffattn_v1_decode", da_v1_decode_params),
                         ("diffattn_grouped_fwd", da_grouped_fwd_params),
                         ("diffattn_grouped_bwd", da_grouped_bwd_params),
                         ("diffattn_v2_decode", da_v2_decode_params),
                         ("diffattn_v2_decode_noalloc", da_v2_decode_params)):
            f = getattr(lib, name)
            f.restype = C.c_int
            f.argtypes = [C.POINTER(st), vp]
        lib.diffattn_v1_fwd_workspace_size.restype = C.c_size_t
        lib.diffattn_v1_fwd_workspace_size.argtypes = [C.c_int] * 6
        lib.diffattn_v1_bwd_workspace_size.restype = C.c_size_t
        lib.diffattn_v1_bwd_workspace_size.argtypes = [C.c_int] * 6
        lib.diffattn_v2_fwd_workspace_size.restype = C.c_size_t
        lib.diffattn_v2_fwd_workspace_size.argtypes = [C.c_int] * 4
        lib.diffattn_v1_decode_num_splits.restype = C.c_int
        lib.diffattn_v1_decode_num_splits.argtypes = [C.c_int] * 3
        lib.diffattn_v1_decode_workspace_size.restype = C.c_size_t
        lib.diffattn_v1_decode_workspace_size.argtypes = [C.c_int] * 5
        lib.diffattn_grouped_fwd_workspace_size.restype = C.c_size_t
        lib.diffattn_grouped_fwd_workspace_size.argtypes = [C.c_int] * 7
        lib.diffattn_grouped_bwd_workspace_size.restype = C.c_size_t
        lib.diffattn_grouped_bwd_workspace_size.argtypes = [C.c_int] * 5
        lib.diffattn_v2_bwd_workspace_size.restype = C.c_size_t
        lib.diffattn_v2_bwd_workspace_size.argtypes = [C.c_int] * 4
        lib.diffattn_v2_decode_num_splits.restype = C.c_int
        lib.diffattn_v2_decode_num_splits.argtypes = [C.c_int] * 3
        lib.diffattn_v2_decode_workspace_size.restype = C.c_size_t
        lib.diffattn_v2_decode_workspace_size.argtypes = [C.c_int] * 7
        lib.diffattn_debug_inject_fault.restype = C.c_int
        lib.diffattn_debug_inject_fault.argtypes = [C.c_int]
        lib.diffattn_get_device_status.restype = C.c_int
        lib.diffattn_get_device_status.argtypes = [vp]
        lib.diffattn_get_device_status_detail.restype = C.c_int
        lib.diffattn_get_device_status_detail.argtypes = [vp, C.POINTER(C.c_uint32)]
        _lib = lib
        return lib


def _status_str(status: int) -> str:
    try:
        return load().diffattn_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return "unknown"


def _check(status: int, what: str):
    if status != DA_OK:
        raise DiffAttnError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _t4(t):
    if t is None:
        return da_t4(None, 0, 0, 0)
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("4-D tensor with a contiguous last dimension expected")
    return da_t4(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DA_BF16
    if t.dtype == torch.float32:
        return DA_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def diffattn_lambda_init(layer: int) -> float:
    return float(load().diffattn_lambda_init(int(layer)))


def diffattn_v1_fwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, lambda_init, *, out=None,
                    causal=True, softmax_scale=0.0, rms_eps=1e-5, rms_weight=None, save=False,
                    saves=None, workspace=None, stream=None):
    """V1 forward.  Returns ``out`` or, with save=True, ``(out, saves)`` where
    saves = dict(lse1, lse2, rstd, o2, lam) are the tensors the backward reads.
    rms_weight: fp32 [d_v] RMSNorm weight (None = unit)."""
    lib = load()
    B, N, H, dqk = q1.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=v.dtype, device=v.device)
    if save and saves is None:
        f32 = dict(dtype=torch.float32, device=v.device)
        saves = dict(lse1=torch.empty((B, H, N), **f32), lse2=torch.empty((B, H, N), **f32),
                     rstd=torch.empty((B, H, N), **f32),
                     o2=torch.empty((B, N, H, dv), dtype=v.dtype, device=v.device),
                     lam=torch.empty((1,), **f32))
    if not save:
        saves = None
    need = lib.diffattn_v1_fwd_workspace_size(B, N, H, dqk, dv, _dtype_code(q1))
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=v.device)
    p = da_v1_fwd_params(
        B, N, H, dqk, dv, _dtype_code(q1), int(causal), float(softmax_scale), float(lambda_init),
        float(rms_eps), _t4(q1), _t4(q2), _t4(k1), _t4(k2), _t4(v), _ptr(lq1), _ptr(lk1),
        _ptr(lq2), _ptr(lk2), _t4(out),
        _ptr(saves["lse1"]) if saves else None, _ptr(saves["lse2"]) if saves else None,
        _ptr(saves["rstd"]) if saves else None, _t4(saves["o2"] if saves else None),
        _ptr(saves["lam"]) if saves else None, _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(rms_weight))
    _check(lib.diffattn_v1_fwd(C.byref(p), _stream(stream)), "diffattn_v1_fwd")
    return (out, saves) if save else out


def diffattn_v1_bwd(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, lambda_init, out, dout, saves, *,
                    causal=True, softmax_scale=0.0, rms_eps=1e-5, rms_weight=None, grads=None,
                    workspace=None, deterministic=False, stream=None):
    """V1 backward.  Returns dict(dq1, dq2, dk1, dk2, dv, dlq1, dlk1, dlq2, dlk2).
    deterministic=True makes dQ (and so every output) bitwise reproducible.
    rms_weight: the forward's RMSNorm weight (None = unit; entries nonzero)."""
    lib = load()
    B, N, H, dqk = q1.shape
    dv = v.shape[-1]
    if grads is None:
        grads = {n: torch.empty_like(t) for n, t in
                 (("dq1", q1), ("dq2", q2), ("dk1", k1), ("dk2", k2), ("dv", v),
                  ("dlq1", lq1), ("dlk1", lk1), ("dlq2", lq2), ("dlk2", lk2))}
    need = lib.diffattn_v1_bwd_workspace_size(B, N, H, dqk, dv, int(bool(deterministic)))
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=v.device)
    p = da_v1_bwd_params(
        B, N, H, dqk, dv, _dtype_code(q1), int(causal), float(softmax_scale), float(lambda_init),
        float(rms_eps), _t4(q1), _t4(q2), _t4(k1), _t4(k2), _t4(v), _ptr(lq1), _ptr(lk1),
        _ptr(lq2), _ptr(lk2), _t4(out), _t4(dout), _ptr(saves["lse1"]), _ptr(saves["lse2"]),
        _ptr(saves["rstd"]), _t4(saves["o2"]), _t4(grads["dq1"]), _t4(grads["dq2"]),
        _t4(grads["dk1"]), _t4(grads["dk2"]), _t4(grads["dv"]), _ptr(grads["dlq1"]),
        _ptr(grads["dlk1"]), _ptr(grads["dlq2"]), _ptr(grads["dlk2"]), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(bool(deterministic)), _ptr(rms_weight))
    _check(lib.diffattn_v1_bwd(C.byref(p), _stream(stream)), "diffattn_v1_bwd")
    return grads


def diffattn_v1_decode_num_splits(B, H, L_max) -> int:
    return int(load().diffattn_v1_decode_num_splits(B, H, L_max))


def diffattn_v1_decode_workspace_size(B, H, d_v, L_max, num_splits=0) -> int:
    return int(load().diffattn_v1_decode_workspace_size(B, H, d_v, L_max, num_splits))


def diffattn_v1_decode(q1, q2, k1_cache, k2_cache, v_cache, lq1, lk1, lq2, lk2, lambda_init, *,
                       seqlens=None, out=None, num_splits=0, softmax_scale=0.0, rms_eps=1e-5,
                       rms_weight=None, workspace=None, stream=None):
    """V1 decode: out [B, H, d_v] for one new token per sequence.
    rms_weight: fp32 [d_v] RMSNorm weight (None = unit)."""
    lib = load()
    B, H, dqk = q1.shape
    L_max, dv = v_cache.shape[1], v_cache.shape[3]
    if out is None:
        out = torch.empty((B, H, dv), dtype=q1.dtype, device=q1.device)
    need = lib.diffattn_v1_decode_workspace_size(B, H, dv, L_max, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q1.device)
    p = da_v1_decode_params(
        B, H, dqk, dv, L_max, float(softmax_scale), float(lambda_init), float(rms_eps), q1.data_ptr(),
        q2.data_ptr(), _t4(k1_cache), _t4(k2_cache), _t4(v_cache), _ptr(seqlens), _ptr(lq1), _ptr(lk1),
        _ptr(lq2), _ptr(lk2), out.data_ptr(), int(num_splits), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _ptr(rms_weight))
    _check(lib.diffattn_v1_decode(C.byref(p), _stream(stream)), "diffattn_v1_decode")
    return out


def diffattn_v2_gate(x, w_lambda, *, gate=None, stream=None):
    """gate = sigmoid(x @ w_lambda) for x [..., d_model] -> fp32 [..., h]."""
    lib = load()
    d_model = x.shape[-1]
    h = w_lambda.shape[1]
    x2 = x.reshape(-1, d_model)
    T = x2.shape[0]
    if gate is None:
        gate = torch.empty((*x.shape[:-1], h), dtype=torch.float32, device=x.device)
    p = da_v2_gate_params(T, d_model, h, x2.data_ptr(), x2.stride(0), w_lambda.data_ptr(),
                          gate.data_ptr())
    _check(lib.diffattn_v2_gate(C.byref(p), _stream(stream)), "diffattn_v2_gate")
    return gate


def diffattn_v2_fwd(q, k, v, *, gate=None, x=None, w_lambda=None, out=None, lse=None,
                    causal=True, softmax_scale=0.0, save=False, saves=None, workspace=None,
                    stream=None):
    """V2 forward: out [B, N, h, d] = O_even - gate * O_odd.  With save=True
    returns ``(out, saves)``, saves = dict(lse, o_heads): what the backward reads."""
    lib = load()
    B, N, H2, d = q.shape
    h = H2 // 2
    hkv = k.shape[2]
    if out is None:
        out = torch.empty((B, N, h, d), dtype=q.dtype, device=q.device)
    if save:
        if saves is None:
            saves = dict(lse=torch.empty((B, H2, N), dtype=torch.float32, device=q.device),
                         o_heads=torch.empty((B, N, H2, d), dtype=q.dtype, device=q.device))
        lse = saves["lse"]
    d_model = 0 if x is None else x.shape[-1]
    need = lib.diffattn_v2_fwd_workspace_size(B, N, h, int(gate is not None))
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    p = da_v2_fwd_params(
        B, N, h, hkv, d, d_model, int(causal), float(softmax_scale), _t4(q), _t4(k), _t4(v),
        _ptr(gate), _ptr(x), _ptr(w_lambda), _t4(out), _ptr(lse),
        _t4(saves["o_heads"] if save else None),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size())
    _check(lib.diffattn_v2_fwd(C.byref(p), _stream(stream)), "diffattn_v2_fwd")
    return (out, saves) if save else out


def diffattn_grouped_fwd(q, k, v, ratio, *, gate=None, x=None, w_lambda=None, out=None, lse=None,
                         o_heads=None, causal=True, softmax_scale=0.0, workspace=None, stream=None):
    """Grouped differential attention: q [B, N, h (ratio+1)/ratio, d] in groups
    of `ratio` signal heads then one noise head; out [B, N, h, d]."""
    lib = load()
    B, N, Hq, d = q.shape
    h = Hq // (ratio + 1) * ratio
    hkv = k.shape[2]
    if out is None:
        out = torch.empty((B, N, h, d), dtype=q.dtype, device=q.device)
    d_model = 0 if x is None else x.shape[-1]
    need = lib.diffattn_grouped_fwd_workspace_size(B, N, h, ratio, d, int(gate is not None),
                                                   int(o_heads is not None))
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    p = da_grouped_fwd_params(
        B, N, h, int(ratio), hkv, d, d_model, int(causal), float(softmax_scale), _t4(q), _t4(k), _t4(v),
        _ptr(gate), _ptr(x), _ptr(w_lambda), _t4(out), _ptr(lse), _t4(o_heads), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size())
    _check(lib.diffattn_grouped_fwd(C.byref(p), _stream(stream)), "diffattn_grouped_fwd")
    return out


def diffattn_v2_bwd_workspace_size(B, N, h, d_model=0) -> int:
    return int(load().diffattn_v2_bwd_workspace_size(B, N, h, d_model))


def diffattn_v2_bwd(q, k, v, dout, saves, *, gate=None, x=None, w_lambda=None, grads=None,
                    want_dx=None, want_dw=None, want_dz=False, causal=True, softmax_scale=0.0,
                    workspace=None, stream=None):
    """V2 backward.  Returns dict(dq, dk, dv) plus dx, dw (when x and w_lambda
    are given, unless want_dx / want_dw say otherwise) and dz (want_dz)."""
    lib = load()
    B, N, H2, d = q.shape
    h = H2 // 2
    hkv = k.shape[2]
    d_model = 0 if x is None else x.shape[-1]
    have_xw = x is not None and w_lambda is not None
    want_dx = have_xw if want_dx is None else want_dx
    want_dw = have_xw if want_dw is None else want_dw
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v))
        if want_dx:
            grads["dx"] = torch.empty((B, N, d_model), dtype=q.dtype, device=q.device)
        if want_dw:
            grads["dw"] = torch.empty((d_model, h), dtype=torch.float32, device=q.device)
        if want_dz:
            grads["dz"] = torch.empty((B, N, h), dtype=torch.float32, device=q.device)
    need = lib.diffattn_v2_bwd_workspace_size(B, N, h, d_model if grads.get("dw") is not None else 0)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    p = da_v2_bwd_params(
        B, N, h, hkv, d, d_model, int(causal), float(softmax_scale), _t4(q), _t4(k), _t4(v),
        _ptr(gate), _ptr(x), _ptr(w_lambda), _t4(saves["o_heads"]), _ptr(saves["lse"]), _t4(dout),
        _t4(grads["dq"]), _t4(grads["dk"]), _t4(grads["dv"]), _ptr(grads.get("dz")),
        _ptr(grads.get("dx")), _ptr(grads.get("dw")), workspace.data_ptr(),
        workspace.numel() * workspace.element_size())
    _check(lib.diffattn_v2_bwd(C.byref(p), _stream(stream)), "diffattn_v2_bwd")
    return grads


def diffattn_grouped_bwd_workspace_size(B, N, h, ratio, d_model=0) -> int:
    return int(load().diffattn_grouped_bwd_workspace_size(B, N, h, ratio, d_model))


def diffattn_grouped_bwd(q, k, v, dout, saves, ratio, *, gate=None, x=None, w_lambda=None, grads=None,
                         want_dx=None, want_dw=None, want_dz=False, causal=True, softmax_scale=0.0,
                         workspace=None, stream=None):
    """Grouped differential attention backward.  saves: dict(o_heads [B, N, Hq,
    d] bf16, lse [B, Hq, N] fp32) written by diffattn_grouped_fwd.  Returns
    dict(dq, dk, dv) plus dx, dw (when x and w_lambda are given, unless
    want_dx / want_dw say otherwise) and dz (want_dz)."""
    lib = load()
    B, N, Hq, d = q.shape
    h = Hq // (ratio + 1) * ratio
    hkv = k.shape[2]
    d_model = 0 if x is None else x.shape[-1]
    have_xw = x is not None and w_lambda is not None
    want_dx = have_xw if want_dx is None else want_dx
    want_dw = have_xw if want_dw is None else want_dw
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v))
        if want_dx:
            grads["dx"] = torch.empty((B, N, d_model), dtype=q.dtype, device=q.device)
        if want_dw:
            grads["dw"] = torch.empty((d_model, h), dtype=torch.float32, device=q.device)
        if want_dz:
            grads["dz"] = torch.empty((B, N, h), dtype=torch.float32, device=q.device)
    need = lib.diffattn_grouped_bwd_workspace_size(B, N, h, ratio,
                                                   d_model if grads.get("dw") is not None else 0)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    p = da_grouped_bwd_params(
        B, N, h, int(ratio), hkv, d, d_model, int(causal), float(softmax_scale), _t4(q), _t4(k), _t4(v),
        _ptr(gate), _ptr(x), _ptr(w_lambda), _t4(saves["o_heads"]), _ptr(saves["lse"]), _t4(dout),
        _t4(grads["dq"]), _t4(grads["dk"]), _t4(grads["dv"]), _ptr(grads.get("dz")),
        _ptr(grads.get("dx")), _ptr(grads.get("dw")), workspace.data_ptr(),
        workspace.numel() * workspace.element_size())
    _check(lib.diffattn_grouped_bwd(C.byref(p), _stream(stream)), "diffattn_grouped_bwd")
    return grads


def diffattn_v2_decode_num_splits(B, h_kv, L_max) -> int:
    return int(load().diffattn_v2_decode_num_splits(B, h_kv, L_max))


def diffattn_v2_decode_workspace_size(B, h, h_kv, d, L_max, num_splits=0, gate_given=False) -> int:
    return int(load().diffattn_v2_decode_workspace_size(B, h, h_kv, d, L_max, num_splits,
                                                        int(gate_given)))


def diffattn_v2_decode(q, k_cache, v_cache, *, seqlens=None, gate=None, x=None, w_lambda=None,
                       out=None, num_splits=0, softmax_scale=0.0, workspace=None, stream=None):
    """V2 decode: out [B, h, d] for one new token per sequence."""
    lib = load()
    B, H2, d = q.shape
    h = H2 // 2
    L_max, hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((B, h, d), dtype=q.dtype, device=q.device)
    d_model = 0 if x is None else x.shape[-1]
    need = lib.diffattn_v2_decode_workspace_size(B, h, hkv, d, L_max, num_splits,
                                                 int(gate is not None))
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    p = da_v2_decode_params(
        B, h, hkv, d, L_max, d_model, float(softmax_scale), q.data_ptr(), _t4(k_cache),
        _t4(v_cache), _ptr(seqlens), _ptr(gate), _ptr(x), _ptr(w_lambda), out.data_ptr(),
        int(num_splits), workspace.data_ptr(), workspace.numel() * workspace.element_size())
    _check(lib.diffattn_v2_decode(C.byref(p), _stream(stream)), "diffattn_v2_decode")
    return out


def diffattn_v2_decode_noalloc(q, k_cache, v_cache, *, seqlens=None, gate=None, x=None,
                               w_lambda=None, out=None, num_splits=0, softmax_scale=0.0,
                               stream=None):
    """V2 decode through the entry point that takes no workspace (its scratch
    is a fixed array inside the library; see include/diffattn.h)."""
    lib = load()
    B, H2, d = q.shape
    h = H2 // 2
    L_max, hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty((B, h, d), dtype=q.dtype, device=q.device)
    d_model = 0 if x is None else x.shape[-1]
    p = da_v2_decode_params(
        B, h, hkv, d, L_max, d_model, float(softmax_scale), q.data_ptr(), _t4(k_cache),
        _t4(v_cache), _ptr(seqlens), _ptr(gate), _ptr(x), _ptr(w_lambda), out.data_ptr(),
        int(num_splits), None, 0)
    _check(lib.diffattn_v2_decode_noalloc(C.byref(p), _stream(stream)), "diffattn_v2_decode_noalloc")
    return out


DA_FAULT_NONE, DA_FAULT_V2_FWD_SKIP_LOAD = 0, 1


def diffattn_debug_inject_fault(fault: int):
    """Test hook: arm a one-shot fault for the next call it applies to."""
    _check(load().diffattn_debug_inject_fault(int(fault)), "diffattn_debug_inject_fault")


def diffattn_get_device_status(stream=None, detail=False):
    lib = load()
    if detail:
        raw = C.c_uint32(0)
        st = lib.diffattn_get_device_status_detail(_stream(stream), C.byref(raw))
        return st, raw.value
    return lib.diffattn_get_device_status(_stream(stream))

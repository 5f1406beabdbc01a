"""ctypes binding of libipttt (include/ipttt.h): argument marshalling only.

Every function takes torch tensors that live on the current CUDA device,
passes their data pointers, sizes and the current torch stream to the C entry
point of the same name, and raises :class:`IptttError` on a non-OK status.  No
step of the layer runs in Python or PyTorch; if ``libipttt.so`` is missing,
loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libipttt.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALLOC, ERR_LAUNCH, ERR_TIMEOUT, ERR_CUDA = range(7)
FP32, BF16 = 0, 1
RULE_MSE, RULE_ADD, RULE_ADD_BLOCKCAUSAL = 0, 1, 2
_RULES = {"mse": RULE_MSE, "add": RULE_ADD, "add_blockcausal": RULE_ADD_BLOCKCAUSAL,
          RULE_MSE: RULE_MSE, RULE_ADD: RULE_ADD, RULE_ADD_BLOCKCAUSAL: RULE_ADD_BLOCKCAUSAL}

# Every symbol include/ipttt.h declares (checked by the ABI tests).
EXPORTS = (
    "ipttt_layer_forward", "ipttt_make_targets", "ipttt_gate_up", "ipttt_chunk_forward",
    "ipttt_workspace_size", "ipttt_sync_status", "ipttt_release", "ipttt_last_launch_count",
    "ipttt_status_string", "ipttt_version", "ipttt_kernel_timing", "ipttt_kernel_timing_read",
    "ipttt_kernel_name", "ipttt_make_targets_noalloc", "ipttt_layer_forward_varlen", "ipttt_layers_forward",
    "ipttt_additive_sums", "ipttt_weight_axpy", "ipttt_set_pool_limit", "ipttt_set_wait_limit",
)
NOALLOC_SCRATCH_BYTES = 16 << 20  # IPTTT_NOALLOC_SCRATCH_BYTES
KERNEL_KINDS = ("gate_up", "conv", "proj", "apply", "residual", "update", "group_sum", "scan", "weight_copy",
                "scores", "engine", "window")


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("d", ctypes.c_int64), ("d_ff", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("w0_per_seq", ctypes.c_int32)]


class IptttError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libipttt.so (built by chunked_weight_mlp_place_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m chunked_weight_mlp_place_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32
        dp = ctypes.POINTER(Dims)
        L.ipttt_layer_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp, vp, dp, vp]
        L.ipttt_set_pool_limit.argtypes = [ctypes.c_size_t]
        L.ipttt_set_wait_limit.argtypes = [ctypes.c_uint64]
        L.ipttt_set_wait_limit.restype = i32
        L.ipttt_additive_sums.argtypes = [vp, vp, i64, vp, dp, vp]
        L.ipttt_weight_axpy.argtypes = [vp, vp, f32, i64, vp]
        L.ipttt_layers_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, i32, vp, vp, dp, vp]
        L.ipttt_layer_forward_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(i64), i64, i64, f32,
                                                 i32, vp, vp, dp, vp]
        L.ipttt_make_targets.argtypes = [vp, vp, vp, vp, i64, i64, dp, vp]
        L.ipttt_make_targets_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, dp, vp]
        L.ipttt_gate_up.argtypes = [vp, vp, vp, vp, i64, dp, vp]
        L.ipttt_chunk_forward.argtypes = [vp, vp, vp, i64, i64, f32, i32, vp, vp, dp, vp]
        L.ipttt_workspace_size.argtypes = [dp, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
        L.ipttt_sync_status.argtypes = [vp]
        L.ipttt_release.argtypes = []
        L.ipttt_last_launch_count.argtypes = []
        L.ipttt_last_launch_count.restype = i64
        L.ipttt_status_string.argtypes = [i32]
        L.ipttt_status_string.restype = ctypes.c_char_p
        L.ipttt_version.argtypes = []
        L.ipttt_kernel_timing.argtypes = [i32]
        L.ipttt_kernel_timing.restype = i32
        L.ipttt_kernel_timing_read.argtypes = [i32, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
        L.ipttt_kernel_timing_read.restype = i32
        L.ipttt_kernel_name.argtypes = [i32]
        L.ipttt_kernel_name.restype = ctypes.c_char_p
        for name in ("ipttt_layer_forward", "ipttt_make_targets", "ipttt_make_targets_noalloc", "ipttt_gate_up",
                     "ipttt_chunk_forward",
                     "ipttt_workspace_size", "ipttt_sync_status", "ipttt_release"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ipttt_status_string(int(status)).decode()


def version() -> int:
    return int(lib().ipttt_version())


def last_launch_count() -> int:
    """Kernels the last call from this thread queued."""
    return int(lib().ipttt_last_launch_count())


def _check(status: int, where: str) -> None:
    if status != OK:
        raise IptttError(status, where)


# ------------------------------------------------------------- tensor helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"activations must be bfloat16 or float32, got {t.dtype}")


def _ptr(t, name: str, dtype=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _shape(t, shape, name: str) -> None:
    """The C-ABI takes sizes, not tensors: a tensor smaller than the sizes say
    would be read or written past its end on the device, so shapes are checked
    here, before the call."""
    if t is not None and tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(int(x) for x in shape)}")


def _rows_per_seq(rows: int, L: int, name: str) -> int:
    if L <= 0 or rows % L:
        raise ValueError(f"{name} has {rows} rows, not a whole number of sequences of L={L}")
    return rows // L


def _w0_shapes(W_o0, batch: int, d_ff: int, d: int):
    if W_o0.dim() == 3:
        _shape(W_o0, (batch, d_ff, d), "W_o0")
    else:
        _shape(W_o0, (d_ff, d), "W_o0")


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def dims(batch: int, d: int, d_ff: int, dtype: int, w0_per_seq: int = 0) -> Dims:
    return Dims(int(batch), int(d), int(d_ff), int(dtype), int(w0_per_seq))


# ------------------------------------------------------------------ entry points
def layer_forward(X, E, W_g, W_u, W_o0, conv_w, P, L: int, B: int, eta: float, rule, O, W_final,
                  stream=None) -> None:
    """ipttt_layer_forward on tensors: X, E (batch*L, d); W_g, W_u (d, d_ff);
    W_o0 (d_ff, d) or (batch, d_ff, d) fp32; conv_w (d, 4) fp32; P (d, d);
    O (batch*L, d) out; W_final (batch, d_ff, d) fp32 out."""
    torch = _torch()
    act = X.dtype
    d, d_ff = W_g.shape
    batch = _rows_per_seq(X.shape[0], L, "X") if L else W_final.shape[0]
    for t, shp, nm in ((X, (batch * L, d), "X"), (E, (batch * L, d), "E"), (W_u, (d, d_ff), "W_u"),
                       (conv_w, (d, 4), "conv_w"), (P, (d, d), "P"), (O, (batch * L, d), "O"),
                       (W_final, (batch, d_ff, d), "W_final")):
        _shape(t, shp, nm)
    _w0_shapes(W_o0, batch, d_ff, d)
    dm = dims(batch, d, d_ff, _dtype_code(X), 1 if W_o0.dim() == 3 else 0)
    st = lib().ipttt_layer_forward(
        _ptr(X, "X", act), _ptr(E, "E", act), _ptr(W_g, "W_g", act), _ptr(W_u, "W_u", act),
        _ptr(W_o0, "W_o0", torch.float32), _ptr(conv_w, "conv_w", torch.float32), _ptr(P, "P", act),
        int(L), int(B), float(eta), _RULES[rule], _ptr(O, "O", act), _ptr(W_final, "W_final", torch.float32),
        ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_layer_forward")


def layer_forward_varlen(X, E, W_g, W_u, W_o0, conv_w, P, cu_seqlens, B: int, eta: float, rule, O, W_final,
                         stream=None) -> None:
    """ipttt_layer_forward_varlen on tensors: packed documents X, E (T, d) with
    boundaries cu_seqlens (n_docs+1 ints, host); W_o0 (d_ff, d) or
    (n_docs, d_ff, d) fp32; O (T, d) out; W_final (n_docs, d_ff, d) fp32 out.
    The fast weight restarts from W_o0 at every document."""
    torch = _torch()
    act = X.dtype
    d, d_ff = W_g.shape
    cu = [int(c) for c in cu_seqlens]
    n_docs = len(cu) - 1
    T = X.shape[0]
    if n_docs < 0 or cu[-1] != T:
        raise ValueError(f"cu_seqlens must end at the number of rows of X ({T})")
    for t, shp, nm in ((E, (T, d), "E"), (W_u, (d, d_ff), "W_u"), (conv_w, (d, 4), "conv_w"), (P, (d, d), "P"),
                       (O, (T, d), "O"), (W_final, (n_docs, d_ff, d), "W_final")):
        _shape(t, shp, nm)
    _w0_shapes(W_o0, n_docs, d_ff, d)
    cu_arr = (ctypes.c_int64 * max(1, len(cu)))(*cu)
    dm = dims(n_docs, d, d_ff, _dtype_code(X), 1 if W_o0.dim() == 3 else 0)
    st = lib().ipttt_layer_forward_varlen(
        _ptr(X, "X", act), _ptr(E, "E", act), _ptr(W_g, "W_g", act), _ptr(W_u, "W_u", act),
        _ptr(W_o0, "W_o0", torch.float32), _ptr(conv_w, "conv_w", torch.float32), _ptr(P, "P", act),
        cu_arr, int(n_docs), int(B), float(eta), _RULES[rule], _ptr(O, "O", act),
        _ptr(W_final, "W_final", torch.float32), ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_layer_forward_varlen")


def layers_forward(X, E, W_g, W_u, W_o0, conv_w, P, L: int, B: int, eta: float, rule, O, W_final,
                   stream=None) -> None:
    """ipttt_layers_forward on tensors: X (n_layers, batch*L, d); E (batch*L, d);
    W_g, W_u (n_layers, d, d_ff); W_o0 (n_layers, d_ff, d) or
    (n_layers, batch, d_ff, d) fp32; conv_w (n_layers, d, 4) fp32; P (n_layers, d, d);
    O (n_layers, batch*L, d) out; W_final (n_layers, batch, d_ff, d) fp32 out."""
    torch = _torch()
    act = X.dtype
    n_layers, d, d_ff = W_g.shape
    batch = _rows_per_seq(X.shape[1], L, "X") if L else W_final.shape[1]
    for t, shp, nm in ((X, (n_layers, batch * L, d), "X"), (E, (batch * L, d), "E"), (W_u, (n_layers, d, d_ff), "W_u"),
                       (conv_w, (n_layers, d, 4), "conv_w"), (P, (n_layers, d, d), "P"),
                       (O, (n_layers, batch * L, d), "O"), (W_final, (n_layers, batch, d_ff, d), "W_final")):
        _shape(t, shp, nm)
    if W_o0.dim() == 4:
        _shape(W_o0, (n_layers, batch, d_ff, d), "W_o0")
    else:
        _shape(W_o0, (n_layers, d_ff, d), "W_o0")
    dm = dims(batch, d, d_ff, _dtype_code(X), 1 if W_o0.dim() == 4 else 0)
    st = lib().ipttt_layers_forward(
        _ptr(X, "X", act), _ptr(E, "E", act), _ptr(W_g, "W_g", act), _ptr(W_u, "W_u", act),
        _ptr(W_o0, "W_o0", torch.float32), _ptr(conv_w, "conv_w", torch.float32), _ptr(P, "P", act),
        int(n_layers), int(L), int(B), float(eta), _RULES[rule], _ptr(O, "O", act),
        _ptr(W_final, "W_final", torch.float32), ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_layers_forward")


def _targets_shapes(E, conv_w, P, V, L: int) -> None:
    d = E.shape[1]
    if L:
        _rows_per_seq(E.shape[0], L, "E")
    _shape(V, E.shape, "V")
    _shape(P, (d, d), "P")
    _shape(conv_w, (d, 4), "conv_w")


def make_targets(E, conv_w, P, V, L: int, B: int, stream=None) -> None:
    """ipttt_make_targets: V = Proj(Conv(E)) with chunk-end padding."""
    torch = _torch()
    act = E.dtype
    d = E.shape[1]
    _targets_shapes(E, conv_w, P, V, L)
    dm = dims(E.shape[0] // L if L else 0, d, 8, _dtype_code(E))
    st = lib().ipttt_make_targets(_ptr(E, "E", act), _ptr(conv_w, "conv_w", torch.float32), _ptr(P, "P", act),
                                  _ptr(V, "V", act), int(L), int(B), ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_make_targets")


def make_targets_noalloc(E, conv_w, P, V, L: int, B: int, stream=None) -> None:
    """ipttt_make_targets_noalloc: the same targets as make_targets, with the
    conv scratch in the library's fixed device array, so nothing is allocated.
    For callers that cannot allocate device memory here (memory already handed
    out by another allocator, or no room for a possibly synchronising
    cudaMalloc).  batch*L*d act elements must fit in NOALLOC_SCRATCH_BYTES."""
    torch = _torch()
    act = E.dtype
    d = E.shape[1]
    _targets_shapes(E, conv_w, P, V, L)
    dm = dims(E.shape[0] // L if L else 0, d, 8, _dtype_code(E))
    st = lib().ipttt_make_targets_noalloc(_ptr(E, "E", act), _ptr(conv_w, "conv_w", torch.float32),
                                          _ptr(P, "P", act), _ptr(V, "V", act), int(L), int(B), ctypes.byref(dm),
                                          _stream(stream))
    if st == ERR_INVALID_ARG and E.shape[0] * d * E.element_size() > NOALLOC_SCRATCH_BYTES:
        raise IptttError(st, f"ipttt_make_targets_noalloc: {E.shape[0]} x {d} conv rows need "
                             f"{E.shape[0] * d * E.element_size()} bytes, more than the fixed "
                             f"{NOALLOC_SCRATCH_BYTES}-byte scratch")
    _check(st, "ipttt_make_targets_noalloc")


def gate_up(X, W_g, W_u, Z, stream=None) -> None:
    """ipttt_gate_up: Z = SiLU(X W_g) * (X W_u)."""
    act = X.dtype
    d, d_ff = W_g.shape
    T = X.shape[0]
    for t, shp, nm in ((X, (T, d), "X"), (W_u, (d, d_ff), "W_u"), (Z, (T, d_ff), "Z")):
        _shape(t, shp, nm)
    dm = dims(1, d, d_ff, _dtype_code(X))
    st = lib().ipttt_gate_up(_ptr(X, "X", act), _ptr(W_g, "W_g", act), _ptr(W_u, "W_u", act), _ptr(Z, "Z", act),
                             int(X.shape[0]), ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_gate_up")


def chunk_forward(Z, V, W_o0, L: int, B: int, eta: float, rule, O, W_final, stream=None) -> None:
    """ipttt_chunk_forward on precomputed Z (batch*L, d_ff) and V (batch*L, d)."""
    torch = _torch()
    act = Z.dtype
    d_ff = Z.shape[1]
    d = V.shape[1]
    batch = _rows_per_seq(Z.shape[0], L, "Z") if L else W_final.shape[0]
    for t, shp, nm in ((V, (batch * L, d), "V"), (O, (batch * L, d), "O"), (W_final, (batch, d_ff, d), "W_final")):
        _shape(t, shp, nm)
    _w0_shapes(W_o0, batch, d_ff, d)
    dm = dims(batch, d, d_ff, _dtype_code(Z), 1 if W_o0.dim() == 3 else 0)
    st = lib().ipttt_chunk_forward(_ptr(Z, "Z", act), _ptr(V, "V", act), _ptr(W_o0, "W_o0", torch.float32),
                                   int(L), int(B), float(eta), _RULES[rule], _ptr(O, "O", act),
                                   _ptr(W_final, "W_final", torch.float32), ctypes.byref(dm), _stream(stream))
    _check(st, "ipttt_chunk_forward")


def set_pool_limit(nbytes: int) -> None:
    """ipttt_set_pool_limit: calls needing more scratch than `nbytes` fail with
    IPTTT_ERR_ALLOC before queuing anything (0 = no limit)."""
    _check(lib().ipttt_set_pool_limit(int(nbytes)), "ipttt_set_pool_limit")


def set_wait_limit(ns: int) -> None:
    """ipttt_set_wait_limit: soft limit (ns) of the tensor-core kernels' pipeline
    waits on the current device; 0 restores the default.  A longer wait makes
    the call's outputs unspecified and ipttt_sync_status report ERR_TIMEOUT."""
    _check(lib().ipttt_set_wait_limit(int(ns)), "ipttt_set_wait_limit")


def copy_weights(W_o0, W, stream=None) -> None:
    """W[s] = W_o0 (or W_o0[s] when W_o0 is per sequence) for every sequence s of
    W (batch, d_ff, d): ipttt_chunk_forward over zero tokens."""
    torch = _torch()
    d_ff, d = W_o0.shape[-2], W_o0.shape[-1]
    dm = dims(W.shape[0], d, d_ff, FP32, 1 if W_o0.dim() == 3 else 0)
    _check(lib().ipttt_chunk_forward(None, None, _ptr(W_o0, "W_o0", torch.float32), 0, 1, 0.0, RULE_ADD, None,
                                     _ptr(W, "W", torch.float32), ctypes.byref(dm), _stream(stream)),
           "ipttt_chunk_forward")


def additive_sums(Z, V, L: int, S, stream=None) -> None:
    """ipttt_additive_sums: S[s] = Z_s^T V_s (fp32, (batch, d_ff, d)) over L tokens per sequence."""
    torch = _torch()
    act = Z.dtype
    batch = _rows_per_seq(Z.shape[0], L, "Z") if L else S.shape[0]
    _shape(V, (batch * L, V.shape[1]), "V")
    _shape(S, (batch, Z.shape[1], V.shape[1]), "S")
    dm = dims(batch, V.shape[1], Z.shape[1], _dtype_code(Z))
    _check(lib().ipttt_additive_sums(_ptr(Z, "Z", act), _ptr(V, "V", act), int(L), _ptr(S, "S", torch.float32),
                                     ctypes.byref(dm), _stream(stream)), "ipttt_additive_sums")


def weight_axpy(W, S, alpha: float, stream=None) -> None:
    """ipttt_weight_axpy: W += alpha * S on fp32 tensors of the same size."""
    torch = _torch()
    if W.numel() != S.numel():
        raise ValueError("W and S differ in size")
    _check(lib().ipttt_weight_axpy(_ptr(W, "W", torch.float32), _ptr(S, "S", torch.float32), float(alpha),
                                   int(W.numel()), _stream(stream)), "ipttt_weight_axpy")


def workspace_size(batch: int, d: int, d_ff: int, dtype: int, L: int, B: int, rule, with_activations=True) -> int:
    out = ctypes.c_size_t(0)
    dm = dims(batch, d, d_ff, dtype)
    _check(lib().ipttt_workspace_size(ctypes.byref(dm), int(L), int(B), _RULES[rule], int(bool(with_activations)),
                                      ctypes.byref(out)), "ipttt_workspace_size")
    return int(out.value)


def sync_status(stream=None) -> int:
    """Synchronise the stream and return the device status (OK, ERR_TIMEOUT, ...)."""
    return int(lib().ipttt_sync_status(_stream(stream)))


def kernel_timing(enable: bool) -> None:
    """Start (clearing the totals) or stop per-kernel CUDA-event timing."""
    _check(lib().ipttt_kernel_timing(1 if enable else 0), "ipttt_kernel_timing")


def kernel_timing_read() -> dict:
    """{kernel name: (launches, total device ms)} since timing was started."""
    out = {}
    for k, name in enumerate(KERNEL_KINDS):
        n, ms = ctypes.c_int64(0), ctypes.c_double(0.0)
        _check(lib().ipttt_kernel_timing_read(k, ctypes.byref(n), ctypes.byref(ms)), "ipttt_kernel_timing_read")
        if n.value:
            out[name] = (int(n.value), float(ms.value))
    return out


def release() -> None:
    _check(lib().ipttt_release(), "ipttt_release")

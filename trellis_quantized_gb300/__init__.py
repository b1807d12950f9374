"""trellis_quantized_gb300 -- Python binding of libexl3 (the EXL3 trellis linear on GB300).

A thin ctypes layer over the C ABI declared in include/exl3.h: every function
here has the name of the C entry point it wraps and only marshals torch
tensors into device pointers, sizes and the current CUDA stream.  All
arithmetic runs in the library's CUDA kernels; there is no CPU path.  If
libexl3.so cannot be built or loaded, importing a function raises.

Tensors: fp16 data is passed as torch.float16 (or any 2-byte dtype holding
binary16 bits), trellis words as a 2-byte integer tensor (torch.int16 or
torch.uint16) shaped [k/16, n/16, 16K], all contiguous on the same CUDA
device.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _build

EXL3_OK = 0
EXL3_ERR_ARG = 1
EXL3_ERR_SHAPE = 2
EXL3_ERR_BITS = 3
EXL3_ERR_CODEBOOK = 4
EXL3_ERR_WORKSPACE = 5
EXL3_ERR_CUDA = 6
EXL3_ERR_DEVICE = 7

EXL3_CB_MCG = 1
EXL3_CB_MUL1 = 2
EXL3_CB_3INST = 3
EXL3_OUT_F16 = 0
EXL3_OUT_F32 = 1

_lock = threading.Lock()
_lib = None


class ExpertProj(ctypes.Structure):
    """exl3_expert_proj: one projection kind for all experts (device pointers)."""
    _fields_ = [("trellis", ctypes.c_void_p), ("suh", ctypes.c_void_p), ("svh", ctypes.c_void_p),
                ("k", ctypes.c_int), ("n", ctypes.c_int), ("K", ctypes.c_int), ("codebook", ctypes.c_int),
                ("nslots", ctypes.c_int)]


class ExpertProjMixed(ctypes.Structure):
    """exl3_expert_proj_mixed: one projection kind with a width per expert
    (device trellis/suh/svh, host widths K[E])."""
    _fields_ = [("trellis", ctypes.c_void_p), ("suh", ctypes.c_void_p), ("svh", ctypes.c_void_p),
                ("K", ctypes.POINTER(ctypes.c_int32)), ("k", ctypes.c_int), ("n", ctypes.c_int),
                ("codebook", ctypes.c_int), ("nslots", ctypes.c_int)]


class Exl3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libexl3 error {code}: {msg}")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load libexl3.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I, Z, L64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int64
        L.exl3_last_error.restype = ctypes.c_char_p
        L.exl3_version.restype = I
        L.exl3_workspace_clear.argtypes = [P, Z, P]
        L.exl3_copy_in.argtypes = [P, P, Z, P]
        L.exl3_check_device_error.argtypes = [P, Z, P, ctypes.POINTER(I)]
        L.exl3_decode_tile.argtypes = [P, I, I, I, I, I, I, I, I, P, L64, P]
        L.exl3_input_rht.argtypes = [P, I, I, P, P, I, P]
        L.exl3_linear_workspace_size.argtypes = [I, I, I, I]
        L.exl3_linear_workspace_size.restype = Z
        L.exl3_linear.argtypes = [P, I, I, I, P, P, P, I, I, P, I, P, Z, P]
        L.exl3_linear_bias.argtypes = [P, I, I, I, P, P, P, P, I, I, P, I, P, Z, P]
        L.exl3_linear_int8_workspace_size.argtypes = [I, I, I, I]
        L.exl3_linear_int8_workspace_size.restype = Z
        L.exl3_linear_int8.argtypes = [P, I, I, I, P, P, P, I, I, ctypes.c_float, P, P, P, P, P, Z, P]
        L.exl3_linear_int8_bias.argtypes = [P, I, I, I, P, P, P, P, I, I, ctypes.c_float, P, P, P, P, P, Z, P]
        L.exl3_moe_workspace_size.argtypes = [I, I, I, P, P]
        L.exl3_moe_workspace_size.restype = Z
        L.exl3_moe_grouped.argtypes = [P, I, I, P, P, I, I, P, P, P, I, P, Z, P]
        L.exl3_linear_gemv_noalloc.argtypes = [P, I, I, P, P, P, I, I, P, I, P]
        L.exl3_noalloc_device_error.argtypes = [P, ctypes.POINTER(I)]
        L.exl3_linear_shards_workspace_size.argtypes = [I, I, I, I, I]
        L.exl3_linear_shards_workspace_size.restype = Z
        L.exl3_linear_shards.argtypes = [P, I, I, I, I, P, P, P, I, I, P, I, P, Z, P]
        L.exl3_linear_shards_var_workspace_size.argtypes = [I, I, I, P, I]
        L.exl3_linear_shards_var_workspace_size.restype = Z
        L.exl3_linear_shards_var.argtypes = [P, I, I, I, P, P, P, P, I, I, P, I, P, Z, P]
        L.exl3_moe_mixed_workspace_size.argtypes = [I, I, I, P, P]
        L.exl3_moe_mixed_workspace_size.restype = Z
        L.exl3_moe_grouped_mixed.argtypes = [P, I, I, P, P, I, I, P, P, P, I, P, Z, P]
        L.exl3_set_weight_prefetch.argtypes = [I]
        L.exl3_set_weight_prefetch.restype = I
        L.exl3_set_row_invariant.argtypes = [I]
        L.exl3_set_row_invariant.restype = I
        _lib = L
        return L


def _check(rc: int):
    if rc != EXL3_OK:
        raise Exl3Error(rc, lib().exl3_last_error().decode())


def _ptr(t, name: str, itemsize: int | None = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if itemsize is not None and t.element_size() != itemsize:
        raise TypeError(f"{name} must have {itemsize}-byte elements, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _ptr_pinned(t, name: str):
    """A pinned host tensor's address (the device addresses pinned memory directly)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    # (is_pinned asks the driver about the address; skipped while a CUDA
    # graph is being captured)
    if t.is_cuda or (not torch.cuda.is_current_stream_capturing() and not t.is_pinned()):
        raise ValueError(f"{name} must be a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


_ws_cache: dict = {}


def workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace of at least nbytes, cached per (device, stream).

    Every libexl3 call leaves its counters at zero again, so one cleared
    workspace serves any number of calls made in stream order."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    key = (dev.index, s.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        exl3_workspace_clear(buf, stream=s)
        _ws_cache[key] = buf
    return buf


# ------------------------------------------------------------------ entry points

def exl3_version() -> int:
    return lib().exl3_version()


def exl3_workspace_clear(ws: torch.Tensor, stream=None):
    _check(lib().exl3_workspace_clear(_ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)))


def exl3_copy_in(src: torch.Tensor, dst: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy a pinned host tensor into a device tensor of the same byte size with
    a kernel chained by programmatic dependent launch (see exl3_copy_in in exl3.h)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst must have the same size in bytes")
    _check(lib().exl3_copy_in(_ptr_pinned(src, "src"), _ptr(dst, "dst"), nbytes, _stream(stream)))
    return dst


def exl3_check_device_error(ws: torch.Tensor, stream=None) -> int:
    err = ctypes.c_int(0)
    _check(lib().exl3_check_device_error(_ptr(ws, "workspace"), ws.numel() * ws.element_size(),
                                         _stream(stream), ctypes.byref(err)))
    return err.value


def exl3_decode_tile(trellis, k: int, n: int, K: int, codebook: int = EXL3_CB_MUL1, tk0: int = 0,
                     tk_cnt: int | None = None, tn0: int = 0, tn_cnt: int | None = None,
                     w_out=None, ld: int | None = None, stream=None) -> torch.Tensor:
    """Dequantised fp16 weights of a tile range (the whole tensor by default)."""
    tk_cnt = k // 16 - tk0 if tk_cnt is None else tk_cnt
    tn_cnt = n // 16 - tn0 if tn_cnt is None else tn_cnt
    if w_out is None:
        ld = 16 * tn_cnt if ld is None else ld
        w_out = torch.empty((16 * tk_cnt, ld), dtype=torch.float16, device=trellis.device)
    elif ld is None:
        ld = w_out.shape[-1]
    _check(lib().exl3_decode_tile(_ptr(trellis, "trellis", 2), k, n, K, codebook, tk0, tk_cnt, tn0, tn_cnt,
                                  _ptr(w_out, "w_out", 2), ld, _stream(stream)))
    return w_out


def exl3_input_rht(x, suh, out_dtype: int = EXL3_OUT_F32, out=None, stream=None) -> torch.Tensor:
    M, k = x.shape
    if out is None:
        out = torch.empty((M, k), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                          device=x.device)
    _check(lib().exl3_input_rht(_ptr(x, "x", 2), M, k, _ptr(suh, "suh", 2), _ptr(out, "out"), out_dtype,
                                _stream(stream)))
    return out


def exl3_linear_workspace_size(M: int, k: int, n: int, K: int) -> int:
    return lib().exl3_linear_workspace_size(M, k, n, K)


def exl3_linear(x, trellis, suh, svh, K: int, codebook: int = EXL3_CB_MUL1, out_dtype: int = EXL3_OUT_F16,
                y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """y = RHT_out(RHT_in(x . suh) @ W) . svh for x [M, k] fp16.  At M = 1, y may be
    a pinned host tensor: the kernels write the result straight into it."""
    M, k = x.shape
    n = trellis.shape[1] * 16
    if y is None:
        y = torch.empty((M, n), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    need = exl3_linear_workspace_size(M, k, n, K)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    yp = _ptr_pinned(y, "y") if (M == 1 and not y.is_cuda) else _ptr(y, "y")
    _check(lib().exl3_linear(_ptr(x, "x", 2), M, k, n, _ptr(trellis, "trellis", 2), _ptr(suh, "suh", 2),
                             _ptr(svh, "svh", 2), K, codebook, yp, out_dtype, _ptr(ws, "workspace"),
                             ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_linear_bias(x, trellis, suh, svh, bias, K: int, codebook: int = EXL3_CB_MUL1,
                     out_dtype: int = EXL3_OUT_F16, y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """y = RHT_out(RHT_in(x . suh) @ W) . svh + bias for x [M, k] fp16, bias [n] fp16."""
    M, k = x.shape
    n = trellis.shape[1] * 16
    if y is None:
        y = torch.empty((M, n), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    need = exl3_linear_workspace_size(M, k, n, K)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_linear_bias(_ptr(x, "x", 2), M, k, n, _ptr(trellis, "trellis", 2), _ptr(suh, "suh", 2),
                                  _ptr(svh, "svh", 2), _ptr(bias, "bias", 2), K, codebook, _ptr(y, "y"), out_dtype,
                                  _ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_linear_shards_workspace_size(M: int, k: int, n: int, K: int, nshards: int) -> int:
    return lib().exl3_linear_shards_workspace_size(M, k, n, K, nshards)


def exl3_linear_shards(x, trellis, suh, svh, K: int, codebook: int = EXL3_CB_MUL1, out_dtype: int = EXL3_OUT_F16,
                       y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """Fused shards over one input: trellis [S, k/16, n/16, 16K], suh [S, k], svh [S, n];
    returns y [S, M, n]."""
    M, k = x.shape
    S = trellis.shape[0]
    n = trellis.shape[2] * 16
    if y is None:
        y = torch.empty((S, M, n), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    need = exl3_linear_shards_workspace_size(M, k, n, K, S)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_linear_shards(_ptr(x, "x", 2), M, k, n, S, _ptr(trellis, "trellis", 2), _ptr(suh, "suh", 2),
                                    _ptr(svh, "svh", 2), K, codebook, _ptr(y, "y"), out_dtype, _ptr(ws, "workspace"),
                                    ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_linear_shards_var_workspace_size(M: int, k: int, widths, K: int) -> int:
    n = (ctypes.c_int * len(widths))(*[int(w) for w in widths])
    return lib().exl3_linear_shards_var_workspace_size(M, k, len(widths), n, K)


def exl3_linear_shards_var(x, trellis, suh, svh, widths, K: int, codebook: int = EXL3_CB_MUL1,
                           out_dtype: int = EXL3_OUT_F16, y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """Fused shards of different widths over one input: trellis flat (shard s's
    [k/16, n_s/16, 16K] tensor right after shard s-1's), suh [S, k], svh [sum n];
    returns y flat, shard-major (shard s an [M, n_s] block)."""
    M, k = x.shape
    S = len(widths)
    n = (ctypes.c_int * S)(*[int(w) for w in widths])
    total = M * sum(int(w) for w in widths)
    if y is None:
        y = torch.empty(total, dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16, device=x.device)
    need = lib().exl3_linear_shards_var_workspace_size(M, k, S, n, K)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_linear_shards_var(_ptr(x, "x", 2), M, k, S, n, _ptr(trellis, "trellis", 2), _ptr(suh, "suh", 2),
                                        _ptr(svh, "svh", 2), K, codebook, _ptr(y, "y"), out_dtype,
                                        _ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_set_row_invariant(enable: bool) -> bool:
    """Make each row of an exl3_linear result independent of the row count and
    of the other rows (same bits at every M); returns the previous setting."""
    return bool(lib().exl3_set_row_invariant(1 if enable else 0))


def exl3_set_weight_prefetch(enable: bool) -> bool:
    """Let M = 1 linears stream their weights while the kernel ahead of them
    on the stream finishes (CUDA programmatic dependent launch); returns the
    previous setting.  Weight buffers must not be written by kernels still in
    flight when a linear reading them is launched."""
    return bool(lib().exl3_set_weight_prefetch(1 if enable else 0))


def exl3_linear_int8_workspace_size(M: int, k: int, n: int, K: int) -> int:
    return lib().exl3_linear_int8_workspace_size(M, k, n, K)


WEIGHT_SCALE = 3.453125 / 127.0


def exl3_linear_int8(x, trellis, suh, svh, K: int, codebook: int = EXL3_CB_MUL1,
                     weight_scale: float = WEIGHT_SCALE, y=None, xq_out=None, row_scale_out=None,
                     acc_out=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """int8 prefill linear: y fp16 [M, n]; optional int8 q_x, fp32 row scales and
    int32 accumulators are written to the given tensors."""
    M, k = x.shape
    n = trellis.shape[1] * 16
    if y is None:
        y = torch.empty((M, n), dtype=torch.float16, device=x.device)
    need = exl3_linear_int8_workspace_size(M, k, n, K)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_linear_int8(_ptr(x, "x", 2), M, k, n, _ptr(trellis, "trellis", 2), _ptr(suh, "suh", 2),
                                  _ptr(svh, "svh", 2), K, codebook, weight_scale, _ptr(y, "y", 2),
                                  _ptr(xq_out, "xq_out", 1), _ptr(row_scale_out, "row_scale_out", 4),
                                  _ptr(acc_out, "acc_out", 4), _ptr(ws, "workspace"),
                                  ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_linear_int8_bias(x, trellis, suh, svh, bias, K: int, codebook: int = EXL3_CB_MUL1,
                          weight_scale: float = WEIGHT_SCALE, y=None, xq_out=None, row_scale_out=None,
                          acc_out=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """int8 prefill linear plus an output bias [n] fp16: y fp16 [M, n]."""
    M, k = x.shape
    n = trellis.shape[1] * 16
    if y is None:
        y = torch.empty((M, n), dtype=torch.float16, device=x.device)
    need = exl3_linear_int8_workspace_size(M, k, n, K)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_linear_int8_bias(_ptr(x, "x", 2), M, k, n, _ptr(trellis, "trellis", 2),
                                       _ptr(suh, "suh", 2), _ptr(svh, "svh", 2), _ptr(bias, "bias", 2), K,
                                       codebook, weight_scale, _ptr(y, "y", 2), _ptr(xq_out, "xq_out", 1),
                                       _ptr(row_scale_out, "row_scale_out", 4), _ptr(acc_out, "acc_out", 4),
                                       _ptr(ws, "workspace"), ws.numel() * ws.element_size(), _stream(stream)))
    return y


def expert_proj(trellis, suh, svh, K: int, codebook: int = EXL3_CB_MUL1) -> ExpertProj:
    """Descriptor of a projection arena: trellis [E, nslots, k/16, n/16, 16K], suh [E, nslots, k],
    svh [E, nslots, n] (CUDA tensors kept alive by the caller)."""
    E, nslots, tk, tn, _ = trellis.shape
    return ExpertProj(_ptr(trellis, "trellis", 2).value, _ptr(suh, "suh", 2).value, _ptr(svh, "svh", 2).value,
                      tk * 16, tn * 16, K, codebook, nslots)


def exl3_moe_workspace_size(T: int, topk: int, E: int, w13: ExpertProj, w2: ExpertProj) -> int:
    return lib().exl3_moe_workspace_size(T, topk, E, ctypes.byref(w13), ctypes.byref(w2))


def exl3_moe_grouped(x, topk_ids, topk_weights, w13: ExpertProj, w2: ExpertProj, E: int,
                     out_dtype: int = EXL3_OUT_F16, y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """Routed-expert contribution y [T, hidden] (gate+up, SiLU, down, weighted combine)."""
    T, hidden = x.shape
    topk = topk_ids.shape[1]
    if y is None:
        y = torch.empty((T, hidden), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    need = exl3_moe_workspace_size(T, topk, E, w13, w2)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_moe_grouped(_ptr(x, "x", 2), T, hidden, _ptr(topk_ids, "topk_ids", 4),
                                  _ptr(topk_weights, "topk_weights", 4), topk, E, ctypes.byref(w13),
                                  ctypes.byref(w2), _ptr(y, "y"), out_dtype, _ptr(ws, "workspace"),
                                  ws.numel() * ws.element_size(), _stream(stream)))
    return y


def expert_proj_mixed(trellis, suh, svh, K, k: int, n: int, codebook: int = EXL3_CB_MUL1) -> ExpertProjMixed:
    """Descriptor of a mixed-width projection arena: trellis flat (expert e's
    slots right after expert e-1's), suh [E, nslots, k], svh [E, nslots, n]
    (CUDA tensors kept alive by the caller), K the E widths (host)."""
    E, nslots, _ = suh.shape
    widths = (ctypes.c_int32 * E)(*[int(w) for w in K])
    d = ExpertProjMixed(_ptr(trellis, "trellis", 2).value, _ptr(suh, "suh", 2).value, _ptr(svh, "svh", 2).value,
                        ctypes.cast(widths, ctypes.POINTER(ctypes.c_int32)), k, n, codebook, nslots)
    d._widths = widths   # keep the host array alive with the descriptor
    return d


def exl3_moe_mixed_workspace_size(T: int, topk: int, E: int, w13: ExpertProjMixed, w2: ExpertProjMixed) -> int:
    return lib().exl3_moe_mixed_workspace_size(T, topk, E, ctypes.byref(w13), ctypes.byref(w2))


def exl3_moe_grouped_mixed(x, topk_ids, topk_weights, w13: ExpertProjMixed, w2: ExpertProjMixed, E: int,
                           out_dtype: int = EXL3_OUT_F16, y=None, workspace_buf=None, stream=None) -> torch.Tensor:
    """Routed-expert contribution y [T, hidden] with a width per expert."""
    T, hidden = x.shape
    topk = topk_ids.shape[1]
    if y is None:
        y = torch.empty((T, hidden), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    need = exl3_moe_mixed_workspace_size(T, topk, E, w13, w2)
    ws = workspace_buf if workspace_buf is not None else workspace(need, x.device, stream)
    _check(lib().exl3_moe_grouped_mixed(_ptr(x, "x", 2), T, hidden, _ptr(topk_ids, "topk_ids", 4),
                                        _ptr(topk_weights, "topk_weights", 4), topk, E, ctypes.byref(w13),
                                        ctypes.byref(w2), _ptr(y, "y"), out_dtype, _ptr(ws, "workspace"),
                                        ws.numel() * ws.element_size(), _stream(stream)))
    return y


def exl3_linear_gemv_noalloc(x, trellis, suh, svh, K: int, codebook: int = EXL3_CB_MUL1,
                             out_dtype: int = EXL3_OUT_F16, y=None, stream=None) -> torch.Tensor:
    """M = 1 linear without a caller workspace, for callers that may not allocate
    device memory: the library's fixed scratch array is used instead."""
    k = x.numel()
    n = trellis.shape[1] * 16
    if y is None:
        y = torch.empty((1, n), dtype=torch.float32 if out_dtype == EXL3_OUT_F32 else torch.float16,
                        device=x.device)
    _check(lib().exl3_linear_gemv_noalloc(_ptr(x, "x", 2), k, n, _ptr(trellis, "trellis", 2),
                                          _ptr(suh, "suh", 2), _ptr(svh, "svh", 2), K, codebook,
                                          _ptr(y, "y"), out_dtype, _stream(stream)))
    return y


def exl3_noalloc_device_error(stream=None) -> int:
    """Device error word of the fixed scratch array used by
    exl3_linear_gemv_noalloc on the current device (waits for the stream,
    then reads and clears it; 0 = no device-side check failed)."""
    v = ctypes.c_int(0)
    _check(lib().exl3_noalloc_device_error(_stream(stream), ctypes.byref(v)))
    return v.value

"""CPU oracle for the EXL3 trellis-quantized linear layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The CUDA library never imports, links or
falls back to anything in this package, and this package never imports the
CUDA library.  The arithmetic lives in ``exl3_oracle.c`` (scalar, float64,
integer-exact trellis and int8 work); this file only marshals numpy arrays.

Every function returns numpy arrays; fp16 tensors are passed and returned as
numpy float16 (their bits are what the C side reads).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exl3_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

MUL1_BOUND = 3.453125


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_f64.restype = ctypes.c_double
        lib.or_f64_to_f16.argtypes = [ctypes.c_double]
        lib.or_f64_to_f16.restype = ctypes.c_uint16
        lib.or_mul1_bytesum.argtypes = [ctypes.c_uint32]
        lib.or_mul1_bytesum.restype = ctypes.c_uint32
        lib.or_mul1_value.argtypes = [ctypes.c_uint32]
        lib.or_mul1_value.restype = ctypes.c_uint16
        lib.or_mul1_sigma.argtypes = []
        lib.or_mul1_sigma.restype = ctypes.c_double
        lib.or_tile_states.argtypes = [P, I, P]
        lib.or_tile_states.restype = None
        lib.or_reconstruct.argtypes = [P, I, I, I, P]
        lib.or_fwht128_f64.argtypes = [P]
        lib.or_fwht128_f64.restype = None
        lib.or_fwht128_f32.argtypes = [P]
        lib.or_fwht128_f32.restype = None
        lib.or_rht_in_f64.argtypes = [P, P, I, I, P]
        lib.or_rht_in_f32.argtypes = [P, P, I, I, P]
        lib.or_rht_out_f64.argtypes = [P, P, I, I]
        lib.or_linear.argtypes = [P, I, I, I, P, P, P, I, P]
        lib.or_linear_w.argtypes = [P, I, I, I, P, P, P, P]
        lib.or_add_bias.argtypes = [P, P, I, I]
        lib.or_quant_act.argtypes = [P, P, I, I, P, P]
        lib.or_quant_weight.argtypes = [ctypes.c_uint16]
        lib.or_quant_weight.restype = ctypes.c_int
        lib.or_int8_acc.argtypes = [P, P, I, I, I, P]
        lib.or_linear_int8.argtypes = [P, I, I, I, P, P, P, I, P, P, P, P, P]
        lib.or_moe.argtypes = [P, I, I, P, P, I, I, P, P, P, I, I, P, P, P, I, P, I, P]
        lib.or_moe_k.argtypes = [P, I, I, P, P, I, I, P, P, P, I, P, P, P, P, P, P, I, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    return a.astype(np.uint16, copy=False)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- scalars ---

def f16_to_f64(bits: int) -> float:
    return _load().or_f16_to_f64(bits)


def f64_to_f16(x: float) -> int:
    return _load().or_f64_to_f16(float(x))


def mul1_bytesum(state: int) -> int:
    return _load().or_mul1_bytesum(state)


def mul1_value_bits(state: int) -> int:
    return _load().or_mul1_value(state)


def mul1_sigma() -> float:
    return _load().or_mul1_sigma()


def codebook_table() -> np.ndarray:
    """fp16 value of every 16-bit state, float16 [65536]."""
    lib = _load()
    return np.array([lib.or_mul1_value(s) for s in range(65536)], dtype=np.uint16).view(np.float16)


def bytesum_table() -> np.ndarray:
    lib = _load()
    return np.array([lib.or_mul1_bytesum(s) for s in range(65536)], dtype=np.int64)


def quant_weight(vbits: int) -> int:
    return _load().or_quant_weight(vbits)


# ---------------------------------------------------------------- arrays ----

def tile_states(words, K: int) -> np.ndarray:
    w = _u16(words)
    assert w.size == 16 * K
    out = np.zeros(256, dtype=np.uint16)
    _load().or_tile_states(_ptr(w), K, _ptr(out))
    return out


def reconstruct(trellis, k: int, n: int, K: int) -> np.ndarray:
    """Dequantised Hadamard-domain weights, float16 [k, n]."""
    t = _u16(trellis)
    W = np.zeros((k, n), dtype=np.uint16)
    _check(_load().or_reconstruct(_ptr(t), k, n, K, _ptr(W)), "reconstruct")
    return W.view(np.float16)


def fwht128_f64(v) -> np.ndarray:
    a = np.array(v, dtype=np.float64).copy()
    assert a.shape == (128,)
    _load().or_fwht128_f64(_ptr(a))
    return a


def fwht128_f32(v) -> np.ndarray:
    a = np.array(v, dtype=np.float32).copy()
    assert a.shape == (128,)
    _load().or_fwht128_f32(_ptr(a))
    return a


def rht_in_f64(x, suh) -> np.ndarray:
    x = _u16(x)
    M, k = x.shape
    out = np.zeros((M, k), dtype=np.float64)
    _check(_load().or_rht_in_f64(_ptr(x), _ptr(_u16(suh)), M, k, _ptr(out)), "rht_in_f64")
    return out


def rht_in_f32(x, suh) -> np.ndarray:
    x = _u16(x)
    M, k = x.shape
    out = np.zeros((M, k), dtype=np.float32)
    _check(_load().or_rht_in_f32(_ptr(x), _ptr(_u16(suh)), M, k, _ptr(out)), "rht_in_f32")
    return out


def rht_out_f64(yp, svh) -> np.ndarray:
    y = np.array(yp, dtype=np.float64, order="C").copy()
    M, n = y.shape
    _check(_load().or_rht_out_f64(_ptr(y), _ptr(_u16(svh)), M, n), "rht_out_f64")
    return y


def add_bias(y, bias) -> np.ndarray:
    """y + bias (fp16 [n], one value per output feature) in float64, in place."""
    M, n = y.shape
    b = _u16(bias)
    if b.shape != (n,):
        raise ValueError(f"bias must have shape ({n},), got {b.shape}")
    _check(_load().or_add_bias(_ptr(y), _ptr(b), M, n), "add_bias")
    return y


def linear(x, trellis, suh, svh, K: int, bias=None) -> np.ndarray:
    """y [M, n] float64 = RHT_out(RHT_in(x . suh) @ W) . svh (+ bias)."""
    x = _u16(x)
    M, k = x.shape
    t = _u16(trellis)
    n = t.shape[1] * 16
    y = np.zeros((M, n), dtype=np.float64)
    _check(_load().or_linear(_ptr(x), M, k, n, _ptr(t), _ptr(_u16(suh)), _ptr(_u16(svh)), K,
                             _ptr(y)), "linear")
    return y if bias is None else add_bias(y, bias)


def linear_w(x, W, suh, svh, bias=None) -> np.ndarray:
    """Linear from dequantised fp16 weights W [k, n] (+ bias)."""
    x = _u16(x)
    M, k = x.shape
    Wb = _u16(W)
    n = Wb.shape[1]
    y = np.zeros((M, n), dtype=np.float64)
    _check(_load().or_linear_w(_ptr(x), M, k, n, _ptr(Wb), _ptr(_u16(suh)), _ptr(_u16(svh)),
                               _ptr(y)), "linear_w")
    return y if bias is None else add_bias(y, bias)


def quant_act(x, suh):
    """(q_x int8 [M,k], row_scale float32 [M]) of the int8 path."""
    x = _u16(x)
    M, k = x.shape
    q = np.zeros((M, k), dtype=np.int8)
    a = np.zeros(M, dtype=np.float32)
    _check(_load().or_quant_act(_ptr(x), _ptr(_u16(suh)), M, k, _ptr(q), _ptr(a)), "quant_act")
    return q, a


def quant_weights(W) -> np.ndarray:
    """q_w int8 of every fp16 weight of W (elementwise)."""
    lib = _load()
    Wb = _u16(W)
    uniq, inv = np.unique(Wb, return_inverse=True)
    q = np.array([lib.or_quant_weight(int(b)) for b in uniq], dtype=np.int64)
    if q.size and (q.min() < -127 or q.max() > 127):
        raise ValueError("weight outside the codebook range: |q_w| > 127")
    return q[inv].reshape(Wb.shape).astype(np.int8)


def int8_acc(qx, qw) -> np.ndarray:
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    qw = np.ascontiguousarray(qw, dtype=np.int8)
    M, k = qx.shape
    n = qw.shape[1]
    acc = np.zeros((M, n), dtype=np.int64)
    _check(_load().or_int8_acc(_ptr(qx), _ptr(qw), M, k, n, _ptr(acc)), "int8_acc")
    return acc


def linear_int8(x, trellis, suh, svh, K: int, bias=None):
    """Returns dict(qx, row_scale, qw, acc (int64), y (float64, + bias if given))."""
    x = _u16(x)
    M, k = x.shape
    t = _u16(trellis)
    n = t.shape[1] * 16
    qx = np.zeros((M, k), dtype=np.int8)
    a = np.zeros(M, dtype=np.float32)
    qw = np.zeros((k, n), dtype=np.int8)
    acc = np.zeros((M, n), dtype=np.int64)
    y = np.zeros((M, n), dtype=np.float64)
    _check(_load().or_linear_int8(_ptr(x), M, k, n, _ptr(t), _ptr(_u16(suh)), _ptr(_u16(svh)), K,
                                  _ptr(qx), _ptr(a), _ptr(qw), _ptr(acc), _ptr(y)), "linear_int8")
    if bias is not None:
        add_bias(y, bias)
    return dict(qx=qx, row_scale=a, qw=qw, acc=acc, y=y)


def moe(x, ids, weights, w13_trellis, w13_suh, w13_svh, K13, w2_trellis, w2_suh, w2_svh, K2,
        tokens=None) -> np.ndarray:
    """Routed-expert output float64 [len(tokens), hidden] for the listed tokens."""
    x = _u16(x)
    T, hidden = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    topk = ids.shape[1]
    t13 = _u16(w13_trellis)
    t2 = _u16(w2_trellis)
    E = t13.shape[0]
    inter = t13.shape[3] * 16
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.zeros((len(tok), hidden), dtype=np.float64)
    _check(_load().or_moe(_ptr(x), T, hidden, _ptr(ids), _ptr(weights), topk, E,
                          _ptr(t13), _ptr(_u16(w13_suh)), _ptr(_u16(w13_svh)), inter, K13,
                          _ptr(t2), _ptr(_u16(w2_suh)), _ptr(_u16(w2_svh)), K2,
                          _ptr(tok), len(tok), _ptr(y)), "moe")
    return y


def moe_k(x, ids, weights, w13_trellis, w13_suh, w13_svh, K13, w2_trellis, w2_suh, w2_svh, K2, inter: int,
          tokens=None) -> np.ndarray:
    """Routed-expert output with a width per expert (K13[e], K2[e]); the trellis
    arenas are flat, expert e packed right after expert e-1."""
    x = _u16(x)
    T, hidden = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    topk = ids.shape[1]
    k13 = np.ascontiguousarray(K13, dtype=np.int32)
    k2 = np.ascontiguousarray(K2, dtype=np.int32)
    E = len(k13)
    if len(k2) != E:
        raise ValueError("K13 and K2 must have one width per expert")
    t13 = _u16(w13_trellis).reshape(-1)
    t2 = _u16(w2_trellis).reshape(-1)
    need13 = int(sum(2 * (hidden // 16) * (inter // 16) * 16 * int(w) for w in k13))
    need2 = int(sum((inter // 16) * (hidden // 16) * 16 * int(w) for w in k2))
    if t13.size != need13 or t2.size != need2:
        raise ValueError(f"arena sizes {t13.size}/{t2.size} words, widths need {need13}/{need2}")
    tok = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.zeros((len(tok), hidden), dtype=np.float64)
    _check(_load().or_moe_k(_ptr(x), T, hidden, _ptr(ids), _ptr(weights), topk, E,
                            _ptr(t13), _ptr(_u16(w13_suh)), _ptr(_u16(w13_svh)), inter, _ptr(k13),
                            _ptr(t2), _ptr(_u16(w2_suh)), _ptr(_u16(w2_svh)), _ptr(k2),
                            _ptr(tok), len(tok), _ptr(y)), "moe_k")
    return y

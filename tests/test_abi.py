"""The C ABI library loads, exports every entry point of include/exl3.h, and
rejects bad arguments before launching anything (runs without a GPU).

Every call below carries at least one argument that validation rejects, so
no kernel is ever launched with the fake device addresses used here.
"""
import ctypes
import os
import re

import pytest

import trellis_quantized_gb300 as tq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
FAKE_MIS = ctypes.c_void_p(0x10002)   # misaligned


def header_functions():
    text = open(os.path.join(ROOT, "include", "exl3.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(exl3_[a-z0-9_]+)\s*\(", text)))


def test_library_builds_and_loads():
    L = tq.lib()
    assert os.path.exists(tq.lib_path())
    assert L.exl3_version() >= 100


def test_every_declared_symbol_is_exported():
    L = tq.lib()
    names = header_functions()
    assert "exl3_linear" in names and "exl3_moe_grouped" in names and "exl3_decode_tile" in names
    for name in names:
        assert hasattr(L, name), f"{name} declared in exl3.h but not exported"


def _err(L):
    return L.exl3_last_error().decode()


def test_every_declared_symbol_has_a_binding_of_the_same_name():
    """The Python layer wraps every C entry point under its own name (the
    error message is read by the wrappers themselves)."""
    missing = [n for n in header_functions() if n != "exl3_last_error" and not hasattr(tq, n)]
    assert not missing, missing


def test_decode_tile_argument_errors():
    L = tq.lib()
    assert L.exl3_decode_tile(None, 128, 128, 4, 2, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_ARG
    assert "trellis" in _err(L)
    assert L.exl3_decode_tile(FAKE_MIS, 128, 128, 4, 2, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_ARG
    assert L.exl3_decode_tile(FAKE, 128, 128, 9, 2, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_BITS
    assert L.exl3_decode_tile(FAKE, 128, 128, 0, 2, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_BITS
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 1, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_CODEBOOK
    assert "refusing" in _err(L)
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 3, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_CODEBOOK
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 7, 0, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_CODEBOOK
    assert L.exl3_decode_tile(FAKE, 120, 128, 4, 2, 0, 7, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_SHAPE
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 2, 4, 8, 0, 8, FAKE, 128, None) == tq.EXL3_ERR_SHAPE
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 2, 0, 8, 0, 8, FAKE, 100, None) == tq.EXL3_ERR_SHAPE
    assert L.exl3_decode_tile(FAKE, 128, 128, 4, 2, 0, 8, 0, 8, FAKE, 132, None) == tq.EXL3_ERR_SHAPE


def test_linear_argument_errors():
    L = tq.lib()
    ws = 1 << 20
    args = lambda **kw: [kw.get("x", FAKE), kw.get("M", 1), kw.get("k", 256), kw.get("n", 256),
                         kw.get("t", FAKE), kw.get("suh", FAKE), kw.get("svh", FAKE), kw.get("K", 4),
                         kw.get("cb", 2), kw.get("y", FAKE), kw.get("od", 0), kw.get("ws", FAKE),
                         kw.get("wsb", ws), None]
    assert L.exl3_linear(*args(x=None)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear(*args(svh=FAKE_MIS)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear(*args(K=9)) == tq.EXL3_ERR_BITS
    assert L.exl3_linear(*args(cb=1)) == tq.EXL3_ERR_CODEBOOK
    assert L.exl3_linear(*args(M=0)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear(*args(k=200)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear(*args(n=64)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear(*args(od=5)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear(*args(ws=None)) == tq.EXL3_ERR_WORKSPACE
    assert L.exl3_linear(*args(wsb=16)) == tq.EXL3_ERR_WORKSPACE
    assert "workspace" in _err(L)


def test_linear_bias_argument_errors():
    """The bias entry points check the bias pointer (required, 16-byte aligned)
    and otherwise share exl3_linear's checks; nothing is launched."""
    L = tq.lib()
    ws = 1 << 20
    args = lambda **kw: [kw.get("x", FAKE), kw.get("M", 1), kw.get("k", 256), kw.get("n", 256),
                         kw.get("t", FAKE), kw.get("suh", FAKE), kw.get("svh", FAKE), kw.get("b", FAKE),
                         kw.get("K", 4), kw.get("cb", 2), kw.get("y", FAKE), kw.get("od", 0), kw.get("ws", FAKE),
                         kw.get("wsb", ws), None]
    assert L.exl3_linear_bias(*args(b=None)) == tq.EXL3_ERR_ARG
    assert "bias" in _err(L)
    assert L.exl3_linear_bias(*args(b=FAKE_MIS)) == tq.EXL3_ERR_ARG
    assert "bias" in _err(L)
    assert L.exl3_linear_bias(*args(K=0)) == tq.EXL3_ERR_BITS
    assert L.exl3_linear_bias(*args(n=200)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_bias(*args(wsb=16)) == tq.EXL3_ERR_WORKSPACE
    i8 = lambda **kw: [FAKE, 4, 256, 256, FAKE, FAKE, FAKE, kw.get("b", FAKE), kw.get("K", 4), 2,
                       kw.get("sw", 3.453125 / 127), FAKE, None, None, None, FAKE, ws, None]
    assert L.exl3_linear_int8_bias(*i8(b=None)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_int8_bias(*i8(b=FAKE_MIS)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_int8_bias(*i8(sw=-1.0)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_int8_bias(*i8(K=9)) == tq.EXL3_ERR_BITS


def test_moe_mixed_argument_errors():
    """Per-expert widths are checked on the host before anything is launched."""
    L = tq.lib()
    E = 4
    Pi = ctypes.POINTER(ctypes.c_int32)
    K13 = (ctypes.c_int32 * E)(3, 3, 4, 4)
    K2 = (ctypes.c_int32 * E)(2, 2, 2, 9)        # expert 3: width 9
    w13 = tq.ExpertProjMixed(FAKE.value, FAKE.value, FAKE.value, ctypes.cast(K13, Pi), 256, 128, 2, 2)
    w2 = tq.ExpertProjMixed(FAKE.value, FAKE.value, FAKE.value, ctypes.cast(K2, Pi), 128, 256, 2, 1)
    call = lambda wsb=1 << 26: L.exl3_moe_grouped_mixed(FAKE, 3, 256, FAKE, FAKE, 2, E, ctypes.byref(w13),
                                                       ctypes.byref(w2), FAKE, 0, FAKE, wsb, None)
    assert call() == tq.EXL3_ERR_BITS and "w2.K[3]" in _err(L)
    K2[3] = 2
    need = L.exl3_moe_mixed_workspace_size(3, 2, E, ctypes.byref(w13), ctypes.byref(w2))
    assert need > 0
    assert call(wsb=need - 1) == tq.EXL3_ERR_WORKSPACE
    w13.codebook = 1
    assert call() == tq.EXL3_ERR_CODEBOOK
    w13.codebook = 2
    w13.nslots = 1
    assert call() == tq.EXL3_ERR_SHAPE
    w13.nslots = 2
    w13.K = None
    assert call() == tq.EXL3_ERR_ARG
    w13.K = ctypes.cast(K13, Pi)
    w2.trellis = FAKE_MIS.value
    assert call() == tq.EXL3_ERR_ARG


def test_linear_shards_argument_errors():
    L = tq.lib()
    args = lambda **kw: [FAKE, kw.get("M", 1), 256, kw.get("n", 256), kw.get("S", 2), FAKE, FAKE,
                         kw.get("svh", FAKE), kw.get("K", 4), kw.get("cb", 2), FAKE, kw.get("od", 0), FAKE,
                         kw.get("wsb", 1 << 24), None]
    assert L.exl3_linear_shards(*args(S=0)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_shards(*args(S=65)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_shards(*args(n=100)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_shards(*args(K=0)) == tq.EXL3_ERR_BITS
    assert L.exl3_linear_shards(*args(cb=3)) == tq.EXL3_ERR_CODEBOOK
    assert L.exl3_linear_shards(*args(od=2)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_shards(*args(svh=FAKE_MIS)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_shards(*args(wsb=64)) == tq.EXL3_ERR_WORKSPACE
    # the workspace covers one shard's exl3_linear at every M
    for M in (1, 7, 300):
        assert L.exl3_linear_shards_workspace_size(M, 5120, 17408, 4, 2) >= L.exl3_linear_workspace_size(
            M, 5120, 17408, 4)
    assert L.exl3_linear_shards_workspace_size(1, 5120, 17408, 4, 0) == 0


def test_linear_shards_var_argument_errors():
    L = tq.lib()
    n = (ctypes.c_int * 3)(5120, 1024, 1024)
    bad = (ctypes.c_int * 3)(5120, 1000, 1024)
    args = lambda **kw: [FAKE, 1, 5120, kw.get("S", 3), kw.get("n", n), FAKE, FAKE, FAKE, kw.get("K", 4), 2, FAKE,
                         0, FAKE, kw.get("wsb", 1 << 26), None]
    assert L.exl3_linear_shards_var(*args(n=None)) == tq.EXL3_ERR_ARG
    assert L.exl3_linear_shards_var(*args(n=bad)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_shards_var(*args(S=0)) == tq.EXL3_ERR_SHAPE
    assert L.exl3_linear_shards_var(*args(K=9)) == tq.EXL3_ERR_BITS
    assert L.exl3_linear_shards_var(*args(wsb=64)) == tq.EXL3_ERR_WORKSPACE
    assert L.exl3_linear_shards_var_workspace_size(1, 5120, 3, n, 4) >= L.exl3_linear_workspace_size(1, 5120, 5120, 4)
    assert L.exl3_linear_shards_var_workspace_size(1, 5120, 3, None, 4) == 0


def test_input_rht_argument_errors():
    L = tq.lib()
    assert L.exl3_input_rht(FAKE, 1, 100, FAKE, FAKE, 1, None) == tq.EXL3_ERR_SHAPE
    assert L.exl3_input_rht(FAKE, 0, 128, FAKE, FAKE, 1, None) == tq.EXL3_ERR_SHAPE
    assert L.exl3_input_rht(FAKE, 1, 128, None, FAKE, 1, None) == tq.EXL3_ERR_ARG
    assert L.exl3_input_rht(FAKE, 1, 128, FAKE, FAKE, 3, None) == tq.EXL3_ERR_ARG


def test_copy_in_argument_errors():
    """NULL or misaligned pointers are rejected; zero bytes enqueue nothing."""
    L = tq.lib()
    assert L.exl3_copy_in(None, FAKE, 64, None) == tq.EXL3_ERR_ARG
    assert "src" in _err(L)
    assert L.exl3_copy_in(FAKE, None, 64, None) == tq.EXL3_ERR_ARG
    assert L.exl3_copy_in(FAKE_MIS, FAKE, 64, None) == tq.EXL3_ERR_ARG
    assert L.exl3_copy_in(FAKE, FAKE_MIS, 64, None) == tq.EXL3_ERR_ARG
    assert L.exl3_copy_in(FAKE, FAKE, 0, None) == tq.EXL3_OK


@pytest.mark.parametrize("M,k,n,K", [(1, 5120, 17408, 4), (4, 5120, 5120, 4), (4096, 5120, 17408, 4),
                                     (1, 128, 128, 1), (64, 4096, 4096, 7)])
def test_workspace_sizes(M, k, n, K):
    size = tq.exl3_linear_workspace_size(M, k, n, K)
    assert size >= 256 and size % 256 == 0
    assert tq.exl3_linear_workspace_size(M, k + 1, n, K) == 0
    assert tq.exl3_linear_workspace_size(M, k, n, 0) == 0


def test_host_settings_round_trip():
    """The row-invariant and weight-prefetch switches return the previous
    setting, and the workspace size does not depend on the row-invariant one
    (it covers both layouts)."""
    sizes = {}
    for inv in (False, True):
        prev = tq.exl3_set_row_invariant(inv)
        assert tq.exl3_set_row_invariant(inv) == inv
        sizes[inv] = [tq.exl3_linear_workspace_size(M, 5120, 512, 4) for M in (1, 16, 300)]
        tq.exl3_set_row_invariant(prev)
    assert sizes[False] == sizes[True]
    prev = tq.exl3_set_weight_prefetch(True)
    assert tq.exl3_set_weight_prefetch(prev) is True

"""The allocation-free M = 1 entry point (exl3_linear_gemv_noalloc).

Callers such as plugin hosts that own the device memory pool, or decode
loops that reserve all memory up front, cannot call cudaMalloc; this entry
point takes no workspace and keeps its scratch in a fixed array inside the
library.  The tests call it through the C ABI twice in a row, with different
shapes so the shared scratch is reused, and compare each result with the
float64 oracle and with the workspace-taking exl3_linear under the tolerance
of the other parity tests; after each call the scratch array's device error
word must read zero.  A further test checks the defining property: once the
first call has loaded the kernels and looked up the array, more calls leave
the device's free memory unchanged.  This file sorts last so a run that stops
at the first failure has already run every other test; it also passes on its
own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _noalloc_raw(x, t, suh, svh, K, y, out_dtype):
    """Direct ctypes call of the C entry point with raw device pointers."""
    L = tq.lib()
    k, n = x.numel(), t.shape[1] * 16
    rc = L.exl3_linear_gemv_noalloc(ctypes.c_void_p(x.data_ptr()), k, n, ctypes.c_void_p(t.data_ptr()),
                                    ctypes.c_void_p(suh.data_ptr()), ctypes.c_void_p(svh.data_ptr()), K,
                                    tq.EXL3_CB_MUL1, ctypes.c_void_p(y.data_ptr()), out_dtype,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == tq.EXL3_OK, L.exl3_last_error().decode()


def _device_error_raw():
    """The scratch array's error word through the C ABI (reads and clears it)."""
    L = tq.lib()
    v = ctypes.c_int(-1)
    rc = L.exl3_noalloc_device_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(v))
    assert rc == tq.EXL3_OK, L.exl3_last_error().decode()
    return v.value


@pytest.mark.parametrize("out_dtype", [tq.EXL3_OUT_F16, tq.EXL3_OUT_F32])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(out_dtype):
    cases = [synth.config2(17408, 1), synth.config3(3, 1)]     # two calls in a row, two shapes
    for case in cases:
        x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
        ref = tq.exl3_linear(x, t, suh, svh, case.K, out_dtype=out_dtype)
        dt = torch.float32 if out_dtype == tq.EXL3_OUT_F32 else torch.float16
        y = torch.empty((1, case.n), dtype=dt, device="cuda")
        _noalloc_raw(x, t, suh, svh, case.K, y, out_dtype)
        assert _device_error_raw() == 0, case.name + ": device error word set"
        got = host(y).astype(np.float64)
        assert_close(got, oracle.linear(case.x, case.trellis, case.suh, case.svh, case.K), case.name + " vs oracle")
        assert_close(got, host(ref).astype(np.float64), case.name + " vs exl3_linear")


def test_noalloc_allocates_no_device_memory():
    """After a first call (kernel loading, scratch address lookup), ten more
    calls of both output types leave cudaMemGetInfo's free bytes unchanged."""
    case = synth.config3(5, 1)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    y16 = torch.empty((1, case.n), dtype=torch.float16, device="cuda")
    y32 = torch.empty((1, case.n), dtype=torch.float32, device="cuda")
    _noalloc_raw(x, t, suh, svh, case.K, y16, tq.EXL3_OUT_F16)
    _noalloc_raw(x, t, suh, svh, case.K, y32, tq.EXL3_OUT_F32)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for i in range(10):
        _noalloc_raw(x, t, suh, svh, case.K, y16 if i % 2 else y32, tq.EXL3_OUT_F16 if i % 2 else tq.EXL3_OUT_F32)
    assert _device_error_raw() == 0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch():
    """n = 2^20 columns (8192 column blocks of 128) needs more partial-sum slots
    than the 2 MiB array holds, so the call is rejected before any launch.  The
    buffers have their full sizes all the same (K = 1 keeps the trellis at 16 MiB)."""
    k, n, K = 128, 1 << 20, 1
    x = torch.zeros(k, dtype=torch.float16, device="cuda")
    t = torch.zeros((k // 16, n // 16, 16 * K), dtype=torch.int16, device="cuda")
    suh = torch.ones(k, dtype=torch.float16, device="cuda")
    svh = torch.ones(n, dtype=torch.float16, device="cuda")
    with pytest.raises(tq.Exl3Error) as e:
        tq.exl3_linear_gemv_noalloc(x, t, suh, svh, K)
    assert e.value.code == tq.EXL3_ERR_SHAPE
    assert "fixed scratch" in str(e.value)

"""The allocation-free M = 1 entry point (exl3_linear_gemv_noalloc).

Callers such as plugin hosts that own the device memory pool, or decode
loops that reserve all memory up front, cannot call cudaMalloc; this entry
point takes no workspace and keeps its scratch in a fixed array inside the
library.  The test calls it through the C ABI twice in a row, with different
shapes so the shared scratch is reused, and compares each result with the
workspace-taking exl3_linear under the tolerance of the other parity tests.
This file sorts last so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import exl3_synth as synth
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


@pytest.mark.parametrize("out_dtype", [tq.EXL3_OUT_F16, tq.EXL3_OUT_F32])
def test_noalloc_matches_workspace_entry_point_twice(out_dtype):
    cases = [synth.config2(17408, 1), synth.config3(3, 1)]     # two calls in a row, two shapes
    for case in cases:
        x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
        ref = tq.exl3_linear(x, t, suh, svh, case.K, out_dtype=out_dtype)
        dt = torch.float32 if out_dtype == tq.EXL3_OUT_F32 else torch.float16
        y = torch.empty((1, case.n), dtype=dt, device="cuda")
        _noalloc_raw(x, t, suh, svh, case.K, y, out_dtype)
        torch.cuda.synchronize()
        assert_close(host(y).astype(np.float64), host(ref).astype(np.float64), case.name + " noalloc")


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

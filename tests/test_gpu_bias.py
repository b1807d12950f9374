"""GPU parity of the linear with an output bias (exl3_linear_bias,
exl3_linear_int8_bias) against the CPU oracle, on every path of the linear.

A checkpoint's EXL3 group holds a bias beside trellis, suh and svh ("EXL3
checkpoints on the native engine (tracker) #832", "What is left").  The
library adds it per output feature after svh, in fp32, before the output is
rounded.  Checks:
  * fp16 and fp32 outputs meet the output tolerance of tests/gpu_util.py
    against the float64 oracle with the same bias;
  * the fp32 output is exactly fp32(y + bias), y the fp32 output of
    exl3_linear on the same inputs (one rounded add, nothing else changes);
  * int8: q_x, row scales and int32 accumulators are unchanged by the bias
    and y meets the tolerance against the oracle's int8 result plus bias.
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu

# (M, k, n, K): M = 1 takes the CUDA-core GEMV (one and several CTAs per
# column block, 128- and 256-column blocks), 2..128 the fused small-M kernel,
# above 128 the reconstruct + GEMM (256-column tiles when n % 256 == 0, else
# 128); n = 640 leaves a ragged last block or tile.
PATHS = [(1, 2048, 1024, 4), (1, 1152, 640, 3), (16, 2048, 1024, 4), (3, 1152, 640, 5),
         (200, 2048, 1024, 4), (129, 1152, 640, 2)]


def _inputs(sub, M, k, n, K):
    case = synth.linear_case(18, sub, M, k, n, K, outlier_rows=0.1)
    return case, synth.bias_for(sub, n)


@pytest.mark.parametrize("M,k,n,K", PATHS)
def test_bias_matches_oracle(M, k, n, K):
    case, b = _inputs(M * 10 + K, M, k, n, K)
    ref = oracle.linear(case.x, case.trellis, case.suh, case.svh, K, bias=b)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = tq.exl3_linear_bias(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), dev(b), K,
                                out_dtype=od)
        assert_close(host(y).astype(np.float64), ref, f"M={M} k={k} n={n} K={K} out={'f32' if od else 'f16'}")


@pytest.mark.parametrize("M,k,n,K", PATHS)
def test_bias_is_one_rounded_add_after_the_output(M, k, n, K):
    case, b = _inputs(M * 10 + K + 5, M, k, n, K)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    y0 = host(tq.exl3_linear(x, t, suh, svh, K, out_dtype=tq.EXL3_OUT_F32))
    yb = host(tq.exl3_linear_bias(x, t, suh, svh, dev(b), K, out_dtype=tq.EXL3_OUT_F32))
    expect = y0 + b.astype(np.float32)[None, :]      # float32 + float32 in numpy: one IEEE rounding
    assert np.array_equal(yb.view(np.uint32), expect.view(np.uint32))


def test_bias_row_invariant_mode():
    """Row-invariant mode adds the bias in the same epilogue: rows alone and
    inside a larger call agree bit for bit, and match the oracle."""
    M, k, n, K = 40, 1024, 768, 4
    case, b = _inputs(400, M, k, n, K)
    x, t, suh, svh, bd = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), dev(b)
    prev = tq.exl3_set_row_invariant(True)
    try:
        full = host(tq.exl3_linear_bias(x, t, suh, svh, bd, K))
        for m in (0, 17, 39):
            one = host(tq.exl3_linear_bias(x[m:m + 1].contiguous(), t, suh, svh, bd, K))
            assert np.array_equal(one.view(np.uint16), full[m:m + 1].view(np.uint16))
    finally:
        tq.exl3_set_row_invariant(prev)
    ref = oracle.linear(case.x, case.trellis, case.suh, case.svh, K, bias=b)
    assert_close(full.astype(np.float64), ref, "row-invariant with bias")


def test_bias_prefill_config4_sampled_rows():
    """The prefill shape (M = 4096, k = 5120, n = 17408) with a bias; the
    oracle evaluates a seeded sample of rows."""
    case = synth.config4()
    b = synth.bias_for(4, case.n)
    rng = np.random.default_rng(41)
    rows = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 8, replace=False)]))
    W = oracle.reconstruct(case.trellis, case.k, case.n, case.K)
    ref = oracle.linear_w(case.x[rows], W, case.suh, case.svh, bias=b)
    y = tq.exl3_linear_bias(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), dev(b), case.K)
    assert_close(host(y)[rows].astype(np.float64), ref, "config 4 with bias")


@pytest.mark.parametrize("M,K", [(37, 3), (1, 7)])
def test_int8_bias(M, K):
    k, n = 640, 384
    case, b = _inputs(500 + M + K, M, k, n, K)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    outs = []
    for bias in (None, dev(b)):
        xq = torch.empty((M, k), dtype=torch.int8, device="cuda")
        rs = torch.empty(M, dtype=torch.float32, device="cuda")
        acc = torch.empty((M, n), dtype=torch.int32, device="cuda")
        if bias is None:
            y = tq.exl3_linear_int8(x, t, suh, svh, K, xq_out=xq, row_scale_out=rs, acc_out=acc)
        else:
            y = tq.exl3_linear_int8_bias(x, t, suh, svh, bias, K, xq_out=xq, row_scale_out=rs, acc_out=acc)
        outs.append((host(xq), host(rs), host(acc), host(y).astype(np.float64)))
    (q0, r0, a0, _), (q1, r1, a1, y1) = outs
    assert np.array_equal(q0, q1) and np.array_equal(r0.view(np.uint32), r1.view(np.uint32))
    assert np.array_equal(a0, a1)
    ref = oracle.linear_int8(case.x, case.trellis, case.suh, case.svh, K, bias=b)
    assert np.array_equal(a1.astype(np.int64), ref["acc"])
    assert_close(y1, ref["y"], f"int8 M={M} K={K} with bias")

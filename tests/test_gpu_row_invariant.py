"""Row-invariant mode of exl3_linear ("EXL3 checkpoints on the native engine
(tracker) #832": a row-invariant linear; "The gate": rows keep one
arithmetic at every row count).

With the mode on, a row's output has the same bits whatever M is and
whichever rows share the call, and still meets the oracle's tolerance.  The
int8 linear is row-invariant in either mode (per-row activation scales and
exact integer accumulation).
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture
def row_invariant():
    prev = tq.exl3_set_row_invariant(True)
    try:
        yield
    finally:
        tq.exl3_set_row_invariant(prev)


def _lin(x, d, K, od):
    return tq.exl3_linear(x, d["t"], d["suh"], d["svh"], K, out_dtype=od)


# (k, n, K): one split per column tile; k split over CTAs (few column tiles);
# an odd width with a k that is not a multiple of 256
SHAPES = [(1024, 768, 4), (5120, 512, 3), (1152, 384, 7)]


@pytest.mark.parametrize("k,n,K", SHAPES)
def test_rows_equal_at_every_row_count(row_invariant, k, n, K):
    case = synth.linear_case(70, k + K, 300, k, n, K, outlier_rows=0.05)
    d = dict(t=dev(case.trellis), suh=dev(case.suh), svh=dev(case.svh))
    x = dev(case.x)
    rows = [0, 1, 16, 31, 32, 33, 127, 128, 129, 255, 299]
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        solo = {m: _lin(x[m:m + 1], d, K, od)[0].clone() for m in rows}
        # row counts around the 32-row chunk boundaries and the small-M /
        # prefill switch of the default mode, and
        # windows that put a row among different neighbours
        for a, b in [(0, 2), (0, 17), (0, 32), (0, 33), (0, 129), (0, 300), (1, 130), (30, 70), (120, 260),
                     (255, 300)]:
            y = _lin(x[a:b], d, K, od)
            for m in rows:
                if a <= m < b:
                    assert torch.equal(y[m - a], solo[m]), f"row {m} differs in rows [{a}, {b}) out={od}"


@pytest.mark.parametrize("k,n,K", SHAPES)
def test_row_invariant_matches_oracle(row_invariant, k, n, K):
    case = synth.linear_case(71, k + K, 131, k, n, K, outlier_rows=0.05)
    d = dict(t=dev(case.trellis), suh=dev(case.suh), svh=dev(case.svh))
    ref = oracle.linear(case.x, case.trellis, case.suh, case.svh, K)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = host(_lin(dev(case.x), d, K, od)).astype(np.float64)
        assert_close(y, ref, f"row-invariant k{k} n{n} K{K} out={od}")


def test_workspace_query_covers_both_modes():
    """The size is queried with the mode off and used with it on (and the
    other way round): both layouts fit."""
    case = synth.linear_case(72, 0, 1, 5120, 512, 4)
    need = tq.exl3_linear_workspace_size(1, case.k, case.n, case.K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    args = (dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), 4)
    y_plain = tq.exl3_linear(*args, workspace_buf=ws).clone()
    prev = tq.exl3_set_row_invariant(True)
    try:
        y_inv = tq.exl3_linear(*args, workspace_buf=ws).clone()
    finally:
        tq.exl3_set_row_invariant(prev)
    assert tq.exl3_check_device_error(ws) == 0
    counters = host(ws[256:256 + 4 * (case.n // 128)]).view(np.int32)
    assert np.all(counters == 0)
    ref = oracle.linear(case.x, case.trellis, case.suh, case.svh, 4)
    assert_close(host(y_plain).astype(np.float64), ref, "plain M=1")
    assert_close(host(y_inv).astype(np.float64), ref, "row-invariant M=1")


def test_int8_rows_equal_at_every_row_count():
    case = synth.linear_case(73, 0, 200, 1024, 512, 4, outlier_rows=0.05)
    t, suh, svh, x = dev(case.trellis), dev(case.suh), dev(case.svh), dev(case.x)
    solo = {m: tq.exl3_linear_int8(x[m:m + 1], t, suh, svh, 4)[0].clone() for m in (0, 5, 130, 199)}
    for a, b in [(0, 200), (0, 131), (5, 6), (100, 200)]:
        y = tq.exl3_linear_int8(x[a:b], t, suh, svh, 4)
        for m, ys in solo.items():
            if a <= m < b:
                assert torch.equal(y[m - a], ys), f"int8 row {m} differs in rows [{a}, {b})"

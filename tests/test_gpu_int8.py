"""GPU parity of the int8 prefill variant ("exl3xpu" README, "Prefill: int8
linears and oneDNN fused attention") against the CPU oracle.

q_x, the per-row activation scales and the int32 accumulators must be
bit-exact; y (fp16) must meet the output tolerance against the float64
evaluation of the same int8 scheme.
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host
from tie_rows import tie_rows

pytestmark = pytest.mark.gpu


def _run_int8(case, rows=None):
    M, k, n = case.M, case.k, case.n
    xq = torch.empty((M, k), dtype=torch.int8, device="cuda")
    rs = torch.empty(M, dtype=torch.float32, device="cuda")
    acc = torch.empty((M, n), dtype=torch.int32, device="cuda")
    y = tq.exl3_linear_int8(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), case.K,
                            xq_out=xq, row_scale_out=rs, acc_out=acc)
    out = dict(qx=host(xq), row_scale=host(rs), acc=host(acc), y=host(y).astype(np.float64))
    if rows is not None:
        out = {key: v[rows] for key, v in out.items()}
    return out


def _check(case, rows=None):
    x = case.x if rows is None else case.x[rows]
    ref = oracle.linear_int8(x, case.trellis, case.suh, case.svh, case.K)
    got = _run_int8(case, rows)
    assert np.array_equal(got["qx"], ref["qx"]), "q_x differs"
    assert np.array_equal(got["row_scale"].view(np.uint32), ref["row_scale"].view(np.uint32)), "row scales differ"
    assert np.array_equal(got["acc"].astype(np.int64), ref["acc"]), "int32 accumulators differ"
    assert_close(got["y"], ref["y"], case.name + " int8")


@pytest.mark.parametrize("K", [1, 3, 4, 8])
def test_int8_small_all_widths(K):
    _check(synth.linear_case(20, K, 37, 640, 384, K, outlier_rows=0.1))


@pytest.mark.parametrize("M", synth.CONFIG3_M)
@pytest.mark.parametrize("K", synth.CONFIG3_K)
def test_int8_config3_all_widths_and_rows(K, M):
    """Every (K, M) pair of the mixed-width layer through the int8 variant:
    q_x, row scales and accumulators bit-exact on every row."""
    _check(synth.config3(K, M))


def test_int8_activation_codes_at_exact_ties():
    """127 activations sit exactly halfway between two codes of the
    definition, where only the fp32 rounding of x' * fp32(127 / amax) decides
    the code: q_x, the row scales and the accumulators must still be
    bit-exact."""
    x, suh, _ = tie_rows()
    case = synth.linear_case(22, 0, x.shape[0], 128, 256, 4)
    case.x, case.suh = x, suh
    _check(case)


def test_int8_config4_sampled_rows():
    case = synth.config4()
    rng = np.random.default_rng(40)
    rows = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 10, replace=False)]))
    _check(case, rows)


def test_int8_extreme_accumulators_are_exact():
    """Every q_x = 127 and every q_w = -127: |acc| = 16129 k exceeds 2^24, so
    an fp32 accumulation over the whole of k would round; the chunked
    accumulation must still be exact.  x = suh at the first element of each
    128-block (0 elsewhere) makes every x' equal 2^-3.5; an all-zero trellis
    makes every weight -3.453125."""
    k, n, M, K = 5120, 256, 3, 2
    case = synth.linear_case(21, 0, M, k, n, K)
    x = np.zeros((M, k), dtype=np.float16)
    x[:, 0::128] = case.suh[0::128]
    case.x = x
    case.trellis = np.zeros_like(case.trellis)
    got = _run_int8(case)
    assert np.all(got["qx"] == 127)
    assert np.all(got["acc"] == -16129 * k)
    _check(case)


def test_int8_zero_rows():
    case = synth.linear_case(22, 0, 5, 512, 256, 4)
    case.x[1] = 0
    case.x[4] = 0
    got = _run_int8(case)
    assert got["row_scale"][1] == 0 and np.all(got["qx"][1] == 0) and np.all(got["acc"][1] == 0)
    _check(case)


def test_int8_rejects_bad_weight_scale():
    case = synth.linear_case(23, 0, 2, 256, 256, 4)
    with pytest.raises(tq.Exl3Error) as e:
        tq.exl3_linear_int8(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), 4, weight_scale=0.0)
    assert e.value.code == tq.EXL3_ERR_ARG


def test_int8_distance_to_fp_path_is_quantisation_sized():
    """For information: the int8 output differs from the fp output by about
    1% (the pages quote +0.17% NLL for the same scheme)."""
    case = synth.config3(4, 64)
    y8 = _run_int8(case)["y"]
    yf = host(tq.exl3_linear(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), 4)).astype(np.float64)
    rel = np.linalg.norm(y8 - yf) / np.linalg.norm(yf)
    assert 1e-4 < rel < 5e-2

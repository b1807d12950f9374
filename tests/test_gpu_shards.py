"""GPU parity of fused shards (exl3_linear_shards): several linears of one
input, each with its own trellis, suh and svh ("exl3xpu" README, "Layout":
fused shards in the vLLM linear method), against the CPU oracle of each
shard.

At M = 1 the shards run in one launch of the GEMV's grouped mode; above, one
linear per shard.  Outputs must meet the tolerance of tests/gpu_util.py; the
per-shard path must give exl3_linear's bits.
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _shards(sub, S, M, k, n, K):
    cases = [synth.linear_case(19, sub * 10 + s, M, k, n, K) for s in range(S)]
    x = cases[0].x                                   # one input for every shard
    t = np.stack([c.trellis for c in cases])
    suh = np.stack([c.suh for c in cases])
    svh = np.stack([c.svh for c in cases])
    return x, t, suh, svh


@pytest.mark.parametrize("S,M,k,n,K", [(2, 1, 2048, 1024, 4), (3, 1, 1152, 640, 3), (2, 1, 5120, 17408, 4),
                                       (4, 1, 256, 384, 8), (3, 7, 1024, 768, 4), (2, 200, 1024, 512, 2)])
def test_shards_match_oracle(S, M, k, n, K):
    x, t, suh, svh = _shards(S * 100 + M, S, M, k, n, K)
    refs = [oracle.linear(x, t[s], suh[s], svh[s], K) for s in range(S)]
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = host(tq.exl3_linear_shards(dev(x), dev(t), dev(suh), dev(svh), K, out_dtype=od))
        assert y.shape == (S, M, n)
        for s in range(S):
            assert_close(y[s].astype(np.float64), refs[s], f"shard {s} of {S}, M={M} out={od}")


def test_shards_above_one_row_are_per_shard_linears():
    S, M, k, n, K = 3, 5, 640, 384, 5
    x, t, suh, svh = _shards(7, S, M, k, n, K)
    xd, td, sd, vd = dev(x), dev(t), dev(suh), dev(svh)
    y = host(tq.exl3_linear_shards(xd, td, sd, vd, K))
    for s in range(S):
        one = host(tq.exl3_linear(xd, td[s].contiguous(), sd[s].contiguous(), vd[s].contiguous(), K))
        assert np.array_equal(y[s].view(np.uint16), one.view(np.uint16))


def test_shards_one_launch_is_deterministic_and_leaves_workspace_clean():
    S, k, n, K = 2, 5120, 5120, 4
    x, t, suh, svh = _shards(8, S, 1, k, n, K)
    xd, td, sd, vd = dev(x), dev(t), dev(suh), dev(svh)
    ws = torch.zeros(tq.exl3_linear_shards_workspace_size(1, k, n, K, S), dtype=torch.uint8, device="cuda")
    y1 = tq.exl3_linear_shards(xd, td, sd, vd, K, workspace_buf=ws).clone()
    y2 = tq.exl3_linear_shards(xd, td, sd, vd, K, workspace_buf=ws).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    counters = host(ws[256:256 + 4 * 2 * (n // 128)]).view(np.int32)
    assert np.all(counters == 0)


# ------------------------------------------------- shards of different widths --

def _var_shards(sub, widths, M, k, K):
    cases = [synth.linear_case(19, 500 + sub * 10 + s, M, k, n, K) for s, n in enumerate(widths)]
    x = cases[0].x
    t = np.concatenate([c.trellis.reshape(-1) for c in cases])
    suh = np.stack([c.suh for c in cases])
    svh = np.concatenate([c.svh for c in cases])
    return x, cases, t, suh, svh


@pytest.mark.parametrize("widths,M,k,K", [((5120, 1024, 1024), 1, 5120, 4), ((384, 128, 640, 256), 1, 1152, 3),
                                          ((256, 512), 1, 256, 8), ((128,) * 9, 1, 512, 2),
                                          ((640, 128, 384), 6, 768, 5)])
def test_var_shards_match_oracle(widths, M, k, K):
    """GQA-style q, k, v; ragged widths (256-column blocks at K = 3 end inside
    a shard); nine shards (more than one launch holds: one linear each); and
    M = 6 (one linear each)."""
    x, cases, t, suh, svh = _var_shards(len(widths) * 7 + M, widths, M, k, K)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = host(tq.exl3_linear_shards_var(dev(x), dev(t), dev(suh), dev(svh), widths, K, out_dtype=od))
        off = 0
        for s, (c, n) in enumerate(zip(cases, widths)):
            ref = oracle.linear(x, c.trellis, c.suh, c.svh, K)
            got = y[off:off + M * n].reshape(M, n).astype(np.float64)
            assert_close(got, ref, f"shard {s} width {n}, M={M} out={od}")
            off += M * n


def test_var_shards_one_launch_is_deterministic_and_leaves_workspace_clean():
    widths, k, K = (5120, 1024, 1024), 5120, 4
    x, _, t, suh, svh = _var_shards(3, widths, 1, k, K)
    xd, td, sd, vd = dev(x), dev(t), dev(suh), dev(svh)
    ws = torch.zeros(tq.exl3_linear_shards_var_workspace_size(1, k, widths, K), dtype=torch.uint8, device="cuda")
    y1 = tq.exl3_linear_shards_var(xd, td, sd, vd, widths, K, workspace_buf=ws).clone()
    y2 = tq.exl3_linear_shards_var(xd, td, sd, vd, widths, K, workspace_buf=ws).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    counters = host(ws[256:256 + 4 * 64]).view(np.int32)
    assert np.all(counters == 0)


def test_var_shards_of_one_width_agree_with_equal_shards():
    """Equal widths through the variable-width entry point: same results as
    exl3_linear_shards within the tolerance (the split of the sums differs)."""
    S, n, k, K = 3, 768, 1024, 4
    x, cases, t, suh, svh = _var_shards(4, (n,) * S, 1, k, K)
    yv = host(tq.exl3_linear_shards_var(dev(x), dev(t), dev(suh), dev(svh), (n,) * S, K,
                                        out_dtype=tq.EXL3_OUT_F32)).reshape(S, 1, n)
    ye = host(tq.exl3_linear_shards(dev(x), dev(t.reshape(S, k // 16, n // 16, 16 * K)), dev(suh),
                                    dev(svh.reshape(S, n)), K, out_dtype=tq.EXL3_OUT_F32))
    for s in range(S):
        assert_close(yv[s].astype(np.float64), ye[s].astype(np.float64), f"shard {s}")

"""GPU parity of libexl3 against the CPU oracle: dequantisation, the input
transform and the linear at M = 1 and above (through the C ABI).

Dequantised weights and the fp32 input transform must match bit for bit;
linear outputs must meet the tolerance in tests/gpu_util.py.  Inputs are the
seeded synthetic workloads of exl3_synth (the shapes of the pages' dense 27B
family: "exl3xpu" README; mixed widths: tracker #832).
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu

BOUND = 3.453125


# ------------------------------------------------------------- dequantise --

@pytest.mark.parametrize("K", range(1, 9))
def test_decode_tile_bit_exact(K):
    case = synth.linear_case(10, K, 1, 256, 384, K)
    ref = oracle.reconstruct(case.trellis, 256, 384, K).view(np.uint16)
    got = host(tq.exl3_decode_tile(dev(case.trellis), 256, 384, K)).view(np.uint16)
    assert np.array_equal(got, ref)


def test_decode_tile_subrange_with_padded_rows():
    K, k, n = 3, 256, 512
    case = synth.linear_case(10, 20, 1, k, n, K)
    ref = oracle.reconstruct(case.trellis, k, n, K).view(np.uint16)
    tk0, tkc, tn0, tnc, ld = 3, 5, 7, 9, 160
    out = torch.full((16 * tkc, ld), 7.0, dtype=torch.float16, device="cuda")
    tq.exl3_decode_tile(dev(case.trellis), k, n, K, tk0=tk0, tk_cnt=tkc, tn0=tn0, tn_cnt=tnc, w_out=out, ld=ld)
    got = host(out).view(np.uint16)
    assert np.array_equal(got[:, :16 * tnc], ref[16 * tk0:16 * (tk0 + tkc), 16 * tn0:16 * (tn0 + tnc)])
    assert np.all(host(out)[:, 16 * tnc:] == 7.0)      # padding untouched


def _all_states_trellis():
    """K = 8 tiles whose byte streams make every (lo, hi) byte pair a state.

    For K = 8, state p is stream bytes p and p+1.  Tile (hi, half) holds bytes
    b[2i] = 128 * half + i and b[2i+1] = hi, so its even states are
    (128 * half + i) | hi << 8: 512 tiles cover all 65536 states."""
    tiles = np.zeros((16, 32, 128), dtype=np.uint16)   # k = 256, n = 512: 512 tiles
    for t in range(512):
        hi, half = t >> 1, t & 1
        b = np.zeros(256, dtype=np.uint8)
        b[0::2] = 128 * half + np.arange(128)
        b[1::2] = hi
        tiles[t // 32, t % 32] = b.view(np.uint16)
    return tiles


def test_codebook_exhaustive_all_65536_states():
    t = _all_states_trellis()
    covered = set()
    for tk in range(16):
        for tn in range(32):
            covered.update(oracle.tile_states(t[tk, tn], 8)[0::2].tolist())
    assert len(covered) == 65536
    ref = oracle.reconstruct(t, 256, 512, 8).view(np.uint16)
    got = host(tq.exl3_decode_tile(dev(t), 256, 512, 8)).view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("K", [1, 5, 8])
def test_decode_special_trellises(K):
    zero = np.zeros((8, 8, 16 * K), dtype=np.uint16)
    got = host(tq.exl3_decode_tile(dev(zero), 128, 128, K)).astype(np.float64)
    assert np.all(got == -BOUND)
    ones = np.full((8, 8, 16 * K), 0xFFFF, dtype=np.uint16)
    got = host(tq.exl3_decode_tile(dev(ones), 128, 128, K)).view(np.uint16)
    assert np.all(got == oracle.mul1_value_bits(0xFFFF))


# --------------------------------------------------------------- transform --

def test_input_rht_bit_exact():
    case = synth.linear_case(11, 0, 7, 1024, 128, 2, outlier_rows=0.3)
    ref = oracle.rht_in_f32(case.x, case.suh)
    x, suh = dev(case.x), dev(case.suh)
    got32 = host(tq.exl3_input_rht(x, suh, tq.EXL3_OUT_F32))
    assert np.array_equal(got32.view(np.uint32), ref.view(np.uint32))
    got16 = host(tq.exl3_input_rht(x, suh, tq.EXL3_OUT_F16))
    assert np.array_equal(got16.view(np.uint16), ref.astype(np.float16).view(np.uint16))


# ------------------------------------------------------------------ linear --

def _run(case, out_dtype):
    y = tq.exl3_linear(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), case.K,
                       out_dtype=out_dtype)
    return host(y).astype(np.float64)


def _check_case(case, ref=None, rows=None):
    if ref is None:
        x = case.x if rows is None else case.x[rows]
        ref = oracle.linear(x, case.trellis, case.suh, case.svh, case.K)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = _run(case, od)
        if rows is not None:
            y = y[rows]
        assert_close(y, ref, f"{case.name} out={'f32' if od else 'f16'}")


def test_linear_config1():
    _check_case(synth.config1())


@pytest.mark.parametrize("n", synth.CONFIG2_N)
def test_linear_config2_m1(n):
    _check_case(synth.config2(n, 1))


@pytest.mark.parametrize("M", synth.CONFIG3_M)
@pytest.mark.parametrize("K", synth.CONFIG3_K)
def test_linear_config3_all_widths_and_rows(K, M):
    """Every (K, M) pair of the mixed-width layer (k = n = 4096, 5% outlier
    rows x20): M = 1 on the GEMV, M = 8 and 64 on the fused tensor-core
    kernel; fp16 and fp32 outputs."""
    _check_case(synth.config3(K, M))


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("k,n", [(128, 128), (384, 384), (1152, 640)])
def test_linear_m1_ragged_shapes(K, k, n):
    """Smallest shape (one block), column counts that leave a CTA half empty,
    and k-ranges that are not a power of two."""
    _check_case(synth.linear_case(12, K * 10 + n // 128, 1, k, n, K))


@pytest.mark.parametrize("M", [4, 16])
@pytest.mark.parametrize("n", synth.CONFIG2_N)
def test_linear_config2_small_m(n, M):
    """The decode sweep's small-M rows at every width (k = 5120, K = 4, n up to
    25600: 1600 tiles along n), fp16 and fp32 outputs."""
    _check_case(synth.config2(n, M))


@pytest.mark.parametrize("M", [2, 3, 31, 127, 128, 129, 200])
def test_linear_small_m_around_path_switch(M):
    """2 <= M <= 128 take the fused decode + tcgen05 kernel, larger M the
    reconstruct + tcgen05 GEMM."""
    _check_case(synth.linear_case(15, M, M, 1024, 768, 4))


@pytest.mark.parametrize("K", range(1, 9))
def test_linear_fused_small_m_all_widths(K):
    """Every K through the fused kernel, with a k that splits unevenly (k/64 = 18)."""
    _check_case(synth.linear_case(16, K, 5, 1152, 384, K, outlier_rows=0.2))


@pytest.mark.parametrize("K,k,M", [(3, 128, 4), (4, 128, 16), (8, 128, 100), (1, 256, 33), (6, 384, 17)])
def test_linear_fused_small_m_short_k(K, k, M):
    """k = 128 is a single pair of k steps (the second decoder group and its
    accumulator stay idle); k = 256 and 384 give one and a half trellis stages;
    M = 33 and 100 use the wide x' layout."""
    _check_case(synth.linear_case(17, K * 1000 + k, M, k, 256, K, outlier_rows=0.1))


def test_linear_prefill_config4_sampled_rows():
    """Full M = 4096 on the GPU; the oracle evaluates a seeded sample of rows
    (rows are independent) including rows of every outlier channel."""
    case = synth.config4()
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 1, 4095], rng.choice(4096, 13, replace=False)]))
    W = oracle.reconstruct(case.trellis, case.k, case.n, case.K)
    ref = oracle.linear_w(case.x[rows], W, case.suh, case.svh)
    _check_case(case, ref=ref, rows=rows)


def test_linear_odd_m_and_zero_rows():
    case = synth.linear_case(13, 0, 37, 640, 384, 6)
    case.x[5] = 0
    _check_case(case)


def test_linear_deterministic_and_workspace_clean():
    case = synth.config2(17408, 1)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    need = tq.exl3_linear_workspace_size(1, case.k, case.n, case.K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y1 = tq.exl3_linear(x, t, suh, svh, 4, workspace_buf=ws).clone()
    y2 = tq.exl3_linear(x, t, suh, svh, 4, workspace_buf=ws).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    # the arrival counters (right after the 256-byte control block) are back at zero
    counters = host(ws[256:256 + 4 * (case.n // 128)]).view(np.int32)
    assert np.all(counters == 0)


def test_linear_rejects_small_workspace():
    case = synth.linear_case(14, 0, 1, 256, 256, 4)
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.Exl3Error) as e:
        tq.exl3_linear(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), 4, workspace_buf=ws)
    assert e.value.code == tq.EXL3_ERR_WORKSPACE


def test_linear_m1_weight_prefetch_chain():
    """With weight prefetch on, M = 1 linears launch as programmatic dependents:
    each may stream weights while the kernel ahead of it runs, but must read
    its input only after that kernel completes.  A chain in which each output
    is the next input (a long linear feeding a short one, directly, through a
    torch kernel, and captured in a CUDA graph) must give bit-for-bit the
    results of the same chain run without prefetch."""
    a = synth.linear_case(18, 0, 1, 5120, 17408, 4)
    b = synth.linear_case(18, 1, 1, 17408, 5120, 3)
    A = [dev(v) for v in (a.x, a.trellis, a.suh, a.svh)]
    B = [dev(v) for v in (b.trellis, b.suh, b.svh)]
    wsa = torch.zeros(tq.exl3_linear_workspace_size(1, a.k, a.n, 4), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros(tq.exl3_linear_workspace_size(1, b.k, b.n, 3), dtype=torch.uint8, device="cuda")
    ya = torch.empty((1, a.n), dtype=torch.float16, device="cuda")
    yb = torch.empty((1, b.n), dtype=torch.float16, device="cuda")

    def chain(via_torch=False):
        tq.exl3_linear(A[0], A[1], A[2], A[3], 4, y=ya, workspace_buf=wsa)
        xb = ya * 1.0 if via_torch else ya
        tq.exl3_linear(xb, B[0], B[1], B[2], 3, y=yb, workspace_buf=wsb)

    prev = tq.exl3_set_weight_prefetch(False)
    try:
        chain()
        ref_a, ref_b = ya.clone(), yb.clone()
        assert_close(host(ref_a).astype(np.float64), oracle.linear(a.x, a.trellis, a.suh, a.svh, 4), "chain head")
        tq.exl3_set_weight_prefetch(True)
        for via_torch in (False, True):
            for _ in range(5):
                yb.fill_(0)
                chain(via_torch)
                assert torch.equal(ya, ref_a) and torch.equal(yb, ref_b)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            chain()
            with torch.cuda.graph(g, stream=s):
                chain()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(5):
            yb.fill_(0)
            g.replay()
            assert torch.equal(ya, ref_a) and torch.equal(yb, ref_b)
        assert tq.exl3_check_device_error(wsa) == 0 and tq.exl3_check_device_error(wsb) == 0
    finally:
        tq.exl3_set_weight_prefetch(prev)


def test_linear_m1_k_too_large_for_gemv_takes_tensor_core_path():
    """At K = 7 and k = 49152, x' and two 56 KB ring stages do not fit in the
    GEMV's shared memory: M = 1 then runs the small-M tensor-core path, with
    the same results; the workspace-free GEMV entry rejects the shape."""
    case = synth.linear_case(19, 0, 1, 49152, 256, 7)
    _check_case(case)
    with pytest.raises(tq.Exl3Error) as e:
        tq.exl3_linear_gemv_noalloc(dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh), 7)
    assert e.value.code == tq.EXL3_ERR_SHAPE


def test_linear_m1_concurrent_streams_share_the_gpu():
    """The GEMV finishes a column block shared by several CTAs in whichever
    CTA arrives last, with no CTA waiting for another, so it does not need
    all its CTAs resident at once.  Four GEMVs on four streams (each with its
    own workspace) run beside a stream of large matmuls that holds SMs; every
    result must be bit-identical to the same linear run alone, with clean
    device error words."""
    case = synth.config2(25600, 1)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    need = tq.exl3_linear_workspace_size(1, case.k, case.n, case.K)
    ref = tq.exl3_linear(x, t, suh, svh, 4, out_dtype=tq.EXL3_OUT_F32).clone()
    assert_close(host(ref).astype(np.float64), oracle.linear(case.x, case.trellis, case.suh, case.svh, 4),
                 "alone")
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)
    hog = torch.cuda.Stream()
    streams = [torch.cuda.Stream() for _ in range(4)]
    wss = [torch.zeros(need, dtype=torch.uint8, device="cuda") for _ in streams]
    ys = [torch.empty((1, case.n), dtype=torch.float32, device="cuda") for _ in streams]
    torch.cuda.synchronize()
    for rep in range(3):
        with torch.cuda.stream(hog):
            b = a
            for _ in range(20):
                b = b @ a * 1e-3
        for s, ws, y in zip(streams, wss, ys):
            with torch.cuda.stream(s):
                for _ in range(5):
                    tq.exl3_linear(x, t, suh, svh, 4, out_dtype=tq.EXL3_OUT_F32, y=y, workspace_buf=ws, stream=s)
        torch.cuda.synchronize()
        for ws, y in zip(wss, ys):
            assert torch.equal(y, ref)
            assert tq.exl3_check_device_error(ws) == 0

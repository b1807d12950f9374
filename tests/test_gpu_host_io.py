"""Host memory at the ends of a decode step: exl3_copy_in brings x from
pinned host memory, and an M = 1 exl3_linear may write y straight into
pinned host memory.

- The copy is bit-exact for sizes with and without a tail of fewer than 16
  bytes, and writes nothing past the destination.
- The copy is ordered against the linears around it: it overwrites a device
  x that the linear before it reads, and the linear after it reads the new x
  (with and without weight prefetch, eagerly and in a CUDA graph).
- A pinned host y gets the same bits as a device y on every M = 1 path: the
  GEMV, the small-M tensor-core kernel that M = 1 takes when x' is too large
  for the GEMV's shared memory, and the row-invariant mode; the result is
  within the parity tolerance of the float64 oracle.
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _pinned(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


@pytest.mark.parametrize("nbytes", [1, 15, 16, 4096 + 7, 30720, (1 << 20) + 3, 8 << 20])
def test_copy_in_is_bit_exact_and_stays_in_bounds(nbytes):
    g = torch.Generator().manual_seed(7000 + nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    guard = 256
    dst = torch.full((nbytes + guard,), 0xAB, dtype=torch.uint8, device="cuda")
    tq.exl3_copy_in(src, dst[:nbytes])
    torch.cuda.synchronize()
    assert torch.equal(dst[:nbytes].cpu(), src)
    assert bool((dst[nbytes:] == 0xAB).all()), "bytes written past the destination"


@pytest.mark.parametrize("prefetch", [False, True])
@pytest.mark.parametrize("graph", [False, True])
def test_copy_in_is_ordered_against_the_linears_around_it(prefetch, graph):
    a = synth.config2(17408, 1)
    b = synth.linear_case(2, 951, 1, 5120, 17408, 4)
    t, suh, svh = dev(a.trellis), dev(a.suh), dev(a.svh)
    refs = [tq.exl3_linear(dev(c.x), t, suh, svh, 4).clone() for c in (a, b)]
    hxs = [_pinned(c.x) for c in (a, b)]
    dx = torch.empty((1, 5120), dtype=torch.int16, device="cuda")
    ys = [torch.empty((1, 17408), dtype=torch.float16, device="cuda") for _ in range(8)]
    ws = tq.workspace(tq.exl3_linear_workspace_size(1, 5120, 17408, 4))
    prev = tq.exl3_set_weight_prefetch(prefetch)
    try:
        def run():
            tq.exl3_copy_in(hxs[0], dx)
            for i in range(8):
                tq.exl3_linear(dx, t, suh, svh, 4, y=ys[i], workspace_buf=ws)
                tq.exl3_copy_in(hxs[(i + 1) % 2], dx)

        torch.cuda.synchronize()
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run()
            for y in ys:
                y.zero_()
            g.replay()
        else:
            run()
        torch.cuda.synchronize()
    finally:
        tq.exl3_set_weight_prefetch(prev)
    for i, y in enumerate(ys):
        assert torch.equal(y, refs[i % 2]), f"linear {i} did not read the x copied before it"
    assert tq.exl3_check_device_error(ws) == 0


# (k, n, K): the GEMV; a k whose fp32 x' does not fit beside two GEMV
# stages at K = 7 (the small-M kernel then runs M = 1); a mixed-width shape
@pytest.mark.parametrize("k,n,K", [(5120, 17408, 4), (24576, 256, 7), (4096, 4096, 3)])
@pytest.mark.parametrize("out_dtype", [tq.EXL3_OUT_F16, tq.EXL3_OUT_F32])
@pytest.mark.parametrize("row_invariant", [False, True])
def test_linear_m1_writes_pinned_host_y(k, n, K, out_dtype, row_invariant):
    case = synth.linear_case(2, 960 + K, 1, k, n, K)
    x, t, suh, svh = dev(case.x), dev(case.trellis), dev(case.suh), dev(case.svh)
    dt = torch.float32 if out_dtype == tq.EXL3_OUT_F32 else torch.float16
    prev = tq.exl3_set_row_invariant(row_invariant)
    try:
        yd = tq.exl3_linear(x, t, suh, svh, K, out_dtype=out_dtype)
        yh = torch.full((1, n), float("nan"), dtype=dt).pin_memory()
        tq.exl3_linear(x, t, suh, svh, K, out_dtype=out_dtype, y=yh)
        torch.cuda.synchronize()
    finally:
        tq.exl3_set_row_invariant(prev)
    assert torch.equal(yh, yd.cpu()), "host y differs from device y"
    assert_close(host(yd).astype(np.float64), oracle.linear(case.x, case.trellis, case.suh, case.svh, K),
                 f"k{k} n{n} K{K}")


def test_decode_step_host_to_host_in_a_graph():
    """The decode-loop form: x for three linears copied in by one exl3_copy_in,
    the linears chained with weight prefetch, their y written to pinned host
    memory; captured in a CUDA graph and replayed."""
    cases = [synth.config2(n, 1) for n in synth.CONFIG2_N]
    hx = _pinned(np.concatenate([c.x.reshape(-1) for c in cases]))
    ny = [c.n for c in cases]
    hy = torch.zeros(sum(ny), dtype=torch.float16).pin_memory()
    dx = torch.empty(hx.shape, dtype=hx.dtype, device="cuda")
    ws = [tq.workspace(tq.exl3_linear_workspace_size(1, c.k, c.n, c.K)).clone().zero_() for c in cases]
    dw = [(dev(c.trellis), dev(c.suh), dev(c.svh)) for c in cases]
    refs = [tq.exl3_linear(dev(c.x), *dw[j], c.K).cpu() for j, c in enumerate(cases)]
    yo = np.cumsum([0] + ny)
    prev = tq.exl3_set_weight_prefetch(True)
    try:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for rep in range(3):
                tq.exl3_copy_in(hx, dx)
                for j, c in enumerate(cases):
                    tq.exl3_linear(dx[j * c.k:(j + 1) * c.k].view(1, -1), *dw[j], c.K,
                                   y=hy[int(yo[j]):int(yo[j + 1])].view(1, -1), workspace_buf=ws[j])
        g.replay()
        torch.cuda.synchronize()
    finally:
        tq.exl3_set_weight_prefetch(prev)
    for j in range(len(cases)):
        assert torch.equal(hy[int(yo[j]):int(yo[j + 1])].view(1, -1), refs[j])
        assert tq.exl3_check_device_error(ws[j]) == 0

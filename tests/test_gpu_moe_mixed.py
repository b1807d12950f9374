"""GPU parity of the routed experts with a width per expert
(exl3_moe_grouped_mixed) against the CPU oracle ("EXL3 checkpoints on the
native engine (tracker) #832": widths 1..8 per tensor, and the Oct 17 comment
keeps each expert's own width in the format).

Each projection's arena packs expert e right after expert e-1 at its own
width.  With more than 32 routed rows every run of consecutive equal widths
is one grouped tile launch; with at most 32 (and at most 8 runs), each
projection is one grouped-GEMV launch over all its runs, whose CTAs split
over the widths present.  Outputs
must meet the tolerance of tests/gpu_util.py against the float64 oracle;
with one width for all experts the call must give the bits of
exl3_moe_grouped's tile path.
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _dev_mixed(c):
    d = dict(x=dev(c.x), ids=dev(c.ids), w=dev(c.weights),
             t13=dev(c.w13.trellis), s13=dev(c.w13.suh), v13=dev(c.w13.svh),
             t2=dev(c.w2.trellis), s2=dev(c.w2.suh), v2=dev(c.w2.svh))
    d["w13"] = tq.expert_proj_mixed(d["t13"], d["s13"], d["v13"], c.w13.K, c.hidden, c.inter)
    d["w2"] = tq.expert_proj_mixed(d["t2"], d["s2"], d["v2"], c.w2.K, c.inter, c.hidden)
    return d


def _oracle(c, tokens=None, ids=None, weights=None):
    return oracle.moe_k(c.x, c.ids if ids is None else ids, c.weights if weights is None else weights,
                        c.w13.trellis, c.w13.suh, c.w13.svh, c.w13.K, c.w2.trellis, c.w2.suh, c.w2.svh, c.w2.K,
                        c.inter, tokens=tokens)


CASES = [
    # (E, topk, T, hidden, inter, K13, K2): runs of 3, 3 and 2 experts with
    # different run boundaries for the two projection kinds
    (8, 2, 37, 256, 128, [3, 3, 3, 4, 4, 4, 5, 5], [2, 2, 6, 6, 6, 6, 1, 1]),
    # every expert its own run, all eight widths
    (8, 3, 20, 256, 256, [1, 8, 2, 7, 3, 6, 4, 5], [8, 1, 7, 2, 6, 3, 5, 4]),
    # one token (decode): eight routed rows over sixteen experts in two runs
    (16, 8, 1, 512, 128, [3] * 8 + [4] * 8, [4] * 8 + [3] * 8),
    # many rows per expert: tiles of 128 rows and a ragged last tile
    (4, 2, 300, 256, 384, [2, 2, 7, 7], [5, 3, 3, 5]),
]


@pytest.mark.parametrize("E,topk,T,hidden,inter,K13,K2", CASES)
def test_moe_mixed_matches_oracle(E, topk, T, hidden, inter, K13, K2):
    c = synth.mixed_moe_case(58, E * 100 + T, T, K13, K2, topk=topk, hidden=hidden, inter=inter)
    d = _dev_mixed(c)
    ref = _oracle(c)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], E, out_dtype=od)
        assert_close(host(y).astype(np.float64), ref, f"mixed E={E} T={T} out={od}")


def test_moe_mixed_config5_shape_two_widths_sampled_tokens():
    """The MoE workload's shape (256 experts, top-8, hidden 2048, inter 512,
    T = 128) with experts 0-127 at K = 3 and 128-255 at K = 4 (down: the
    other way round); the oracle evaluates a seeded sample of tokens."""
    K13 = [3] * 128 + [4] * 128
    K2 = [4] * 128 + [3] * 128
    c = synth.mixed_moe_case(59, 0, 128, K13, K2)
    d = _dev_mixed(c)
    y = host(tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E)).astype(np.float64)
    tokens = np.array([0, 5, 77, 127], dtype=np.int32)
    assert_close(y[tokens], _oracle(c, tokens=tokens), "mixed config-5 shape")


def test_moe_mixed_one_width_is_the_uniform_tile_path():
    """One width for all experts: the packed arena is the uniform layout, and
    with more than 32 routed rows both entry points run the same tile kernels
    over the same experts, so the outputs are identical."""
    c = synth.moe_case(57, 0, 64, E=32, topk=8, hidden=512, inter=256, K=3)
    x, ids, w = dev(c.x), dev(c.ids), dev(c.weights)
    t13, s13, v13 = dev(c.w13.trellis), dev(c.w13.suh), dev(c.w13.svh)
    t2, s2, v2 = dev(c.w2.trellis), dev(c.w2.suh), dev(c.w2.svh)
    uni = tq.exl3_moe_grouped(x, ids, w, tq.expert_proj(t13, s13, v13, 3), tq.expert_proj(t2, s2, v2, 3), c.E,
                              out_dtype=tq.EXL3_OUT_F32)
    K = [3] * c.E
    mix = tq.exl3_moe_grouped_mixed(x, ids, w, tq.expert_proj_mixed(t13, s13, v13, K, 512, 256),
                                    tq.expert_proj_mixed(t2, s2, v2, K, 256, 512), c.E, out_dtype=tq.EXL3_OUT_F32)
    assert np.array_equal(host(uni).view(np.uint32), host(mix).view(np.uint32))


def test_moe_mixed_invalid_expert_id_is_reported_and_skipped():
    c = synth.mixed_moe_case(60, 0, 5, [3, 4, 4, 2], [2, 2, 5, 5], topk=2, hidden=256, inter=128)
    d = _dev_mixed(c)
    bad_ids = c.ids.copy()
    bad_ids[3, 0] = -1                             # outside [0, E)
    ws = torch.zeros(tq.exl3_moe_mixed_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y = tq.exl3_moe_grouped_mixed(d["x"], dev(bad_ids), d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws)
    assert tq.exl3_check_device_error(ws) != 0
    ref_ids = bad_ids.copy()
    ref_ids[3, 0] = 0
    ref_w = c.weights.copy()
    ref_w[3, 0] = 0.0
    assert_close(host(y).astype(np.float64), _oracle(c, ids=ref_ids, weights=ref_w), "mixed invalid id")


@pytest.mark.parametrize("T", [1, 4, 16, 32])
def test_moe_mixed_few_tokens_grouped_gemv(T):
    """Up to 32 routed rows, or up to 1.25 per expert, take the few-token
    path: per projection one grouped M = 1 GEMV launch whose CTAs split over
    the widths of the routed experts (found on the device, each CTA keeping
    its width's unit list in shared memory: 8 to 256 units here).  The MoE
    workload's shape with two widths per projection; deterministic, with the
    arrival counters back at zero."""
    K13 = [3] * 128 + [4] * 128
    K2 = [4] * 128 + [3] * 128
    c = synth.mixed_moe_case(61, T, T, K13, K2)
    d = _dev_mixed(c)
    ws = torch.zeros(tq.exl3_moe_mixed_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y1 = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws,
                                   out_dtype=tq.EXL3_OUT_F32).clone()
    y2 = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws,
                                   out_dtype=tq.EXL3_OUT_F32).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    assert np.all(host(ws[256:256 + 4 * 8192]).view(np.int32) == 0)
    assert_close(host(y1).astype(np.float64), _oracle(c), f"mixed few tokens T={T}")


def test_moe_mixed_few_tokens_width_without_units():
    """Every routed expert has width 3, so no CTA of either launch takes the
    width-5 experts' runs; the launches must still run only the routed
    width and leave the chain ordered."""
    c = synth.mixed_moe_case(62, 0, 3, [3, 3, 3, 3, 5, 5, 5, 5], [3, 3, 3, 3, 5, 5, 5, 5], topk=2, hidden=512,
                             inter=256)
    c.ids[:] = np.array([[0, 1], [2, 3], [1, 2]], dtype=np.int32)
    d = _dev_mixed(c)
    y = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, out_dtype=tq.EXL3_OUT_F32)
    assert_close(host(y).astype(np.float64), _oracle(c), "mixed width without units")


def test_moe_mixed_few_tokens_all_ids_invalid():
    """No valid expert id: no CTA has a share, every unit's combine row is
    -1, the output is zero and the error word is set."""
    c = synth.mixed_moe_case(63, 0, 2, [3, 4], [4, 3], topk=2, hidden=256, inter=128)
    d = _dev_mixed(c)
    bad = np.full_like(c.ids, 5)
    ws = torch.zeros(tq.exl3_moe_mixed_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y = tq.exl3_moe_grouped_mixed(d["x"], dev(bad), d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws)
    assert tq.exl3_check_device_error(ws) != 0
    assert np.all(host(y) == 0)


@pytest.mark.parametrize("E", [8, 10])
def test_moe_mixed_few_tokens_alternating_widths(E):
    """Widths alternating per expert: 8 experts give 8 runs per projection
    (one launch holds their 8 tensor maps); 10 give 10 runs, more than one
    launch holds, so the call takes the tile kernels."""
    K13 = [3 if e % 2 == 0 else 4 for e in range(E)]
    K2 = [4 if e % 2 == 0 else 2 for e in range(E)]
    c = synth.mixed_moe_case(64, E, 4, K13, K2, topk=6, hidden=256, inter=256)
    d = _dev_mixed(c)
    y = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], d["w13"], d["w2"], E, out_dtype=tq.EXL3_OUT_F32)
    assert_close(host(y).astype(np.float64), _oracle(c), f"mixed alternating widths E={E}")

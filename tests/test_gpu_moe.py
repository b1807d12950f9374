"""GPU parity of the grouped routed-expert path against the CPU oracle
("exl3xpu" README, "MoE (routed experts)"; Arc 140V MoE post, sections 2.A-2.D).

The seeded workloads have the pages' MoE shape (256 experts, top-8, hidden
2048, inter 512, K = 3); outputs must meet the tolerance of tests/gpu_util.py
against the float64 oracle.  Large token counts are checked on a seeded
sample of tokens (each token's output depends on its own routing only).
"""
import numpy as np
import pytest
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _dev_case(c):
    d = dict(x=dev(c.x), ids=dev(c.ids), w=dev(c.weights),
             t13=dev(c.w13.trellis), s13=dev(c.w13.suh), v13=dev(c.w13.svh),
             t2=dev(c.w2.trellis), s2=dev(c.w2.suh), v2=dev(c.w2.svh))
    d["w13"] = tq.expert_proj(d["t13"], d["s13"], d["v13"], c.w13.K)
    d["w2"] = tq.expert_proj(d["t2"], d["s2"], d["v2"], c.w2.K)
    return d


def _run(c, d, out_dtype=tq.EXL3_OUT_F16, ids=None, weights=None):
    ids = d["ids"] if ids is None else ids
    weights = d["w"] if weights is None else weights
    y = tq.exl3_moe_grouped(d["x"], ids, weights, d["w13"], d["w2"], c.E, out_dtype=out_dtype)
    return host(y).astype(np.float64)


def _oracle(c, tokens=None, ids=None, weights=None):
    return oracle.moe(c.x, c.ids if ids is None else ids, c.weights if weights is None else weights,
                      c.w13.trellis, c.w13.suh, c.w13.svh, c.w13.K, c.w2.trellis, c.w2.suh, c.w2.svh, c.w2.K,
                      tokens=tokens)


@pytest.mark.parametrize("T", [1, 128])
def test_moe_config5_full(T):
    c = synth.config5(T)
    d = _dev_case(c)
    ref = _oracle(c)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        assert_close(_run(c, d, od), ref, f"{c.name} out={od}")


def test_moe_config5_t4096_sampled_tokens():
    """T = 4096 in full on the GPU (fp16 and fp32 outputs); the oracle
    evaluates a seeded sample of tokens."""
    c = synth.config5(4096)
    d = _dev_case(c)
    rng = np.random.default_rng(50)
    tokens = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 14, replace=False)])).astype(np.int32)
    ref = _oracle(c, tokens=tokens)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        y = _run(c, d, od)
        assert_close(y[tokens], ref, f"{c.name} sampled out={od}")


@pytest.mark.parametrize("E,topk,T", [(4, 2, 3), (1, 1, 5), (8, 8, 37), (1000, 4, 300)])
def test_moe_small_shapes(E, topk, T):
    """Few experts (many rows per expert), a single expert, all experts hit,
    and 1000 experts (the routing step bins units in several chunks)."""
    c = synth.moe_case(51, E * 10 + topk, T, E=E, topk=topk, hidden=256, inter=128, K=4)
    d = _dev_case(c)
    assert_close(_run(c, d), _oracle(c), f"moe E{E} top{topk} T{T}")


@pytest.mark.parametrize("K,K2,hidden,inter", [(8, 8, 256, 128), (5, 5, 512, 256), (1, 7, 256, 384), (6, 2, 768, 128)])
def test_moe_widths_and_shapes(K, K2, hidden, inter):
    """Every width on both projections (different widths for gate+up and down),
    down projections of one and several k-step pairs, odd numbers of 128-row
    output tiles."""
    c = synth.moe_case(55, K * 10 + K2, 40, E=6, topk=3, hidden=hidden, inter=inter, K=K, K2=K2)
    d = _dev_case(c)
    assert_close(_run(c, d), _oracle(c), f"moe K{K}/{K2} h{hidden} i{inter}")


def test_moe_many_rows_one_expert_spans_tiles():
    """300 rows on one expert: its rows cross two 128-row tiles plus a partial one."""
    c = synth.moe_case(52, 0, 150, E=3, topk=2, hidden=512, inter=256, K=2)
    c.ids[:, 0] = 1
    c.ids[:, 1] = (np.arange(150) % 2) * 2        # experts 0 and 2 alternate in slot 1
    d = _dev_case(c)
    assert_close(_run(c, d), _oracle(c), "moe one expert with 150+ rows")


def test_moe_expert_beyond_one_256_row_tile():
    """400 tokens, top-2 over 3 experts, every first slot on expert 1: 800
    routed rows (at least 96 per expert) take 256-row tiles, expert 1's 400
    rows span two of them (256 + 144) and its epilogue runs in 128-row
    chunks; experts 0 and 2 hold 200 rows each in one tile."""
    c = synth.moe_case(52, 1, 400, E=3, topk=2, hidden=512, inter=256, K=3)
    c.ids[:, 0] = 1
    c.ids[:, 1] = (np.arange(400) % 2) * 2
    d = _dev_case(c)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        assert_close(_run(c, d, od), _oracle(c), f"moe 256-row tiles out={od}")


def test_moe_expert_beyond_one_160_row_tile():
    """240 tokens, top-2 over 4 experts: 480 routed rows (120 per expert on
    average, between 96 and 136) take 160-row tiles; every first slot on
    expert 1 gives it 240 rows over two tiles (160 + 80), whose epilogue runs
    in a 128-row and a 32-row chunk; experts 0 and 2 hold 120 rows each."""
    c = synth.moe_case(52, 2, 240, E=4, topk=2, hidden=512, inter=256, K=3)
    c.ids[:, 0] = 1
    c.ids[:, 1] = (np.arange(240) % 2) * 2
    d = _dev_case(c)
    for od in (tq.EXL3_OUT_F16, tq.EXL3_OUT_F32):
        assert_close(_run(c, d, od), _oracle(c), f"moe 160-row tiles out={od}")


def test_moe_invalid_expert_id_is_reported_and_skipped():
    c = synth.moe_case(53, 0, 4, E=4, topk=2, hidden=256, inter=128, K=3)
    d = _dev_case(c)
    bad_ids = c.ids.copy()
    bad_ids[2, 1] = 7                              # outside [0, E)
    ws = torch.zeros(tq.exl3_moe_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y = tq.exl3_moe_grouped(d["x"], dev(bad_ids), d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws)
    assert tq.exl3_check_device_error(ws) != 0
    # the bad slot contributes nothing: same as routing it anywhere with weight 0
    ref_ids = bad_ids.copy()
    ref_ids[2, 1] = 0
    ref_w = c.weights.copy()
    ref_w[2, 1] = 0.0
    assert_close(host(y).astype(np.float64), _oracle(c, ids=ref_ids, weights=ref_w), "moe invalid id")


def test_moe_slot_order_does_not_matter():
    c = synth.moe_case(54, 0, 16, E=16, topk=4, hidden=256, inter=128, K=3)
    d = _dev_case(c)
    y1 = _run(c, d)
    perm = [3, 1, 0, 2]
    y2 = _run(c, d, ids=dev(np.ascontiguousarray(c.ids[:, perm])),
              weights=dev(np.ascontiguousarray(c.weights[:, perm])))
    assert np.max(np.abs(y1 - y2)) <= 2e-3 * max(1.0, np.abs(y1).max())


@pytest.mark.parametrize("E,topk,T,hidden,inter,K", [(8, 2, 17, 1024, 256, 4), (16, 4, 10, 2048, 128, 3),
                                                     (4, 4, 9, 512, 384, 5)])
def test_moe_gateup_split_over_k(E, topk, T, hidden, inter, K):
    """Few tokens (but more than 32 routed rows, so the tile kernels run): the
    gate+up projection is split over k across CTAs and the last CTA of each
    tile adds the partial sums in split order.  Same result on a second call
    (fixed order) and the arrival counters are back at zero."""
    c = synth.moe_case(56, E * 100 + T, T, E=E, topk=topk, hidden=hidden, inter=inter, K=K)
    d = _dev_case(c)
    ws = torch.zeros(tq.exl3_moe_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y1 = tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws).clone()
    y2 = tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    assert int(ws[256:256 + 4 * 8192].view(torch.int32).abs().sum()) == 0
    assert_close(host(y1).astype(np.float64), _oracle(c), f"moe split E{E} T{T}")


@pytest.mark.parametrize("T,E,topk,hidden,inter,K,K2", [(4, 256, 8, 2048, 512, 3, 3), (2, 16, 8, 512, 256, 8, 2),
                                                        (3, 6, 3, 256, 384, 1, 7), (1, 4, 2, 768, 128, 6, 5),
                                                        (16, 256, 8, 2048, 512, 3, 3), (32, 256, 8, 2048, 512, 3, 3),
                                                        (9, 96, 8, 512, 256, 4, 6)])
def test_moe_few_tokens_grouped_gemv(T, E, topk, hidden, inter, K, K2):
    """Up to 32 routed rows, or up to 1.25 per expert, take the few-token
    path: gate and up as grouped M = 1 GEMVs over (unit, slot), SiLU, down as
    grouped GEMVs times the routing weight, and the combine.  32 rows at the
    pages' shape is the first boundary, 128 and 256 rows over 256 experts
    (T = 16, and T = 32, whose CTAs' shares span five gate/up ops) and 72
    over 96 lie under the second; also mixed widths and odd tile counts.  Deterministic, with the arrival counters back at zero."""
    c = synth.moe_case(57, T * 100 + K, T, E=E, topk=topk, hidden=hidden, inter=inter, K=K, K2=K2)
    d = _dev_case(c)
    ws = torch.zeros(tq.exl3_moe_workspace_size(c.T, c.topk, c.E, d["w13"], d["w2"]), dtype=torch.uint8,
                     device="cuda")
    y1 = tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws).clone()
    y2 = tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], d["w13"], d["w2"], c.E, workspace_buf=ws).clone()
    assert torch.equal(y1, y2)
    assert tq.exl3_check_device_error(ws) == 0
    counters = host(ws[256:256 + 4 * 1024]).view(np.int32)
    assert np.all(counters == 0)
    assert_close(host(y1).astype(np.float64), _oracle(c), f"moe few tokens T{T} E{E} K{K}/{K2}")

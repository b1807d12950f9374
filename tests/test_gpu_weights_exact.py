"""The weights every fast kernel contracts with, checked weight by weight.

Dequantised weights must be bit-exact to the oracle ("exl3xpu" README,
"Correctness").  exl3_decode_tile is compared directly in test_gpu_linear.py;
the kernels below never write their weights out, so they are checked here:

* The prefill GEMM's transposed fp16 weights (the reconstruct kernel's
  workspace) and the int8 variant's integer weight codes are read back from
  the workspace and compared bit for bit with the oracle.
* The fused kernels (the M = 1 GEMV, its grouped form behind the fused
  shards, and the small-M tensor-core kernel whose decoder the grouped
  expert kernels share) are probed one input row at a time.  With svh = 1
  and x = suh . H[:, j] on the 128-block of input j (zero elsewhere), the
  input transform gives x' = 2^3.5 e_j, so y' = x'_j W[j, :] and the block
  Hadamard of the fp32 output gives back row j of the weights the kernel
  used.  It must equal (B - 510) sigma, B the oracle's byte sum of each
  weight's state, within fp32 rounding (one codebook step is sigma = 0.0068,
  so a weight decoded from a wrong state, window or tile fails), and the
  oracle's fp16 weight within its rounding.
* The grouped expert kernels get per-token probes: every token routed to one
  expert with weight 1 and an input that is a one-hot probe of the gate and
  up projections (both given the same suh), so each token's output depends
  on one row of that expert's gate and up weights; outputs are compared per
  token with the oracle.
"""
import functools

import numpy as np
import pytest
import scipy.linalg
import torch

import exl3_synth as synth
import oracle
import trellis_quantized_gb300 as tq
from gpu_util import REL_L2, dev, host

pytestmark = pytest.mark.gpu

ALIGN = 256
CTRL_BYTES = 256
COUNTER_BYTES = 8192 * 4
DATA_OFF = CTRL_BYTES + COUNTER_BYTES          # first data byte of every workspace
X_PRIME_F32 = float(np.float32(128.0) * np.float32(2.0 ** -3.5))   # x'_j of a probe in fp32
X_PRIME_F16 = float(np.float16(X_PRIME_F32))                       # ... rounded to fp16
W_TOL = 2e-5                                   # fp32 rounding of y' and of the output transform


def _align(v):
    return (v + ALIGN - 1) // ALIGN * ALIGN


@functools.lru_cache(maxsize=1)
def _bytesum():
    return oracle.bytesum_table()


def _exact_rows(trellis, K, rows):
    """(B - 510) sigma of input rows `rows` (float64 [len(rows), n]) and the
    oracle's fp16 weights of the same rows."""
    kt, nt = trellis.shape[:2]
    table = _bytesum()
    sigma = oracle.mul1_sigma()
    B = np.empty((len(rows), nt * 16), dtype=np.int64)
    states = {}
    for i, j in enumerate(rows):
        tk, r = divmod(int(j), 16)
        if tk not in states:
            states[tk] = [oracle.tile_states(trellis[tk, tn], K) for tn in range(nt)]
        for tn in range(nt):
            B[i, 16 * tn:16 * tn + 16] = table[states[tk][tn][16 * r:16 * r + 16]]
    W16 = oracle.reconstruct(trellis, kt * 16, nt * 16, K)[np.asarray(rows)].astype(np.float64)
    return (B - 510) * sigma, W16


def _probe_x(suh, rows):
    """x [len(rows), k] fp16: row m is the one-hot probe of input j = rows[m]."""
    H = scipy.linalg.hadamard(128)
    x = np.zeros((len(rows), suh.size), dtype=np.float16)
    for m, j in enumerate(rows):
        b, i = divmod(int(j), 128)
        x[m, 128 * b:128 * b + 128] = (suh[128 * b:128 * b + 128].astype(np.float64) * H[:, i]).astype(np.float16)
    return x


def _recover(y32, xj):
    """Row of Hadamard-domain weights from an fp32 output row (svh = 1)."""
    y = np.asarray(y32, dtype=np.float64).reshape(-1, 128)
    H = scipy.linalg.hadamard(128) / np.sqrt(128.0)
    return (y @ H).reshape(-1) / xj


def _assert_rows(Wrec, exact, W16, what):
    err = np.abs(Wrec - exact)
    assert err.max() <= W_TOL, f"{what}: max |W - (B-510) sigma| = {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert np.all(np.abs(Wrec - W16) <= np.abs(W16) * 2.0 ** -11 + W_TOL), f"{what}: beyond fp16 rounding"


def _probe_rows(kt, rng, extra=8):
    """All 16 rows of the first and last tile rows plus a seeded sample."""
    rows = list(range(16)) + list(range(16 * (kt - 1), 16 * kt))
    rows += sorted(rng.choice(16 * kt, size=extra, replace=False).tolist())
    return sorted(set(rows))


# ------------------------------------------------------- written weights --

def test_prefill_reconstructed_weights_bit_exact_config4():
    """M = 4096, k = 5120, n = 17408, K = 4: the transposed fp16 weights the
    tcgen05 GEMM reads (workspace: x' [M][k] fp16, then Wt [n][k] fp16)."""
    c = synth.config4()
    need = tq.exl3_linear_workspace_size(c.M, c.k, c.n, c.K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    tq.exl3_linear(dev(c.x), dev(c.trellis), dev(c.suh), dev(c.svh), c.K, workspace_buf=ws)
    torch.cuda.synchronize()
    wt_off = _align(DATA_OFF + 2 * c.M * c.k)
    assert wt_off + 2 * c.k * c.n <= need
    wt = host(ws[wt_off:wt_off + 2 * c.k * c.n]).view(np.uint16).reshape(c.n, c.k)
    ref = oracle.reconstruct(c.trellis, c.k, c.n, c.K).view(np.uint16)
    assert np.array_equal(wt, ref.T), "transposed reconstruct differs from the oracle"


@pytest.mark.parametrize("K", [2, 4, 7])
def test_int8_weight_codes_bit_exact(K):
    """The int8 variant's weight codes (integer-valued fp16 q_w [n][k] after
    the integer-valued q_x [M][k] in the workspace) against the oracle's
    q_w = RNE(v 127 / 3.453125)."""
    c = synth.linear_case(30, K, 200, 1024, 640, K)
    need = tq.exl3_linear_int8_workspace_size(c.M, c.k, c.n, c.K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    tq.exl3_linear_int8(dev(c.x), dev(c.trellis), dev(c.suh), dev(c.svh), K, workspace_buf=ws)
    torch.cuda.synchronize()
    off = _align(DATA_OFF + 2 * c.M * c.k)
    qw = host(ws[off:off + 2 * c.k * c.n]).view(np.float16).reshape(c.n, c.k)
    ref = oracle.quant_weights(oracle.reconstruct(c.trellis, c.k, c.n, K))
    assert np.array_equal(qw.astype(np.float64), ref.T.astype(np.float64))


# ------------------------------------------------------- one-hot probes --

def _probe_case(sub, k, n, K):
    c = synth.linear_case(31, sub, 1, k, n, K)
    c.svh = np.ones(n, dtype=np.float16)
    return c


@pytest.mark.parametrize("K", range(1, 9))
def test_gemv_decoder_one_hot_probes(K):
    """M = 1 GEMV (k = 512, n = 640: column blocks shared by several CTAs)."""
    c = _probe_case(K, 512, 640, K)
    rows = _probe_rows(c.k // 16, np.random.default_rng(K))
    exact, W16 = _exact_rows(c.trellis, K, rows)
    t, suh, svh = dev(c.trellis), dev(c.suh), dev(c.svh)
    xs = _probe_x(c.suh, rows)
    for i, j in enumerate(rows):
        y = tq.exl3_linear(dev(xs[i:i + 1]), t, suh, svh, K, out_dtype=tq.EXL3_OUT_F32)
        _assert_rows(_recover(host(y)[0], X_PRIME_F32), exact[i], W16[i], f"GEMV K{K} row {j}")


def test_gemv_decoder_one_hot_probes_config3_width():
    """The mixed-width layer's shape at K = 4 (k = n = 4096)."""
    c = _probe_case(100, 4096, 4096, 4)
    rows = _probe_rows(c.k // 16, np.random.default_rng(100), extra=4)
    exact, W16 = _exact_rows(c.trellis, 4, rows)
    t, suh, svh = dev(c.trellis), dev(c.suh), dev(c.svh)
    xs = _probe_x(c.suh, rows)
    for i, j in enumerate(rows):
        y = tq.exl3_linear(dev(xs[i:i + 1]), t, suh, svh, 4, out_dtype=tq.EXL3_OUT_F32)
        _assert_rows(_recover(host(y)[0], X_PRIME_F32), exact[i], W16[i], f"GEMV cfg3 width row {j}")


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("M", [16, 128])
def test_small_m_decoder_one_hot_probes(K, M):
    """The fused tensor-core kernel (2 <= M <= 128), whose item decoder the
    grouped expert kernels share: every input row of k = 512, M probes per
    call (x' rounded to fp16 there)."""
    c = _probe_case(200 + K, 512, 384, K)
    rows = list(range(c.k))
    exact, W16 = _exact_rows(c.trellis, K, rows)
    t, suh, svh = dev(c.trellis), dev(c.suh), dev(c.svh)
    xs = _probe_x(c.suh, rows)
    for s in range(0, len(rows), M):
        y = host(tq.exl3_linear(dev(xs[s:s + M]), t, suh, svh, K, out_dtype=tq.EXL3_OUT_F32))
        for m in range(y.shape[0]):
            _assert_rows(_recover(y[m], X_PRIME_F16), exact[s + m], W16[s + m], f"small-M K{K} M{M} row {rows[s + m]}")


@pytest.mark.parametrize("K", [3, 4, 8])
def test_grouped_gemv_decoder_one_hot_probes(K):
    """The grouped GEMV (the few-token expert path's kernel) through fused
    shards of one input: three shards with a common suh, each probed row
    recovered from every shard's output."""
    S, k, n = 3, 512, 384
    cs = [_probe_case(300 + 10 * K + s, k, n, K) for s in range(S)]
    suh = cs[0].suh
    tr = np.stack([c.trellis for c in cs])
    t = dev(tr)
    su = dev(np.stack([suh] * S))
    sv = dev(np.ones((S, n), dtype=np.float16))
    rows = _probe_rows(k // 16, np.random.default_rng(300 + K))
    xs = _probe_x(suh, rows)
    exact = [_exact_rows(cs[s].trellis, K, rows) for s in range(S)]
    for i, j in enumerate(rows):
        y = host(tq.exl3_linear_shards(dev(xs[i:i + 1]), t, su, sv, K, out_dtype=tq.EXL3_OUT_F32))
        for s in range(S):
            _assert_rows(_recover(y[s, 0], X_PRIME_F32), exact[s][0][i], exact[s][1][i], f"shard {s} K{K} row {j}")


def test_shards_of_different_widths_decoder_one_hot_probes():
    """gemv_shards_kernel: one trellis map per shard, widths 512 + 128 + 384."""
    K, k, widths = 5, 384, (512, 128, 384)
    cs = [_probe_case(400 + s, k, w, K) for s, w in enumerate(widths)]
    suh = cs[0].suh
    t = dev(np.concatenate([c.trellis.reshape(-1) for c in cs]))
    su = dev(np.stack([suh] * len(widths)))
    sv = dev(np.ones(sum(widths), dtype=np.float16))
    rows = _probe_rows(k // 16, np.random.default_rng(400))
    xs = _probe_x(suh, rows)
    exact = [_exact_rows(c.trellis, K, rows) for c in cs]
    for i, j in enumerate(rows):
        y = host(tq.exl3_linear_shards_var(dev(xs[i:i + 1]), t, su, sv, widths, K, out_dtype=tq.EXL3_OUT_F32))
        off = 0
        for s, w in enumerate(widths):
            _assert_rows(_recover(y[off:off + w], X_PRIME_F32), exact[s][0][i], exact[s][1][i],
                         f"var shard {s} row {j}")
            off += w


# ------------------------------------------------ grouped expert probes --

@pytest.mark.parametrize("T,K,K2", [(96, 2, 5), (64, 4, 4), (12, 3, 6)])
def test_grouped_expert_per_token_probes(T, K, K2):
    """Top-1 routing with weight 1 over 4 experts, token t a one-hot probe of
    gate/up input row j_t: T = 96 and 64 take the 128-row tile kernels,
    T = 12 the few-token grouped GEMV.  Each token's output must match the
    oracle on its own (rel-L2 per token), so a wrong row of any expert's gate
    or up weights, or a wrong down weight row, fails its token."""
    E, hidden, inter = 4, 512, 256
    c = synth.moe_case(58, T * 10 + K, T, E=E, topk=1, hidden=hidden, inter=inter, K=K, K2=K2)
    c.w13.suh[:, 1] = c.w13.suh[:, 0]                       # gate and up share suh: one probe serves both
    c.ids[:, 0] = np.arange(T, dtype=np.int32) % E
    c.weights[:] = 1.0
    rows = np.random.default_rng(58 + T).permutation(hidden)[:T]
    for t in range(T):
        c.x[t] = _probe_x(c.w13.suh[c.ids[t, 0], 0], [rows[t]])[0]
    d = {key: dev(v) for key, v in dict(x=c.x, ids=c.ids, w=c.weights, t13=c.w13.trellis, s13=c.w13.suh,
                                         v13=c.w13.svh, t2=c.w2.trellis, s2=c.w2.suh, v2=c.w2.svh).items()}
    w13 = tq.expert_proj(d["t13"], d["s13"], d["v13"], K)
    w2 = tq.expert_proj(d["t2"], d["s2"], d["v2"], K2)
    y = host(tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], w13, w2, E, out_dtype=tq.EXL3_OUT_F32)).astype(np.float64)
    ref = oracle.moe(c.x, c.ids, c.weights, c.w13.trellis, c.w13.suh, c.w13.svh, K, c.w2.trellis, c.w2.suh,
                     c.w2.svh, K2)
    for t in range(T):
        rel = np.linalg.norm(y[t] - ref[t]) / np.linalg.norm(ref[t])
        assert rel <= REL_L2, f"token {t} (expert {c.ids[t, 0]}, probe row {rows[t]}): rel-L2 {rel:.2e}"

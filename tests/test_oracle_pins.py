"""Pins of the CPU oracle to facts other than itself (runs without a GPU).

Each test ties one part of the oracle to something independent: hand-derived
worked examples (tests/golden), the bound the pages print, library routines
(numpy's binary16 conversion, scipy's Sylvester Hadamard, numpy integer
matmul, scipy's logistic function), closed forms and structural invariants.
Sources: "exl3xpu" README ("Prefill: int8 linears and oneDNN fused
attention", "MoE (routed experts)", "Adding a model"); "Bringing EXL3 Trellis
Quantization to 35B MoE on Intel Arc 140V" (sections 1 and 2.B); "EXL3
checkpoints on the native engine (tracker) #832".
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import exl3_synth as synth
import oracle
from tie_rows import tie_rows

BOUND = 3.453125
H128 = scipy.linalg.hadamard(128).astype(np.float64)   # Sylvester, natural order


def block_hadamard(dim):
    """Orthonormal block-diagonal Hadamard of size dim (128-blocks), from scipy."""
    Hn = H128 / np.sqrt(128.0)
    return scipy.linalg.block_diag(*([Hn] * (dim // 128)))


# ----------------------------------------------------------------- binary16 --

def test_f16_decode_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        # exact midpoints between neighbouring fp16 values (ties to even)
        (np.arange(0, 4000, dtype=np.float64) + 0.5) * 2.0 ** -10,
        (np.arange(0, 2000, dtype=np.float64) + 0.5) * 2.0 ** -24,   # subnormal ties
        [65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 6.0e-8, 2.0 ** -25, 0.0, -0.0],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_f16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- codebook --

def test_codebook_worked_examples(golden):
    for state, bsum, bits, value in golden("codebook_worked.txt"):
        s = int(state, 16)
        assert oracle.mul1_bytesum(s) == int(bsum)
        assert oracle.mul1_value_bits(s) == int(bits, 16)
        assert oracle.f16_to_f64(int(bits, 16)) == float(value)


def test_codebook_bound_bruteforce_all_states():
    """Every value satisfies |v| <= 3.453125 and the bound is attained (at s=0)."""
    v = oracle.codebook_table().astype(np.float64)
    assert np.max(np.abs(v)) == BOUND
    assert v[0] == -BOUND
    sigma = oracle.mul1_sigma()
    assert sigma * 2 ** 18 == 1775.0                       # sigma is an fp16 value
    assert np.float16(510 * sigma) == np.float16(BOUND)    # the bound fixes sigma
    assert np.float16(510 * 1.0 / 147.8) != np.float16(BOUND)  # unit-variance scale would not


def test_codebook_is_fp16_of_affine_bytesum_and_near_gaussian():
    b = oracle.bytesum_table()
    v = oracle.codebook_table().astype(np.float64)
    # sum of four uniform bytes: mean 510, std sqrt(4*(256^2-1)/12) = 147.80
    assert abs(b.mean() - 510.0) < 1.0
    assert abs(b.std() - np.sqrt(4 * (256 ** 2 - 1) / 12)) < 0.5
    assert b.min() >= 0 and b.max() <= 1020
    # v depends on the state only through B, monotonically, with v = 0 at B = 510
    order = np.argsort(b, kind="stable")
    assert np.all(np.diff(v[order]) >= 0)
    assert np.all(v[b == 510] == 0.0)
    # the value of each B is the fp16 rounding of (B - 510) * sigma (numpy's rounding)
    sigma = oracle.mul1_sigma()
    assert np.array_equal(v, ((b - 510) * sigma).astype(np.float16).astype(np.float64))
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


# ------------------------------------------------------------------ trellis --

def test_single_bit_trellis_states(golden):
    for row in golden("trellis_single_bit.txt"):
        K, b = int(row[0]), int(row[1])
        words = np.zeros(16 * K, dtype=np.uint16)
        words[b // 16] = 1 << (b % 16)
        expect = np.zeros(256, dtype=np.uint16)
        for item in row[2:]:
            p, s = item.split(":")
            expect[int(p)] = int(s, 16)
        assert np.array_equal(oracle.tile_states(words, K), expect), f"K={K} bit={b}"


@pytest.mark.parametrize("K", range(1, 9))
def test_shift_register_property(K):
    """Consecutive states overlap in 16-K bits, including the wrap 255 -> 0."""
    rng = np.random.default_rng(100 + K)
    mask = (1 << (16 - K)) - 1
    for _ in range(20):
        words = rng.integers(0, 1 << 16, size=16 * K, dtype=np.uint16)
        s = oracle.tile_states(words, K).astype(np.int64)
        nxt = np.roll(s, -1)
        assert np.array_equal(s >> K, nxt & mask)
        # the K fresh bits of state p+1 are stream bits [pK+16, pK+16+K)
        bits = np.unpackbits(words.view(np.uint8), bitorder="little")
        L = 256 * K
        for p in (0, 100, 255):
            fresh = sum(int(bits[(p * K + 16 + j) % L]) << j for j in range(K))
            assert (int(nxt[p]) >> (16 - K)) == fresh


@pytest.mark.parametrize("K", [1, 4, 8])
def test_special_trellises(K):
    zero = np.zeros(16 * K, dtype=np.uint16)
    ones = np.full(16 * K, 0xFFFF, dtype=np.uint16)
    assert np.all(oracle.tile_states(zero, K) == 0)
    assert np.all(oracle.tile_states(ones, K) == 0xFFFF)
    W0 = oracle.reconstruct(np.zeros((2, 2, 16 * K), np.uint16), 32, 32, K)
    assert np.all(W0.astype(np.float64) == -BOUND)


def test_tile_and_intra_tile_placement():
    # tile (tk=1, tn=0) all ones, every other tile zero -> rows 16..31, cols 0..15
    K = 2
    t = np.zeros((2, 2, 16 * K), dtype=np.uint16)
    t[1, 0, :] = 0xFFFF
    W = oracle.reconstruct(t, 32, 32, K).view(np.uint16)
    expect = np.full((32, 32), 0xC2E8, dtype=np.uint16)
    expect[16:32, 0:16] = 0x34A9
    assert np.array_equal(W, expect)
    # K=8, stream bit 136 of tile (0,1): p=16 -> state 0x100, p=17 -> state 0x001
    K = 8
    t = np.zeros((1, 2, 16 * K), dtype=np.uint16)
    t[0, 1, 8] = 1 << 8
    W = oracle.reconstruct(t, 16, 32, K).view(np.uint16)
    expect = np.full((16, 32), 0xC2E8, dtype=np.uint16)
    expect[1, 16 + 0] = 0xBC41   # p = 16 = row 1, column 0 of tile tn=1
    expect[1, 16 + 1] = 0x1EEF   # p = 17 = row 1, column 1
    assert np.array_equal(W, expect)


def test_reconstruct_rejects_bad_arguments():
    t = np.zeros((8, 8, 16), dtype=np.uint16)
    for K in (0, 9):
        with pytest.raises(ValueError):
            oracle.reconstruct(t, 128, 128, K)
    with pytest.raises(ValueError):
        oracle.linear(np.zeros((1, 120), np.float16), np.zeros((7, 8, 16), np.uint16),
                      np.ones(120, np.float16), np.ones(128, np.float16), 1)


# ----------------------------------------------------------------- Hadamard --

def test_fwht_is_sylvester_hadamard():
    cols = np.stack([oracle.fwht128_f64(np.eye(128)[j]) for j in range(128)], axis=1)
    assert np.array_equal(cols, H128)
    assert np.array_equal(cols @ cols.T, 128.0 * np.eye(128))
    i = np.arange(128)
    pop = np.array([[bin(a & b).count("1") for b in i] for a in i])
    assert np.array_equal(cols, (-1.0) ** pop)


def test_fwht_matches_matrix_product():
    rng = np.random.default_rng(7)
    for _ in range(10):
        v = rng.integers(-1000, 1000, 128).astype(np.float64)
        assert np.array_equal(oracle.fwht128_f64(v), H128 @ v)
        assert np.array_equal(oracle.fwht128_f32(v.astype(np.float32)).astype(np.float64), H128 @ v)
        w = rng.standard_normal(128)
        assert np.max(np.abs(oracle.fwht128_f64(w) - H128 @ w)) < 1e-12
    Hn = H128 / np.sqrt(128)
    assert np.max(np.abs(Hn @ Hn - np.eye(128))) < 1e-14


U32 = 2.0 ** -24                                       # binary32 unit roundoff
C_RHT = 2.0 ** -3.5                                    # 1/sqrt(128)


def test_rht_in_f32_exact_sums_are_one_rounding_from_the_definition():
    # With exact butterflies the only errors are fp32(2^-3.5) and the final
    # product, so every x' is within 2u (relative) of S * 2^-3.5, and a zero
    # sum stays exactly zero. A wrong scale, sign or position fails this.
    x, suh, S = tie_rows()
    a32 = oracle.rht_in_f32(x, suh).astype(np.float64)
    exact = S * C_RHT
    assert np.array_equal(a32 == 0, S == 0)
    assert np.all(np.abs(a32 - exact) <= (2 * U32 + U32 * U32) * np.abs(exact))


def test_rht_in_f32_within_the_pairwise_summation_bound():
    # Forward error of a 7-level butterfly tree in binary32 (pairwise
    # summation, Higham's gamma_7 bound) plus the two roundings of the scale:
    #   |x'32 - x'| <= c * gamma_7 * (1 + 3u) * sum_j |x_j suh_j| + (2u + u^2) |x'|
    # per element, with x' the float64 transform pinned above.
    case = synth.linear_case(90, 0, 3, 512, 128, 2, outlier_rows=0.3)
    a64 = oracle.rht_in_f64(case.x, case.suh)
    a32 = oracle.rht_in_f32(case.x, case.suh).astype(np.float64)
    v = np.abs(case.x.astype(np.float64) * case.suh.astype(np.float64))
    l1 = v.reshape(3, 4, 128).sum(axis=2).repeat(128, axis=1)
    gamma7 = 7 * U32 / (1 - 7 * U32)
    bound = C_RHT * gamma7 * (1 + 3 * U32) * l1 + (2 * U32 + U32 * U32) * np.abs(a64)
    assert np.all(np.abs(a32 - a64) <= bound * (1 + 1e-9) + 1e-300)
    # the bound is tight enough to matter: it sits far below the 1e-5 level
    assert np.max(bound) < 1e-5 * np.max(np.abs(a64))


# ------------------------------------------------------------ the linear -----

@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("k,n", [(128, 128), (256, 128), (128, 256), (256, 256)])
def test_transform_form_bruteforce(K, k, n):
    """y == x @ (diag(suh) Hn W Hn diag(svh)) with explicit scipy matrices."""
    case = synth.linear_case(91, K * 10 + k // 128 + 4 * (n // 128), 3, k, n, K)
    W = oracle.reconstruct(case.trellis, k, n, K).astype(np.float64)
    Weff = (np.diag(case.suh.astype(np.float64)) @ block_hadamard(k) @ W
            @ block_hadamard(n) @ np.diag(case.svh.astype(np.float64)))
    ref = case.x.astype(np.float64) @ Weff
    got = oracle.linear(case.x, case.trellis, case.suh, case.svh, K)
    assert np.max(np.abs(got - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("K,k,n", [(2, 128, 256), (4, 256, 128), (7, 256, 256)])
def test_bias_is_the_offset_of_the_affine_map(K, k, n):
    """With a bias, y == x @ W_eff + b (the textbook affine map, explicit scipy
    matrices): the bias is added per output feature after svh, outside the
    Hadamard domain.  Adding it before the output transform would spread it
    over each 128-block and fail this."""
    case = synth.linear_case(91, 100 + K, 3, k, n, K)
    b = synth.bias_for(K, n)
    W = oracle.reconstruct(case.trellis, k, n, K).astype(np.float64)
    Weff = (np.diag(case.suh.astype(np.float64)) @ block_hadamard(k) @ W
            @ block_hadamard(n) @ np.diag(case.svh.astype(np.float64)))
    ref = case.x.astype(np.float64) @ Weff + b.astype(np.float64)[None, :]
    got = oracle.linear(case.x, case.trellis, case.suh, case.svh, K, bias=b)
    assert np.max(np.abs(got - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))
    # the dequantised-weight form takes the same bias
    got_w = oracle.linear_w(case.x, oracle.reconstruct(case.trellis, k, n, K), case.suh, case.svh, bias=b)
    assert np.max(np.abs(got_w - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))
    with pytest.raises(ValueError):
        oracle.linear(case.x, case.trellis, case.suh, case.svh, K, bias=b[:-1])


def test_one_hot_probe_recovers_a_weight_row():
    """x = suh * (H e_j) gives x' = sqrt(128) e_j, so Hn y = sqrt(128) W[j, :] (svh = 1)."""
    K, k, n = 3, 256, 256
    case = synth.linear_case(92, 0, 1, k, n, K)
    W = oracle.reconstruct(case.trellis, k, n, K).astype(np.float64)
    svh = np.ones(n, np.float16)
    for j in (0, 5, 129, 255):
        e = np.zeros(k)
        e[j] = 1.0
        x = (block_hadamard(k) @ e * np.sqrt(128.0) * case.suh.astype(np.float64)).astype(np.float16)
        y = oracle.linear(x[None, :], case.trellis, case.suh, svh, K)[0]
        row = block_hadamard(n) @ y / np.sqrt(128.0)
        assert np.max(np.abs(row - W[j])) < 1e-9


@pytest.mark.parametrize("K", [2, 5])
def test_constant_state_closed_form(K):
    """All-ones words give one state c everywhere, so W = v(c) and y' = v(c) sum(x') in
    every column; H of a constant block is 128 * e_0, which leaves one spike per block:
    y[128b] = svh[128b] * 128 * v(c) * sum_b' x[128b'] suh[128b'], every other y = 0."""
    k, n = 384, 256
    case = synth.linear_case(93, K, 2, k, n, K)
    t = np.full_like(case.trellis, 0xFFFF)
    vc = oracle.f16_to_f64(oracle.mul1_value_bits(0xFFFF))
    y = oracle.linear(case.x, t, case.suh, case.svh, K)
    xs = case.x.astype(np.float64) * case.suh.astype(np.float64)
    for r in range(2):
        s = xs[r, 0::128].sum()
        expect = np.zeros(n)
        expect[0::128] = case.svh.astype(np.float64)[0::128] * 128.0 * vc * s
        assert np.max(np.abs(y[r] - expect)) <= 1e-9 * max(1.0, np.abs(expect).max())


# --------------------------------------------------------------------- int8 --

def test_int8_weight_quant_worked_examples(golden):
    for bits, q in golden("int8_weight_quant.txt"):
        assert oracle.quant_weight(int(bits, 16)) == int(q)


def test_int8_weight_quant_range_over_codebook():
    v = oracle.codebook_table()
    q = oracle.quant_weights(v).astype(np.int64)
    assert q.min() == -127 and np.abs(q).max() <= 127
    # q_w is the nearest integer to v / s_w (within one half, ties aside)
    sw = BOUND / 127.0
    assert np.max(np.abs(q - v.astype(np.float64) / sw)) <= 0.5 + 1e-9


def test_int8_activation_quant_properties():
    case = synth.linear_case(94, 0, 6, 512, 128, 4, outlier_rows=0.2)
    x = case.x.copy()
    x[3] = 0                                     # a zero row -> q = 0, a = 0
    q, a = oracle.quant_act(x, case.suh)
    xr = oracle.rht_in_f32(x, case.suh).astype(np.float64)
    assert a[3] == 0 and np.all(q[3] == 0)
    for r in (0, 1, 2, 4, 5):
        amax = np.abs(xr[r]).max()
        assert np.float32(amax / 127) == a[r]
        assert np.abs(q[r]).max() == 127
        assert np.max(np.abs(q[r] * np.float64(a[r]) - xr[r])) <= 0.5 * a[r] * (1 + 1e-5)


def _rne(t):
    """Round-half-even of exact rationals (Fractions) to integers."""
    out = []
    for f in t:
        lo = f.numerator // f.denominator
        rem = f - lo
        out.append(lo + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2) else 0))
    return np.array(out, dtype=np.float64)


def test_int8_activation_quant_reading_is_multiply_by_fp32_inverse():
    # Which of three plausible roundings the int8 path takes is a reading of
    # "Prefill: int8 linears" (per-row absmax scale, codes in [-127, 127]):
    #   (a) RNE(fp32(x' * fp32(127 / amax)))   -- this library's reading
    #   (b) RNE(fp32(x' / a_r)), a_r = fp32(amax / 127)
    #   (c) RNE of the exact rational x' * 127 / amax
    # They agree except near halfway points. The rows of tie_rows put 127
    # elements exactly at halfway points of the definition, where fp32
    # rounding decides; the oracle must match (a) everywhere and differ from
    # (b) and (c) at many of these elements, so that the pin separates them.
    x, suh, S = tie_rows()
    q, a = oracle.quant_act(x, suh)
    xr = oracle.rht_in_f32(x, suh)
    amax = np.abs(xr).max(axis=1)
    assert np.array_equal(amax, np.abs(xr[:, 0]))
    ties = S * 127 % 508 == 254                        # 127 S / 508 = m + 1/2
    assert ties.sum() == 127
    qa = np.rint(xr * (np.float32(127) / amax)[:, None]).astype(np.float64)
    qb = np.rint(xr / (amax / np.float32(127))[:, None]).astype(np.float64)
    qc = np.array([_rne([Fraction(float(t)) * 127 / Fraction(float(m)) for t in row])
                   for row, m in zip(xr, amax)])
    assert np.abs(qa).max() <= 127
    assert np.array_equal(q.astype(np.float64), qa)
    assert np.array_equal(qa[~ties], qc[~ties])        # off the ties all agree
    assert (qa != qb)[ties].sum() >= 20
    assert (qa != qc)[ties].sum() >= 20
    assert np.array_equal(a, (amax / np.float32(127)).astype(np.float32))


def test_int8_accumulators_and_output():
    case = synth.linear_case(95, 0, 5, 512, 256, 4)
    res = oracle.linear_int8(case.x, case.trellis, case.suh, case.svh, 4)
    W = oracle.reconstruct(case.trellis, 512, 256, 4)
    assert np.array_equal(res["qw"], oracle.quant_weights(W))
    q, a = oracle.quant_act(case.x, case.suh)
    assert np.array_equal(res["qx"], q) and np.array_equal(res["row_scale"], a)
    acc = res["qx"].astype(np.int64) @ res["qw"].astype(np.int64)
    assert np.array_equal(res["acc"], acc)
    assert np.abs(acc).max() < 2 ** 31
    # the int8 output is the fp output up to quantisation error (about 1%)
    yf = oracle.linear(case.x, case.trellis, case.suh, case.svh, 4)
    rel = np.linalg.norm(res["y"] - yf) / np.linalg.norm(yf)
    assert 1e-4 < rel < 3e-2
    # dequantisation uses the per-row scale and the static weight scale
    yp = acc * a[:, None].astype(np.float64) * (BOUND / 127.0)
    ref = yp @ block_hadamard(256) * case.svh.astype(np.float64)
    assert np.max(np.abs(res["y"] - ref)) <= 1e-9 * np.abs(ref).max()
    # an output bias is added to the dequantised result, per output feature
    b = synth.bias_for(95, 256)
    resb = oracle.linear_int8(case.x, case.trellis, case.suh, case.svh, 4, bias=b)
    assert np.array_equal(resb["acc"], res["acc"])
    refb = ref + b.astype(np.float64)[None, :]
    assert np.max(np.abs(resb["y"] - refb)) <= 1e-9 * np.abs(refb).max()


# ---------------------------------------------------------------------- MoE --

def _moe_small(sub, T=3, E=4, topk=2, hidden=256, inter=128, K=3):
    return synth.moe_case(96, sub, T, E=E, topk=topk, hidden=hidden, inter=inter, K=K)


def _dense_expert(c, e):
    """Dense effective matrices (gate, up, down) of expert e via scipy Hadamards."""
    h, i, K = c.hidden, c.inter, c.K
    mats = []
    for proj, slot, k, n in ((c.w13, 0, h, i), (c.w13, 1, h, i), (c.w2, 0, i, h)):
        W = oracle.reconstruct(proj.trellis[e, slot], k, n, proj.K).astype(np.float64)
        mats.append(np.diag(proj.suh[e, slot].astype(np.float64)) @ block_hadamard(k) @ W
                    @ block_hadamard(n) @ np.diag(proj.svh[e, slot].astype(np.float64)))
    return mats


def test_moe_matches_dense_composition():
    c = _moe_small(0)
    got = oracle.moe(c.x, c.ids, c.weights, c.w13.trellis, c.w13.suh, c.w13.svh, c.K,
                     c.w2.trellis, c.w2.suh, c.w2.svh, c.K)
    ref = np.zeros((c.T, c.hidden))
    for t in range(c.T):
        xt = c.x[t].astype(np.float64)
        for s in range(c.topk):
            G, U, D = _dense_expert(c, int(c.ids[t, s]))
            g, u = xt @ G, xt @ U
            h = g * scipy.special.expit(g) * u
            ref[t] += float(c.weights[t, s]) * (h @ D)
    assert np.max(np.abs(got - ref)) <= 1e-9 * np.abs(ref).max()


def test_moe_weight_on_down_output_and_slot_symmetry():
    c = _moe_small(1, T=2, topk=3)
    args = (c.w13.trellis, c.w13.suh, c.w13.svh, c.K, c.w2.trellis, c.w2.suh, c.w2.svh, c.K)
    base = oracle.moe(c.x, c.ids, c.weights, *args)
    perm = [2, 0, 1]
    permuted = oracle.moe(c.x, c.ids[:, perm], c.weights[:, perm], *args)
    assert np.max(np.abs(base - permuted)) <= 1e-12 * np.abs(base).max()
    # all slots on one expert with weights summing to one == that expert's chain
    ids = np.full_like(c.ids, 2)
    w = np.array([[0.5, 0.25, 0.25]] * c.T, dtype=np.float32)
    one = oracle.moe(c.x, ids, w, *args)
    single = oracle.moe(c.x, ids[:, :1], np.ones((c.T, 1), np.float32), *args)
    assert np.max(np.abs(one - single)) <= 1e-12 * np.abs(single).max()
    # scaling the weight scales the output linearly (weight is not on the input)
    half = oracle.moe(c.x, ids[:, :1], np.full((c.T, 1), 0.5, np.float32), *args)
    assert np.max(np.abs(2 * half - single)) <= 1e-12 * np.abs(single).max()


def test_moe_token_sampling_matches_full():
    c = _moe_small(2, T=5)
    args = (c.w13.trellis, c.w13.suh, c.w13.svh, c.K, c.w2.trellis, c.w2.suh, c.w2.svh, c.K)
    full = oracle.moe(c.x, c.ids, c.weights, *args)
    part = oracle.moe(c.x, c.ids, c.weights, *args, tokens=[4, 1])
    assert np.array_equal(part, full[[4, 1]])


# ------------------------------------------------ MoE with per-expert widths --

def _mixed_dense_expert(c, e):
    """Dense effective (gate, up, down) of expert e of a mixed-width case: the
    expert's tensors are cut out of the flat arenas at offsets summed here
    from the widths, then dequantised and wrapped in scipy Hadamards."""
    h, i = c.hidden, c.inter
    mats = []
    for proj, slot, k, n in ((c.w13, 0, h, i), (c.w13, 1, h, i), (c.w2, 0, i, h)):
        sizes = [proj.nslots * (k // 16) * (n // 16) * 16 * int(w) for w in proj.K]
        start = int(np.sum(sizes[:e])) + slot * sizes[e] // proj.nslots
        K = int(proj.K[e])
        words = proj.trellis[start:start + (k // 16) * (n // 16) * 16 * K].reshape(k // 16, n // 16, 16 * K)
        W = oracle.reconstruct(words, k, n, K).astype(np.float64)
        mats.append(np.diag(proj.suh[e, slot].astype(np.float64)) @ block_hadamard(k) @ W
                    @ block_hadamard(n) @ np.diag(proj.svh[e, slot].astype(np.float64)))
    return mats


def test_moe_mixed_widths_match_dense_composition():
    """Per-expert widths: every expert decoded at its own K from its own place
    in the packed arena, composed with scipy's logistic function."""
    c = synth.mixed_moe_case(97, 0, 3, [1, 3, 8, 3], [2, 5, 4, 7], topk=2, hidden=256, inter=128)
    got = oracle.moe_k(c.x, c.ids, c.weights, c.w13.trellis, c.w13.suh, c.w13.svh, c.w13.K,
                       c.w2.trellis, c.w2.suh, c.w2.svh, c.w2.K, c.inter)
    ref = np.zeros((c.T, c.hidden))
    for t in range(c.T):
        xt = c.x[t].astype(np.float64)
        for s_ in range(c.topk):
            G, U, D = _mixed_dense_expert(c, int(c.ids[t, s_]))
            g, u = xt @ G, xt @ U
            ref[t] += float(c.weights[t, s_]) * ((g * scipy.special.expit(g) * u) @ D)
    assert np.max(np.abs(got - ref)) <= 1e-9 * np.abs(ref).max()


def test_moe_mixed_with_equal_widths_is_the_uniform_definition():
    """Equal widths in the packed arena are the [E][nslots][k/16][n/16][16K]
    layout, so the two entry points must agree exactly."""
    c = _moe_small(5, T=4, E=5, topk=3, K=4)
    base = oracle.moe(c.x, c.ids, c.weights, c.w13.trellis, c.w13.suh, c.w13.svh, 4,
                      c.w2.trellis, c.w2.suh, c.w2.svh, 4)
    K = np.full(c.E, 4, dtype=np.int32)
    mixed = oracle.moe_k(c.x, c.ids, c.weights, c.w13.trellis.reshape(-1), c.w13.suh, c.w13.svh, K,
                         c.w2.trellis.reshape(-1), c.w2.suh, c.w2.svh, K, c.inter)
    assert np.array_equal(base, mixed)
    with pytest.raises(ValueError):
        oracle.moe_k(c.x, c.ids, c.weights, c.w13.trellis.reshape(-1)[:-16], c.w13.suh, c.w13.svh, K,
                     c.w2.trellis.reshape(-1), c.w2.suh, c.w2.svh, K, c.inter)

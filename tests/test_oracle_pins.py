"""Pins of the fp64 oracle to what the pages and mathematics fix.

Each test states the passage it follows. None of them re-types the oracle's
formula: they compare against printed values, closed forms, invariants,
brute force written a different way, or an independent high-precision route.
"""
import math
import os

import mpmath
import numpy as np
import pytest

import alibi_inputs as gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TAU_D = math.log(2.0 ** -126)


# ------------------------------------------------------------------ slopes

def test_slopes_printed_tables():
    # "ALiBi: Attention with Linear Biases", "Different heads, different distance
    # penalties": four heads -> 0.25, 0.0625, 0.015625, 0.00390625; eight heads ->
    # 0.5, 0.25, ..., 0.00390625; six heads -> the printed head/slope table.
    assert list(oracle.slopes(4)) == [0.25, 0.0625, 0.015625, 0.00390625]
    assert list(oracle.slopes(8)) == [0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.00390625]
    assert list(oracle.slopes(6)) == [0.25, 0.0625, 0.015625, 0.00390625, 0.5, 0.125]
    # dev.to "ALiBi: give a Transformer position sense...", head_slopes(8) output.
    assert list(oracle.slopes_f32(8)) == [0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.00390625]


@pytest.mark.parametrize("H,first,second,last", [
    (16, -0.5, -1.0, -8.0),     # BLOOM row of Table 1 ("When Attention Goes Blind", sec. 4)
    (64, -0.125, -0.25, -8.0),  # Falcon-RW row of Table 1
    (32, -0.25, -0.5, -8.0),    # MPT row of Table 1
])
def test_slopes_model_rows(H, first, second, last):
    m = oracle.slopes(H)
    assert m[0] == pytest.approx(2.0 ** first, rel=1e-15)
    assert m[1] == pytest.approx(2.0 ** second, rel=1e-15)
    assert m[-1] == pytest.approx(2.0 ** last, rel=1e-15)
    assert np.all(np.diff(m) < 0)


@pytest.mark.parametrize("H", [2, 4, 8, 16, 32, 64, 128])
def test_slope_ratio_power_of_two(H):
    # "ALiBi: Attention with Linear Biases": the ratio between consecutive slopes is 2^(-8/H).
    m = oracle.slopes(H)
    assert np.allclose(m[1:] / m[:-1], 2.0 ** (-8.0 / H), rtol=1e-14, atol=0)
    assert m[0] == pytest.approx(2.0 ** (-8.0 / H), rel=1e-15)


def test_slopes_nonpow2_keep_pow2_prefix():
    # Non-power-of-two head counts keep the schedule of the largest smaller power
    # of two, then append entries of the 2x schedule ("ALiBi: Attention with
    # Linear Biases"); the appended ones are every other entry starting at the first.
    for H in [3, 5, 6, 7, 9, 12, 20, 40, 71, 100]:
        c = 1 << (H.bit_length() - 1)
        m = oracle.slopes(H)
        assert np.array_equal(m[:c], oracle.slopes(c))
        assert np.array_equal(m[c:], oracle.slopes(2 * c)[0::2][: H - c])


def test_slopes_f32_correctly_rounded():
    # C1 reading: the fp32 slope is the exact real 2^(-num/den) rounded once to
    # fp32 (round to nearest even). Independent route: 200-bit mpmath, rounded
    # to a 24-bit significand.
    mpmath.mp.prec = 200
    for H in range(1, 257):
        got = oracle.slopes_f32(H)
        for h in range(H):
            num, den = oracle.slope_exponent(H, h)
            exact = mpmath.power(2, mpmath.mpf(-num) / den)
            with mpmath.workprec(24):
                want = float(+exact)
            assert float(got[h]) == want, (H, h)


# -------------------------------------------------------------------- bias

def _worked_values():
    rows = []
    with open(os.path.join(GOLDEN, "worked_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, m, i, j, want = line.split()[:5]
            rows.append((float(a), float(m), int(i), int(j), float(want)))
    return rows


@pytest.mark.parametrize("a,m,i,j,want", _worked_values())
def test_worked_biased_logits(a, m, i, j, want):
    got = a + oracle.bias(m, i, j, causal=True)
    assert got == pytest.approx(want, abs=1e-12)


def test_extrapolation_values_exact():
    # "What length extrapolation means": -3.99609375 at 1023 and -7.99609375 at
    # 2047 for slope 0.00390625 are exact binary fractions.
    assert oracle.bias(0.00390625, 1023, 0) == -3.99609375
    assert oracle.bias(0.00390625, 2047, 0) == -7.99609375


def test_translation_invariance_and_zero_diagonal():
    # dev.to page asserts: b[7,3] == b[6,2] (distance 4) and b[5,5] == 0.
    assert oracle.bias(0.25, 7, 3) == oracle.bias(0.25, 6, 2)
    assert oracle.bias(0.25, 5, 5) == 0.0
    for s in range(0, 50, 7):
        for i in range(8):
            for j in range(i + 1):
                assert oracle.bias(0.25, i + s, j + s) == oracle.bias(0.25, i, j)


def test_causal_mask_and_symmetric_distance():
    # Future keys are excluded regardless of content ("From distance to a
    # normalized weight"); the non-causal distance is |i - j| ("ALiBi and
    # Relative Position Bias", "The mechanics").
    assert oracle.bias(0.5, 3, 4) == -math.inf
    assert oracle.bias(0.5, 3, 7, causal=False) == oracle.bias(0.5, 7, 3, causal=False) == -2.0


# ----------------------------------------------------------- full attention

def _p4_golden():
    mats, cur = {}, None
    with open(os.path.join(GOLDEN, "p4_seed42_weights.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("head"):
                _, h, _, m = line.split()
                cur = (int(h), float(m))
                mats[cur] = []
            else:
                mats[cur].append([float(x) for x in line.split()])
    return {k: np.array(v) for k, v in mats.items()}


def test_p4_printed_weight_matrices():
    # "ALiBi in Attention: Complete Implementation", seed-42 example: the printed
    # 8x8 causal weights of heads 1 and 4 (3 decimals).
    q, k, v = gen.generate(gen.WORKLOADS["p4_example"])
    _, _, w = oracle.attention(q.f32, k.f32, v.f32, want_weights=True)
    m = oracle.slopes(4)
    for (h, slope), want in _p4_golden().items():
        assert m[h] == slope
        assert np.abs(w[0, h] - want).max() <= 5e-4 + 1e-9, h


def test_rows_sum_to_one_and_mask():
    # Every query row of every head normalises to one ("ALiBi: Attention with
    # Linear Biases", "From distance to a normalized weight"); masked entries
    # are exactly zero.
    q, k, v = gen.random_case(7, 2, 3, 40, 16, dtype="fp32")
    _, _, w = oracle.attention(q.f32, k.f32, v.f32, want_weights=True)
    assert np.allclose(w.sum(-1), 1.0, atol=1e-13)
    assert np.all(w[..., np.triu_indices(40, 1)[0], np.triu_indices(40, 1)[1]] == 0.0)


def test_equal_scores_ratio_is_exp_minus_slope():
    # "ALiBi: Attention with Linear Biases", "From distance to a normalized
    # weight": the ratio of two allowed keys' weights is free of the softmax
    # denominator, and at equal content scores one more token of distance scales
    # it by e^{-m_h}.
    rng = np.random.default_rng(1)
    B, H, N, d = 1, 4, 24, 8
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    krow = rng.standard_normal(d).astype(np.float32)
    k = np.broadcast_to(krow, (B, H, N, d)).copy()
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    _, _, w = oracle.attention(q, k, v, want_weights=True)
    m = oracle.slopes(H)
    for h in range(H):
        for i in range(1, N):
            ratios = w[0, h, i, :i] / w[0, h, i, 1:i + 1]
            assert np.allclose(ratios, math.exp(-m[h]), rtol=1e-12)


def test_zero_keys_closed_form():
    # With K = 0 every content score is 0 and row i's weights are the normalised
    # geometric sequence e^{-m (i-j)} / sum_{t=0}^{i} e^{-m t}; the sum is
    # (1 - e^{-m (i+1)}) / (1 - e^{-m}).
    rng = np.random.default_rng(2)
    B, H, N, d = 1, 6, 33, 16
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = np.zeros_like(q)
    v = rng.standard_normal((B, H, N, d)).astype(np.float32)
    out, lse, w = oracle.attention(q, k, v, want_weights=True)
    m = oracle.slopes(H)
    for h in range(H):
        r = math.exp(-m[h])
        for i in range(N):
            z = (1.0 - r ** (i + 1)) / (1.0 - r)
            want = np.array([r ** (i - j) / z for j in range(i + 1)])
            assert np.allclose(w[0, h, i, :i + 1], want, rtol=1e-12, atol=0)
            assert lse[0, h, i] == pytest.approx(math.log(z), rel=1e-12, abs=1e-14)
        assert np.allclose(out[0, h], w[0, h] @ v[0, h].astype(np.float64), atol=1e-12)


def test_zero_slope_is_uniform_prefix_average():
    # Slopes -> 0 with equal scores: uniform weights 1/(i+1), output = running mean of V.
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 20, 4)).astype(np.float32)
    k = np.zeros_like(q)
    v = rng.standard_normal((1, 1, 20, 4)).astype(np.float32)
    out, _, w = oracle.attention(q, k, v, m=np.zeros(1), want_weights=True)
    for i in range(20):
        assert np.allclose(w[0, 0, i, :i + 1], 1.0 / (i + 1), rtol=1e-13)
        assert np.allclose(out[0, 0, i], v[0, 0, :i + 1].astype(np.float64).mean(0), atol=1e-13)


def _brute_force_row(q, k, v, slope, i, causal=True):
    """Per-element softmax by direct summation: no max shift, no reuse of the oracle."""
    d = len(q[i])
    keys = range(i + 1) if causal else range(len(k))
    num = {}
    for j in keys:
        score = math.fsum(float(q[i][t]) * float(k[j][t]) for t in range(d)) / math.sqrt(d)
        num[j] = math.exp(score - slope * abs(i - j))
    den = math.fsum(num.values())
    w = {j: num[j] / den for j in keys}
    o = [math.fsum(w[j] * float(v[j][t]) for j in keys) for t in range(len(v[0]))]
    return o, math.log(den), w


@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_tiny(causal):
    q, k, v = gen.random_case(11, 1, 3, 13, 8, dtype="fp32")
    out, lse, w = oracle.attention(q.f32, k.f32, v.f32, causal=causal, want_weights=True)
    m = oracle.slopes(3)
    for h in range(3):
        for i in range(13):
            o_bf, lse_bf, w_bf = _brute_force_row(q.f32[0, h], k.f32[0, h], v.f32[0, h], m[h], i, causal)
            assert np.allclose(out[0, h, i], o_bf, atol=1e-12, rtol=0)
            assert lse[0, h, i] == pytest.approx(lse_bf, abs=1e-12)
            for j, wj in w_bf.items():
                assert w[0, h, i, j] == pytest.approx(wj, abs=1e-13)


def test_selected_rows_match_full():
    q, k, v = gen.random_case(5, 2, 3, 50, 16, dtype="bf16")
    out, lse, _ = oracle.attention(q.f32, k.f32, v.f32)
    rows = np.array([0, 49, 50, 123, 299])
    o2, l2, _ = oracle.attention(q.f32, k.f32, v.f32, rows=rows)
    assert np.array_equal(o2, out.reshape(-1, 16)[rows])
    assert np.array_equal(l2, lse.reshape(-1)[rows])


def test_decode_equals_last_prefill_row():
    # A decode query at true position L-1 sees exactly what prefill row L-1 sees
    # ("ALiBi: Attention with Linear Biases", KV-cache paragraph).
    B, H, L, d = 2, 5, 77, 32
    q, k, v = gen.random_case(9, B, H, L, d, dtype="bf16")
    out_p, lse_p, _ = oracle.attention(q.f32, k.f32, v.f32)
    qd = q.f32[:, :, L - 1, :]
    out_d, lse_d = oracle.decode(qd, k.f32, v.f32)
    assert np.allclose(out_d, out_p[:, :, L - 1], atol=1e-13)
    assert np.allclose(lse_d, lse_p[:, :, L - 1], atol=1e-13)


# ------------------------------------------------------- numerical failure

def test_table4_thresholds():
    # "When Attention Goes Blind", App. A Table 4 (printed to 4 decimals).
    t = oracle.thresholds()
    assert round(t["underflow_bf16"], 4) == -92.1886
    assert round(t["underflow_fp32"], 4) == -103.2789
    assert round(t["denorm_bf16"], 4) == -87.3365
    assert round(t["denorm_fp32"], 4) == -87.3365
    assert round(t["overflow_bf16"], 4) == 88.7189
    assert round(t["overflow_fp32"], 4) == 88.7228
    # sec. 3.2 text: tau_fp32 ~ -103.27, tau_bf16 ~ -92.18 (truncated to 2 decimals)
    assert math.trunc(t["underflow_fp32"] * 100) / 100 == -103.27
    assert math.trunc(t["underflow_bf16"] * 100) / 100 == -92.18
    # the thresholds are where the formats' exponentials actually flush
    assert np.float32(math.exp(t["underflow_fp32"])) > 0 and np.float32(math.exp(t["underflow_fp32"] - 1)) == 0
    assert np.float32(math.exp(t["denorm_fp32"])) == np.finfo(np.float32).tiny


def test_table1_blindness_distances():
    # "When Attention Goes Blind", Table 1: BLOOM (16 heads) delta_1 = 124,
    # delta_H = 22,358; Falcon-RW (64 heads) delta_1 = 95, delta_H = 22,358.
    # The printed values are the crossing points rounded to the nearest integer,
    # with tau = ln 2^-126 (the reading that reproduces every printed value).
    for H, d1, dH in [(16, 124, 22358), (64, 95, 22358)]:
        m = oracle.slopes(H)
        assert round(oracle.blindness_real(m[0])) == d1
        assert round(oracle.blindness_real(m[-1])) == dH


def test_table8_default_row_nine_heads():
    # Table 8 "ALiBi (default)" for the 9-head model of Table 7, listed sorted.
    want = [124, 175, 349, 699, 1397, 2795, 5590, 11179, 22358]
    got = sorted(round(oracle.blindness_real(x)) for x in oracle.slopes(9))
    assert got == want
    # integer definition min{D : -m D <= tau} agrees with ceil of the crossing point
    for x in oracle.slopes(9):
        D = oracle.blindness_int(x)
        assert -x * D <= TAU_D < -x * (D - 1)


def test_log_scaled_blindness():
    # sec. 3.4 "Log-scaled Distances": delta_1 moves from 124 to 4.37e53.
    m1 = oracle.slopes(16)[0]
    assert round(oracle.blindness_real(m1)) == 124
    assert float(f"{oracle.blindness_real(m1, log_distance=True):.2e}") == 4.37e53


def test_underflow_counter_is_shift_invariant():
    # The counted quantity is the max-subtracted exponent ("When Attention Goes
    # Blind", App. B.1 stable softmax and sec. 3.2), so a content score shared by
    # every key of a row (identical K rows) leaves the counts of the A = 0 case.
    B, H, N, d = 1, 8, 200, 8
    rng = np.random.default_rng(4)
    q = (3.0 * rng.standard_normal((B, H, N, d))).astype(np.float32)
    k = np.broadcast_to(rng.standard_normal(d).astype(np.float32), (B, H, N, d)).copy()
    cnt, _ = oracle.underflow_counts_per_head(q, k, TAU_D)
    cnt0, _ = oracle.underflow_counts_per_head(np.zeros_like(q), k, TAU_D)
    assert np.array_equal(cnt, cnt0) and cnt0.sum() > 0


def test_underflow_counter_closed_form():
    # With Q = 0 (A = 0) the max-subtracted exponent of key j in row i is
    # -m (i - j); a causal pair underflows iff i - j >= w := min{D : -m D <= tau}.
    # Per head the count is sum_{D=w}^{N-1} (N - D) = (N-w)(N-w+1)/2.
    B, H, N, d = 1, 16, 300, 8
    q = np.zeros((B, H, N, d), np.float32)
    k = np.random.default_rng(0).standard_normal((B, H, N, d)).astype(np.float32)
    cnt, _ = oracle.underflow_counts_per_head(q, k, TAU_D)
    for h, x in enumerate(oracle.slopes(H)):
        w = int(oracle.blindness_int(x))
        want = (N - w) * (N - w + 1) // 2 if w < N else 0
        assert cnt[h] == want, h


@pytest.mark.parametrize("band", [0.0, 1.25, 3.65])
def test_underflow_band_closed_form(band):
    # The counter's second output is the number of entries whose max-subtracted
    # exponent lies within +-band of tau: the entries whose side of the "<= tau"
    # crossing ("When Attention Goes Blind", sec. 3.2) depends on rounding. With
    # Q = 0 row i's exponent at distance D is exactly -m D (the diagonal holds
    # the max), so per head the count is the sum of (N - D) over the distances
    # D < N with |-m D - tau| <= band, evaluated here in exact rationals. tau is
    # chosen so that -m D = tau exactly for the dyadic slopes (ties at band 0
    # and at both edges of band 1.25 count), and 0.3 has no tie.
    from fractions import Fraction
    N, tau = 300, -25.0
    m = np.array([0.25, 0.5, 0.0625, 0.3, 0.125])
    q = np.zeros((1, m.size, N, 4), np.float32)
    k = np.random.default_rng(1).standard_normal(q.shape).astype(np.float32)
    cnt, near = oracle.underflow_counts_per_head(q, k, tau, m=m, band=band)
    for h, mh in enumerate(m):
        fm, ft, fb = Fraction(float(mh)), Fraction(tau), Fraction(band)
        want_near = sum(N - D for D in range(N) if abs(-fm * D - ft) <= fb)
        want_cnt = sum(N - D for D in range(N) if -fm * D <= ft)
        assert near[h] == want_near, (h, band)
        assert cnt[h] == want_cnt, h
    # the tie at band 0: slope 0.25 reaches -25 at D = 100 exactly
    if band == 0.0:
        assert near[0] == N - 100 and near[1] == N - 50 and near[3] == 0


def test_fraction_36_6_percent():
    # sec. 3.3 / Fig. 1b: at a token distance of 2048, 36.6% of the entries of a
    # 16-head bf16 layer have underflowed (A = 0). Reading: the last row of a
    # 2048-token context, averaged over the 16 heads.
    H, N = 16, 2048
    q = np.zeros((1, H, N, 4), np.float32)
    k = np.zeros_like(q)
    rows = [h * N + (N - 1) for h in range(H)]
    cnt, _ = oracle.underflow_rows(q, k, TAU_D, rows=rows)
    frac = float(np.mean(cnt / N))
    assert round(100 * frac, 1) == 36.6


def test_fraction_88_3_percent_out_of_window():
    # sec. 5.2: a steep head with an effective window of 124 tokens in a
    # 2048-token context has 88.3% of its (causal) entries out of window.
    N = 2048
    m = np.array([oracle.slopes(16)[0]])  # delta = 124
    q = np.zeros((1, 1, N, 4), np.float32)
    cnt, _ = oracle.underflow_counts_per_head(q, q.copy(), TAU_D, m=m)
    assert round(100 * cnt[0] / (N * (N + 1) / 2), 1) == 88.3


# ------------------------------------------------------------- mitigations

def test_clamp_variant():
    # sec. 3.4 "Clamping": B* = max(B, c_clamp), c_clamp = -87 (sec. 4.3). With
    # A = 0, every key beyond distance 87/m keeps weight ratio e^{-87} to the
    # diagonal instead of underflowing.
    N, m = 400, 0.5
    q = np.zeros((1, 1, N, 4), np.float32)
    _, _, w = oracle.attention(q, q, q, m=np.array([m]), want_weights=True, variant=oracle.CLAMP, c_clamp=-87.0)
    row = w[0, 0, N - 1]
    far = row[: N - 1 - 174]  # distances >= 175 > 87 / 0.5
    assert np.allclose(far / row[N - 1], math.exp(-87.0), rtol=1e-12)
    assert oracle.bias(m, 500, 0, variant=oracle.CLAMP) == -87.0


def test_logdist_variant():
    # sec. 3.4 "Log-scaled Distances": D* = log(D + 1), so with A = 0 the weight
    # ratio to the diagonal is (D + 1)^{-m}.
    N, m = 64, 0.7
    q = np.zeros((1, 1, N, 4), np.float32)
    _, _, w = oracle.attention(q, q, q, m=np.array([m]), want_weights=True, variant=oracle.LOGDIST)
    row = w[0, 0, N - 1]
    D = np.arange(N - 1, -1, -1, dtype=np.float64)
    assert np.allclose(row / row[-1], (D + 1.0) ** (-m), rtol=1e-12)


def test_softcap_variant():
    # sec. 3.4 "Soft Capping": A* = z tanh(A / z), z = 50. One key with A = 100
    # (d = 1, q = k = 10): LSE = 50 tanh(2).
    q = np.full((1, 1, 1, 1), 10.0, np.float32)
    _, lse, _ = oracle.attention(q, q, q, m=np.array([0.5]), variant=oracle.SOFTCAP, z_cap=50.0)
    assert lse[0, 0, 0] == pytest.approx(50.0 * math.tanh(2.0), abs=1e-12)
    _, lse_plain, _ = oracle.attention(q, q, q, m=np.array([0.5]))
    assert lse_plain[0, 0, 0] == pytest.approx(100.0, abs=1e-12)


# Table 8 ("When Attention Goes Blind", App. F): expected blindness distances of
# the trained 9-head models, rounded to the nearest integer.
TABLE8_SCHEDULES = {
    "Steep": (128, 512, [128, 152, 181, 215, 256, 304, 362, 431, 512]),
    "Safe": (2048, 4096, [2048, 2233, 2435, 2656, 2896, 3158, 3444, 3756, 4096]),
    "Wide": (16, 4096, [16, 32, 64, 128, 256, 512, 1024, 2048, 4096]),
    "Explicit": (32, 8192, [32, 64, 128, 256, 512, 1024, 2048, 4096, 8192]),
}


@pytest.mark.parametrize("name", sorted(TABLE8_SCHEDULES))
def test_table8_explicit_schedules(name):
    # sec. 4.2 names only delta_1 and delta_H for Steep / Safe / Wide; Table 8's
    # middle columns fix the spacing as geometric over the nine heads.
    d1, dH, want = TABLE8_SCHEDULES[name]
    m = oracle.slopes_explicit(9, d1, dH)
    assert [round(oracle.blindness_real(x)) for x in m] == want
    # slopes fall head by head and the steepest head is the first
    assert np.all(np.diff(m) < 0)


def test_explicit_slopes_section_3_4_example():
    # sec. 3.4 "Robust Slopes": for a 2048 context the targets double from 32
    # to 2048, i.e. seven heads.
    m = oracle.slopes_explicit(7, 32, 2048)
    assert [round(oracle.blindness_real(x)) for x in m] == [32, 64, 128, 256, 512, 1024, 2048]
    # the crossing sits on the target up to rounding, so the integer definition
    # lands on it or one token past it
    for x, want in zip(m, [32, 64, 128, 256, 512, 1024, 2048]):
        assert oracle.blindness_int(x) in (want, want + 1)


def test_explicit_slopes_log_distance_adaptation():
    # sec. 4.3: with log-scaled distances (E+L) the slopes become
    # m_h = -tau / log(delta_h + 1), so the log-distance crossing lands on delta_h.
    m = oracle.slopes_explicit(9, 32, 8192, log_distance=True)
    for x, want in zip(m, TABLE8_SCHEDULES["Explicit"][2]):
        assert math.isclose(oracle.blindness_real(x, log_distance=True), want, rel_tol=1e-9)
        assert math.isclose(x, -TAU_D / math.log(want + 1), rel_tol=1e-12)
    # with linear distances the same slopes go blind after only log(delta + 1) tokens
    assert round(oracle.blindness_real(m[0])) == round(math.log(33))


def test_explicit_slopes_edges():
    # one head takes delta_first; equal ends give equal slopes; tau scales them
    assert math.isclose(oracle.slopes_explicit(1, 100, 5000)[0], -TAU_D / 100, rel_tol=1e-15)
    assert np.allclose(oracle.slopes_explicit(4, 300, 300), -TAU_D / 300, rtol=1e-15)
    assert np.allclose(oracle.slopes_explicit(5, 16, 256, tau=-1.0), 1.0 / (16 * 2.0 ** np.arange(5)),
                       rtol=1e-14)
    for bad in [(0, 16, 64), (4, 0, 64), (4, 16, -1), (4, 16, float("inf"))]:
        with pytest.raises(RuntimeError):
            oracle.slopes_explicit(*bad)
    with pytest.raises(RuntimeError):
        oracle.slopes_explicit(4, 16, 64, tau=0.5)

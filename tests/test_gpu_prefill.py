"""bf16 tcgen05 prefill vs the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_BF16_LSE, assert_bf16_out, assert_close, dev, host64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


def run_bf16(ab, q, k, v):
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    out, lse = ab.alibi_attn_fwd(qd, kd, vd)
    ab.alibi_check_error()
    return host64(out), host64(lse)


@pytest.mark.parametrize("B,H,N,d", [
    (1, 1, 1, 64), (1, 2, 7, 128), (1, 1, 64, 64), (1, 3, 127, 128), (2, 2, 128, 64), (1, 2, 129, 128),
    (1, 1, 255, 64), (1, 2, 256, 128), (1, 1, 257, 128), (1, 3, 383, 64), (2, 3, 1000, 64), (1, 4, 700, 128),
    (1, 1, 1537, 128),
])
def test_prefill_shape_sweep(ab, B, H, N, d):
    q, k, v = gen.random_case(7 + N + d + H, B, H, N, d, dtype="bf16")
    out, lse = run_bf16(ab, q, k, v)
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")


def test_heads6_n1024_full(ab):
    # B=2, H=6 (non-power-of-two slopes), N=1024, d=64, bf16 N(0, 1): every row
    q, k, v = gen.generate(gen.WORKLOADS["heads6_n1024"])
    out, lse = run_bf16(ab, q, k, v)
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")


@pytest.mark.parametrize("name", ["layer_n2048", "long_n16384"])
def test_full_size_sampled_rows(ab, name):
    # the full-size workloads, in the launch configuration the benchmark times;
    # the oracle checks rows of EVERY (b, h): the tile edges, the ragged tail, the
    # last row and random rows (35-43 per head)
    w = gen.WORKLOADS[name]
    q, k, v = gen.generate(w)
    out, lse = run_bf16(ab, q, k, v)
    rows = sample_rows(w.B, w.H, w.N, max_heads=w.B * w.H, per_head=16 if w.N > 4096 else 24, seed=w.N)
    assert len(np.unique(rows // w.N)) == w.B * w.H
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, rows=rows)
    assert_bf16_out(out.reshape(-1, w.d)[rows], ro)
    assert_close(lse.reshape(-1)[rows], rl, TOL_BF16_LSE, "lse")
    # properties at every row: finite, outputs inside the convex hull of V's range
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    vmax = np.abs(v.f32).max()
    assert np.abs(out).max() <= vmax * (1 + 2 ** -8)


def test_repeatable_and_lse_optional(ab):
    import torch
    q, k, v = gen.random_case(3, 1, 2, 300, 128, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o1, l1 = ab.alibi_attn_fwd(qd, kd, vd)
    o2, l2 = ab.alibi_attn_fwd(qd, kd, vd)
    o3, l3 = ab.alibi_attn_fwd(qd, kd, vd, want_lse=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o4, _ = ab.alibi_attn_fwd(qd, kd, vd)
    s.synchronize()
    ab.alibi_check_error()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3) and torch.equal(o1, o4)


def test_equal_scores_recency_on_gpu(ab):
    # identical K rows: each row's weights fall by e^{-m} per token of distance
    # ("ALiBi: Attention with Linear Biases", "From distance to a normalized
    # weight"); with V = one-hot positions the output exposes the weights.
    import torch
    H, N, d = 4, 128, 128
    rng = np.random.default_rng(5)
    q = gen.make_tensor(rng.standard_normal((1, H, N, d)), (1, H, N, d), "bf16")
    k = gen.make_tensor(np.broadcast_to(rng.standard_normal(d), (1, H, N, d)), (1, H, N, d), "bf16")
    v = gen.make_tensor(np.broadcast_to(np.eye(N, d), (1, H, N, d)), (1, H, N, d), "bf16")
    out, lse = run_bf16(ab, q, k, v)
    m = oracle.slopes(H)
    for h in range(H):
        i = N - 1
        w = out[0, h, i, : i + 1]
        want = np.exp(-m[h] * (i - np.arange(i + 1)))
        want /= want.sum()
        assert np.abs(w - want).max() <= 1e-2 * max(1.0, want.max())


def test_lazy_rescale_with_divergent_rows(ab):
    # Rows of one warp disagree on raising the running max: even rows meet low
    # scores on their diagonal tile and high scores one tile back, odd rows the
    # reverse. Scores reach +-sigma |u|^2 / sqrt(d) with sigma = 40, well past
    # the 2^8 lazy-rescale threshold.
    H, N, d = 1, 384, 128
    rng = np.random.default_rng(8)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    sign_q = np.where(np.arange(N) % 2 == 0, 1.0, -1.0)
    q = 40.0 * sign_q[:, None] * u[None, :] + 0.1 * rng.standard_normal((N, d))
    tile = np.arange(N) // 128
    k = np.where((tile % 2 == 0)[:, None], 1.0, -1.0) * u[None, :] * 6.0 + 0.1 * rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    qt, kt, vt = (gen.make_tensor(x[None, None], (1, H, N, d), "bf16") for x in (q, k, v))
    out, lse = run_bf16(ab, qt, kt, vt)
    ro, rl, _ = oracle.attention(qt.f32, kt.f32, vt.f32)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("B,H,N,d", [(1, 2, 7, 16), (1, 4, 300, 16), (2, 3, 129, 32), (1, 4, 700, 32)])
def test_prefill_small_head_sizes(ab, B, H, N, d, causal):
    # d = 16 and 32 run the d = 64 tiles with a 64-column TMA box over the narrower rows
    q, k, v = gen.random_case(61 + N + d, B, H, N, d, dtype="bf16")
    out, lse = ab.alibi_attn_fwd(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=causal)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, causal=causal)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_prefill_small_head_skip_is_bit_identical(ab):
    import torch
    q, k, v = gen.random_case(71, 1, 4, 2000, 32, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o0, l0 = ab.alibi_attn_fwd(qd, kd, vd)
    o1, l1 = ab.alibi_attn_fwd(qd, kd, vd, skip_underflow=True)
    ab.alibi_check_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("seed,B,H,N,d,sq", [(101, 1, 8, 2048, 128, 3.0), (102, 2, 6, 1024, 64, 3.0),
                                             (106, 2, 16, 1024, 128, 3.0), (107, 1, 4, 3000, 64, 4.0)])
def test_peaked_weights_with_normal_values(ab, seed, B, H, N, d, sq):
    # Q, K ~ N(0, sq^2) make the weights peaked (logits of tens); V ~ N(0, 1)
    # reaches |v| ~ 5. The bf16 rounding of P moves an output by at most 2^-8 of the
    # weighted mean of |v| (unit roundoff of bf16), so these rows sit closest to the
    # 1e-2 bound; they are judged at exactly that bound (plus half a bf16 ulp of the
    # value for the output's own rounding), and against the 2^-8 max|v| worst case.
    n = B * H * N * d
    q = gen.make_tensor(gen.normal(seed, 0, n, scale=sq), (B, H, N, d), "bf16")
    k = gen.make_tensor(gen.normal(seed, 1, n, scale=sq), (B, H, N, d), "bf16")
    v = gen.make_tensor(gen.normal(seed, 2, n, scale=1.0), (B, H, N, d), "bf16")
    out, lse = run_bf16(ab, q, k, v)
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")
    from gpu_helpers import half_ulp_bf16
    before_store = np.abs(out - ro) - half_ulp_bf16(ro)
    assert before_store.max() <= 2.0 ** -8 * np.abs(v.f32).max()


def test_concurrent_host_threads(ab):
    # Several host threads call the prefill at once, each on its own stream and with
    # its own head count, so the per-device kernel set-up and the per-head-count slope
    # tables are first created concurrently (the C calls run without the GIL). Every
    # result must equal the same call made alone.
    import threading
    import torch
    shapes = [(1, h, 300 + 17 * i, 128 if i % 2 else 64) for i, h in enumerate((3, 5, 7, 9, 11, 13))]
    inputs = []
    for i, (B, H, N, d) in enumerate(shapes):
        q, k, v = gen.random_case(500 + i, B, H, N, d, dtype="bf16")
        inputs.append(tuple(dev(t, "bf16") for t in (q, k, v)))
    results = [None] * len(shapes)
    errors = []
    start = threading.Barrier(len(shapes))

    def work(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            for causal in (True, False):
                with torch.cuda.stream(s):
                    out, lse = ab.alibi_attn_fwd(*inputs[i], causal=causal, stream=s)
                s.synchronize()
                results[i] = results[i] or {}
                results[i][causal] = (out, lse)
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    ab.alibi_check_error()
    assert not errors, errors
    for i in range(len(shapes)):
        for causal in (True, False):
            out, lse = ab.alibi_attn_fwd(*inputs[i], causal=causal)
            ab.alibi_check_error()
            assert torch.equal(out, results[i][causal][0]) and torch.equal(lse, results[i][causal][1]), (i, causal)

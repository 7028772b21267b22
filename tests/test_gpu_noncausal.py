"""causal = 0: the symmetric bias -m_h |i - j| over every key ("ALiBi and Relative
Position Bias" (quantmemo.com), "The mechanics"; the encoder models of "When
Attention Goes Blind", Table 5), in the tensor-core prefill and the fp32 path,
against the oracle's causal = 0 rows."""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_BF16_LSE, TOL_F32, assert_bf16_out, assert_close, dev, host64, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


def run_bf16(ab, q, k, v):
    out, lse = ab.alibi_attn_fwd(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=False)
    ab.alibi_check_error()
    return host64(out), host64(lse)


# single tile, ragged single tile, one Q block with and without a second Q tile,
# ragged last KV tile, several blocks (the wrap-around walk), both head sizes
@pytest.mark.parametrize("B,H,N,d", [
    (1, 1, 1, 64), (1, 2, 7, 128), (1, 1, 128, 64), (1, 3, 127, 128), (1, 2, 129, 128), (1, 1, 255, 64),
    (1, 2, 256, 128), (1, 1, 257, 128), (1, 3, 383, 64), (2, 3, 1000, 64), (1, 4, 700, 128), (1, 1, 1537, 128),
])
def test_noncausal_shape_sweep(ab, B, H, N, d):
    q, k, v = gen.random_case(101 + N + d + H, B, H, N, d, dtype="bf16")
    out, lse = run_bf16(ab, q, k, v)
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, causal=False)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")


@pytest.mark.parametrize("name", ["heads6_n1024", "layer_n2048", "long_n16384"])
def test_noncausal_workloads_sampled_rows(ab, name):
    # rows of every (b, h): tile edges, the ragged tail, the last row, random rows
    w = gen.WORKLOADS[name]
    q, k, v = gen.generate(w)
    out, lse = run_bf16(ab, q, k, v)
    rows = sample_rows(w.B, w.H, w.N, max_heads=w.B * w.H, per_head=8 if w.N > 4096 else 16, seed=w.N + 1)
    assert len(np.unique(rows // w.N)) == w.B * w.H
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, causal=False, rows=rows)
    assert_bf16_out(out.reshape(-1, w.d)[rows], ro)
    assert_close(lse.reshape(-1)[rows], rl, TOL_BF16_LSE, "lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_noncausal_symmetric_closed_form(ab):
    # identical K rows: row i's weights are exp(-m |i - j|) / sum over all j, so the
    # output with V = one-hot positions exposes a two-sided geometric profile
    H, N, d = 4, 128, 128
    rng = np.random.default_rng(15)
    q = gen.make_tensor(rng.standard_normal((1, H, N, d)), (1, H, N, d), "bf16")
    k = gen.make_tensor(np.broadcast_to(rng.standard_normal(d), (1, H, N, d)), (1, H, N, d), "bf16")
    v = gen.make_tensor(np.broadcast_to(np.eye(N, d), (1, H, N, d)), (1, H, N, d), "bf16")
    out, _ = run_bf16(ab, q, k, v)
    m = oracle.slopes(H)
    for h in range(H):
        for i in (0, 40, 64, N - 1):
            want = np.exp(-m[h] * np.abs(i - np.arange(N)))
            want /= want.sum()
            assert np.abs(out[0, h, i] - want).max() <= 1e-2 * max(1.0, want.max())
    # the profile is symmetric about the query: weights of i - D and i + D agree
    h, i = H - 1, 64
    assert np.abs(out[0, h, i, i - 20:i] - out[0, h, i, i + 20:i:-1]).max() <= 4e-3


def test_noncausal_ragged_keys_are_masked(ab):
    # N = 130: the last KV tile holds 2 real keys and 126 zero-filled ones. With
    # every real score very negative, unmasked padding (score 0) would dominate.
    H, N, d = 2, 130, 64
    rng = np.random.default_rng(16)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    q = 12.0 * np.broadcast_to(u, (1, H, N, d))
    k = -12.0 * np.broadcast_to(u, (1, H, N, d)) + 0.01 * rng.standard_normal((1, H, N, d))
    v = rng.standard_normal((1, H, N, d))
    qt, kt, vt = (gen.make_tensor(x, (1, H, N, d), "bf16") for x in (q, k, v))
    out, lse = run_bf16(ab, qt, kt, vt)
    ro, rl, _ = oracle.attention(qt.f32, kt.f32, vt.f32, causal=False)
    assert_bf16_out(out, ro)
    assert_close(lse, rl, TOL_BF16_LSE, "lse")


def test_noncausal_differs_from_causal(ab):
    # the parity above is not vacuous: future keys change every row but the last
    q, k, v = gen.random_case(17, 1, 2, 300, 64, dtype="bf16")
    o_nc, _ = run_bf16(ab, q, k, v)
    o_c, _ = ab.alibi_attn_fwd(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=True)
    o_c = host64(o_c)
    assert np.abs(o_nc[0, :, :-1] - o_c[0, :, :-1]).max() > 0.05
    assert np.abs(o_nc[0, :, -1] - o_c[0, :, -1]).max() <= 1e-2


@pytest.mark.parametrize("combo", [("clamp",), ("logdist",), ("softcap",), ("clamp", "logdist", "softcap")])
def test_noncausal_mitigations(ab, combo):
    abi = {"clamp": 2, "logdist": 4, "softcap": 8}
    orc = {"clamp": oracle.CLAMP, "logdist": oracle.LOGDIST, "softcap": oracle.SOFTCAP}
    q, k, _ = gen.random_case(19, 1, 3, 777, 128, dtype="bf16", sigma=4.0)
    _, _, v = gen.random_case(20, 1, 3, 777, 128, dtype="bf16")
    out, lse = ab.alibi_attn_fwd_ex(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=False,
                                    flags=sum(abi[c] for c in combo), clamp_min=-3.0, softcap_z=50.0)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, causal=False, variant=sum(orc[c] for c in combo),
                                 c_clamp=-3.0, z_cap=50.0)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


@pytest.mark.parametrize("B,H,N,d", [(1, 4, 64, 16), (2, 3, 100, 64), (1, 2, 77, 200)])
def test_noncausal_fp32_path_and_weights(ab, B, H, N, d):
    q, k, v = gen.random_case(23 + N, B, H, N, d, dtype="fp32", sigma=0.5)
    qd, kd, vd = dev(q, "fp32"), dev(k, "fp32"), dev(v, "fp32")
    out, lse = ab.alibi_attn_fwd_f32(qd, kd, vd, causal=False)
    P = ab.alibi_attn_probs_f32_ex(qd, kd, lse, causal=False)
    ab.alibi_check_error()
    ro, rl, rw = oracle.attention(q.f32, k.f32, v.f32, causal=False, want_weights=True)
    assert_close(host64(out), ro, TOL_F32, "out")
    assert_close(host64(lse), rl, TOL_F32, "lse")
    assert_close(host64(P), rw, TOL_F32, "weights")
    # every row's weights sum to one over all N keys
    assert np.abs(host64(P).sum(axis=-1) - 1.0).max() <= 1e-5

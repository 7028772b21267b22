"""Backward pass (dQ, dK, dV of sum(dO * O)) through the C ABI against the fp64
oracle's gradients, which are pinned to finite differences of the forward.

Tolerances. fp32 path: max-abs error <= 1e-5 x max(1, max |G|) per gradient
tensor G (the 1e-5 of the forward, scaled to the gradient's magnitude). bf16
tensor-core path: a bound per element, derived from where the kernels round
(gpu_helpers.bf16_grad_bounds): P^T enters dV += P^T dO and dS enters dQ and dK
rounded to bf16 (unit roundoff 2^-8), and D_i = dO_i . O_i is taken from the
forward's bf16 output, which is off by half an ulp plus the forward's own P
rounding. Each gradient element must lie within twice its bound plus half a bf16
ulp (the result's own rounding). Measured on the GB300 over this file's cases:
dQ and dK reach at most 0.26 of the bound, dV 0.96 (a key with a single
contributing query, where P's rounding is the whole error). The decoder-layer
workload is checked at full size on every head and element; the identities at
full size keep a coarse 5% bound.
"""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import assert_grad, assert_grad_bound, bf16_grad_bounds, dev, host64

pytestmark = pytest.mark.gpu

TOL_F32_REL = 1e-5


def check_bf16(got, q, k, v, do, refs, causal=True, m=None, variant=0, c_clamp=-87.0, z_cap=50.0, what=("dq", "dk", "dv")):
    """The tensor-core gradients against the oracle's within the derived per-element bounds."""
    rq, rk, rv, _, rowdot = refs
    E = bf16_grad_bounds(q, k, v, do, rowdot, causal=causal, m=m, variant=variant, c_clamp=c_clamp, z_cap=z_cap)
    for g, r, e, name in zip(got, (rq, rk, rv), E, ("dq", "dk", "dv")):
        if name in what:
            assert_grad_bound(g, r, e, name)


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


check_grad = assert_grad


def cases(seed, B, H, N, d, dtype):
    q, k, v = gen.random_case(seed, B, H, N, d, dtype=dtype)
    do, _, _ = gen.random_case(seed + 1000, B, H, N, d, dtype=dtype)
    return q, k, v, do


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("B,H,N,d", [(1, 4, 64, 16), (2, 3, 100, 64), (1, 2, 77, 200), (1, 1, 1, 32)])
def test_bwd_f32_vs_oracle(ab, B, H, N, d, causal):
    q, k, v, do = cases(11 + N + d, B, H, N, d, "fp32")
    qd, kd, vd, dod = (dev(t, "fp32") for t in (q, k, v, do))
    out, lse = ab.alibi_attn_fwd_f32(qd, kd, vd, causal=causal)
    dq, dk, dv = ab.alibi_attn_bwd_f32(qd, kd, vd, out, lse, dod, causal=causal)
    ab.alibi_check_error()
    rq, rk, rv, _, _ = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, causal=causal)
    check_grad(host64(dq), rq, TOL_F32_REL, "dq")
    check_grad(host64(dk), rk, TOL_F32_REL, "dk")
    check_grad(host64(dv), rv, TOL_F32_REL, "dv")


def run_bf16(ab, q, k, v, do, causal=True, slopes=None):
    qd, kd, vd, dod = (dev(t, "bf16") for t in (q, k, v, do))
    if slopes is None:
        out, lse = ab.alibi_attn_fwd(qd, kd, vd, causal=causal)
    else:
        out, lse = ab.alibi_attn_fwd_ex(qd, kd, vd, causal=causal, slopes=slopes)
    dq, dk, dv = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dod, causal=causal, slopes=slopes)
    ab.alibi_check_error()
    return host64(dq), host64(dk), host64(dv)


# single tile, ragged tiles, several tiles (both kernels' walks), both head sizes
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 64), (1, 2, 7, 128), (1, 2, 128, 64), (1, 3, 129, 128),
                                     (2, 2, 300, 64), (1, 4, 513, 128), (1, 2, 1000, 128)])
def test_bwd_bf16_vs_oracle(ab, B, H, N, d, causal):
    q, k, v, do = cases(21 + N + d, B, H, N, d, "bf16")
    got = run_bf16(ab, q, k, v, do, causal)
    refs = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, causal=causal)
    check_bf16(got, q.f32, k.f32, v.f32, do.f32, refs, causal=causal)


def test_bwd_bf16_explicit_slopes(ab):
    H, N, d = 9, 600, 64
    m = ab.alibi_slopes_explicit(H, 16, 4096)
    q, k, v, do = cases(31, 1, H, N, d, "bf16")
    got = run_bf16(ab, q, k, v, do, slopes=m)
    refs = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, m=m.astype(np.float64))
    check_bf16(got, q.f32, k.f32, v.f32, do.f32, refs, m=m.astype(np.float64))


def test_bwd_identities_at_layer_size(ab):
    # layer_n2048 shapes (B=4, H=32, N=2048, d=128): rows of P sum to one and rows of dS
    # to zero, so per (b, h): sum_j dV_j = sum_i dO_i and sum_j dK_j = 0.
    w = gen.WORKLOADS["layer_n2048"]
    q, k, v = gen.generate(w)
    do, _, _ = gen.random_case(77, w.B, w.H, w.N, w.d, dtype="bf16")
    dq, dk, dv = run_bf16(ab, q, k, v, do)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    sum_do = do.f32.astype(np.float64).sum(axis=2)
    assert np.abs(dv.sum(axis=2) - sum_do).max() <= 0.05 * max(1.0, np.abs(sum_do).max())
    assert np.abs(dk.sum(axis=2)).max() <= 0.05 * max(1.0, np.abs(dk).sum(axis=2).max())


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_bwd_every_head_at_layer_size(ab, causal):
    # The decoder-layer workload at full size (B=4, H=32, N=2048, d=128; its K and V
    # exceed half the L2, so the backward's kernels run in the blocked work order),
    # with either mask:
    # dQ, dK and dV of every (b, h), every element, against the oracle within the
    # derived per-element bounds. The oracle's gradients come from one threaded call;
    # the bounds, which need each head's weights, are formed eight heads at a time.
    w = gen.WORKLOADS["layer_n2048"]
    q, k, v = gen.generate(w)
    do, _, _ = gen.random_case(77, w.B, w.H, w.N, w.d, dtype="bf16")
    dq, dk, dv = run_bf16(ab, q, k, v, do, causal=causal)
    refs = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, causal=causal)
    m_all = oracle.slopes(w.H)
    for b in range(w.B):
        for h0 in range(0, w.H, 8):
            sl = (slice(b, b + 1), slice(h0, h0 + 8))
            check_bf16((dq[sl], dk[sl], dv[sl]), q.f32[sl], k.f32[sl], v.f32[sl], do.f32[sl],
                       tuple(r[sl] for r in refs), causal=causal, m=m_all[h0:h0 + 8])


def test_bwd_deterministic(ab):
    import torch
    q, k, v, do = cases(41, 1, 4, 700, 128, "bf16")
    qd, kd, vd, dod = (dev(t, "bf16") for t in (q, k, v, do))
    out, lse = ab.alibi_attn_fwd(qd, kd, vd)
    g1 = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dod)
    g2 = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dod)
    ab.alibi_check_error()
    assert all(torch.equal(a, b) for a, b in zip(g1, g2))


def test_bwd_far_keys_get_exactly_zero_gradient(ab):
    # "When Attention Goes Blind" sec. 5.1: a weight that underflowed carries no
    # gradient. Slope 1 (blindness distance 88), dO nonzero only for rows 150 and
    # beyond: in fp64 key 0 still gets a tiny dV (below e^-140), on the GPU exactly 0.
    H, N, d = 2, 256, 64
    q, k, v, do = cases(51, 1, H, N, d, "bf16")
    dob = do.f32.copy()
    dob[:, :, :150] = 0.0
    do = gen.make_tensor(dob, dob.shape, "bf16")
    m = np.ones(H, np.float32)
    dq, dk, dv = run_bf16(ab, q, k, v, do, slopes=m)
    _, rk, rv, _, _ = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, m=m.astype(np.float64))
    assert (np.abs(rv[0, :, 0]) > 0).any() and np.abs(rv[0, :, 0]).max() < 1e-55
    assert not dv[0, :, 0].any() and not dk[0, :, 0].any()
    # keys within reach of the nonzero rows do get gradient
    assert np.abs(dv[0, :, 200]).max() > 0


ABI = {"clamp": 2, "logdist": 4, "softcap": 8}
ORC = {"clamp": oracle.CLAMP, "logdist": oracle.LOGDIST, "softcap": oracle.SOFTCAP}


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("combo,d", [(("clamp",), 128), (("logdist",), 128), (("softcap",), 128),
                                     (("clamp", "logdist", "softcap"), 128), (("clamp", "logdist", "softcap"), 64)],
                         ids=["clamp", "logdist", "softcap", "all3", "all3_d64"])
def test_bwd_mitigations(ab, combo, d, causal):
    # sigma = 3 on Q and K with z = 8 puts many logits on the curved part of the cap
    # (its derivative factor matters); c_clamp = -3 makes the clamp bind.
    B, H, N = 1, 3, 300
    q, k, _ = gen.random_case(61, B, H, N, d, dtype="bf16", sigma=3.0)
    _, _, v = gen.random_case(62, B, H, N, d, dtype="bf16")
    do, _, _ = gen.random_case(63, B, H, N, d, dtype="bf16")
    flags = sum(ABI[c] for c in combo)
    kw = dict(flags=flags, clamp_min=-3.0, softcap_z=8.0)
    qd, kd, vd, dod = (dev(t, "bf16") for t in (q, k, v, do))
    out, lse = ab.alibi_attn_fwd_ex(qd, kd, vd, causal=causal, **kw)
    dq, dk, dv = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dod, causal=causal, **kw)
    ab.alibi_check_error()
    variant = sum(ORC[c] for c in combo)
    refs = oracle.attention_bwd(q.f32, k.f32, v.f32, do.f32, causal=causal, variant=variant, c_clamp=-3.0, z_cap=8.0)
    check_bf16((host64(dq), host64(dk), host64(dv)), q.f32, k.f32, v.f32, do.f32, refs, causal=causal,
               variant=variant, c_clamp=-3.0, z_cap=8.0)
    if "softcap" in combo:
        # the cap's derivative is not vacuous on these inputs: 1 - tanh^2(A / z) is far from 1
        a = q.f32[0, 0].astype(np.float64) @ k.f32[0, 0].astype(np.float64).T / np.sqrt(d)
        assert np.mean(1.0 - np.tanh(a / 8.0) ** 2) < 0.8


def test_bwd_long_context_prefix_rows_and_identities(ab):
    # long_n16384 (B=1, H=16, N=16384, d=128) in the launch configuration the benchmark
    # times. Causal rows depend only on earlier keys, so dQ of rows below 2048 equals the
    # oracle's dQ of the 2048-prefix problem; over all heads, rows of P sum to one and
    # rows of dS to zero: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 per (b, h).
    w = gen.WORKLOADS["long_n16384"]
    q, k, v = gen.generate(w)
    do, _, _ = gen.random_case(78, w.B, w.H, w.N, w.d, dtype="bf16")
    dq, dk, dv = run_bf16(ab, q, k, v, do)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    sum_do = do.f32.astype(np.float64).sum(axis=2)
    assert np.abs(dv.sum(axis=2) - sum_do).max() <= 0.05 * max(1.0, np.abs(sum_do).max())
    assert np.abs(dk.sum(axis=2)).max() <= 0.05 * max(1.0, np.abs(dk).sum(axis=2).max())
    n = 2048
    for h in (0, 7, 15):  # the shallowest, a middle and the steepest head
        sl = (slice(0, 1), slice(h, h + 1), slice(0, n))
        m = oracle.slopes(w.H)[h:h + 1]
        refs = oracle.attention_bwd(q.f32[sl], k.f32[sl], v.f32[sl], do.f32[sl], m=m)
        check_bf16((dq[sl], None, None), q.f32[sl], k.f32[sl], v.f32[sl], do.f32[sl], refs, m=m, what=("dq",))

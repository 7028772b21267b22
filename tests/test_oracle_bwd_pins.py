"""Pins of the oracle's backward pass (gradients of sum(dO * attention)).

The pages give the forward only ("When Attention Goes Blind" sec. 3.1 eq. 1-4)
and remark (sec. 5.1) that only nonzero weights carry gradient. The gradient
is therefore pinned to the forward itself, by finite differences of the
oracle's own fp64 forward on inputs where every perturbed value is exact, and
by identities every correct gradient satisfies.
"""
import numpy as np
import pytest

import oracle

H_STEP = 2.0 ** -10  # perturbation; inputs are multiples of it, so x +- 2h is exact in fp32


def grid_inputs(seed, B, H, N, d, scale=1.0):
    """Normal-ish inputs rounded to multiples of 2^-10 (|x| < 8): exact in fp32 with room
    for the +-2h perturbations of the finite differences."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(4):
        x = np.clip(scale * rng.standard_normal((B, H, N, d)), -7.0, 7.0)
        out.append((np.round(x / H_STEP) * H_STEP).astype(np.float32))
    return out


def loss(q, k, v, dout, **kw):
    o, _, _ = oracle.attention(q, k, v, **kw)
    return float(np.sum(o * dout.astype(np.float64)))


def fd_grad(which, idx, q, k, v, dout, **kw):
    """Four-point central difference (error O(h^4)) of the loss in one input coordinate."""
    vals = []
    for s in (2, 1, -1, -2):
        ins = [a.copy() for a in (q, k, v)]
        ins[which][idx] += np.float32(s * H_STEP)
        vals.append(loss(*ins, dout, **kw))
    return (-vals[0] + 8 * vals[1] - 8 * vals[2] + vals[3]) / (12 * H_STEP)


CASES = [
    dict(causal=True), dict(causal=False),
    dict(causal=True, variant=oracle.SOFTCAP, z_cap=1.5),        # cap factor matters at z = 1.5
    dict(causal=True, variant=oracle.CLAMP, c_clamp=-1.0),
    dict(causal=False, variant=oracle.LOGDIST | oracle.CLAMP | oracle.SOFTCAP, c_clamp=-2.0, z_cap=2.0),
]


@pytest.mark.parametrize("kw", CASES, ids=["causal", "noncausal", "softcap", "clamp", "all3_noncausal"])
def test_gradients_match_finite_differences(kw):
    B, H, N, d = 1, 2, 7, 4
    q, k, v, dout = grid_inputs(1, B, H, N, d)
    m = np.array([0.7, 0.15])
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, dout, m=m, **kw)
    rng = np.random.default_rng(2)
    for which, g in ((0, dq), (1, dk), (2, dv)):
        for _ in range(10):
            idx = tuple(int(rng.integers(0, s)) for s in (B, H, N, d))
            want = fd_grad(which, idx, q, k, v, dout, m=m, **kw)
            assert abs(g[idx] - want) <= 1e-9 * max(1.0, abs(want)), (which, idx, g[idx], want)


def test_gradient_identities():
    # rows of w sum to one: sum_j dV_j = sum_i dO_i; rows of dx sum to zero: sum_j dK_j = 0
    B, H, N, d = 2, 3, 40, 8
    q, k, v, dout = grid_inputs(3, B, H, N, d)
    for causal in (True, False):
        dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, dout, causal=causal)
        assert np.abs(dv.sum(axis=2) - dout.astype(np.float64).sum(axis=2)).max() <= 1e-12
        assert np.abs(dk.sum(axis=2)).max() <= 1e-12
        # and the LSE of pass 1 is the forward's
        _, lse, _ = oracle.attention(q, k, v, causal=causal)
        _, _, _, lse_b, _ = oracle.attention_bwd(q, k, v, dout, causal=causal)
        assert np.abs(lse - lse_b).max() <= 1e-12


def test_constant_keys_give_zero_dq_and_constant_values_zero_dqk():
    B, H, N, d = 1, 2, 30, 8
    q, k, v, dout = grid_inputs(4, B, H, N, d)
    kc = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq, _, _, _, _ = oracle.attention_bwd(q, kc, v, dout)
    assert np.abs(dq).max() <= 1e-12   # same k everywhere: sum_j dx_ij k = 0
    vc = np.broadcast_to(v[:, :, :1], v.shape).copy()
    dq, dk, _, _, _ = oracle.attention_bwd(q, k, vc, dout)
    assert np.abs(dq).max() <= 1e-12 and np.abs(dk).max() <= 1e-12  # output independent of the weights


def test_single_token():
    q, k, v, dout = grid_inputs(5, 1, 1, 1, 4)
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, dout)
    assert np.array_equal(dv, dout.astype(np.float64)) and not dq.any() and not dk.any()


def test_far_keys_carry_tiny_but_nonzero_gradient_in_fp64():
    # sec. 5.1: in fp64 a key far past the blindness distance keeps a tiny nonzero
    # weight, so it still receives gradient (an fp32 flush-to-zero exponential would
    # give exactly 0). Only rows at distance >= 150 from key 0 have nonzero dO, so
    # dV_0 is made of weights below e^-140 alone; it must equal the forward weights'
    # sum_i w_i0 dO_i.
    N, d = 200, 4
    q, k, v, dout = grid_inputs(6, 1, 1, N, d, scale=0.1)
    dout[:, :, :150] = 0.0
    m = np.array([1.0])  # blindness distance 88 under tau = ln 2^-126
    _, _, dv, _, _ = oracle.attention_bwd(q, k, v, dout, m=m)
    _, _, w = oracle.attention(q, k, v, m=m, want_weights=True)
    want = w[0, 0, :, 0] @ dout[0, 0].astype(np.float64)
    assert np.all(w[0, 0, 150:, 0] < np.exp(-140.0)) and np.all(w[0, 0, 150:, 0] > 0)
    assert np.all(np.abs(dv[0, 0, 0]) > 0) and np.all(np.abs(dv[0, 0, 0]) < 1e-55)
    assert np.allclose(dv[0, 0, 0], want, rtol=1e-12, atol=0)

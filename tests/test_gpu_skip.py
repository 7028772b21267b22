"""Exact underflow-tile skipping (alibi_attn_fwd_ex with ALIBI_FWD_SKIP_UNDERFLOW).

Leaving out KV tiles whose weights flush to zero must not change a single bit
of the output or the LSE ("When Attention Goes Blind", sec. 3.2-3.3 and 5.2:
past the blindness distance the weights are exactly zero)."""
import math

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


def both(ab, q, k, v):
    import torch
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o0, l0 = ab.alibi_attn_fwd(qd, kd, vd)
    o1, l1 = ab.alibi_attn_fwd(qd, kd, vd, skip_underflow=True)
    plan = ab.alibi_attn_skip_plan(qd, kd)
    ab.alibi_check_error()
    return o0, l0, o1, l1, plan.cpu().numpy()


def skipped_fraction(plan, B, H, N):
    NQB = (N + 255) // 256
    NQT = (N + 127) // 128
    tot = skip = 0
    for w, first in enumerate(plan):
        qb = w % NQB
        for qt in (2 * qb, 2 * qb + 1):
            if qt < NQT:
                tot += qt + 1
                skip += min(first, qt + 1)
    return skip / tot


@pytest.mark.parametrize("name", ["long_n16384", "layer_n2048", "heads6_n1024"])
def test_skip_is_bit_identical(ab, name):
    import torch
    w = gen.WORKLOADS[name]
    q, k, v = gen.generate(w)
    o0, l0, o1, l1, plan = both(ab, q, k, v)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    NQB = (w.N + 255) // 256
    assert all(0 <= plan[i] <= 2 * (i % NQB) for i in range(len(plan)))
    frac = skipped_fraction(plan, w.B, w.H, w.N)
    if name == "long_n16384":
        # most causal pairs of the 16-head long-context layer are past the blindness distance
        assert frac > 0.4, frac
    # and the skipping result still matches the oracle
    rows = sample_rows(w.B, w.H, w.N, max_heads=6, per_head=8)
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, rows=rows)
    assert_bf16_out(host64(o1).reshape(-1, w.d)[rows], ro)
    assert_close(host64(l1).reshape(-1)[rows], rl, TOL_BF16_LSE, "lse")


def test_skip_at_the_flush_margin(ab):
    # A = 0 (Q = 0): every exponent is exactly -m (i - j) log2(e); tiles straddle the
    # flush threshold 2^-126 for several heads. Skipped or not, the result is identical.
    import torch
    H, N, d = 16, 3000, 128
    q = gen.make_tensor(np.zeros((1, H, N, d)), (1, H, N, d), "bf16")
    _, k, v = gen.random_case(3, 1, H, N, d, dtype="bf16")
    o0, l0, o1, l1, plan = both(ab, q, k, v)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert plan.max() > 0


def test_skipped_entries_truly_underflow():
    # Independent check of the plan's bound on sampled items: every entry the plan
    # leaves out has x_ij - max_j x_ij <= -126 (base 2) against the oracle's exact
    # row maxima, i.e. its weight is below the smallest normal fp32 number.
    import torch
    import alibi_positional_bias_gb300 as ab
    w = gen.WORKLOADS["long_n16384"].with_n(4096)
    q, k, _ = gen.generate(w)
    plan = ab.alibi_attn_skip_plan(dev(q, "bf16"), dev(k, "bf16")).cpu().numpy()
    ab.alibi_check_error()
    m = oracle.slopes(w.H)
    NQB = (w.N + 255) // 256
    rng = np.random.default_rng(0)
    checked = 0
    for item in rng.choice(len(plan), size=24, replace=False):
        first = int(plan[item])
        if first == 0:
            continue
        bh, qb = divmod(int(item), NQB)
        h = bh % w.H
        rows = np.arange(256 * qb, min(w.N, 256 * qb + 256))
        Q = q.f32[0, h, rows].astype(np.float64)
        K = k.f32[0, h].astype(np.float64)
        x = (Q @ K.T) / math.sqrt(w.d) - m[h] * (rows[:, None] - np.arange(w.N)[None, :])
        x[np.arange(w.N)[None, :] > rows[:, None]] = -np.inf
        M = x.max(axis=1)
        skipped = x[:, : 128 * first] - M[:, None]
        assert (skipped * math.log2(math.e) <= -126.0).all()
        checked += 1
    assert checked > 5


def test_skip_more_heads_than_grid_rows(ab):
    # B*H = 70000 (b, h) pairs, past the 65535 a second grid dimension holds: the
    # plan's key-norm pass runs on a one-dimensional grid. N = 300 gives every head
    # a second 256-row block whose far tiles the steep heads of the 100-head
    # schedule leave out; the output must stay bit-identical to the dense kernel.
    import torch
    B, H, N, d = 700, 100, 300, 16
    g = torch.Generator(device="cuda").manual_seed(70000)
    q, k, v = (torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o0, l0 = ab.alibi_attn_fwd(q, k, v)
    o1, l1 = ab.alibi_attn_fwd(q, k, v, skip_underflow=True)
    plan = ab.alibi_attn_skip_plan(q, k).cpu().numpy()
    ab.alibi_check_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert plan.max() > 0  # some tiles were left out


@pytest.mark.parametrize("N", [1_540_000, 1_600_000])
def test_skip_plan_longest_sequences(ab, N):
    # The plan's work order is a counting sort over item lengths in one CTA's
    # shared memory (one int per possible length: 128-key tiles + 1). At 1.54M keys
    # the 12033 bins still fit the 48 KB a launch gets by default; at 1.6M (12501
    # bins) the plan keeps the nominal order instead. Both stay bit-identical to
    # the dense kernel.
    import torch
    B, H, d = 1, 1, 16
    g = torch.Generator(device="cuda").manual_seed(N)
    q, k, v = (torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o0, l0 = ab.alibi_attn_fwd(q, k, v)
    o1, l1 = ab.alibi_attn_fwd(q, k, v, skip_underflow=True)
    ab.alibi_check_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)

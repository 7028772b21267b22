"""Caller-chosen slopes in the tensor-core prefill: the robust / explicit
schedules of "When Attention Goes Blind" (sec. 3.4 "Robust Slopes", sec. 4.2
configurations, Table 8) against the oracle given the same fp32 slopes."""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_BF16_LSE, assert_bf16_out, assert_close, dev, host64

pytestmark = pytest.mark.gpu

# (delta_first, delta_last) of the Table 8 rows, nine heads each
SCHEDULES = {"Steep": (128, 512), "Safe": (2048, 4096), "Wide": (16, 4096), "Explicit": (32, 8192)}


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("name", sorted(SCHEDULES))
def test_table8_schedules(ab, name, causal):
    H, N, d = 9, 1100, 64
    m = ab.alibi_slopes_explicit(H, *SCHEDULES[name])
    q, k, v = gen.random_case(40 + len(name), 1, H, N, d, dtype="bf16")
    out, lse = ab.alibi_attn_fwd_ex(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=causal, slopes=m)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, m=m.astype(np.float64), causal=causal)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_explicit_log_distance_combination(ab):
    # E+L (sec. 4.3): slopes adapted to log-scaled distances, run with ALIBI_FWD_LOGDIST
    H, N, d = 9, 900, 128
    m = ab.alibi_slopes_explicit(H, 32, 8192, log_distance=True)
    q, k, v = gen.random_case(48, 1, H, N, d, dtype="bf16")
    out, lse = ab.alibi_attn_fwd_ex(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), flags=4, slopes=m)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, m=m.astype(np.float64), variant=oracle.LOGDIST)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_default_slopes_passed_explicitly_are_bit_identical(ab):
    import torch
    q, k, v = gen.random_case(49, 2, 6, 600, 128, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o0, l0 = ab.alibi_attn_fwd(qd, kd, vd)
    o1, l1 = ab.alibi_attn_fwd_ex(qd, kd, vd, slopes=ab.alibi_slopes(6))
    ab.alibi_check_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_zero_slopes_are_plain_attention(ab, causal):
    # m = 0 removes the bias: plain (masked) softmax attention
    H, N, d = 3, 300, 64
    q, k, v = gen.random_case(50, 1, H, N, d, dtype="bf16")
    out, lse = ab.alibi_attn_fwd_ex(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), causal=causal,
                                    slopes=np.zeros(H, np.float32))
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, m=np.zeros(H), causal=causal)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_skip_with_steep_schedule_is_bit_identical(ab):
    # The Steep schedule (delta_H = 512) blinds every head early, so exact underflow
    # skipping leaves out most far tiles; the result must not move by a bit.
    import torch
    H, N, d = 9, 4096, 128
    m = ab.alibi_slopes_explicit(H, *SCHEDULES["Steep"])
    q, k, v = gen.random_case(51, 1, H, N, d, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o0, l0 = ab.alibi_attn_fwd_ex(qd, kd, vd, slopes=m)
    o1, l1 = ab.alibi_attn_fwd_ex(qd, kd, vd, flags=1, slopes=m)
    ab.alibi_check_error()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    rows = np.array([h * N + i for h in range(H) for i in (0, 127, 128, 1000, 2047, 4095)])
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, m=m.astype(np.float64), rows=rows)
    assert_bf16_out(host64(o1).reshape(-1, d)[rows], ro)
    assert_close(host64(l1).reshape(-1)[rows], rl, TOL_BF16_LSE, "lse")

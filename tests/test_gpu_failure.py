"""Failure detection without a GPU fault: a bounded device-side wait that is made
to run out (a barrier nothing arrives on, or a Q tile the prefill producer leaves
out) must come back as ALIBI_ERR_TIMEOUT, the kernel must drain its own work and
return, and the context must stay usable afterwards. An error left uncollected
must not spoil later calls."""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_BF16_LSE, assert_bf16_out, assert_close, dev, host64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    ab.alibi_check_error()  # start clean
    ab.alibi_selftest_timeout()
    with pytest.raises(ab.AlibiError) as exc:
        ab.alibi_check_error()
    assert exc.value.status == ab.ALIBI_ERR_TIMEOUT
    ab.alibi_check_error()  # the status word was cleared
    q, k, v = gen.random_case(4, 1, 2, 200, 128, dtype="bf16")
    out, lse = ab.alibi_attn_fwd(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"))
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_kernel_timeout_drains_and_context_survives(d):
    # the prefill kernel's own failure path: every CTA's first item's Q tiles are never
    # loaded, the MMA issuer's wait for them runs out after 20 ms, the other roles
    # stop, the issued loads and MMAs are waited for and TMEM is freed
    import torch
    import alibi_positional_bias_gb300 as ab
    ab.load()
    ab.alibi_check_error()
    q, k, v = gen.random_case(11, 1, 2, 300, d, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    ab.alibi_selftest_fwd_timeout(qd, kd, vd, wait_us=20000)
    with pytest.raises(ab.AlibiError) as exc:
        ab.alibi_check_error()
    assert exc.value.status == ab.ALIBI_ERR_TIMEOUT
    ab.alibi_check_error()
    out, lse = ab.alibi_attn_fwd(qd, kd, vd)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_uncollected_timeout_does_not_void_later_calls():
    # a timeout nobody collected with alibi_check_error stays in the status word;
    # prefill and backward launched after it still compute correct results, and
    # the next check still reports the timeout
    import torch
    import alibi_positional_bias_gb300 as ab
    ab.load()
    ab.alibi_check_error()
    ab.alibi_selftest_timeout()
    q, k, v = gen.random_case(12, 1, 2, 333, 128, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    out, lse = ab.alibi_attn_fwd(qd, kd, vd)
    dout = torch.randn_like(out)
    dq, dk, dv = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dout)
    out2, lse2 = ab.alibi_attn_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    with pytest.raises(ab.AlibiError) as exc:
        ab.alibi_check_error()
    assert exc.value.status == ab.ALIBI_ERR_TIMEOUT
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # the backward after the stale error equals one run on a clean word
    dq2, dk2, dv2 = ab.alibi_attn_bwd(qd, kd, vd, out, lse, dout)
    ab.alibi_check_error()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)

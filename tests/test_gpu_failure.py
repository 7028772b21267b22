"""Failure detection without a GPU fault: a bounded device-side wait that is made
to run out (a barrier nothing arrives on) must come back as ALIBI_ERR_TIMEOUT,
and the context must stay usable afterwards."""
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

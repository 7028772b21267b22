"""The mitigations of "When Attention Goes Blind" sec. 3.4 in the tensor-core
prefill (clamped bias, log-scaled distance, soft-capped logits, and their
combinations) against the oracle's pinned variants (c_clamp = -87 and z = 50 as
in sec. 4.3)."""
import itertools

import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_BF16_LSE, assert_bf16_out, assert_close, dev, host64

pytestmark = pytest.mark.gpu

# ABI flag -> oracle variant bit
ABI = {"clamp": 2, "logdist": 4, "softcap": 8}
ORC = {"clamp": oracle.CLAMP, "logdist": oracle.LOGDIST, "softcap": oracle.SOFTCAP}
COMBOS = [c for r in (1, 2, 3) for c in itertools.combinations(("clamp", "logdist", "softcap"), r)]


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


@pytest.mark.parametrize("combo", COMBOS, ids=["+".join(c) for c in COMBOS])
@pytest.mark.parametrize("B,H,N,d,sigma,c_clamp", [(1, 4, 1000, 64, 1.0, -87.0), (1, 3, 777, 128, 4.0, -87.0),
                                                   (2, 2, 300, 128, 1.0, -3.0)])
def test_mitigation_variants(ab, combo, B, H, N, d, sigma, c_clamp):
    # c_clamp = -87 is the paper's choice (sec. 4.3); -3 makes the clamp change the output itself.
    # sigma scales Q and K only (large logits exercise the soft cap); V stays N(0, 1), the
    # scale the bf16 output tolerance is stated for.
    q, k, _ = gen.random_case(31 + N + d, B, H, N, d, dtype="bf16", sigma=sigma)
    _, _, v = gen.random_case(32 + N + d, B, H, N, d, dtype="bf16")
    flags = sum(ABI[c] for c in combo)
    out, lse = ab.alibi_attn_fwd_ex(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), flags=flags,
                                    clamp_min=c_clamp, softcap_z=50.0)
    ab.alibi_check_error()
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, variant=sum(ORC[c] for c in combo), c_clamp=c_clamp,
                                 z_cap=50.0)
    assert_bf16_out(host64(out), ro)
    assert_close(host64(lse), rl, TOL_BF16_LSE, "lse")


def test_variants_change_the_result(ab):
    # each mitigation must actually act on these inputs (otherwise the parity test is vacuous)
    import torch
    q, k, _ = gen.random_case(5, 1, 4, 1000, 128, dtype="bf16", sigma=4.0)
    _, _, v = gen.random_case(6, 1, 4, 1000, 128, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    _, l0 = ab.alibi_attn_fwd(qd, kd, vd)
    for c in ("clamp", "logdist", "softcap"):
        _, l1 = ab.alibi_attn_fwd_ex(qd, kd, vd, flags=ABI[c], clamp_min=-3.0)
        assert (l1 - l0).abs().max().item() > 1e-2, c
    ab.alibi_check_error()

"""fp32 reference-precision path vs the fp64 oracle (through the C ABI)."""
import os

import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import TOL_F32, assert_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


def run_f32(ab, q, k, v):
    qd, kd, vd = dev(q, "fp32"), dev(k, "fp32"), dev(v, "fp32")
    out, lse = ab.alibi_attn_fwd_f32(qd, kd, vd)
    P = ab.alibi_attn_probs_f32(qd, kd, lse)
    ab.alibi_check_error()
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), P.cpu().numpy().astype(np.float64)


def test_tiny_fp32_workload(ab):
    # B=1, H=4, N=64, d=16, fp32 N(0, 0.5^2) from seed 42: outputs and full weights
    q, k, v = gen.generate(gen.WORKLOADS["tiny_fp32"])
    out, lse, P = run_f32(ab, q, k, v)
    ro, rl, rw = oracle.attention(q.f32, k.f32, v.f32, want_weights=True)
    assert_close(out, ro, TOL_F32, "out")
    assert_close(lse, rl, TOL_F32, "lse")
    assert_close(P, rw, TOL_F32, "weights")


def test_p4_printed_matrices_on_gpu(ab):
    # "ALiBi in Attention: Complete Implementation", seed-42 example, heads 1 and 4
    q, k, v = gen.generate(gen.WORKLOADS["p4_example"])
    _, _, P = run_f32(ab, q, k, v)
    golden = os.path.join(os.path.dirname(__file__), "golden", "p4_seed42_weights.txt")
    mats, cur = {}, None
    for line in open(golden):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("head"):
            cur = int(line.split()[1])
            mats[cur] = []
        else:
            mats[cur].append([float(x) for x in line.split()])
    for h, m in mats.items():
        assert np.abs(P[0, h] - np.array(m)).max() <= 5e-4 + 1e-9


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 16), (1, 2, 7, 1), (2, 3, 33, 33), (1, 2, 100, 64),
                                     (1, 1, 65, 128), (1, 2, 40, 256), (2, 5, 130, 16)])
def test_fp32_shape_sweep(ab, B, H, N, d):
    q, k, v = gen.random_case(100 + N + d, B, H, N, d, dtype="fp32", sigma=0.5)
    out, lse, P = run_f32(ab, q, k, v)
    ro, rl, rw = oracle.attention(q.f32, k.f32, v.f32, want_weights=True)
    assert_close(out, ro, TOL_F32, "out")
    assert_close(lse, rl, TOL_F32, "lse")
    assert_close(P, rw, TOL_F32, "weights")

"""bf16 underflow counter vs the fp64 oracle, and closed forms at full size."""
import math

import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import dev

pytestmark = pytest.mark.gpu
TAU_D = math.log(2.0 ** -126)


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


def band_for(H, N):
    # The kernel forms x_ij - M_i in fp32: the bias m (i - j) reaches m_max N and
    # carries relative error ~2^-22 (slope rounding + product), the dot product
    # ~1e-5 absolute. Entries closer than this to tau may be classified either way.
    return 4e-7 * float(oracle.slopes(H).max()) * N + 1e-4


def gpu_counts(ab, q, k):
    c = ab.alibi_attn_underflow_bf16(dev(q, "bf16"), dev(k, "bf16"), TAU_D)
    ab.alibi_check_error()
    return c.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("name,n", [("heads6_n1024", None), ("long_n16384", 2048), ("layer_n2048", 512)])
def test_counts_match_oracle(ab, name, n):
    # causal rows depend only on earlier keys, so an N-prefix of a workload is a
    # complete problem of its own
    w = gen.WORKLOADS[name] if n is None else gen.WORKLOADS[name].with_n(n)
    q, k, _ = gen.generate(w)
    got = gpu_counts(ab, q, k)
    want, near = oracle.underflow_counts_per_head(q.f32, k.f32, TAU_D, band=band_for(w.H, w.N))
    diff = np.abs(got - want.astype(np.int64))
    assert (diff <= near.astype(np.int64)).all(), (got, want, near)


def test_zero_logits_closed_form_full_size(ab):
    # A = 0 (Q = 0): per head the count is (N - w)(N - w + 1)/2 with
    # w = min{D : -m D <= tau}, at the long-context size N = 16384.
    import torch
    H, N, d = 16, 16384, 128
    q = torch.zeros((1, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((1, H, N, d), generator=torch.Generator().manual_seed(0)).to(torch.bfloat16).cuda()
    c = ab.alibi_attn_underflow_bf16(q, k, TAU_D).cpu().numpy()
    ab.alibi_check_error()
    for h, m in enumerate(oracle.slopes(H)):
        w = int(oracle.blindness_int(m))
        want = (N - w) * (N - w + 1) // 2 if w < N else 0
        # exact except where m D lands within rounding of tau for some distance D
        assert abs(int(c[h]) - want) <= N, (h, int(c[h]), want)


def test_counts_more_heads_than_grid_rows(ab):
    # B*H = 70000 (b, h) pairs: more than the 65535 rows a y grid dimension can hold
    w = gen.Workload("uf", "prefill", 700, 100, 8, 16, "bf16", seed=17)
    q, k, _ = gen.generate(w)
    got = gpu_counts(ab, q, k)
    want, near = oracle.underflow_counts_per_head(q.f32, k.f32, TAU_D, band=band_for(w.H, w.N))
    diff = np.abs(got - want.astype(np.int64))
    assert (diff <= near.astype(np.int64)).all(), (got, want, near)


@pytest.mark.parametrize("B,H,L,d", [(2, 40, 8192, 128), (3, 5, 1000, 64), (1, 4, 1, 128), (2, 3, 777, 16)])
def test_decode_row_counts_match_oracle(ab, B, H, L, d):
    # The decode row is prefill row L-1 of the same sequence ("ALiBi: Attention with
    # Linear Biases", KV-cache paragraph): the oracle counts it as that row of a
    # prefill problem whose other query rows are never read.
    w = gen.Workload("ufdec", "decode", B, H, L, d, "bf16", seed=23 + L)
    q, k, _ = gen.generate(w)
    c = ab.alibi_decode_underflow_bf16(dev(q, "bf16"), dev(k, "bf16"), TAU_D)
    ab.alibi_check_error()
    got = c.cpu().numpy().astype(np.int64)
    qfull = np.zeros((B, H, L, d), np.float32)
    qfull[:, :, L - 1] = q.f32
    rows = np.arange(B * H, dtype=np.int64) * L + (L - 1)
    cnt, near = oracle.underflow_rows(qfull, k.f32, TAU_D, rows=rows, band=band_for(H, L))
    want = cnt.reshape(B, H).sum(0).astype(np.int64)
    nr = near.reshape(B, H).sum(0).astype(np.int64)
    assert (np.abs(got - want) <= nr).all(), (got, want, nr)
    if L > 2000:
        assert want.sum() > 0  # the steep heads do underflow at this length

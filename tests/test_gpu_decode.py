"""bf16 split-K decode vs the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest

import alibi_inputs as gen
import oracle
from gpu_helpers import assert_bf16_out, dev, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


@pytest.mark.parametrize("B,H,L", [(1, 1, 1), (1, 3, 5), (2, 2, 16), (1, 2, 17), (1, 4, 100), (2, 3, 513),
                                   (1, 1, 1000), (3, 5, 4097), (1, 2, 20000), (4, 40, 300)])
def test_decode_sweep(ab, B, H, L):
    w = gen.Workload("dec", "decode", B, H, L, 128, "bf16", seed=11 + L)
    q, k, v = gen.generate(w)
    out = ab.alibi_attn_decode(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"))
    ab.alibi_check_error()
    ro, _ = oracle.decode(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("B,H,L", [(1, 3, 5), (2, 2, 129), (1, 4, 1000), (3, 5, 4097), (1, 2, 20000)])
def test_decode_head_sizes(ab, B, H, L, d):
    # the smaller head sizes: one key row per d/8 lanes, with and without split-K
    w = gen.Workload("dec", "decode", B, H, L, d, "bf16", seed=31 + L + d)
    q, k, v = gen.generate(w)
    out = ab.alibi_attn_decode(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"))
    out2 = ab.alibi_attn_decode_noalloc(dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), out.clone())
    ab.alibi_check_error()
    ro, _ = oracle.decode(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    assert np.array_equal(host64(out), host64(out2))


def test_decode_matches_prefill_last_row(ab):
    # decode at position L-1 sees what prefill row L-1 sees (same kernel family, same inputs)
    B, H, L = 1, 4, 777
    q, k, v = gen.random_case(21, B, H, L, 128, dtype="bf16")
    qd = gen.make_tensor(q.f32[:, :, L - 1, :], (B, H, 128), "bf16")
    out = ab.alibi_attn_decode(dev(qd, "bf16"), dev(k, "bf16"), dev(v, "bf16"))
    ab.alibi_check_error()
    ro, _, _ = oracle.attention(q.f32, k.f32, v.f32, rows=[h * L + L - 1 for h in range(H)])
    assert_bf16_out(host64(out).reshape(H, 128), ro)


def test_decode_full_size_every_head(ab):
    # B=64 sequences, H=40 (32-head schedule + alternating 64-head entries),
    # L=8192, d=128: the benchmark's launch; the oracle checks every one of the
    # 2560 (b, h), one sequence at a time (inputs regenerated on the host from
    # the same counter streams)
    import torch
    w = gen.WORKLOADS["decode_l8192"]
    qs, ks, _ = w.shapes()
    qd = torch.empty(qs, dtype=torch.bfloat16, device="cuda")
    kd = torch.empty(ks, dtype=torch.bfloat16, device="cuda")
    vd = torch.empty(ks, dtype=torch.bfloat16, device="cuda")
    for i, t in enumerate((qd, kd, vd)):
        gen.fill_device(w, i, t)
    out = host64(ab.alibi_attn_decode(qd, kd, vd))
    ab.alibi_check_error()
    assert np.isfinite(out).all()
    m = oracle.slopes(w.H)
    per_q, per_kv = w.H * w.d, w.H * w.N * w.d
    for b in range(w.B):
        q = gen.make_tensor(gen.tensor_values(w, 0, b * per_q, per_q), (1, w.H, w.d), "bf16")
        k = gen.make_tensor(gen.tensor_values(w, 1, b * per_kv, per_kv), (1, w.H, w.N, w.d), "bf16")
        v = gen.make_tensor(gen.tensor_values(w, 2, b * per_kv, per_kv), (1, w.H, w.N, w.d), "bf16")
        ro, _ = oracle.decode(q.f32, k.f32, v.f32, m=m)
        assert_bf16_out(out[b], ro[0], what=f"out[{b}]")


def test_decode_more_heads_than_grid_rows(ab):
    # B*H = 71680 (b, h) pairs: more than the 65535 rows a y grid dimension can hold;
    # dense and skipping decode both against the oracle, every head
    B, H, L, d = 1024, 70, 20, 16
    w = gen.Workload("dec", "decode", B, H, L, d, "bf16", seed=91)
    q, k, v = gen.generate(w)
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    out = ab.alibi_attn_decode(qd, kd, vd)
    knorm = ab.alibi_kv_block_norms(kd)
    out_s = ab.alibi_attn_decode_skip(qd, kd, vd, knorm)
    ab.alibi_check_error()
    ro, _ = oracle.decode(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    assert_bf16_out(host64(out_s), ro)
    # block norms of the last (b, h), computed directly
    kl = k.f32[-1, -1].astype(np.float64)
    assert abs(float(knorm[-1, -1, 0]) - np.sqrt((kl * kl).sum(axis=1)).max()) <= 1e-5 * np.sqrt((kl * kl).sum(axis=1)).max()

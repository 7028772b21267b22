"""Decode that skips provably underflowed cache rows (alibi_attn_decode_skip with
the block norms of alibi_kv_block_norms): "When Attention Goes Blind" sec. 3.2-3.3
and 5.2, where past a head's blindness distance every weight is exactly zero."""
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


def ref_norms(k: np.ndarray) -> np.ndarray:
    B, H, L, d = k.shape
    nb = (L + 63) // 64
    pad = np.zeros((B, H, nb * 64, d))
    pad[:, :, :L] = k
    return np.sqrt((pad.reshape(B, H, nb, 64, d) ** 2).sum(-1)).max(-1)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_block_norms(ab, d):
    w = gen.Workload("kn", "decode", 2, 3, 1000, d, "bf16", seed=7 + d)
    _, k, _ = gen.generate(w)
    kn = host64(ab.alibi_kv_block_norms(dev(k, "bf16")))
    ab.alibi_check_error()
    want = ref_norms(k.f32.astype(np.float64))
    assert np.abs(kn - want).max() <= 1e-6 * want.max()


def test_block_norms_tail_refresh(ab):
    # appending keys: refreshing the blocks from the old length's block on equals a full pass
    import torch
    w = gen.Workload("kn", "decode", 1, 4, 1500, 128, "bf16", seed=9)
    _, k, _ = gen.generate(w)
    kd = dev(k, "bf16")
    full = ab.alibi_kv_block_norms(kd)
    part = ab.alibi_kv_block_norms(kd[:, :, :1000].contiguous())
    tail = torch.zeros_like(full)
    tail[:, :, : part.shape[2]] = part
    ab.alibi_kv_block_norms(kd, knorm=tail, blk_begin=1000 // 64)
    ab.alibi_check_error()
    assert torch.equal(tail, full)


@pytest.mark.parametrize("B,H,L,d", [(1, 3, 5, 128), (2, 8, 700, 128), (2, 40, 4097, 128), (1, 32, 20000, 64),
                                     (3, 16, 3000, 32), (2, 12, 5000, 16)])
def test_decode_skip_vs_oracle(ab, B, H, L, d):
    w = gen.Workload("dsk", "decode", B, H, L, d, "bf16", seed=41 + L + d)
    q, k, v = gen.generate(w)
    kd = dev(k, "bf16")
    kn = ab.alibi_kv_block_norms(kd)
    out = ab.alibi_attn_decode_skip(dev(q, "bf16"), kd, dev(v, "bf16"), kn)
    dense = ab.alibi_attn_decode(dev(q, "bf16"), kd, dev(v, "bf16"))
    ab.alibi_check_error()
    ro, _ = oracle.decode(q.f32, k.f32, v.f32)
    assert_bf16_out(host64(out), ro)
    # the omitted weights are below 2^-127 of the largest: the two kernels agree to bf16 rounding
    assert np.abs(host64(out) - host64(dense)).max() <= 2.0 ** -7


def test_decode_skip_never_reads_skipped_rows(ab):
    # Rows 0..2047 of a 4096-long cache get K = 0 and V = NaN. For the steep heads of the
    # 32-head schedule (m_h >= 2^-17/4, heads 0..16) those rows lie past the blindness
    # distance: the skipping decode must not read them (finite output equal to the oracle
    # without them), while the dense decode does read them (0 x NaN = NaN).
    B, H, L, d = 1, 32, 4096, 128
    w = gen.Workload("nan", "decode", B, H, L, d, "bf16", seed=77)
    q, k, v = gen.generate(w)
    kf, vf = k.f32.copy(), v.f32.copy()
    kf[:, :, :2048] = 0.0
    v0 = vf.copy()
    v0[:, :, :2048] = 0.0
    vf[:, :, :2048] = np.nan
    kt, vt = gen.make_tensor(kf, kf.shape, "bf16"), gen.make_tensor(vf, vf.shape, "bf16")
    kd = dev(kt, "bf16")
    kn = ab.alibi_kv_block_norms(kd)
    out = host64(ab.alibi_attn_decode_skip(dev(q, "bf16"), kd, dev(vt, "bf16"), kn))
    dense = host64(ab.alibi_attn_decode(dev(q, "bf16"), kd, dev(vt, "bf16")))
    ab.alibi_check_error()
    steep = slice(0, 17)
    ro, _ = oracle.decode(q.f32, kf, v0)
    assert np.isfinite(out[:, steep]).all()
    assert_bf16_out(out[:, steep], ro[:, steep])
    assert np.isnan(dense[:, steep]).any()


def test_decode_skip_full_size(ab):
    # the benchmark's decode workload (B=64, H=40, L=8192, d=128) on sampled heads
    import torch
    w = gen.WORKLOADS["decode_l8192"]
    qs, ks, _ = w.shapes()
    qd = torch.empty(qs, dtype=torch.bfloat16, device="cuda")
    kd = torch.empty(ks, dtype=torch.bfloat16, device="cuda")
    vd = torch.empty(ks, dtype=torch.bfloat16, device="cuda")
    for i, t in enumerate((qd, kd, vd)):
        gen.fill_device(w, i, t)
    kn = ab.alibi_kv_block_norms(kd)
    out = host64(ab.alibi_attn_decode_skip(qd, kd, vd, kn))
    dense = host64(ab.alibi_attn_decode(qd, kd, vd))
    ab.alibi_check_error()
    assert np.isfinite(out).all()
    assert np.abs(out - dense).max() <= 2.0 ** -7
    m = oracle.slopes(w.H)
    for b, h in [(0, 0), (63, 39), (5, 3), (17, 20)]:
        qh = gen.head_slice(w, 0, b, h)
        kh = gen.head_slice(w, 1, b, h)
        vh = gen.head_slice(w, 2, b, h)
        ro, _ = oracle.decode(qh.f32[None, None], kh.f32[None, None], vh.f32[None, None], m=m[h:h + 1])
        assert_bf16_out(out[b, h][None, None], ro)

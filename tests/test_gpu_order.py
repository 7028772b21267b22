"""Work order of dense launches whose streamed tiles exceed half the L2.

Such launches (prefill, and the backward's dK/dV and dQ kernels) run their items
in the blocked order (csrc/work_order.h) from tables the library builds once per
shape. Every item computes the same values in either order, so output, LSE and
gradients must be bit-identical to the nominal order (ALIBI_FWD_NOMINAL_ORDER),
for the plain kernels, the mitigation kernels and the D = 64 kernels, causal
and not, on shapes that take the blocked order: several block counts per head,
a ragged N with an odd number of tiles, and a launch made while its stream is
being captured (which keeps the nominal order until the shape has a table). The
ragged prefill is also checked against the oracle on sampled rows of every
head."""
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


def blocked_regime(B, H, N, d):
    # the prefill's rule (causal or not): K and V above half the L2, at most 16
    # blocks of 256 rows per head
    import torch
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return 4 * B * H * N * d > l2 / 2 and 2 <= (N + 255) // 256 <= 16


def both_orders(ab, q, k, v, flags=0, **kw):
    o1, l1 = ab.alibi_attn_fwd_ex(q, k, v, flags=flags, **kw)
    o2, l2 = ab.alibi_attn_fwd_ex(q, k, v, flags=flags | ab.ALIBI_FWD_NOMINAL_ORDER, **kw)
    ab.alibi_check_error()
    return o1, l1, o2, l2


@pytest.mark.parametrize("B,H,N,d", [
    (4, 32, 2048, 128),    # the decoder-layer shape: 8 blocks per head
    (16, 32, 1024, 128),   # 4 blocks per head, 512 heads
    (4, 32, 4096, 128),    # 16 blocks per head
    (16, 32, 1024, 64),    # the D = 64 kernel
    (32, 32, 1024, 32),    # head size 32 on the D = 64 kernel
    (64, 32, 1024, 16),    # head size 16 on the D = 64 kernel
])
def test_blocked_order_bit_identical(ab, B, H, N, d):
    import torch
    assert blocked_regime(B, H, N, d)
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + N + d)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    o1, l1, o2, l2 = both_orders(ab, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.isfinite(o1).all() and torch.isfinite(l1).all()


@pytest.mark.parametrize("B,H,N,d", [(4, 32, 2048, 128), (16, 32, 1024, 64), (8, 20, 1900, 128)])
def test_blocked_order_noncausal(ab, B, H, N, d):
    # the symmetric bias over all keys: every item has the same length and the
    # blocked order is taken as it is; forward and backward bit-identical
    import torch
    assert blocked_regime(B, H, N, d)
    g = torch.Generator(device="cuda").manual_seed(B + H + N + d + 77)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    do = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    o1, l1 = ab.alibi_attn_fwd_ex(q, k, v, causal=False)
    o2, l2 = ab.alibi_attn_fwd_ex(q, k, v, causal=False, flags=ab.ALIBI_FWD_NOMINAL_ORDER)
    g1 = ab.alibi_attn_bwd(q, k, v, o1, l1, do, causal=False)
    g2 = ab.alibi_attn_bwd(q, k, v, o1, l1, do, causal=False, flags=ab.ALIBI_FWD_NOMINAL_ORDER)
    ab.alibi_check_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b, name in zip(g1, g2, ("dq", "dk", "dv")):
        assert torch.equal(a, b), name


def test_blocked_order_mitigation_kernel(ab):
    import torch
    B, H, N, d = 4, 32, 2048, 128
    g = torch.Generator(device="cuda").manual_seed(11)
    q = (3 * torch.randn(B, H, N, d, device="cuda", generator=g)).bfloat16()
    k = (3 * torch.randn(B, H, N, d, device="cuda", generator=g)).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    o1, l1, o2, l2 = both_orders(ab, q, k, v, flags=ab.ALIBI_FWD_CLAMP | ab.ALIBI_FWD_SOFTCAP, clamp_min=-20.0,
                                 softcap_z=30.0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # the symmetric bias with log-scaled distances
    o1 = ab.alibi_attn_fwd_ex(q, k, v, causal=False, flags=ab.ALIBI_FWD_LOGDIST)
    o2 = ab.alibi_attn_fwd_ex(q, k, v, causal=False, flags=ab.ALIBI_FWD_LOGDIST | ab.ALIBI_FWD_NOMINAL_ORDER)
    ab.alibi_check_error()
    assert torch.equal(o1[0], o2[0]) and torch.equal(o1[1], o2[1])


def test_blocked_order_ragged_vs_oracle(ab):
    # N = 1900: 15 Q tiles, so the last block of every head has one Q tile
    import torch
    B, H, N, d = 8, 20, 1900, 128
    assert blocked_regime(B, H, N, d)
    q, k, v = gen.random_case(1900, B, H, N, d, dtype="bf16")
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    o1, l1, o2, l2 = both_orders(ab, qd, kd, vd)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    out, lse = host64(o1), host64(l1)
    rows = sample_rows(B, H, N, max_heads=B * H, per_head=12, seed=N)
    assert len(np.unique(rows // N)) == B * H
    ro, rl, _ = oracle.attention(q.f32, k.f32, v.f32, rows=rows)
    assert_bf16_out(out.reshape(-1, d)[rows], ro)
    assert_close(lse.reshape(-1)[rows], rl, TOL_BF16_LSE, "lse")


def test_blocked_order_under_capture(ab):
    # a shape first launched inside a stream capture keeps the nominal order (no
    # table can be built there); replaying the graph, and a later launch of the
    # same shape outside capture (which builds the table), give identical results
    import torch
    B, H, N, d = 24, 16, 1024, 128   # a shape no other test launches
    assert blocked_regime(B, H, N, d)
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    # one launch of another shape first, so nothing but the launch itself is left to
    # happen inside the capture
    ab.alibi_attn_fwd(q[:1, :1].contiguous(), k[:1, :1].contiguous(), v[:1, :1].contiguous())
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ab.alibi_attn_fwd(q, k, v, out=out, lse=lse)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ab.alibi_check_error()
    o2, l2 = ab.alibi_attn_fwd(q, k, v)
    o3, l3 = ab.alibi_attn_fwd_ex(q, k, v, flags=ab.ALIBI_FWD_NOMINAL_ORDER)
    ab.alibi_check_error()
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert torch.equal(o2, o3) and torch.equal(l2, l3)


@pytest.mark.parametrize("B,H,N,d,flags", [
    (1, 16, 16384, 128, 0),    # the long-context shape: 128 tiles per head (the backward has no
                               # limit on tiles per head)
    (4, 32, 2048, 128, 0),     # the decoder-layer shape: 16 tiles per head
    (16, 32, 1024, 64, 0),     # the D = 64 kernels, 8 tiles per head
    (8, 20, 1900, 128, 0),     # 15 tiles per head: a ragged last tile
    (4, 32, 2048, 128, 2 | 8),  # clamp + soft cap: the mitigation kernels
])
def test_backward_blocked_order_bit_identical(ab, B, H, N, d, flags):
    # the backward's two kernels take their own blocked orders on the same rule;
    # dQ, dK and dV do not depend on the order (each item writes its own tile)
    import torch
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert 4 * B * H * N * d > l2 / 2  # the backward's rule: the footprint alone
    g = torch.Generator(device="cuda").manual_seed(B + H + N + d + flags)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    do = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    kw = dict(clamp_min=-20.0, softcap_z=30.0)
    out, lse = ab.alibi_attn_fwd_ex(q, k, v, flags=flags, **kw)
    g1 = ab.alibi_attn_bwd(q, k, v, out, lse, do, flags=flags, **kw)
    g2 = ab.alibi_attn_bwd(q, k, v, out, lse, do, flags=flags | ab.ALIBI_FWD_NOMINAL_ORDER, **kw)
    ab.alibi_check_error()
    for a, b, name in zip(g1, g2, ("dq", "dk", "dv")):
        assert torch.equal(a, b), name
        assert torch.isfinite(a).all(), name


def test_blocked_order_from_concurrent_threads(ab):
    # four host threads launch the same new shape (no table yet) on their own streams:
    # one builds the table while the others wait for it; every result equals the
    # nominal order's
    import threading
    import torch
    B, H, N, d = 20, 16, 1024, 128   # a shape no other test launches
    assert blocked_regime(B, H, N, d)
    g = torch.Generator(device="cuda").manual_seed(9)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    ref_o, ref_l = ab.alibi_attn_fwd_ex(q, k, v, flags=ab.ALIBI_FWD_NOMINAL_ORDER)
    torch.cuda.synchronize()
    results, errors = [None] * 4, []

    def worker(t):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                results[t] = ab.alibi_attn_fwd(q, k, v)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    ab.alibi_check_error()
    for o, l in results:
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_backward_blocked_order_in_a_graph(ab):
    # forward and backward of a blocked-order shape captured in a CUDA graph (the
    # tables exist from a first call; the backward's kernels launch as programmatic
    # dependents inside the graph) and replayed: equal to the direct calls
    import torch
    B, H, N, d = 4, 32, 2048, 128
    assert blocked_regime(B, H, N, d)
    g = torch.Generator(device="cuda").manual_seed(21)
    q = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    k = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    v = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    do = torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16()
    o_ref, l_ref = ab.alibi_attn_fwd(q, k, v)
    g_ref = ab.alibi_attn_bwd(q, k, v, o_ref, l_ref, do)
    torch.cuda.synchronize()
    out, lse = torch.empty_like(q), torch.empty(B, H, N, device="cuda")
    grads = [torch.empty_like(q) for _ in range(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ab.alibi_attn_fwd(q, k, v, out=out, lse=lse)
        ab.alibi_attn_bwd(q, k, v, out, lse, do, *grads)
    for _ in range(2):
        for t in (out, lse, *grads):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        ab.alibi_check_error()
        assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)
        for a, b, name in zip(grads, g_ref, ("dq", "dk", "dv")):
            assert torch.equal(a, b), name


CACHE_CHILD = r"""
import torch
import alibi_positional_bias_gb300 as ab
ab.load()
B, H, d = 4, 32, 128
l2 = torch.cuda.get_device_properties(0).L2_cache_size
g = torch.Generator(device="cuda").manual_seed(3)
NMAX = 1100 + 4 * 263
flat = [torch.randn(B * H * NMAX * d, device="cuda", generator=g).bfloat16() for _ in range(3)]
checked = 0
for t in range(264):
    N = 1100 + 4 * t                  # 264 shapes, 5 to 9 blocks per head
    assert 4 * B * H * N * d > l2 / 2
    q, k, v = (f[: B * H * N * d].view(B, H, N, d) for f in flat)
    o1, l1 = ab.alibi_attn_fwd(q, k, v)
    if t in (0, 100, 255, 256, 263):  # before and past the 256 cached shapes
        o2, l2_ = ab.alibi_attn_fwd_ex(q, k, v, flags=ab.ALIBI_FWD_NOMINAL_ORDER)
        assert torch.equal(o1, o2) and torch.equal(l1, l2_), t
        checked += 1
ab.alibi_check_error()
print("ok", checked)
"""


def test_work_order_cache_full():
    # more blocked-order shapes than the library caches tables for (256): the shapes
    # past the cap keep the nominal order, with identical results and no error. A
    # child process, so the full cache does not change the order other tests see.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", CACHE_CHILD], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert r.stdout.strip().endswith("ok 5")


def test_blocked_order_random_shapes(ab):
    # 16 seeded random launches above half the L2 (ragged N, every head size, either
    # mask, plain or mitigated): forward and (d = 64 / 128) backward bit-identical to
    # the nominal order
    import random
    import torch
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    rng = random.Random(2026)
    done = 0
    while done < 16:
        d = rng.choice([16, 32, 64, 128])
        B, H, N = rng.randint(1, 32), rng.randint(1, 64), rng.randint(300, 8192)
        causal = rng.random() < 0.7
        if 4 * B * H * N * d <= l2 / 2 or B * H * N * d > 2 ** 31:
            continue
        flags = rng.choice([0, 0, 0, ab.ALIBI_FWD_CLAMP, ab.ALIBI_FWD_LOGDIST, ab.ALIBI_FWD_SOFTCAP])
        g = torch.Generator(device="cuda").manual_seed(done)
        q, k, v, do = (torch.randn(B, H, N, d, device="cuda", generator=g).bfloat16() for _ in range(4))
        kw = dict(causal=causal, clamp_min=-30.0, softcap_z=40.0)
        o1, l1 = ab.alibi_attn_fwd_ex(q, k, v, flags=flags, **kw)
        o2, l2_ = ab.alibi_attn_fwd_ex(q, k, v, flags=flags | ab.ALIBI_FWD_NOMINAL_ORDER, **kw)
        assert torch.equal(o1, o2) and torch.equal(l1, l2_), (B, H, N, d, causal, flags)
        if d in (64, 128):
            g1 = ab.alibi_attn_bwd(q, k, v, o1, l1, do, flags=flags, **kw)
            g2 = ab.alibi_attn_bwd(q, k, v, o1, l1, do, flags=flags | ab.ALIBI_FWD_NOMINAL_ORDER, **kw)
            assert all(torch.equal(a, b) for a, b in zip(g1, g2)), (B, H, N, d, causal, flags)
        ab.alibi_check_error()
        done += 1

"""The library's calls inside CUDA graphs (a serving loop captures a decode step once
and replays it): capture on torch's graph stream, replay, and compare with direct calls."""
import pytest

import alibi_inputs as gen
from gpu_helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ab():
    import alibi_positional_bias_gb300 as ab
    ab.load()
    return ab


@pytest.mark.parametrize("B,H,L", [(1, 40, 8192), (64, 8, 1024)])  # split (counters, merging CTA) and single pass
def test_decode_graph_replay(ab, B, H, L):
    import torch
    w = gen.Workload("dec", "decode", B, H, L, 128, "bf16", seed=5)
    q, k, v = gen.generate(w)
    qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
    ref = ab.alibi_attn_decode(qd, kd, vd)
    out = torch.empty_like(ref)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ab.alibi_attn_decode(qd, kd, vd, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    ab.alibi_check_error()
    assert torch.equal(out, ref)
    # a new query in the same buffer, replayed without re-capture
    qd.copy_(torch.flip(qd, dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ab.alibi_attn_decode(qd, kd, vd))


def test_prefill_and_backward_graph_replay(ab):
    import torch
    q, k, v = gen.random_case(7, 1, 4, 1000, 128, dtype="bf16")
    do, _, _ = gen.random_case(8, 1, 4, 1000, 128, dtype="bf16")
    qd, kd, vd, dod = (dev(t, "bf16") for t in (q, k, v, do))
    out_r, lse_r = ab.alibi_attn_fwd(qd, kd, vd)
    grads_r = ab.alibi_attn_bwd(qd, kd, vd, out_r, lse_r, dod)
    out, lse = torch.empty_like(out_r), torch.empty_like(lse_r)
    grads = [torch.empty_like(qd) for _ in range(3)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ab.alibi_attn_fwd(qd, kd, vd, out=out, lse=lse)
        ab.alibi_attn_bwd(qd, kd, vd, out, lse, dod, *grads)
    g.replay()
    torch.cuda.synchronize()
    ab.alibi_check_error()
    assert torch.equal(out, out_r) and torch.equal(lse, lse_r)
    assert all(torch.equal(a, b) for a, b in zip(grads, grads_r))

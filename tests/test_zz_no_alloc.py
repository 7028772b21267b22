"""The allocation-free decode entry point, for callers that cannot allocate.

Some callers (a server whose allocator reserved the whole GPU, a real-time
decode loop, a runtime that forbids allocations outside its arena) cannot let
the library allocate the split-K partials buffer. alibi_attn_decode_noalloc
keeps them in a fixed device buffer instead. Its output must match
alibi_attn_decode's on consecutive calls, whatever the previous call left in
the shared buffer.
"""
import ctypes

import numpy as np
import pytest

import alibi_inputs as gen
from gpu_helpers import assert_bf16_out, dev, host64

pytestmark = pytest.mark.gpu


def _noalloc(lib, qd, kd, vd, out, B, H, L, d):
    import torch
    return lib.alibi_attn_decode_noalloc(ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()),
                                         ctypes.c_void_p(vd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         B, H, L, d, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("B,H,L", [(1, 2, 3000), (2, 3, 1000), (4, 40, 300)])
def test_noalloc_decode_matches_decode_twice(B, H, L, d):
    import torch
    import alibi_positional_bias_gb300 as ab
    lib = ab.load()
    for call, seed in enumerate((31 + L + d, 77 + L + d)):  # two calls in a row, different inputs
        w = gen.Workload("noalloc", "decode", B, H, L, d, "bf16", seed=seed)
        q, k, v = gen.generate(w)
        qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
        ref = ab.alibi_attn_decode(qd, kd, vd)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, qd, kd, vd, out, B, H, L, d)
        assert st == 0, ab.alibi_status_str(st)
        ab.alibi_check_error()
        got, want = host64(out), host64(ref)
        assert np.isfinite(got).all(), f"call {call}"
        assert_bf16_out(got, want, what=f"call {call}")


def test_noalloc_decode_refuses_plans_beyond_its_buffer():
    # A split plan whose partials outgrow the fixed 4 MiB buffer is refused with
    # ALIBI_ERR_UNSUPPORTED before anything runs, and out is left as it was. The
    # shape is the smallest found whose plan (B*H*S*(d+4)*4 bytes, S from the
    # library's own split rule on this GPU) passes 4 MiB: B=51, H=40, L=23552,
    # d=128. The caches are real allocations of that size (uninitialised, 24.6 GB),
    # so even a wrong refusal could only read memory the test owns.
    import torch
    import alibi_positional_bias_gb300 as ab
    lib = ab.load()
    B, H, L, d = 51, 40, 23552, 128
    S = ab.alibi_attn_decode_splits(B, H, L, d)
    need = B * H * S * (d + 4) * 4
    if need <= 4 << 20:
        pytest.skip(f"on this GPU the plan ({S} splits) fits the buffer")
    kd = torch.empty((B, H, L, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    qd = torch.zeros((B, H, d), dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, qd, kd, vd, out, B, H, L, d) == ab.ALIBI_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    del kd, vd
    torch.cuda.empty_cache()

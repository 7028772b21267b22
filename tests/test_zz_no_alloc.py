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


@pytest.mark.parametrize("B,H,L", [(1, 2, 3000), (2, 3, 1000), (4, 40, 300)])
def test_noalloc_decode_matches_decode_twice(B, H, L):
    import torch
    import alibi_positional_bias_gb300 as ab
    lib = ab.load()
    for call, seed in enumerate((31 + L, 77 + L)):  # two calls in a row, different inputs
        w = gen.Workload("noalloc", "decode", B, H, L, 128, "bf16", seed=seed)
        q, k, v = gen.generate(w)
        qd, kd, vd = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16")
        ref = ab.alibi_attn_decode(qd, kd, vd)
        out = torch.full_like(ref, float("nan"))
        st = lib.alibi_attn_decode_noalloc(ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()),
                                           ctypes.c_void_p(vd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                           B, H, L, 128, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, ab.alibi_status_str(st)
        ab.alibi_check_error()
        got, want = host64(out), host64(ref)
        assert np.isfinite(got).all(), f"call {call}"
        assert_bf16_out(got, want, what=f"call {call}")

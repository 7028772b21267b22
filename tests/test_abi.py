"""The C-ABI library: builds, loads, exports every declared symbol, and its
host-only paths (slopes, argument validation) behave. No device work here."""
import ctypes
import os
import re

import mpmath
import numpy as np
import pytest

import alibi_positional_bias_gb300 as ab
import oracle
from alibi_positional_bias_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ab.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(alibi_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_abi():
    names = declared_symbols()
    for n in ["alibi_slopes", "alibi_attn_fwd", "alibi_attn_decode", "alibi_attn_fwd_f32",
              "alibi_attn_probs_f32", "alibi_attn_underflow_bf16", "alibi_status_str", "alibi_check_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n, ok in ab.exported_symbols(declared_symbols()).items() if not ok]
    assert not missing, missing


def test_library_exports_nothing_undeclared(lib):
    # visibility is hidden by default: only the extern "C" ABI is exported
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ab.lib_path()], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("alibi_")}
    assert exported == set(declared_symbols())


def test_version_and_status_strings(lib):
    assert ab.alibi_version() >= 100
    for s in (0, -1, -2, -3, -4, -5):
        assert ab.alibi_status_str(s).startswith("ALIBI_")


def test_slopes_match_printed_tables(lib):
    # "ALiBi: Attention with Linear Biases", slope tables for 4, 8 and 6 heads.
    assert list(ab.alibi_slopes(4)) == [0.25, 0.0625, 0.015625, 0.00390625]
    assert list(ab.alibi_slopes(8)) == [0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.00390625]
    assert list(ab.alibi_slopes(6)) == [0.25, 0.0625, 0.015625, 0.00390625, 0.5, 0.125]


def test_slopes_bit_exact_vs_oracle_all_h(lib):
    for H in range(1, 1025):
        assert np.array_equal(ab.alibi_slopes(H).view(np.uint32), oracle.slopes_f32(H).view(np.uint32)), H


def test_slopes_correctly_rounded_large_h(lib):
    mpmath.mp.prec = 200
    for H in (257, 300, 1000, 2047, 4096):
        got = ab.alibi_slopes(H)
        for h in range(0, H, max(1, H // 97)):
            num, den = oracle.slope_exponent(H, h)
            exact = mpmath.power(2, mpmath.mpf(-num) / den)  # at 200 bits
            with mpmath.workprec(24):
                want = float(+exact)
            assert float(got[h]) == want, (H, h)


def test_slopes_rejects_bad_h(lib):
    buf = (ctypes.c_float * 4)()
    assert lib.alibi_slopes(0, buf) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_slopes(-3, buf) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_slopes(4, None) == ab.ALIBI_ERR_INVALID


# Argument validation happens on the host before any CUDA call, so these run
# without a GPU. The fake pointer values are never dereferenced.
P = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10008)  # not 16-byte aligned


def test_fwd_argument_errors(lib):
    f = lib.alibi_attn_fwd
    assert f(None, P, P, P, P, 1, 1, 8, 64, 1, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, 0, 1, 8, 64, 1, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, 1, 1, 0, 64, 1, None) == ab.ALIBI_ERR_INVALID
    assert f(MIS, P, P, P, P, 1, 1, 8, 64, 1, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 64, 2, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 48, 1, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, 1, 300, 8, 64, 1, None) == ab.ALIBI_ERR_UNSUPPORTED


def _opt(flags=0, clamp=0.0, z=0.0, slopes=None):
    m = None if slopes is None else np.ascontiguousarray(slopes, dtype=np.float32)
    o = ab.AlibiFwdOptions(flags, clamp, z, None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return ctypes.byref(o), m  # keep m alive with the struct


def test_fwd_ex_flags_and_plan_errors(lib):
    def f(H, d, causal, *opt):
        o, keep = _opt(*opt)
        return lib.alibi_attn_fwd_ex(P, P, P, P, P, 1, H, 8, d, causal, o, None)
    assert f(1, 64, 1, 32) == ab.ALIBI_ERR_INVALID                      # unknown flag
    assert f(1, 48, 1, 1) == ab.ALIBI_ERR_UNSUPPORTED                   # head size
    assert f(1, 64, 1, 2, 1.0) == ab.ALIBI_ERR_INVALID                  # clamp >= 0
    assert f(1, 64, 1, 8, 0.0, -5.0) == ab.ALIBI_ERR_INVALID            # z <= 0
    assert f(1, 64, 1, 1 | 4) == ab.ALIBI_ERR_INVALID                   # skip + logdist
    assert f(1, 64, 0, 1) == ab.ALIBI_ERR_UNSUPPORTED                   # skip needs the causal range
    assert f(2, 64, 1, 0, 0.0, 0.0, [0.5, -0.25]) == ab.ALIBI_ERR_INVALID         # negative slope
    assert f(2, 64, 1, 0, 0.0, 0.0, [0.5, float("nan")]) == ab.ALIBI_ERR_INVALID  # non-finite slope
    assert f(2, 64, 1, 0, 0.0, 0.0, [0.5, float("inf")]) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_skip_plan(P, P, 1, 1, 8, 64, None, None, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_skip_plan(P, P, 1, 1, 8, 48, None, P, None) == ab.ALIBI_ERR_UNSUPPORTED
    neg = (ctypes.c_float * 2)(0.5, -1.0)
    assert lib.alibi_attn_skip_plan(P, P, 1, 2, 8, 64, neg, P, None) == ab.ALIBI_ERR_INVALID


def test_decode_and_aux_argument_errors(lib):
    assert lib.alibi_attn_decode(None, P, P, P, 1, 1, 8, 128, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_decode(P, P, P, P, 1, 1, 0, 128, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_decode(P, P, P, P, 1, 1, 8, 48, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_decode(P, P, P, P, 1, 1, 8, 256, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_fwd_f32(P, P, P, P, P, 1, 1, 8, 512, 1, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_probs_f32(P, P, None, P, 1, 1, 8, 16, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_probs_f32_ex(P, P, P, P, 1, 1, 8, 16, 2, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_fwd_f32(P, P, P, P, P, 1, 1, 8, 16, 3, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_underflow_bf16(P, P, 1, 1, 8, 48, ctypes.c_float(-87.0), P, None) == \
        ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_underflow_bf16(P, P, 1, 1, 8, 64, ctypes.c_float(float("nan")), P, None) == \
        ab.ALIBI_ERR_INVALID
    st = lib.alibi_selftest_fwd_timeout
    assert st(P, P, P, P, P, 1, 1, 8, 64, 0, None) == ab.ALIBI_ERR_INVALID          # wait limit below 1 us
    assert st(P, P, P, P, P, 1, 1, 8, 64, 1000001, None) == ab.ALIBI_ERR_INVALID    # above one second
    assert st(None, P, P, P, P, 1, 1, 8, 64, 100, None) == ab.ALIBI_ERR_INVALID
    assert st(P, P, P, P, P, 1, 1, 8, 48, 100, None) == ab.ALIBI_ERR_UNSUPPORTED


def test_large_head_counts_are_bounded_on_the_host(lib):
    # work items (256-row blocks of every (b, h)) are counted in 32-bit integers:
    # B*H*ceil(N/256) beyond 2^31 - 1 is refused before any launch
    f = lib.alibi_attn_fwd
    assert f(P, P, P, P, P, 1 << 16, 1 << 8, 1 << 15, 64, 1, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_skip_plan(P, P, 1 << 16, 1 << 8, 1 << 15, 64, None, P, None) == ab.ALIBI_ERR_UNSUPPORTED


def test_explicit_slopes_bit_exact_vs_oracle(lib):
    # host-only: the library's robust-slope schedule against the oracle's, rounded once
    import oracle
    for H, d1, dH, logd in [(9, 128, 512, False), (9, 2048, 4096, False), (9, 16, 4096, False),
                            (9, 32, 8192, False), (9, 32, 8192, True), (7, 32, 2048, False), (1, 100, 5000, False),
                            (64, 10, 1e6, True), (256, 3, 3e5, False)]:
        got = ab.alibi_slopes_explicit(H, d1, dH, log_distance=logd)
        want = oracle.slopes_explicit(H, d1, dH, log_distance=logd).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (H, d1, dH, logd)
    for bad in [(0, 16, 64), (4, 0, 64), (4, 16, float("nan")), (4, 16, -1.0)]:
        with pytest.raises(ab.AlibiError):
            ab.alibi_slopes_explicit(*bad)
    with pytest.raises(ab.AlibiError):
        ab.alibi_slopes_explicit(4, 16, 64, tau=0.0)


def test_bwd_argument_errors(lib):
    f = lib.alibi_attn_bwd
    assert f(None, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 1, None, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, P, P, P, MIS, 1, 1, 8, 64, 1, None, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 2, None, None) == ab.ALIBI_ERR_INVALID
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 32, 1, None, None) == ab.ALIBI_ERR_UNSUPPORTED
    o, keep = _opt(1)  # skipping has no backward
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 1, o, None) == ab.ALIBI_ERR_UNSUPPORTED
    o, keep = _opt(2, 1.0)  # clamp >= 0
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 1, o, None) == ab.ALIBI_ERR_INVALID
    o, keep = _opt(32)  # unknown flag
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 1, o, None) == ab.ALIBI_ERR_INVALID
    o, keep = _opt(0, 0.0, 0.0, [float("nan")])
    assert f(P, P, P, P, P, P, P, P, P, 1, 1, 8, 64, 1, o, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_bwd_f32(P, P, P, P, P, P, P, P, P, 1, 1, 8, 300, 1, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_bwd_f32(P, P, P, None, P, P, P, P, P, 1, 1, 8, 16, 1, None) == ab.ALIBI_ERR_INVALID


def test_decode_skip_argument_errors(lib):
    assert lib.alibi_kv_block_norms(None, P, 1, 1, 8, 128, 0, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_kv_block_norms(P, P, 1, 1, 8, 128, 2, None) == ab.ALIBI_ERR_INVALID     # blk_begin > ceil(L/64)
    assert lib.alibi_kv_block_norms(P, P, 1, 1, 8, 128, -1, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_kv_block_norms(P, P, 1, 1, 8, 48, 0, None) == ab.ALIBI_ERR_UNSUPPORTED
    assert lib.alibi_attn_decode_skip(P, P, P, None, P, 1, 1, 8, 128, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_decode_skip(P, P, P, P, MIS, 1, 1, 8, 128, None) == ab.ALIBI_ERR_INVALID
    assert lib.alibi_attn_decode_skip(P, P, P, P, P, 1, 1, 8, 96, None) == ab.ALIBI_ERR_UNSUPPORTED

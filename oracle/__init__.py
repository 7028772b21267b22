"""fp64 CPU oracle for ALiBi causal attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product path (``alibi_positional_bias_gb300``)
never does, and this package never imports the product path.

The arithmetic lives in ``alibi_oracle.c`` (plain C, fp64, one query row at a
time); this module compiles it with gcc on first use and marshals numpy
arrays. Every function is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "alibi_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
# Test hook: tests/test_oracle_mutations.py points the pin suite at deliberately
# broken builds of alibi_oracle.c to show that each plausible mistake is caught.
_SO_OVERRIDE = os.environ.get("ALIBI_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

CLAMP, LOGDIST, SOFTCAP = 1, 2, 4


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no fast-math: IEEE fp64)."""
    if _SO_OVERRIDE:
        return _SO_OVERRIDE
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        compile_to(_SRC, tmp)
        os.replace(tmp, _SO)
    return _SO


def compile_to(src: str, out: str) -> None:
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", out, src, "-lm"],
                   check=True)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        f32p, f64p, i64p = P(ctypes.c_float), P(ctypes.c_double), P(ctypes.c_long)
        u64p = P(ctypes.c_ulonglong)
        I, D = ctypes.c_int, ctypes.c_double
        lib.oracle_slope_exponent.argtypes = [I, I, P(I), P(I)]
        lib.oracle_slopes.argtypes = [I, f64p]
        lib.oracle_slopes_f32.argtypes = [I, f32p]
        lib.oracle_slopes_explicit.argtypes = [I, D, D, D, I, f64p]
        lib.oracle_bias.argtypes = [D, ctypes.c_long, ctypes.c_long, I]
        lib.oracle_bias.restype = D
        lib.oracle_bias_ex.argtypes = [D, ctypes.c_long, ctypes.c_long, I, I, D]
        lib.oracle_bias_ex.restype = D
        lib.oracle_attn_rows.argtypes = [f32p, f32p, f32p, f64p, I, I, I, I, I, I, D, D, i64p,
                                         ctypes.c_long, f64p, f64p, f64p, I]
        lib.oracle_attn_bwd.argtypes = [f32p, f32p, f32p, f32p, f64p, I, I, I, I, I, I, D, D, f64p, f64p, f64p,
                                        f64p, f64p, I]
        lib.oracle_attn_decode.argtypes = [f32p, f32p, f32p, f64p, I, I, I, I, f64p, f64p, I]
        lib.oracle_underflow_rows.argtypes = [f32p, f32p, f64p, I, I, I, I, D, D, i64p, ctypes.c_long,
                                              u64p, u64p, I]
        lib.oracle_thresholds.argtypes = [f64p]
        lib.oracle_thresholds.restype = None
        lib.oracle_blindness_real.argtypes = [D, D, D, I]
        lib.oracle_blindness_real.restype = D
        lib.oracle_blindness_int.argtypes = [D, D, D, I]
        lib.oracle_blindness_int.restype = D
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _check(rc: int):
    if rc != 0:
        raise RuntimeError(f"oracle call failed with status {rc}")


def slope_exponent(H: int, h: int) -> tuple[int, int]:
    """(num, den) with m_h = 2^(-num/den)."""
    n, d = ctypes.c_int(), ctypes.c_int()
    _check(_load().oracle_slope_exponent(H, h, ctypes.byref(n), ctypes.byref(d)))
    return n.value, d.value


def slopes(H: int) -> np.ndarray:
    """fp64 ALiBi slopes for H heads."""
    m = np.empty(H, dtype=np.float64)
    _check(_load().oracle_slopes(H, _ptr(m, ctypes.c_double)))
    return m


def slopes_f32(H: int) -> np.ndarray:
    """ALiBi slopes rounded once to fp32."""
    m = np.empty(H, dtype=np.float32)
    _check(_load().oracle_slopes_f32(H, _ptr(m, ctypes.c_float)))
    return m


def slopes_explicit(H: int, delta_first: float, delta_last: float, tau: float | None = None,
                    log_distance: bool = False) -> np.ndarray:
    """fp64 slopes whose zero-logit blindness distances run geometrically from
    delta_first to delta_last ("When Attention Goes Blind", sec. 3.4 "Robust
    Slopes", sec. 4.3, Table 8). tau defaults to ln 2^-126."""
    tau = tau_denorm() if tau is None else float(tau)
    m = np.empty(H, dtype=np.float64)
    _check(_load().oracle_slopes_explicit(int(H), float(delta_first), float(delta_last), tau,
                                          int(bool(log_distance)), _ptr(m, ctypes.c_double)))
    return m


def bias(m: float, i: int, j: int, causal: bool = True, variant: int = 0, c_clamp: float = -87.0) -> float:
    return _load().oracle_bias_ex(float(m), int(i), int(j), int(bool(causal)), int(variant), float(c_clamp))


def attention(q, k, v, m=None, causal=True, rows=None, want_weights=False, variant=0,
              c_clamp=-87.0, z_cap=50.0, nthreads=0):
    """Oracle attention over [B, H, N, d] inputs.

    Returns (out, lse, weights). With ``rows`` (flat (b*H + h)*N + i indices) the
    results are per requested row; otherwise out is [B, H, N, d], lse [B, H, N]
    and weights [B, H, N, N] (when requested).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, N, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    m = slopes(H) if m is None else np.ascontiguousarray(m, dtype=np.float64)
    lib = _load()
    if rows is None:
        nrows = B * H * N
        rows_p = None
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_a.size
        rows_p = _ptr(rows_a, ctypes.c_long)
    out = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    w = np.empty((nrows, N), dtype=np.float64) if want_weights else None
    _check(lib.oracle_attn_rows(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                                _ptr(m, ctypes.c_double), B, H, N, d, int(bool(causal)), int(variant),
                                float(c_clamp), float(z_cap), rows_p, nrows, _ptr(out, ctypes.c_double),
                                _ptr(lse, ctypes.c_double), _ptr(w, ctypes.c_double) if w is not None else None,
                                int(nthreads)))
    if rows is None:
        out = out.reshape(B, H, N, d)
        lse = lse.reshape(B, H, N)
        if w is not None:
            w = w.reshape(B, H, N, N)
    return out, lse, w


def attention_bwd(q, k, v, dout, m=None, causal=True, variant=0, c_clamp=-87.0, z_cap=50.0, nthreads=0):
    """Oracle gradients (dq, dk, dv) [B, H, N, d] of sum(dout * attention(q, k, v)),
    plus the per-row LSE and sum_j w_ij (dout_i . v_j) [B, H, N]."""
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    B, H, N, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape
    m = slopes(H) if m is None else np.ascontiguousarray(m, dtype=np.float64)
    dq, dk, dv = (np.empty((B, H, N, d), dtype=np.float64) for _ in range(3))
    lse, rowdot = np.empty((B, H, N), dtype=np.float64), np.empty((B, H, N), dtype=np.float64)
    p64 = lambda a: _ptr(a, ctypes.c_double)  # noqa: E731
    _check(_load().oracle_attn_bwd(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                                   _ptr(dout, ctypes.c_float), p64(m), B, H, N, d, int(bool(causal)), int(variant),
                                   float(c_clamp), float(z_cap), p64(dq), p64(dk), p64(dv), p64(lse), p64(rowdot),
                                   int(nthreads)))
    return dq, dk, dv, lse, rowdot


def decode(q, kcache, vcache, m=None, nthreads=0):
    """Oracle decode: q [B, H, d] at position L-1 against caches [B, H, L, d]."""
    q, kc, vc = _f32(q), _f32(kcache), _f32(vcache)
    B, H, L, d = kc.shape
    assert q.shape == (B, H, d) and vc.shape == kc.shape
    m = slopes(H) if m is None else np.ascontiguousarray(m, dtype=np.float64)
    out = np.empty((B, H, d), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    _check(_load().oracle_attn_decode(_ptr(q, ctypes.c_float), _ptr(kc, ctypes.c_float), _ptr(vc, ctypes.c_float),
                                      _ptr(m, ctypes.c_double), B, H, L, d, _ptr(out, ctypes.c_double),
                                      _ptr(lse, ctypes.c_double), int(nthreads)))
    return out, lse


def underflow_rows(q, k, tau, m=None, rows=None, band=1e-3, nthreads=0):
    """Per-row counts of allowed keys with x_ij - M_i <= tau, and of keys within band of tau."""
    q, k = _f32(q), _f32(k)
    B, H, N, d = q.shape
    m = slopes(H) if m is None else np.ascontiguousarray(m, dtype=np.float64)
    if rows is None:
        nrows, rows_p = B * H * N, None
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rows_p = rows_a.size, _ptr(rows_a, ctypes.c_long)
    cnt = np.zeros(nrows, dtype=np.uint64)
    near = np.zeros(nrows, dtype=np.uint64)
    _check(_load().oracle_underflow_rows(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(m, ctypes.c_double),
                                         B, H, N, d, float(tau), float(band), rows_p, nrows,
                                         _ptr(cnt, ctypes.c_ulonglong), _ptr(near, ctypes.c_ulonglong),
                                         int(nthreads)))
    return cnt, near


def underflow_counts_per_head(q, k, tau, m=None, band=1e-3, nthreads=0):
    """Whole-matrix causal counts per head: (count[H], near[H])."""
    B, H, N, _ = np.shape(q)
    cnt, near = underflow_rows(q, k, tau, m=m, band=band, nthreads=nthreads)
    return (cnt.reshape(B, H, N).sum(axis=(0, 2)), near.reshape(B, H, N).sum(axis=(0, 2)))


def thresholds() -> dict:
    t = np.empty(6, dtype=np.float64)
    _load().oracle_thresholds(_ptr(t, ctypes.c_double))
    return {"underflow_bf16": t[0], "underflow_fp32": t[1], "denorm_bf16": t[2], "denorm_fp32": t[3],
            "overflow_bf16": t[4], "overflow_fp32": t[5]}


def tau_denorm() -> float:
    """ln 2^-126: the threshold the pages' own blindness numbers use."""
    return thresholds()["denorm_fp32"]


def blindness_real(m: float, eps: float = 0.0, tau: float | None = None, log_distance: bool = False) -> float:
    tau = tau_denorm() if tau is None else tau
    return _load().oracle_blindness_real(float(m), float(eps), float(tau), int(bool(log_distance)))


def blindness_int(m: float, eps: float = 0.0, tau: float | None = None, log_distance: bool = False) -> float:
    tau = tau_denorm() if tau is None else tau
    return _load().oracle_blindness_int(float(m), float(eps), float(tau), int(bool(log_distance)))

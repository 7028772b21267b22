"""GB300-native ALiBi attention: Python binding of the C ABI (include/alibi.h).

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libalibi_gb300.so``. There is no CPU fallback; if the library
is missing or fails to load, every call raises.

The functions carry the names of the C entry points. Tensors are torch CUDA
tensors (torch supplies device memory and streams); ``stream`` defaults to
torch's current stream on the tensors' device.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np

from . import _build

__all__ = [
    "AlibiError", "load", "lib_path", "exported_symbols", "alibi_version", "alibi_status_str", "alibi_slopes",
    "alibi_attn_fwd", "alibi_attn_fwd_ex", "alibi_attn_skip_plan", "alibi_attn_fwd_f32", "alibi_attn_decode", "alibi_attn_decode_splits", "alibi_attn_probs_f32",
    "alibi_attn_underflow_bf16", "alibi_check_error", "alibi_attn_decode_noalloc", "alibi_selftest_timeout",
    "alibi_selftest_fwd_timeout", "alibi_decode_underflow_bf16",
    "alibi_slopes_explicit", "alibi_attn_probs_f32_ex", "AlibiFwdOptions", "alibi_attn_bwd", "alibi_attn_bwd_f32",
    "alibi_kv_block_norms", "alibi_attn_decode_skip",
]

ALIBI_OK, ALIBI_ERR_INVALID, ALIBI_ERR_UNSUPPORTED, ALIBI_ERR_CUDA, ALIBI_ERR_TIMEOUT, ALIBI_ERR_CHECK = 0, -1, -2, -3, -4, -5
ALIBI_FWD_SKIP_UNDERFLOW, ALIBI_FWD_CLAMP, ALIBI_FWD_LOGDIST, ALIBI_FWD_SOFTCAP = 1, 2, 4, 8
ALIBI_FWD_NOMINAL_ORDER = 16

_lock = threading.Lock()
_lib = None


class AlibiFwdOptions(ctypes.Structure):
    """The C struct alibi_fwd_options (include/alibi.h)."""
    _fields_ = [("flags", ctypes.c_uint), ("clamp_min", ctypes.c_float), ("softcap_z", ctypes.c_float),
                ("slopes", ctypes.POINTER(ctypes.c_float))]


class AlibiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {alibi_status_str(status)} ({status})")


def checks_build() -> bool:
    """True when ALIBI_CHECKS=1 selects the debug-checks library (every TMA coordinate,
    TMEM address and shared-memory operand tested in the kernels; slower)."""
    return os.environ.get("ALIBI_CHECKS", "0") == "1"


def lib_path() -> str:
    return _build.LIB_CHECKS if checks_build() else _build.LIB


def load(build_if_missing: bool = False):
    """Load the CUDA library (optionally building it first). Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if build_if_missing and not os.path.exists(path):
            _build.build(checks=checks_build())
        if not os.path.exists(path):
            raise RuntimeError(f"ALiBi CUDA library not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.alibi_version.restype = I
        lib.alibi_status_str.argtypes = [I]
        lib.alibi_status_str.restype = ctypes.c_char_p
        lib.alibi_slopes.argtypes = [I, ctypes.POINTER(F)]
        lib.alibi_attn_fwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, vp]
        lib.alibi_attn_fwd_f32.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, vp]
        lib.alibi_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, ctypes.POINTER(AlibiFwdOptions), vp]
        lib.alibi_slopes_explicit.argtypes = [I, ctypes.c_double, ctypes.c_double, ctypes.c_double, I,
                                              ctypes.POINTER(F)]
        lib.alibi_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I,
                                        ctypes.POINTER(AlibiFwdOptions), vp]
        lib.alibi_attn_bwd_f32.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, vp]
        lib.alibi_kv_block_norms.argtypes = [vp, vp, I, I, I, I, I, vp]
        lib.alibi_attn_decode_skip.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, vp]
        lib.alibi_attn_probs_f32_ex.argtypes = [vp, vp, vp, vp, I, I, I, I, I, vp]
        lib.alibi_attn_fwd_ex.restype = I
        lib.alibi_attn_skip_plan.argtypes = [vp, vp, I, I, I, I, ctypes.POINTER(F), vp, vp]
        lib.alibi_attn_skip_plan.restype = I
        lib.alibi_attn_decode.argtypes = [vp, vp, vp, vp, I, I, I, I, vp]
        lib.alibi_attn_probs_f32.argtypes = [vp, vp, vp, vp, I, I, I, I, vp]
        lib.alibi_attn_decode_splits.argtypes = [I, I, I, I]
        lib.alibi_attn_decode_noalloc.argtypes = [vp, vp, vp, vp, I, I, I, I, vp]
        lib.alibi_attn_decode_noalloc.restype = I
        lib.alibi_attn_underflow_bf16.argtypes = [vp, vp, I, I, I, I, F, vp, vp]
        lib.alibi_check_error.argtypes = [vp]
        lib.alibi_selftest_timeout.argtypes = [vp]
        lib.alibi_selftest_timeout.restype = I
        lib.alibi_selftest_fwd_timeout.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, vp]
        lib.alibi_selftest_fwd_timeout.restype = I
        lib.alibi_decode_underflow_bf16.argtypes = [vp, vp, I, I, I, I, F, vp, vp]
        lib.alibi_decode_underflow_bf16.restype = I
        for name in ("alibi_attn_fwd", "alibi_attn_fwd_f32", "alibi_attn_decode", "alibi_attn_decode_splits",
                     "alibi_attn_probs_f32",
                     "alibi_attn_underflow_bf16", "alibi_check_error", "alibi_slopes"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def exported_symbols(names) -> dict:
    """Which of ``names`` the loaded library exports (no device work)."""
    lib = load()
    return {n: hasattr(lib, n) for n in names}


def _check(status: int, where: str):
    if status != ALIBI_OK:
        raise AlibiError(status, where)


def _stream(stream, device):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# --------------------------------------------------------------------- entry points

def alibi_version() -> int:
    return load().alibi_version()


def alibi_status_str(status: int) -> str:
    try:
        return load().alibi_status_str(int(status)).decode()
    except Exception:  # library unavailable while formatting an error
        return f"status {status}"


def alibi_slopes(H: int) -> np.ndarray:
    """fp32 ALiBi slopes for H heads (host computation in the library)."""
    out = np.empty(H, dtype=np.float32)
    _check(load().alibi_slopes(int(H), out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))), "alibi_slopes")
    return out


def alibi_attn_fwd(q, k, v, out=None, lse=None, causal: bool = True, stream=None, want_lse: bool = True,
                   skip_underflow: bool = False):
    """bf16 prefill on the tensor cores (causal, or symmetric bias over all keys).
    q, k, v: [B, H, N, d] bf16 CUDA tensors.

    ``skip_underflow`` leaves out KV tiles whose weights provably flush to zero
    (alibi_attn_fwd_ex with ALIBI_FWD_SKIP_UNDERFLOW); the result is bit-identical.
    """
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.bfloat16, q.shape, "k")
    _need(v, torch.bfloat16, q.shape, "v")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, q.shape, "out")
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, (B, H, N), "lse")
    if skip_underflow:
        opt = AlibiFwdOptions(ALIBI_FWD_SKIP_UNDERFLOW, 0.0, 0.0, None)
        _check(load().alibi_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                        int(bool(causal)), ctypes.byref(opt), _stream(stream, q.device)),
               "alibi_attn_fwd_ex")
    else:
        _check(load().alibi_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                     int(bool(causal)), _stream(stream, q.device)), "alibi_attn_fwd")
    return out, lse


def alibi_attn_fwd_ex(q, k, v, out=None, lse=None, causal: bool = True, flags: int = 0, clamp_min: float = -87.0,
                      softcap_z: float = 50.0, slopes=None, stream=None):
    """Prefill with options (ALIBI_FWD_* flags): exact underflow skipping, or the
    clamp / log-distance / soft-cap mitigations with their parameters, and
    optionally caller-chosen per-head slopes (H values, natural-log units)."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.bfloat16, q.shape, "k")
    _need(v, torch.bfloat16, q.shape, "v")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, q.shape, "out")
    _need(lse, torch.float32, (B, H, N), "lse")
    m = None
    if slopes is not None:
        m = np.ascontiguousarray(slopes, dtype=np.float32)
        if m.shape != (H,):
            raise ValueError(f"slopes: expected shape ({H},), got {m.shape}")
    opt = AlibiFwdOptions(int(flags), float(clamp_min), float(softcap_z),
                          None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    _check(load().alibi_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)),
                                    ctypes.byref(opt), _stream(stream, q.device)),
           "alibi_attn_fwd_ex")
    return out, lse


def alibi_slopes_explicit(H: int, delta_first: float, delta_last: float, tau: float | None = None,
                          log_distance: bool = False) -> np.ndarray:
    """fp32 slopes whose zero-logit blindness distances run geometrically from
    delta_first (head 0) to delta_last (head H-1); tau defaults to ln 2^-126."""
    tau = -126.0 * math.log(2.0) if tau is None else tau
    out = np.empty(H, dtype=np.float32)
    _check(load().alibi_slopes_explicit(int(H), float(delta_first), float(delta_last), float(tau),
                                        int(bool(log_distance)), out.ctypes.data_as(ctypes.POINTER(ctypes.c_float))),
           "alibi_slopes_explicit")
    return out


def alibi_attn_bwd(q, k, v, out, lse, dout, dq=None, dk=None, dv=None, causal: bool = True, slopes=None,
                   flags: int = 0, clamp_min: float = -87.0, softcap_z: float = 50.0, stream=None):
    """bf16 backward on the tensor cores: (dq, dk, dv) of sum(dout * out) for the
    forward's out and lse. All tensors [B, H, N, d] bf16 CUDA tensors, lse fp32.
    flags / clamp_min / softcap_z / slopes must be those the forward ran with."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    for t, name in ((k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, q.shape, name)
    _need(lse, torch.float32, (B, H, N), "lse")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, torch.bfloat16, q.shape, name)
    m = None
    if slopes is not None:
        m = np.ascontiguousarray(slopes, dtype=np.float32)
        if m.shape != (H,):
            raise ValueError(f"slopes: expected shape ({H},), got {m.shape}")
    opt = AlibiFwdOptions(int(flags), float(clamp_min), float(softcap_z),
                          None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    _check(load().alibi_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, N, d, int(bool(causal)), ctypes.byref(opt),
                                 _stream(stream, q.device)), "alibi_attn_bwd")
    return dq, dk, dv


def alibi_attn_bwd_f32(q, k, v, out, lse, dout, causal: bool = True, stream=None):
    """fp32 backward (reference precision). All tensors fp32 CUDA tensors."""
    import torch
    _need(q, torch.float32, None, "q")
    B, H, N, d = q.shape
    for t, name in ((k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.float32, q.shape, name)
    _need(lse, torch.float32, (B, H, N), "lse")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    _check(load().alibi_attn_bwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                     _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), _stream(stream, q.device)),
           "alibi_attn_bwd_f32")
    return dq, dk, dv


def alibi_attn_skip_plan(q, k, first_tile=None, slopes=None, stream=None):
    """Per work item (b*H + h, 256-row block): the first 128-key tile the skipping
    prefill computes. Returns an int32 CUDA tensor [B*H*ceil(N/256)]."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.bfloat16, q.shape, "k")
    items = B * H * ((N + 255) // 256)
    if first_tile is None:
        first_tile = torch.empty(items, dtype=torch.int32, device=q.device)
    _need(first_tile, torch.int32, (items,), "first_tile")
    m = None if slopes is None else np.ascontiguousarray(slopes, dtype=np.float32)
    if m is not None and m.shape != (H,):
        raise ValueError(f"slopes: expected shape ({H},), got {m.shape}")
    _check(load().alibi_attn_skip_plan(_ptr(q), _ptr(k), B, H, N, d,
                                       None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                       _ptr(first_tile), _stream(stream, q.device)),
           "alibi_attn_skip_plan")
    return first_tile


def alibi_attn_fwd_f32(q, k, v, out=None, lse=None, causal: bool = True, stream=None):
    """fp32 prefill (reference precision), causal or symmetric. q, k, v: [B, H, N, d] fp32 CUDA tensors."""
    import torch
    _need(q, torch.float32, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.float32, q.shape, "k")
    _need(v, torch.float32, q.shape, "v")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, q.shape, "out")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _need(lse, torch.float32, (B, H, N), "lse")
    _check(load().alibi_attn_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                     int(bool(causal)), _stream(stream, q.device)), "alibi_attn_fwd_f32")
    return out, lse


def alibi_attn_decode(q, kcache, vcache, out=None, stream=None):
    """bf16 decode: q [B, H, d] at position L-1 against caches [B, H, L, d]."""
    import torch
    _need(kcache, torch.bfloat16, None, "kcache")
    B, H, L, d = kcache.shape
    _need(vcache, torch.bfloat16, kcache.shape, "vcache")
    _need(q, torch.bfloat16, (B, H, d), "q")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, (B, H, d), "out")
    _check(load().alibi_attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), B, H, L, d,
                                    _stream(stream, q.device)), "alibi_attn_decode")
    return out


def alibi_kv_block_norms(kcache, knorm=None, blk_begin: int = 0, stream=None):
    """Maximum key norm per 64-key block of a bf16 cache [B, H, L, d] -> fp32 [B, H, ceil(L/64)].
    Only blocks >= blk_begin are recomputed (refresh the tail after appending keys)."""
    import torch
    _need(kcache, torch.bfloat16, None, "kcache")
    B, H, L, d = kcache.shape
    nblk = (L + 63) // 64
    if knorm is None:
        knorm = torch.empty((B, H, nblk), dtype=torch.float32, device=kcache.device)
    _need(knorm, torch.float32, (B, H, nblk), "knorm")
    _check(load().alibi_kv_block_norms(_ptr(kcache), _ptr(knorm), B, H, L, d, int(blk_begin),
                                       _stream(stream, kcache.device)), "alibi_kv_block_norms")
    return knorm


def alibi_attn_decode_skip(q, kcache, vcache, knorm, out=None, stream=None):
    """Decode that skips cache rows whose weights are provably below 2^-127 of the
    largest (needs the cache's block norms from alibi_kv_block_norms)."""
    import torch
    _need(kcache, torch.bfloat16, None, "kcache")
    B, H, L, d = kcache.shape
    _need(vcache, torch.bfloat16, kcache.shape, "vcache")
    _need(q, torch.bfloat16, (B, H, d), "q")
    _need(knorm, torch.float32, (B, H, (L + 63) // 64), "knorm")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, (B, H, d), "out")
    _check(load().alibi_attn_decode_skip(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(knorm), _ptr(out), B, H, L, d,
                                         _stream(stream, q.device)), "alibi_attn_decode_skip")
    return out


def alibi_attn_decode_noalloc(q, kcache, vcache, out, stream=None):
    """Decode without any device allocation (for callers that cannot allocate).

    Same result as alibi_attn_decode, but the split-K partials live in a fixed
    4 MiB buffer inside the library, so ``out`` must be supplied by the caller.
    Calls that overlap on the GPU share that buffer and race: order them.
    """
    import torch
    _need(kcache, torch.bfloat16, None, "kcache")
    B, H, L, d = kcache.shape
    _need(vcache, torch.bfloat16, kcache.shape, "vcache")
    _need(q, torch.bfloat16, (B, H, d), "q")
    _need(out, torch.bfloat16, (B, H, d), "out")
    _check(load().alibi_attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), B, H, L, d,
                                            _stream(stream, q.device)), "alibi_attn_decode_noalloc")
    return out


def alibi_attn_decode_splits(B: int, H: int, L: int, d: int) -> int:
    """KV splits alibi_attn_decode uses for this shape (1 = single kernel, no partials)."""
    s = load().alibi_attn_decode_splits(int(B), int(H), int(L), int(d))
    if s < 0:
        raise AlibiError(s, "alibi_attn_decode_splits")
    return s


def alibi_attn_probs_f32(q, k, lse, P=None, stream=None):
    """fp32 causal attention weights [B, H, N, N] from the LSE of alibi_attn_fwd_f32."""
    return alibi_attn_probs_f32_ex(q, k, lse, P, causal=True, stream=stream)


def alibi_attn_probs_f32_ex(q, k, lse, P=None, causal: bool = True, stream=None):
    """fp32 attention weights [B, H, N, N] from the LSE of alibi_attn_fwd_f32 (either mask)."""
    import torch
    _need(q, torch.float32, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.float32, q.shape, "k")
    _need(lse, torch.float32, (B, H, N), "lse")
    if P is None:
        P = torch.empty((B, H, N, N), dtype=torch.float32, device=q.device)
    _need(P, torch.float32, (B, H, N, N), "P")
    _check(load().alibi_attn_probs_f32_ex(_ptr(q), _ptr(k), _ptr(lse), _ptr(P), B, H, N, d, int(bool(causal)),
                                          _stream(stream, q.device)), "alibi_attn_probs_f32_ex")
    return P


def alibi_attn_underflow_bf16(q, k, tau: float, counts=None, stream=None):
    """Per-head counts of causal pairs whose max-subtracted exponent is <= tau."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.bfloat16, q.shape, "k")
    if counts is None:
        counts = torch.empty((H,), dtype=torch.int64, device=q.device)
    _need(counts, torch.int64, (H,), "counts")
    _check(load().alibi_attn_underflow_bf16(_ptr(q), _ptr(k), B, H, N, d, ctypes.c_float(tau), _ptr(counts),
                                            _stream(stream, q.device)), "alibi_attn_underflow_bf16")
    return counts


def alibi_decode_underflow_bf16(q, kcache, tau: float, counts=None, stream=None):
    """Per-head counts of cached keys whose max-subtracted exponent at the decode row is <= tau."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, d = q.shape
    _need(kcache, torch.bfloat16, None, "kcache")
    if kcache.dim() != 4 or tuple(kcache.shape[:2]) != (B, H) or kcache.shape[3] != d:
        raise ValueError("kcache must be [B, H, L, d] matching q [B, H, d]")
    L = kcache.shape[2]
    if counts is None:
        counts = torch.empty((H,), dtype=torch.int64, device=q.device)
    _need(counts, torch.int64, (H,), "counts")
    _check(load().alibi_decode_underflow_bf16(_ptr(q), _ptr(kcache), B, H, L, d, ctypes.c_float(tau), _ptr(counts),
                                              _stream(stream, q.device)), "alibi_decode_underflow_bf16")
    return counts


def alibi_selftest_timeout(stream=None) -> None:
    """Launch the failure-path self-test (a bounded wait that must time out)."""
    import torch
    _check(load().alibi_selftest_timeout(_stream(stream, torch.cuda.current_device())), "alibi_selftest_timeout")


def alibi_selftest_fwd_timeout(q, k, v, wait_us: int = 20000, out=None, lse=None, stream=None):
    """Run the prefill kernel with one Q load left out and a short wait limit (failure-path self-test)."""
    import torch
    _need(q, torch.bfloat16, None, "q")
    B, H, N, d = q.shape
    _need(k, torch.bfloat16, q.shape, "k")
    _need(v, torch.bfloat16, q.shape, "v")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(load().alibi_selftest_fwd_timeout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                             int(wait_us), _stream(stream, q.device)), "alibi_selftest_fwd_timeout")
    return out, lse


def alibi_check_error(stream=None, device=None) -> None:
    """Synchronise and raise if a kernel recorded a device-side failure."""
    _check(load().alibi_check_error(_stream(stream, device)), "alibi_check_error")

"""Seeded synthetic inputs for the ALiBi attention workloads.

Shared by the fp64 oracle tests, the GPU parity tests and the benchmark. This
package holds no attention arithmetic: only random-number generation,
storage-format rounding (fp32 -> bf16) and the shapes of the named workloads.

Generators
----------
* ``legacy``: numpy's legacy Mersenne-Twister stream (``np.random.seed(s);
  np.random.randn(...) * scale``). The worked example of "ALiBi in Attention:
  Complete Implementation" (seed-42 example) draws Q, K, V this way, in that
  order, with scale 0.5; the tiny fp32 workload follows it.
* ``counter``: a counter-based stream built on the SplitMix64 output function
  (Steele, Lea & Flood, OOPSLA 2014), implemented in ``gen.c`` (threaded).
  Element n of stream (seed, stream_id) depends on nothing else, so any slice
  of a tensor can be regenerated on its own. Normals use Box-Muller (cosine
  branch) in fp64; uniforms use 53 random bits. Stream ids: q = 0, k = 1, v = 2.

Samples are rounded to fp32 (RNE); bf16 tensors are rounded again to bf16
(RNE on the fp32 bit pattern) and carried as ``uint16`` bit patterns plus
their exact fp32 widening.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_SO = os.path.join(_HERE, "_build", "libgen.so")
_lock = threading.Lock()
_lib = None

GOLDEN = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


def build() -> str:
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, dbl, fp = ctypes.c_uint64, ctypes.c_double, ctypes.POINTER(ctypes.c_float)
            lib.gen_stream_key.argtypes = [u64, u64]
            lib.gen_stream_key.restype = u64
            lib.gen_normal_f32.argtypes = [u64, u64, u64, u64, dbl, fp, ctypes.c_int]
            lib.gen_normal_f32.restype = None
            lib.gen_uniform_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, fp, ctypes.c_int]
            lib.gen_uniform_f32.restype = None
            _lib = lib
    return _lib


# ------------------------------------------------------------ raw streams

def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (numpy cross-check of gen.c)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, sid: int) -> int:
    return int(_load().gen_stream_key(seed & _M64, sid & _M64))


def counter_u64(seed: int, sid: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs (numpy); element n = mix64(key + (n + 1) G)."""
    k1 = int(mix64(np.array([(seed + GOLDEN) & _M64], dtype=np.uint64))[0])
    key = int(mix64(np.array([((k1 ^ sid) + GOLDEN) & _M64], dtype=np.uint64))[0])
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (n + np.uint64(1)) * np.uint64(GOLDEN))


def normal(seed: int, sid: int, count: int, start: int = 0, scale: float = 1.0, nthreads: int = 0) -> np.ndarray:
    """fp32 N(0, scale^2) samples n = start .. start+count-1 of stream (seed, sid)."""
    out = np.empty(count, dtype=np.float32)
    _load().gen_normal_f32(seed & _M64, sid & _M64, start, count, float(scale),
                           out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), nthreads)
    return out


def uniform(seed: int, sid: int, count: int, lo: float, hi: float, start: int = 0, nthreads: int = 0) -> np.ndarray:
    """fp32 U(lo, hi) samples of stream (seed, sid)."""
    out = np.empty(count, dtype=np.float32)
    _load().gen_uniform_f32(seed & _M64, sid & _M64, start, count, float(lo), float(hi),
                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), nthreads)
    return out


def legacy_normal(seed: int, shapes, scale: float) -> list[np.ndarray]:
    """numpy legacy MT19937 normals, drawn in the order of ``shapes``."""
    st = np.random.RandomState(seed)
    return [st.randn(*s) * scale for s in shapes]


# --------------------------------------------------------------- rounding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Tensor:
    """One synthetic tensor: exact fp32 values, plus bf16 bits when stored as bf16."""
    f32: np.ndarray
    bf16: np.ndarray | None = None

    @property
    def shape(self):
        return self.f32.shape


def make_tensor(f32: np.ndarray, shape, dtype: str) -> Tensor:
    f32 = np.ascontiguousarray(f32, dtype=np.float32).reshape(shape)
    if dtype == "fp32":
        return Tensor(f32=f32)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(f32)
        return Tensor(f32=bf16_bits_to_f32(bits).reshape(shape), bf16=bits.reshape(shape))
    raise ValueError(dtype)


# -------------------------------------------------------------- workloads

@dataclass
class Workload:
    """A named synthetic workload (shapes, dtype and value distributions)."""
    name: str
    kind: str               # "prefill" or "decode"
    B: int
    H: int
    N: int                  # prefill tokens, or decode KV-cache length L
    d: int
    dtype: str              # "fp32" or "bf16"
    q_dist: str = "normal"  # "normal" (N(0, sigma^2)), "uniform" (U(-1, 1)) or "zero"
    k_dist: str = "normal"
    v_dist: str = "normal"
    sigma: float = 1.0
    seed: int = 42
    generator: str = "counter"  # "counter" or "legacy"
    note: str = ""
    extra: dict = field(default_factory=dict)

    def shapes(self):
        if self.kind == "prefill":
            s = (self.B, self.H, self.N, self.d)
            return s, s, s
        return (self.B, self.H, self.d), (self.B, self.H, self.N, self.d), (self.B, self.H, self.N, self.d)

    def with_n(self, n: int) -> "Workload":
        return Workload(**{**self.__dict__, "N": n})


WORKLOADS = {
    # The seed-42 worked example of "ALiBi in Attention: Complete Implementation":
    # Q, K, V ~ randn(4, 8, 16) * 0.5 without a batch axis (B = 1 here).
    "p4_example": Workload("p4_example", "prefill", 1, 4, 8, 16, "fp32", sigma=0.5, generator="legacy",
                           note="legacy MT19937 seed 42, randn(4,8,16)*0.5 for Q, K, V in order"),
    "tiny_fp32": Workload("tiny_fp32", "prefill", 1, 4, 64, 16, "fp32", sigma=0.5, generator="legacy",
                          note="legacy MT19937 seed 42, randn(B,H,N,d)*0.5 for Q, K, V in order"),
    "heads6_n1024": Workload("heads6_n1024", "prefill", 2, 6, 1024, 64, "bf16"),
    "layer_n2048": Workload("layer_n2048", "prefill", 4, 32, 2048, 128, "bf16"),
    "long_n16384": Workload("long_n16384", "prefill", 1, 16, 16384, 128, "bf16", v_dist="uniform"),
    "decode_l8192": Workload("decode_l8192", "decode", 64, 40, 8192, 128, "bf16"),
}


def tensor_values(w: Workload, idx: int, start: int = 0, count: int | None = None) -> np.ndarray:
    """fp32 values of tensor idx (0 = q, 1 = k, 2 = v) of a counter workload, flat
    elements [start, start + count), before bf16 rounding."""
    shape = w.shapes()[idx]
    total = int(np.prod(shape))
    count = total - start if count is None else count
    dist = (w.q_dist, w.k_dist, w.v_dist)[idx]
    if dist == "normal":
        return normal(w.seed, idx, count, start=start, scale=w.sigma)
    if dist == "uniform":
        return uniform(w.seed, idx, count, -1.0, 1.0, start=start)
    if dist == "zero":
        return np.zeros(count, dtype=np.float32)
    raise ValueError(dist)


def generate(w: Workload, scale_n: int | None = None):
    """Return (q, k, v) ``Tensor``s for workload ``w`` (``scale_n`` overrides N / L)."""
    if scale_n is not None:
        w = w.with_n(scale_n)
    qs, ks, vs = w.shapes()
    if w.generator == "legacy":
        shp = [(w.H, w.N, w.d)] * 3 if w.name == "p4_example" else [qs, ks, vs]
        q, k, v = legacy_normal(w.seed, shp, w.sigma)
        return tuple(make_tensor(x.astype(np.float32), s, w.dtype) for x, s in zip((q, k, v), (qs, ks, vs)))
    return tuple(make_tensor(tensor_values(w, i), s, w.dtype) for i, s in enumerate((qs, ks, vs)))


def head_slice(w: Workload, idx: int, b: int, h: int) -> Tensor:
    """One (b, h) slab of tensor idx of a counter workload, regenerated on its own."""
    shape = w.shapes()[idx]
    per = int(np.prod(shape[2:]))
    start = (b * w.H + h) * per
    return make_tensor(tensor_values(w, idx, start, per), shape[2:], w.dtype)


def random_case(seed: int, B: int, H: int, N: int, d: int, dtype: str = "bf16", sigma: float = 1.0,
                v_dist: str = "normal", kind: str = "prefill", q_dist: str = "normal", k_dist: str = "normal"):
    """A small ad-hoc case of the same recipe (shape sweeps, edge cases)."""
    w = Workload(f"case{seed}", kind, B, H, N, d, dtype, q_dist=q_dist, k_dist=k_dist, v_dist=v_dist,
                 sigma=sigma, seed=seed)
    return generate(w)


def fill_device(w: Workload, idx: int, dst, chunk: int = 1 << 27, start: int = 0) -> None:
    """Write tensor idx of workload w into the contiguous torch CUDA tensor ``dst``
    (bf16 or fp32) chunk by chunk, without materialising it on the host.

    ``start`` is the flat element offset of ``dst`` inside the workload's tensor
    (a rank's shard of a global batch is a contiguous slice)."""
    import torch
    total = dst.numel()
    assert start + total <= int(np.prod(w.shapes()[idx])) and dst.is_contiguous()
    flat = dst.view(-1)
    for s in range(0, total, chunk):
        c = min(chunk, total - s)
        vals = tensor_values(w, idx, start + s, c)
        if dst.dtype == torch.bfloat16:
            host = torch.from_numpy(f32_to_bf16_bits(vals).view(np.int16)).view(torch.bfloat16)
        else:
            host = torch.from_numpy(vals)
        flat[s:s + c].copy_(host)

"""Seeded synthetic inputs for the ALiBi attention workloads.

This module is shared by the fp64 oracle tests, the GPU parity tests and the
benchmark. It holds no attention arithmetic: only random-number generation,
storage-format rounding (fp32 -> bf16) and the shapes of the named workloads.

Generators
----------
* ``legacy_normal``: numpy's legacy Mersenne-Twister stream
  (``np.random.seed(s); np.random.randn(...) * scale``). The worked example of
  "ALiBi in Attention: Complete Implementation" (seed-42 example) draws Q, K, V
  this way, in that order, with scale 0.5; the tiny fp32 workload follows it.
* ``counter_normal`` / ``counter_uniform``: a counter-based generator built from
  the published SplitMix64 output function (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014). Element ``n`` of
  stream ``(seed, stream_id)`` depends on nothing else, so any slice can be
  regenerated independently. Normals use the Box-Muller transform
  (cosine branch) on two uniforms drawn from elements ``2n`` and ``2n+1``.

Rounding: samples are drawn in fp64, rounded to fp32 (RNE), and for bf16
tensors rounded again to bf16 (RNE on the fp32 bit pattern). bf16 tensors are
returned as ``uint16`` bit patterns plus their exact fp32 widening.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output (finalisation) function on a uint64 array."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream_id: int) -> np.uint64:
    base = np.array([(seed & 0xFFFFFFFFFFFFFFFF)], dtype=np.uint64)
    k = _mix64(base + _GOLDEN)
    k = _mix64(k ^ np.uint64(stream_id & 0xFFFFFFFFFFFFFFFF) + _GOLDEN)
    return k[0]


def counter_u64(seed: int, stream_id: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit outputs n = start .. start+count-1 of stream (seed, stream_id)."""
    key = _stream_key(seed, stream_id)
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + (n + np.uint64(1)) * _GOLDEN)


def counter_uniform01(seed: int, stream_id: int, count: int, start: int = 0) -> np.ndarray:
    """Uniform fp64 samples in [0, 1) with 53 random bits."""
    return (counter_u64(seed, stream_id, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def counter_normal(seed: int, stream_id: int, count: int) -> np.ndarray:
    """N(0, 1) fp64 samples via Box-Muller (cosine branch)."""
    out = np.empty(count, dtype=np.float64)
    chunk = 1 << 22
    for s in range(0, count, chunk):
        c = min(chunk, count - s)
        u = counter_uniform01(seed, stream_id, 2 * c, start=2 * s)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))  # 1 - u1 lies in (0, 1]
        out[s:s + c] = r * np.cos(2.0 * np.pi * u2)
    return out


def counter_uniform(seed: int, stream_id: int, count: int, lo: float, hi: float) -> np.ndarray:
    """U(lo, hi) fp64 samples."""
    return lo + (hi - lo) * counter_uniform01(seed, stream_id, count)


def legacy_normal(seed: int, shapes, scale: float) -> list[np.ndarray]:
    """numpy legacy MT19937 normals, drawn in the order of ``shapes``."""
    st = np.random.RandomState(seed)
    return [st.randn(*s) * scale for s in shapes]


# --------------------------------------------------------------------- rounding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
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


def make_tensor(samples_f64: np.ndarray, shape, dtype: str) -> Tensor:
    f32 = samples_f64.astype(np.float32).reshape(shape)
    if dtype == "fp32":
        return Tensor(f32=np.ascontiguousarray(f32))
    if dtype == "bf16":
        bits = f32_to_bf16_bits(f32)
        return Tensor(f32=bf16_bits_to_f32(bits).reshape(shape), bf16=bits.reshape(shape))
    raise ValueError(dtype)


# --------------------------------------------------------------------- workloads

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
    q_dist: str = "normal"  # "normal" (N(0, sigma^2)) or "uniform" (U(-1, 1))
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


WORKLOADS = {
    # The seed-42 worked example of "ALiBi in Attention: Complete Implementation":
    # Q, K, V ~ randn(4, 8, 16) * 0.5 without a batch axis (B = 1 here).
    "p4_example": Workload("p4_example", "prefill", 1, 4, 8, 16, "fp32", sigma=0.5,
                           generator="legacy", note="legacy MT19937 seed 42, randn(4,8,16)*0.5"),
    "tiny_fp32": Workload("tiny_fp32", "prefill", 1, 4, 64, 16, "fp32", sigma=0.5,
                          generator="legacy", note="legacy MT19937 seed 42, randn(B,H,N,d)*0.5"),
    "heads6_n1024": Workload("heads6_n1024", "prefill", 2, 6, 1024, 64, "bf16"),
    "layer_n2048": Workload("layer_n2048", "prefill", 4, 32, 2048, 128, "bf16"),
    "long_n16384": Workload("long_n16384", "prefill", 1, 16, 16384, 128, "bf16", v_dist="uniform"),
    "decode_l8192": Workload("decode_l8192", "decode", 64, 40, 8192, 128, "bf16"),
}


def generate(w: Workload, scale_n: int | None = None):
    """Return (q, k, v) ``Tensor``s for workload ``w``.

    ``scale_n`` overrides N (or L) to draw a smaller instance of the same recipe.
    """
    if scale_n is not None:
        w = Workload(**{**w.__dict__, "N": scale_n})
    qs, ks, vs = w.shapes()
    if w.generator == "legacy":
        if w.name == "p4_example":
            shp = [(w.H, w.N, w.d)] * 3
        else:
            shp = [qs, ks, vs]
        q, k, v = legacy_normal(w.seed, shp, w.sigma)
        return tuple(make_tensor(x.ravel(), s, w.dtype) for x, s in zip((q, k, v), (qs, ks, vs)))
    out = []
    for sid, (shape, dist) in enumerate(zip((qs, ks, vs), (w.q_dist, w.k_dist, w.v_dist))):
        n = int(np.prod(shape))
        if dist == "normal":
            x = counter_normal(w.seed, sid, n) * w.sigma
        elif dist == "uniform":
            x = counter_uniform(w.seed, sid, n, -1.0, 1.0)
        elif dist == "zero":
            x = np.zeros(n)
        else:
            raise ValueError(dist)
        out.append(make_tensor(x, shape, w.dtype))
    return tuple(out)


def random_case(seed: int, B: int, H: int, N: int, d: int, dtype: str = "bf16",
                sigma: float = 1.0, v_dist: str = "normal", kind: str = "prefill"):
    """A small ad-hoc case of the same recipe (used by shape sweeps)."""
    w = Workload(f"case{seed}", kind, B, H, N, d, dtype, v_dist=v_dist, sigma=sigma, seed=seed)
    return generate(w)

"""Helpers for the GPU parity tests: device upload, tolerances, row sampling."""
import numpy as np

import alibi_inputs as gen


def dev(t: "gen.Tensor", dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(t.bf16).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(t.f32)).cuda()


def host64(x) -> np.ndarray:
    return x.float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |ref| (the rounding error of storing ref in bf16)."""
    a = np.abs(ref)
    _, e = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^e, f in [0.5, 1)
    return np.where(a > 0, np.ldexp(1.0, e - 9), 0.0)


# Tolerances stated for this operator: fp32 path out/weights max-abs <= 1e-5;
# bf16 path out max-abs <= 1e-2 before the final store (plus half a bf16 ulp of
# the value for the unavoidable rounding of the bf16 output), LSE <= 1e-3.
TOL_F32 = 1e-5
TOL_BF16_OUT = 1e-2
TOL_BF16_LSE = 1e-3


def assert_bf16_out(got: np.ndarray, ref: np.ndarray, what: str = "out"):
    err = np.abs(got - ref)
    lim = TOL_BF16_OUT + half_ulp_bf16(ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements exceed tolerance; "
                           f"max err {err.max():.3e} (max err - lim {(err - lim).max():.3e})")
    return float(err.max())


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float, what: str):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err.max() <= tol, f"{what}: max err {err.max():.3e} > {tol:.1e}"
    return float(err.max())


def sample_rows(B: int, H: int, N: int, max_heads: int = 8, per_head: int = 24, seed: int = 0) -> np.ndarray:
    """Flat (b*H + h)*N + i row indices: tile edges, the ragged tail and random rows."""
    rng = np.random.default_rng(seed)
    BH = B * H
    heads = np.arange(BH) if BH <= max_heads else np.unique(
        np.concatenate([[0, BH - 1], rng.choice(BH, max_heads - 2, replace=False)]))
    fixed = [0, 1, 2, 63, 64, 126, 127, 128, 129, 255, 256, 257, 383, 384, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = []
    for bh in heads:
        rr = set(i for i in fixed if 0 <= i < N)
        rr |= set(rng.integers(0, N, size=per_head).tolist())
        rows.extend(int(bh) * N + i for i in sorted(rr))
    return np.array(rows, dtype=np.int64)


def assert_grad(got: np.ndarray, ref: np.ndarray, rel: float, what: str, bf16: bool = False):
    """Per (b, h): |got - ref| <= rel * max(1, max |ref|) (+ half a bf16 ulp of ref for bf16 results)."""
    B, H = ref.shape[:2]
    for b in range(B):
        for h in range(H):
            g, r = got[b, h], ref[b, h]
            scale = max(1.0, float(np.abs(r).max()))
            lim = rel * scale + (half_ulp_bf16(r) if bf16 else 0.0)
            err = np.abs(g - r)
            assert np.isfinite(g).all(), f"{what}[{b},{h}]: non-finite"
            assert (err <= lim).all(), (f"{what}[{b},{h}]: max err {err.max():.3e}, scale {scale:.3e}, "
                                        f"worst excess {(err - lim).max():.3e}")

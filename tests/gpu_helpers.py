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


def bf16_grad_bounds(q, k, v, do, rowdot, causal=True, m=None, variant=0, c_clamp=-87.0, z_cap=50.0):
    """Per-element error bounds (E_dq, E_dk, E_dv) of the tensor-core backward, from
    where it rounds, with the oracle's weights W, output O and row sums D = rowdot:

    - P^T enters dV += P^T dO rounded to bf16 (unit roundoff 2^-8):
        E_dv[j] = 2^-8 sum_i W_ij |dO_i|;
    - dS = P (dP - D) enters dQ += dS K and dK += dS^T Q rounded to bf16, and D is
      taken from the forward's bf16 output, itself off by half an ulp plus the forward's
      own P rounding (2^-8 sum_j W_ij |v_j|), so
        dD_i = sum_t |dO_it| (2^-9 |O_it| + 2^-8 sum_j W_ij |v_jt|),
        E_dq[i] = sum_j W_ij (2^-8 |dP_ij - D_i| + dD_i) |K_j| / sqrt(d),
        E_dk[j] = sum_i W_ij (2^-8 |dP_ij - D_i| + dD_i) |Q_i| / sqrt(d).
    A soft cap's derivative factor is at most one, so the bounds hold for it too.
    q, k, v, do: fp32 arrays of the exact (bf16) values, [B, H, N, d]."""
    import oracle
    out, _, W = oracle.attention(q, k, v, m=m, causal=causal, want_weights=True, variant=variant,
                                 c_clamp=c_clamp, z_cap=z_cap)
    q64, k64, v64, do64 = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    d = q64.shape[-1]
    dP = do64 @ np.swapaxes(v64, -1, -2)
    G = W * np.abs(dP - rowdot[..., None])
    dD = 2.0 ** -9 * (np.abs(do64) * np.abs(out)).sum(-1) + \
        2.0 ** -8 * (W * (np.abs(do64) @ np.swapaxes(np.abs(v64), -1, -2))).sum(-1)
    Ew = 2.0 ** -8 * G + W * dD[..., None]
    E_dq = Ew @ np.abs(k64) / np.sqrt(d)
    E_dk = np.swapaxes(Ew, -1, -2) @ np.abs(q64) / np.sqrt(d)
    E_dv = 2.0 ** -8 * (np.swapaxes(W, -1, -2) @ np.abs(do64))
    return E_dq, E_dk, E_dv


def assert_grad_bound(got: np.ndarray, ref: np.ndarray, bound: np.ndarray, what: str):
    """|got - ref| <= 2 x bound + half a bf16 ulp of ref + 2^-20 max(1, max|ref|) per (b, h)
    (the factor 2 and the last term cover the fp32 accumulations and the LSE)."""
    B, H = ref.shape[:2]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            g, r, e = got[b, h], ref[b, h], bound[b, h]
            lim = 2.0 * e + half_ulp_bf16(r) + 2.0 ** -20 * max(1.0, float(np.abs(r).max()))
            err = np.abs(g - r)
            assert np.isfinite(g).all(), f"{what}[{b},{h}]: non-finite"
            assert (err <= lim).all(), (f"{what}[{b},{h}]: {(err > lim).sum()} elements over the bound; "
                                        f"worst excess {(err - lim).max():.3e}, max err {err.max():.3e}")
            worst = max(worst, float(((err - half_ulp_bf16(r)) / np.maximum(e, 1e-30)).max()))
    return worst

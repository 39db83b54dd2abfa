"""Tolerance rules of the GPU parity tests (shared by the test modules).

Normwise = max|x - ref| / max|ref|:
  fp32 inputs  Y normwise <= 1e-5, dQ/dK/dV normwise <= 1e-4
  bf16 inputs  Y max abs err <= 1e-2 plus half a bf16 ulp of the oracle value
               (and <= 1e-2 with no allowance wherever |ref| < 2),
               each gradient max abs err <= 2e-2 * max|ref|
  both         L max abs err <= 1e-4 (rows with an empty allowed set: exactly -inf)
A gradient that is identically zero in exact arithmetic has its denominator
floored at 1e-3 x the largest max|ref| over dQ, dK, dV of the same call.
With fp32 inputs and a single key (n = 1) dQ and dK are zero in exact
arithmetic and the computed ones are the rounding of dP - delta, a difference of
two width-long fp32 dot products that cancel: they are held element by element
to 2^-18 x sum |dY| |V| times c |K| (dQ) or c |Q| (dK) instead.
"""
import numpy as np
import torch


def _np(t):
    return t.detach().to(torch.float64).cpu().numpy()


TOL = {"f32": dict(y=1e-5, g=1e-4, L=1e-4), "bf16": dict(y=1e-2, g=2e-2, L=1e-4)}


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def compare(dtype, got, ref, heads=None):
    """Assert the tolerance rules; got are torch tensors, ref numpy float64 arrays."""
    tol = TOL[dtype]
    errs = {}
    gscale = max((float(np.abs(ref[k]).max()) for k in ("dQ", "dK", "dV") if k in ref),
                 default=0.0)
    for key in ("Y", "L", "dQ", "dK", "dV"):
        if key not in ref:
            continue
        g = got[key]
        if heads is not None:
            g = g.reshape((-1,) + tuple(g.shape[2:]))[heads]
        g = _np(g).reshape(ref[key].shape)
        r = ref[key]
        if key == "L":
            fin = np.isfinite(r)
            assert np.array_equal(np.isfinite(g), fin), "L finiteness differs"
            err = float(np.abs(g[fin] - r[fin]).max()) if fin.any() else 0.0
            bound = tol["L"]
        elif key == "Y" and dtype == "bf16":
            excess = np.abs(g - r) - half_ulp_bf16(r)
            err = float(excess.max()) if excess.size else 0.0
            bound = tol["y"]
            # Where |Y| < 2 the bf16 rounding is at most 2^-8: there the plain
            # 1e-2 bar holds without the half-ulp allowance.
            small = np.abs(r) < 2.0
            if small.any():
                plain = float(np.abs(g - r)[small].max())
                assert plain <= tol["y"], f"Y (|ref| < 2): max abs err {plain:.3e} > {tol['y']}"
                errs["Y_plain_small"] = (plain, tol["y"])
        elif key == "Y":
            err = float(np.abs(g - r).max())
            bound = tol["y"] * float(np.abs(r).max())
        else:
            err = float(np.abs(g - r).max())
            bound = tol["g"] * max(float(np.abs(r).max()), 1e-3 * gscale)
        assert np.isfinite(g).all() or key == "L", f"{key} has non-finite values"
        errs[key] = (err, bound)
        assert err <= bound, f"{key}: max abs err {err:.3e} > bound {bound:.3e}"
    return errs


def single_key_cancellation(got, Q, K, V, dY, c):
    """fp32, one key per slice: p = 1, so gamma = dP - delta = 0 in exact
    arithmetic ("Exact tiled softmax attention with block-recomputed
    vector-Jacobian products", Reverse procedure), dQ = dK = 0 and dV = dY.
    The computed dQ and dK are the rounding of that cancellation; Q, K, V, dY
    are float64 arrays [..., 1, width]."""
    cancel = 2.0 ** -18 * np.sum(np.abs(dY) * np.abs(V), axis=-1, keepdims=True)
    dq, dk, dv = (_np(got[k]).reshape(r.shape) for k, r in (("dQ", Q), ("dK", K), ("dV", V)))
    assert np.all(np.abs(dq) <= c * np.abs(K) * cancel), "dQ beyond the cancellation bound"
    assert np.all(np.abs(dk) <= c * np.abs(Q) * cancel), "dK beyond the cancellation bound"
    assert np.allclose(dv, dY, rtol=1e-6, atol=0), "dV differs from dY"

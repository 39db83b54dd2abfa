"""GPU parity of dropout with a replayed mask (attn_fwd_dropout / attn_bwd_dropout)
against the float64 oracle (dense.forward_dropout / backward_dropout, whose keep
decisions come from oracle.philox, written separately from the CUDA generator).

Tolerances are those of test_gpu_parity.  On top of them, two bit-exact checks
read the realised mask back out of the kernels: with Q = 0 every allowed p_ij
is 1/|A_i|, so with V = I the forward gives Y_ij = xi_ij s / |A_i| (xi is where
Y is nonzero), and with dY = I the reverse pass gives dV_ji = xi_ij s / |A_i|
(the replayed xi, transposed).
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense, philox
from tolerances import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


def _run(ex, w, x, q, seed, path="auto"):
    dev = torch.device("cuda:0")
    prev = ex.set_path(path)
    try:
        qq, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
        bm = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
        y, L = ex.fwd(qq, k, v, w.scale, w.mask, w.window, bm, dropout_p=q, seed=seed)
        dq, dk, dv = ex.bwd(qq, k, v, y, g, L, w.scale, w.mask, w.window, bm, dropout_p=q,
                            seed=seed)
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    return dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv)


def _oracle(w, x, q, seed):
    Q, K, V, G = x.as_f64()
    Y, L = dense.forward_dropout(Q, K, V, w.scale, w.mask_kind, w.window, x.bitmask, q, seed)
    dQ, dK, dV, _ = dense.backward_dropout(Q, K, V, G, w.scale, w.mask_kind, w.window,
                                           x.bitmask, q, seed)
    return dict(Y=Y, L=L, dQ=dQ, dK=dK, dV=dV)


CASES = [
    # (B, H, n, d, v, dtype, mask, window, q, seed)
    (1, 2, 300, 64, 64, "bf16", "causal", 0, 0.1, 1),
    (2, 1, 333, 128, 128, "bf16", "none", 0, 0.5, 0xDEADBEEF12345678),
    (1, 2, 520, 128, 128, "bf16", "window", 100, 0.25, 7),
    (1, 2, 390, 64, 64, "bf16", "bitmask", 0, 0.3, 99),
    (1, 1, 257, 80, 96, "bf16", "causal", 0, 0.2, 3),
    (1, 2, 300, 64, 64, "f32", "causal", 0, 0.1, 11),
    (1, 1, 257, 48, 24, "f32", "bitmask", 0, 0.4, 5),
]


@pytest.mark.parametrize("path", ["auto", "simt"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_dropout_parity(ex, case, path):
    B, H, n, d, v, dtype, mask, window, q, seed = case
    w = workloads.small(B, H, n, d, v, dtype, mask, 1 / math.sqrt(d), window=window,
                        seed=CASES.index(case) + 40)
    x = workloads.make_inputs(w)
    compare(dtype, _run(ex, w, x, q, seed, path), _oracle(w, x, q, seed))


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("path", ["auto", "simt"])
def test_realised_mask_is_bit_exact_in_both_passes(ex, dtype, d, path):
    """Y and dV reveal xi exactly (Q = 0, V = I, dY = I, causal, n = v)."""
    B, H, n = 2, 3, d
    seed, q = 0x0123_4567_89AB_CDEF, 0.3
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    dev = torch.device("cuda:0")
    Q = torch.zeros(B, H, n, d, dtype=tdt, device=dev)
    K = torch.randn(B, H, n, d, generator=torch.Generator().manual_seed(1)).to(tdt).to(dev)
    eye = torch.eye(n, dtype=tdt, device=dev).expand(B, H, n, n).contiguous()
    prev = ex.set_path(path)
    try:
        y, L = ex.fwd(Q, K, eye, 1.0, "causal", dropout_p=q, seed=seed)
        dq, dk, dv = ex.bwd(Q, K, eye, y, eye, L, 1.0, "causal", dropout_p=q, seed=seed)
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    tri = np.tril(np.ones((n, n), dtype=bool))
    Y = y.float().cpu().numpy().reshape(B * H, n, n)
    dV = dv.float().cpu().numpy().reshape(B * H, n, n)
    s = philox.keep_scale(q)
    for bh in range(B * H):
        keep = philox.keep_mask(bh, n, n, q, seed) & tri
        assert np.array_equal(Y[bh] != 0, keep), f"forward mask differs in slice {bh}"
        assert np.array_equal(dV[bh].T != 0, keep), f"replayed mask differs in slice {bh}"
        # The kept values are s / (i + 1) (bf16-rounded for bf16 outputs).
        want = (s / (np.arange(n) + 1.0))[:, None] * keep
        assert np.abs(Y[bh] - want).max() <= 4e-3 * s


def test_zero_probability_is_the_plain_call(ex):
    w = workloads.small(1, 2, 300, 128, 128, "bf16", "causal", 1 / math.sqrt(128), seed=3)
    x = workloads.make_inputs(w)
    a = _run(ex, w, x, 0.0, 5)
    dev = torch.device("cuda:0")
    qq, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    lib = ex.load_library()
    import ctypes
    shape = ex.Shape(1, 2, 300, 128, 128, 1)
    y = torch.empty_like(qq)
    L = torch.empty(qq.shape[:-1], dtype=torch.float32, device=dev)
    ws = ex.workspace(ex.fwd_workspace_size(shape, "causal"), dev)
    st = lib.attn_fwd_dropout(ctypes.byref(shape), ex._ptr(qq), ex._ptr(k), ex._ptr(v),
                              1 / math.sqrt(128), 1, 0, None, 0.0, 5, ex._ptr(y), ex._ptr(L),
                              ex._ptr(ws), ws.numel(), ex._stream(None))
    torch.cuda.synchronize()
    assert st == 0
    assert torch.equal(y, a["Y"]) and torch.equal(L, a["L"])


def test_same_seed_same_result_other_seed_differs(ex):
    w = workloads.small(1, 1, 256, 64, 64, "bf16", "none", 0.125, seed=8)
    x = workloads.make_inputs(w)
    a = _run(ex, w, x, 0.2, 42)
    b = _run(ex, w, x, 0.2, 42)
    c = _run(ex, w, x, 0.2, 43)
    for key in ("Y", "dQ", "dK", "dV"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["Y"], c["Y"])
    assert torch.equal(a["L"], c["L"])  # L is the undropped statistic


def test_bad_probability_is_rejected(ex):
    w = workloads.small(1, 1, 64, 64, 64, "bf16", "none", 0.125, seed=8)
    x = workloads.make_inputs(w)
    for q in (1.0, -0.5, float("nan")):
        with pytest.raises(ex.ExattnError):
            _run(ex, w, x, q, 1)


def test_dropout_benchmark_size_sampled_heads(ex):
    """The benchmark workload with dropout 0.1 (bench.py --dropout 0.1, seed 1234),
    compared with the oracle on sampled heads."""
    from oracle import masks
    from sampling import head_slices
    w = workloads.workload(3)
    x = workloads.make_inputs(w)
    q, seed = 0.1, 1234
    got = _run(ex, w, x, q, seed)
    heads = [0, 77, w.B * w.H - 1]
    Q, K, V, G = (head_slices(t, heads) for t in (x.Q, x.K, x.V, x.dY))
    allowed = masks.allowed_matrix(w.n, w.mask_kind)
    ks = philox.keep_scale(q)
    ref = {key: [] for key in ("Y", "L", "dQ", "dK", "dV")}
    for idx, h in enumerate(heads):
        keep = philox.keep_mask(h, w.n, w.n, q, seed)
        yy, ll = dense.head_forward_dropout(Q[idx], K[idx], V[idx], w.scale, allowed, keep, ks)
        a, b, c, _ = dense.head_backward_dropout(Q[idx], K[idx], V[idx], G[idx], w.scale,
                                                 allowed, keep, ks)
        for key, val in zip(("Y", "L", "dQ", "dK", "dV"), (yy, ll, a, b, c)):
            ref[key].append(val)
    compare("bf16", got, {key: np.stack(val) for key, val in ref.items()}, heads=heads)

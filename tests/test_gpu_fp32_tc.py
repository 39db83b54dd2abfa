"""GPU parity of the 3xTF32 tensor-core forward for fp32 inputs (d, v <= 128,
multiples of 4; widths other than 64 and 128 zero-padded) against the float64 oracle, at the fp32 bar: Y normwise <= 1e-5,
L max abs <= 1e-4 (tests/tolerances.py).  The same cases also run the SIMT
kernels, and the launch counter shows which path ran: the tensor-core forward
is two launches (the K/V split and the kernel), the SIMT forward one."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense
from tolerances import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


CASES = [
    # (B, H, nq, nk, d, mask, window)
    (1, 2, 300, 300, 64, "none", 0),
    (1, 2, 333, 333, 128, "causal", 0),
    (2, 1, 1000, 1000, 128, "window", 200),
    (1, 2, 390, 390, 64, "bitmask", 0),
    (1, 1, 257, 777, 128, "causal", 0),     # nq < nk
    (1, 1, 300, 100, 64, "causal", 0),      # nq > nk: 200 rows before every key
    (1, 1, 64, 1, 64, "none", 0),
    (1, 4, 2048, 2048, 128, "causal", 0),
]


def _data(case, seed):
    B, H, nq, nk, d, mask, window = case
    Q, K, V, dY, bm = workloads.make_decode_inputs(B, H, nq, nk, d, d, "f32", mask, seed=seed,
                                                   with_dy=True)
    return Q, K, V, bm


@pytest.mark.parametrize("path", ["auto", "simt"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fp32_forward_parity(ex, case, path):
    B, H, nq, nk, d, mask, window = case
    Q, K, V, bm = _data(case, CASES.index(case) + 90)
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (Q, K, V))
    bmt = None if bm is None else torch.from_numpy(bm.view(np.int32)).to(dev)
    c = 1 / math.sqrt(d)
    prev = ex.set_path(path)
    try:
        n0 = ex.launch_count()
        y, L = ex.fwd(q, k, v, c, mask, window, bmt)
        launches = ex.launch_count() - n0
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    assert launches == (2 if path == "auto" else 1)
    kind = workloads.MASK_KINDS[mask]
    Yr, Lr = dense.forward_rect(Q.double().numpy(), K.double().numpy(), V.double().numpy(), c,
                                kind, window, bm)
    compare("f32", dict(Y=y, L=L), dict(Y=Yr, L=Lr))


PADDED = [
    # (B, H, n, d, v, mask, window): widths that run zero-padded on the kernel of
    # width 64 or 128, with their own row strides in memory
    (2, 8, 1000, 80, 96, "bitmask", 0),    # the irregular workload's shape
    (1, 2, 300, 48, 24, "causal", 0),      # width-64 kernel
    (1, 1, 257, 100, 36, "window", 70),    # d above 64: width-128 kernel, v far below
    (1, 1, 200, 4, 128, "none", 0),        # one 16-byte piece of Q, K
]


@pytest.mark.parametrize("path", ["auto", "simt"])
@pytest.mark.parametrize("case", PADDED, ids=lambda c: "-".join(map(str, c)))
def test_fp32_padded_widths_forward_and_reverse(ex, case, path):
    """fp32 widths other than 64 and 128 (multiples of 4): the 3xTF32 forward and
    the register-tiled SIMT reverse pass on zero-padded kernels, Y and L and the
    gradients against the oracle at the fp32 bar; outputs NaN-filled first so
    that a column left unwritten fails."""
    B, H, n, d, v, mask, window = case
    w = workloads.small(B, H, n, d, v, "f32", mask, 0.1, window=window, seed=600 + d + v)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, vv, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    bm = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
    prev = ex.set_path(path)
    try:
        y = torch.full((B, H, n, v), float("nan"), device=dev)
        L = torch.full((B, H, n), float("nan"), device=dev)
        n0 = ex.launch_count()
        ex.fwd(q, k, vv, w.scale, mask, window, bm, y=y, L=L)
        launches = ex.launch_count() - n0
        dq, dk, dv = ex.bwd(q, k, vv, y, g, L, w.scale, mask, window, bm)
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    assert launches == (2 if path == "auto" else 1)
    Q, K, V, G = x.as_f64()
    Yr, Lr = dense.forward(Q, K, V, w.scale, w.mask_kind, window, x.bitmask)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, w.mask_kind, window, x.bitmask)
    compare("f32", dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv), dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))


def test_fp32_forward_then_reverse(ex):
    """Y and L of the tensor-core forward feed the (SIMT) reverse pass."""
    w = workloads.small(1, 2, 500, 128, 128, "f32", "causal", 1 / math.sqrt(128), seed=4)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, "causal")
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, "causal")
    torch.cuda.synchronize()
    Q, K, V, G = x.as_f64()
    Yr, Lr = dense.forward(Q, K, V, w.scale, w.mask_kind)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, w.mask_kind)
    compare("f32", dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv), dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))


def test_fp32_large_magnitudes_keep_the_fp32_bar(ex):
    """Peaked rows (scores up to ~40): the split keeps the relative accuracy."""
    g = torch.Generator().manual_seed(12)
    dev = torch.device("cuda:0")
    Q = torch.randn(1, 2, 512, 128, generator=g) * 3.0
    K = torch.randn(1, 2, 512, 128, generator=g) * 3.0
    V = torch.randn(1, 2, 512, 128, generator=g)
    y, L = ex.fwd(Q.to(dev), K.to(dev), V.to(dev), 1 / math.sqrt(128), "causal")
    torch.cuda.synchronize()
    Yr, Lr = dense.forward(Q.double().numpy(), K.double().numpy(), V.double().numpy(),
                           1 / math.sqrt(128), workloads.MASK_CAUSAL)
    compare("f32", dict(Y=y, L=L), dict(Y=Yr, L=Lr))


def test_fp32_benchmark_step_full_size_sampled_heads(ex):
    """The benchmark workload in fp32 (bench.py --dtype f32): the 3xTF32 forward and
    the register-tiled reverse pass, compared with the oracle on sampled heads."""
    import dataclasses
    from oracle import masks
    from sampling import head_slices
    w = dataclasses.replace(workloads.workload(3), dtype="f32")
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, w.mask)
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, w.mask)
    torch.cuda.synchronize()
    heads = [0, 77, w.B * w.H - 1]
    Q, K, V, G = (head_slices(t, heads) for t in (x.Q, x.K, x.V, x.dY))
    allowed = masks.allowed_matrix(w.n, w.mask_kind)
    ref = {key: [] for key in ("Y", "L", "dQ", "dK", "dV")}
    for h in range(len(heads)):
        yy, ll = dense.head_forward(Q[h], K[h], V[h], w.scale, allowed)
        a, b, cc, _ = dense.head_backward(Q[h], K[h], V[h], G[h], w.scale, allowed)
        for key, val in zip(("Y", "L", "dQ", "dK", "dV"), (yy, ll, a, b, cc)):
            ref[key].append(val)
    compare("f32", dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv),
            {key: np.stack(val) for key, val in ref.items()}, heads=heads)

"""GPU parity of the 3xTF32 tensor-core reverse pass for fp32 inputs (d = v = 64)
against the float64 oracle, at the fp32 bar of tests/tolerances.py: dQ, dK, dV
normwise <= 1e-4 (Y normwise <= 1e-5, L <= 1e-4 for the forward that feeds it).

The reverse pass is four launches on this path (delta, the tf32 split of the
operands, the dQ kernel, the dK/dV kernel); the launch counter checks that it
ran.  The cases cover the workload of n = 256 (full, causal and the shared-X
self-attention form), ragged lengths over several 128-row blocks, every mask
kind, nq != nk in both directions, a one-row problem and a long sequence.  The
outputs are filled with NaN first: every row must be written, none twice."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense
from tolerances import compare

pytestmark = pytest.mark.gpu

BWD32_LAUNCHES = 4


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


def _run(ex, q, k, v, g, c, mask, window, bm, path="auto"):
    dev = q.device
    bmt = None if bm is None else torch.from_numpy(bm.view(np.int32)).to(dev)
    prev = ex.set_path(path)
    try:
        y, L = ex.fwd(q, k, v, c, mask, window, bmt)
        outs = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        n0 = ex.launch_count()
        dq, dk, dv = ex.bwd(q, k, v, y, g, L, c, mask, window, bmt, dq=outs[0], dk=outs[1],
                            dv=outs[2])
        launches = ex.launch_count() - n0
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    return dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv), launches


CASES = [
    # (B, H, nq, nk, mask, window)
    (1, 1, 256, 256, "none", 0),        # the n = 256 fp32 workload, full mask
    (1, 1, 256, 256, "causal", 0),      # ... and causal
    (1, 2, 300, 300, "none", 0),
    (2, 2, 333, 333, "causal", 0),
    (1, 2, 1000, 1000, "window", 200),
    (1, 2, 390, 390, "bitmask", 0),
    (1, 1, 257, 777, "causal", 0),      # nq < nk
    (1, 1, 300, 100, "causal", 0),      # nq > nk: 200 rows before every key
    (1, 1, 2, 2, "none", 0),
    (1, 3, 129, 129, "causal", 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fp32_reverse_parity(ex, case):
    B, H, nq, nk, mask, window = case
    Q, K, V, dY, bm = workloads.make_decode_inputs(B, H, nq, nk, 64, 64, "f32", mask,
                                                   seed=CASES.index(case) + 300, with_dy=True)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (Q, K, V, dY))
    c = 1 / math.sqrt(64)
    got, launches = _run(ex, q, k, v, g, c, mask, window, bm)
    assert launches == BWD32_LAUNCHES
    kind = workloads.MASK_KINDS[mask]
    Qd, Kd, Vd, Gd = (t.double().numpy() for t in (Q, K, V, dY))
    Yr, Lr = dense.forward_rect(Qd, Kd, Vd, c, kind, window, bm)
    dQ, dK, dV = dense.backward_rect(Qd, Kd, Vd, Gd, c, kind, window, bm)[:3]
    if nq > nk and mask == "causal":  # rows before every key: exactly zero gradient
        assert torch.all(got["dQ"][:, :, : nq - nk] == 0)
    compare("f32", got, dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))


def test_fp32_reverse_single_key(ex):
    """n = 1: p = 1, so gamma = dP - delta = 0 and dQ = dK = 0 in exact arithmetic,
    while dV = dY.  The computed dQ and dK are the rounding of that cancellation:
    |dP - delta| is held to 2^-18 of |dY| |V| summed over the width (the two
    64-term fp32 dot products it subtracts), times c |K| or c |Q|."""
    g0 = torch.Generator().manual_seed(57)
    Q, K, V, dY = (torch.randn(3, 2, 1, 64, generator=g0) for _ in range(4))
    dev = torch.device("cuda:0")
    c = 0.125
    got, launches = _run(ex, *(t.to(dev) for t in (Q, K, V, dY)), c, "none", 0, None)
    assert launches == BWD32_LAUNCHES
    cancel = 2.0 ** -18 * (dY.abs() * V.abs()).sum(-1, keepdim=True)  # per slice
    assert torch.all(got["dQ"].cpu().abs() <= c * K.abs() * cancel)
    assert torch.all(got["dK"].cpu().abs() <= c * Q.abs() * cancel)
    assert torch.allclose(got["dV"].cpu(), dY, rtol=1e-6, atol=0)


def test_fp32_reverse_self_attention_workload(ex):
    """The shared-X form of the n = 256 workload (Q = K = V = X, scale 1): dX =
    dQ + dK + dV against the oracle's three gradients summed."""
    w = workloads.workload(1, "self")
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    X, g = x.Q.to(dev), x.dY.to(dev)
    got, launches = _run(ex, X, X, X, g, w.scale, "none", 0, None)
    assert launches == BWD32_LAUNCHES
    Q, K, V, G = x.as_f64()
    Yr, Lr = dense.forward(Q, K, V, w.scale, w.mask_kind)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, w.mask_kind)
    compare("f32", got, dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))
    dx = (got["dQ"] + got["dK"] + got["dV"]).double().cpu().numpy()
    ref = dQ + dK + dV
    assert np.abs(dx - ref).max() <= 1e-4 * np.abs(ref).max()


@pytest.mark.parametrize("variant", ["none", "causal"])
def test_fp32_reverse_workload1(ex, variant):
    w = workloads.workload(1, variant)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    got, launches = _run(ex, q, k, v, g, w.scale, w.mask, 0, None)
    assert launches == BWD32_LAUNCHES
    Q, K, V, G = x.as_f64()
    Yr, Lr = dense.forward(Q, K, V, w.scale, w.mask_kind)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, w.mask_kind)
    compare("f32", got, dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))


@pytest.mark.parametrize("n,heads", [(4096, 2), (6144, 1)])
def test_fp32_reverse_long_sequence_accumulation(ex, n, heads):
    """Long rows: dV and dK gather up to n / 32 query steps and dQ n / 32 key
    steps.  The dK/dV partial sums leave the fp32 TMEM accumulators every 32
    steps (without that, dK reached a normwise error of 5.7e-5 at n = 4096 and
    grew with n); the errors stay within the 1e-4 bar."""
    g0 = torch.Generator().manual_seed(55 + n)
    Q, K, V, dY = (torch.randn(1, heads, n, 64, generator=g0) for _ in range(4))
    dev = torch.device("cuda:0")
    c = 1 / 8.0
    got, launches = _run(ex, *(t.to(dev) for t in (Q, K, V, dY)), c, "causal", 0, None)
    assert launches == BWD32_LAUNCHES
    Qd, Kd, Vd, Gd = (t.double().numpy() for t in (Q, K, V, dY))
    Yr, Lr = dense.forward(Qd, Kd, Vd, c, workloads.MASK_CAUSAL)
    dQ, dK, dV, _ = dense.backward(Qd, Kd, Vd, Gd, c, workloads.MASK_CAUSAL)
    errs = compare("f32", got, dict(Y=Yr, L=Lr, dQ=dQ, dK=dK, dV=dV))
    print(f"normwise gradient errors at n = {n}:",
          {k: v[0] / v[1] * 1e-4 for k, v in errs.items() if k in ("dQ", "dK", "dV")})


def test_fp32_reverse_matches_the_simt_kernels(ex):
    """The tensor-core and SIMT reverse passes agree to the fp32 bar."""
    g0 = torch.Generator().manual_seed(56)
    Q, K, V, dY = (torch.randn(2, 2, 700, 64, generator=g0) for _ in range(4))
    dev = torch.device("cuda:0")
    args = [t.to(dev) for t in (Q, K, V, dY)]
    tc, n_tc = _run(ex, *args, 0.125, "causal", 0, None)
    simt, n_simt = _run(ex, *args, 0.125, "causal", 0, None, path="simt")
    assert n_tc == BWD32_LAUNCHES and n_simt != BWD32_LAUNCHES
    for key in ("dQ", "dK", "dV"):
        a, b = tc[key].double(), simt[key].double()
        assert float((a - b).abs().max()) <= 1e-4 * float(b.abs().max()), key

"""GPU parity of cross-attention (nq query rows against nk keys; attn_fwd_qk /
attn_bwd_qk through the binding) against the float64 oracle (forward_rect /
backward_rect: queries aligned to the end of the keys).  Tolerances as in
test_gpu_parity (tests/tolerances.py).  Cases cover the tensor-core kernels
(bf16, d = v in {64, 128}) and the SIMT kernels, nq < nk and nq > nk (rows
before every key: empty under the causal mask), ragged tails of both lengths
and every mask kind."""
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


def _inputs(case, seed):
    B, H, nq, nk, d, v, dtype, mask, window = case[:9]
    Q, K, V, dY, bm = workloads.make_decode_inputs(B, H, nq, nk, d, v, dtype, mask, seed=seed,
                                                   with_dy=True)
    return Q, K, V, dY, bm


def _run(ex, case, x, path="auto", dropout=(0.0, 0)):
    B, H, nq, nk, d, v, dtype, mask, window = case[:9]
    dev = torch.device("cuda:0")
    Q, K, V, dY, bm = x
    prev = ex.set_path(path)
    try:
        q, k, vv, g = (t.to(dev) for t in (Q, K, V, dY))
        bmt = None if bm is None else torch.from_numpy(bm.view(np.int32)).to(dev)
        c = 1 / math.sqrt(d)
        y, L = ex.fwd(q, k, vv, c, mask, window, bmt, dropout_p=dropout[0], seed=dropout[1])
        dq, dk, dv = ex.bwd(q, k, vv, y, g, L, c, mask, window, bmt, dropout_p=dropout[0],
                            seed=dropout[1])
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    return dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv)


def _oracle(case, x, dropout=None):
    B, H, nq, nk, d, v, dtype, mask, window = case[:9]
    Q, K, V, dY, bm = (t if t is None or isinstance(t, np.ndarray) else t.double().numpy()
                       for t in x)
    kind = workloads.MASK_KINDS[mask]
    c = 1 / math.sqrt(d)
    Y, L = dense.forward_rect(Q, K, V, c, kind, window, bm, dropout)
    dQ, dK, dV, _ = dense.backward_rect(Q, K, V, dY, c, kind, window, bm, dropout)
    return dict(Y=Y, L=L, dQ=dQ, dK=dK, dV=dV)


CASES = [
    # (B, H, nq, nk, d, v, dtype, mask, window)
    (1, 2, 200, 700, 128, 128, "bf16", "causal", 0),
    (2, 1, 333, 129, 64, 64, "bf16", "none", 0),
    (1, 2, 300, 100, 128, 128, "bf16", "causal", 0),     # 200 rows before every key
    (1, 2, 150, 1000, 64, 64, "bf16", "window", 300),
    (1, 1, 257, 520, 128, 128, "bf16", "bitmask", 0),
    (1, 2, 128, 384, 64, 64, "bf16", "causal", 0),       # whole tiles
    (1, 1, 130, 77, 80, 96, "bf16", "window", 20),       # widths padded to 128
    (1, 2, 90, 301, 64, 64, "f32", "causal", 0),
    (1, 1, 250, 60, 48, 24, "f32", "bitmask", 0),
]


@pytest.mark.parametrize("path", ["auto", "simt"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_cross_attention_parity(ex, case, path):
    x = _inputs(case, CASES.index(case) + 60)
    got = _run(ex, case, x, path)
    compare(case[6], got, _oracle(case, x))
    nq, nk = case[2], case[3]
    if case[7] == "causal" and nq > nk:
        assert np.isneginf(got["L"].cpu().numpy()[..., : nq - nk]).all()
        assert (got["dQ"][..., : nq - nk, :] == 0).all()


@pytest.mark.parametrize("case", [CASES[0], CASES[7]], ids=lambda c: "-".join(map(str, c)))
def test_cross_attention_with_dropout(ex, case):
    x = _inputs(case, 77)
    compare(case[6], _run(ex, case, x, dropout=(0.2, 31)), _oracle(case, x, (0.2, 31)))


def test_equal_lengths_match_the_square_call(ex):
    """attn_fwd_qk / attn_bwd_qk with nq == nk give bitwise the attn_fwd / attn_bwd results."""
    import ctypes
    w = workloads.small(1, 2, 300, 128, 128, "bf16", "causal", 1 / math.sqrt(128), seed=5)
    xi = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (xi.Q, xi.K, xi.V, xi.dY))
    y, L = ex.fwd(q, k, v, w.scale, "causal")
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, "causal")
    lib = ex.load_library()
    shape = ex.QKShape(1, 2, 300, 300, 128, 128, 1)
    y2, L2 = torch.empty_like(y), torch.empty_like(L)
    ws = ex.workspace(lib.exattn_fwd_qk_workspace_size(ctypes.byref(shape), 1), dev)
    assert lib.attn_fwd_qk(ctypes.byref(shape), ex._ptr(q), ex._ptr(k), ex._ptr(v), w.scale, 1,
                           0, None, 0.0, 0, ex._ptr(y2), ex._ptr(L2), ex._ptr(ws), ws.numel(),
                           ex._stream(None)) == 0
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    wb = ex.workspace(lib.exattn_bwd_qk_workspace_size(ctypes.byref(shape), 1), dev)
    assert lib.attn_bwd_qk(ctypes.byref(shape), ex._ptr(q), ex._ptr(k), ex._ptr(v), ex._ptr(y),
                           ex._ptr(g), ex._ptr(L), w.scale, 1, 0, None, 0.0, 0, ex._ptr(dq2),
                           ex._ptr(dk2), ex._ptr(dv2), ex._ptr(wb), wb.numel(),
                           ex._stream(None)) == 0
    torch.cuda.synchronize()
    for a, b in ((y, y2), (L, L2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)


def test_cross_benchmark_size_sampled_heads(ex):
    """bench.py --nk 8192: the benchmark workload's 4096 queries against 8192 keys,
    forward and reverse, sampled heads against the oracle."""
    import dataclasses
    from sampling import head_slices
    w = dataclasses.replace(workloads.workload(3), nk=8192)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, w.mask)
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, w.mask)
    torch.cuda.synchronize()
    heads = [0, w.B * w.H - 1]
    Q, K, V, G = (head_slices(t, heads)[:, None] for t in (x.Q, x.K, x.V, x.dY))
    Yr, Lr = dense.forward_rect(Q, K, V, w.scale, w.mask_kind)
    dQ, dK, dV, _ = dense.backward_rect(Q, K, V, G, w.scale, w.mask_kind)
    ref = dict(Y=Yr[:, 0], L=Lr[:, 0], dQ=dQ[:, 0], dK=dK[:, 0], dV=dV[:, 0])
    compare("bf16", dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv), ref, heads=heads)

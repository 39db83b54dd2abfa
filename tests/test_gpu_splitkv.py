"""GPU parity of the split-KV forward (attn_fwd_splitkv) against the float64
oracle: nq queries at the end of an nk-key sequence, keys cut into chunks whose
summaries are merged with the star rule.  The result must not depend on the
number of chunks.  Tolerances as in test_gpu_parity (bf16 Y: 1e-2 plus half a
bf16 ulp of the reference; fp32 Y: 1e-5 normwise; L: 1e-4)."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense, masks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


def _half_ulp_bf16(x):
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def _check(dtype, Y, L, Yr, Lr):
    Y = Y.double().cpu().numpy()
    L = L.double().cpu().numpy()
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(L), fin)
    if fin.any():
        assert np.abs(L[fin] - Lr[fin]).max() <= 1e-4
    if dtype == "bf16":
        assert (np.abs(Y - Yr) - _half_ulp_bf16(Yr)).max() <= 1e-2
    else:
        assert np.abs(Y - Yr).max() <= 1e-5 * max(np.abs(Yr).max(), 1e-30)
    assert np.all(Y[~fin] == 0)


CASES = [
    # (B, H, nq, nk, d, v, dtype, mask, window)
    (1, 2, 1, 1000, 128, 128, "bf16", "none", 0),
    (2, 2, 4, 777, 64, 64, "bf16", "causal", 0),
    (1, 2, 16, 2048, 128, 128, "bf16", "window", 300),
    (1, 1, 8, 513, 80, 96, "f32", "bitmask", 0),
    (1, 2, 64, 300, 64, 64, "f32", "causal", 0),
    (1, 1, 3, 4099, 256, 256, "f32", "none", 0),
    (1, 1, 33, 190, 32, 16, "bf16", "bitmask", 0),
    # nq <= 4 (nq = 1 only for the tensor-core shapes below) runs the
    # register-resident kernel; these cover each lane-group
    # layout (8 or 16 lanes per key row, 32 lanes with one or two 16-byte
    # pieces each), rows wider than the pieces in use, and d != v.
    (1, 2, 2, 3000, 80, 96, "f32", "bitmask", 0),
    (2, 1, 1, 5000, 256, 256, "bf16", "window", 700),
    (1, 3, 4, 2500, 16, 32, "bf16", "causal", 0),
    (1, 1, 1, 2049, 128, 128, "f32", "causal", 0),
    (1, 2, 3, 1500, 64, 64, "f32", "window", 64),
    # bf16, d = v in {64, 128}, nq >= 2: chunks on the tensor-core forward (summary
    # mode, 128-key chunks), then the merge kernel.
    (1, 2, 2, 4100, 128, 128, "bf16", "causal", 0),
    (2, 1, 3, 999, 64, 64, "bf16", "window", 200),
    (1, 1, 4, 2100, 64, 64, "bf16", "bitmask", 0),
    (2, 2, 2, 260, 128, 128, "bf16", "none", 0),
    (1, 2, 8, 1000, 128, 128, "bf16", "causal", 0),
    (2, 2, 64, 3000, 64, 64, "bf16", "bitmask", 0),
    (1, 1, 5, 129, 128, 128, "bf16", "none", 0),
    (1, 2, 40, 5000, 128, 128, "bf16", "window", 1000),
    (1, 1, 17, 300, 64, 64, "bf16", "causal", 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_splitkv_matches_oracle_for_every_split_count(ex, case):
    B, H, nq, nk, d, v, dtype, mask, window = case
    Q, K, V, bm = workloads.make_decode_inputs(B, H, nq, nk, d, v, dtype, mask,
                                               seed=CASES.index(case) + 7)
    Yr, Lr = dense.forward_rect(*(t.double().numpy() for t in (Q, K, V)), 1 / math.sqrt(d),
                                workloads.MASK_KINDS[mask], window, bm)
    dev = torch.device("cuda:0")
    q, k, v_ = (t.to(dev) for t in (Q, K, V))
    bmt = None if bm is None else torch.from_numpy(bm.view(np.int32)).to(dev)
    for splits in (1, 2, 5, 16, 4096):
        Y, L = ex.fwd_splitkv(q, k, v_, 1 / math.sqrt(d), mask, window, bmt, num_splits=splits)
        torch.cuda.synchronize()
        _check(dtype, Y, L, Yr, Lr)


@pytest.mark.parametrize("nq,d,mask", [(2, 128, "causal"), (4, 64, "bitmask"), (3, 128, "none")])
def test_register_kernel_on_tensor_core_shapes(ex, nq, d, mask):
    """With the kernel path set to SIMT, bf16 d = v in {64, 128} and nq in 2..4
    run the register kernel on the tensor-core plan's 128-key chunks."""
    B, H, nk = 1, 2, 1500
    Q, K, V, bm = workloads.make_decode_inputs(B, H, nq, nk, d, d, "bf16", mask, seed=40 + nq)
    Yr, Lr = dense.forward_rect(*(t.double().numpy() for t in (Q, K, V)), 1 / math.sqrt(d),
                                workloads.MASK_KINDS[mask], 0, bm)
    dev = torch.device("cuda:0")
    q, k, v_ = (t.to(dev) for t in (Q, K, V))
    bmt = None if bm is None else torch.from_numpy(bm.view(np.int32)).to(dev)
    prev = ex.set_path("simt")
    try:
        for splits in (1, 3, 0):
            Y, L = ex.fwd_splitkv(q, k, v_, 1 / math.sqrt(d), mask, 0, bmt, num_splits=splits)
            torch.cuda.synchronize()
            _check("bf16", Y, L, Yr, Lr)
    finally:
        ex.set_path(prev)


@pytest.mark.parametrize("nq,nk", [(8, 5), (4, 2), (20, 7)])
def test_more_queries_than_keys_gives_empty_rows(ex, nq, nk):
    """With nq > nk under the causal mask the first nq - nk queries precede every
    key: their allowed sets are empty (Y = 0, L = -inf, status EMPTY_ROW)."""
    B, H, d = 1, 1, 64
    Q, K, V, _ = workloads.make_decode_inputs(B, H, nq, nk, d, d, "bf16", seed=3)
    Yr, Lr = dense.forward_rect(*(t.double().numpy() for t in (Q, K, V)), 0.125, masks.CAUSAL)
    dev = torch.device("cuda:0")
    shape = ex.QKShape(B, H, nq, nk, d, d, 1)
    ws = ex.workspace(ex.load_library().exattn_splitkv_workspace_size(
        __import__("ctypes").byref(shape), 2), dev)
    Y, L = ex.fwd_splitkv(*(t.to(dev) for t in (Q, K, V)), 0.125, "causal", num_splits=2, ws=ws)
    assert ex.device_status(ws) == 5
    _check("bf16", Y, L, Yr, Lr)
    assert np.isneginf(L.cpu().numpy()[0, 0, :nq - nk]).all()


@pytest.mark.parametrize("nq", [1, 4, 6])
def test_splitkv_agrees_with_last_rows_of_full_forward(ex, nq):
    """The decode problem is the last nq rows of the square problem."""
    n, d = 700, 128
    w = workloads.small(1, 2, n, d, d, "bf16", "causal", 1 / math.sqrt(d), seed=11)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (x.Q, x.K, x.V))
    y_full, L_full = ex.fwd(q, k, v, w.scale, "causal")
    y_dec, L_dec = ex.fwd_splitkv(q[:, :, -nq:].contiguous(), k, v, w.scale, "causal",
                                  num_splits=7)
    torch.cuda.synchronize()
    assert (y_dec.float() - y_full[:, :, -nq:].float()).abs().max() <= 2e-2
    assert (L_dec - L_full[:, :, -nq:]).abs().max() <= 1e-4


@pytest.mark.parametrize("nq", [1, 4, 16])
def test_decode_benchmark_size_sampled_heads(ex, nq):
    """bench.py --decode (B=8, H=32, nk=16384, d=v=128, bf16, causal, automatic
    chunk count): the register kernel for nq = 1, the tensor-core chunks for 4
    and 16; sampled heads against the oracle."""
    from sampling import head_slices
    w = workloads.decode_workload(nq)
    Q, K, V, _ = workloads.make_decode_inputs(w.B, w.H, w.nq, w.nk, w.d, w.v, w.dtype, w.mask,
                                              seed=w.seed)
    dev = torch.device("cuda:0")
    Y, L = ex.fwd_splitkv(Q.to(dev), K.to(dev), V.to(dev), w.scale, w.mask, num_splits=0)
    torch.cuda.synchronize()
    heads = [0, 100, w.B * w.H - 1]
    Qh, Kh, Vh = (head_slices(t, heads) for t in (Q, K, V))
    Yr, Lr = dense.forward_rect(Qh[:, None], Kh[:, None], Vh[:, None], w.scale,
                                workloads.MASK_KINDS[w.mask])
    Yg = Y.reshape(-1, nq, w.v)[heads]
    Lg = L.reshape(-1, nq)[heads]
    _check("bf16", Yg, Lg, Yr[:, 0], Lr[:, 0])

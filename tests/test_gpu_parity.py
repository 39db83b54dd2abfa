"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (fixed for this method; normwise = max|x - ref| / max|ref|):
  fp32 inputs  Y normwise <= 1e-5, dQ/dK/dV normwise <= 1e-4
  bf16 inputs  Y max abs err <= 1e-2, each gradient max abs err <= 2e-2 * max|ref|
  both         L max abs err <= 1e-4 (rows with an empty allowed set: exactly -inf)
A bf16 Y cannot be closer to the exact value than half a bf16 ulp of it (0.0156
for |Y| in [4, 8)), so the bf16 Y bound is 1e-2 plus that half ulp of the
oracle value, element by element.
A gradient that is identically zero in exact arithmetic (e.g. dQ when every
row allows a single key) has max|ref| = 0; its denominator is floored at
1e-3 x the largest max|ref| over dQ, dK, dV of the same call, so rounding
noise of the fp32 sums is not held to a zero bound.
The oracle sees the inputs exactly as the GPU does (bf16 values upcast to
float64).  Small cases span several 128-row tiles and a ragged tail; the
benchmark-sized workloads run at full size in the benchmark's launch
configuration and are compared on whole sampled heads.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense, masks
from tolerances import TOL, compare, half_ulp_bf16, single_key_cancellation  # noqa: F401

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


def _np(t):
    return t.detach().to(torch.float64).cpu().numpy()


def run_gpu(ex, w, x, path="auto", self_attention=False, dy=None):
    """Forward + reverse on cuda:0 through the C ABI; returns float64 numpy outputs."""
    dev = torch.device("cuda:0")
    prev = ex.set_path(path)
    try:
        q = x.Q.to(dev)
        k = q if self_attention else x.K.to(dev)
        v = q if self_attention else x.V.to(dev)
        g = (x.dY if dy is None else dy).to(dev)
        bm = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
        y, L = ex.fwd(q, k, v, w.scale, w.mask, w.window, bm)
        dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, w.mask, w.window, bm)
        torch.cuda.synchronize()
    finally:
        ex.set_path(prev)
    return dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv)


def oracle_all(w, x, kind=None):
    Q, K, V, G = x.as_f64()
    kind = w.mask_kind if kind is None else kind
    Y, L = dense.forward(Q, K, V, w.scale, kind, w.window, x.bitmask)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, kind, w.window, x.bitmask)
    return dict(Y=Y, L=L, dQ=dQ, dK=dK, dV=dV)


# --------------------------------------------------------------------------- #
# Small cases: several tiles, ragged tails, every mask kind, both kernel paths
# --------------------------------------------------------------------------- #

SMALL = [
    # (B, H, n, d, v, dtype, mask, window)
    (1, 2, 300, 64, 64, "bf16", "none", 0),
    (1, 2, 300, 64, 64, "bf16", "causal", 0),
    (2, 1, 333, 128, 128, "bf16", "causal", 0),
    (1, 2, 520, 128, 128, "bf16", "window", 100),
    (1, 2, 390, 64, 64, "bf16", "bitmask", 0),
    (1, 1, 257, 80, 96, "bf16", "bitmask", 0),
    (1, 1, 200, 16, 32, "bf16", "causal", 0),
    # widths padded to the tensor-core kernels' 64 or 128 (zero-filled loads, clipped stores)
    (1, 2, 300, 112, 72, "bf16", "window", 77),
    (2, 1, 257, 48, 64, "bf16", "none", 0),
    (1, 1, 190, 8, 8, "bf16", "causal", 0),
    (1, 2, 260, 96, 40, "bf16", "causal", 0),     # Y's second box past its columns
    (1, 1, 200, 40, 128, "bf16", "none", 0),      # Q, K boxes past their columns
    (1, 1, 300, 128, 8, "bf16", "window", 64),    # one 8-column box of V, Y, dY, dV
    (1, 2, 150, 8, 120, "bf16", "none", 0),       # one 8-column box of Q, K, dQ, dK
    (1, 2, 300, 64, 64, "f32", "none", 0),
    (1, 2, 300, 64, 64, "f32", "causal", 0),
    (1, 1, 333, 80, 96, "f32", "window", 45),
    (1, 1, 257, 48, 24, "f32", "bitmask", 0),
    (1, 1, 150, 200, 256, "f32", "causal", 0),
    (1, 1, 140, 256, 256, "bf16", "none", 0),
]


def _small_inputs(case, seed):
    B, H, n, d, v, dtype, mask, window = case
    w = workloads.small(B, H, n, d, v, dtype, mask, 1.0 / math.sqrt(d), window=window,
                        seed=seed)
    return w, workloads.make_inputs(w)


@pytest.mark.parametrize("path", ["auto", "simt", "atomic_dq"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_small_parity(ex, case, path):
    w, x = _small_inputs(case, seed=1000 + SMALL.index(case))
    got = run_gpu(ex, w, x, path)
    compare(w.dtype, got, oracle_all(w, x))


@pytest.mark.parametrize("n", [1, 2, 3, 127, 128, 129, 255, 1000])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_lengths(ex, n, dtype):
    for mask in ("none", "causal"):
        w = workloads.small(1, 1, n, 64, 64, dtype, mask, 0.125, seed=n)
        x = workloads.make_inputs(w)
        got, ref = run_gpu(ex, w, x), oracle_all(w, x)
        if dtype == "f32" and n == 1:
            # dQ = dK = 0 exactly; the computed ones are a cancellation's rounding.
            compare(dtype, got, {k: ref[k] for k in ("Y", "L", "dV")})
            single_key_cancellation(got, *x.as_f64(), w.scale)
        else:
            compare(dtype, got, ref)


def test_window_wider_than_n_is_causal(ex):
    w = workloads.small(1, 2, 300, 64, 64, "bf16", "window", 0.125, window=5000, seed=3)
    x = workloads.make_inputs(w)
    compare("bf16", run_gpu(ex, w, x), oracle_all(w, x, kind=masks.CAUSAL))


def test_one_allowed_key_per_row(ex):
    n = 260
    w = workloads.small(1, 1, n, 64, 64, "bf16", "bitmask", 0.125, seed=4)
    x = workloads.make_inputs(w)
    perm = np.random.default_rng(0).permutation(n)
    allowed = np.zeros((n, n), dtype=bool)
    allowed[np.arange(n), perm] = True
    x.bitmask = workloads.pack_bitmask(allowed)
    got = run_gpu(ex, w, x)
    ref = oracle_all(w, x)
    compare("bf16", got, ref)
    # Y_i is exactly the (bf16) value row V_pi(i).
    assert np.array_equal(_np(got["Y"])[0, 0], x.V.double().numpy()[0, 0][perm])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bitmask_tile_table_across_words(ex, dtype):
    """n = 4500 keys: the kernels' bitmask tile tables span several 32-block
    words (128-key blocks: 36; the fp32 forward's 64-key blocks: 71). Key blocks
    cycle through three kinds: every pair allowed (FULL), a random 30% (PARTIAL)
    and none but the diagonal (EMPTY for all rows except the block's own 128)."""
    n = 4500
    w = workloads.small(1, 1, n, 64, 64, dtype, "bitmask", 0.125, seed=21)
    x = workloads.make_inputs(w)
    rng = np.random.default_rng(21)
    kind = (np.arange(n) // 128) % 3
    allowed = np.zeros((n, n), dtype=bool)
    allowed[:, kind == 0] = True
    part = kind == 1
    allowed[:, part] = rng.random((n, int(part.sum()))) < 0.3
    allowed[np.arange(n), np.arange(n)] = True
    x.bitmask = workloads.pack_bitmask(allowed)
    compare(dtype, run_gpu(ex, w, x), oracle_all(w, x))


def test_empty_allowed_set_reports_and_stays_finite(ex):
    n = 200
    w = workloads.small(1, 1, n, 64, 64, "bf16", "bitmask", 0.125, seed=5)
    x = workloads.make_inputs(w)
    allowed = masks.allowed_matrix(n, masks.BITMASK, bitmask=x.bitmask)
    empty = [0, 77, 199]
    allowed[empty] = False
    x.bitmask = workloads.pack_bitmask(allowed)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    bm = torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
    shape = ex.Shape(1, 1, n, 64, 64, 1)
    ws = ex.workspace(ex.fwd_workspace_size(shape, "bitmask"), dev)
    y, L = ex.fwd(q, k, v, w.scale, "bitmask", 0, bm, ws=ws)
    assert ex.device_status(ws) == 5
    wsb = ex.workspace(ex.bwd_workspace_size(shape, "bitmask"), dev)
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, "bitmask", 0, bm, ws=wsb)
    assert ex.device_status(wsb) == 5  # the reverse pass saw L = -inf rows
    Yn, Ln = _np(y)[0, 0], _np(L)[0, 0]
    assert np.all(Yn[empty] == 0) and np.all(np.isneginf(Ln[empty]))
    assert np.all(_np(dq)[0, 0][empty] == 0)
    # The oracle needs nonempty rows: give the empty rows a dummy key and G_i = 0,
    # which removes every contribution of those rows.
    allowed2 = allowed.copy()
    allowed2[empty, 0] = True
    x2 = workloads.Inputs(x.Q, x.K, x.V, x.dY.clone(), workloads.pack_bitmask(allowed2))
    x2.dY[0, 0, empty] = 0
    ref = oracle_all(w, x2)
    keep = torch.from_numpy(np.setdiff1d(np.arange(n), empty))
    for key in ("Y", "L", "dQ"):
        ref[key] = ref[key][0, 0][keep.numpy()]
    got = dict(Y=y[0, 0][keep], L=L[0, 0][keep], dQ=dq[0, 0][keep], dK=dk, dV=dv)
    compare("bf16", got, ref)
    for t in (y, L, dq, dk, dv):
        assert torch.isfinite(t.float()).logical_or(torch.isneginf(t.float())).all()


def test_self_attention_aliasing(ex):
    """Q = K = V = X passed as one buffer (workload 1, self variant)."""
    w = workloads.workload(1, "self")
    x = workloads.make_inputs(w)
    got = run_gpu(ex, w, x, self_attention=True)
    compare("f32", got, oracle_all(w, x))
    # Shared-input accumulation: dX = dQ + dK + dV matches the oracle's sum.
    Q, K, V, G = x.as_f64()
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, 0)
    dX = _np(got["dQ"]) + _np(got["dK"]) + _np(got["dV"])
    ref = dQ + dK + dV
    assert np.abs(dX - ref).max() <= 1e-4 * np.abs(ref).max()


def test_guard_regions_untouched(ex):
    """Outputs sit inside NaN-filled buffers; nothing outside them is written.  The
    40/72-wide case runs on the 128-wide kernels: the second 64-column box of dQ
    and dK is skipped and that of Y and dV is clipped to 8 columns."""
    dev = torch.device("cuda:0")
    for dtype, d, vw in (("bf16", 128, 128), ("f32", 128, 128), ("bf16", 40, 72)):
        w = workloads.small(1, 2, 333, d, vw, dtype, "causal", 0.09, seed=8)
        x = workloads.make_inputs(w)
        q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
        pad = 4096
        outs = {}
        for name, shape, dt in (("y", v.shape, q.dtype), ("L", q.shape[:-1], torch.float32),
                                ("dq", q.shape, q.dtype), ("dk", k.shape, q.dtype),
                                ("dv", v.shape, q.dtype)):
            numel = int(np.prod(shape))
            buf = torch.full((numel + 2 * pad,), float("nan"), dtype=dt, device=dev)
            outs[name] = (buf, buf[pad:pad + numel].view(shape))
        y, L = ex.fwd(q, k, v, w.scale, "causal", y=outs["y"][1], L=outs["L"][1])
        ex.bwd(q, k, v, y, g, L, w.scale, "causal", dq=outs["dq"][1], dk=outs["dk"][1],
               dv=outs["dv"][1])
        torch.cuda.synchronize()
        for name, (buf, view) in outs.items():
            assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[-pad:].float()).all(), name
            assert not torch.isnan(view.float()).any(), name
        compare(dtype, dict(Y=y, L=L, dQ=outs["dq"][1], dK=outs["dk"][1], dV=outs["dv"][1]),
                oracle_all(w, x))


def test_device_status_ok_and_misalignment(ex):
    dev = torch.device("cuda:0")
    w = workloads.small(1, 1, 64, 64, 64, "bf16", "none", 0.125)
    x = workloads.make_inputs(w)
    q, k, v = (t.to(dev) for t in (x.Q, x.K, x.V))
    shape = ex.Shape(1, 1, 64, 64, 64, 1)
    ws = ex.workspace(ex.fwd_workspace_size(shape, 0), dev)
    ex.fwd(q, k, v, w.scale, "none", ws=ws)
    assert ex.device_status(ws) == 0
    flat = torch.empty(q.numel() + 1, dtype=q.dtype, device=dev)
    bad_q = flat[1:].view(q.shape)
    with pytest.raises(ex.ExattnError) as e:
        ex.fwd(bad_q, k, v, w.scale, "none")
    assert e.value.status == 3


# --------------------------------------------------------------------------- #
# The five benchmark-shaped workloads
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("variant", ["none", "causal"])
def test_workload1_single_head_fp32(ex, variant):
    w = workloads.workload(1, variant)
    x = workloads.make_inputs(w)
    compare("f32", run_gpu(ex, w, x), oracle_all(w, x))


@pytest.mark.parametrize("variant", ["", "bf16"])
def test_workload5_irregular_bitmask(ex, variant):
    w = workloads.workload(5, variant)
    x = workloads.make_inputs(w)
    compare(w.dtype, run_gpu(ex, w, x), oracle_all(w, x))


def _sampled_heads(ex, w, heads):
    x = workloads.make_inputs(w)
    got = run_gpu(ex, w, x)
    Q, K, V, G = x.as_f64()
    Y, L = dense.forward(Q, K, V, w.scale, w.mask_kind, w.window, x.bitmask, heads=heads)
    dQ, dK, dV, _ = dense.backward(Q, K, V, G, w.scale, w.mask_kind, w.window, x.bitmask,
                                   heads=heads)
    return compare(w.dtype, got, dict(Y=Y, L=L, dQ=dQ, dK=dK, dV=dV), heads=heads)


# Workloads 2 and 3 at full size: tests/test_gpu_fullsize.py (every slice on
# sampled rows and identities, whole gradients on one slice per item group).


@pytest.mark.parametrize("variant", ["", "window"])
def test_workload4_full_size_sampled_head(ex, variant):
    w = workloads.workload(4, variant)
    _sampled_heads(ex, w, [w.B * w.H - 1])


def test_bounded_wait_times_out_and_reports(ex):
    """A device wait on a barrier nothing arrives on gives up after its limit,
    records EXATTN_TIMEOUT and returns; the context stays usable."""
    import ctypes
    dev = torch.device("cuda:0")
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    lib = ex.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.exattn_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 2000, stream) == 0
    assert ex.device_status(ws) == 7
    words = ws.view(torch.int32).cpu().tolist()
    assert words[1] == 1 and words[2] == 1
    assert words[3] < 500_000          # the second waiter stopped long before its 1 s limit
    # The context is still usable: a normal call afterwards succeeds.
    w = workloads.small(1, 1, 128, 64, 64, "bf16", "causal", 0.125)
    x = workloads.make_inputs(w)
    y, L = ex.fwd(x.Q.to(dev), x.K.to(dev), x.V.to(dev), w.scale, "causal")
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()

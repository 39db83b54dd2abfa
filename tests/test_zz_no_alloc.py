"""attn_bwd_noalloc: the reverse pass for callers that cannot allocate device
memory (and so cannot hand attn_bwd a workspace), e.g. a plugin whose host gives
it only its input and output buffers.  It runs on a scratch array inside the
library instead of a caller workspace.

Each case calls the new entry point twice in a row through the C ABI (the
second call reuses the array that the first one left behind) and checks both
results against attn_bwd with an ordinary torch-allocated workspace.  On the
tensor-core path both calls run the same deterministic kernels on the same
inputs, so the results must be bitwise equal; the SIMT path adds dQ with fp32
atomics in any order, so there the gradient tolerances of the parity tests
apply.  Further cases go through the Python wrapper (its shape checks and the
status word read back from the scratch array).  The file runs last so that a
failure here cannot hide any other test; it also passes on its own in a fresh
process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

GRAD_TOL = {"bf16": 2e-2, "f32": 1e-4}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


@pytest.mark.parametrize("case", [
    (2, 4, 1000, 128, "bf16", "causal"),   # tensor-core reverse kernel
    (1, 2, 300, 64, "f32", "bitmask"),     # SIMT reverse kernel
], ids=lambda c: "-".join(map(str, c)))
def test_noalloc_matches_attn_bwd_twice(ex, case):
    B, H, n, d, dtype, mask = case
    w = workloads.small(B, H, n, d, d, dtype, mask, 1.0 / math.sqrt(d), seed=77)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    bm = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
    y, L = ex.fwd(q, k, v, w.scale, mask, 0, bm)
    ref = ex.bwd(q, k, v, y, g, L, w.scale, mask, 0, bm)
    lib = ex.load_library()
    shape = ex.Shape(B, H, n, d, d, 0 if dtype == "f32" else 1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        st = lib.attn_bwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(y),
                                  _ptr(g), _ptr(L), ctypes.c_float(w.scale),
                                  ex.MASK_CAUSAL if mask == "causal" else ex.MASK_BITMASK, 0,
                                  _ptr(bm), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), stream)
        assert st == 0, lib.exattn_last_error()
        torch.cuda.synchronize()
        assert lib.exattn_noalloc_device_status(stream) == 0
        for name, got, want in zip(("dQ", "dK", "dV"), outs, ref):
            if dtype == "bf16":  # tensor-core kernels: no atomics, same order
                assert torch.equal(got, want), (call, name)
                continue
            gd, wd = got.double(), want.double()
            assert torch.isfinite(gd).all(), (call, name)
            bound = GRAD_TOL[dtype] * float(wd.abs().max())
            err = float((gd - wd).abs().max())
            assert err <= bound, (call, name, err, bound)


def test_noalloc_wrapper_window_mask_d64(ex):
    """The Python wrapper: bf16, d = 64, the window mask, bitwise attn_bwd."""
    B, H, n, d = 1, 3, 700, 64
    w = workloads.small(B, H, n, d, d, "bf16", "window", 0.125, seed=78, window=200)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, "window", 200)
    ref = ex.bwd(q, k, v, y, g, L, w.scale, "window", 200)
    for _ in range(2):
        got = ex.bwd_noalloc(q, k, v, y, g, L, w.scale, "window", 200, check_status=True)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_status_word_reports_empty_rows(ex):
    """An empty allowed set is a device-side condition: the kernels record
    EXATTN_EMPTY_ROW in the status word inside the scratch array, and
    exattn_noalloc_device_status reads it back; the next call clears it."""
    n, d = 256, 64
    w = workloads.small(1, 2, n, d, d, "bf16", "bitmask", 0.125, seed=79)
    x = workloads.make_inputs(w)
    words = x.bitmask.copy()
    words[[3, 200]] = 0  # rows 3 and 200 allow no key
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    bm = torch.from_numpy(words.view(np.int32)).to(dev)
    y, L = ex.fwd(q, k, v, w.scale, "bitmask", 0, bm)
    with pytest.raises(ex.ExattnError) as e:
        ex.bwd_noalloc(q, k, v, y, g, L, w.scale, "bitmask", 0, bm, check_status=True)
    assert e.value.status == 5
    assert ex.noalloc_device_status() == 5
    bm_full = torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
    y2, L2 = ex.fwd(q, k, v, w.scale, "bitmask", 0, bm_full)
    ex.bwd_noalloc(q, k, v, y2, g, L2, w.scale, "bitmask", 0, bm_full)
    assert ex.noalloc_device_status() == 0


def test_noalloc_wrapper_rejects_a_key_length_unlike_q(ex):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device=dev)
    L = torch.zeros(1, 1, 128, device=dev)
    with pytest.raises(ValueError):
        ex.bwd_noalloc(q, k, k, q, q, L, 0.1, "causal")


def test_noalloc_rejects_problems_beyond_the_static_array(ex):
    """A problem needing more than 64 MiB of scratch is refused before any work
    is queued (the buffers are never touched: null pointers are passed)."""
    lib = ex.load_library()
    big = ex.Shape(4, 32, 4096, 128, 128, 1)
    assert ex.bwd_workspace_size(big, "causal") > 64 << 20
    st = lib.attn_bwd_noalloc(ctypes.byref(big), None, None, None, None, None, None,
                              ctypes.c_float(0.1), ex.MASK_CAUSAL, 0, None, None, None, None,
                              None)
    assert st == 4
    assert b"64 MiB" in lib.exattn_last_error()

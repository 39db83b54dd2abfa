"""GPU: attn_step_host (forward and reverse pass on host tensors, copies and
kernels overlapped over chunks of slices) gives bitwise the results of attn_fwd
and attn_bwd on the same data (fp32 dQ, which the SIMT reverse pass adds with
atomics, to summation order); the slice counts cover one chunk, equal chunks
and a short last chunk, and every mask kind.  The device calls themselves are
checked against the float64 oracle in test_gpu_parity."""
import math

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


CASES = [
    # (B, H, n, d, v, dtype, mask, window)
    (2, 8, 300, 128, 128, "bf16", "causal", 0),    # 16 slices: 4 chunks of 4
    (1, 3, 200, 64, 64, "bf16", "none", 0),        # 3 slices: one chunk
    (2, 41, 136, 64, 64, "bf16", "window", 50),    # 82 slices: 8 chunks, the last one short
    (1, 9, 130, 64, 64, "f32", "bitmask", 0),      # fp32, bitmask copied from the host
    (1, 4, 1000, 128, 128, "bf16", "causal", 0),
    (1, 6, 260, 80, 96, "bf16", "causal", 0),      # widths padded to the 128-wide kernels
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_host_step_matches_the_device_calls(ex, case):
    B, H, n, d, vw, dtype, mask, window = case
    w = workloads.small(B, H, n, d, vw, dtype, mask, 1 / math.sqrt(d), seed=CASES.index(case) + 5)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    bm = None
    if mask == "bitmask":
        bm = torch.from_numpy(x.bitmask.view(np.int32))
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, mask, window, None if bm is None else bm.to(dev))
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, mask, window,
                        None if bm is None else bm.to(dev))
    pin = [t.contiguous().pin_memory() for t in (x.Q, x.K, x.V, x.dY)]
    got = ex.step_host(*pin, w.scale, mask, window, bm, device=dev)
    torch.cuda.synchronize()
    for name, a, b in zip(("Y", "L", "dQ", "dK", "dV"), got, (y, L, dq, dk, dv)):
        b = b.cpu()
        if dtype == "f32" and name == "dQ":
            # The fp32 reverse pass adds dQ with atomics: equal up to summation order.
            tol = 1e-5 * b.abs().max().item()
            assert (a - b).abs().max().item() <= tol, name
        else:
            assert torch.equal(a, b), name


def test_host_step_status_reports_empty_rows(ex):
    """A bitmask row with no allowed key: Y = 0, L = -inf and the status word of
    the step's workspace (the OR over the chunks) says EMPTY_ROW."""
    n, d = 64, 64
    words = np.ones((n, 2), dtype=np.uint32) * 0xFFFFFFFF
    words[5] = 0
    g = torch.Generator().manual_seed(3)
    Q, K, V, G = (torch.randn(1, 9, n, d, generator=g).to(torch.bfloat16).pin_memory()
                  for _ in range(4))
    dev = torch.device("cuda:0")
    shape = ex.Shape(1, 9, n, d, d, 1)
    lib = ex.load_library()
    import ctypes
    ws = ex.workspace(lib.exattn_host_step_workspace_size(ctypes.byref(shape), 3), dev)
    y, L, dq, dk, dv = ex.step_host(Q, K, V, G, 0.125, "bitmask", 0,
                                    torch.from_numpy(words.view(np.int32)), ws=ws, device=dev)
    assert ex.device_status(ws) == 5  # EXATTN_EMPTY_ROW
    assert torch.isneginf(L[:, :, 5]).all()
    assert (y[:, :, 5] == 0).all()


def test_host_step_from_threads_that_exit(ex):
    """attn_step_host keeps its streams and events per host thread and releases
    them when the thread exits.  Several short-lived threads each run a step
    (making and, at exit, destroying their own set); the results match the
    main thread's bitwise, and the main thread's calls still work afterwards."""
    import threading

    w = workloads.small(1, 5, 256, 64, 64, "bf16", "causal", 0.125, seed=31)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    pin = [t.contiguous().pin_memory() for t in (x.Q, x.K, x.V, x.dY)]
    want = ex.step_host(*pin, w.scale, "causal", 0, None, device=dev)
    torch.cuda.synchronize()
    want = [t.clone() for t in want]
    results, errors = {}, []

    def worker(idx):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            out = ex.step_host(*pin, w.scale, "causal", 0, None, stream=s, device=dev)
            s.synchronize()
            results[idx] = [t.clone() for t in out]
        except Exception as e:  # reported below, in the main thread
            errors.append(repr(e))

    for rnd in range(3):
        threads = [threading.Thread(target=worker, args=(4 * rnd + i,)) for i in range(4)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
    assert not errors, errors
    assert len(results) == 12
    for got in results.values():
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    again = ex.step_host(*pin, w.scale, "causal", 0, None, device=dev)
    torch.cuda.synchronize()
    for a, b in zip(again, want):
        assert torch.equal(a, b)

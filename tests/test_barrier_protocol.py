"""CPU checks of the tensor-core kernels' mbarrier protocols (no GPU).

Every wait in those kernels is a parity wait, which is correct only while the
barrier never runs two phases ahead of its waiter, and every arrival must land
in the phase it belongs to.  `barrier_model` writes out each kernel's roles
and barrier operations from its source and runs them under many random
schedules, with the tensor pipe in issue order and TMA copies in any order.

The dQ kernel once waited for dS(t) on one barrier after issuing S(t + 1); the
elementwise warps could then complete dS(t) and dS(t + 1) before the MMA
warp's first poll.  That form is kept in the model (two_ds=False) to show that
the search finds such a schedule; the kernel now uses one barrier per block
parity.
"""
import random

import pytest

import barrier_model as bm

N_SCHEDULES = 400


def _search(factory, make_work, seed, n=N_SCHEDULES, **kw):
    rnd = random.Random(seed)
    failures = []
    for s in range(n):
        work = make_work(rnd)
        r = bm.run_kernel(factory, work, s, **kw)
        if r:
            failures.append((r, work, s))
    return failures


def _counts(rnd):
    return bm.random_counts(rnd, rnd.randint(1, 8))


def test_dq_kernel_protocol_holds():
    assert _search(bm.dq_kernel, _counts, 11) == []


def test_dq_kernel_protocol_holds_with_two_warps_and_deep_rings():
    assert _search(bm.dq_kernel, _counts, 12, ew_warps=2, NK=5, NV=3) == []


def test_dq_kernel_single_ds_barrier_is_found_broken():
    failures = _search(bm.dq_kernel, _counts, 13, two_ds=False)
    assert failures, "the search should find the double completion of the one dS barrier"
    kinds = {f[0].split(" ")[0] for f in failures}
    msgs = " ".join(f[0] for f in failures)
    assert "DS0" in msgs and ("parity wait misses" in msgs or "counted in phase" in msgs), kinds


def test_kv_kernel_protocol_holds():
    assert _search(bm.kv_kernel, _counts, 21) == []


def test_kv_kernel_protocol_holds_with_two_warps():
    assert _search(bm.kv_kernel, _counts, 22, ew_warps=2) == []


def test_forward_kernel_protocol_holds():
    items = lambda rnd: bm.random_fwd_items(rnd, rnd.randint(1, 8))
    assert _search(bm.fwd_kernel, items, 31) == []


def test_forward_kernel_protocol_holds_deeper_ring():
    items = lambda rnd: bm.random_fwd_items(rnd, rnd.randint(1, 6))
    assert _search(bm.fwd_kernel, items, 32, NS=6, warps_per_tile=1) == []


def test_atomic_kernel_protocol_holds():
    assert _search(bm.atomic_kernel, lambda rnd: rnd.randint(0, 9), 41) == []


@pytest.mark.parametrize("factory,drop,kw", [
    (bm.dq_kernel, "QFREE", {}), (bm.dq_kernel, "SFREE", {}), (bm.dq_kernel, "DPART", {}),
    (bm.dq_kernel, "DREAD", {}), (bm.dq_kernel, "EPI", {}),
    (bm.kv_kernel, "ACCFREE", {}), (bm.kv_kernel, "P", {}), (bm.fwd_kernel, "OREAD0", {})])
def test_model_catches_a_missing_wait(factory, drop, kw):
    """Planted mistakes in the model: a role that no longer waits on one barrier
    is caught by some schedule, so the checks are not vacuous."""
    if factory is bm.fwd_kernel:
        make = lambda rnd: bm.random_fwd_items(rnd, rnd.randint(3, 8))
    else:
        make = lambda rnd: bm.random_counts(rnd, rnd.randint(3, 8), (0, 1, 2, 3))
    assert _search(factory, make, 51, n=200, skip_waits={drop}, **kw)


def test_fp32_reverse_kernels_protocol_holds():
    steps = lambda rnd: rnd.randint(0, 11)
    assert _search(bm.kv32_kernel, steps, 61) == []
    assert _search(bm.kv32_kernel, steps, 65, NSS=2, NV=2, promote=1, ew_warps=3) == []
    assert _search(bm.q32_kernel, steps, 62) == []
    assert _search(bm.q32_kernel, steps, 63, NST=2, ew_warps=3) == []


@pytest.mark.parametrize("factory,drop,kw", [
    (bm.kv32_kernel, "QSE0", {}), (bm.kv32_kernel, "QTE0", {}), (bm.kv32_kernel, "SP0", {}),
    # with four vector slots the T-half ring already orders a slot's reuse;
    # with two, the vector ring's own release is what does
    (bm.kv32_kernel, "VE0", {"NV": 2}),
    (bm.q32_kernel, "SP0", {}), (bm.q32_kernel, "DS0", {})])
def test_fp32_reverse_model_catches_a_missing_wait(factory, drop, kw):
    assert _search(factory, lambda rnd: rnd.randint(3, 11), 64, n=200, skip_waits={drop}, **kw)

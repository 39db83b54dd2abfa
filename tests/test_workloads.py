"""The seeded input recipe shared by the parity tests and the benchmark: the five
workloads' shapes, dtypes, masks, scales and seeds; determinism; the bit-row
mask format and density; the allowed-pair counts behind the algorithmic flops;
and the decode workload's algorithmic bytes."""
import math

import numpy as np
import pytest
import torch

import workloads

# (k, variant) -> (B, H, n, d, v, dtype, mask, scale, window, qk_gain)
EXPECTED = {
    (1, ""): (1, 1, 256, 64, 64, "f32", "causal", 1 / 8, 0, 1.0),
    (1, "none"): (1, 1, 256, 64, 64, "f32", "none", 1 / 8, 0, 1.0),
    (1, "self"): (1, 1, 256, 64, 64, "f32", "none", 1.0, 0, 1.0),
    (2, ""): (8, 16, 2048, 64, 64, "bf16", "none", 1 / 8, 0, 1.0),
    (3, ""): (4, 32, 4096, 128, 128, "bf16", "causal", 1 / math.sqrt(128), 0, 1.0),
    (4, ""): (1, 16, 16384, 128, 128, "bf16", "causal", 1 / math.sqrt(128), 0, 1.5),
    (4, "window"): (1, 16, 16384, 128, 128, "bf16", "window", 1 / math.sqrt(128), 1024, 1.5),
    (5, ""): (2, 8, 1000, 80, 96, "f32", "bitmask", 0.1, 0, 1.0),
    (5, "bf16"): (2, 8, 1000, 80, 96, "bf16", "bitmask", 0.1, 0, 1.0),
}


@pytest.mark.parametrize("key", list(EXPECTED), ids=lambda k: f"{k[0]}{k[1]}")
def test_workload_table(key):
    k, variant = key
    w = workloads.workload(k, variant)
    B, H, n, d, v, dtype, mask, scale, window, gain = EXPECTED[key]
    assert (w.B, w.H, w.n, w.d, w.v, w.dtype, w.mask) == (B, H, n, d, v, dtype, mask)
    assert w.scale == pytest.approx(scale, rel=1e-15)
    assert w.window == window and w.qk_gain == gain
    assert w.seed == workloads.SEED_BASE + k
    assert w.n_keys == n
    assert w.self_attention == (variant == "self")


def test_unknown_workload_is_rejected():
    with pytest.raises(ValueError):
        workloads.workload(6)


def _unpack(bits, cols):
    rows, W = bits.shape
    out = np.zeros((rows, W * 32), dtype=bool)
    for b in range(32):
        out[:, b::32] = (bits >> np.uint32(b)) & np.uint32(1)
    return out[:, :cols]


def test_pack_bitmask_layout():
    """Bit j % 32 of word j // 32 of row i is key j of row i."""
    rng = np.random.default_rng(0)
    allowed = rng.random((7, 70)) < 0.4
    bits = workloads.pack_bitmask(allowed)
    assert bits.dtype == np.uint32 and bits.shape == (7, 3)
    assert np.array_equal(_unpack(bits, 70), allowed)
    # Columns past the last key are zero.
    assert (bits[:, 2] >> np.uint32(6)).max() == 0
    one = np.zeros((1, 64), dtype=bool)
    one[0, 33] = True
    assert workloads.pack_bitmask(one).tolist() == [[0, 2]]


def test_inputs_are_deterministic_and_in_the_workload_dtype():
    w = workloads.small(1, 2, 100, 16, 24, "bf16", "bitmask", 0.2, seed=5)
    a, b = workloads.make_inputs(w), workloads.make_inputs(w)
    for x, y, shape in zip((a.Q, a.K, a.V, a.dY), (b.Q, b.K, b.V, b.dY),
                           ((1, 2, 100, 16), (1, 2, 100, 16), (1, 2, 100, 24), (1, 2, 100, 24))):
        assert x.dtype == torch.bfloat16 and tuple(x.shape) == shape
        assert torch.equal(x, y)
    assert np.array_equal(a.bitmask, b.bitmask)
    c = workloads.make_inputs(workloads.small(1, 2, 100, 16, 24, "bf16", "bitmask", 0.2, seed=6))
    assert not torch.equal(a.Q, c.Q)
    # The oracle's float64 copies are exact.
    q64 = a.as_f64()[0]
    assert q64.dtype == np.float64 and np.array_equal(q64, a.Q.float().numpy())


def test_bitmask_density_and_diagonal():
    w = workloads.workload(5)
    x = workloads.make_inputs(w, heads=1)
    allowed = _unpack(x.bitmask, w.n)
    assert allowed.shape == (1000, 1000)
    assert allowed.diagonal().all()  # every allowed-key set is nonempty
    off = allowed[~np.eye(1000, dtype=bool)]
    # 999 000 Bernoulli(0.3) draws: standard deviation ~4.6e-4.
    assert abs(off.mean() - 0.3) < 3e-3


def test_value_recipe():
    """N(0, 1) draws; Q and K scaled by the gain; self-attention X ~ N(0, 0.25)."""
    w = workloads.small(1, 4, 512, 64, 64, "f32", "none", 0.1, qk_gain=1.5, seed=3)
    x = workloads.make_inputs(w)
    assert float(x.Q.std()) == pytest.approx(1.5, rel=0.02)
    assert float(x.K.std()) == pytest.approx(1.5, rel=0.02)
    assert float(x.V.std()) == pytest.approx(1.0, rel=0.02)
    assert float(x.dY.std()) == pytest.approx(1.0, rel=0.02)
    s = workloads.make_inputs(workloads.workload(1, "self"))
    assert s.Q is s.K and s.K is s.V
    assert float(s.Q.std()) == pytest.approx(0.5, rel=0.05)
    assert float(s.dY.std()) == pytest.approx(1.0, rel=0.05)


def _pairs_brute(n, nk, mask, window):
    off = nk - n
    total = 0
    for i in range(n):
        for j in range(nk):
            a = i + off  # absolute position of query i
            if mask == "none":
                total += 1
            elif mask == "causal":
                total += j <= a
            else:
                total += a - window + 1 <= j <= a
    return total


@pytest.mark.parametrize("n,nk", [(1, 1), (7, 7), (130, 130), (40, 100), (100, 40)])
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal", 0), ("window", 1),
                                         ("window", 17)])
def test_allowed_pairs_per_head(n, nk, mask, window):
    w = workloads.small(1, 1, n, 8, 8, "f32", mask, 1.0, window=window)
    w.nk = nk
    assert w.allowed_pairs_per_head() == _pairs_brute(n, nk, mask, window)


def test_bitmask_pair_count_is_not_guessed():
    with pytest.raises(ValueError):
        workloads.workload(5).allowed_pairs_per_head()


def test_decode_workload_bytes():
    """One decode step reads Q, K, V once and writes Y and L."""
    w = workloads.decode_workload(1)
    assert (w.B, w.H, w.nq, w.nk, w.d, w.v, w.dtype, w.mask) == (8, 32, 1, 16384, 128, 128,
                                                                  "bf16", "causal")
    assert w.bytes_moved() == 2_147_615_744
    assert workloads.decode_workload(4).bytes_moved() == 8 * 32 * (
        4 * 128 * 2 + 16384 * 256 * 2 + 4 * (128 * 2 + 4))


def test_decode_inputs_mask_keeps_each_querys_own_key():
    Q, K, V, dY, bits = workloads.make_decode_inputs(1, 2, 5, 70, 8, 8, "f32", "bitmask",
                                                     seed=4, p_allow=0.0, with_dy=True)
    assert tuple(Q.shape) == (1, 2, 5, 8) and tuple(K.shape) == (1, 2, 70, 8)
    assert tuple(dY.shape) == (1, 2, 5, 8)
    allowed = _unpack(bits, 70)
    # p_allow = 0: only the query's own position i + nk - nq is allowed.
    assert [list(np.flatnonzero(r)) for r in allowed] == [[65], [66], [67], [68], [69]]

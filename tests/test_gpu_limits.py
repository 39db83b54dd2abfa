"""GPU runs at the library's size limits, checked on outputs the oracle can form
one row at a time and on identities that hold at any size.

  * the longest sequence the library accepts (n = 2^20, one head, bf16,
    causal, tensor-core kernels): sampled rows of Y and L against the oracle's
    row forward; Sum_j dK_j = 0 and Sum_j dV_j = Sum_i dY_i, which hold exactly
    in real arithmetic ("Exact tiled softmax attention with block-recomputed
    vector-Jacobian products", Reverse procedure: Sum_j gamma_ij = 0 and
    Sum_j p_ij = 1);
  * the most (batch, head) slices one call takes (65535, the grid's y limit),
    compared head by head on a sample;
  * a bitmask longer than the tensor-core kernels' tile table (n = 40000: the
    SIMT kernels run it), sampled rows plus the same identities.
Bounds: the bf16 row outputs as in tests/tolerances.py; the identities to 2e-2
of the size of the sums involved (bf16 outputs summed over 2^20 rows)."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import dense, masks
from tolerances import compare, half_ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ex():
    import exact_tiled_softmax_gb300 as mod
    mod.load_library()
    assert torch.cuda.is_available()
    return mod


def _rows_and_identities(ex, Q, K, V, G, c, mask, rows, allowed_row, bits=None):
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (Q, K, V, G))
    bm = None if bits is None else torch.from_numpy(bits.view(np.int32)).to(dev)
    y, L = ex.fwd(q, k, v, c, mask, 0, bm)
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, c, mask, 0, bm)
    torch.cuda.synchronize()
    Qd, Kd, Vd = (t[0, 0].double().numpy() for t in (Q, K, V))
    Y = y[0, 0].double().cpu().numpy()
    Lg = L[0, 0].double().cpu().numpy()
    for i in rows:
        yr, lr = dense.row_forward(Qd, Kd, Vd, c, allowed_row(i), i)
        assert abs(Lg[i] - lr) <= 1e-4, (i, Lg[i], lr)
        assert (np.abs(Y[i] - yr) - half_ulp_bf16(yr)).max() <= 1e-2, i
    dK = dk[0, 0].double().cpu().numpy()
    dV = dv[0, 0].double().cpu().numpy()
    sum_dy = G[0, 0].double().numpy().sum(axis=0)
    assert np.abs(dV.sum(axis=0) - sum_dy).max() <= 2e-2 * np.abs(sum_dy).max()
    assert np.abs(dK.sum(axis=0)).max() <= 2e-2 * np.abs(dK).sum(axis=0).max()
    assert np.isfinite(dq.float().cpu().numpy()).all()


def test_longest_sequence(ex):
    n, d = 1 << 20, 64
    g = torch.Generator().manual_seed(2026)
    Q, K, V, G = (torch.randn(1, 1, n, d, generator=g).to(torch.bfloat16) for _ in range(4))
    rows = [0, 1, 12345, n // 2, n - 1]
    _rows_and_identities(ex, Q, K, V, G, 1 / math.sqrt(d), "causal", rows,
                         lambda i: np.arange(n) <= i)


def test_most_slices(ex):
    w = workloads.small(65535, 1, 3, 64, 64, "bf16", "causal", 0.125, seed=17)
    x = workloads.make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, g = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    y, L = ex.fwd(q, k, v, w.scale, "causal")
    dq, dk, dv = ex.bwd(q, k, v, y, g, L, w.scale, "causal")
    torch.cuda.synchronize()
    heads = [0, 32767, 65534]
    sel = lambda t: t[heads].double().numpy()  # noqa: E731
    Q, K, V, G = (sel(t.reshape(-1, 3, 64)) for t in (x.Q, x.K, x.V, x.dY))
    allowed = masks.allowed_matrix(3, masks.CAUSAL)
    ref = {key: [] for key in ("Y", "L", "dQ", "dK", "dV")}
    for h in range(len(heads)):
        yy, ll = dense.head_forward(Q[h], K[h], V[h], w.scale, allowed)
        a, b, cc, _ = dense.head_backward(Q[h], K[h], V[h], G[h], w.scale, allowed)
        for key, val in zip(("Y", "L", "dQ", "dK", "dV"), (yy, ll, a, b, cc)):
            ref[key].append(val)
    compare("bf16", dict(Y=y, L=L, dQ=dq, dK=dk, dV=dv),
            {key: np.stack(val) for key, val in ref.items()}, heads=heads)


def test_long_bitmask_beyond_the_tile_table(ex):
    """Row i allows keys j <= i whose bit j % 32 is set in a per-row 32-bit
    pattern (its own position always set): built word by word, no n x n draw."""
    n, d = 40000, 64
    W = (n + 31) // 32
    rng = np.random.default_rng(40000)
    pattern = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    i = np.arange(n)
    pattern |= (np.uint32(1) << (i % 32).astype(np.uint32))
    words = np.repeat(pattern[:, None], W, axis=1)
    w_idx = np.arange(W)[None, :]
    last = (i // 32)[:, None]
    words[w_idx > last] = 0
    tail = (np.uint64(1) << ((i % 32) + 1).astype(np.uint64)) - np.uint64(1)
    words[i, i // 32] &= tail.astype(np.uint32)
    g = torch.Generator().manual_seed(4)
    Q, K, V, G = (torch.randn(1, 1, n, d, generator=g).to(torch.bfloat16) for _ in range(4))

    def allowed_row(r):
        bits = (words[r][np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1
        return bits.astype(bool)

    _rows_and_identities(ex, Q, K, V, G, 0.125, "bitmask", [0, 31, 32, 20000, n - 1],
                         allowed_row, bits=words.astype(np.uint32))

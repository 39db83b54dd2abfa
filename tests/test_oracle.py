"""Pins for the float64 oracle (CPU only).

Each pin ties the oracle to something other than itself: hand-worked values
(re-derived here with exact rationals), the pages' own block procedures at
every block size, a library routine (torch's float64 scaled-dot-product
attention and autograd), central finite differences, and invariants that the
mathematics fixes.  ``test_planted_mistakes_are_caught`` plants typical mistakes
in a copy of the oracle and checks that the same pins reject every one.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import dense, masks, tiled
from workloads import pack_bitmask

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

def _load(path):
    with open(path) as f:
        return json.load(f)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
KINDS = {"none": masks.NONE, "causal": masks.CAUSAL}


def _expr(x):
    """Evaluate a fixture entry: a number or an expression in rationals and ln(k)."""
    if isinstance(x, (int, float)):
        return float(x)
    return float(eval(x, {"__builtins__": {}}, {"ln": math.log}))


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    """Normwise relative error max|a-b| / max|b|."""
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------- #
# Hand-worked cases (re-derived exactly, then compared with the fixture)
# --------------------------------------------------------------------------- #

def test_hand_cases_rederived_exactly():
    """The 3x3 Q=0 case has rational outputs: re-derive them with Fractions."""
    V = [Fraction(1), Fraction(2), Fraction(3)]
    K = [Fraction(1), Fraction(0), Fraction(-1)]
    G = [Fraction(1)] * 3
    Y, dQ = [], []
    dV = [Fraction(0)] * 3
    for i in range(3):
        p = [Fraction(1, i + 1) if j <= i else Fraction(0) for j in range(3)]
        y = sum(p[j] * V[j] for j in range(3))
        Y.append(y)
        gam = [p[j] * (G[i] * V[j] - G[i] * y) for j in range(3)]
        dQ.append(sum(gam[j] * K[j] for j in range(3)))
        for j in range(3):
            dV[j] += p[j] * G[i]
    case = _load(GOLDEN)["cases"][2]
    assert [Fraction(s) for s in case["Y"]] == Y
    assert [Fraction(s) for s in case["dQ"]] == dQ
    assert [Fraction(s) for s in case["dV"]] == dV
    # 2x2 full: p_11 = 2/3 (e^{ln 2} = 2 against e^0 = 1), p_21 = 1/2.
    p = [[Fraction(2, 3), Fraction(1, 3)], [Fraction(1, 2), Fraction(1, 2)]]
    Vv = [Fraction(1), Fraction(0)]
    Yf = [sum(p[i][j] * Vv[j] for j in range(2)) for i in range(2)]
    gam = [[p[i][j] * (Vv[j] - Yf[i]) for j in range(2)] for i in range(2)]
    case = _load(GOLDEN)["cases"][0]
    assert [Fraction(s) for s in case["Y"]] == Yf
    # dK_j = sum_i gamma_ij Q_i with Q = (1, 0)
    assert [Fraction(s) for s in case["dK"]] == [gam[0][0], gam[0][1]]
    assert [Fraction(s) for s in case["dV"]] == [p[0][j] + p[1][j] for j in range(2)]
    # dQ_i = gamma_i1 * ln 2 (K_2 = 0): coefficients 2/9 and 1/4
    assert gam[0][0] == Fraction(2, 9) and gam[1][0] == Fraction(1, 4)


def _hand_failures(head_forward, head_backward):
    out = []
    for case in _load(GOLDEN)["cases"]:
        arr = {k: np.array([[_expr(x) for x in row] for row in case[k]])
               for k in ("Q", "K", "V", "G")}
        n = arr["Q"].shape[0]
        allowed = masks.allowed_matrix(n, KINDS[case["mask"]])
        Y, L = head_forward(arr["Q"], arr["K"], arr["V"], case["c"], allowed)
        dQ, dK, dV = head_backward(arr["Q"], arr["K"], arr["V"], arr["G"], case["c"],
                                   allowed)[:3]
        got = {"Y": Y[:, 0], "L": L, "dQ": dQ[:, 0], "dK": dK[:, 0], "dV": dV[:, 0]}
        for key, val in got.items():
            want = np.array([_expr(x) for x in case[key]])
            if not np.allclose(val, want, rtol=0, atol=1e-14):
                out.append(f"hand case '{case['name']}' {key}: {val} != {want}")
    return out


# --------------------------------------------------------------------------- #
# Pins shared by the real oracle and the planted-mistake copies
# --------------------------------------------------------------------------- #

def _fd_failures(head_forward, head_backward, self_attention=False):
    """Central differences of f = <G, Y> against the reverse pass, rel err <= 1e-5."""
    out = []
    r = _rng(11)
    for kind, n, d, v, c in [(masks.NONE, 3, 2, 3, 0.7), (masks.CAUSAL, 4, 3, 2, 1.3)]:
        allowed = masks.allowed_matrix(n, kind)
        Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
        G = r.normal(size=(n, v))
        if self_attention:
            X = r.normal(size=(n, d))
            G = r.normal(size=(n, d))
            Q = K = V = X
        dQ, dK, dV = head_backward(Q, K, V, G, c, allowed)[:3]
        h = 1e-6

        def f(q, k, vv):
            return float((G * head_forward(q, k, vv, c, allowed)[0]).sum())

        if self_attention:
            num = np.zeros_like(X)
            for idx in np.ndindex(*X.shape):
                e = np.zeros_like(X)
                e[idx] = h
                num[idx] = (f(X + e, X + e, X + e) - f(X - e, X - e, X - e)) / (2 * h)
            err = _rel(dQ + dK + dV, num)
            if err > 1e-5:
                out.append(f"finite differences, shared X: rel err {err:.2e}")
            continue
        for name, grad, which in (("dQ", dQ, 0), ("dK", dK, 1), ("dV", dV, 2)):
            base = [Q, K, V]
            num = np.zeros_like(base[which])
            for idx in np.ndindex(*base[which].shape):
                e = np.zeros_like(base[which])
                e[idx] = h
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[which] += e
                minus[which] -= e
                num[idx] = (f(*plus) - f(*minus)) / (2 * h)
            err = _rel(grad, num)
            if err > 1e-5:
                out.append(f"finite differences {name} (kind {kind}): rel err {err:.2e}")
    return out


def _torch_failures(head_forward, head_backward):
    """torch's float64 scaled_dot_product_attention + autograd + logsumexp."""
    out = []
    r = _rng(5)
    for kind, n, d, v, c in [(masks.NONE, 37, 8, 5, 0.31), (masks.CAUSAL, 41, 6, 9, 1.7),
                             (masks.WINDOW, 29, 4, 4, 0.5), (masks.BITMASK, 33, 7, 3, 0.9)]:
        bitmask = None
        if kind == masks.BITMASK:
            a = r.random((n, n)) < 0.3
            np.fill_diagonal(a, True)
            bitmask = pack_bitmask(a)
        allowed = masks.allowed_matrix(n, kind, window=5, bitmask=bitmask)
        Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
        G = r.normal(size=(n, v))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        tm = torch.tensor(allowed)
        ty = torch.nn.functional.scaled_dot_product_attention(
            tq[None], tk[None], tv[None], attn_mask=tm, scale=c)[0]
        (ty * torch.tensor(G)).sum().backward()
        s = (tq @ tk.T * c).masked_fill(~tm, float("-inf"))
        tL = torch.logsumexp(s, dim=1)
        Y, L = head_forward(Q, K, V, c, allowed)
        dQ, dK, dV = head_backward(Q, K, V, G, c, allowed)[:3]
        for name, mine, ref in (("Y", Y, ty.detach().numpy()), ("L", L, tL.detach().numpy()),
                                ("dQ", dQ, tq.grad.numpy()), ("dK", dK, tk.grad.numpy()),
                                ("dV", dV, tv.grad.numpy())):
            err = _rel(mine, ref)
            if err > 1e-12:
                out.append(f"torch cross-check {name} (kind {kind}): rel err {err:.2e}")
    return out


def _invariant_failures(head_forward, head_backward):
    out = []
    r = _rng(7)
    n, d, v, c = 23, 5, 4, 0.8
    for kind in (masks.NONE, masks.CAUSAL, masks.WINDOW):
        allowed = masks.allowed_matrix(n, kind, window=4)
        Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
        G = r.normal(size=(n, v))
        Y, L = head_forward(Q, K, V, c, allowed)
        dQ, dK, dV, delta = head_backward(Q, K, V, G, c, allowed)
        # Y_i is a convex combination of the allowed V_j: inside their column range.
        for i in range(n):
            Va = V[allowed[i]]
            if (Y[i] < Va.min(0) - 1e-12).any() or (Y[i] > Va.max(0) + 1e-12).any():
                out.append(f"Y row {i} outside the hull of its allowed values")
                break
        # delta_i = G_i . Y_i (the D identity of the backward section).
        if _rel(delta, (G * Y).sum(1)) > 1e-12:
            out.append("delta != G.Y")
        # sum_j gamma_ij = 0  =>  sum_j dK_j = 0;  sum_j p_ij = 1  =>  sum_j dV_j = sum_i G_i.
        if np.abs(dK.sum(0)).max() > 1e-12 * max(1.0, np.abs(dK).max()):
            out.append("sum_j dK_j != 0")
        if _rel(dV.sum(0), G.sum(0)) > 1e-12:
            out.append("sum_j dV_j != sum_i G_i")
        # Adding a constant row w to every V_j shifts Y by w and leaves dQ, dK alone.
        w = r.normal(size=v)
        Y2, L2 = head_forward(Q, K, V + w, c, allowed)
        dQ2, dK2 = head_backward(Q, K, V + w, G, c, allowed)[:2]
        if _rel(Y2, Y + w) > 1e-12 or _rel(L2, L) > 1e-14:
            out.append("V + 1w^T does not shift Y by w")
        if _rel(dQ2, dQ) > 1e-10 or _rel(dK2, dK) > 1e-10:
            out.append("V + 1w^T changes dQ or dK")
        # Scale: (Q a, c / a) gives the same scores.
        Y3 = head_forward(Q * 2.5, K, V, c / 2.5, allowed)[0]
        if _rel(Y3, Y) > 1e-12:
            out.append("scale c not applied to <Q_i, K_j>")
        # Logsumexp: L_i >= max allowed score and L_i <= max + ln|A_i|.
        s = np.where(allowed, c * Q @ K.T, -np.inf)
        smax = s.max(1)
        if (L < smax - 1e-12).any() or (L > smax + np.log(allowed.sum(1)) + 1e-12).any():
            out.append("L outside [max s, max s + ln|A_i|]")
    # Full mask: permuting the keys (with their values) leaves Y unchanged and
    # permutes dK and dV the same way.
    allowed = np.ones((n, n), dtype=bool)
    Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
    G = r.normal(size=(n, v))
    perm = r.permutation(n)
    Y = head_forward(Q, K, V, c, allowed)[0]
    Yp = head_forward(Q, K[perm], V[perm], c, allowed)[0]
    dK, dV = head_backward(Q, K, V, G, c, allowed)[1:3]
    dKp, dVp = head_backward(Q, K[perm], V[perm], G, c, allowed)[1:3]
    if _rel(Yp, Y) > 1e-12 or _rel(dKp, dK[perm]) > 1e-10 or _rel(dVp, dV[perm]) > 1e-12:
        out.append("key permutation equivariance broken")
    return out


def _special_failures(head_forward, head_backward):
    out = []
    r = _rng(9)
    n, d, v, c = 9, 3, 4, 0.6
    Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
    G = r.normal(size=(n, v))
    # One allowed key per row (a permutation): Y_i = V_pi(i), L_i = s_i,pi(i), dQ = 0.
    pi = r.permutation(n)
    allowed = np.zeros((n, n), dtype=bool)
    allowed[np.arange(n), pi] = True
    Y, L = head_forward(Q, K, V, c, allowed)
    dQ = head_backward(Q, K, V, G, c, allowed)[0]
    if _rel(Y, V[pi]) > 1e-15:
        out.append("single key: Y_i != V_j")
    if _rel(L, c * (Q * K[pi]).sum(1)) > 1e-14:
        out.append("single key: L_i != s_ij")
    if np.abs(dQ).max() > 1e-15:
        out.append("single key: dQ != 0")
    # Q = 0 under the causal mask: uniform p = 1/|A_i|, L_i = ln |A_i|, Y_i = prefix mean.
    allowed = masks.allowed_matrix(n, masks.CAUSAL)
    Y, L = head_forward(np.zeros((n, d)), K, V, c, allowed)
    if _rel(Y, np.cumsum(V, 0) / np.arange(1, n + 1)[:, None]) > 1e-14:
        out.append("Q=0: Y != prefix mean")
    if _rel(L, np.log(np.arange(1, n + 1))) > 1e-14:
        out.append("Q=0: L != ln |A_i|")
    return out


def _tiled_failures(head_forward, head_backward):
    """The page's block procedures agree with the definition under test."""
    out = []
    r = _rng(3)
    n, d, v, c = 19, 4, 5, 0.9
    for kind in (masks.NONE, masks.CAUSAL, masks.WINDOW):
        allowed = masks.allowed_matrix(n, kind, window=6)
        Q, K, V = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v))
        G = r.normal(size=(n, v))
        Y, L = head_forward(Q, K, V, c, allowed)
        Yt, m, l, Lt = tiled.summary_forward(Q, K, V, c, allowed, 4)
        if _rel(Yt, Y) > 1e-12 or _rel(Lt, L) > 1e-12:
            out.append(f"summary forward disagrees (kind {kind})")
        got = head_backward(Q, K, V, G, c, allowed)[:3]
        want = tiled.recompute_backward(Q, K, V, G, Yt, m, l, c, allowed, 4)[:3]
        for name, a, b in zip(("dQ", "dK", "dV"), got, want):
            if _rel(a, b) > 1e-11:
                out.append(f"recompute backward {name} disagrees (kind {kind})")
    return out


def pin_failures(head_forward, head_backward):
    return (_hand_failures(head_forward, head_backward)
            + _fd_failures(head_forward, head_backward)
            + _fd_failures(head_forward, head_backward, self_attention=True)
            + _torch_failures(head_forward, head_backward)
            + _invariant_failures(head_forward, head_backward)
            + _special_failures(head_forward, head_backward)
            + _tiled_failures(head_forward, head_backward))


def test_oracle_passes_every_pin():
    assert pin_failures(dense.head_forward, dense.head_backward) == []


# --------------------------------------------------------------------------- #
# Block-size exactness (O1) and the recompute reverse pass (O2)
# --------------------------------------------------------------------------- #

def _case(n, d, v, kind, seed, window=3, p=0.3):
    r = _rng(seed)
    bitmask = None
    if kind == masks.BITMASK:
        a = r.random((n, n)) < p
        np.fill_diagonal(a, True)
        bitmask = pack_bitmask(a)
    allowed = masks.allowed_matrix(n, kind, window=window, bitmask=bitmask)
    return (r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v)),
            r.normal(size=(n, v)), allowed)


ALL_KINDS = (masks.NONE, masks.CAUSAL, masks.WINDOW, masks.BITMASK)


@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 33])
@pytest.mark.parametrize("kind", ALL_KINDS)
def test_every_block_size_gives_the_dense_result(n, kind):
    Q, K, V, G, allowed = _case(n, 5, 3, kind, seed=100 + n)
    c = 0.45
    Y, L = dense.head_forward(Q, K, V, c, allowed)
    for b in range(1, n + 1):
        Ys, m, l, Ls = tiled.summary_forward(Q, K, V, c, allowed, b)
        Yo, Lo = tiled.online_forward(Q, K, V, c, allowed, b)
        assert _rel(Ys, Y) <= 1e-12 and _rel(Ls, L) <= 1e-12, b
        assert _rel(Yo, Y) <= 1e-12 and _rel(Lo, L) <= 1e-12, b


@pytest.mark.parametrize("kind", ALL_KINDS)
def test_block_sizes_at_n256(kind):
    Q, K, V, G, allowed = _case(256, 16, 12, kind, seed=256, window=40)
    c = 0.25
    Y, L = dense.head_forward(Q, K, V, c, allowed)
    dQ, dK, dV, _ = dense.head_backward(Q, K, V, G, c, allowed)
    for b in (1, 2, 3, 16, 31, 64, 100, 256):
        Ys, m, l, Ls = tiled.summary_forward(Q, K, V, c, allowed, b)
        assert _rel(Ys, Y) <= 1e-12 and _rel(Ls, L) <= 1e-12, b
        got = tiled.recompute_backward(Q, K, V, G, Ys, m, l, c, allowed, b)
        for a, ref in zip(got[:3], (dQ, dK, dV)):
            assert _rel(a, ref) <= 1e-11, b


def test_delta_identity_rowwise():
    """sum_j p_ij dP_ij = G_i . Y_i per row (backward section, D identity)."""
    for kind in ALL_KINDS:
        Q, K, V, G, allowed = _case(64, 8, 8, kind, seed=21)
        Y, _ = dense.head_forward(Q, K, V, 0.3, allowed)
        delta = dense.head_backward(Q, K, V, G, 0.3, allowed)[3]
        gy = (G * Y).sum(1)
        assert np.all(np.abs(delta - gy) <= 1e-12 * np.maximum(1.0, np.abs(gy)))


def test_batched_layout_matches_heads():
    r = _rng(2)
    Q, K, V, G = (r.normal(size=(2, 3, 10, 4)) for _ in range(4))
    Y, L = dense.forward(Q, K, V, 0.5, masks.CAUSAL)
    dQ, dK, dV, delta = dense.backward(Q, K, V, G, 0.5, masks.CAUSAL)
    allowed = masks.allowed_matrix(10, masks.CAUSAL)
    y, l = dense.head_forward(Q[1, 2], K[1, 2], V[1, 2], 0.5, allowed)
    assert np.array_equal(Y[1, 2], y) and np.array_equal(L[1, 2], l)
    g = dense.head_backward(Q[1, 2], K[1, 2], V[1, 2], G[1, 2], 0.5, allowed)
    assert np.array_equal(dK[1, 2], g[1]) and np.array_equal(dV[1, 2], g[2])
    Ys, Ls = dense.forward(Q, K, V, 0.5, masks.CAUSAL, heads=[5])
    assert np.array_equal(Ys[0], y)
    yi, li = dense.row_forward(Q[1, 2], K[1, 2], V[1, 2], 0.5, allowed[7], 7)
    assert _rel(yi, y[7]) < 1e-15 and abs(li - l[7]) < 1e-15


def test_row_backward_against_torch_autograd_and_hand_cases():
    """dense.row_backward, the one-row reverse pass behind the sampled full-size
    checks: every row's dQ_i against torch's float64 autograd through SDPA on
    the four mask kinds, delta_i against G_i . Y_i (torch's Y), and the dQ
    column of the hand-worked cases exactly."""
    r = _rng(6)
    for kind, n, d, v, c in [(masks.NONE, 23, 8, 5, 0.31), (masks.CAUSAL, 31, 6, 9, 1.7),
                             (masks.WINDOW, 19, 4, 4, 0.5), (masks.BITMASK, 27, 7, 3, 0.9)]:
        bitmask = None
        if kind == masks.BITMASK:
            a = r.random((n, n)) < 0.3
            np.fill_diagonal(a, True)
            bitmask = pack_bitmask(a)
        allowed = masks.allowed_matrix(n, kind, window=4, bitmask=bitmask)
        Q, K, V, G = (r.normal(size=(n, w)) for w in (d, d, v, v))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        ty = torch.nn.functional.scaled_dot_product_attention(
            tq[None], tk[None], tv[None], attn_mask=torch.tensor(allowed), scale=c)[0]
        (ty * torch.tensor(G)).sum().backward()
        tdq, Yt = tq.grad.numpy(), ty.detach().numpy()
        rows = [dense.row_backward(Q, K, V, G, c, allowed[i], i) for i in range(n)]
        dq = np.stack([x[0] for x in rows])
        delta = np.array([x[1] for x in rows])
        assert _rel(dq, tdq) <= 1e-12, kind
        assert _rel(delta, (G * Yt).sum(axis=1)) <= 1e-12, kind
    for case in _load(GOLDEN)["cases"]:
        arr = {k: np.array([[_expr(x) for x in row] for row in case[k]])
               for k in ("Q", "K", "V", "G")}
        n = arr["Q"].shape[0]
        allowed = masks.allowed_matrix(n, KINDS[case["mask"]])
        want = np.array([_expr(x) for x in case["dQ"]])
        for i in range(n):
            got = dense.row_backward(arr["Q"], arr["K"], arr["V"], arr["G"], case["c"],
                                     allowed[i], i)[0]
            assert abs(got[0] - want[i]) <= 1e-14, (case["name"], i)


def test_empty_allowed_set_is_rejected():
    allowed = np.ones((3, 3), dtype=bool)
    allowed[1] = False
    z = np.zeros((3, 2))
    with pytest.raises(ValueError):
        dense.head_forward(z, z, z, 1.0, allowed)
    with pytest.raises(ValueError):
        tiled.summary_forward(z, z, z, 1.0, allowed, 2)


# --------------------------------------------------------------------------- #
# Mask readings, checked by plain membership loops
# --------------------------------------------------------------------------- #

def test_mask_readings():
    n = 45
    for i in range(n):
        for j in range(n):
            assert masks.allowed_matrix(n, masks.CAUSAL)[i, j] == (j <= i)
    win = masks.allowed_matrix(n, masks.WINDOW, window=7)
    for i in range(n):
        assert set(np.nonzero(win[i])[0]) == set(range(max(0, i - 6), i + 1))
    r = _rng(4)
    a = r.random((n, n)) < 0.4
    words = pack_bitmask(a)
    assert words.shape == (n, 2) and words.dtype == np.uint32
    for i in range(n):
        for j in range(n):
            bit = (int(words[i, j // 32]) >> (j % 32)) & 1
            assert bit == int(a[i, j])
    assert np.array_equal(masks.allowed_matrix(n, masks.BITMASK, bitmask=words), a)
    # A window wider than n is the causal mask.
    assert np.array_equal(masks.allowed_matrix(n, masks.WINDOW, window=10 * n),
                          masks.allowed_matrix(n, masks.CAUSAL))


# --------------------------------------------------------------------------- #
# Planted mistakes: a copy of the oracle with one fault at a time must fail a pin
# --------------------------------------------------------------------------- #

def _mutant(fault):
    def fwd(Q, K, V, c, allowed):
        cc = 1.0 if fault == "no_scale" else c
        s = cc * (K @ Q.T) if fault == "transposed_scores" else cc * (Q @ K.T)
        al = allowed.T if fault == "transposed_mask" else allowed
        s = np.where(al, s, -np.inf)
        m = s.max(1)
        e = np.exp(s - m[:, None])
        l = e.sum(1)
        Y = (e / l[:, None]) @ V
        L = np.log(l) if fault == "L_without_max" else m + np.log(l)
        return Y, L

    def bwd(Q, K, V, G, c, allowed):
        s = np.where(allowed, c * (Q @ K.T), -np.inf)
        e = np.exp(s - s.max(1)[:, None])
        P = e / e.sum(1)[:, None]
        dV = P @ G if fault == "dV_untransposed" else P.T @ G
        dP = G @ V.T
        delta = (P * dP).sum(1)
        if fault == "no_delta":
            delta = 0 * delta
        if fault == "delta_sign":
            delta = -delta
        dS = P * (dP - delta[:, None])
        dQ = c * (dS.T @ K) if fault == "dQ_transposed" else c * (dS @ K)
        dK = dS.T @ Q if fault == "dK_no_scale" else c * (dS.T @ Q)
        if fault == "dK_uses_K":
            dK = c * (dS.T @ K)
        return dQ, dK, dV, delta

    return fwd, bwd


FAULTS = ["no_scale", "transposed_scores", "transposed_mask", "L_without_max",
          "dV_untransposed", "no_delta", "delta_sign", "dQ_transposed", "dK_no_scale",
          "dK_uses_K"]


def test_unfaulted_copy_passes():
    assert pin_failures(*_mutant(None)) == []


@pytest.mark.parametrize("fault", FAULTS)
def test_planted_mistakes_are_caught(fault):
    assert pin_failures(*_mutant(fault)), f"no pin caught {fault}"


# --------------------------------------------------------------------------- #
# Queries aligned to the end of a longer key sequence (decode / split-KV)
# --------------------------------------------------------------------------- #

def test_rect_mask_reading_reduces_to_square_and_to_last_rows():
    n = 70
    r = _rng(12)
    a = r.random((n, n)) < 0.3
    np.fill_diagonal(a, True)
    for kind, kw in ((masks.NONE, {}), (masks.CAUSAL, {}), (masks.WINDOW, dict(window=9)),
                     (masks.BITMASK, dict(bitmask=pack_bitmask(a)))):
        sq = masks.allowed_matrix(n, kind, **kw)
        assert np.array_equal(masks.allowed_matrix_rect(n, n, kind, **kw), sq)
        # The last nq rows of the square problem are the nq-query problem
        # (bit rows restricted to those queries).
        nq = 5
        if kind == masks.BITMASK:
            kw = dict(bitmask=pack_bitmask(a[-nq:]))
        assert np.array_equal(masks.allowed_matrix_rect(nq, n, kind, **kw), sq[-nq:])
    # Plain membership check of the causal decode reading.
    got = masks.allowed_matrix_rect(3, 10, masks.CAUSAL)
    for i in range(3):
        assert set(np.nonzero(got[i])[0]) == set(range(0, 10 - 3 + i + 1))


def test_rect_forward_equals_last_rows_of_square_forward():
    r = _rng(13)
    B, H, n, d, v, nq = 1, 2, 50, 6, 5, 7
    Q, K, V = r.normal(size=(B, H, n, d)), r.normal(size=(B, H, n, d)), r.normal(size=(B, H, n, v))
    for kind in (masks.NONE, masks.CAUSAL, masks.WINDOW):
        Y, L = dense.forward(Q, K, V, 0.4, kind, 8)
        Yr, Lr = dense.forward_rect(Q[:, :, -nq:], K, V, 0.4, kind, 8)
        assert _rel(Yr, Y[:, :, -nq:]) <= 1e-15 and _rel(Lr, L[:, :, -nq:]) <= 1e-15


def test_split_merge_is_exact_for_every_split():
    """Summaries of disjoint key chunks merged with the star rule give the
    dense result, whatever the chunks (the split-KV reading of the Forward
    procedure)."""
    r = _rng(14)
    nq, nk, d, v, c = 4, 45, 5, 3, 0.6
    Q, K, V = r.normal(size=(nq, d)), r.normal(size=(nk, d)), r.normal(size=(nk, v))
    allowed = masks.allowed_matrix_rect(nq, nk, masks.CAUSAL)
    Y, L = dense.head_forward(Q, K, V, c, allowed)
    for splits in (1, 2, 3, 7, 45):
        bounds = np.linspace(0, nk, splits + 1).astype(int)
        m = np.full(nq, -np.inf)
        l = np.zeros(nq)
        z = np.zeros((nq, v))
        for a0, a1 in zip(bounds[:-1], bounds[1:]):
            s = c * Q @ K[a0:a1].T
            bm, bl, bz = tiled.block_summary(s, allowed[:, a0:a1], V[a0:a1])
            ne = allowed[:, a0:a1].any(axis=1)
            first = ne & ~np.isfinite(m)
            both = ne & np.isfinite(m)
            m[first], l[first], z[first] = bm[first], bl[first], bz[first]
            if both.any():
                mm, ml, mz = tiled.merge(m[both], l[both], z[both], bm[both], bl[both], bz[both])
                m[both], l[both], z[both] = mm, ml, mz
        assert _rel(z / l[:, None], Y) <= 1e-12 and _rel(m + np.log(l), L) <= 1e-12


# --------------------------------------------------------------------------- #
# Dropout with a replayed mask (oracle.philox and the dropout forms of dense)
# --------------------------------------------------------------------------- #

from oracle import philox  # noqa: E402

DROPOUT_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dropout_cases.json")


def _hex(xs):
    return np.array([int(x, 16) for x in xs], dtype=np.uint32)


def test_philox_known_answer_vectors():
    cases = _load(DROPOUT_GOLDEN)["philox4x32_10"]
    for c in cases:
        got = philox.philox4x32_10(_hex(c["ctr"]), _hex(c["key"]))
        assert np.array_equal(got, _hex(c["out"])), c


def test_dropout_mask_layout_golden():
    c = _load(DROPOUT_GOLDEN)["mask_case"]
    u = philox.random_u16(c["bh"], c["row"] + 1, 8, c["seed"])[c["row"]]
    assert np.array_equal(u, _hex(c["u16"]))
    assert philox.threshold(c["q"]) == c["threshold"]
    assert philox.keep_scale(c["q"]) == c["scale"]
    keep = philox.keep_mask(c["bh"], 1, 8, c["q"], c["seed"])[0]
    assert keep.astype(int).tolist() == c["keep"]


def test_dropout_mask_matches_its_stated_counter_layout():
    """The vectorised mask equals scalar generator calls with the documented
    counter (j // 8, i, bh, 0) and key (seed low, seed high)."""
    seed, bh, rows, cols = 0x1234_5678_9ABC_DEF0, 37, 13, 45
    u = philox.random_u16(bh, rows, cols, seed)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
    for i, j in [(0, 0), (5, 9), (12, 44), (7, 31), (3, 40)]:
        out = philox.philox4x32_10(np.array([j // 8, i, bh, 0], dtype=np.uint32), key)
        w = out[(j % 8) // 2]
        assert u[i, j] == ((int(w) >> (16 * (j % 2))) & 0xFFFF)


def test_dropout_threshold_and_rate():
    assert philox.threshold(0.0) == 0 and philox.keep_scale(0.0) == 1.0
    assert philox.threshold(0.1) == 6554
    assert philox.threshold(0.9999999) == 65535
    with pytest.raises(ValueError):
        philox.threshold(1.0)
    with pytest.raises(ValueError):
        philox.threshold(-0.1)
    # Keep rate over 512 x 512 entries within 5 standard deviations of 1 - t/65536.
    for q in (0.1, 0.5):
        keep = philox.keep_mask(3, 512, 512, q, seed=99)
        p = 1 - philox.threshold(q) / 65536
        sd = math.sqrt(p * (1 - p) / keep.size)
        assert abs(keep.mean() - p) <= 5 * sd
    # Different slices and seeds give different masks.
    a = philox.keep_mask(0, 64, 64, 0.5, 1)
    assert not np.array_equal(a, philox.keep_mask(1, 64, 64, 0.5, 1))
    assert not np.array_equal(a, philox.keep_mask(0, 64, 64, 0.5, 2))


def _drop_case(seed=21, n=5, d=3, v=4, q=0.4):
    r = _rng(seed)
    Q, K, V, G = (r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, v)),
                  r.normal(size=(n, v)))
    allowed = masks.allowed_matrix(n, masks.CAUSAL)
    keep = philox.keep_mask(2, n, n, q, seed=7)
    return Q, K, V, G, allowed, keep, philox.keep_scale(q)


def dropout_pin_failures(fwd, bwd):
    """The dropout pins as one list of failures (used for the planted mistakes)."""
    fails = []
    c = 0.7
    # q = 0 reduces to the plain oracle.
    Q, K, V, G, allowed, _, _ = _drop_case()
    ones = np.ones_like(allowed)
    Y0, L0 = dense.head_forward(Q, K, V, c, allowed)
    Y1, L1 = fwd(Q, K, V, c, allowed, ones, 1.0)
    if _rel(Y1, Y0) > 1e-14 or _rel(L1, L0) > 1e-14:
        fails.append("q0_forward")
    g0 = dense.head_backward(Q, K, V, G, c, allowed)
    g1 = bwd(Q, K, V, G, c, allowed, ones, 1.0)
    if any(_rel(a, b) > 1e-13 for a, b in zip(g1[:3], g0[:3])):
        fails.append("q0_backward")
    # Central finite differences of <G, Y> with the realised mask held fixed.
    Q, K, V, G, allowed, keep, ks = _drop_case()
    grads = bwd(Q, K, V, G, c, allowed, keep, ks)
    for which, X in enumerate((Q, K, V)):
        num = np.zeros_like(X)
        h = 1e-6
        for idx in np.ndindex(X.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            yp = np.sum(G * fwd(*args, c, allowed, keep, ks)[0])
            args[which][idx] -= 2 * h
            ym = np.sum(G * fwd(*args, c, allowed, keep, ks)[0])
            num[idx] = (yp - ym) / (2 * h)
        if _rel(grads[which], num) > 1e-5:
            fails.append(f"fd_{'QKV'[which]}")
    # delta is G . Y with the dropped Y (the identity survives dropout).
    Y, L = fwd(Q, K, V, c, allowed, keep, ks)
    if _rel(grads[3], np.sum(G * Y, axis=1)) > 1e-12:
        fails.append("delta_identity")
    # L is the undropped statistic.
    if _rel(L, dense.head_forward(Q, K, V, c, allowed)[1]) > 1e-14:
        fails.append("L_undropped")
    # Unbiased: the mean of Y over many masks approaches the plain Y.
    n = Q.shape[0]
    acc = np.zeros_like(Y)
    for sd in range(400):
        kp = philox.keep_mask(0, n, n, 0.5, seed=1000 + sd)
        acc += fwd(Q, K, V, c, allowed, kp, philox.keep_scale(0.5))[0]
    if _rel(acc / 400, dense.head_forward(Q, K, V, c, allowed)[0]) > 0.15:
        fails.append("unbiased")
    return fails


def test_dropout_oracle_pins():
    assert dropout_pin_failures(dense.head_forward_dropout, dense.head_backward_dropout) == []


def _dropout_mutant(fault):
    def fwd(Q, K, V, c, allowed, keep, ks):
        s = np.where(allowed, c * (Q @ K.T), -np.inf)
        m = s.max(1)
        e = np.exp(s - m[:, None])
        if fault == "mask_in_sum":
            e_l = e * keep
            l = np.where(e_l.sum(1) > 0, e_l.sum(1), 1.0)
        else:
            l = e.sum(1)
        P = e / l[:, None]
        kk = keep.T if fault == "mask_transposed" else keep
        sc = 1.0 if fault == "no_keep_scale" else ks
        Y = (P * kk * sc) @ V
        return Y, m + np.log(l)

    def bwd(Q, K, V, G, c, allowed, keep, ks):
        s = np.where(allowed, c * (Q @ K.T), -np.inf)
        e = np.exp(s - s.max(1)[:, None])
        P = e / e.sum(1)[:, None]
        xs = keep * ks
        dV = (P if fault == "dV_undropped" else P * xs).T @ G
        dP = G @ V.T
        if fault != "dP_unmasked":
            dP = dP * xs
        delta = (P * dP).sum(1)
        if fault == "delta_undropped":
            delta = (P * (G @ V.T)).sum(1)
        dS = P * (dP - delta[:, None])
        return c * (dS @ K), c * (dS.T @ Q), dV, delta

    return fwd, bwd


DROPOUT_FAULTS = ["mask_in_sum", "mask_transposed", "no_keep_scale", "dV_undropped",
                  "dP_unmasked", "delta_undropped"]


def test_dropout_unfaulted_copy_passes():
    assert dropout_pin_failures(*_dropout_mutant(None)) == []


@pytest.mark.parametrize("fault", DROPOUT_FAULTS)
def test_dropout_planted_mistakes_are_caught(fault):
    assert dropout_pin_failures(*_dropout_mutant(fault)), f"no pin caught {fault}"


def test_batched_dropout_uses_each_heads_own_mask():
    r = _rng(31)
    B, H, n, d = 2, 3, 9, 4
    Q, K, V, G = (r.normal(size=(B, H, n, d)) for _ in range(4))
    Y, L = dense.forward_dropout(Q, K, V, 0.5, masks.CAUSAL, q=0.3, seed=5)
    allowed = masks.allowed_matrix(n, masks.CAUSAL)
    for b in range(B):
        for h in range(H):
            keep = philox.keep_mask(b * H + h, n, n, 0.3, 5)
            y, l = dense.head_forward_dropout(Q[b, h], K[b, h], V[b, h], 0.5, allowed, keep,
                                              philox.keep_scale(0.3))
            assert np.array_equal(Y[b, h], y) and np.array_equal(L[b, h], l)
    g = dense.backward_dropout(Q, K, V, G, 0.5, masks.CAUSAL, q=0.3, seed=5, heads=[4])
    keep = philox.keep_mask(4, n, n, 0.3, 5)
    ref = dense.head_backward_dropout(Q[1, 1], K[1, 1], V[1, 1], G[1, 1], 0.5, allowed, keep,
                                      philox.keep_scale(0.3))
    for a, b_ in zip(g, ref):
        assert np.array_equal(a[0], b_)


# --------------------------------------------------------------------------- #
# Cross-attention, nq != nk (queries aligned to the end of the keys)
# --------------------------------------------------------------------------- #

def test_rect_backward_equals_square_problem_with_leading_rows_silenced():
    """The nq-query problem is the square nk problem whose first nk - nq rows
    get a zero upstream gradient: same dK and dV, dQ of the last nq rows."""
    r = _rng(41)
    B, H, nk, nq, d, v = 1, 2, 40, 13, 5, 6
    Q = r.normal(size=(B, H, nk, d))
    K, V, G = r.normal(size=(B, H, nk, d)), r.normal(size=(B, H, nk, v)), r.normal(size=(B, H, nk, v))
    Gz = G.copy()
    Gz[:, :, : nk - nq] = 0.0
    for kind, w in ((masks.NONE, 0), (masks.CAUSAL, 0), (masks.WINDOW, 7)):
        dQ, dK, dV, _ = dense.backward(Q, K, V, Gz, 0.3, kind, w)
        rq, rk, rv, rd = dense.backward_rect(Q[:, :, -nq:], K, V, G[:, :, -nq:], 0.3, kind, w)
        assert _rel(rk, dK) <= 1e-13 and _rel(rv, dV) <= 1e-13
        assert _rel(rq, dQ[:, :, -nq:]) <= 1e-13
        Y, _ = dense.forward_rect(Q[:, :, -nq:], K, V, 0.3, kind, w)
        assert _rel(rd, np.sum(G[:, :, -nq:] * Y, axis=-1)) <= 1e-12


def test_rect_matches_torch_autograd_with_explicit_mask():
    r = _rng(42)
    nq, nk, d, v, c = 9, 23, 4, 3, 0.45
    Q, K, V, G = (r.normal(size=s) for s in ((nq, d), (nk, d), (nk, v), (nq, v)))
    for kind, w in ((masks.CAUSAL, 0), (masks.WINDOW, 5)):
        allowed = masks.allowed_matrix_rect(nq, nk, kind, w)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        y = torch.nn.functional.scaled_dot_product_attention(
            tq[None], tk[None], tv[None], attn_mask=torch.tensor(allowed)[None], scale=c)[0]
        y.backward(torch.tensor(G))
        Y, L = dense.forward_rect(Q[None, None], K[None, None], V[None, None], c, kind, w)
        dQ, dK, dV, _ = dense.backward_rect(Q[None, None], K[None, None], V[None, None],
                                            G[None, None], c, kind, w)
        assert _rel(Y[0, 0], y.detach().numpy()) <= 1e-13
        assert _rel(dQ[0, 0], tq.grad.numpy()) <= 1e-12
        assert _rel(dK[0, 0], tk.grad.numpy()) <= 1e-12
        assert _rel(dV[0, 0], tv.grad.numpy()) <= 1e-12


def test_rect_rows_before_every_key_are_empty_and_inert():
    """nq > nk under the causal mask: the first nq - nk queries precede every key.
    Their Y, dQ and delta are 0, L is -inf, and the other rows' gradients are
    those of the problem without them."""
    r = _rng(43)
    nq, nk, d, v = 10, 6, 3, 4
    Q, K, V, G = (r.normal(size=(1, 1) + s) for s in ((nq, d), (nk, d), (nk, v), (nq, v)))
    Y, L = dense.forward_rect(Q, K, V, 0.5, masks.CAUSAL)
    dQ, dK, dV, dl = dense.backward_rect(Q, K, V, G, 0.5, masks.CAUSAL)
    e = nq - nk
    assert np.all(Y[0, 0, :e] == 0) and np.all(np.isneginf(L[0, 0, :e]))
    assert np.all(dQ[0, 0, :e] == 0) and np.all(dl[0, 0, :e] == 0)
    sq = dense.backward(Q[:, :, e:], K, V, G[:, :, e:], 0.5, masks.CAUSAL)
    assert _rel(dK, sq[1]) <= 1e-14 and _rel(dV, sq[2]) <= 1e-14
    assert _rel(dQ[:, :, e:], sq[0]) <= 1e-14


def test_rect_backward_finite_differences():
    r = _rng(44)
    nq, nk, d, v, c = 3, 5, 2, 3, 0.8
    Q, K, V, G = (r.normal(size=(1, 1) + s) for s in ((nq, d), (nk, d), (nk, v), (nq, v)))
    grads = dense.backward_rect(Q, K, V, G, c, masks.CAUSAL)
    for which, X in enumerate((Q, K, V)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += 1e-6
            yp = np.sum(G * dense.forward_rect(*args, c, masks.CAUSAL)[0])
            args[which][idx] -= 2e-6
            ym = np.sum(G * dense.forward_rect(*args, c, masks.CAUSAL)[0])
            num[idx] = (yp - ym) / 2e-6
        assert _rel(grads[which], num) <= 1e-5


def test_rect_dropout_reduces_to_square_dropout_and_to_plain():
    """nq == nk with dropout is the square dropout oracle; q = 0 is forward_rect."""
    r = _rng(45)
    B, H, n, d = 1, 2, 11, 4
    Q, K, V, G = (r.normal(size=(B, H, n, d)) for _ in range(4))
    for kind in (masks.NONE, masks.CAUSAL):
        Y1, L1 = dense.forward_rect(Q, K, V, 0.6, kind, dropout=(0.3, 9))
        Y2, L2 = dense.forward_dropout(Q, K, V, 0.6, kind, q=0.3, seed=9)
        assert _rel(Y1, Y2) <= 1e-15 and _rel(L1, L2) <= 1e-15
        g1 = dense.backward_rect(Q, K, V, G, 0.6, kind, dropout=(0.3, 9))
        g2 = dense.backward_dropout(Q, K, V, G, 0.6, kind, q=0.3, seed=9)
        for a, b in zip(g1, g2):
            assert _rel(a, b) <= 1e-14
        Y3, _ = dense.forward_rect(Q, K, V, 0.6, kind, dropout=(0.0, 9))
        assert _rel(Y3, dense.forward_rect(Q, K, V, 0.6, kind)[0]) <= 1e-15

"""Dense float64 attention: the plain definition (oracle; test infrastructure only).

The method computes, up to rounding order, exactly the dense softmax attention
("Exact tiled softmax attention with block-recomputed vector-Jacobian
products", Inputs: "exact real arithmetic"; "txf-modern-flash-attention",
Constraints: the same output for every block size).  So the oracle is that
definition written out, one (batch, head) slice at a time, in float64:

  s_ij = c * <Q_i, K_j>            for j in A_i, and -inf otherwise
  m_i  = max_j s_ij,   l_i = sum_j exp(s_ij - m_i),   p_ij = exp(s_ij - m_i) / l_i
  Y    = P V,          L_i = m_i + ln l_i           (the retained statistic)

and the vector-Jacobian product for an upstream G = dY with the statistics held
fixed (Reverse procedure of the same page; "python-flash-attention-online-
softmax-block-recompute", The fix, item 2):

  dV = P^T G,   dP = G V^T,   delta_i = sum_j p_ij dP_ij,
  dS = P o (dP - delta),   dQ = c dS K,   dK = c dS^T Q.

delta is formed from P and dP, NOT as G_i . Y_i, so that the identity
delta_i = G_i . Y_i (HarshvardhanJ/FlashAttention, backward section) stays a
real check on it.  Rows of S are always formed whole; rows are only processed
in groups to bound memory.  No online recurrence appears here.
"""
import numpy as np

from .masks import allowed_matrix

ROW_GROUP = 1024


def _check_rows(allowed):
    if not allowed.any(axis=1).all():
        raise ValueError("every allowed-key set A_i must be nonempty")


def head_forward(Q, K, V, c, allowed):
    """One head. Q [n,d], K [n,d], V [n,v] float64; allowed [n,n] bool -> (Y, L)."""
    _check_rows(allowed)
    n = Q.shape[0]
    Y = np.empty((n, V.shape[1]))
    L = np.empty(n)
    for r0 in range(0, n, ROW_GROUP):
        r1 = min(n, r0 + ROW_GROUP)
        s = c * (Q[r0:r1] @ K.T)
        s = np.where(allowed[r0:r1], s, -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=1)
        Y[r0:r1] = (e / l[:, None]) @ V
        L[r0:r1] = m + np.log(l)
    return Y, L


def head_backward(Q, K, V, G, c, allowed):
    """One head. Returns (dQ, dK, dV, delta) for the upstream G [n,v]."""
    _check_rows(allowed)
    n = Q.shape[0]
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    delta = np.empty(n)
    for r0 in range(0, n, ROW_GROUP):
        r1 = min(n, r0 + ROW_GROUP)
        s = c * (Q[r0:r1] @ K.T)
        s = np.where(allowed[r0:r1], s, -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        P = e / e.sum(axis=1)[:, None]
        Gr = G[r0:r1]
        dV += P.T @ Gr
        dP = Gr @ V.T
        dl = (P * dP).sum(axis=1)
        dS = P * (dP - dl[:, None])
        dQ[r0:r1] = c * (dS @ K)
        dK += c * (dS.T @ Q[r0:r1])
        delta[r0:r1] = dl
    return dQ, dK, dV, delta


def _heads(x):
    """View [..., n, f] as [heads, n, f]."""
    return x.reshape(-1, x.shape[-2], x.shape[-1])


def forward(Q, K, V, c, mask_kind, window=0, bitmask=None, heads=None):
    """Batched forward over [B,H,n,*] float64 arrays -> (Y [B,H,n,v], L [B,H,n]).

    ``heads`` (optional) is a list of flat (b*H + h) indices; only those heads
    are computed and the result has a leading axis of len(heads).
    """
    n = Q.shape[-2]
    allowed = allowed_matrix(n, mask_kind, window, bitmask)
    q, k, vv = _heads(Q), _heads(K), _heads(V)
    idx = range(q.shape[0]) if heads is None else heads
    out = [head_forward(q[h], k[h], vv[h], c, allowed) for h in idx]
    Y = np.stack([o[0] for o in out])
    L = np.stack([o[1] for o in out])
    if heads is None:
        Y = Y.reshape(V.shape[:-2] + Y.shape[-2:])
        L = L.reshape(Q.shape[:-1])
    return Y, L


def backward(Q, K, V, G, c, mask_kind, window=0, bitmask=None, heads=None):
    """Batched reverse pass -> (dQ, dK, dV, delta), same layout rules as ``forward``."""
    n = Q.shape[-2]
    allowed = allowed_matrix(n, mask_kind, window, bitmask)
    q, k, vv, g = _heads(Q), _heads(K), _heads(V), _heads(G)
    idx = range(q.shape[0]) if heads is None else heads
    out = [head_backward(q[h], k[h], vv[h], g[h], c, allowed) for h in idx]
    res = [np.stack([o[t] for o in out]) for t in range(4)]
    if heads is None:
        res[0] = res[0].reshape(Q.shape)
        res[1] = res[1].reshape(K.shape)
        res[2] = res[2].reshape(V.shape)
        res[3] = res[3].reshape(Q.shape[:-1])
    return tuple(res)


def row_forward(Q, K, V, c, allowed_row, i):
    """A single output row Y_i and L_i of one head (for sampled full-size checks)."""
    if not allowed_row.any():
        raise ValueError("every allowed-key set A_i must be nonempty")
    s = np.where(allowed_row, c * (K @ Q[i]), -np.inf)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return (e @ V) / l, m + np.log(l)


def row_backward(Q, K, V, G, c, allowed_row, i):
    """dQ_i and delta_i of one head's row i (for sampled full-size checks).

    The Reverse procedure of "Exact tiled softmax attention with block-recomputed
    vector-Jacobian products" restricted to one query row: p_ij from the row's
    own scores, dP_ij = G_i . V_j, delta_i = sum_j p_ij dP_ij (formed this way,
    not as G_i . Y_i), gamma_ij = p_ij (dP_ij - delta_i), dQ_i = c sum_j gamma_ij K_j.
    """
    if not allowed_row.any():
        raise ValueError("every allowed-key set A_i must be nonempty")
    s = np.where(allowed_row, c * (K @ Q[i]), -np.inf)
    e = np.exp(s - s.max())
    p = e / e.sum()
    dP = V @ G[i]
    delta = p @ dP
    gamma = p * (dP - delta)
    return c * (gamma @ K), delta


def _rect_keep(h, nq, nk, dropout):
    from .philox import keep_mask, keep_scale
    q, seed = dropout
    return keep_mask(h, nq, nk, q, seed), keep_scale(q)


def forward_rect(Q, K, V, c, mask_kind, window=0, bitmask=None, dropout=None):
    """Forward for nq queries against nk keys ([B,H,nq,d], [B,H,nk,d], [B,H,nk,v]),
    queries aligned to the end of the keys (masks.allowed_matrix_rect).
    Rows whose allowed set is empty get Y_i = 0 and L_i = -inf (the library's
    convention for inputs outside the method's domain).  ``dropout`` = (q, seed)
    applies the replayed keep mask of flat head h (philox.keep_mask(h, nq, nk))."""
    from .masks import allowed_matrix_rect
    nq, nk = Q.shape[-2], K.shape[-2]
    allowed = allowed_matrix_rect(nq, nk, mask_kind, window, bitmask)
    q, k, vv = _heads(Q), _heads(K), _heads(V)
    Y = np.zeros((q.shape[0], nq, vv.shape[-1]))
    L = np.full((q.shape[0], nq), -np.inf)
    rows = allowed.any(axis=1)
    for h in range(q.shape[0]):
        if rows.any():
            if dropout is None:
                y, l = head_forward(q[h][rows], k[h], vv[h], c, allowed[rows])
            else:
                keep, ks = _rect_keep(h, nq, nk, dropout)
                y, l = head_forward_dropout(q[h][rows], k[h], vv[h], c, allowed[rows],
                                            keep[rows], ks)
            Y[h][rows] = y
            L[h][rows] = l
    return Y.reshape(V.shape[:-2] + (nq, V.shape[-1])), L.reshape(Q.shape[:-1])


# --------------------------------------------------------------------------- #
# Dropout with a replayed mask ("Exact tiled softmax attention with block-
# recomputed vector-Jacobian products", Reverse procedure, closing remark: the
# reverse pass must use the forward pass's realised mask).  Reading: the mask
# xi acts on the normalised probabilities, kept entries scaled by
# s = 1 / (1 - q):
#
#   Y_i = sum_j p_ij xi_ij s V_j,     L_i = m_i + ln l_i  (undropped statistics)
#
# whose vector-Jacobian product for G = dY is
#
#   dV_j += p_ij xi_ij s G_i,   dP_ij = xi_ij s G_i . V_j,
#   delta_i = sum_j p_ij dP_ij  (= G_i . Y_i),   gamma_ij = p_ij (dP_ij - delta_i),
#   dQ_i += c gamma_ij K_j,     dK_j += c gamma_ij Q_i.
# --------------------------------------------------------------------------- #

def head_forward_dropout(Q, K, V, c, allowed, keep, kscale):
    """One head with the realised keep mask ``keep`` [n,n] and factor ``kscale``."""
    _check_rows(allowed)
    n = Q.shape[0]
    Y = np.empty((n, V.shape[1]))
    L = np.empty(n)
    for r0 in range(0, n, ROW_GROUP):
        r1 = min(n, r0 + ROW_GROUP)
        s = np.where(allowed[r0:r1], c * (Q[r0:r1] @ K.T), -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=1)
        P = e / l[:, None]
        Y[r0:r1] = (P * keep[r0:r1] * kscale) @ V
        L[r0:r1] = m + np.log(l)
    return Y, L


def head_backward_dropout(Q, K, V, G, c, allowed, keep, kscale):
    """One head: (dQ, dK, dV, delta) with the same realised mask as the forward."""
    _check_rows(allowed)
    n = Q.shape[0]
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    delta = np.empty(n)
    for r0 in range(0, n, ROW_GROUP):
        r1 = min(n, r0 + ROW_GROUP)
        s = np.where(allowed[r0:r1], c * (Q[r0:r1] @ K.T), -np.inf)
        e = np.exp(s - s.max(axis=1)[:, None])
        P = e / e.sum(axis=1)[:, None]
        xs = keep[r0:r1] * kscale
        Gr = G[r0:r1]
        dV += (P * xs).T @ Gr
        dP = (Gr @ V.T) * xs
        dl = (P * dP).sum(axis=1)
        dS = P * (dP - dl[:, None])
        dQ[r0:r1] = c * (dS @ K)
        dK += c * (dS.T @ Q[r0:r1])
        delta[r0:r1] = dl
    return dQ, dK, dV, delta


def _dropout_heads(Q, n, q, seed, idx):
    from .philox import keep_mask, keep_scale
    return [keep_mask(h, n, n, q, seed) for h in idx], keep_scale(q)


def forward_dropout(Q, K, V, c, mask_kind, window=0, bitmask=None, q=0.0, seed=0, heads=None):
    """Batched dropout forward; the mask of flat head h is philox.keep_mask(h, ...)."""
    n = Q.shape[-2]
    allowed = allowed_matrix(n, mask_kind, window, bitmask)
    qh, kh, vh = _heads(Q), _heads(K), _heads(V)
    idx = list(range(qh.shape[0])) if heads is None else list(heads)
    keeps, ks = _dropout_heads(Q, n, q, seed, idx)
    out = [head_forward_dropout(qh[h], kh[h], vh[h], c, allowed, kp, ks)
           for h, kp in zip(idx, keeps)]
    Y = np.stack([o[0] for o in out])
    L = np.stack([o[1] for o in out])
    if heads is None:
        Y = Y.reshape(V.shape[:-2] + Y.shape[-2:])
        L = L.reshape(Q.shape[:-1])
    return Y, L


def backward_dropout(Q, K, V, G, c, mask_kind, window=0, bitmask=None, q=0.0, seed=0,
                     heads=None):
    """Batched dropout reverse pass -> (dQ, dK, dV, delta)."""
    n = Q.shape[-2]
    allowed = allowed_matrix(n, mask_kind, window, bitmask)
    qh, kh, vh, gh = _heads(Q), _heads(K), _heads(V), _heads(G)
    idx = list(range(qh.shape[0])) if heads is None else list(heads)
    keeps, ks = _dropout_heads(Q, n, q, seed, idx)
    out = [head_backward_dropout(qh[h], kh[h], vh[h], gh[h], c, allowed, kp, ks)
           for h, kp in zip(idx, keeps)]
    res = [np.stack([o[t] for o in out]) for t in range(4)]
    if heads is None:
        res[0] = res[0].reshape(Q.shape)
        res[1] = res[1].reshape(K.shape)
        res[2] = res[2].reshape(V.shape)
        res[3] = res[3].reshape(Q.shape[:-1])
    return tuple(res)


def backward_rect(Q, K, V, G, c, mask_kind, window=0, bitmask=None, dropout=None):
    """Reverse pass for nq queries against nk keys (``forward_rect``'s alignment):
    -> (dQ [..,nq,d], dK [..,nk,d], dV [..,nk,v], delta [..,nq]).  Rows whose
    allowed set is empty contribute nothing (dQ_i = 0, delta_i = 0).
    ``dropout`` as for ``forward_rect``."""
    from .masks import allowed_matrix_rect
    nq, nk = Q.shape[-2], K.shape[-2]
    allowed = allowed_matrix_rect(nq, nk, mask_kind, window, bitmask)
    q, k, vv, g = _heads(Q), _heads(K), _heads(V), _heads(G)
    rows = allowed.any(axis=1)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(vv)
    delta = np.zeros((q.shape[0], nq))
    for h in range(q.shape[0]):
        if rows.any():
            if dropout is None:
                a, b, cc, dl = head_backward(q[h][rows], k[h], vv[h], g[h][rows], c,
                                             allowed[rows])
            else:
                keep, ks = _rect_keep(h, nq, nk, dropout)
                a, b, cc, dl = head_backward_dropout(q[h][rows], k[h], vv[h], g[h][rows], c,
                                                     allowed[rows], keep[rows], ks)
            dQ[h][rows] = a
            dK[h] = b
            dV[h] = cc
            delta[h][rows] = dl
    return (dQ.reshape(Q.shape), dK.reshape(K.shape), dV.reshape(V.shape),
            delta.reshape(Q.shape[:-1]))

"""The pages' block procedures in float64 (oracle; test infrastructure only).

These are not what the parity tests compare the GPU against (that is
``dense``); they restate the block algorithms of the pages so that the tests
can pin ``dense`` to them: identical results for every key-block size b.

Block sets, from "Exact tiled softmax attention with block-recomputed
vector-Jacobian products", Inputs: J_t = {(t-1)b+1 .. min(tb, n)} (here
0-indexed: keys t*b .. min((t+1)*b, n) - 1).

Summary of a nonempty key set I for row i (the page's Sigma_i(I); its body was
lost from the page, and this is the reading that agrees with the page's own
Y_i = z_i / l_i and p_ij = exp(s_ij - m_i) / l_i, and with the running-max
rule of "txf-modern-flash-attention", Constraints and Hints):

  Sigma_i(I) = (m, l, z),  m = max_{j in I} s_ij,
               l = sum_{j in I} exp(s_ij - m),   z = sum_{j in I} exp(s_ij - m) V_j

Merge (the page's star):  (m1,l1,z1) * (m2,l2,z2) = (M, a1 l1 + a2 l2, a1 z1 + a2 z2)
with M = max(m1, m2), a1 = exp(m1 - M), a2 = exp(m2 - M).  The empty summary
"bottom" is represented by a per-row flag.

Row operations are applied to all rows of a block at once with numpy; each
row still follows the per-row procedure exactly (its own I, skip, copy or
merge).
"""
import numpy as np


def key_blocks(n, b):
    """The key blocks J_t as (start, stop) pairs, the last one possibly shorter."""
    return [(t, min(t + b, n)) for t in range(0, n, b)]


def block_summary(s_blk, allowed_blk, V_blk):
    """Sigma_i(I) for every row at once; rows with I empty get (-inf, 0, 0)."""
    s = np.where(allowed_blk, s_blk, -np.inf)
    m = s.max(axis=1)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(allowed_blk, np.exp(s - safe_m[:, None]), 0.0)
    return m, e.sum(axis=1), e @ V_blk


def merge(m1, l1, z1, m2, l2, z2):
    """The star merge of two summaries (both nonempty)."""
    M = np.maximum(m1, m2)
    a1 = np.exp(m1 - M)
    a2 = np.exp(m2 - M)
    return M, a1 * l1 + a2 * l2, a1[:, None] * z1 + a2[:, None] * z2


def summary_forward(Q, K, V, c, allowed, b):
    """Forward procedure of the page (summary / skip / copy-or-merge), block size b.

    Returns (Y, m, l, L) for one head, L = m + ln l.
    """
    n = Q.shape[0]
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    z = np.zeros((n, V.shape[1]))
    have = np.zeros(n, dtype=bool)                  # False: summary is "bottom"
    for j0, j1 in key_blocks(n, b):
        nonempty = allowed[:, j0:j1].any(axis=1)    # I = J_t intersect A_i
        if not nonempty.any():
            continue
        s_blk = c * (Q @ K[j0:j1].T)
        bm, bl, bz = block_summary(s_blk, allowed[:, j0:j1], V[j0:j1])
        copy = nonempty & ~have
        mix = nonempty & have
        m[copy], l[copy], z[copy] = bm[copy], bl[copy], bz[copy]
        if mix.any():
            mm, ml, mz = merge(m[mix], l[mix], z[mix], bm[mix], bl[mix], bz[mix])
            m[mix], l[mix], z[mix] = mm, ml, mz
        have |= nonempty
    if not have.all():
        raise ValueError("every allowed-key set A_i must be nonempty")
    Y = z / l[:, None]
    return Y, m, l, m + np.log(l)


def online_forward(Q, K, V, c, allowed, b):
    """The running-statistics recurrence of the hint code ("txf-modern-flash-
    attention", Hints; "What Ordinary Autograd Saves ...", The implementation
    under test): running max, correction exp(old - new) applied to the running
    sum and output, normalisation once at the end.  A correction taken from a
    running max of -inf is 0 (that page's empty-key guard).  Returns (Y, L)."""
    n = Q.shape[0]
    run_max = np.full(n, -np.inf)
    run_sum = np.zeros(n)
    run_out = np.zeros((n, V.shape[1]))
    for j0, j1 in key_blocks(n, b):
        s = np.where(allowed[:, j0:j1], c * (Q @ K[j0:j1].T), -np.inf)
        new_max = np.maximum(run_max, s.max(axis=1))
        ref = np.where(np.isfinite(new_max), new_max, 0.0)
        corr = np.where(np.isneginf(run_max), 0.0, np.exp(run_max - ref))
        probs = np.exp(s - ref[:, None])
        run_sum = corr * run_sum + probs.sum(axis=1)
        run_out = corr[:, None] * run_out + probs @ V[j0:j1]
        run_max = new_max
    return run_out / run_sum[:, None], run_max + np.log(run_sum)


def recompute_backward(Q, K, V, G, Y, m, l, c, allowed, b):
    """Reverse procedure of the page, block by block, with frozen (m, l):

    delta_i = sum_a G_ia Y_ia; for every block J_t and j in J_t intersect A_i:
    p_ij = exp(s_ij - m_i) / l_i, gamma_ij = p_ij (sum_a G_ia V_ja - delta_i),
    dQ_i += c gamma_ij K_j, dK_j += c gamma_ij Q_i, dV_j += p_ij G_i.
    Returns (dQ, dK, dV, delta).
    """
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    delta = (G * Y).sum(axis=1)
    for j0, j1 in key_blocks(Q.shape[0], b):
        a = allowed[:, j0:j1]
        if not a.any():
            continue
        s = c * (Q @ K[j0:j1].T)
        p = np.where(a, np.exp(s - m[:, None]) / l[:, None], 0.0)
        gamma = p * (G @ V[j0:j1].T - delta[:, None])
        dQ += c * (gamma @ K[j0:j1])
        dK[j0:j1] += c * (gamma.T @ Q)
        dV[j0:j1] += p.T @ G
    return dQ, dK, dV, delta

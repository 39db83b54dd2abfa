"""Allowed-key sets A_i (oracle; test infrastructure only).

The pages fix only that each A_i is a nonempty subset of the keys and that the
caller owns the mask storage ("Exact tiled softmax attention ...", Inputs).
The four concrete kinds below are the readings used throughout, 0-indexed:

  none     A_i = {0 .. n-1}
  causal   A_i = {0 .. i}                       (j <= i)
  window   A_i = {max(0, i-w+1) .. i}           (w keys ending at the diagonal)
  bitmask  j in A_i  iff  bit (j mod 32) of word [i*ceil(n/32) + j div 32] is 1

For nq queries against nk keys (a decode step, a chunk of new queries), query
i sits at absolute position i + (nk - nq): the queries are the LAST nq
positions of the key sequence, so causal reads j <= i + nk - nq and the window
{i + nk - nq - w + 1 .. i + nk - nq}; bit rows are [nq][ceil(nk/32)].  With
nq = nk this is the square reading above.

Written as explicit membership tests over index grids; nothing is shared with
the kernels' tile classification.
"""
import numpy as np

NONE, CAUSAL, WINDOW, BITMASK = 0, 1, 2, 3


def allowed_matrix(n, mask_kind, window=0, bitmask=None):
    """Boolean [n, n] matrix: entry (i, j) is True when key j is in A_i."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    if mask_kind == NONE:
        return np.ones((n, n), dtype=bool)
    if mask_kind == CAUSAL:
        return j <= i
    if mask_kind == WINDOW:
        if window < 1:
            raise ValueError("window must be >= 1")
        return (j <= i) & (j >= i - window + 1)
    if mask_kind == BITMASK:
        words = np.asarray(bitmask, dtype=np.uint32).reshape(n, (n + 31) // 32)
        word = words[np.arange(n)[:, None], np.arange(n)[None, :] // 32]
        bit = (word >> (np.arange(n)[None, :] % 32).astype(np.uint32)) & np.uint32(1)
        return bit.astype(bool)
    raise ValueError(f"unknown mask kind {mask_kind}")


def allowed_matrix_rect(nq, nk, mask_kind, window=0, bitmask=None):
    """Boolean [nq, nk]: key j in A_i for queries aligned to the end of the keys."""
    off = nk - nq
    i = np.arange(nq)[:, None] + off
    j = np.arange(nk)[None, :]
    if mask_kind == NONE:
        return np.ones((nq, nk), dtype=bool)
    if mask_kind == CAUSAL:
        return j <= i
    if mask_kind == WINDOW:
        if window < 1:
            raise ValueError("window must be >= 1")
        return (j <= i) & (j >= i - window + 1)
    if mask_kind == BITMASK:
        words = np.asarray(bitmask, dtype=np.uint32).reshape(nq, (nk + 31) // 32)
        word = words[np.arange(nq)[:, None], np.arange(nk)[None, :] // 32]
        bit = (word >> (np.arange(nk)[None, :] % 32).astype(np.uint32)) & np.uint32(1)
        return bit.astype(bool)
    raise ValueError(f"unknown mask kind {mask_kind}")

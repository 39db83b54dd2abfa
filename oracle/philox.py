"""Counter-based random bits and the dropout keep mask (oracle; test infrastructure only).

"Exact tiled softmax attention with block-recomputed vector-Jacobian
products", Reverse procedure (closing remark): the base method has no dropout,
and a dropout extension must use, in the reverse pass, exactly the dropout mask
that the forward pass realised.  A counter-based generator gives that without
storing the mask: the keep decision of entry (b, h, i, j) is a pure function of
(seed, b*H + h, i, j), recomputed wherever it is needed.

Generator: Philox-4x32 with 10 rounds, as published by Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011).  A counter of
four 32-bit words and a key of two are mapped to four 32-bit outputs by ten
rounds of

    (hi0, lo0) = M0 * c0,  (hi1, lo1) = M1 * c2          (64-bit products)
    c = (hi1 ^ c1 ^ k0,  lo1,  hi0 ^ c3 ^ k1,  lo0)

with the key advanced by the Weyl constants (W0, W1) between rounds.

Mask layout (this library's own definition; the CUDA path implements the same
definition separately):
    counter = (j // 8, i, bh, 0),  key = (seed mod 2^32, seed div 2^32)
    output word w = (j % 8) // 2, half h = j % 2:  u_ij = (word >> 16 h) & 0xFFFF
    keep_ij  <=>  u_ij >= t,   t = min(65535, floor(q * 65536 + 1/2))
with the drop probability q read as a float32.  The realised drop rate is
t / 65536, and the kept entries are scaled by 65536 / (65536 - t).
"""
import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """ctr uint32 [..., 4], key uint32 [..., 2] (broadcast against ctr) -> uint32 [..., 4]."""
    ctr = np.asarray(ctr, dtype=np.uint32)
    key = np.asarray(key, dtype=np.uint32)
    c0, c1, c2, c3 = (ctr[..., k].astype(np.uint64) for k in range(4))
    k0 = key[..., 0].astype(np.uint64)
    k1 = key[..., 1].astype(np.uint64)
    for _ in range(10):
        p0 = np.uint64(M0) * c0          # < 2^64: exact in uint64
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(W0)) & _MASK32
        k1 = (k1 + np.uint64(W1)) & _MASK32
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def threshold(q):
    """The 16-bit drop threshold t of a drop probability q in [0, 1) (read as float32)."""
    q32 = float(np.float32(q))
    if not (0.0 <= q32 < 1.0):
        raise ValueError("the drop probability must lie in [0, 1)")
    return min(65535, int(np.floor(q32 * 65536.0 + 0.5)))


def keep_scale(q):
    """Factor 1 / (1 - t/65536) applied to kept entries."""
    return 65536.0 / (65536 - threshold(q))


def random_u16(bh, rows, cols, seed):
    """The 16-bit values u_ij for rows 0..rows-1 and keys 0..cols-1 of slice bh."""
    nb = (cols + 7) // 8
    i = np.arange(rows, dtype=np.uint32)
    jb = np.arange(nb, dtype=np.uint32)
    ctr = np.zeros((rows, nb, 4), dtype=np.uint32)
    ctr[..., 0] = jb[None, :]
    ctr[..., 1] = i[:, None]
    ctr[..., 2] = np.uint32(bh)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint32)
    out = philox4x32_10(ctr, key)                          # [rows, nb, 4]
    u = np.empty((rows, nb, 8), dtype=np.uint32)
    u[..., 0::2] = out & np.uint32(0xFFFF)                 # j % 2 == 0: low half
    u[..., 1::2] = out >> np.uint32(16)                    # j % 2 == 1: high half
    return u.reshape(rows, nb * 8)[:, :cols]


def keep_mask(bh, rows, cols, q, seed):
    """Boolean keep mask [rows, cols] of slice bh (all True when t = 0)."""
    t = threshold(q)
    return random_u16(bh, rows, cols, seed) >= t

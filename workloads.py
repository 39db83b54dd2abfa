"""Seeded synthetic inputs for exact masked attention.

This module only draws random numbers and packs the allowed-key mask into the
bit-row format that both the CUDA library and the oracle read.  It holds none
of the attention arithmetic, so both sides of every parity test can take their
inputs from here without sharing any of the method.

Recipe (same for every workload):
  * one CPU ``torch.Generator`` seeded with ``seed``;
  * fp32 ``randn`` drawn in the order Q, K, V, dY, then the mask;
  * Q and K multiplied by ``qk_gain`` (1.5 for the peaked-row workload), the
    self-attention variant draws a single X with standard deviation 0.5;
  * cast to the workload dtype (bf16 rounds to nearest even); the oracle then
    gets the rounded values upcast to float64, which is exact.
  * the random bitmask allows each key with probability ``p_allow`` and always
    allows the diagonal, so every allowed-key set is nonempty.

Bitmask format: row i of the mask is ``W = ceil(n/32)`` uint32 words; key j
is allowed for query i when bit ``j % 32`` of word ``i*W + j//32`` is set.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BITMASK = 0, 1, 2, 3
MASK_KINDS = {"none": MASK_NONE, "causal": MASK_CAUSAL,
              "window": MASK_WINDOW, "bitmask": MASK_BITMASK}

SEED_BASE = 20261200


@dataclass
class Workload:
    """Shape, dtype, mask and value recipe of one synthetic attention problem."""
    name: str
    B: int
    H: int
    n: int
    d: int
    v: int
    dtype: str                 # "f32" or "bf16"
    mask: str                  # "none" | "causal" | "window" | "bitmask"
    scale: float
    window: int = 0
    qk_gain: float = 1.0
    p_allow: float = 0.3
    self_attention: bool = False
    seed: int = SEED_BASE
    extra: dict = field(default_factory=dict)
    nk: int = 0                # keys (0: n, self-attention shapes); queries sit at the end

    @property
    def n_keys(self) -> int:
        return self.nk or self.n

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def mask_kind(self) -> int:
        return MASK_KINDS[self.mask]

    def allowed_pairs_per_head(self) -> int:
        """|A| = sum_i |A_i| for the arithmetic masks (bitmask: unknown here); query
        i sits at position i + nk - n, so it sees min(nk, i + nk - n + 1) keys
        under the causal mask and at most ``window`` of them under the window."""
        n, nk = self.n, self.n_keys
        if self.mask == "none":
            return n * nk
        off = nk - n
        if self.mask == "causal":
            return sum(max(0, min(nk, i + off + 1)) for i in range(n))
        if self.mask == "window":
            return sum(max(0, min(nk, i + off + 1, self.window)) for i in range(n))
        raise ValueError("bitmask pair count depends on the drawn mask")


def workload(k: int, variant: str = "") -> Workload:
    """The five benchmark-shaped workloads, numbered 1..5.

    1  single head, n=256, d=v=64, fp32, scale 1/8; variants "none", "causal",
       "self" (Q=K=V=X, X ~ N(0, 0.25), scale 1, full mask)
    2  B=8, H=16, n=2048, d=v=64, bf16, scale 1/8, full mask
    3  B=4, H=32, n=4096, d=v=128, bf16, scale 1/sqrt(128), causal
    4  B=1, H=16, n=16384, d=v=128, bf16, Q,K x1.5, causal or "window" (1024)
    5  B=2, H=8, n=1000, d=80, v=96, fp32 or "bf16", scale 0.1, random bitmask
    """
    seed = SEED_BASE + k
    if k == 1:
        if variant == "self":
            return Workload("attn-n256-d64-f32-self", 1, 1, 256, 64, 64, "f32", "none",
                            1.0, self_attention=True, seed=seed)
        mask = variant or "causal"
        return Workload(f"attn-n256-d64-f32-{mask}", 1, 1, 256, 64, 64, "f32", mask,
                        1.0 / 8.0, seed=seed)
    if k == 2:
        return Workload("attn-b8h16-n2048-d64-bf16-full", 8, 16, 2048, 64, 64, "bf16",
                        "none", 1.0 / 8.0, seed=seed)
    if k == 3:
        return Workload("attn-b4h32-n4096-d128-bf16-causal", 4, 32, 4096, 128, 128, "bf16",
                        "causal", 1.0 / math.sqrt(128.0), seed=seed)
    if k == 4:
        if variant == "window":
            return Workload("attn-b1h16-n16384-d128-bf16-window1024", 1, 16, 16384, 128, 128,
                            "bf16", "window", 1.0 / math.sqrt(128.0), window=1024,
                            qk_gain=1.5, seed=seed)
        return Workload("attn-b1h16-n16384-d128-bf16-causal", 1, 16, 16384, 128, 128, "bf16",
                        "causal", 1.0 / math.sqrt(128.0), qk_gain=1.5, seed=seed)
    if k == 5:
        dt = "bf16" if variant == "bf16" else "f32"
        return Workload(f"attn-b2h8-n1000-d80-v96-{dt}-bitmask", 2, 8, 1000, 80, 96, dt,
                        "bitmask", 0.1, p_allow=0.3, seed=seed)
    raise ValueError(f"no workload {k}")


def pack_bitmask(allowed: np.ndarray) -> np.ndarray:
    """Pack a boolean [rows, cols] allowed matrix into uint32 bit rows
    [rows, ceil(cols/32)] (bit j % 32 of word j // 32 is key j)."""
    rows, cols = allowed.shape
    W = (cols + 31) // 32
    padded = np.zeros((rows, W * 32), dtype=bool)
    padded[:, :cols] = allowed
    bits = padded.reshape(rows, W, 32).astype(np.uint64)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (bits * weights).sum(axis=2).astype(np.uint32)


@dataclass
class Inputs:
    """CPU tensors of one problem, in the workload dtype, plus the mask words."""
    Q: torch.Tensor
    K: torch.Tensor
    V: torch.Tensor
    dY: torch.Tensor
    bitmask: np.ndarray | None   # uint32 [n, ceil(n/32)] or None

    def as_f64(self):
        """Exact float64 numpy copies of (Q, K, V, dY) for the oracle."""
        return tuple(t.to(torch.float64).numpy() for t in (self.Q, self.K, self.V, self.dY))


def make_inputs(w: Workload, heads: int | None = None) -> Inputs:
    """Draw the seeded inputs of workload ``w``.

    ``heads`` limits the draw to the first ``heads`` (batch*head) slices; since
    every head is drawn as one contiguous block of the same stream this is NOT
    the same numbers as the full draw sliced, so callers that compare against a
    full-size run must draw the full size and slice instead.
    """
    B, H = (w.B, w.H) if heads is None else (1, heads)
    if w.n_keys != w.n:  # cross-attention: the decode-shape generator with dY
        Q, K, V, dY, bm = make_decode_inputs(B, H, w.n, w.n_keys, w.d, w.v, w.dtype, w.mask,
                                             seed=w.seed, p_allow=w.p_allow, with_dy=True)
        return Inputs(Q, K, V, dY, bm)
    g = torch.Generator().manual_seed(w.seed)
    n, d, v = w.n, w.d, w.v
    if w.self_attention:
        X = 0.5 * torch.randn(B, H, n, d, generator=g)
        dY = torch.randn(B, H, n, d, generator=g)
        X = X.to(w.torch_dtype)
        Q = K = V = X
        dY = dY.to(w.torch_dtype)
    else:
        Q = torch.randn(B, H, n, d, generator=g) * w.qk_gain
        K = torch.randn(B, H, n, d, generator=g) * w.qk_gain
        V = torch.randn(B, H, n, v, generator=g)
        dY = torch.randn(B, H, n, v, generator=g)
        Q, K, V, dY = (t.to(w.torch_dtype) for t in (Q, K, V, dY))
    bitmask = None
    if w.mask == "bitmask":
        allowed = (torch.rand(n, n, generator=g) < w.p_allow).numpy()
        np.fill_diagonal(allowed, True)
        bitmask = pack_bitmask(allowed)
    return Inputs(Q, K, V, dY, bitmask)


def make_decode_inputs(B, H, nq, nk, d, v, dtype, mask="none", seed=1, p_allow=0.3,
                       with_dy=False):
    """Q [B,H,nq,d], K [B,H,nk,d], V [B,H,nk,v] (N(0,1), drawn in that order) for
    nq queries at the end of an nk-key sequence, plus bit rows [nq][ceil(nk/32)]
    for the bitmask (each key allowed with p_allow, the query's own position
    i + nk - nq always allowed when it is a key).  ``with_dy`` also draws an
    upstream gradient dY [B,H,nq,v] right after V and returns it fifth."""
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    Q = torch.randn(B, H, nq, d, generator=g).to(tdt)
    K = torch.randn(B, H, nk, d, generator=g).to(tdt)
    V = torch.randn(B, H, nk, v, generator=g).to(tdt)
    dY = torch.randn(B, H, nq, v, generator=g).to(tdt) if with_dy else None
    bitmask = None
    if mask == "bitmask":
        allowed = (torch.rand(nq, nk, generator=g) < p_allow).numpy()
        rows = np.arange(nq)
        own = nk - nq + rows
        allowed[rows[own >= 0], own[own >= 0]] = True
        bitmask = pack_bitmask(allowed)
    if with_dy:
        return Q, K, V, dY, bitmask
    return Q, K, V, bitmask


@dataclass
class DecodeWorkload:
    """nq new queries at the end of an nk-key sequence (a decode step)."""
    name: str
    B: int
    H: int
    nq: int
    nk: int
    d: int
    v: int
    dtype: str
    mask: str
    scale: float
    window: int = 0
    seed: int = SEED_BASE + 100

    def bytes_moved(self) -> int:
        """Algorithmic HBM bytes of one step: read Q, K, V once, write Y and L."""
        e = 4 if self.dtype == "f32" else 2
        per = self.nq * self.d * e + self.nk * (self.d + self.v) * e + self.nq * (self.v * e + 4)
        return self.B * self.H * per


def decode_workload(nq: int = 1) -> DecodeWorkload:
    """Decode step of the long-context training shape: B=8, H=32, d=v=128,
    bf16, causal, nk=16384 keys (K and V 1 GiB each, far beyond L2)."""
    return DecodeWorkload(f"decode-b8h32-nq{nq}-nk16384-d128-bf16-causal", 8, 32, nq, 16384,
                          128, 128, "bf16", "causal", 1.0 / math.sqrt(128.0))


def random_bitmask(n: int, p_allow: float, seed: int, diagonal: bool = True) -> np.ndarray:
    """A seeded random bit-row mask (diagonal forced on unless ``diagonal`` is False)."""
    g = torch.Generator().manual_seed(seed)
    allowed = (torch.rand(n, n, generator=g) < p_allow).numpy()
    if diagonal:
        np.fill_diagonal(allowed, True)
    return pack_bitmask(allowed)


def small(B, H, n, d, v, dtype, mask, scale, window=0, seed=1, qk_gain=1.0,
          p_allow=0.3) -> Workload:
    """An ad-hoc small workload for parity and edge-case tests."""
    return Workload(f"attn-b{B}h{H}-n{n}-d{d}-v{v}-{dtype}-{mask}", B, H, n, d, v, dtype,
                    mask, scale, window=window, qk_gain=qk_gain, p_allow=p_allow,
                    seed=seed)

"""The C ABI without a GPU: the library loads, exports every function that
include/exattn.h declares, and rejects bad arguments on the host before any
CUDA call (so these calls are safe on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "exattn.h")


@pytest.fixture(scope="session")
def lib():
    import exact_tiled_softmax_gb300 as ex
    if not os.path.exists(ex.library_path()):
        from exact_tiled_softmax_gb300 import build
        build.build()
    return ex.load_library()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text,
                       flags=re.M)
    return sorted(set(names) - {"defined"})


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("attn_fwd", "attn_bwd", "exattn_fwd_workspace_size",
                 "exattn_bwd_workspace_size", "exattn_device_status", "exattn_status_string",
                 "exattn_set_path"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(8):
        assert lib.exattn_status_string(code)
    assert lib.exattn_status_string(99) == b"unknown status"


def _shape(B=1, H=1, n=16, d=64, v=64, dtype=1):
    import exact_tiled_softmax_gb300 as ex
    return ex.Shape(B, H, n, d, v, dtype)


def test_workspace_sizes_are_linear_in_n(lib):
    import exact_tiled_softmax_gb300 as ex
    s1 = ex.bwd_workspace_size(_shape(n=1024, d=128), "causal")
    s2 = ex.bwd_workspace_size(_shape(n=2048, d=128), "causal")
    s4 = ex.bwd_workspace_size(_shape(n=4096, d=128), "causal")
    # status word + delta and L log2(e) (4n each, n padded to 128) + dQ
    # accumulator (4nd): no n^2 term.
    assert s2 - s1 == 1024 * (8 + 4 * 128)
    assert s4 - s2 == 2048 * (8 + 4 * 128)
    assert ex.fwd_workspace_size(_shape(n=4096), "causal") == 256
    assert ex.bwd_workspace_size(_shape(n=0), "none") == 0


def test_host_side_argument_checks(lib):
    """Bad arguments return a status before any device work is queued."""
    vp = ctypes.c_void_p
    good = vp(1 << 20)          # never dereferenced: every call below fails its checks first
    ws = vp(1 << 21)

    def fwd(shape, mask=0, window=0, bitmask=None, q=good, ws_ptr=ws, ws_bytes=1 << 20):
        return lib.attn_fwd(ctypes.byref(shape), q, good, good, 1.0, mask, window, bitmask,
                            good, good, ws_ptr, ws_bytes, None)

    assert fwd(_shape(n=0)) == 1                      # INVALID_ARG
    assert fwd(_shape(dtype=7)) == 1
    assert fwd(_shape(d=300)) == 2                    # UNSUPPORTED
    assert fwd(_shape(d=20, dtype=1)) == 2            # bf16 needs multiples of 8
    assert fwd(_shape(), mask=9) == 1
    assert fwd(_shape(), mask=2, window=0) == 1       # window must be >= 1
    assert fwd(_shape(), mask=3, bitmask=None) == 1   # bitmask required
    assert fwd(_shape(), q=None) == 1
    assert fwd(_shape(), q=vp((1 << 20) + 2)) == 3    # MISALIGNED
    assert fwd(_shape(), ws_ptr=vp((1 << 21) + 16)) == 3
    assert fwd(_shape(), ws_bytes=8) == 4             # WORKSPACE_TOO_SMALL
    assert lib.attn_bwd(None, good, good, good, good, good, good, 1.0, 0, 0, None, good, good,
                        good, ws, 1 << 30, None) == 1


def test_host_step_checks_and_workspace(lib):
    """attn_step_host rejects bad arguments before any CUDA call; its workspace
    holds the nine tensors plus one chunk's working space, so it is linear in n."""
    vp = ctypes.c_void_p
    good, ws = vp(1 << 20), vp(1 << 21)

    def step(shape, mask=0, window=0, bitmask=None, q=good, ws_ptr=ws, ws_bytes=1 << 40):
        return lib.attn_step_host(ctypes.byref(shape), q, good, good, good, 1.0, mask, window,
                                  bitmask, good, good, good, good, good, ws_ptr, ws_bytes, None)

    assert step(_shape(n=0)) == 1                      # INVALID_ARG
    assert step(_shape(d=300)) == 2                    # UNSUPPORTED
    assert step(_shape(), mask=3, bitmask=None) == 1   # bitmask required
    assert step(_shape(), mask=2, window=0) == 1
    assert step(_shape(), q=None) == 1
    assert step(_shape(), ws_ptr=vp((1 << 21) + 16)) == 3
    assert step(_shape(), ws_bytes=8) == 4             # WORKSPACE_TOO_SMALL

    def size(n):
        return lib.exattn_host_step_workspace_size(ctypes.byref(_shape(n=n, d=128)), 1)

    s1, s2, s4 = size(1024), size(2048), size(4096)
    assert s1 > 0 and s4 - s2 == 2 * (s2 - s1)
    assert lib.exattn_host_step_workspace_size(None, 0) == 0


def test_path_switch(lib):
    import exact_tiled_softmax_gb300 as ex
    assert ex.set_path("simt") == "auto"
    assert ex.set_path("auto") == "simt"
    assert lib.exattn_set_path(5) == -1


def _qk(B=1, H=1, nq=1, nk=1000, d=128, v=128, dtype=1):
    import exact_tiled_softmax_gb300 as ex
    return ex.QKShape(B, H, nq, nk, d, v, dtype)


def test_splitkv_workspace_and_split_plan(lib):
    """Summaries are 4 (2 + v) bytes per (slice, chunk, query) plus the status
    word and a chunk counter per slice; chunks are whole multiples of 32 keys; 0 picks the count from the
    shape alone."""
    size = lambda shape, splits: lib.exattn_splitkv_workspace_size(ctypes.byref(shape), splits)

    def chunks(shape, splits):
        rows = shape.batch * shape.heads * shape.nq
        counters = (4 * shape.batch * shape.heads + 255) // 256 * 256
        body = size(shape, splits) - 256 - counters
        per = 4 * (2 + shape.v)
        for c in range(1, 5000):  # padding of the m and l arrays is < 2 x 256 bytes
            if 0 <= body - c * rows * per < 512:
                return c
        raise AssertionError(body)

    assert chunks(_qk(nk=1000), 1) == 1
    assert chunks(_qk(nk=1000), 4) == 4        # 250 keys -> chunks of 256
    assert chunks(_qk(nk=1000), 16) == 16      # 63 -> 64 keys per chunk
    assert chunks(_qk(nk=1000), 40) == 32      # 25 -> 32 keys: only 32 chunks
    assert chunks(_qk(nk=1000), 4096) == 32
    # auto: 4864 CTAs over the slices, >= 256 keys per chunk
    assert chunks(_qk(B=8, H=32, nk=16384), 0) == 19
    assert chunks(_qk(B=1, H=1, nk=1000), 0) == 4
    assert chunks(_qk(B=64, H=64, nk=1000), 0) == 2
    assert chunks(_qk(B=128, H=64, nk=1000), 0) == 1
    # bf16, d = v = 128, nq >= 2 (tensor-core chunks): chunks are multiples of 128
    # keys, and auto aims at 8 waves of one CTA per SM (1216 CTAs).
    assert chunks(_qk(nq=8, nk=1000), 4) == 4        # 250 -> 256 keys
    assert chunks(_qk(nq=8, nk=1000), 16) == 8       # 63 -> 128 keys
    assert chunks(_qk(B=8, H=32, nq=8, nk=16384), 0) == 5
    assert chunks(_qk(nq=8, nk=1000, d=80, v=80), 16) == 16   # not a tensor-core shape
    assert chunks(_qk(nq=2, nk=1000), 16) == 8       # two queries: tensor-core chunks
    assert chunks(_qk(nq=2, nk=1000, dtype=0), 16) == 16      # fp32: register kernel
    assert size(_qk(nq=65), 1) == 0            # more than 64 queries
    assert size(_qk(d=20, dtype=1), 1) == 0    # bf16 rows need 8-element pieces
    assert size(_qk(d=20, dtype=0), 1) != 0    # fp32: 4-element pieces
    assert size(_qk(d=18, dtype=0), 1) == 0
    assert size(_qk(), -1) == 0
    assert size(_qk(), 4097) == 0


def test_splitkv_host_side_argument_checks(lib):
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    ws = vp(1 << 21)

    def call(shape, mask=0, window=0, bitmask=None, q=good, splits=1, ws_ptr=ws,
             ws_bytes=1 << 30):
        return lib.attn_fwd_splitkv(ctypes.byref(shape), q, good, good, 1.0, mask, window,
                                    bitmask, splits, good, good, ws_ptr, ws_bytes, None)

    assert call(_qk(nq=0)) == 1
    assert call(_qk(nq=65)) == 2
    assert call(_qk(d=264)) == 2
    assert call(_qk(), mask=2, window=0) == 1
    assert call(_qk(), mask=3) == 1
    assert call(_qk(), splits=-1) == 1
    assert call(_qk(), q=None) == 1
    assert call(_qk(), q=vp((1 << 20) + 8)) == 3
    assert call(_qk(), ws_ptr=vp((1 << 21) + 64)) == 3
    assert call(_qk(), ws_bytes=100) == 4


@pytest.mark.parametrize("bad", ["k_len", "k_heads", "k_width", "v_len", "y", "dy", "L", "L_dtype",
                                 "dq"])
def test_binding_rejects_mismatched_shapes_before_any_launch(lib, bad):
    """The library trusts the sizes in its shape argument, so the Python binding
    checks every tensor against q, k and v first.  CPU tensors: a ValueError
    here means nothing reached the library (which would need device memory)."""
    import torch
    import exact_tiled_softmax_gb300 as ex
    B, H, n, d = 1, 2, 32, 64
    bf = torch.bfloat16
    t = dict(q=torch.zeros(B, H, n, d, dtype=bf), k=torch.zeros(B, H, n, d, dtype=bf),
             v=torch.zeros(B, H, n, d, dtype=bf), y=torch.zeros(B, H, n, d, dtype=bf),
             dy=torch.zeros(B, H, n, d, dtype=bf), L=torch.zeros(B, H, n),
             dq=torch.zeros(B, H, n, d, dtype=bf))
    change = {"k_len": ("k", (B, H, n + 8, d)), "k_heads": ("k", (B, H + 1, n, d)),
              "k_width": ("k", (B, H, n, d + 8)), "v_len": ("v", (B, H, n + 8, d)),
              "y": ("y", (B, H, n, d + 8)), "dy": ("dy", (B, H, n - 1, d)),
              "L": ("L", (B, H, n + 1)), "dq": ("dq", (B, H, n, d - 8))}
    if bad == "L_dtype":
        t["L"] = torch.zeros(B, H, n, dtype=torch.float64)
    else:
        name, shape = change[bad]
        t[name] = torch.zeros(shape, dtype=torch.float32 if name == "L" else bf)
    count = lib.exattn_launch_count()
    with pytest.raises(ValueError):
        ex.bwd_noalloc(t["q"], t["k"], t["v"], t["y"], t["dy"], t["L"], 0.1, "causal",
                       dq=t["dq"])
    if bad not in ("k_len", "v_len"):  # a different key length is cross-attention for bwd
        with pytest.raises(ValueError):
            ex.bwd(t["q"], t["k"], t["v"], t["y"], t["dy"], t["L"], 0.1, "causal", dq=t["dq"])
    assert lib.exattn_launch_count() == count


def test_binding_rejects_bad_bitmasks_workspaces_and_outputs_before_the_library():
    """The library takes the bitmask, the workspace and step_host's outputs as
    bare pointers and sizes it trusts, so the binding checks them first: these
    calls raise ValueError on CPU tensors without reaching any CUDA call."""
    import torch
    import exact_tiled_softmax_gb300 as ex
    q = torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16)
    words = 100 * 4  # rows x ceil(100 / 32)
    short = torch.zeros(words - 1, dtype=torch.int32)
    wide = torch.zeros(words, dtype=torch.int64)
    strided = torch.zeros(2 * words, dtype=torch.int32)[::2]
    for bm in (short, wide, strided):
        with pytest.raises(ValueError):
            ex.fwd(q, k, k, 0.1, "bitmask", 0, bm)
        with pytest.raises(ValueError):
            ex.bwd(q, k, k, q, q, torch.zeros(1, 2, 100), 0.1, "bitmask", 0, bm)
    # decode shape: 3 query rows against 1000 keys read 3 * 32 words
    qd = torch.zeros(1, 2, 3, 64, dtype=torch.bfloat16)
    kd = torch.zeros(1, 2, 1000, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ex.fwd_splitkv(qd, kd, kd, 0.1, "bitmask", 0, torch.zeros(3 * 32 - 1, dtype=torch.int32))
    ex._check_aux(qd, 1000, ex.MASK_BITMASK, torch.zeros(3, 32, dtype=torch.int32))
    ex._check_aux(q, 100, ex.MASK_BITMASK, torch.zeros(100, 4, dtype=torch.int32))
    # another kind of mask reads no words: only the form of a given bitmask is checked
    ex._check_aux(q, 100, ex.MASK_CAUSAL, torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError):
        ex._check_aux(q, 100, ex.MASK_CAUSAL, wide)
    # a workspace on another device than q
    with pytest.raises(ValueError):
        ex._check_aux(q, 100, ex.MASK_CAUSAL, None, torch.zeros(1, dtype=torch.uint8,
                                                                 device="meta"))
    # step_host: outputs of the wrong shape, dtype or place
    dev = torch.device("cuda", 0)
    good = (torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16), torch.zeros(1, 2, 100),
            torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16),
            torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16),
            torch.zeros(1, 2, 100, 64, dtype=torch.bfloat16))
    for i, bad in ((0, torch.zeros(1, 2, 99, 64, dtype=torch.bfloat16)),
                   (1, torch.zeros(1, 2, 100, dtype=torch.float64)),
                   (3, torch.zeros(1, 2, 100, 32, dtype=torch.bfloat16)),
                   (4, torch.zeros(1, 2, 64, 100, dtype=torch.bfloat16).transpose(2, 3))):
        out = list(good)
        out[i] = bad
        with pytest.raises(ValueError):
            ex.step_host(q, k, k, q, 0.1, "causal", out=tuple(out), device=dev)
    with pytest.raises(ValueError):
        ex.step_host(q, k, k, q, 0.1, "bitmask", 0, short, out=good, device=dev)

"""The benchmark's choice of roofline on CPU: which kernel, bound and peak each
shape and kernel path reports, when a zero-padded width is flagged, and when the
captured DRAM traffic is used (only for the kernel the capture was taken of)."""
import types

import pytest

import bench

PEAKS = {"bf16_tflops": 1856.1, "sm_max_mhz": 2070.0}


def _w(d, v, dtype="bf16"):
    return types.SimpleNamespace(d=d, v=v, dtype=dtype, name=f"attn-d{d}-v{v}-{dtype}")


def _args(path="auto", dropout=0.0):
    return types.SimpleNamespace(path=path, dropout=dropout)


@pytest.fixture
def no_traffic(monkeypatch):
    """read_traffic stubbed: records the tags asked for, answers 1.0."""
    asked = []

    def fake(tag, workload):
        asked.append(tag)
        return 1.0

    monkeypatch.setattr(bench, "read_traffic", fake)
    return asked


@pytest.mark.parametrize("which,tag", [("fwd", "tc_fwd"), ("bwd", "tc_bwd_split")])
def test_bf16_native_widths_use_the_tensor_peak_and_the_capture(no_traffic, which, tag):
    r = bench.kernel_roofline(_args(), _w(128, 128), which, 928.05, PEAKS, "measured")
    assert r["kernel"] == tag and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == PEAKS["bf16_tflops"]
    assert r["frac"] == pytest.approx(0.5)
    assert r["traffic"] == 1.0 and no_traffic == [tag]
    assert "padded_to" not in r


@pytest.mark.parametrize("d,v,to", [(80, 96, 128), (48, 64, 64), (8, 8, 64), (40, 128, 128),
                                    (128, 8, 128)])
def test_bf16_padded_widths_report_the_kernel_width_and_no_capture(no_traffic, d, v, to):
    for which in ("fwd", "bwd"):
        r = bench.kernel_roofline(_args(), _w(d, v), which, 100.0, PEAKS, "measured")
        assert r["bound"] == "tensor" and r["padded_to"] == to
        # The capture was taken at d = v = 128: it says nothing about a padded launch.
        assert r["traffic"] is None
    assert no_traffic == []


@pytest.mark.parametrize("d,v", [(72, 136), (136, 64), (256, 256)])
def test_bf16_widths_outside_the_tensor_kernels_are_alu_bound(no_traffic, d, v):
    r = bench.kernel_roofline(_args(), _w(d, v), "fwd", 10.0, PEAKS, "measured")
    assert r["kernel"] == "simt_fwd" and r["bound"] == "alu"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)


def test_atomic_reverse_form_takes_only_native_widths(no_traffic):
    r = bench.kernel_roofline(_args("atomic_dq"), _w(128, 128), "bwd", 1.0, PEAKS, "measured")
    assert r["kernel"] == "tc_bwd_atomic"
    r = bench.kernel_roofline(_args("atomic_dq"), _w(80, 96), "bwd", 1.0, PEAKS, "measured")
    assert r["kernel"] == "simt_bwd"
    # Its forward is the ordinary tensor-core forward, padded as usual.
    r = bench.kernel_roofline(_args("atomic_dq"), _w(80, 96), "fwd", 1.0, PEAKS, "measured")
    assert r["kernel"] == "tc_fwd" and r["padded_to"] == 128


def test_simt_path_is_alu_bound_for_every_shape(no_traffic):
    for which in ("fwd", "bwd"):
        r = bench.kernel_roofline(_args("simt"), _w(128, 128), which, 1.0, PEAKS, "measured")
        assert r["kernel"] == f"simt_{which}" and r["bound"] == "alu"


def test_fp32_forward_uses_the_derived_tf32_peak(no_traffic):
    r = bench.kernel_roofline(_args(), _w(128, 128, "f32"), "fwd", 90.0, PEAKS, "measured")
    assert r["kernel"] == "tc32_fwd"
    assert r["peak"] == pytest.approx(PEAKS["bf16_tflops"] * 1.1 / 2.25)
    assert r["tensor_work_frac"] == pytest.approx(3 * r["frac"])
    # With dropout, or for the reverse pass of d = 128, fp32 runs on the SIMT kernels.
    assert bench.kernel_roofline(_args(dropout=0.1), _w(128, 128, "f32"), "fwd", 1.0, PEAKS,
                                 "measured")["kernel"] == "simt_fwd"
    assert bench.kernel_roofline(_args(), _w(128, 128, "f32"), "bwd", 1.0, PEAKS,
                                 "measured")["kernel"] == "simt_bwd"


def test_fp32_reverse_of_width_64_is_the_3xtf32_kernel_pair(no_traffic):
    r = bench.kernel_roofline(_args(), _w(64, 64, "f32"), "bwd", 90.0, PEAKS, "measured")
    assert r["kernel"] == "tc32_bwd" and r["bound"] == "tensor"
    assert r["peak"] == pytest.approx(PEAKS["bf16_tflops"] * 1.1 / 2.25)
    # 7 products per tile, each three tf32 products, against the convention's 5
    assert r["tensor_work_frac"] == pytest.approx(21 / 5 * r["frac"])
    for args, w in ((_args("simt"), _w(64, 64, "f32")), (_args(dropout=0.1), _w(64, 64, "f32")),
                    (_args("atomic_dq"), _w(64, 64, "f32")), (_args(), _w(80, 96, "f32"))):
        assert bench.kernel_roofline(args, w, "bwd", 1.0, PEAKS, "measured")["kernel"] == "simt_bwd"


def test_read_traffic_rejects_a_changed_source_or_another_launch(tmp_path, monkeypatch):
    """An entry counts only for the workload launch it was taken on, and only
    while its kernel source hashes to the recorded prefix."""
    import hashlib
    csrc = tmp_path / "exact_tiled_softmax_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# comment\n"
        f"kernel=tc_fwd launch=attn-x source=k.cu source_sha={sha} bytes_per_launch=12345 "
        "measured_on=x\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("tc_fwd", "attn-x") == 12345.0
    assert bench.read_traffic("tc_fwd", "attn-y") is None
    assert bench.read_traffic("tc_bwd_split", "attn-x") is None
    src.write_bytes(b"__global__ void k() { }\n")
    assert bench.read_traffic("tc_fwd", "attn-x") is None


def test_committed_traffic_entries_name_bench_workloads():
    """Every committed entry names the launch of a workload that bench.py runs."""
    import workloads
    names = {workloads.workload(3).name, workloads.decode_workload(1).name,
             workloads.decode_workload(4).name,
             workloads.workload(3).name + "-as-f32", workloads.workload(2).name + "-as-f32"}
    path = bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt")
    with open(path) as f:
        entries = [dict(p.split("=", 1) for p in line.split())
                   for line in f if line.strip() and not line.startswith("#")]
    assert entries
    for e in entries:
        assert e.get("launch") in names, e


def test_decode_kernel_rule_matches_the_library_plan():
    """bench.py names the decode kernels from the shape; the library's plan tells
    the tensor-core chunks apart (whole 128-key chunks, against 32 keys for the
    other kernels).  With nk = 1000 and 16 chunks asked for, a 128-key plan
    gives 8 chunks and a 32-key plan 16."""
    import ctypes
    import dataclasses
    import exact_tiled_softmax_gb300 as ex
    import workloads
    lib = ex.load_library()
    base = workloads.decode_workload(1)
    for dtype in ("bf16", "f32"):
        for d, v in ((64, 64), (128, 128), (80, 96), (128, 64), (32, 32)):
            for nq in (1, 2, 3, 4, 5, 16, 64):
                w = dataclasses.replace(base, B=1, H=1, nq=nq, nk=1000, d=d, v=v, dtype=dtype)
                shape = ex.QKShape(1, 1, nq, 1000, d, v, 0 if dtype == "f32" else 1)
                size = lib.exattn_splitkv_workspace_size(ctypes.byref(shape), 16)
                assert size > 0
                rows = nq
                body = size - 256 - 256 - 2 * ((4 * rows * 16 + 255) // 256 * 256)
                chunks = 8 if body < 16 * rows * 4 * v else 16
                kind = bench.decode_kernels(w)
                assert (kind == "tc") == (chunks == 8), (dtype, d, v, nq, kind, chunks)
                assert kind == "tc" or kind == ("reg" if nq <= 4 else "smem")

"""The benchmark's record of DRAM traffic per launch (profiles/traffic.txt):
a figure is reported only while the code it was measured on is unchanged.
These checks run on a copy of the sources, without a GPU."""
import os
import shutil

import pytest

import bench

CSRC = os.path.join(bench.ROOT, "bf16_gemm_skinny_gb300", "csrc")


@pytest.fixture()
def srcdir(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d)
    return str(d)


def _append(path, text):
    with open(path, "a") as f:
        f.write(text)


def _insert_after(path, marker, text):
    with open(path) as f:
        s = f.read()
    i = s.index(marker) + len(marker)
    with open(path, "w") as f:
        f.write(s[:i] + text + s[i:])


def test_digest_is_the_package_sources_by_default(srcdir):
    for kernel in bench.KERNEL_SOURCES:
        assert bench.source_digest(kernel) == bench.source_digest(kernel, srcdir)


def test_comments_and_layout_do_not_count(srcdir):
    before = bench.source_digest("gemm", srcdir)
    path = os.path.join(srcdir, "gemm_tcgen05.cuh")
    _insert_after(path, "struct Params {", "\n    // a comment\n    /* and another */\n\n")
    assert bench.source_digest("gemm", srcdir) == before


def test_kernel_code_counts(srcdir):
    before = bench.source_digest("gemm", srcdir)
    _insert_after(os.path.join(srcdir, "gemm_tcgen05.cuh"), "struct Params {", "\n    int unused_field;\n")
    assert bench.source_digest("gemm", srcdir) != before


def test_planner_counts_but_other_host_code_does_not(srcdir):
    api = os.path.join(srcdir, "api.cu")
    before = bench.source_digest("gemm", srcdir)
    _append(api, "\nint an_unrelated_host_function() { return 1; }\n")
    assert bench.source_digest("gemm", srcdir) == before
    _insert_after(api, "struct GemmPlan {", "\n    int another_choice = 0;\n")
    assert bench.source_digest("gemm", srcdir) != before


def test_host_launch_code_after_the_marker_does_not_count(srcdir):
    before = bench.source_digest("gemv", srcdir)
    _append(os.path.join(srcdir, "gemv.cu"), "\nstatic int host_helper() { return 2; }\n")
    assert bench.source_digest("gemv", srcdir) == before


def test_missing_marker_is_an_error(srcdir):
    path = os.path.join(srcdir, "api.cu")
    with open(path) as f:
        s = f.read()
    with open(path, "w") as f:
        f.write(s.replace("// Elements a stored matrix", "// (marker removed)"))
    with pytest.raises(RuntimeError):
        bench.source_digest("gemm", srcdir)


def test_recorded_figures_are_per_launch_byte_counts():
    for key in ("gemm_f16_8192x8192x16384", "gemv_bf16_34816x5120_n1"):
        v = bench.committed_traffic(key)
        # None only when the code has changed since the figure was measured
        assert v is None or v > 3.5e8

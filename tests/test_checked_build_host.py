"""The checked debug build without a GPU: its range test is right at the edges,
it builds from the same sources, exports what the header declares and says
which build it is; and the scratch size the library reports is the header's.
No kernel is launched here."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import memory_bound_normalization_gb300 as pkg
from memory_bound_normalization_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")

# A host program over the range test the checked kernels use (span_in is a
# host and device function): each line prints one verdict.
SPAN_PROGRAM = r"""
#include <cstdio>
#include "common.cuh"
int main() {
    alignas(16) static unsigned char buf[256];
    const unsigned char* b = buf;
    const int64_t ext = 256;
    const struct { const void* p; int64_t n; } cases[] = {
        {b, 16}, {b + 240, 16}, {b + 241, 16}, {b + 256, 0}, {b + 256, 1},
        {b - 1, 1}, {b, 256}, {b, 257}, {b + 16, -1}, {b + 100, 0},
    };
    for (const auto& c : cases) std::printf("%d\n", rmsn::span_in(c.p, c.n, b, ext) ? 1 : 0);
    std::printf("%d\n", rmsn::span_in(b, 0, b, 0) ? 1 : 0);
    std::printf("%d\n", rmsn::span_in(b, 1, b, 0) ? 1 : 0);
    return 0;
}
"""
SPAN_EXPECTED = [1, 1, 0, 1, 0, 0, 1, 0, 0, 1, 1, 0]


def test_span_in_edges(tmp_path):
    src = tmp_path / "span.cu"
    src.write_text(SPAN_PROGRAM)
    exe = tmp_path / "span"
    cmd = [libbuild._nvcc(), *libbuild.ARCH, "-std=c++17", "-I", libbuild.INCLUDE, "-I",
           libbuild.CSRC, str(src), "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert [int(v) for v in out] == SPAN_EXPECTED


@pytest.fixture(scope="module")
def checked_lib():
    path = libbuild.build(checked=True)
    assert path == libbuild.CHECKED_LIB_PATH
    lib = ctypes.CDLL(path)
    lib.rmsnorm_version.restype = ctypes.c_char_p
    return lib


def test_checked_build_exports_and_names_itself(checked_lib):
    for name in pkg.EXPORTS:
        assert hasattr(checked_lib, name), f"{name} missing from the checked build"
    assert checked_lib.rmsnorm_version().decode().endswith("+checks")


def test_checked_variant_is_opt_in(monkeypatch):
    monkeypatch.delenv("RMSNORM_LIBRARY_VARIANT", raising=False)
    assert pkg.library_path() == libbuild.LIB_PATH
    monkeypatch.setenv("RMSNORM_LIBRARY_VARIANT", "checked")
    assert pkg.library_path() == libbuild.CHECKED_LIB_PATH


def test_checked_sources_are_the_same():
    # one source list for both builds: the variant differs only by the macro
    plans = libbuild._variant_jobs(True, [])[0]
    assert [c[0][-3] for c in plans] == [os.path.join(libbuild.CSRC, s)
                                         for s in libbuild.SOURCES]
    assert all("-DRMSNORM_CHECKS" in c[0] for c in plans)
    assert not any("-DRMSNORM_CHECKS" in c[0] for c in libbuild._variant_jobs(False, [])[0])


def test_noalloc_scratch_size_matches_header():
    libbuild.build()
    text = open(HEADER).read()
    m = re.search(r"#define RMSNORM_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "scratch size macro not found in the header"
    assert pkg.rmsnorm_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_status_codes_match_header():
    text = open(HEADER).read()
    codes = dict(re.findall(r"RMSNORM_(ERR_[A-Z_]+|OK) = (\d+)", text))
    for name, value in codes.items():
        assert getattr(pkg, name) == int(value), name
    assert pkg.ERR_OUT_OF_BOUNDS == 7

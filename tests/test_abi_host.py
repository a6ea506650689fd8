"""Host-only checks of the C ABI: the library builds, loads, exports every entry
point declared in include/fp8q.h, and rejects bad arguments on the host before
any CUDA call (these paths run without a GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import build as fqbuild

HEADER = os.path.join(ROOT, "include", "fp8q.h")

OK, INVALID, SHAPE, ALIGN, UNSUP = 0, 1, 2, 3, 4
FAKE = 0x10000          # a 16-byte aligned address; never dereferenced by rejected calls


@pytest.fixture(scope="module")
def lib():
    fqbuild.build()
    return fq.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^(?:fp8_status|const char\*)\s+(\w+)\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ("fp8_amax", "fp8_compute_scale", "amax_history_update", "fp8_quantize",
                     "fp8_cast_transpose", "fp8_scaled_gemm", "fp8_get_device_status", "fp8_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # the binding exposes the same names
    for name in declared_functions():
        assert hasattr(fq, name), name


def test_status_strings(lib):
    for st in fq.Status:
        assert lib.fp8_status_string(int(st)).decode() == "FP8_" + st.name


def test_amax_rejects(lib):
    assert lib.fp8_amax(None, 4, 4, FAKE, None) == INVALID          # null x with elements
    assert lib.fp8_amax(FAKE, -1, 4, FAKE, None) == INVALID
    assert lib.fp8_amax(FAKE, 4, 4, None, None) == INVALID          # null amax
    assert lib.fp8_amax(FAKE + 2, 4, 4, FAKE, None) == ALIGN


def test_f32_entry_points_reject(lib):
    assert lib.fp8_amax_f32(None, 4, 4, FAKE, None) == INVALID       # null x with elements
    assert lib.fp8_amax_f32(FAKE, 4, 4, None, None) == INVALID       # null amax
    assert lib.fp8_amax_f32(FAKE + 4, 4, 4, FAKE, None) == ALIGN     # x not 16-byte aligned
    ct = lib.fp8_cast_transpose_f32
    T, B1, B128, MXT = 0, 1, 2, 4
    assert ct(FAKE, 128, 128, T, 0, FAKE, None, None, None, None, None, None) == INVALID    # nothing requested
    assert ct(FAKE, 128, 128, T, 0, None, None, FAKE, None, None, None, None) == INVALID    # per-tensor scale
    assert ct(FAKE, 100, 256, B128, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE   # rows % 128
    assert ct(FAKE, 128, 96, MXT, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE     # cols % 128
    assert ct(FAKE + 8, 128, 128, B1, 0, None, None, FAKE, FAKE, None, None, None) == ALIGN
    assert ct(FAKE, 0, 128, B1, 0, None, None, None, None, None, None, None) == OK          # empty: no-op


def test_floor_rule_mx_recipes_are_checked_like_mx(lib):
    ct = lib.fp8_cast_transpose
    MXF, MXFT = 5, 6
    assert ct(FAKE, 128, 96, MXF, 0, None, None, FAKE, FAKE, None, None, None) != SHAPE      # 96 % 32 == 0
    assert ct(FAKE, 128, 100, MXF, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE     # cols % 32
    assert ct(FAKE, 128, 96, MXFT, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE     # tiled: cols % 128
    assert ct(FAKE, 128, 128, 7, 0, None, None, FAKE, FAKE, None, None, None) == INVALID     # no recipe 7
    g = lib.fp8_scaled_gemm
    # empty GEMMs return on the host: the pairing checks come first
    assert g(FAKE, 0, 4, FAKE, FAKE, 0, MXFT, FAKE, 0, 0, 0, FAKE, 0, None) == OK             # MX x MX-floor
    assert g(FAKE, 0, MXFT, FAKE, FAKE, 0, MXFT, FAKE, 0, 0, 0, FAKE, 0, None) == OK
    assert g(FAKE, 0, MXF, FAKE, FAKE, 0, MXFT, FAKE, 0, 0, 0, FAKE, 0, None) == UNSUP       # row-major scales
    assert lib.fp8_dequantize(FAKE, 128, 100, MXF, 0, FAKE, FAKE, None) == SHAPE


def test_scale_and_history_reject(lib):
    assert lib.fp8_compute_scale(FAKE, 7, FAKE, FAKE, None) == INVALID    # bad format
    assert lib.fp8_compute_scale(None, 0, FAKE, FAKE, None) == INVALID
    assert lib.fp8_compute_scale(FAKE + 1, 0, FAKE, FAKE, None) == ALIGN
    assert lib.amax_history_update(FAKE, 0, FAKE, FAKE, 0, FAKE, FAKE, None) == INVALID   # len 0
    assert lib.amax_history_update(None, 16, FAKE, FAKE, 0, FAKE, FAKE, None) == INVALID


def test_cast_transpose_rejects(lib):
    ct = lib.fp8_cast_transpose
    T, B1, B128, MX, MXT = 0, 1, 2, 3, 4
    # nothing requested
    assert ct(FAKE, 128, 128, T, 0, FAKE, None, None, None, None, None, None) == INVALID
    # per-tensor needs a scale
    assert ct(FAKE, 128, 128, T, 0, None, None, FAKE, None, None, None, None) == INVALID
    # bad recipe / format
    assert ct(FAKE, 128, 128, 9, 0, None, None, FAKE, FAKE, None, None, None) == INVALID
    assert ct(FAKE, 128, 128, B1, 3, None, None, FAKE, FAKE, None, None, None) == INVALID
    # block recipes need their scale outputs
    assert ct(FAKE, 128, 128, B1, 0, None, None, FAKE, None, None, None, None) == INVALID
    # blocked dimensions
    assert ct(FAKE, 100, 200, B1, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE      # cols % 128
    assert ct(FAKE, 100, 256, B1, 0, None, None, None, None, FAKE, FAKE, None) == SHAPE      # col copy: rows % 128
    assert ct(FAKE, 128, 200, B128, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE
    assert ct(FAKE, 64, 48, MX, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE        # cols % 32
    assert ct(FAKE, 48, 64, MX, 0, None, None, None, None, FAKE, FAKE, None) == SHAPE        # rows % 32
    assert ct(FAKE, 160, 256, MXT, 0, None, None, FAKE, FAKE, None, None, None) == SHAPE     # tiled: % 128
    # alignment
    assert ct(FAKE + 8, 128, 128, B1, 0, None, None, FAKE, FAKE, None, None, None) == ALIGN
    assert ct(FAKE, 128, 128, B1, 0, None, None, FAKE + 4, FAKE, None, None, None) == ALIGN
    assert ct(FAKE, 128, 128, B1, 0, None, None, FAKE, FAKE + 2, None, None, None) == ALIGN
    assert ct(FAKE, 128, 128, MXT, 0, None, None, FAKE, FAKE + 4, None, None, None) == ALIGN
    # quantize = row-wise only, needs q
    assert lib.fp8_quantize(FAKE, 128, 128, B1, 0, None, None, None, FAKE, None) == INVALID


def test_gemm_rejects(lib):
    g = lib.fp8_scaled_gemm
    T, B1, B128, MX, MXT = 0, 1, 2, 3, 4
    args = lambda ra, rb, M=256, N=256, K=256, out=0, a=FAKE, c=FAKE: (a, 0, ra, FAKE, FAKE, 0, rb, FAKE, M, N, K, c,
                                                                       out, None)
    assert g(*args(T, B1)) == UNSUP
    assert g(*args(MX, MX)) == UNSUP          # row-major MX scales: quantize with the tiled layout
    assert g(*args(B128, B1)) == UNSUP
    assert g(*args(7, T)) == INVALID
    assert g(*args(T, T, out=5)) == INVALID
    assert g(*args(T, T, M=200)) == SHAPE
    assert g(*args(T, T, K=100)) == SHAPE
    assert g(*args(B1, B128, N=130)) == SHAPE
    assert g(*args(T, T, a=FAKE + 8)) == ALIGN
    assert g(*args(T, T, c=FAKE + 4)) == ALIGN
    assert g(*args(T, T, a=None)) == INVALID
    assert g(*args(T, T, M=-1)) == INVALID
    # empty outputs are a no-op that needs no device
    assert g(*args(T, T, M=0)) == OK
    assert g(*args(T, T, N=0)) == OK


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(OSError):
        fq.load_library(str(tmp_path / "missing.so"))


def test_gemm_amax_rejects(lib):
    g = lib.fp8_scaled_gemm_amax
    T, B1 = 0, 1

    def args(ra=T, rb=T, M=256, N=256, K=256, c=FAKE, amax=FAKE, scale=FAKE, fc=0, cq=FAKE, sinv=FAKE):
        return (FAKE, 0, ra, FAKE, FAKE, 0, rb, FAKE, M, N, K, c, 0, amax, scale, fc, cq, sinv, None)

    assert g(*args(amax=None, cq=None)) == INVALID           # nothing fused requested
    assert g(*args(scale=None)) == INVALID                   # the FP8 copy needs its scale
    assert g(*args(cq=None)) == INVALID                      # scale_inv only with the FP8 copy
    assert g(*args(fc=4)) == INVALID
    assert g(*args(T, B1)) == UNSUP
    assert g(*args(M=200)) == SHAPE
    assert g(*args(cq=FAKE + 8)) == ALIGN
    assert g(*args(amax=FAKE + 2)) == ALIGN
    assert g(*args(c=FAKE + 4)) == ALIGN


def test_dequantize_rejects(lib):
    dq = lib.fp8_dequantize
    T, B1, B128, MX, MXT = 0, 1, 2, 3, 4
    assert dq(FAKE, 128, 128, 9, 0, FAKE, FAKE, None) == INVALID        # bad recipe
    assert dq(FAKE, 128, 128, T, 2, FAKE, FAKE, None) == INVALID        # bad format
    assert dq(None, 128, 128, T, 0, FAKE, FAKE, None) == INVALID
    assert dq(FAKE, 128, 128, T, 0, None, FAKE, None) == INVALID
    assert dq(FAKE, 128, 100, B1, 0, FAKE, FAKE, None) == SHAPE
    assert dq(FAKE, 100, 128, B128, 0, FAKE, FAKE, None) == SHAPE
    assert dq(FAKE, 128, 48, MX, 0, FAKE, FAKE, None) == SHAPE
    assert dq(FAKE, 160, 128, MXT, 0, FAKE, FAKE, None) == SHAPE
    assert dq(FAKE + 8, 128, 128, T, 0, FAKE, FAKE, None) == ALIGN
    assert dq(FAKE, 128, 128, T, 0, FAKE, FAKE + 2, None) == ALIGN
    assert dq(FAKE, 128, 128, B1, 0, FAKE + 1, FAKE, None) == ALIGN
    assert dq(FAKE, 0, 128, T, 0, None, None, None) == OK                # empty: no-op


def test_allreduce_rejects(lib):
    ar = lib.fp8_allreduce_sum
    assert ar(FAKE, 0, 64, 0, FAKE, FAKE, FAKE, FAKE, None) == INVALID        # no ranks
    assert ar(FAKE, 2, 64, 5, FAKE, FAKE, FAKE, FAKE, None) == INVALID        # bad format
    assert ar(None, 2, 64, 0, FAKE, FAKE, FAKE, FAKE, None) == INVALID
    assert ar(FAKE, 2, 60, 0, FAKE, FAKE, FAKE, FAKE, None) == SHAPE          # n % 8
    assert ar(FAKE + 8, 2, 64, 0, FAKE, FAKE, FAKE, FAKE, None) == ALIGN
    assert ar(FAKE, 2, 64, 0, FAKE, FAKE + 4, FAKE, FAKE, None) == ALIGN
    assert ar(FAKE, 2, 64, 0, FAKE, FAKE, FAKE, FAKE + 8, None) == ALIGN
    assert ar(FAKE, 2, 0, 0, None, None, None, None, None) == OK               # empty: no-op


def test_allreduce_noalloc_rejects(lib):
    ar = lib.fp8_allreduce_sum_noalloc
    assert ar(FAKE, 1025, 64, 0, FAKE, FAKE, FAKE, None) == SHAPE       # more ranks than the scratch holds
    assert ar(FAKE, 0, 64, 0, FAKE, FAKE, FAKE, None) == INVALID
    assert ar(FAKE, 2, 64, 3, FAKE, FAKE, FAKE, None) == INVALID        # bad format
    assert ar(FAKE, 2, 60, 0, FAKE, FAKE, FAKE, None) == SHAPE          # n % 8
    assert ar(FAKE + 8, 2, 64, 0, FAKE, FAKE, FAKE, None) == ALIGN
    assert ar(FAKE, 2, 0, 0, None, None, None, None) == OK               # empty: no-op


def test_cast_multi_rejects(lib):
    job = fq.CastJob
    T, B1 = 0, 1
    good = job(FAKE, 128, 128, B1, 0, None, None, FAKE, FAKE, None, None)
    bad_shape = job(FAKE, 128, 100, B1, 0, None, None, FAKE, FAKE, None, None)
    bad_align = job(FAKE + 8, 128, 128, B1, 0, None, None, FAKE, FAKE, None, None)
    arr = (job * 5)(good, good, good, good, good)
    assert lib.fp8_cast_transpose_multi(arr, 5, None) == INVALID      # more than 4 jobs
    assert lib.fp8_cast_transpose_multi(None, 1, None) == INVALID
    assert lib.fp8_cast_transpose_multi(arr, 0, None) == OK
    arr2 = (job * 2)(bad_shape, good)
    assert lib.fp8_cast_transpose_multi(arr2, 2, None) == SHAPE      # checked before any device work
    arr3 = (job * 2)(bad_align, good)
    assert lib.fp8_cast_transpose_multi(arr3, 2, None) == ALIGN

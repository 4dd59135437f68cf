"""CPU checks of the C-ABI library: it builds, loads, exports every function
include/csf.h declares, and its host-only paths (sizes, argument checks that
return before any CUDA call) behave as documented.  No GPU needed."""
import ctypes
import os
import re

import pytest

from lossless_nvfp4_scale_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def csf():
    build.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf as mod
    return mod


def declared_functions():
    text = open(os.path.join(ROOT, "include", "csf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csf_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(csf):
    names = declared_functions()
    assert {"csf_prepare", "csf_prepare_static", "csf_decode", "csf_decode_pair", "csf_sizes"} <= set(names)
    lib = ctypes.CDLL(build.LIB)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/csf.h but not exported"


def test_abi_version_and_status_strings(csf):
    assert csf.lib.csf_abi_version() == 5
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "buffer too small"),
                       (3, "unsupported geometry"), (4, "CUDA error")]:
        assert csf.lib.csf_status_string(code).decode() == text


@pytest.mark.parametrize("kind,E,R,C", [(0, 512, 1024, 100), (0, 512, 2048, 50), (1, 384, 2048, 160),
                                        (0, 1, 1, 1), (1, 3, 5, 7)])
def test_sizes(csf, kind, E, R, C):
    sz = csf.sizes(kind, E, R, C)
    n = E * R * C
    assert sz["dense"] == n and sz["base"] == E * R and sz["exc_index"] == 4 * (E * R + 1)
    packed = (n + 1) // 2 if kind == 0 else (n + 7) // 8
    assert sz["offsets"] == (packed + 15) // 16 * 16
    assert sz["escapes"] == (0 if kind == 0 else sz["offsets"])
    assert sz["prepare_scratch"] >= 16 + 8
    assert sz["blocked"] == E * (-(-R // 128) * 128) * (-(-C // 4) * 4)
    tiles = E * (-(-R // 128)) * (-(-C // 4))
    assert sz["tiled_codes"] == tiles * (256 if kind == 0 else 128)
    assert sz["tiled_bases"] == E * (-(-R // 128)) * 128 and sz["tiled_index"] == 4 * (tiles + 1)


def test_sizes_rejects_bad_geometry(csf):
    with pytest.raises(csf.CsfError, match="invalid argument"):
        csf.sizes(2, 1, 1, 1)
    with pytest.raises(csf.CsfError, match="invalid argument"):
        csf.sizes(0, 0, 1, 1)
    with pytest.raises(csf.CsfError, match="unsupported"):
        csf.sizes(0, 1 << 16, 1 << 16, 1)


def test_null_arguments_rejected_before_cuda(csf):
    # All of these return before the library touches the CUDA runtime.
    assert csf.lib.csf_decode(None, None, 0, None, 0, None) == 1
    assert csf.lib.csf_decode_pair(None, None, 0, None, None, 0, None, 0, None) == 1
    assert csf.lib.csf_prepare(None, None, 0, None, 0, None) == 1
    g = csf.Geometry(0, 1, 1, 32)
    st = csf.CStack(g, 16, 16, None, 16, 16, 0, None)
    # ws too small for the geometry.
    assert csf.lib.csf_decode(ctypes.byref(st), 16, 31, None, 0, None) == 2
    # offsets not 16-byte aligned.
    st_bad = csf.CStack(g, 16, 17, None, 16, 16, 0, None)
    assert csf.lib.csf_decode(ctypes.byref(st_bad), 16, 64, None, 0, None) == 1
    # MXFP4 without an escape plane.
    st_mx = csf.CStack(csf.Geometry(1, 1, 1, 32), 16, 16, None, 16, 16, 0, None)
    assert csf.lib.csf_decode(ctypes.byref(st_mx), 16, 64, None, 0, None) == 1
    # pair with different expert counts.
    st2 = csf.CStack(csf.Geometry(0, 2, 1, 32), 16, 16, None, 16, 16, 0, None)
    assert csf.lib.csf_decode_pair(ctypes.byref(st), 16, 64, ctypes.byref(st2), 16, 64, None, 0, None) == 1
    # routed decode with too many experts for the shared-memory active list.
    big = csf.CStack(csf.Geometry(0, 8193, 1, 32), 16, 16, None, 16, 16, 0, None)
    assert csf.lib.csf_decode(ctypes.byref(big), 16, 8193 * 32, 16, 0, None) == 3


def test_decode_rows_argument_checks_before_cuda(csf):
    # csf_decode_rows rejects bad part counts and row ranges on the host,
    # before any CUDA call (the pointers below are never dereferenced).
    g = csf.Geometry(0, 2, 10, 32)
    st = csf.CStack(g, 16, 16, None, 16, 16, 0, None)

    def parts(*ranges, stack=st):
        arr = (csf.CDecodePart * len(ranges))()
        for i, (lo, hi) in enumerate(ranges):
            arr[i] = csf.CDecodePart(ctypes.pointer(stack), 16, 1 << 30, lo, hi)
        return arr

    assert csf.lib.csf_decode_rows(None, 1, None, 0, None) == 1
    assert csf.lib.csf_decode_rows(parts((0, 5)), 0, None, 0, None) == 1
    assert csf.lib.csf_decode_rows(parts((0, 5), (0, 5), (0, 5)), 3, None, 0, None) == 1
    for bad in [(-1, 5), (5, 5), (6, 5), (0, 11)]:
        assert csf.lib.csf_decode_rows(parts(bad), 1, None, 0, None) == 1, bad
    nul = (csf.CDecodePart * 1)()
    nul[0] = csf.CDecodePart(None, 16, 640, 0, 5)
    assert csf.lib.csf_decode_rows(nul, 1, None, 0, None) == 1
    # Parts with different expert counts.
    other = csf.CStack(csf.Geometry(0, 3, 10, 32), 16, 16, None, 16, 16, 0, None)
    two = (csf.CDecodePart * 2)()
    two[0] = csf.CDecodePart(ctypes.pointer(st), 16, 640, 0, 5)
    two[1] = csf.CDecodePart(ctypes.pointer(other), 16, 960, 0, 5)
    assert csf.lib.csf_decode_rows(two, 2, None, 0, None) == 1
    # A partial row range keeps the per-expert work list in shared memory.
    big = csf.CStack(csf.Geometry(0, 8193, 2, 32), 16, 16, None, 16, 16, 0, None)
    assert csf.lib.csf_decode_rows(parts((0, 1), stack=big), 1, None, 0, None) == 3


def test_expand_argument_checks_before_cuda(csf):
    # csf_expand checks its parts before it enqueues a wait, a launch or a
    # record (nothing below reaches the CUDA runtime).
    st = csf.CStack(csf.Geometry(0, 2, 10, 32), 16, 16, None, 16, 16, 0, None)
    assert csf.lib.csf_expand(None, 1, None, None, None) == 1
    arr = (csf.CDecodePart * 3)()
    for i in range(3):
        arr[i] = csf.CDecodePart(ctypes.pointer(st), 16, 1 << 20, 0, 10)
    assert csf.lib.csf_expand(arr, 0, None, None, None) == 1
    assert csf.lib.csf_expand(arr, 3, None, None, None) == 1
    bad = (csf.CDecodePart * 1)()
    bad[0] = csf.CDecodePart(ctypes.pointer(st), 16, 1 << 20, 4, 4)
    assert csf.lib.csf_expand(bad, 1, None, None, None) == 1
    small = (csf.CDecodePart * 1)()
    small[0] = csf.CDecodePart(ctypes.pointer(st), 16, 639, 0, 10)
    assert csf.lib.csf_expand(small, 1, None, None, None) == 2


def test_blocked_layout_argument_checks_before_cuda(csf):
    # The blocked layout's own checks return before any CUDA call.
    g = csf.Geometry(0, 2, 256, 100)
    st = csf.CStack(g, 16, 16, None, 16, 16, 0, None)
    nb = csf.sizes(0, 2, 256, 100)["blocked"]

    def one(ws=16, nbytes=nb, lo=0, hi=256, layout=csf.LAYOUT_BLOCKED, stack=st):
        arr = (csf.CDecodePart * 1)()
        arr[0] = csf.CDecodePart(ctypes.pointer(stack), ws, nbytes, lo, hi, layout)
        return csf.lib.csf_decode_rows(arr, 1, None, 0, None)

    assert one(ws=24) == 1                       # workspace not 16-byte aligned
    assert one(lo=64) == 1 and one(hi=200) == 1  # rows off the 128-row boundaries
    assert one(nbytes=nb - 1) == 2               # smaller than the blocked size
    assert one(layout=7) == 1                    # unknown layout
    mixed = (csf.CDecodePart * 2)()
    mixed[0] = csf.CDecodePart(ctypes.pointer(st), 16, nb, 0, 256, csf.LAYOUT_BLOCKED)
    mixed[1] = csf.CDecodePart(ctypes.pointer(st), 16, nb, 0, 256, csf.LAYOUT_ROWS)
    assert csf.lib.csf_decode_rows(mixed, 2, None, 0, None) == 1


def test_expand_scales_needs_the_workspace(csf):
    # Host-side check of the binding: a compressed stack without its
    # workspace is an error (no CUDA call is made).
    class Fake:
        pass
    with pytest.raises(csf.CsfError, match="workspace"):
        csf.expand_scales([(Fake(), None)])
    assert csf.expand_scales([(None, None)]) is False


def test_static_prepare_host_checks(csf):
    # The allocation-free prepare checks its arguments on the host before any
    # CUDA call: NULLs are refused, and so is a geometry whose look-back words
    # (16 + 8 per 128-row tile) exceed the built-in 256 KiB array.
    fn = csf.lib.csf_prepare_static
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(csf.CStack), ctypes.c_uint64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(None, None, 0, None) == 1
    g = csf.Geometry(0, 8192, 1024, 100)
    st = csf.CStack(g, 256, 256, None, 256, 256, 0, None)
    assert fn(256, ctypes.byref(st), 0, None) == 2
    g = csf.Geometry(0, 4, 64, 8)
    st = csf.CStack(g, 256, 256, None, 256, 256, 0, None)
    assert fn(None, ctypes.byref(st), 0, None) == 1

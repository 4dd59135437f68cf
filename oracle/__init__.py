"""CPU oracle for the CSF scale codec -- TEST INFRASTRUCTURE ONLY.

Plain, slow, single-threaded reference of what the CSF method computes
(encode, decode, routed and row-range decode, decode into the block-scaled
GEMM scale layout, the tile-packed form and its decode, index check), written
in plain C
(``csf_oracle.c``) and reached through ``ctypes``.  Only the test suite, the
smoke check and the benchmark's CPU-baseline leg may import this package.  It
shares no code with the CUDA library, and the product path never routes
through it.

Pages followed (cited by title and paragraph; they have no numbered sections):
  "finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)",
  format and helpers paragraphs; "NVFP4-CSF: expand_scales() for
  ahead-of-call scale expansion (canonical twin of #477)", commit message on
  one-bit MXFP4 and four-bit NVFP4 offsets; "Load native FP4 experts with
  optional lossless CSF scales", encoding plus index paragraph.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

NVFP4 = 0
MXFP4 = 1
OK, ERR_ARG, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no vector intrinsics)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
        os.close(fd)
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.csfo_stream_bytes.argtypes = [ctypes.c_int, _i64, _i64, _i64,
                                          _u64p, _u64p, _u64p, _u64p]
        lib.csfo_stream_bytes.restype = None
        lib.csfo_encode.argtypes = [ctypes.c_int, _i64, _i64, _i64, _u8p,
                                    _u8p, _u8p, _u8p, _u32p, _u8p,
                                    ctypes.c_uint64, _u64p]
        lib.csfo_encode.restype = ctypes.c_int
        lib.csfo_decode.argtypes = [ctypes.c_int, _i64, _i64, _i64, _u8p, _u8p,
                                    _u8p, _u32p, _u8p, ctypes.c_uint64, _i64p,
                                    _i64, _i64, _u8p]
        lib.csfo_decode.restype = ctypes.c_int
        lib.csfo_decode_blocked.argtypes = lib.csfo_decode.argtypes
        lib.csfo_decode_blocked.restype = ctypes.c_int
        lib.csfo_blocked_bytes.argtypes = [_i64, _i64, _i64]
        lib.csfo_blocked_bytes.restype = ctypes.c_uint64
        lib.csfo_tiled_code_bytes.argtypes = [ctypes.c_int, _i64, _i64, _i64]
        lib.csfo_tiled_code_bytes.restype = ctypes.c_uint64
        lib.csfo_tiled_pack.argtypes = [ctypes.c_int, _i64, _i64, _i64, _u8p, _u8p, _u8p, _u32p, _u8p,
                                        ctypes.c_uint64, _u8p, _u8p, _u32p, _u8p, ctypes.c_uint64, _u64p]
        lib.csfo_tiled_pack.restype = ctypes.c_int
        lib.csfo_tiled_decode.argtypes = [ctypes.c_int, _i64, _i64, _i64, _u8p, _u8p, _u32p, _u8p,
                                          ctypes.c_uint64, _i64p, _u8p]
        lib.csfo_tiled_decode.restype = ctypes.c_int
        lib.csfo_check.argtypes = [ctypes.c_int, _i64, _i64, _i64, _u8p, _u8p,
                                   _u32p, ctypes.c_uint64]
        lib.csfo_check.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(typ)


def stream_bytes(kind: int, E: int, R: int, C: int) -> dict:
    """Exact byte lengths of the packed streams (no allocation padding)."""
    vals = [ctypes.c_uint64() for _ in range(4)]
    _load().csfo_stream_bytes(kind, E, R, C, *[ctypes.byref(v) for v in vals])
    ob, eb, bb, ie = (v.value for v in vals)
    return {"offsets": ob, "escapes": eb, "base": bb, "index_entries": ie}


def encode(kind: int, dense: np.ndarray) -> dict:
    """Encode a dense [E, R, C] uint8 stack.  Returns the packed streams."""
    dense = np.ascontiguousarray(dense, dtype=np.uint8)
    E, R, C = dense.shape
    sz = stream_bytes(kind, E, R, C)
    base = np.zeros(sz["base"], np.uint8)
    offsets = np.zeros(sz["offsets"], np.uint8)
    escapes = np.zeros(sz["escapes"], np.uint8)
    index = np.zeros(sz["index_entries"], np.uint32)
    cap = dense.size
    exc = np.zeros(max(cap, 1), np.uint8)
    num = ctypes.c_uint64()
    st = _load().csfo_encode(kind, E, R, C, _ptr(dense, _u8p), _ptr(base, _u8p),
                             _ptr(offsets, _u8p), _ptr(escapes, _u8p),
                             _ptr(index, _u32p), _ptr(exc, _u8p), cap,
                             ctypes.byref(num))
    if st != OK:
        raise RuntimeError(f"oracle encode failed with status {st}")
    return {"kind": kind, "shape": (E, R, C), "base": base, "offsets": offsets,
            "escapes": escapes, "exc_index": index,
            "exc_bytes": exc[:num.value].copy(), "num_exc": num.value}


def decode(enc: dict, expert_start=None, out: np.ndarray | None = None, rows=None):
    """Decode a stack; returns (dense [E, R, C] uint8, status).

    ``expert_start`` (E+1 integers) selects the active experts; planes of
    inactive experts in ``out`` are left as they were.  ``rows`` = (lo, hi)
    writes only rows lo <= r < hi of each selected expert (default: all).
    """
    E, R, C = enc["shape"]
    lo, hi = (0, R) if rows is None else rows
    if out is None:
        out = np.zeros((E, R, C), np.uint8)
    assert out.dtype == np.uint8 and out.shape == (E, R, C)
    es = None
    if expert_start is not None:
        es = np.ascontiguousarray(np.asarray(expert_start, dtype=np.int64))
        assert es.shape == (E + 1,)
    exc = enc["exc_bytes"] if enc["exc_bytes"].size else np.zeros(1, np.uint8)
    st = _load().csfo_decode(enc["kind"], E, R, C, _ptr(enc["base"], _u8p),
                             _ptr(enc["offsets"], _u8p),
                             _ptr(enc["escapes"] if enc["escapes"].size else None, _u8p),
                             _ptr(enc["exc_index"], _u32p), _ptr(exc, _u8p),
                             enc["num_exc"], _ptr(es, _i64p), lo, hi, _ptr(out, _u8p))
    return out, st


def blocked_bytes(E: int, R: int, C: int) -> int:
    """Bytes of a stack in the 128 x 4 tiled scale-operand layout."""
    return int(_load().csfo_blocked_bytes(E, R, C))


def decode_blocked(enc: dict, expert_start=None, out: np.ndarray | None = None, rows=None):
    """Decode into the 128 x 4 tiled scale-operand layout of block-scaled
    GEMMs (flat uint8 of blocked_bytes(E, R, C)); returns (out, status).
    ``rows`` = (lo, hi) with lo a multiple of 128 and hi a multiple of 128 or
    R; tiles outside the selected row blocks and experts keep their bytes."""
    E, R, C = enc["shape"]
    lo, hi = (0, R) if rows is None else rows
    if out is None:
        out = np.zeros(blocked_bytes(E, R, C), np.uint8)
    assert out.dtype == np.uint8 and out.size == blocked_bytes(E, R, C)
    es = None
    if expert_start is not None:
        es = np.ascontiguousarray(np.asarray(expert_start, dtype=np.int64))
        assert es.shape == (E + 1,)
    exc = enc["exc_bytes"] if enc["exc_bytes"].size else np.zeros(1, np.uint8)
    st = _load().csfo_decode_blocked(enc["kind"], E, R, C, _ptr(enc["base"], _u8p),
                                     _ptr(enc["offsets"], _u8p),
                                     _ptr(enc["escapes"] if enc["escapes"].size else None, _u8p),
                                     _ptr(enc["exc_index"], _u32p), _ptr(exc, _u8p),
                                     enc["num_exc"], _ptr(es, _i64p), lo, hi, _ptr(out, _u8p))
    return out, st


def tiled_pack(enc: dict) -> dict:
    """Tile-packed form of a CSF stack (codes, bases and exceptions in the
    order of the block-scaled GEMM scale tiles; see csf_oracle.c)."""
    kind = enc["kind"]
    E, R, C = enc["shape"]
    nrb, ncb = -(-R // 128), -(-C // 4)
    codes = np.zeros(int(_load().csfo_tiled_code_bytes(kind, E, R, C)), np.uint8)
    bases = np.zeros(E * nrb * 128, np.uint8)
    tile_index = np.zeros(E * nrb * ncb + 1, np.uint32)
    cap = max(enc["num_exc"], 1)
    t_exc = np.zeros(cap, np.uint8)
    num = ctypes.c_uint64()
    exc = enc["exc_bytes"] if enc["exc_bytes"].size else np.zeros(1, np.uint8)
    st = _load().csfo_tiled_pack(kind, E, R, C, _ptr(enc["base"], _u8p), _ptr(enc["offsets"], _u8p),
                                 _ptr(enc["escapes"] if enc["escapes"].size else None, _u8p),
                                 _ptr(enc["exc_index"], _u32p), _ptr(exc, _u8p), enc["num_exc"],
                                 _ptr(codes, _u8p), _ptr(bases, _u8p), _ptr(tile_index, _u32p),
                                 _ptr(t_exc, _u8p), cap, ctypes.byref(num))
    if st != OK:
        raise RuntimeError(f"oracle tiled_pack failed with status {st}")
    return {"kind": kind, "shape": (E, R, C), "codes": codes, "bases": bases, "tile_index": tile_index,
            "exc_bytes": t_exc[:num.value].copy(), "num_exc": num.value}


def tiled_decode(tp: dict, expert_start=None, out: np.ndarray | None = None):
    """Decode a tile-packed stack into the block-scaled GEMM scale layout;
    returns (out, status).  Tiles of inactive experts keep their bytes."""
    E, R, C = tp["shape"]
    if out is None:
        out = np.zeros(blocked_bytes(E, R, C), np.uint8)
    es = None
    if expert_start is not None:
        es = np.ascontiguousarray(np.asarray(expert_start, dtype=np.int64))
    exc = tp["exc_bytes"] if tp["exc_bytes"].size else np.zeros(1, np.uint8)
    st = _load().csfo_tiled_decode(tp["kind"], E, R, C, _ptr(tp["codes"], _u8p), _ptr(tp["bases"], _u8p),
                                   _ptr(tp["tile_index"], _u32p), _ptr(exc, _u8p), tp["num_exc"],
                                   _ptr(es, _i64p), _ptr(out, _u8p))
    return out, st


def check(enc: dict) -> int:
    """OK if the index agrees with the escape codes, else ERR_CORRUPT."""
    E, R, C = enc["shape"]
    return _load().csfo_check(enc["kind"], E, R, C, _ptr(enc["offsets"], _u8p),
                              _ptr(enc["escapes"] if enc["escapes"].size else None, _u8p),
                              _ptr(enc["exc_index"], _u32p), enc["num_exc"])

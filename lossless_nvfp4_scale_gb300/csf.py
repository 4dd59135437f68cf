"""Python binding of libcsf.so (the CSF C ABI in include/csf.h).

Argument marshalling only: every step of prepare and decode runs in the CUDA
kernels of the library.  PyTorch supplies device memory and streams.  Importing
this module fails loudly when the compiled library is missing; there is no CPU
fallback.

Typical use::

    stack = csf.prepare(dense_u8_cuda, csf.NVFP4)        # [E, R, C] uint8
    ws = torch.empty_like(dense_u8_cuda)
    csf.decode(stack, ws)                                 # whole stack
    csf.decode(stack, ws, expert_start=start_i32_cuda)    # routed experts only
    csf.decode_pair(gate, down, gate_ws, down_ws, expert_start)
    csf.decode(stack, ws, rows=(0, R // 2))               # gate half of fused gate/up
    sf = csf.decode(stack, layout=csf.LAYOUT_BLOCKED)     # GEMM scale-operand layout
    tp = csf.tiled_pack(stack)                            # stage-readable tile-packed form
    sf = csf.tiled_decode(tp)                             # same bytes as the line above
    sums = csf.tiled_checksums(tp)                        # each tile rebuilt in shared memory only
    ev = csf.expand_scales([(gate, gate_ws), (down, down_ws)], side_stream, after=last_read)
    torch.cuda.current_stream().wait_event(ev)            # before the call that reads them
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

NVFP4 = 0
MXFP4 = 1
DEV_ERR_CORRUPT = 0x1
DEV_ERR_CAPACITY = 0x2
DEV_ERR_TIMEOUT = 0x4
LAYOUT_ROWS = 0      # row-major [E][R][C]
LAYOUT_BLOCKED = 1   # 128 x 4 tiled scale-operand layout of block-scaled GEMMs

_c_i32 = ctypes.c_int32
_c_u64 = ctypes.c_uint64
_c_vp = ctypes.c_void_p


class Geometry(ctypes.Structure):
    """csf_geometry: kind, experts E, rows R per expert, scale bytes C per row."""
    _fields_ = [("kind", _c_i32), ("num_experts", _c_i32), ("rows", _c_i32), ("cols", _c_i32)]


class Sizes(ctypes.Structure):
    """csf_sizes_t: allocation sizes in bytes for one geometry."""
    _fields_ = [("dense", _c_u64), ("base", _c_u64), ("offsets", _c_u64), ("escapes", _c_u64),
                ("exc_index", _c_u64), ("prepare_scratch", _c_u64), ("blocked", _c_u64),
                ("tiled_codes", _c_u64), ("tiled_bases", _c_u64), ("tiled_index", _c_u64)]


class CStack(ctypes.Structure):
    """csf_stack: the device buffers of a compressed stack."""
    _fields_ = [("g", Geometry), ("base", _c_vp), ("offsets", _c_vp), ("escapes", _c_vp),
                ("exc_index", _c_vp), ("exc_bytes", _c_vp), ("num_exc", _c_u64),
                ("error_word", _c_vp)]


class CDecodePart(ctypes.Structure):
    """csf_decode_part: one stack of a row-range or expansion call."""
    _fields_ = [("stack", ctypes.POINTER(CStack)), ("ws", _c_vp), ("ws_bytes", ctypes.c_size_t),
                ("row_lo", _c_i32), ("row_hi", _c_i32), ("layout", _c_i32)]


class CTiled(ctypes.Structure):
    """csf_tiled: the device buffers of a tile-packed stack."""
    _fields_ = [("g", Geometry), ("codes", _c_vp), ("bases", _c_vp), ("tile_index", _c_vp),
                ("exc_bytes", _c_vp), ("num_exc", _c_u64), ("error_word", _c_vp)]


class CsfError(RuntimeError):
    """A csf_* call returned an error status, or its arguments were rejected
    before the call."""


def _load():
    path = os.environ.get("CSF_LIBRARY", _build.LIB)
    if not os.path.exists(path):
        raise CsfError(f"{path} is missing: build it with `python -m lossless_nvfp4_scale_gb300.build` "
                       "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    lib.csf_status_string.argtypes = [ctypes.c_int]
    lib.csf_status_string.restype = ctypes.c_char_p
    lib.csf_abi_version.argtypes = []
    lib.csf_abi_version.restype = ctypes.c_int
    lib.csf_sizes.argtypes = [ctypes.POINTER(Geometry), ctypes.POINTER(Sizes)]
    lib.csf_sizes.restype = ctypes.c_int
    lib.csf_prepare.argtypes = [_c_vp, ctypes.POINTER(CStack), _c_u64, _c_vp, ctypes.c_size_t, _c_vp]
    lib.csf_prepare.restype = ctypes.c_int
    lib.csf_decode.argtypes = [ctypes.POINTER(CStack), _c_vp, ctypes.c_size_t, _c_vp, ctypes.c_int, _c_vp]
    lib.csf_decode.restype = ctypes.c_int
    lib.csf_decode_pair.argtypes = [ctypes.POINTER(CStack), _c_vp, ctypes.c_size_t,
                                    ctypes.POINTER(CStack), _c_vp, ctypes.c_size_t,
                                    _c_vp, ctypes.c_int, _c_vp]
    lib.csf_decode_pair.restype = ctypes.c_int
    lib.csf_decode_rows.argtypes = [ctypes.POINTER(CDecodePart), ctypes.c_int, _c_vp, ctypes.c_int, _c_vp]
    lib.csf_decode_rows.restype = ctypes.c_int
    lib.csf_expand.argtypes = [ctypes.POINTER(CDecodePart), ctypes.c_int, _c_vp, _c_vp, _c_vp]
    lib.csf_expand.restype = ctypes.c_int
    lib.csf_tiled_pack.argtypes = [ctypes.POINTER(CStack), ctypes.POINTER(CTiled), _c_u64, _c_vp]
    lib.csf_tiled_pack.restype = ctypes.c_int
    lib.csf_tiled_decode.argtypes = [ctypes.POINTER(CTiled), _c_vp, ctypes.c_size_t, _c_vp, ctypes.c_int, _c_vp]
    lib.csf_tiled_decode.restype = ctypes.c_int
    lib.csf_tiled_checksum.argtypes = [ctypes.POINTER(CTiled), _c_vp, ctypes.c_size_t, _c_vp, ctypes.c_int, _c_vp]
    lib.csf_tiled_checksum.restype = ctypes.c_int
    lib.csf_selftest_lookback_timeout.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.csf_selftest_lookback_timeout.restype = ctypes.c_int
    return lib


lib = _load()


def _check(status: int, what: str):
    if status != 0:
        raise CsfError(f"{what}: {lib.csf_status_string(status).decode()} (status {status})")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def sizes(kind: int, E: int, R: int, C: int) -> dict:
    """csf_sizes for a geometry, as a dict of field name -> bytes."""
    g = Geometry(kind, E, R, C)
    out = Sizes()
    _check(lib.csf_sizes(ctypes.byref(g), ctypes.byref(out)), "csf_sizes")
    return {f: getattr(out, f) for f, _ in Sizes._fields_}


def _pad16(n: int) -> int:
    return max(16, (n + 15) // 16 * 16)


@dataclass
class Stack:
    """A compressed stack held in device memory (buffers padded as the ABI asks)."""
    kind: int
    E: int
    R: int
    C: int
    base: torch.Tensor
    offsets: torch.Tensor
    escapes: torch.Tensor | None
    exc_index: torch.Tensor     # int32 storage of the uint32 index
    exc_bytes: torch.Tensor
    num_exc: int
    error_word: torch.Tensor    # int32[1]

    @property
    def shape(self):
        return (self.E, self.R, self.C)

    @property
    def dense_bytes(self) -> int:
        return self.E * self.R * self.C

    def stream_bytes(self) -> dict:
        """Exact byte lengths of the packed streams (without allocation padding)."""
        n = self.dense_bytes
        off = (n + 1) // 2 if self.kind == NVFP4 else (n + 7) // 8
        return {"base": self.E * self.R, "offsets": off,
                "escapes": 0 if self.kind == NVFP4 else (n + 7) // 8,
                "exc_index": 4 * (self.E * self.R + 1), "exc_bytes": self.num_exc}

    def cstruct(self) -> CStack:
        return CStack(Geometry(self.kind, self.E, self.R, self.C), self.base.data_ptr(),
                      self.offsets.data_ptr(),
                      self.escapes.data_ptr() if self.escapes is not None else None,
                      self.exc_index.data_ptr(), self.exc_bytes.data_ptr(), self.num_exc,
                      self.error_word.data_ptr())

    def errors(self) -> int:
        """Device error bits (synchronises on the current stream)."""
        return int(self.error_word.item())


def empty_stack(kind: int, E: int, R: int, C: int, exc_capacity: int = 0, device=None) -> Stack:
    """Allocate the buffers of a stack for a geometry (contents undefined)."""
    device = torch.device(device if device is not None else "cuda")
    sz = sizes(kind, E, R, C)
    u8 = dict(dtype=torch.uint8, device=device)
    return Stack(kind, E, R, C,
                 base=torch.empty(_pad16(sz["base"]), **u8),
                 offsets=torch.empty(sz["offsets"], **u8),
                 escapes=torch.empty(sz["escapes"], **u8) if kind == MXFP4 else None,
                 exc_index=torch.empty(E * R + 1, dtype=torch.int32, device=device),
                 exc_bytes=torch.empty(_pad16(exc_capacity), **u8),
                 num_exc=0,
                 error_word=torch.zeros(1, dtype=torch.int32, device=device))


def prepare_scratch(kind: int, E: int, R: int, C: int, device=None) -> torch.Tensor:
    """A device scratch buffer for prepare_async (its contents need no
    initialisation: each prepare clears what it uses on its stream)."""
    n = sizes(kind, E, R, C)["prepare_scratch"]
    return torch.empty(_pad16(n), dtype=torch.uint8, device=device if device is not None else "cuda")


def prepare_async(dense: torch.Tensor, out: Stack, scratch: torch.Tensor, exc_capacity: int | None = None,
                  stream=None) -> None:
    """Launch csf_prepare into `out` (no host sync).  exc_index[rows] holds the
    exception total when it completes."""
    if not dense.is_cuda or dense.dtype != torch.uint8 or not dense.is_contiguous():
        raise CsfError("prepare: dense must be a contiguous uint8 CUDA tensor")
    if dense.numel() != out.dense_bytes:
        raise CsfError("prepare: dense size does not match the stack geometry")
    cap = out.exc_bytes.numel() if exc_capacity is None else exc_capacity
    cs = out.cstruct()
    _check(lib.csf_prepare(dense.data_ptr(), ctypes.byref(cs), cap, scratch.data_ptr(), scratch.numel(),
                           _stream(stream)), "csf_prepare")


def prepare(dense: torch.Tensor, kind: int, stream=None) -> Stack:
    """Encode a dense [E, R, C] uint8 CUDA stack on the GPU.

    One pass over the dense bytes into an exception staging buffer of E*R*C
    bytes, then one 4-byte device-to-host read of the exception total, then a
    copy of the exceptions into an exact-size (16-byte padded) buffer.
    """
    if dense.dim() != 3:
        raise CsfError("prepare: dense must be [E, R, C]")
    E, R, C = (int(x) for x in dense.shape)
    dev = dense.device
    st = empty_stack(kind, E, R, C, exc_capacity=E * R * C, device=dev)
    scratch = prepare_scratch(kind, E, R, C, device=dev)
    prepare_async(dense, st, scratch, stream=stream)
    total = int(st.exc_index[E * R].item()) & 0xFFFFFFFF
    exc = torch.zeros(_pad16(total), dtype=torch.uint8, device=dev)
    exc[:total].copy_(st.exc_bytes[:total])
    st.exc_bytes = exc
    st.num_exc = total
    return st


def upload(enc: dict, device=None) -> Stack:
    """Copy a host-side encoded stack (numpy arrays: base, offsets, escapes,
    exc_index, exc_bytes, num_exc, shape, kind) into padded device buffers."""
    kind = int(enc["kind"])
    E, R, C = enc["shape"]
    st = empty_stack(kind, E, R, C, exc_capacity=int(enc["num_exc"]), device=device)
    st.base.zero_()
    st.offsets.zero_()
    st.exc_bytes.zero_()
    st.base[:E * R].copy_(torch.from_numpy(enc["base"]))
    st.offsets[:enc["offsets"].size].copy_(torch.from_numpy(enc["offsets"]))
    if kind == MXFP4:
        st.escapes.zero_()
        st.escapes[:enc["escapes"].size].copy_(torch.from_numpy(enc["escapes"]))
    st.exc_index.copy_(torch.from_numpy(enc["exc_index"].view("int32")))
    n = int(enc["num_exc"])
    if n:
        st.exc_bytes[:n].copy_(torch.from_numpy(enc["exc_bytes"][:n]))
    st.num_exc = n
    return st


def _es(expert_start):
    if expert_start is None:
        return None, 0
    if not expert_start.is_cuda or expert_start.dtype not in (torch.int32, torch.int64):
        raise CsfError("expert_start must be an int32 or int64 CUDA tensor")
    if not expert_start.is_contiguous():
        raise CsfError("expert_start must be contiguous")
    return expert_start.data_ptr(), 1 if expert_start.dtype == torch.int64 else 0


def _check_es(stack: Stack, expert_start):
    if expert_start is not None and expert_start.numel() != stack.E + 1:
        raise CsfError("expert_start must have E+1 entries")


def blocked_bytes(stack: Stack) -> int:
    """Workspace bytes of a stack in the scale-operand layout (LAYOUT_BLOCKED)."""
    return sizes(stack.kind, stack.E, stack.R, stack.C)["blocked"]


def _ws_for(stack: Stack, ws, what: str, layout: int = LAYOUT_ROWS) -> torch.Tensor:
    if ws is None:
        if layout == LAYOUT_BLOCKED:
            ws = torch.empty(blocked_bytes(stack), dtype=torch.uint8, device=stack.base.device)
        else:
            ws = torch.empty(stack.shape, dtype=torch.uint8, device=stack.base.device)
    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise CsfError(f"{what}: workspaces must be contiguous uint8 CUDA tensors")
    return ws


def _parts(parts, layout=LAYOUT_ROWS):
    """Marshal (stack, ws, (lo, hi) or None) triples into csf_decode_part
    structs; returns the array and the stack structs it points to."""
    cs = [p[0].cstruct() for p in parts]
    arr = (CDecodePart * len(parts))()
    for i, ((stack, ws, rows), c) in enumerate(zip(parts, cs)):
        lo, hi = (0, stack.R) if rows is None else rows
        arr[i] = CDecodePart(ctypes.pointer(c), ws.data_ptr(), ws.numel(), lo, hi, layout)
    return arr, cs


def _decode_rows(parts, expert_start, stream, layout=LAYOUT_ROWS):
    arr, _keep = _parts(parts, layout)
    ptr, is64 = _es(expert_start)
    _check(lib.csf_decode_rows(arr, len(parts), ptr, is64, _stream(stream)), "csf_decode_rows")


def _event_handle(ev, stream) -> int:
    # torch creates the CUDA event at its first record; record it once on the
    # stream that will use it so that a handle exists (a later record or wait
    # through the library supersedes this one).
    if ev.cuda_event == 0:
        ev.record(stream)
    return ev.cuda_event


def expand_scales(parts, stream=None, after: torch.cuda.Event | None = None,
                  done: torch.cuda.Event | None = None, layout: int = LAYOUT_ROWS) -> torch.cuda.Event | bool:
    """Ahead-of-call expansion (csf_expand): decode every expert of the given
    stacks into their workspaces on `stream` (a side stream, typically),
    after `after` (recorded by the previous reader of the workspaces), and
    record `done` for the consumer to wait on.  `layout` = LAYOUT_BLOCKED
    writes the GEMM scale-operand layout.

    `parts` is a list of (stack, ws) or (stack, ws, (lo, hi)); entries whose
    stack is None (scales that are not compressed) are skipped, and False is
    returned when nothing is left to expand."""
    if any(p[0] is not None and p[1] is None for p in parts):
        raise CsfError("expand_scales: every compressed stack needs the workspace it expands into")
    todo = [(p[0], _ws_for(p[0], p[1], "expand_scales", layout), p[2] if len(p) > 2 else None)
            for p in parts if p[0] is not None]
    if not todo:
        return False
    s = stream if stream is not None else torch.cuda.current_stream()
    after_h = None
    if after is not None:
        if after.cuda_event == 0:
            raise CsfError("expand_scales: `after` has never been recorded")
        after_h = after.cuda_event
        s.wait_event(after)        # before the handle record below (csf_expand waits again)
    if done is None:
        done = torch.cuda.Event()
    done_h = _event_handle(done, s)
    for i in range(0, len(todo), 2):
        chunk = todo[i:i + 2]
        arr, _keep = _parts(chunk, layout)
        last = i + 2 >= len(todo)
        _check(lib.csf_expand(arr, len(chunk), after_h if i == 0 else None, done_h if last else None,
                              s.cuda_stream), "csf_expand")
    return done


def decode(stack: Stack, ws: torch.Tensor | None = None, expert_start: torch.Tensor | None = None,
           stream=None, rows: tuple[int, int] | None = None, layout: int = LAYOUT_ROWS) -> torch.Tensor:
    """Decode into `ws` (uint8 CUDA, >= E*R*C bytes, any byte offset).  With
    `expert_start` only experts with routed tokens are written; with
    `rows=(lo, hi)` only rows lo <= r < hi of each of them (csf_decode_rows).
    `layout=LAYOUT_BLOCKED` writes the 128 x 4 tiled scale-operand layout of
    block-scaled GEMMs (flat, blocked_bytes(stack), 16-byte aligned)."""
    ws = _ws_for(stack, ws, "decode", layout)
    _check_es(stack, expert_start)
    if rows is not None or layout != LAYOUT_ROWS:
        _decode_rows([(stack, ws, rows)], expert_start, stream, layout)
        return ws
    ptr, is64 = _es(expert_start)
    cs = stack.cstruct()
    _check(lib.csf_decode(ctypes.byref(cs), ws.data_ptr(), ws.numel(), ptr, is64, _stream(stream)),
           "csf_decode")
    return ws


def decode_pair(gate: Stack, down: Stack, gate_ws: torch.Tensor | None = None,
                down_ws: torch.Tensor | None = None, expert_start: torch.Tensor | None = None,
                stream=None, gate_rows: tuple[int, int] | None = None,
                down_rows: tuple[int, int] | None = None, layout: int = LAYOUT_ROWS):
    """Decode a gate(/up) and a down stack in one launch with shared routing;
    `gate_rows`/`down_rows` restrict each to a row range of every expert."""
    gate_ws = _ws_for(gate, gate_ws, "decode_pair", layout)
    down_ws = _ws_for(down, down_ws, "decode_pair", layout)
    _check_es(gate, expert_start)
    if gate_rows is not None or down_rows is not None or layout != LAYOUT_ROWS:
        _decode_rows([(gate, gate_ws, gate_rows), (down, down_ws, down_rows)], expert_start, stream, layout)
        return gate_ws, down_ws
    ptr, is64 = _es(expert_start)
    g, d = gate.cstruct(), down.cstruct()
    _check(lib.csf_decode_pair(ctypes.byref(g), gate_ws.data_ptr(), gate_ws.numel(),
                               ctypes.byref(d), down_ws.data_ptr(), down_ws.numel(),
                               ptr, is64, _stream(stream)), "csf_decode_pair")
    return gate_ws, down_ws


@dataclass
class Tiled:
    """A tile-packed stack in device memory (csf_tiled: stage-readable, each
    128 x 4 scale tile decodes on its own)."""
    kind: int
    E: int
    R: int
    C: int
    codes: torch.Tensor
    bases: torch.Tensor
    tile_index: torch.Tensor    # int32 storage of the uint32 index
    exc_bytes: torch.Tensor
    num_exc: int
    error_word: torch.Tensor

    @property
    def shape(self):
        return (self.E, self.R, self.C)

    def cstruct(self) -> CTiled:
        return CTiled(Geometry(self.kind, self.E, self.R, self.C), self.codes.data_ptr(), self.bases.data_ptr(),
                      self.tile_index.data_ptr(), self.exc_bytes.data_ptr(), self.num_exc,
                      self.error_word.data_ptr())

    def errors(self) -> int:
        return int(self.error_word.item())


def tiled_pack(stack: Stack, stream=None) -> Tiled:
    """Convert a CSF stack to its tile-packed form on the GPU (csf_tiled_pack)."""
    sz = sizes(stack.kind, stack.E, stack.R, stack.C)
    dev = stack.base.device
    u8 = dict(dtype=torch.uint8, device=dev)
    t = Tiled(stack.kind, stack.E, stack.R, stack.C,
              codes=torch.empty(sz["tiled_codes"], **u8), bases=torch.empty(_pad16(sz["tiled_bases"]), **u8),
              tile_index=torch.empty(sz["tiled_index"] // 4, dtype=torch.int32, device=dev),
              exc_bytes=torch.zeros(_pad16(stack.num_exc), **u8), num_exc=stack.num_exc,
              error_word=torch.zeros(1, dtype=torch.int32, device=dev))
    cs, ct = stack.cstruct(), t.cstruct()
    _check(lib.csf_tiled_pack(ctypes.byref(cs), ctypes.byref(ct), stack.num_exc, _stream(stream)), "csf_tiled_pack")
    return t


def tiled_decode(t: Tiled, ws: torch.Tensor | None = None, expert_start: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Decode a tile-packed stack into the block-scaled GEMM scale layout
    (flat uint8 of csf_sizes().blocked bytes, 16-byte aligned)."""
    if ws is None:
        ws = torch.empty(sizes(t.kind, t.E, t.R, t.C)["blocked"], dtype=torch.uint8, device=t.codes.device)
    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise CsfError("tiled_decode: ws must be a contiguous uint8 CUDA tensor")
    if expert_start is not None and expert_start.numel() != t.E + 1:
        raise CsfError("expert_start must have E+1 entries")
    ptr, is64 = _es(expert_start)
    ct = t.cstruct()
    _check(lib.csf_tiled_decode(ctypes.byref(ct), ws.data_ptr(), ws.numel(), ptr, is64, _stream(stream)),
           "csf_tiled_decode")
    return ws


def tiled_checksums(t: Tiled, sums: torch.Tensor | None = None, expert_start: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Rebuild every tile of a tile-packed stack in shared memory with the
    device decoder of include/csf_tile.cuh (as a GEMM pipeline stage would)
    and return one 32-bit checksum per tile (csf_tiled_checksum): sum of
    w_i * (2i + 1) mod 2^32 over the tile's 128 little-endian words, as int32
    storage of uint32 values [E * T]."""
    tiles = sizes(t.kind, t.E, t.R, t.C)["tiled_index"] // 4 - 1
    if sums is None:
        sums = torch.zeros(tiles, dtype=torch.int32, device=t.codes.device)
    if sums.dtype != torch.int32 or not sums.is_cuda or not sums.is_contiguous():
        raise CsfError("tiled_checksums: sums must be a contiguous int32 CUDA tensor")
    if expert_start is not None and expert_start.numel() != t.E + 1:
        raise CsfError("expert_start must have E+1 entries")
    ptr, is64 = _es(expert_start)
    ct = t.cstruct()
    _check(lib.csf_tiled_checksum(ctypes.byref(ct), sums.data_ptr(), sums.numel(), ptr, is64, _stream(stream)),
           "csf_tiled_checksum")
    return sums


def selftest_lookback_timeout() -> int:
    """Run the library's failure-detection self-test of the prepare's bounded
    look-back wait (a small internal stack whose first tile is never taken) and
    return the device error word of that run; CSF_DEV_ERR_TIMEOUT is set when
    the wait gave up as designed.  Synchronous."""
    word = ctypes.c_uint32(0)
    _check(lib.csf_selftest_lookback_timeout(ctypes.byref(word)), "csf_selftest_lookback_timeout")
    return int(word.value)

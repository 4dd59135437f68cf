"""The stage-readable tile-packed form read per tile, in shared memory.

include/csf_tile.cuh is the device-side decoder a consumer kernel (a GEMM
pipeline stage) calls to rebuild one 128 x 4 tile of scales in shared memory
("NVFP4-CSF: expand_scales() ... (canonical twin of #477)", commit message on
packed experts whose stages rebuild their scales in shared memory).  These
tests (1) build a separate consumer kernel against the header alone
(tests/csf_tile_probe.cu): each warp decodes its tiles into its own shared
buffer and copies them out, and every byte is compared with the oracle's
tile-packed decode, with and without routing (inactive experts left
poisoned); (2) check csf_tiled_checksum, which reads every tile through the
same decoder into shared memory and writes one checksum per tile, against
checksums computed from the oracle's decode.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from lossless_nvfp4_scale_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def csf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_nvfp4_scale_gb300 import build
    build.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf as mod
    return mod


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    from lossless_nvfp4_scale_gb300 import build
    out = str(tmp_path_factory.mktemp("probe") / "libcsf_tile_probe.so")
    subprocess.run([build.nvcc(), *build.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-cudart", "shared", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "csf_tile_probe.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    vp = ctypes.c_void_p
    lib.csf_tile_probe.argtypes = [vp, vp, vp, vp, ctypes.c_uint32, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, vp, ctypes.c_int, vp, vp]
    lib.csf_tile_probe.restype = ctypes.c_int
    return lib


def _dense(kind, E, R, C, seed):
    w = 14 if kind == 0 else 1
    return synth.random_rows(seed, E * R, C, spread=3 * w + 3, replace_p=0.08).reshape(E, R, C)


CASES = [(0, 3, 130, 100), (0, 2, 256, 52), (0, 4, 37, 7), (1, 3, 130, 160), (1, 2, 200, 33), (0, 1, 1, 1)]


@pytest.mark.parametrize("kind,E,R,C", CASES)
@pytest.mark.parametrize("routing", [None, np.int32, np.int64])
def test_device_tile_decoder_in_shared_memory(csf, probe, kind, E, R, C, routing):
    dense = _dense(kind, E, R, C, seed=E * 1000 + C)
    enc = oracle.encode(kind, dense)
    tp_want = oracle.tiled_pack(enc)
    start = None
    if routing is not None:
        start = np.zeros(E + 1, np.int64)
        start[1:] = np.cumsum([(e % 2) * 3 for e in range(E)])         # odd experts active
        start = start.astype(routing)
    want, status = oracle.tiled_decode(tp_want, start, np.full(oracle.blocked_bytes(E, R, C), 0xFF, np.uint8))
    assert status == oracle.OK
    st = csf.prepare(torch.from_numpy(dense).cuda(), kind)
    tp = csf.tiled_pack(st)
    out = torch.full((oracle.blocked_bytes(E, R, C),), 0xFF, dtype=torch.uint8, device="cuda")
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    es = torch.from_numpy(start).cuda() if start is not None else None
    rc = probe.csf_tile_probe(tp.codes.data_ptr(), tp.bases.data_ptr(), tp.tile_index.data_ptr(),
                              tp.exc_bytes.data_ptr(), tp.num_exc, kind, E, R, C,
                              es.data_ptr() if es is not None else None,
                              1 if routing is np.int64 else 0, out.data_ptr(), bad.data_ptr())
    assert rc == 0
    assert int(bad.item()) == 0
    assert np.array_equal(out.cpu().numpy(), want)


def _checksums(blocked: np.ndarray) -> np.ndarray:
    w = blocked.view("<u4").reshape(-1, 128).astype(np.uint64)
    k = 2 * np.arange(128, dtype=np.uint64) + 1
    return ((w * k).sum(axis=1) & 0xFFFFFFFF).astype(np.uint32)


@pytest.mark.parametrize("kind,E,R,C", CASES + [(0, 512, 1024, 100)])
def test_tiled_checksums_match_the_oracle(csf, kind, E, R, C):
    dense = synth.gate_stack(seed=4) if E == 512 else _dense(kind, E, R, C, seed=7 + C)
    enc = oracle.encode(kind, dense)
    blocked, status = oracle.decode_blocked(enc)
    assert status == oracle.OK
    want = _checksums(blocked)
    tp = csf.tiled_pack(csf.prepare(torch.from_numpy(dense).cuda(), kind))
    got = csf.tiled_checksums(tp).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, want)
    # routed: only active experts' entries are written
    start = synth.routing(E=E, active=min(E, 3), tokens=10, seed=C).astype(np.int32)
    sums = torch.full((want.size,), -1, dtype=torch.int32, device="cuda")
    csf.tiled_checksums(tp, sums, expert_start=torch.from_numpy(start).cuda())
    got = sums.cpu().numpy().view(np.uint32).reshape(E, -1)
    active = start[1:] > start[:-1]
    assert np.array_equal(got[active], want.reshape(E, -1)[active])
    assert (got[~active] == 0xFFFFFFFF).all()
    assert tp.errors() == 0

"""GPU parity of the tile-packed (stage-readable) CSF form: the GPU
conversion from a CSF stack against the oracle's packing (every byte of
codes, bases, tile index and exception stream), and the GPU decode into the
block-scaled GEMM scale layout against the oracle (also with routing)."""
import numpy as np
import pytest
import torch

import oracle
from lossless_nvfp4_scale_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_nvfp4_scale_gb300 import build
    build.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf as mod
    return mod


def _check_pack(csf, t, tp):
    assert np.array_equal(t.codes.cpu().numpy(), tp["codes"])
    assert np.array_equal(t.bases[:tp["bases"].size].cpu().numpy(), tp["bases"])
    assert np.array_equal(t.tile_index.cpu().numpy().view(np.uint32), tp["tile_index"])
    assert np.array_equal(t.exc_bytes[:tp["num_exc"]].cpu().numpy(), tp["exc_bytes"])


SHAPES = [(0, 1, 1, 1), (0, 2, 128, 4), (0, 3, 200, 7), (0, 2, 256, 100), (0, 3, 300, 50), (0, 2, 130, 600),
          (1, 2, 130, 160), (1, 3, 64, 33), (1, 2, 512, 160), (1, 2, 100, 17), (0, 4, 37, 99)]


@pytest.mark.parametrize("kind,E,R,C", SHAPES)
@pytest.mark.parametrize("routed", [False, np.int64, np.int32])
def test_tiled_pack_and_decode(csf, kind, E, R, C, routed):
    w = 14 if kind == 0 else 1
    dense = synth.random_rows(E + R + C, E * R, C, spread=w + 5, replace_p=0.1).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    tp = oracle.tiled_pack(enc)
    up = csf.upload(enc)
    t = csf.tiled_pack(up)
    torch.cuda.synchronize()
    assert t.errors() == 0
    _check_pack(csf, t, tp)
    nb = oracle.blocked_bytes(E, R, C)
    start = None
    if routed:
        start = np.concatenate([[0], np.cumsum((np.arange(E) % 2 == 0) * 3)]).astype(routed)
    ws = torch.full((nb,), 0xA5, dtype=torch.uint8, device="cuda")
    csf.tiled_decode(t, ws, expert_start=None if start is None else torch.from_numpy(start).cuda())
    want, st = oracle.tiled_decode(tp, start, np.full(nb, 0xA5, np.uint8))
    assert st == oracle.OK
    assert np.array_equal(ws.cpu().numpy(), want)
    assert t.errors() == 0


def test_tiled_full_gate(csf):
    dense = synth.stack("gate")
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    t = csf.tiled_pack(up)
    sf = csf.tiled_decode(t)
    want, _ = oracle.decode_blocked(enc)
    assert np.array_equal(sf.cpu().numpy(), want)
    # The same bytes as the blocked-layout decode of the CSF stack itself.
    assert torch.equal(sf, csf.decode(up, layout=csf.LAYOUT_BLOCKED))
    assert t.errors() == 0 and up.errors() == 0


def test_tiled_corrupt_inputs_set_the_error_word(csf):
    dense = _d = synth.random_rows(3, 4 * 64, 8, spread=19, replace_p=0.08).reshape(4, 64, 8)
    enc = oracle.encode(0, dense)
    bad = dict(enc)
    bad["exc_index"] = enc["exc_index"].copy()
    bad["exc_index"][100:] += 1                     # CSF index off by one from row 100
    t = csf.tiled_pack(csf.upload(bad))
    torch.cuda.synchronize()
    assert t.errors() & csf.DEV_ERR_CORRUPT
    good = csf.tiled_pack(csf.upload(enc))
    idx = good.tile_index.clone()
    good.tile_index[1:] += 1                        # tile index off by one: decode reports it
    csf.tiled_decode(good)
    assert good.errors() & csf.DEV_ERR_CORRUPT
    good.tile_index.copy_(idx)
    good.error_word.zero_()
    csf.tiled_decode(good)
    assert good.errors() == 0


@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_tiled_decode_no_active_expert_writes_nothing(csf, dtype):
    dense = synth.random_rows(5, 3 * 130, 20, spread=19, replace_p=0.1).reshape(3, 130, 20)
    enc = oracle.encode(0, dense)
    t = csf.tiled_pack(csf.upload(enc))
    nb = oracle.blocked_bytes(3, 130, 20)
    ws = torch.full((nb,), 0x5A, dtype=torch.uint8, device="cuda")
    start = torch.from_numpy(np.full(4, 7, dtype)).cuda()
    csf.tiled_decode(t, ws, expert_start=start)
    assert bool((ws == 0x5A).all())
    assert t.errors() == 0

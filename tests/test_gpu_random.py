"""Randomised GPU parity: many seeded configurations at once.

Each case draws a kind, a geometry (ragged rows and columns, R below and above
the unit and tile sizes), a routing prefix (int32 or int64, empty, full or
sparse), a row range, an output layout and a workspace byte offset, decodes
through the C ABI into a poisoned workspace, and compares every byte with the
oracle (prepare is compared too).  Bit-exact: integer byte work.
"""
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


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    kind = int(rng.integers(0, 2))
    E = int(rng.integers(1, 9))
    R = int(rng.choice([1, 3, 16, 37, 64, 128, 130, 200, 256, 300]))
    C = int(rng.choice([1, 2, 3, 7, 8, 17, 31, 32, 33, 50, 63, 64, 65, 100, 128, 160, 255, 300]))
    w = 14 if kind == 0 else 1
    dense = synth.random_rows(seed, E * R, C, spread=int(rng.integers(w, 3 * w + 4)),
                              replace_p=float(rng.choice([0.0, 0.02, 0.1, 0.4]))).reshape(E, R, C)
    mode = rng.choice(["all", "none", "sparse", "first_last"])
    counts = {"all": np.ones(E), "none": np.zeros(E), "sparse": (rng.random(E) < 0.4).astype(float),
              "first_last": np.r_[1, np.zeros(max(E - 2, 0)), 1][:E]}[mode]
    start = np.concatenate([[0], np.cumsum(counts * rng.integers(1, 5, size=E))]).astype(np.int64)
    routed = bool(rng.integers(0, 2))
    layout = int(rng.integers(0, 2))
    if layout == 1:
        blocks = -(-R // 128)
        b0 = int(rng.integers(0, blocks))
        b1 = int(rng.integers(b0 + 1, blocks + 1))
        rows = (128 * b0, min(128 * b1, R)) if rng.random() < 0.6 else None
    else:
        lo = int(rng.integers(0, R))
        rows = (lo, int(rng.integers(lo + 1, R + 1))) if rng.random() < 0.6 else None
    offset = 0 if layout == 1 else int(rng.choice([0, 1, 3, 16]))
    return kind, dense, (start if routed else None), rng.choice([np.int32, np.int64]), rows, layout, offset


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration(csf, seed):
    kind, dense, start, itype, rows, layout, offset = _case(seed)
    E, R, C = dense.shape
    enc = oracle.encode(kind, dense)
    if seed % 4 == 0:   # GPU prepare against the oracle's streams
        st = csf.prepare(torch.from_numpy(dense).cuda(), kind)
        assert st.num_exc == enc["num_exc"]
        assert np.array_equal(st.exc_index.cpu().numpy().view(np.uint32), enc["exc_index"])
    up = csf.upload(enc)
    es = None if start is None else torch.from_numpy(start.astype(itype)).cuda()
    if layout == 1:
        n = oracle.blocked_bytes(E, R, C)
        ws = torch.full((n,), 0xA7, dtype=torch.uint8, device="cuda")
        csf.decode(up, ws, expert_start=es, rows=rows, layout=csf.LAYOUT_BLOCKED)
        want, st_ = oracle.decode_blocked(enc, start, np.full(n, 0xA7, np.uint8), rows=rows)
        got = ws.cpu().numpy()
    else:
        n = dense.size
        buf = torch.full((n + 32,), 0xA7, dtype=torch.uint8, device="cuda")
        csf.decode(up, buf[offset:offset + n], expert_start=es, rows=rows)
        want, st_ = oracle.decode(enc, start, np.full(dense.shape, 0xA7, np.uint8), rows=rows)
        host = buf.cpu().numpy()
        assert (host[:offset] == 0xA7).all() and (host[offset + n:] == 0xA7).all()
        got = host[offset:offset + n].reshape(dense.shape)
    assert st_ == oracle.OK
    assert np.array_equal(got, want), (kind, dense.shape, rows, layout, offset)
    assert up.errors() == 0

"""Parity beyond 2^32 elements: the seeded 512 x 1024 x 100 gate stack
repeated 84 times along the expert axis (43,008 experts, 4.40e9 scales, rows
and element offsets past 32 bits).  Every repeat encodes like the first, so
the oracle's encoding of one block pins the GPU prepare's streams at the far
end of the stack (index entries, bases, offsets, exception bytes of the last
block); the row-major decode must give back the whole dense stack, and the
blocked-layout decode of the last expert must match the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from lossless_nvfp4_scale_gb300 import synth

pytestmark = pytest.mark.gpu

REPEATS = 84


@pytest.fixture(scope="module")
def csf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_nvfp4_scale_gb300 import build
    build.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf as mod
    return mod


def test_stack_past_2_32_elements(csf):
    block = synth.stack("gate")                                  # 512 x 1024 x 100
    Eb, R, C = block.shape
    enc = oracle.encode(oracle.NVFP4, block)
    E = Eb * REPEATS
    assert E * R * C > 1 << 32
    dense = torch.from_numpy(block).cuda().repeat(REPEATS, 1, 1)
    st = csf.prepare(dense, csf.NVFP4)
    torch.cuda.synchronize()
    assert st.errors() == 0
    ne, rb = enc["num_exc"], Eb * R
    assert st.num_exc == REPEATS * ne
    idx = st.exc_index
    for j in (1, REPEATS // 2, REPEATS - 1, REPEATS):
        assert (int(idx[j * rb].item()) & 0xFFFFFFFF) == j * ne
    last = REPEATS - 1
    nb = block.size // 2                                         # offset bytes per block
    assert np.array_equal(st.base[last * rb:(last + 1) * rb].cpu().numpy(), enc["base"])
    assert np.array_equal(st.offsets[last * nb:(last + 1) * nb].cpu().numpy(), enc["offsets"])
    assert np.array_equal(st.exc_bytes[last * ne:(last + 1) * ne].cpu().numpy(), enc["exc_bytes"])
    want_idx = enc["exc_index"][:-1].astype(np.int64) + last * ne
    got_idx = idx[last * rb:(last + 1) * rb].cpu().numpy().view(np.uint32).astype(np.int64)
    assert np.array_equal(got_idx, want_idx)
    ws = csf.decode(st)
    assert torch.equal(ws, dense)
    del ws
    sf = csf.decode(st, layout=csf.LAYOUT_BLOCKED)
    per = oracle.blocked_bytes(1, R, C)
    one = oracle.encode(oracle.NVFP4, block[-1:])
    want, status = oracle.decode_blocked(one)
    assert status == oracle.OK
    assert np.array_equal(sf[(E - 1) * per:].cpu().numpy(), want)
    assert st.errors() == 0

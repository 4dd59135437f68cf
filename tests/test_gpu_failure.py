"""Failure detection on the GPU without a fault: the prepare's decoupled
look-back wait is bounded, and when it runs out (a status word that nothing
writes) the kernel reports CSF_DEV_ERR_TIMEOUT through the device error word
and finishes; the context stays usable for the next prepare and decode."""
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


def test_lookback_wait_gives_up_and_reports(csf):
    word = csf.selftest_lookback_timeout()
    assert word & csf.DEV_ERR_TIMEOUT
    assert not word & ~(csf.DEV_ERR_TIMEOUT | csf.DEV_ERR_CORRUPT | csf.DEV_ERR_CAPACITY)
    # The context still works: a prepare and a decode right after match the oracle.
    dense = synth.stack("tiny")
    st = csf.prepare(torch.from_numpy(dense).cuda(), csf.NVFP4)
    ws = csf.decode(st)
    torch.cuda.synchronize()
    assert st.errors() == 0
    assert np.array_equal(ws.cpu().numpy(), dense)
    enc = oracle.encode(oracle.NVFP4, dense)
    assert np.array_equal(st.exc_index.cpu().numpy().view(np.uint32), enc["exc_index"])

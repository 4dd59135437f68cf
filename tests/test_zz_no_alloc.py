"""csf_prepare_static: GPU prepare for callers that cannot allocate.

Some users of this library cannot call cudaMalloc (a plugin whose host process
owns all device memory, code where an allocation would synchronise the device
or disturb a stream capture).  csf_prepare_static keeps the prepare kernel's
scratch in a device array inside the library instead of taking a scratch
buffer.  These tests call it through the C ABI and require the same bytes as
the existing csf_prepare entry point (bit-exact, the bar of every test here),
on two calls in a row, since every call reuses the one built-in array.

This file is collected last, so a run that stops at the first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import ctypes

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
    fn = mod.lib.csf_prepare_static
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(mod.CStack), ctypes.c_uint64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return mod


def _np(t):
    return t.detach().cpu().numpy()


def _static_prepare(csf, dense, kind):
    E, R, C = (int(x) for x in dense.shape)
    st = csf.empty_stack(kind, E, R, C, exc_capacity=E * R * C)
    for t in (st.base, st.offsets, st.exc_bytes) + ((st.escapes,) if st.escapes is not None else ()):
        t.fill_(0xEE)                                   # outputs start as garbage
    st.exc_index.fill_(-1)
    cs = st.cstruct()
    rc = csf.lib.csf_prepare_static(dense.data_ptr(), ctypes.byref(cs), st.exc_bytes.numel(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == 0, csf.lib.csf_status_string(rc).decode()
    torch.cuda.synchronize()
    st.num_exc = int(st.exc_index[E * R].item()) & 0xFFFFFFFF
    return st


@pytest.mark.parametrize("kind,shape", [(0, (4, 64, 8)), (0, (5, 37, 100)), (1, (2, 37, 160)),
                                        (0, (512, 1024, 100)), (1, (384, 2048, 160))])
def test_static_prepare_matches_prepare_on_two_calls(csf, kind, shape):
    if shape[0] >= 384:
        dense_np = synth.gate_stack(seed=3) if kind == 0 else synth.mxfp4_stack(seed=3)
    else:
        w = 14 if kind == 0 else 1
        dense_np = synth.random_rows(11, shape[0] * shape[1], shape[2], spread=3 * w + 3,
                                     replace_p=0.08).reshape(shape)
    dense = torch.from_numpy(dense_np).cuda()
    ref = csf.prepare(dense, kind)                     # the existing entry point
    sb = ref.stream_bytes()
    if shape[0] < 384:
        # small stacks: the existing entry point's streams are also the oracle's
        enc = oracle.encode(kind, dense_np)
        assert ref.num_exc == enc["num_exc"]
        assert np.array_equal(_np(ref.offsets[:enc["offsets"].size]), enc["offsets"])
        assert np.array_equal(_np(ref.exc_bytes[:ref.num_exc]), enc["exc_bytes"][:enc["num_exc"]])
    for call in range(2):
        st = _static_prepare(csf, dense, kind)
        assert st.errors() == 0, f"call {call}: device error {st.errors():#x}"
        assert st.num_exc == ref.num_exc
        assert np.array_equal(_np(st.base[:sb["base"]]), _np(ref.base[:sb["base"]]))
        assert np.array_equal(_np(st.offsets), _np(ref.offsets))
        if kind == 1:
            assert np.array_equal(_np(st.escapes), _np(ref.escapes))
        assert np.array_equal(_np(st.exc_index), _np(ref.exc_index))
        assert np.array_equal(_np(st.exc_bytes[:st.num_exc]), _np(ref.exc_bytes[:ref.num_exc]))
        ws = csf.decode(st)
        assert torch.equal(ws, dense)


def test_static_prepare_rejects_geometry_beyond_builtin_scratch(csf):
    # 8192 x 1024 rows of 100 bytes need more than 256 KiB of look-back words.
    # The call must refuse before touching any pointer or the device.
    g = csf.Geometry(0, 8192, 1024, 100)
    st = csf.CStack(g, 256, 256, None, 256, 256, 0, None)
    rc = csf.lib.csf_prepare_static(256, ctypes.byref(st), 0, None)
    assert rc == 2 and csf.lib.csf_status_string(rc).decode() == "buffer too small"

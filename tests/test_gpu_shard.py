"""Expert-range split of one stack (the multi-GPU partition), on one GPU.

The codec shards along the expert axis with no exchange step ("Load native FP4
experts with optional lossless CSF scales": tensor-parallel workers compress
their slices independently).  Each rank prepares the sub-stack of its
contiguous experts [e0, e1) and decodes it with the routing view
expert_start[e0 : e1 + 1].  These tests run the two shards of a 2-way split
one after the other on one GPU -- the kernels of the two ranks never wait on
one another, so nothing needs two GPUs -- and require every byte of each
shard's decode, in a 0xFF-poisoned workspace, to equal the matching slice of
the oracle's decode of the WHOLE stack under the same routing.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_nvfp4_scale_gb300 import shard, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lossless_nvfp4_scale_gb300 import build
    build.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf as mod
    return mod


@pytest.fixture(scope="module")
def gate():
    dense = synth.gate_stack(seed=0)
    return dense, oracle.encode(oracle.NVFP4, dense)


def _routings(E):
    eight = synth.routing(E=E, active=8, tokens=64, seed=0)
    # experts on both sides of the split boundary E/2 active, and the boundary itself
    edge = np.zeros(E + 1, np.int64)
    counts = np.zeros(E, np.int64)
    counts[[0, E // 2 - 1, E // 2, E // 2 + 1, E - 1]] = [3, 1, 2, 5, 1]
    np.cumsum(counts, out=edge[1:])
    return {"8of512": eight, "boundary": edge}


@pytest.mark.parametrize("world", [2, 3])
def test_shards_full_decode_equal_slices(csf, gate, world):
    dense, _ = gate
    d = torch.from_numpy(dense).cuda()
    seen = []
    for rank in range(world):
        st, e0, e1 = shard.prepare_shard(d, csf.NVFP4, world, rank)
        seen.append((e0, e1))
        assert st.shape == (e1 - e0, 1024, 100) and st.errors() == 0
        ws = csf.decode(st)
        assert torch.equal(ws, d[e0:e1])
    assert seen[0][0] == 0 and seen[-1][1] == 512
    assert all(a[1] == b[0] for a, b in zip(seen, seen[1:]))


@pytest.mark.parametrize("route", ["8of512", "boundary"])
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_shards_routed_decode_equal_slices_of_whole_routed_decode(csf, gate, route, dtype):
    dense, enc = gate
    E = dense.shape[0]
    start = _routings(E)[route].astype(dtype)
    poison = np.full(dense.shape, 0xFF, np.uint8)
    want, status = oracle.decode(enc, start.astype(np.int64), poison)
    assert status == oracle.OK
    d = torch.from_numpy(dense).cuda()
    start_d = torch.from_numpy(start).cuda()
    for rank in range(2):
        st, e0, e1 = shard.prepare_shard(d, csf.NVFP4, 2, rank)
        # the shard's streams are the oracle's encoding of its sub-stack
        sub = oracle.encode(oracle.NVFP4, dense[e0:e1])
        assert st.num_exc == sub["num_exc"]
        assert np.array_equal(st.exc_index.cpu().numpy().view(np.uint32), sub["exc_index"])
        view = shard.routing_view(start_d, e0, e1)
        assert view.data_ptr() == start_d.data_ptr() + e0 * start_d.element_size()
        ws = torch.full((e1 - e0, 1024, 100), 0xFF, dtype=torch.uint8, device="cuda")
        csf.decode(st, ws, expert_start=view)
        assert np.array_equal(ws.cpu().numpy(), want[e0:e1]), f"rank {rank} ({e0}, {e1})"
        assert st.errors() == 0


def test_shard_pair_decode_with_routing_view(csf, gate):
    # gate and down shards of the same expert range decode in one paired
    # launch with the shared routing view.
    dense, enc = gate
    down = synth.down_stack(seed=0)
    start = synth.routing(E=512, active=8, tokens=64, seed=1)
    want_g, sg = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
    want_d, sd = oracle.decode(oracle.encode(oracle.NVFP4, down), start, np.full(down.shape, 0xFF, np.uint8))
    assert sg == oracle.OK and sd == oracle.OK
    dg, dd = torch.from_numpy(dense).cuda(), torch.from_numpy(down).cuda()
    start_d = torch.from_numpy(start).cuda()
    for rank in range(2):
        g, e0, e1 = shard.prepare_shard(dg, csf.NVFP4, 2, rank)
        dn, f0, f1 = shard.prepare_shard(dd, csf.NVFP4, 2, rank)
        assert (e0, e1) == (f0, f1)
        gw = torch.full((e1 - e0, 1024, 100), 0xFF, dtype=torch.uint8, device="cuda")
        dw = torch.full((e1 - e0, 2048, 50), 0xFF, dtype=torch.uint8, device="cuda")
        csf.decode_pair(g, dn, gw, dw, expert_start=shard.routing_view(start_d, e0, e1))
        assert np.array_equal(gw.cpu().numpy(), want_g[e0:e1])
        assert np.array_equal(dw.cpu().numpy(), want_d[e0:e1])

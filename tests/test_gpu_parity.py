"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer byte work, so the bar is bit-exact everywhere.  Inputs are the seeded
synthetic stacks of lossless_nvfp4_scale_gb300.synth; expected values come
from the oracle only.  Covers small ragged geometries (several work units,
ragged tails, odd C, C < chunk), the full-size stacks of the pages' workloads
(512 x 1024 x 100 gate, 512 x 2048 x 50 down, 384 x 2048 x 160 MXFP4) in the
launch configuration the benchmark times, routed decode into a poisoned
workspace, row-range decode (the gate half of a fused gate/up stack), paired
decode, odd-offset workspaces with guard bytes, CUDA-graph
replay, both routing integer types, and corrupt or over-capacity inputs
(planted on the CPU) reported through the device error word.
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


def _np(t):
    return t.detach().cpu().numpy()


def assert_stack_matches(st, enc):
    E, R, C = enc["shape"]
    sb = st.stream_bytes()
    assert st.num_exc == enc["num_exc"]
    assert np.array_equal(_np(st.base[:E * R]), enc["base"])
    assert np.array_equal(_np(st.offsets[:sb["offsets"]]), enc["offsets"])
    if enc["kind"] == oracle.MXFP4:
        assert np.array_equal(_np(st.escapes[:sb["escapes"]]), enc["escapes"])
    assert np.array_equal(_np(st.exc_index).view(np.uint32), enc["exc_index"])
    assert np.array_equal(_np(st.exc_bytes[:st.num_exc]), enc["exc_bytes"])
    # Allocation padding past the stream is written as zeros.
    assert not _np(st.offsets[sb["offsets"]:]).any()


def _dense_cuda(dense):
    return torch.from_numpy(dense).cuda()


def test_tiny_workload_seed0_round_trip(csf):
    # The 4 x 64 x 8 NVFP4 workload (base U[0x20,0x60], offsets U{0..14}, 3%
    # random bytes, seed 0): GPU encode and decode against the oracle.
    dense = synth.stack("tiny")
    enc = oracle.encode(0, dense)
    st = csf.prepare(_dense_cuda(dense), 0)
    assert st.errors() == 0
    assert_stack_matches(st, enc)
    assert np.array_equal(_np(csf.decode(st)), dense)
    assert np.array_equal(_np(csf.decode(csf.upload(enc))), dense)


SMALL = [
    (0, 1, 1, 1), (0, 1, 1, 31), (0, 3, 5, 7), (0, 2, 33, 17), (0, 5, 37, 100), (0, 7, 13, 3),
    (0, 4, 64, 8), (0, 3, 40, 64), (0, 2, 3, 1000), (0, 5, 37, 50), (0, 3, 41, 33), (0, 2, 9, 63),
    (1, 1, 1, 1), (1, 3, 5, 7), (1, 2, 37, 160), (1, 4, 9, 33), (1, 3, 11, 128), (1, 2, 5, 500),
]


def _small_dense(kind, E, R, C, seed):
    w = 14 if kind == 0 else 1
    return synth.random_rows(seed, E * R, C, spread=3 * w + 3, replace_p=0.08).reshape(E, R, C)


@pytest.mark.parametrize("kind,E,R,C", SMALL)
def test_prepare_and_decode_small(csf, kind, E, R, C):
    dense = _small_dense(kind, E, R, C, seed=E * 1000 + R * 10 + C)
    enc = oracle.encode(kind, dense)
    st = csf.prepare(_dense_cuda(dense), kind)
    torch.cuda.synchronize()
    assert st.errors() == 0
    assert_stack_matches(st, enc)
    # Decode the oracle's stream (independent of the GPU prepare).
    up = csf.upload(enc)
    ws = torch.full(dense.shape, 0x5A, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws)
    assert np.array_equal(_np(ws), dense)
    assert up.errors() == 0


@pytest.mark.parametrize("kind,E,R,C", [(0, 6, 5, 7), (0, 5, 37, 100), (1, 6, 9, 33), (1, 4, 37, 160),
                                        (0, 9, 13, 3)])
@pytest.mark.parametrize("is64", [False, True])
def test_routed_small_poisoned(csf, kind, E, R, C, is64):
    dense = _small_dense(kind, E, R, C, seed=7 + C)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    counts = np.zeros(E, np.int64)
    counts[[0, E // 2, E - 1]] = [2, 1, 3]          # first, middle and last experts
    start = np.concatenate([[0], np.cumsum(counts)])
    es = torch.from_numpy(start.astype(np.int64 if is64 else np.int32)).cuda()
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws, expert_start=es)
    want, st = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
    assert st == oracle.OK
    assert np.array_equal(_np(ws), want)
    assert up.errors() == 0


@pytest.mark.parametrize("kind,E,R,C", [(0, 12, 32, 100), (0, 7, 64, 50), (1, 10, 8, 160), (0, 6, 5, 7)])
def test_routed_runs_of_consecutive_experts(csf, kind, E, R, C):
    # Runs of consecutive active experts (one segment may run through a run
    # when experts start on unit boundaries), with gaps, at both ends, and
    # with a warp range that ends inside a run.
    dense = _small_dense(kind, E, R, C, seed=E + R + C)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    patterns = [np.ones(E, np.int64), np.r_[np.ones(3), np.zeros(1), np.ones(E - 4)],
                np.r_[np.zeros(1), np.ones(E - 2), np.zeros(1)], (np.arange(E) % 3 != 1).astype(np.int64)]
    for counts in patterns:
        start = np.concatenate([[0], np.cumsum(counts.astype(np.int64))])
        ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
        csf.decode(up, ws, expert_start=torch.from_numpy(start).cuda())
        want, _ = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
        assert np.array_equal(_np(ws), want), counts
    assert up.errors() == 0


@pytest.mark.parametrize("E", [1300, 8192])
def test_routed_many_experts_varying_units(csf, E):
    # Experts whose unit counts differ (R not a multiple of the unit rows)
    # keep per-expert prefix arrays in shared memory: 12*E + 8 bytes on top of
    # the static staging buffers, past the default 48 KB window at E = 1300.
    R, C = 5, 7
    dense = _small_dense(0, E, R, C, seed=E)
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    counts = np.zeros(E, np.int64)
    counts[np.arange(0, E, 97)] = 1
    counts[E - 1] = 2
    start = np.concatenate([[0], np.cumsum(counts)])
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws, expert_start=torch.from_numpy(start.astype(np.int32)).cuda())
    want, _ = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
    assert np.array_equal(_np(ws), want)
    assert up.errors() == 0


def test_routed_edge_cases(csf):
    dense = _small_dense(0, 8, 16, 100, seed=3)
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    E = 8
    cases = {
        "none": np.zeros(E + 1, np.int64),
        "all": np.arange(E + 1, dtype=np.int64),
        "last": np.concatenate([np.zeros(E, np.int64), [5]]),
        "zero-length groups": np.array([0, 0, 4, 4, 4, 9, 9, 9, 9], np.int64),
        "decreasing": np.array([5, 3, 4, 4, -1, 0, 0, 2, 2], np.int64),
    }
    for name, start in cases.items():
        ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
        csf.decode(up, ws, expert_start=torch.from_numpy(start.astype(np.int32)).cuda())
        want, _ = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
        assert np.array_equal(_np(ws), want), name


# Rows per expert that are (second line) and are not (first line) a multiple
# of the rows of one work unit: equal or varying unit counts per expert.
ROW_RANGE_SHAPES = [(0, 5, 10, 7), (0, 4, 38, 100), (0, 3, 12, 50), (0, 6, 9, 3), (1, 4, 10, 33),
                    (1, 3, 38, 160),
                    (0, 4, 32, 100), (0, 5, 64, 50), (0, 3, 64, 8), (1, 3, 8, 160), (1, 2, 128, 33)]


@pytest.mark.parametrize("kind,E,R,C", ROW_RANGE_SHAPES)
@pytest.mark.parametrize("routed", [False, True])
def test_row_range_small_poisoned(csf, kind, E, R, C, routed):
    # Rows [lo, hi) of each (routed) expert against the oracle, into a
    # poisoned workspace: halves of a fused gate/up expert, single rows at
    # either end, a range that starts mid-unit, and the whole expert.
    dense = _small_dense(kind, E, R, C, seed=11 + C + R)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    start = None
    if routed:
        counts = np.zeros(E, np.int64)
        counts[[0, E - 1]] = [3, 1]
        start = np.concatenate([[0], np.cumsum(counts)])
    es = None if start is None else torch.from_numpy(start.astype(np.int32)).cuda()
    for lo, hi in [(0, R // 2), (R // 2, R), (0, 1), (R - 1, R), (1, R - 1), (3, 7), (0, R)]:
        ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
        csf.decode(up, ws, expert_start=es, rows=(lo, hi))
        want, st = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8), rows=(lo, hi))
        assert st == oracle.OK
        assert np.array_equal(_np(ws), want), (lo, hi)
    assert up.errors() == 0


@pytest.mark.parametrize("offset", [0, 1, 16])
@pytest.mark.parametrize("routed", [False, True])
@pytest.mark.parametrize("I,Rd", [(19, 37), (16, 64), (16, 37)])
def test_row_range_pair_gate_half_and_down(csf, offset, routed, I, Rd):
    # A fused gate/up stack (R = 2*I rows per expert) decodes only its gate
    # half [0, I) while the down stack decodes whole, in one launch, into
    # odd-offset workspaces with guard bytes.
    E = 6
    gu = _small_dense(0, E, 2 * I, 100, seed=5)
    dn = _small_dense(0, E, Rd, 50, seed=6)
    genc, denc = oracle.encode(0, gu), oracle.encode(0, dn)
    g_up, d_up = csf.upload(genc), csf.upload(denc)
    start = np.array([0, 2, 2, 5, 5, 5, 6], np.int64) if routed else None
    es = None if start is None else torch.from_numpy(start).cuda()
    gbuf = torch.full((gu.size + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    dbuf = torch.full((dn.size + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    gws, dws = gbuf[offset:offset + gu.size], dbuf[offset:offset + dn.size]
    csf.decode_pair(g_up, d_up, gws, dws, expert_start=es, gate_rows=(0, I))
    gwant, _ = oracle.decode(genc, start, np.full(gu.shape, 0xAB, np.uint8), rows=(0, I))
    dwant, _ = oracle.decode(denc, start, np.full(dn.shape, 0xAB, np.uint8))
    gh, dh = _np(gbuf), _np(dbuf)
    assert np.array_equal(gh[offset:offset + gu.size], gwant.ravel())
    assert np.array_equal(dh[offset:offset + dn.size], dwant.ravel())
    assert (gh[:offset] == 0xAB).all() and (gh[offset + gu.size:] == 0xAB).all()
    assert (dh[:offset] == 0xAB).all() and (dh[offset + dn.size:] == 0xAB).all()
    assert g_up.errors() == 0 and d_up.errors() == 0


@pytest.mark.parametrize("shift", [0, 1, 3, 8])
@pytest.mark.parametrize("kind,E,R,C,replace_p", [(0, 5, 64, 100, 0.02), (0, 3, 40, 100, 0.3),
                                                  (1, 3, 16, 160, 0.05)])
def test_exception_stream_at_any_alignment(csf, shift, kind, E, R, C, replace_p):
    # The exception stream may start at any byte (the decoder stages it in
    # 16-byte pieces only when it is 16-byte aligned); sparse and dense
    # exception rates (a warp step's exceptions within or beyond one staged
    # chunk).
    w = 14 if kind == 0 else 1
    dense = synth.random_rows(shift + C, E * R, C, spread=w + 3, replace_p=replace_p).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    n = up.num_exc
    pad = (n + 15) // 16 * 16
    buf = torch.full((pad + 32,), 0xEE, dtype=torch.uint8, device="cuda")
    buf[shift:shift + n].copy_(up.exc_bytes[:n])
    up.exc_bytes = buf[shift:shift + pad + 16]
    ws = torch.full(dense.shape, 0x5A, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws)
    assert np.array_equal(_np(ws), dense)
    assert up.errors() == 0


@pytest.mark.parametrize("offset", [0, 1, 3, 8, 15, 16, 17])
def test_odd_offset_workspace_with_guards(csf, offset):
    for kind, shape in ((0, (3, 40, 100)), (1, (2, 37, 160))):
        dense = _small_dense(kind, *shape, seed=offset)
        up = csf.upload(oracle.encode(kind, dense))
        n = dense.size
        buf = torch.full((n + 64,), 0xAB, dtype=torch.uint8, device="cuda")
        ws = buf[offset:offset + n]
        csf.decode(up, ws)
        host = _np(buf)
        assert np.array_equal(host[offset:offset + n], dense.ravel())
        assert (host[:offset] == 0xAB).all() and (host[offset + n:] == 0xAB).all()
        # routed into an odd-offset workspace: inactive planes keep the guard value
        start = np.array([0, 1] + [1] * (shape[0] - 1), np.int32)
        buf.fill_(0xAB)
        csf.decode(up, buf[offset:offset + n], expert_start=torch.from_numpy(start).cuda())
        host = _np(buf)
        plane = shape[1] * shape[2]
        assert np.array_equal(host[offset:offset + plane], dense[0].ravel())
        assert (host[offset + plane:] == 0xAB).all() and (host[:offset] == 0xAB).all()


def test_special_streams(csf):
    # All-escape rows (decoder only) and a zero-exception stack.
    exc = np.arange(100, 100 + 3 * 40, dtype=np.uint8)
    enc = {"kind": 0, "shape": (1, 3, 40), "base": np.array([1, 2, 3], np.uint8),
           "offsets": np.full(60, 0xFF, np.uint8), "escapes": np.zeros(0, np.uint8),
           "exc_index": np.array([0, 40, 80, 120], np.uint32), "exc_bytes": exc, "num_exc": 120}
    ws = csf.decode(csf.upload(enc))
    assert np.array_equal(_np(ws).ravel(), exc)
    dense = np.full((2, 16, 100), 0x40, np.uint8)
    dense[:, :, 1::2] = 0x4E
    enc = oracle.encode(0, dense)
    assert enc["num_exc"] == 0
    st = csf.prepare(_dense_cuda(dense), 0)
    assert_stack_matches(st, enc)
    assert np.array_equal(_np(csf.decode(st)), dense)


def test_corrupt_index_sets_error_word(csf):
    dense = synth.stack("tiny")
    enc = oracle.encode(0, dense)
    bad = dict(enc)
    bad["exc_index"] = enc["exc_index"].copy()
    bad["exc_index"][100:] += 1          # planted on the CPU: row 99's step is off by one
    assert oracle.check(bad) == oracle.ERR_CORRUPT
    up = csf.upload(bad)
    csf.decode(up)
    assert up.errors() & csf.DEV_ERR_CORRUPT
    bad = dict(enc)
    bad["num_exc"] = enc["num_exc"] - 3  # stream shorter than the index says
    bad["exc_bytes"] = enc["exc_bytes"][:-3]
    up = csf.upload(bad)
    csf.decode(up)
    assert up.errors() & csf.DEV_ERR_CORRUPT
    good = csf.upload(enc)
    csf.decode(good)
    assert good.errors() == 0


def test_prepare_capacity_overflow_reports_and_keeps_index(csf):
    dense = synth.stack("tiny")
    enc = oracle.encode(0, dense)
    E, R, C = dense.shape
    st = csf.empty_stack(0, E, R, C, exc_capacity=16)
    scratch = csf.prepare_scratch(0, E, R, C)
    csf.prepare_async(_dense_cuda(dense), st, scratch, exc_capacity=5)
    torch.cuda.synchronize()
    assert st.errors() & csf.DEV_ERR_CAPACITY
    assert np.array_equal(_np(st.exc_index).view(np.uint32), enc["exc_index"])
    assert np.array_equal(_np(st.exc_bytes[:5]), enc["exc_bytes"][:5])


def test_cuda_graph_replay_with_repoisoning(csf):
    dense = synth.gate_stack(E=16, R=64)
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    start = synth.routing(E=16, active=4, tokens=16, seed=1)
    es = torch.from_numpy(start).cuda()
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    want, _ = oracle.decode(enc, start, np.full(dense.shape, 0xFF, np.uint8))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        csf.decode(up, ws, expert_start=es)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        csf.decode(up, ws, expert_start=es)
    for _ in range(8):
        ws.fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_np(ws), want)


# ---------------------------------------------------------------- full sizes

@pytest.fixture(scope="module")
def gate(csf):
    dense = synth.stack("gate")
    enc = oracle.encode(0, dense)
    return dense, enc


@pytest.fixture(scope="module")
def down(csf):
    dense = synth.stack("down")
    enc = oracle.encode(0, dense)
    return dense, enc


def test_full_gate_prepare_and_decode(csf, gate):
    dense, enc = gate
    d = _dense_cuda(dense)
    st = csf.prepare(d, 0)
    assert st.errors() == 0
    assert_stack_matches(st, enc)
    ws = torch.empty_like(d)
    csf.decode(st, ws)
    assert torch.equal(ws, d)
    up = csf.upload(enc)
    ws.fill_(0)
    csf.decode(up, ws)
    assert torch.equal(ws, d) and up.errors() == 0


@pytest.mark.parametrize("is64", [False, True])
def test_full_gate_routed_8_of_512_poisoned(csf, gate, is64):
    dense, enc = gate
    d = _dense_cuda(dense)
    up = csf.upload(enc)
    start = synth.routing(E=512, active=8, tokens=64, seed=0, dtype=np.int64 if is64 else np.int32)
    active = np.flatnonzero(np.diff(start.astype(np.int64)) > 0)
    assert active.size == 8
    ws = torch.full_like(d, 0xFF)
    csf.decode(up, ws, expert_start=torch.from_numpy(start).cuda())
    mask = torch.zeros(512, dtype=torch.bool, device="cuda")
    mask[torch.from_numpy(active).cuda()] = True
    assert torch.equal(ws[mask], d[mask])
    assert bool((ws[~mask] == 0xFF).all())


@pytest.mark.parametrize("routed", [False, True])
def test_full_gate_row_range(csf, gate, routed):
    # The full gate stack read as fused gate/up (rows [0, 512) of each
    # 1024-row expert are the gate half), in the launch the benchmark times.
    dense, enc = gate
    d = _dense_cuda(dense)
    up = csf.upload(enc)
    es = None
    mask = torch.ones(512, dtype=torch.bool, device="cuda")
    if routed:
        start = synth.routing(E=512, active=8, tokens=64, seed=0)
        es = torch.from_numpy(start).cuda()
        mask[:] = False
        mask[torch.from_numpy(np.flatnonzero(np.diff(start.astype(np.int64)) > 0)).cuda()] = True
    for lo, hi in [(0, 512), (512, 1024), (5, 1000)]:
        ws = torch.full_like(d, 0xFF)
        csf.decode(up, ws, expert_start=es, rows=(lo, hi))
        assert torch.equal(ws[mask][:, lo:hi], d[mask][:, lo:hi])
        assert bool((ws[mask][:, :lo] == 0xFF).all()) and bool((ws[mask][:, hi:] == 0xFF).all())
        assert bool((ws[~mask] == 0xFF).all())
    assert up.errors() == 0


def test_full_pair_decode(csf, gate, down):
    (gd, genc), (dd, denc) = gate, down
    g_up, d_up = csf.upload(genc), csf.upload(denc)
    gdc, ddc = _dense_cuda(gd), _dense_cuda(dd)
    gws, dws = torch.full_like(gdc, 0xFF), torch.full_like(ddc, 0xFF)
    csf.decode_pair(g_up, d_up, gws, dws)
    assert torch.equal(gws, gdc) and torch.equal(dws, ddc)
    start = synth.routing(E=512, active=8, tokens=64, seed=0)
    active = torch.from_numpy(np.flatnonzero(np.diff(start.astype(np.int64)) > 0)).cuda()
    gws.fill_(0xFF)
    dws.fill_(0xFF)
    csf.decode_pair(g_up, d_up, gws, dws, expert_start=torch.from_numpy(start).cuda())
    mask = torch.zeros(512, dtype=torch.bool, device="cuda")
    mask[active] = True
    assert torch.equal(gws[mask], gdc[mask]) and torch.equal(dws[mask], ddc[mask])
    assert bool((gws[~mask] == 0xFF).all()) and bool((dws[~mask] == 0xFF).all())
    assert g_up.errors() == 0 and d_up.errors() == 0
    # GPU prepare of the heavy-tailed down stack matches the oracle.
    st = csf.prepare(ddc, 0)
    assert_stack_matches(st, denc)


def test_full_mxfp4_prepare_and_decode(csf):
    dense = synth.stack("mxfp4")
    enc = oracle.encode(1, dense)
    d = _dense_cuda(dense)
    st = csf.prepare(d, 1)
    assert st.errors() == 0
    assert_stack_matches(st, enc)
    ws = torch.empty_like(d)
    csf.decode(st, ws)
    assert torch.equal(ws, d)
    start = synth.routing(E=384, active=8, tokens=64, seed=0)
    active = torch.from_numpy(np.flatnonzero(np.diff(start.astype(np.int64)) > 0)).cuda()
    ws.fill_(0xFF)
    csf.decode(st, ws, expert_start=torch.from_numpy(start).cuda())
    mask = torch.zeros(384, dtype=torch.bool, device="cuda")
    mask[active] = True
    assert torch.equal(ws[mask], d[mask]) and bool((ws[~mask] == 0xFF).all())


def _low_and_high_base_stack(seed, E, R, C, high_experts):
    # Rows centred low (bases well under 240) except in `high_experts`, whose
    # rows sit at the top of the byte range (bases above 240, values that
    # reach 255); 3% random bytes everywhere.
    rng = np.random.default_rng(seed)
    centre = rng.integers(0x20, 0x60, size=(E, R, 1))
    centre[list(high_experts)] = rng.integers(241, 250, size=(len(high_experts), R, 1))
    vals = np.minimum(centre + rng.integers(0, 15, size=(E, R, C)), 255)
    repl = rng.integers(0, 256, size=(E, R, C))
    return np.where(rng.random((E, R, C)) < 0.03, repl, vals).astype(np.uint8)


@pytest.mark.parametrize("C", [20, 50, 64, 66, 68, 100])
def test_word_wise_and_general_segments_in_one_launch(csf, C):
    # A warp segment whose bases are all <= 240 takes plain adds: the
    # word-wise expansion when C is a multiple of 4 and at least 64, else the
    # plain-add variant of the general expansion (C < 32, 32 <= C < 64, and
    # C >= 64 with boundaries inside words); segments with a higher base take
    # the general loop.  Both kinds of segment meet in every launch below.
    E, R = 6, 300
    dense = _low_and_high_base_stack(11 + C, E, R, C, high_experts=(3, 5))
    enc = oracle.encode(0, dense)
    assert (enc["base"] > 240).any() and (enc["base"] <= 240).any()
    st = csf.upload(enc)
    assert np.array_equal(_np(csf.decode(st)), dense)
    start = torch.from_numpy(np.array([0, 1, 1, 4, 6, 6, 9], np.int32)).cuda()    # experts 0, 2, 3, 5
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    csf.decode(st, ws, expert_start=start)
    want, status = oracle.decode(enc, start.cpu().numpy(), np.full(dense.shape, 0xFF, np.uint8))
    assert status == oracle.OK and np.array_equal(_np(ws), want)
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    csf.decode(st, ws, rows=(0, 150))
    want, status = oracle.decode(enc, None, np.full(dense.shape, 0xFF, np.uint8), rows=(0, 150))
    assert status == oracle.OK and np.array_equal(_np(ws), want)
    sf = csf.decode(st, layout=csf.LAYOUT_BLOCKED)
    want, status = oracle.decode_blocked(enc)
    assert status == oracle.OK and np.array_equal(_np(sf), want)
    assert st.errors() == 0


def _mx_low_and_high_base_stack(seed, E, R, C, high_experts):
    # MXFP4-shaped rows: base + {0, 1} for 85% of entries, else random; bases
    # low except in `high_experts`, whose rows centre on 254 / 255 (bases
    # above 254 reach the general loop).
    rng = np.random.default_rng(seed)
    centre = rng.integers(100, 130, size=(E, R, 1))
    centre[list(high_experts)] = rng.integers(254, 256, size=(len(high_experts), R, 1))
    vals = np.minimum(centre + rng.integers(0, 2, size=(E, R, C)), 255)
    repl = rng.integers(0, 256, size=(E, R, C))
    return np.where(rng.random((E, R, C)) < 0.15, repl, vals).astype(np.uint8)


@pytest.mark.parametrize("C", [64, 128, 132, 160])
def test_mxfp4_word_wise_and_general_segments_in_one_launch(csf, C):
    E, R = 5, 260
    dense = _mx_low_and_high_base_stack(23 + C, E, R, C, high_experts=(1, 4))
    enc = oracle.encode(1, dense)
    assert (enc["base"] > 254).any() and (enc["base"] <= 254).any()
    st = csf.upload(enc)
    assert np.array_equal(_np(csf.decode(st)), dense)
    start = torch.from_numpy(np.array([0, 2, 3, 3, 5, 8], np.int64)).cuda()       # experts 0, 1, 3, 4
    ws = torch.full(dense.shape, 0xFF, dtype=torch.uint8, device="cuda")
    csf.decode(st, ws, expert_start=start)
    want, status = oracle.decode(enc, start.cpu().numpy(), np.full(dense.shape, 0xFF, np.uint8))
    assert status == oracle.OK and np.array_equal(_np(ws), want)
    sf = csf.decode(st, layout=csf.LAYOUT_BLOCKED)
    want, status = oracle.decode_blocked(enc)
    assert status == oracle.OK and np.array_equal(_np(sf), want)
    assert st.errors() == 0


# Row widths that reach every way the two row kernels read a staged row:
# 16-byte vectors (C % 16 == 0), aligned words (C % 4 == 0) and byte-shifted
# words (C % 4 != 0); narrow rows run double-buffered and wide ones (C of 200
# and more) single-buffered; ragged last tiles and tiles whose byte count is
# not a multiple of 16 (tail loaded plainly).  Rows wider than 255 bytes take
# the single-pass kernel with the decoupled look-back.
PREP_WIDTHS = [(0, 3, 150, 48), (0, 3, 150, 128), (0, 2, 130, 200), (0, 2, 70, 252), (0, 3, 131, 100),
               (0, 2, 140, 8), (0, 2, 133, 72), (0, 3, 129, 7), (0, 2, 150, 50), (0, 2, 135, 255),
               (0, 2, 60, 256), (1, 3, 150, 160), (1, 2, 100, 200), (1, 2, 140, 96), (1, 2, 131, 100),
               (1, 3, 129, 33), (1, 2, 140, 8), (1, 2, 50, 300)]


def _least_scratch_bytes(csf, kind, E, R, C):
    # The smallest scratch csf_prepare accepts for rows of up to 255 bytes:
    # 16 bytes and 8 per 128-row tile.  It takes the two-kernel path instead
    # of the fused one.  Wider rows have one path, whose scratch csf_sizes()
    # reports.
    if C > 255:
        return csf.sizes(kind, E, R, C)["prepare_scratch"]
    return 16 + 8 * -(-(E * R) // 128)


def _prepare_with_scratch(csf, d, kind, nbytes):
    E, R, C = (int(x) for x in d.shape)
    st = csf.empty_stack(kind, E, R, C, exc_capacity=E * R * C)
    scratch = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")   # no initialisation needed
    csf.prepare_async(d, st, scratch)
    st.num_exc = int(st.exc_index[E * R].item()) & 0xFFFFFFFF
    return st


@pytest.mark.parametrize("kind,E,R,C", PREP_WIDTHS)
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("path", ["fused", "two_kernels"])
def test_prepare_rows_every_staging_path(csf, kind, E, R, C, offset, path):
    # A dense pointer one byte off alignment takes plain loads; aligned ones
    # take the bulk copies where the row layout allows.  The scratch size
    # csf_sizes() reports takes the fused path (one pass per tile, then the
    # placing kernel); the least accepted size takes the base and encode
    # kernels.  All give the oracle's streams, with a ragged last tile of rows.
    dense = _small_dense(kind, E, R, C, seed=C + 17 * E)
    enc = oracle.encode(kind, dense)
    buf = torch.zeros(dense.size + offset, dtype=torch.uint8, device="cuda")
    d = buf[offset:].view(E, R, C)
    d.copy_(_dense_cuda(dense))
    if path == "fused":
        st = csf.prepare(d, kind)
    else:
        st = _prepare_with_scratch(csf, d, kind, _least_scratch_bytes(csf, kind, E, R, C))
    torch.cuda.synchronize()
    assert st.errors() == 0
    assert_stack_matches(st, enc)


@pytest.mark.parametrize("kind,C", [(0, 100), (1, 160), (0, 50)])
def test_prepare_both_paths_full_size(csf, kind, C):
    # Full-size stacks (the gate, MXFP4 and down shapes) through both paths,
    # in a scratch filled with garbage, agree with the oracle.
    dense = {(0, 100): synth.gate_stack, (1, 160): synth.mxfp4_stack, (0, 50): synth.down_stack}[(kind, C)](seed=3)
    enc = oracle.encode(kind, dense)
    E, R, _ = dense.shape
    d = _dense_cuda(dense)
    for nbytes in (csf.sizes(kind, E, R, C)["prepare_scratch"], _least_scratch_bytes(csf, kind, E, R, C)):
        st = _prepare_with_scratch(csf, d, kind, nbytes)
        torch.cuda.synchronize()
        assert st.errors() == 0
        assert_stack_matches(st, enc)


def _adversarial_rows(kind, C, seed):
    """Rows built against the prepare's fast base search: around the median m
    of the bytes at columns 0, C/4, C/2, 3C/4 and C-1 it histograms each
    NVFP4 row in 32 bins, and counts the values m-1, m, m+1 of each MXFP4
    row; it then proves the best window there against the bytes it cannot
    see.  These rows defeat the anchor or the proof, or sit on the edges of
    the byte range, so both the fast and the exact paths run."""
    rng = np.random.default_rng(seed)
    w = 14 if kind == 0 else 1
    rows = []
    probes = sorted({0, C // 4, C // 2, (3 * C) // 4, C - 1})
    for _ in range(6):
        rows.append(rng.integers(0, 256, C))                                 # flat: no dominant window
        b = int(rng.integers(0, 256 - w))
        r = b + rng.integers(0, w + 1, C)
        r[probes] = (b + 128 + rng.integers(0, 60, len(probes))) % 256       # every probe an outlier
        rows.append(r)
        b1, b2 = int(rng.integers(0, 100)), int(rng.integers(140, 256 - w))
        half = np.concatenate([b1 + rng.integers(0, w + 1, C // 2), b2 + rng.integers(0, w + 1, C - C // 2)])
        rows.append(rng.permutation(half))                                    # twin clusters: tie or near tie
        rows.append(np.clip(255 - rng.integers(0, w + 3, C), 0, 255))          # at the top of the range
        rows.append(np.clip(rng.integers(0, w + 3, C), 0, 255))                # at the bottom
        b = int(rng.integers(40, 200))
        r = b + rng.integers(0, w + 1, C)
        edge = rng.random(C) < 0.35                                           # many bytes just past the window
        r[edge] = b + w + 1 + rng.integers(0, 18, edge.sum())
        low = rng.random(C) < 0.15
        r[low] = b - 1 - rng.integers(0, 18, low.sum())
        rows.append(np.clip(r, 0, 255))
        rows.append(np.full(C, int(rng.integers(0, 256))))                    # constant
        rows.append((np.arange(C) * 7 + int(rng.integers(0, 256))) % 256)      # every value once or so
        if kind == 1:
            # MXFP4: the counted values m-1, m, m+1 against the windows beside them
            probes_at = np.zeros(C, bool)
            probes_at[probes] = True
            m = int(rng.integers(3, 250))
            r = np.where(rng.random(C) < 0.5, m - 2, m - 1)                  # best window just below m - 1
            r[probes_at] = m
            rows.append(r)
            r = np.where(rng.random(C) < 0.5, m + 2, m + 3)                  # best window just above m + 1
            r[probes_at] = m
            rows.append(r)
            r = rng.choice([m - 1, m, m + 1], C)                              # [m-1, m] and [m, m+1] tie or nearly
            rows.append(r)
            r = np.where(rng.random(C) < 0.4, m, m + 1)
            r[rng.random(C) < 0.3] = m + 2                                    # a third value beside the window
            rows.append(r)
            rows.append(rng.choice([253, 254, 255], C))                       # median at the top: m - 1 clamped
            rows.append(rng.choice([0, 1, 2], C))                             # median 0: no window below
    return np.array(rows, dtype=np.uint8)


@pytest.mark.parametrize("kind,C", [(0, 100), (0, 50), (0, 7), (0, 160), (0, 255), (1, 160), (1, 100), (1, 33),
                                    (1, 5)])
def test_prepare_adversarial_rows(csf, kind, C):
    rows = _adversarial_rows(kind, C, seed=C + 1000 * kind)
    E = 2
    R = -(-rows.shape[0] // E)
    dense = np.resize(rows, (E * R, C)).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    st = csf.prepare(_dense_cuda(dense), kind)
    assert st.errors() == 0
    assert_stack_matches(st, enc)
    assert np.array_equal(_np(csf.decode(st)), dense)


@pytest.mark.parametrize("Cm", [160, 33])
@pytest.mark.parametrize("routed", [False, True])
@pytest.mark.parametrize("layout", ["rows", "blocked"])
@pytest.mark.parametrize("half", [False, True])
def test_pair_of_different_kinds(csf, Cm, routed, layout, half):
    # A pair may mix kinds (an NVFP4 stack and an MXFP4 one, different R and C):
    # the launch runs the kernel instance that holds both segment decoders,
    # whole-stack or per expert (routing, the gate half of a fused stack).
    E = 5
    gu = _small_dense(0, E, 256, 100, seed=31)                 # fused gate/up, gate half decoded
    mx = _small_dense(1, E, 300, Cm, seed=32)
    genc, menc = oracle.encode(0, gu), oracle.encode(1, mx)
    g_up, m_up = csf.upload(genc), csf.upload(menc)
    start = np.array([0, 1, 1, 4, 4, 6], np.int32) if routed else None
    es = None if start is None else torch.from_numpy(start).cuda()
    gr = (0, 128) if half else None
    if layout == "rows":
        gws = torch.full(gu.shape, 0x3C, dtype=torch.uint8, device="cuda")
        mws = torch.full(mx.shape, 0x3C, dtype=torch.uint8, device="cuda")
        csf.decode_pair(g_up, m_up, gws, mws, expert_start=es, gate_rows=gr)
        gw, gs = oracle.decode(genc, start, np.full(gu.shape, 0x3C, np.uint8), rows=gr)
        mw, ms = oracle.decode(menc, start, np.full(mx.shape, 0x3C, np.uint8))
    else:
        gws = torch.full((oracle.blocked_bytes(E, 256, 100),), 0x3C, dtype=torch.uint8, device="cuda")
        mws = torch.full((oracle.blocked_bytes(E, 300, Cm),), 0x3C, dtype=torch.uint8, device="cuda")
        csf.decode_pair(g_up, m_up, gws, mws, expert_start=es, gate_rows=gr, layout=csf.LAYOUT_BLOCKED)
        gw, gs = oracle.decode_blocked(genc, start, np.full(gws.numel(), 0x3C, np.uint8), rows=gr)
        mw, ms = oracle.decode_blocked(menc, start, np.full(mws.numel(), 0x3C, np.uint8))
    assert gs == oracle.OK and ms == oracle.OK
    assert np.array_equal(_np(gws).ravel(), gw.ravel())
    assert np.array_equal(_np(mws).ravel(), mw.ravel())
    assert g_up.errors() == 0 and m_up.errors() == 0


@pytest.mark.parametrize("kind,C", [(0, 100), (1, 160)])
def test_prepare_fused_into_unaligned_exception_buffer(csf, kind, C):
    # The placing kernel copies whole words into a 4-byte aligned exception
    # buffer; any other alignment takes its byte-by-byte copy.
    E, R = 4, 1000
    dense = _small_dense(kind, E, R, C, seed=91 + kind)
    enc = oracle.encode(kind, dense)
    for off in (1, 2, 3):
        st = csf.empty_stack(kind, E, R, C, exc_capacity=E * R * C)
        buf = torch.full((E * R * C + 16,), 0xEE, dtype=torch.uint8, device="cuda")
        st.exc_bytes = buf[off:off + E * R * C]
        csf.prepare_async(_dense_cuda(dense), st, csf.prepare_scratch(kind, E, R, C))
        torch.cuda.synchronize()
        st.num_exc = int(st.exc_index[E * R].item()) & 0xFFFFFFFF
        assert st.errors() == 0
        assert_stack_matches(st, enc)
        assert (_np(buf[:off]) == 0xEE).all() and (_np(buf[off + st.num_exc:]) == 0xEE).all()


@pytest.mark.parametrize("tiles", [8192, 8193])
def test_prepare_at_the_fused_tile_limit(csf, tiles):
    # Up to 8192 tiles of 128 rows the reported scratch takes the fused path;
    # one more tile and csf_sizes() reports the two-kernel scratch.
    E, R, C = 1, tiles * 128 - 5, 8
    dense = synth.random_rows(tiles, E * R, C, spread=20, replace_p=0.05).reshape(E, R, C)
    enc = oracle.encode(0, dense)
    need = csf.sizes(0, E, R, C)["prepare_scratch"]
    assert (need > 16 + 8 * tiles) == (tiles <= 8192)
    st = csf.prepare(_dense_cuda(dense), 0)
    assert st.errors() == 0
    assert_stack_matches(st, enc)

"""GPU tests of ahead-of-call expansion (csf_expand / csf.expand_scales).

The pages' expand_scales ("NVFP4-CSF: expand_scales() for ahead-of-call scale
expansion" body and its canonical-twin commit message) expands a layer's
scales into the shared scratch on a side stream while other work runs; the
caller orders scratch reuse, expansion and the reading call with events.
These tests build that ordering with real hazards: a long kernel keeps the
previous reader of the workspace busy, so an expansion that did not wait for
it would overwrite bytes still to be read.  Expected bytes come from the
seeded inputs (which the oracle round-trips in the parity tests).
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


def _layer(csf, seed, E=16, I=64, Rd=128):
    # One MoE layer: a fused gate/up stack (2*I rows) and a down stack.
    gu = synth.random_rows(seed, E * 2 * I, 100, spread=17, replace_p=0.03).reshape(E, 2 * I, 100)
    dn = synth.random_rows(seed + 1, E * Rd, 50, spread=17, replace_p=0.05).reshape(E, Rd, 50)
    return (gu, csf.upload(oracle.encode(0, gu))), (dn, csf.upload(oracle.encode(0, dn)))


SLEEP = 20_000_000   # device cycles (~10 ms): the previous reader is still busy


def test_expansion_waits_for_the_previous_reader(csf):
    (g1, s1g), (d1, s1d) = _layer(csf, 1)
    (g2, s2g), (d2, s2d) = _layer(csf, 2)
    gws = torch.empty(g1.shape, dtype=torch.uint8, device="cuda")
    dws = torch.empty(d1.shape, dtype=torch.uint8, device="cuda")
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    csf.decode_pair(s1g, s1d, gws, dws)                 # layer 1's scales
    torch.cuda._sleep(SLEEP)                            # layer 1's attention
    out1g, out1d = gws.clone(), dws.clone()             # layer 1's MoE reads them
    read1 = torch.cuda.Event()
    read1.record(main)
    ev = csf.expand_scales([(s2g, gws), (s2d, dws)], side, after=read1)
    main.wait_event(ev)
    out2g, out2d = gws.clone(), dws.clone()             # layer 2's MoE
    torch.cuda.synchronize()
    assert np.array_equal(out1g.cpu().numpy(), g1) and np.array_equal(out1d.cpu().numpy(), d1)
    assert np.array_equal(out2g.cpu().numpy(), g2) and np.array_equal(out2d.cpu().numpy(), d2)
    assert s1g.errors() == s2g.errors() == s2d.errors() == 0


def test_consumer_waits_for_the_expansion(csf):
    # Poisoned scratch; the side stream is held back by a long kernel, so a
    # consumer that did not wait for `done` would read the poison.
    (g1, s1g), (d1, s1d) = _layer(csf, 3)
    gws = torch.full(g1.shape, 0xA5, dtype=torch.uint8, device="cuda")
    dws = torch.full(d1.shape, 0xA5, dtype=torch.uint8, device="cuda")
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    side.wait_stream(main)
    with torch.cuda.stream(side):
        torch.cuda._sleep(SLEEP)
    ev = csf.expand_scales([(s1g, gws), (s1d, dws)], side)
    main.wait_event(ev)
    outg, outd = gws.clone(), dws.clone()
    torch.cuda.synchronize()
    assert np.array_equal(outg.cpu().numpy(), g1) and np.array_equal(outd.cpu().numpy(), d1)


def test_gate_half_and_more_than_two_stacks(csf):
    # Row ranges pass through; more than two stacks go out as several
    # launches on the same stream with one wait and one final record.
    (g1, s1g), (d1, s1d) = _layer(csf, 4)
    (g2, s2g), (d2, s2d) = _layer(csf, 5)
    I = g1.shape[1] // 2
    wss = [torch.full(a.shape, 0xFF, dtype=torch.uint8, device="cuda") for a in (g1, d1, g2, d2)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    ev = csf.expand_scales([(s1g, wss[0], (0, I)), (s1d, wss[1]), (s2g, wss[2]), (s2d, wss[3])], side)
    torch.cuda.current_stream().wait_event(ev)
    h = [w.cpu().numpy() for w in wss]
    assert np.array_equal(h[0][:, :I], g1[:, :I]) and (h[0][:, I:] == 0xFF).all()
    assert np.array_equal(h[1], d1) and np.array_equal(h[2], g2) and np.array_equal(h[3], d2)


def test_nothing_compressed_returns_false(csf):
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert csf.expand_scales([(None, ws)]) is False


def test_expansion_inside_a_cuda_graph(csf):
    # Fork to the side stream and join back inside one captured graph; each
    # replay poisons the workspace first, then expands and reads it.
    (g1, s1g), (d1, s1d) = _layer(csf, 6)
    gws = torch.empty(g1.shape, dtype=torch.uint8, device="cuda")
    dws = torch.empty(d1.shape, dtype=torch.uint8, device="cuda")
    outg, outd = torch.empty_like(gws), torch.empty_like(dws)
    side = torch.cuda.Stream()
    csf.expand_scales([(s1g, gws), (s1d, dws)], side)   # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        gws.fill_(0x77)
        dws.fill_(0x77)
        poisoned = torch.cuda.Event()
        poisoned.record(cap)
        ev = csf.expand_scales([(s1g, gws), (s1d, dws)], side, after=poisoned)
        cap.wait_event(ev)
        outg.copy_(gws)
        outd.copy_(dws)
    for _ in range(3):
        outg.zero_()
        outd.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(outg.cpu().numpy(), g1) and np.array_equal(outd.cpu().numpy(), d1)


def test_concurrent_host_threads_on_separate_streams(csf):
    # Several host threads call the library at once, each on its own stream
    # with its own stacks and workspaces (the library's per-device state is
    # set up once under a lock; calls share nothing else).
    import threading
    layers = [_layer(csf, 20 + k, E=8, I=64, Rd=64) for k in range(4)]
    results = [None] * len(layers)
    errors = []

    def work(k):
        try:
            (g, sg), (d, sd) = layers[k]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    gws, dws = csf.decode_pair(sg, sd)
                    half = csf.decode(sg, rows=(0, g.shape[1] // 2))
            stream.synchronize()
            results[k] = (gws.cpu().numpy(), dws.cpu().numpy(), half.cpu().numpy())
        except Exception as exc:   # reported below
            errors.append(exc)

    torch.cuda.synchronize()                            # uploads done before other streams read them
    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(layers))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k, ((g, _), (d, _)) in enumerate(layers):
        gw, dw, half = results[k]
        assert np.array_equal(gw, g) and np.array_equal(dw, d)
        assert np.array_equal(half[:, :g.shape[1] // 2], g[:, :g.shape[1] // 2])

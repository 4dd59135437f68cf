"""GPU tests of decode into the scale-operand layout of block-scaled GEMMs.

csf_decode_rows / csf_expand with CSF_LAYOUT_BLOCKED write the 128 x 4 tiled
layout that Blackwell block-scaled GEMMs read.  Parity: bit-exact against the
oracle's blocked decode (small ragged shapes, several items per expert, row
ranges, routing, pairs, the full gate stack), padding included.  Pin of the
layout itself, independent of the oracle: a cuBLASLt NVFP4 GEMM through
PyTorch consumes the decoded scales and must match an fp64 product computed
from the row-major scales, while the same GEMM fed the row-major bytes must
not.
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


def _dense(kind, E, R, C, seed, replace_p=0.08):
    w = 14 if kind == 0 else 1
    return synth.random_rows(seed, E * R, C, spread=w + 3, replace_p=replace_p).reshape(E, R, C)


SHAPES = [(0, 1, 1, 1), (0, 2, 128, 4), (0, 3, 200, 7), (0, 2, 256, 100), (0, 3, 300, 50), (0, 2, 1000, 100),
          (0, 2, 640, 12), (0, 1, 129, 255), (0, 2, 130, 600), (1, 2, 130, 160), (1, 3, 64, 33), (1, 2, 512, 160),
          (0, 1, 128, 2000), (1, 2, 100, 17), (1, 2, 130, 300), (1, 1, 200, 1000)]


@pytest.mark.parametrize("kind,E,R,C", SHAPES)
def test_blocked_matches_oracle_poisoned(csf, kind, E, R, C):
    dense = _dense(kind, E, R, C, seed=E * 7 + R + C)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    nb = oracle.blocked_bytes(E, R, C)
    assert csf.blocked_bytes(up) == nb
    ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws, layout=csf.LAYOUT_BLOCKED)
    want, st = oracle.decode_blocked(enc)
    assert st == oracle.OK
    assert np.array_equal(ws.cpu().numpy(), want)
    assert up.errors() == 0


@pytest.mark.parametrize("kind,E,R,C", [(0, 4, 300, 100), (1, 3, 384, 160), (0, 5, 512, 50), (0, 3, 384, 400),
                                        (1, 3, 300, 520)])
@pytest.mark.parametrize("routed", [False, True])
def test_blocked_row_blocks_and_routing(csf, kind, E, R, C, routed):
    dense = _dense(kind, E, R, C, seed=R + C)
    enc = oracle.encode(kind, dense)
    up = csf.upload(enc)
    nb = oracle.blocked_bytes(E, R, C)
    start = None
    if routed:
        counts = np.zeros(E, np.int64)
        counts[[0, E - 1]] = [2, 5]
        start = np.concatenate([[0], np.cumsum(counts)])
    es = None if start is None else torch.from_numpy(start.astype(np.int32)).cuda()
    for lo, hi in [(0, R), (0, 128), (128, R), (256, R), (128, 256)]:
        ws = torch.full((nb,), 0x5A, dtype=torch.uint8, device="cuda")
        csf.decode(up, ws, expert_start=es, rows=(lo, hi), layout=csf.LAYOUT_BLOCKED)
        want, _ = oracle.decode_blocked(enc, start, np.full(nb, 0x5A, np.uint8), rows=(lo, hi))
        assert np.array_equal(ws.cpu().numpy(), want), (lo, hi)
    assert up.errors() == 0


@pytest.mark.parametrize("routed", [False, True])
def test_blocked_pair_gate_half_and_down(csf, routed):
    E, I = 6, 256
    gu, dn = _dense(0, E, 2 * I, 100, seed=1), _dense(0, E, 300, 50, seed=2)
    genc, denc = oracle.encode(0, gu), oracle.encode(0, dn)
    g_up, d_up = csf.upload(genc), csf.upload(denc)
    start = np.array([0, 3, 3, 3, 4, 4, 9], np.int64) if routed else None
    es = None if start is None else torch.from_numpy(start).cuda()
    gws = torch.full((oracle.blocked_bytes(E, 2 * I, 100),), 0xEE, dtype=torch.uint8, device="cuda")
    dws = torch.full((oracle.blocked_bytes(E, 300, 50),), 0xEE, dtype=torch.uint8, device="cuda")
    csf.decode_pair(g_up, d_up, gws, dws, expert_start=es, gate_rows=(0, I), layout=csf.LAYOUT_BLOCKED)
    gw, _ = oracle.decode_blocked(genc, start, np.full(gws.numel(), 0xEE, np.uint8), rows=(0, I))
    dw, _ = oracle.decode_blocked(denc, start, np.full(dws.numel(), 0xEE, np.uint8))
    assert np.array_equal(gws.cpu().numpy(), gw) and np.array_equal(dws.cpu().numpy(), dw)


def test_blocked_side_stream_expansion(csf):
    E, R, C = 4, 256, 100
    dense = _dense(0, E, R, C, seed=3)
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    ws = torch.full((oracle.blocked_bytes(E, R, C),), 0x11, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    ev = csf.expand_scales([(up, ws)], side, layout=csf.LAYOUT_BLOCKED)
    torch.cuda.current_stream().wait_event(ev)
    want, _ = oracle.decode_blocked(enc)
    assert np.array_equal(ws.cpu().numpy(), want)


def test_blocked_argument_errors(csf):
    E, R, C = 2, 256, 100
    up = csf.upload(oracle.encode(0, _dense(0, E, R, C, seed=4)))
    nb = oracle.blocked_bytes(E, R, C)
    buf = torch.zeros(nb + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(csf.CsfError, match="invalid argument"):
        csf.decode(up, buf[1:1 + nb], layout=csf.LAYOUT_BLOCKED)         # not 16-byte aligned
    with pytest.raises(csf.CsfError, match="invalid argument"):
        csf.decode(up, buf[:nb], rows=(0, 100), layout=csf.LAYOUT_BLOCKED)
    with pytest.raises(csf.CsfError, match="too small"):
        csf.decode(up, buf[:nb - 16], layout=csf.LAYOUT_BLOCKED)


def test_blocked_full_gate(csf):
    dense = synth.stack("gate")
    enc = oracle.encode(0, dense)
    up = csf.upload(enc)
    want, _ = oracle.decode_blocked(enc)
    ws = torch.full((want.size,), 0xAB, dtype=torch.uint8, device="cuda")
    csf.decode(up, ws, layout=csf.LAYOUT_BLOCKED)
    assert np.array_equal(ws.cpu().numpy(), want)
    start = synth.routing(E=512, active=8, tokens=64, seed=0)
    ws.fill_(0xAB)
    csf.decode(up, ws, expert_start=torch.from_numpy(start).cuda(), layout=csf.LAYOUT_BLOCKED)
    want_r, _ = oracle.decode_blocked(enc, start, np.full(want.size, 0xAB, np.uint8))
    assert np.array_equal(ws.cpu().numpy(), want_r)
    assert up.errors() == 0


# ------------------------------------------------ pin through a real GEMM

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def _fp4_values(packed: np.ndarray) -> np.ndarray:
    # Two e2m1 codes per byte; the order inside a byte does not matter for the
    # product below (both operands share it and a byte never straddles a
    # 16-element scale block).
    return np.stack([E2M1[packed & 0xF], E2M1[packed >> 4]], axis=-1).reshape(packed.shape[0], -1)


def _e4m3(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _nvfp4_gemm(a, b_t, sa, sb):
    """D = A B^T with NVFP4 block scales through PyTorch (cuBLASLt)."""
    F = torch.nn.functional
    if hasattr(F, "scaled_mm") and hasattr(F, "ScalingType"):
        return F.scaled_mm(a, b_t, sa, F.ScalingType.BlockWise1x16, sb, F.ScalingType.BlockWise1x16,
                           swizzle_a=F.SwizzleType.SWIZZLE_32_4_4, swizzle_b=F.SwizzleType.SWIZZLE_32_4_4,
                           output_dtype=torch.bfloat16)
    return torch._scaled_mm(a, b_t, sa, sb, out_dtype=torch.bfloat16)


def test_blocked_scales_drive_a_real_nvfp4_gemm(csf):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this PyTorch has no fp4 dtype")
    M, N, K = 128, 256, 1600
    C = K // 16
    rng = np.random.default_rng(0)
    # B's scales: CSF-coded e4m3 bytes with exceptions, all finite and of
    # moderate size (no NaN codes).
    base = rng.integers(0x30, 0x40, size=(N, 1))
    sb_dense = (base + rng.integers(0, 15, size=(N, C))).astype(np.uint8)
    repl = rng.random((N, C)) < 0.05
    sb_dense[repl] = rng.integers(0x20, 0x50, size=int(repl.sum()))
    enc = oracle.encode(0, sb_dense.reshape(1, N, C))
    assert enc["num_exc"] > 0
    up = csf.upload(enc)
    sb = csf.decode(up, layout=csf.LAYOUT_BLOCKED)
    a_codes = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b_codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    a = torch.from_numpy(a_codes).cuda().view(torch.float4_e2m1fn_x2)
    b_t = torch.from_numpy(b_codes).cuda().view(torch.float4_e2m1fn_x2).t()
    sa = torch.full((M * C,), 0x38, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)   # 1.0
    try:
        d = _nvfp4_gemm(a, b_t, sa, sb.view(torch.float8_e4m3fn))
        torch.cuda.synchronize()
    except (RuntimeError, TypeError, NotImplementedError) as err:
        pytest.skip(f"NVFP4 scaled GEMM not available in this PyTorch: {err}")
    bf = _fp4_values(b_codes) * np.repeat(_e4m3(sb_dense), 16, axis=1)
    ref = _fp4_values(a_codes) @ bf.T
    got = d.float().cpu().numpy().astype(np.float64)
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < 1e-2, err
    # Control: the row-major scale bytes in the same buffer give a wrong product.
    flat = torch.from_numpy(sb_dense.reshape(-1).copy()).cuda().view(torch.float8_e4m3fn)
    d2 = _nvfp4_gemm(a, b_t, sa, flat).float().cpu().numpy().astype(np.float64)
    assert np.linalg.norm(d2 - ref) / np.linalg.norm(ref) > 0.1


def test_blocked_corrupt_index_sets_error_word(csf):
    # Corruptions planted on the CPU, as in the row-major test: one row's
    # index step off by one, and a stream shorter than the index says.
    for kind in (0, 1):
        dense = _dense(kind, 4, 64, 8, seed=kind)
        enc = oracle.encode(kind, dense)
        assert enc["num_exc"] > 10
        bad = dict(enc)
        bad["exc_index"] = enc["exc_index"].copy()
        bad["exc_index"][100:] += 1
        assert oracle.check(bad) == oracle.ERR_CORRUPT
        up = csf.upload(bad)
        csf.decode(up, layout=csf.LAYOUT_BLOCKED)
        assert up.errors() & csf.DEV_ERR_CORRUPT
        bad = dict(enc)
        bad["num_exc"] = enc["num_exc"] - 3
        bad["exc_bytes"] = enc["exc_bytes"][:-3]
        up = csf.upload(bad)
        csf.decode(up, layout=csf.LAYOUT_BLOCKED)
        assert up.errors() & csf.DEV_ERR_CORRUPT
        good = csf.upload(enc)
        csf.decode(good, layout=csf.LAYOUT_BLOCKED)
        assert good.errors() == 0

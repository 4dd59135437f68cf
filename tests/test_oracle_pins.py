"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test fixes a part of the codec by something independent of the oracle's
own code: bytes worked out by hand from the format reading, closed forms,
exhaustive brute force on tiny rows, invariants, and the size figures the
"finegrained-kernels: decode losslessly compressed NVFP4 scales (CSF)" page
reports for its 512-expert stacks (size paragraph).

Format reading being pinned (from that page's format paragraph and the
"NVFP4-CSF: expand_scales() ... (canonical twin of #477)" commit message on
one-bit MXFP4 and four-bit NVFP4 offsets): one base byte per row; NVFP4
nibbles 0..14 are offsets and 15 is the escape code, element i in byte i>>1,
even element in the low nibble; MXFP4 has an LSB-first offset bit plane and
an escape bit plane; exceptions row-major; exc_index = exclusive per-row
prefix with the total last; base = smallest present value whose window
[v, v+w] covers the most bytes (w = 14 NVFP4, 1 MXFP4).
"""
import numpy as np
import pytest

import oracle
from lossless_nvfp4_scale_gb300 import synth

W = {oracle.NVFP4: 14, oracle.MXFP4: 1}


# ---------------------------------------------------------------- hand-worked

def test_hand_example_nvfp4():
    # Row 0: 0x30, 0x3E, 0x31 all fit the window [0x30, 0x3E]: base 0x30,
    # offsets 0, 14, 1.  Row 1: 0xFF, 0x00, 0x05: window [0x00, 0x0E] holds two
    # bytes, every other window one: base 0x00, 0xFF is an exception.
    # Nibbles in element order: 0, E, 1, F, 0, 5 -> bytes E0 F1 50.
    dense = np.array([[[0x30, 0x3E, 0x31], [0xFF, 0x00, 0x05]]], np.uint8)
    enc = oracle.encode(oracle.NVFP4, dense)
    assert enc["base"].tolist() == [0x30, 0x00]
    assert enc["offsets"].tolist() == [0xE0, 0xF1, 0x50]
    assert enc["exc_index"].tolist() == [0, 0, 1]
    assert enc["exc_bytes"].tolist() == [0xFF]
    assert enc["num_exc"] == 1
    out, st = oracle.decode(enc)
    assert st == oracle.OK and np.array_equal(out, dense)


def test_hand_example_mxfp4():
    # Row: 120 121 121 120 7 254 121 120 120 0.  Window [120, 121] holds 7
    # bytes: base 120; offset bits 0 1 1 0 . . 1 0 0 . ; escapes at 4, 5, 9.
    # Offset plane (LSB first): 0b01000110 = 0x46, 0x00.
    # Escape plane: 0b00110000 = 0x30, 0b10 = 0x02.
    dense = np.array([[[120, 121, 121, 120, 7, 254, 121, 120, 120, 0]]], np.uint8)
    enc = oracle.encode(oracle.MXFP4, dense)
    assert enc["base"].tolist() == [120]
    assert enc["offsets"].tolist() == [0x46, 0x00]
    assert enc["escapes"].tolist() == [0x30, 0x02]
    assert enc["exc_index"].tolist() == [0, 3]
    assert enc["exc_bytes"].tolist() == [7, 254, 0]
    out, st = oracle.decode(enc)
    assert st == oracle.OK and np.array_equal(out, dense)


def test_hand_tie_break_smallest_present():
    # MXFP4 windows [10,11] and [20,21] both hold two bytes: the smaller wins.
    enc = oracle.encode(oracle.MXFP4, np.array([[[20, 21, 10, 11]]], np.uint8))
    assert enc["base"].tolist() == [10]
    assert enc["exc_bytes"].tolist() == [20, 21]
    # NVFP4 [5, 19]: window [5, 19] holds both; base 5, offsets 0 and 14.
    enc = oracle.encode(oracle.NVFP4, np.array([[[5, 19]]], np.uint8))
    assert enc["base"].tolist() == [5] and enc["offsets"].tolist() == [0xE0]
    # NVFP4 [5, 20]: two windows of one byte: base 5, 20 is an exception.
    enc = oracle.encode(oracle.NVFP4, np.array([[[5, 20]]], np.uint8))
    assert enc["base"].tolist() == [5] and enc["offsets"].tolist() == [0xF0]
    assert enc["exc_bytes"].tolist() == [20]


def test_hand_decode_wraps_mod_256():
    # A hand-made (non-canonical) stack: element 0 (low nibble) has offset 14
    # on base 0xF8, which wraps to 0x06; element 1 has offset 0.
    enc = {"kind": oracle.NVFP4, "shape": (1, 1, 2),
           "base": np.array([0xF8], np.uint8), "offsets": np.array([0x0E], np.uint8),
           "escapes": np.zeros(0, np.uint8), "exc_index": np.array([0, 0], np.uint32),
           "exc_bytes": np.zeros(0, np.uint8), "num_exc": 0}
    out, st = oracle.decode(enc)
    assert st == oracle.OK and out.ravel().tolist() == [0x06, 0xF8]


def test_hand_all_escape_rows_decode_in_order():
    # Every nibble is the escape code: each row is its exception bytes in order.
    exc = np.arange(100, 112, dtype=np.uint8)
    enc = {"kind": oracle.NVFP4, "shape": (1, 3, 4),
           "base": np.array([1, 2, 3], np.uint8), "offsets": np.full(6, 0xFF, np.uint8),
           "escapes": np.zeros(0, np.uint8), "exc_index": np.array([0, 4, 8, 12], np.uint32),
           "exc_bytes": exc, "num_exc": 12}
    out, st = oracle.decode(enc)
    assert st == oracle.OK and out.ravel().tolist() == exc.tolist()
    assert oracle.check(enc) == oracle.OK


# --------------------------------------------------------- exhaustive / brute

@pytest.mark.parametrize("kind", [oracle.NVFP4, oracle.MXFP4])
def test_exhaustive_c1(kind):
    # Every single-byte row: base is the byte, offset 0, no exception.
    dense = np.arange(256, dtype=np.uint8).reshape(1, 256, 1)
    enc = oracle.encode(kind, dense)
    assert np.array_equal(enc["base"], dense.ravel())
    assert enc["num_exc"] == 0
    assert not enc["offsets"].any()
    out, st = oracle.decode(enc)
    assert st == oracle.OK and np.array_equal(out, dense)


@pytest.mark.parametrize("kind", [oracle.NVFP4, oracle.MXFP4])
def test_exhaustive_c2_closed_form(kind):
    # Every pair (a, b): base = min(a, b) (one window holds both, or two
    # one-byte windows tie and the smaller wins); one exception, max(a, b),
    # exactly when |a - b| > w.
    a, b = np.meshgrid(np.arange(256), np.arange(256), indexing="ij")
    dense = np.stack([a.ravel(), b.ravel()], axis=1).astype(np.uint8).reshape(1, 65536, 2)
    enc = oracle.encode(kind, dense)
    lo = np.minimum(a, b).ravel()
    hi = np.maximum(a, b).ravel()
    far = (hi - lo) > W[kind]
    assert np.array_equal(enc["base"], lo.astype(np.uint8))
    steps = np.diff(enc["exc_index"].astype(np.int64))
    assert np.array_equal(steps, far.astype(np.int64))
    assert np.array_equal(enc["exc_bytes"], hi[far].astype(np.uint8))
    out, st = oracle.decode(enc)
    assert st == oracle.OK and np.array_equal(out, dense)


def _brute_rows(rows: np.ndarray, w: int):
    """Brute force over all 256 window starts, independent of the oracle."""
    best_counts, bases = [], []
    for x in rows:
        counts = np.array([np.count_nonzero((x >= v) & (x <= v + w)) for v in range(256)])
        present = np.zeros(256, bool)
        present[x] = True
        m = counts[present].max()
        best_counts.append(counts.max())
        bases.append(int(np.flatnonzero(present & (counts == m))[0]))
    return np.array(best_counts), np.array(bases)


@pytest.mark.parametrize("kind", [oracle.NVFP4, oracle.MXFP4])
@pytest.mark.parametrize("C", [1, 3, 7, 8, 15, 16, 17, 50, 100, 160])
def test_minimal_exceptions_and_base_brute_force(kind, C):
    rows = synth.random_rows(seed=C * 7 + kind, rows=64, C=C,
                             spread=3 * W[kind] + 3, replace_p=0.1)
    enc = oracle.encode(kind, rows.reshape(1, 64, C))
    best, bases = _brute_rows(rows, W[kind])
    # The global maximum over all 256 starts is reached at a present value.
    assert np.array_equal(enc["base"], bases.astype(np.uint8))
    steps = np.diff(enc["exc_index"].astype(np.int64))
    assert np.array_equal(steps, C - best)
    out, st = oracle.decode(enc)
    assert st == oracle.OK and np.array_equal(out.reshape(64, C), rows)


def _nibbles(offsets: np.ndarray, n: int) -> np.ndarray:
    lo = offsets & 0xF
    hi = offsets >> 4
    return np.stack([lo, hi], axis=1).ravel()[:n]


def test_constant_rows_and_extremes():
    dense = np.full((2, 3, 5), 0x77, np.uint8)
    enc = oracle.encode(oracle.NVFP4, dense)
    assert (enc["base"] == 0x77).all() and not enc["offsets"].any() and enc["num_exc"] == 0
    # A row holding 0 and 255 always has at least one exception.
    row = np.array([[[0, 255, 7, 3]]], np.uint8)
    for kind in (oracle.NVFP4, oracle.MXFP4):
        assert oracle.encode(kind, row)["num_exc"] >= 1


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("name", ["tiny"])
def test_index_invariants_and_escape_counts(name):
    dense = synth.stack(name)
    E, R, C = dense.shape
    enc = oracle.encode(oracle.NVFP4, dense)
    idx = enc["exc_index"].astype(np.int64)
    assert idx[0] == 0 and (np.diff(idx) >= 0).all() and idx[-1] == enc["num_exc"]
    nib = _nibbles(enc["offsets"], E * R * C).reshape(E * R, C)
    assert np.array_equal(np.diff(idx), (nib == 0xF).sum(axis=1))
    # Escaped positions hold exactly the bytes outside [base, base+14], in order.
    flat = dense.reshape(E * R, C)
    assert np.array_equal(enc["exc_bytes"], flat[nib == 0xF])
    off_ok = nib != 0xF
    recon = (enc["base"][:, None].astype(np.int64) + nib) & 0xFF
    assert np.array_equal(recon[off_ok], flat[off_ok])
    assert oracle.check(enc) == oracle.OK


def test_check_flags_inconsistent_index():
    enc = oracle.encode(oracle.NVFP4, synth.stack("tiny"))
    bad = dict(enc)
    bad["exc_index"] = enc["exc_index"].copy()
    bad["exc_index"][5] += 1
    assert oracle.check(bad) == oracle.ERR_CORRUPT
    bad = dict(enc)
    bad["num_exc"] = enc["num_exc"] - 1
    bad["exc_bytes"] = enc["exc_bytes"][:-1]
    assert oracle.check(bad) == oracle.ERR_CORRUPT
    _, st = oracle.decode(bad)
    assert st == oracle.ERR_CORRUPT


def test_routed_decode_equals_masked_full_decode():
    dense = synth.stack("tiny")
    enc = oracle.encode(oracle.NVFP4, dense)
    start = np.array([0, 3, 3, 4, 4], np.int64)        # experts 0 and 2 active
    out = np.full(dense.shape, 0xFF, np.uint8)
    out, st = oracle.decode(enc, start, out)
    assert st == oracle.OK
    assert np.array_equal(out[[0, 2]], dense[[0, 2]])
    assert (out[[1, 3]] == 0xFF).all()
    # Decreasing or negative steps count as inactive.
    out2, _ = oracle.decode(enc, np.array([5, 3, 4, 4, -1], np.int64),
                            np.full(dense.shape, 0xAA, np.uint8))
    assert np.array_equal(out2[1], dense[1]) and (out2[[0, 2, 3]] == 0xAA).all()


@pytest.mark.parametrize("kind", [oracle.NVFP4, oracle.MXFP4])
def test_row_range_decode_is_the_input_rows(kind):
    """Row-range decode ("decode only consumed gate halves", [B478] pairing
    commit message): rows [lo, hi) of each written expert are the original
    input rows and every other byte keeps its old value.  Rows that start
    mid-expert take their exceptions from their own index entry, which a
    rank counted from the expert's first row would get wrong."""
    E, R, C = 3, 10, 9
    dense = synth.random_rows(7, E * R, C, spread=24, replace_p=0.3).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    assert enc["num_exc"] > 20
    for lo, hi in [(0, R), (0, R // 2), (R // 2, R), (3, 4), (7, 10)]:
        out, st = oracle.decode(enc, None, np.full(dense.shape, 0x5A, np.uint8), rows=(lo, hi))
        assert st == oracle.OK
        assert np.array_equal(out[:, lo:hi], dense[:, lo:hi])
        assert (out[:, :lo] == 0x5A).all() and (out[:, hi:] == 0x5A).all()
    # Routing and row range together; an empty range writes nothing.
    start = np.array([0, 0, 2, 2], np.int64)               # expert 1 only
    out, _ = oracle.decode(enc, start, np.full(dense.shape, 0x5A, np.uint8), rows=(2, 6))
    assert np.array_equal(out[1, 2:6], dense[1, 2:6])
    out[1, 2:6] = 0x5A
    assert (out == 0x5A).all()
    out, st = oracle.decode(enc, None, np.full(dense.shape, 0x5A, np.uint8), rows=(4, 4))
    assert st == oracle.OK and (out == 0x5A).all()
    for bad in [(-1, 3), (2, R + 1), (5, 4)]:
        assert oracle.decode(enc, None, None, rows=bad)[1] == oracle.ERR_ARG


# ------------------------------------------------------------------- sizes

@pytest.mark.parametrize("kind,E,R,C", [(0, 3, 5, 7), (0, 2, 4, 100), (1, 3, 5, 7), (1, 2, 4, 160)])
def test_stream_sizes_closed_form(kind, E, R, C):
    sz = oracle.stream_bytes(kind, E, R, C)
    n = E * R * C
    if kind == oracle.NVFP4:
        assert sz["offsets"] == (n + 1) // 2 and sz["escapes"] == 0
    else:
        assert sz["offsets"] == (n + 7) // 8 == sz["escapes"]
    assert sz["base"] == E * R and sz["index_entries"] == E * R + 1
    enc = oracle.encode(kind, synth.random_rows(1, E * R, C).reshape(E, R, C))
    assert enc["offsets"].size == sz["offsets"] and enc["base"].size == E * R


def _golden_sizes():
    """The size figures printed on the finegrained-kernels page (size
    paragraph), from tests/golden/csf_sizes.txt: name -> (dense, compressed)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "csf_sizes.txt")
    out = {}
    with open(path) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                name, dense, comp, _unit = ln.split("\t")
                out[name] = (float(dense), float(comp))
    return out


def test_size_against_pages_figures():
    # The size paragraph reports 28.68 MB (gate, C=100) and 27.99 MB (down,
    # C=50) for 52.43 MB dense per 512-expert stack.  Offsets (N/2) plus one
    # base byte per row must not exceed those, which a byte-per-scale or
    # 8-bit-offset layout would; the rest is the exception stream: the
    # implied exception rates must be "a few percent".
    g = _golden_sizes()
    dense_bytes = 512 * 1024 * 100
    assert abs(g["gate_stack"][0] * 1e6 - dense_bytes) < 0.01e6
    assert abs(g["down_stack"][0] * 1e6 - dense_bytes) < 0.01e6
    for (_, reported_mb), C in ((g["gate_stack"], 100), (g["down_stack"], 50)):
        reported = reported_mb * 1e6
        rows = dense_bytes // C
        fixed = dense_bytes / 2 + rows
        assert fixed < reported
        rate = (reported - fixed) / dense_bytes
        assert 0.005 < rate < 0.05
    # The whole checkpoint's planes (gate, up and down of every layer) shrink
    # from 7.03 to 3.69 GiB: above the 4-bit floor of one half, by less than a
    # base byte per 16 scales plus a few percent of exceptions.
    dense, comp = g["all_planes"]
    assert 0.5 < comp / dense < 0.5 + 1 / 16 + 0.05
    # A synthetic gate-shaped stack at a few percent exceptions lands in the
    # pages' 53-55% band, and its size is the closed form exactly.
    dense = synth.gate_stack(E=8, replace_p=0.039)
    enc = oracle.encode(oracle.NVFP4, dense)
    total = enc["offsets"].size + enc["base"].size + enc["num_exc"]
    n = dense.size
    assert total == (n + 1) // 2 + n // 100 + enc["num_exc"]
    assert 0.53 <= total / n <= 0.55


# ------------------------------------------- scale-operand (blocked) layout
# The 128 x 4 tiled scale layout that Blackwell block-scaled GEMMs read
# (cuBLASLt's documented block-scaling-factor layout; PyTorch calls it the
# 32_4_4 swizzle): per expert, 128-row x 4-column tiles of 512 bytes, row
# blocks outer and column blocks inner; inside a tile, 16-byte line b holds
# rows b, b+32, b+64, b+96 with four columns each.

def _reshape_form(dense: np.ndarray) -> np.ndarray:
    """The layout written as a tensor permutation, independent of the
    oracle's index arithmetic: pad to (128k, 4m), split into 128 x 4 tiles,
    order tiles row-block-major, then within a tile view rows as (4, 32) and
    move the 32 outermost."""
    E, R, C = dense.shape
    RP, CP = -(-R // 128) * 128, -(-C // 4) * 4
    pad = np.zeros((E, RP, CP), np.uint8)
    pad[:, :R, :C] = dense
    t = pad.reshape(E, RP // 128, 128, CP // 4, 4).transpose(0, 1, 3, 2, 4)   # E, rb, cb, 128, 4
    t = t.reshape(E, RP // 128, CP // 4, 4, 32, 4).transpose(0, 1, 2, 4, 3, 5)  # rows as (4, 32) -> (32, 4)
    return t.reshape(-1)


def test_blocked_layout_hand_lines():
    # dense[r, c] = r: line b of the tile is rows b, b+32, b+64, b+96, each
    # repeated for its four columns.
    R, C = 128, 4
    dense = np.repeat(np.arange(R, dtype=np.uint8)[:, None], C, axis=1)[None]
    out, st = oracle.decode_blocked(oracle.encode(oracle.NVFP4, dense))
    assert st == oracle.OK and out.size == 512
    assert out[:16].tolist() == [0] * 4 + [32] * 4 + [64] * 4 + [96] * 4
    assert out[16:32].tolist() == [1] * 4 + [33] * 4 + [65] * 4 + [97] * 4
    assert out[496:].tolist() == [31] * 4 + [63] * 4 + [95] * 4 + [127] * 4
    # dense[r, c] = c: every 4-byte group is 0 1 2 3.
    dense = np.tile(np.arange(C, dtype=np.uint8), (R, 1))[None]
    out, _ = oracle.decode_blocked(oracle.encode(oracle.NVFP4, dense))
    assert (out.reshape(-1, 4) == np.arange(4)).all()
    # Two column blocks (C = 8): tile (row block 0, column block 1) follows
    # tile 0 and holds columns 4..7.
    dense = np.tile(np.arange(8, dtype=np.uint8), (R, 1))[None]
    out, _ = oracle.decode_blocked(oracle.encode(oracle.NVFP4, dense))
    assert (out[:512].reshape(-1, 4) == np.arange(4)).all()
    assert (out[512:].reshape(-1, 4) == np.arange(4, 8)).all()


@pytest.mark.parametrize("kind,E,R,C", [(0, 2, 128, 4), (0, 3, 200, 7), (0, 2, 256, 100), (1, 2, 130, 160),
                                        (0, 1, 1, 1), (1, 3, 64, 33)])
def test_blocked_layout_equals_reshape_form_and_pads_zero(kind, E, R, C):
    w = 14 if kind == oracle.NVFP4 else 1
    dense = synth.random_rows(E + R + C, E * R, C, spread=w + 3, replace_p=0.1).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    out, st = oracle.decode_blocked(enc, out=np.full(oracle.blocked_bytes(E, R, C), 0xAB, np.uint8))
    assert st == oracle.OK
    assert np.array_equal(out, _reshape_form(dense))
    # Every byte written once: the padding is zero, the rest a permutation.
    ones = np.full_like(dense, 0xFF)
    po, _ = oracle.decode_blocked(oracle.encode(kind, ones))
    assert int((po == 0xFF).sum()) == dense.size and int((po == 0).sum()) == po.size - dense.size


def test_blocked_row_blocks_and_routing_leave_other_tiles():
    E, R, C = 3, 300, 12                        # row blocks [0,128) [128,256) [256,300)+pad
    dense = synth.random_rows(9, E * R, C, spread=17, replace_p=0.1).reshape(E, R, C)
    enc = oracle.encode(oracle.NVFP4, dense)
    full, _ = oracle.decode_blocked(enc)
    per_expert = full.size // E
    tile_rows = 3 * 512                         # bytes of one row block (3 column blocks)
    start = np.array([0, 1, 1, 4], np.int64)   # experts 0 and 2
    for lo, hi in [(128, 256), (128, R), (0, 128), (256, R)]:
        out, st = oracle.decode_blocked(enc, start, np.full(full.size, 0x5A, np.uint8), rows=(lo, hi))
        assert st == oracle.OK
        want = np.full(full.size, 0x5A, np.uint8)
        for e in (0, 2):
            a = e * per_expert + (lo // 128) * tile_rows
            b = e * per_expert + (-(-hi // 128)) * tile_rows
            want[a:b] = full[a:b]
        assert np.array_equal(out, want), (lo, hi)
    for bad in [(1, 128), (0, 100), (128, 128), (0, R + 1)]:
        assert oracle.decode_blocked(enc, None, None, rows=bad)[1] == oracle.ERR_ARG


# ------------------------------------------------ tile-packed (stage-readable)
# The same per-row bases and codes stored in GEMM-tile order: inside a 128 x 4
# tile, position q = 16*b + 4*a + c is row b + 32*a, column c (the tile's byte
# order in the blocked layout); bases in the same line order per row block.

def test_tiled_hand_worked_tile():
    R, C = 128, 4
    base = 0x20 + (np.arange(R) % 8)
    dense = (base[:, None] + np.arange(C)[None, :]).astype(np.uint8)
    dense[33, 2] = 0xFF                                  # row 33 = line 1, a = 1; column 2 -> q = 22
    enc = oracle.encode(oracle.NVFP4, dense[None])
    assert enc["base"].tolist() == base.tolist()
    tp = oracle.tiled_pack(enc)
    # codes: nibbles 0 1 2 3 per line-row group -> bytes 0x10 0x32, except q = 22 (escape 15)
    want = np.tile(np.array([0x10, 0x32], np.uint8), 128)
    want[11] = 0x3F
    assert np.array_equal(tp["codes"], want)
    # bases in line order: byte 4*b + a = base of row b + 32*a
    assert tp["bases"].tolist() == [0x20 + (b % 8) for b in range(32) for a in range(4)]
    assert tp["tile_index"].tolist() == [0, 1] and tp["exc_bytes"].tolist() == [0xFF]


def test_tiled_mxfp4_bits():
    R, C = 128, 8                                        # two column tiles
    dense = np.full((R, C), 120, np.uint8)
    dense[:, 1] = 121                                    # offset bit 1 in column 1
    dense[5, 6] = 7                                      # exception: row 5 (line 5, a = 0), tile 1, c = 2
    enc = oracle.encode(oracle.MXFP4, dense[None])
    tp = oracle.tiled_pack(enc)
    t0, t1 = tp["codes"][:128], tp["codes"][128:]
    # tile 0: offset bit set at every q with q % 4 == 1 -> 0x22 in every byte; no escapes
    assert (t0[:64] == 0x22).all() and not t0[64:].any()
    # tile 1 (columns 4..7): no offsets; escape at q = 16*5 + 2 = 82 -> byte 10, bit 2
    assert not t1[:64].any()
    esc = np.zeros(64, np.uint8)
    esc[10] = 0x04
    assert np.array_equal(t1[64:], esc)
    assert tp["tile_index"].tolist() == [0, 0, 1] and tp["exc_bytes"].tolist() == [7]


@pytest.mark.parametrize("kind,E,R,C", [(0, 3, 200, 7), (0, 2, 256, 100), (1, 2, 130, 160), (1, 3, 64, 33),
                                        (0, 1, 1, 1), (0, 2, 300, 50)])
def test_tiled_round_trip_equals_blocked_decode(kind, E, R, C):
    w = W[kind]
    dense = synth.random_rows(R + C, E * R, C, spread=w + 5, replace_p=0.1).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    tp = oracle.tiled_pack(enc)
    assert tp["num_exc"] == enc["num_exc"]
    assert sorted(tp["exc_bytes"].tolist()) == sorted(enc["exc_bytes"].tolist())
    nb = oracle.blocked_bytes(E, R, C)
    out, st = oracle.tiled_decode(tp, None, np.full(nb, 0xAB, np.uint8))
    want, _ = oracle.decode_blocked(enc)
    assert st == oracle.OK and np.array_equal(out, want)
    start = np.concatenate([[0], np.cumsum(np.arange(E) % 2)]).astype(np.int64)   # odd experts
    out, _ = oracle.tiled_decode(tp, start, np.full(nb, 0xAB, np.uint8))
    want, _ = oracle.decode_blocked(enc, start, np.full(nb, 0xAB, np.uint8))
    assert np.array_equal(out, want)


@pytest.mark.parametrize("kind,E,R,C", [(0, 3, 300, 50), (1, 2, 260, 33), (0, 2, 128, 100)])
def test_tiled_row_block_ranges_match_csf(kind, E, R, C):
    # A 128-row block is a run of consecutive rows, so its exceptions take the
    # same range of the tile-ordered stream as of CSF's row-major one: the
    # tile index at a block's first tile is the CSF index at its first row,
    # and the bytes in that range are the same bytes, reordered.  (The GPU
    # conversion from CSF relies on this to place each block without a scan.)
    w = W[kind]
    dense = synth.random_rows(E * R + C, E * R, C, spread=w + 7, replace_p=0.12).reshape(E, R, C)
    enc = oracle.encode(kind, dense)
    tp = oracle.tiled_pack(enc)
    nrb, ncb = -(-R // 128), -(-C // 4)
    T = nrb * ncb
    for e in range(E):
        for rb in range(nrb):
            r0 = e * R + 128 * rb
            r1 = e * R + min(128 * (rb + 1), R)
            lo, hi = int(enc["exc_index"][r0]), int(enc["exc_index"][r1])
            t0 = e * T + rb * ncb
            assert int(tp["tile_index"][t0]) == lo
            assert int(tp["tile_index"][t0 + ncb]) == hi
            assert sorted(tp["exc_bytes"][lo:hi].tolist()) == sorted(enc["exc_bytes"][lo:hi].tolist())

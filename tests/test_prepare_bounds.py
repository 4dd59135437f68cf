"""The GPU prepare's fast base search, restated on the CPU and checked against
the oracle's canonical base rule.

The base of a row is the smallest byte present in it whose window [v, v+w]
(w = 14 NVFP4, 1 MXFP4) holds the most of its bytes ("finegrained-kernels:
decode losslessly compressed NVFP4 scales (CSF)", format paragraph; the
smallest-value tie rule is this library's reading).  The prepare kernels do
not evaluate all 256 windows: they look near the median m of five of the
row's bytes (columns 0, C/4, C/2, 3C/4, C-1) and accept the answer only when
a bound proves no other window can beat it; otherwise the row's warp applies
the exact rule.  These tests restate the two bounds in Python, as the kernels
state them, and require that every row the bound accepts gets exactly the
oracle's base and window count.  They also check that the fallback stays rare
on the synthetic stacks, which is what the kernels' speed relies on.

  NVFP4: 32 bins for the values [a, a + 32), a = clamp(m - 16, 0, 224), plus
    the count of bytes outside them.  The best window lying inside the bins
    is accepted when windows starting below a (at most out + bytes in
    [a, a + w)) hold strictly fewer bytes and windows past the bins (at most
    out + bytes in the last w bins) hold no more; with a + 32 = 256 every
    window is inside.
  MXFP4: counts c0, c1, c2 of the values a, a + 1, a + 2, a = clamp(m - 1, 0,
    253); the better of the windows at a and a + 1 is accepted when windows
    below a hold at most C - c1 - c2 < M bytes and windows above a + 1 at
    most C - c0 - c1 <= M.
"""
import numpy as np
import pytest

import oracle
from lossless_nvfp4_scale_gb300 import synth


def _median5(row):
    C = row.size
    return int(np.sort(row[[0, C // 4, C // 2, (3 * C) // 4, C - 1]].astype(np.int64))[2])


def _fast_nvfp4(row):
    w, n = 14, 32
    C = row.size
    a = min(max(_median5(row) - 16, 0), 256 - n)
    d = row.astype(np.int64) - a
    inside = (d >= 0) & (d < n)
    h = np.bincount(d[inside], minlength=n)
    out = C - int(inside.sum())
    top = a + n == 256
    best = None                                      # (count, -value): ties go to the smaller value
    for j in range(n):
        if h[j] == 0:
            continue
        if j + w < n:
            cnt = int(h[j:j + w + 1].sum())
        elif top:
            cnt = int(h[j:].sum())                   # truncated at 255
        else:
            continue                                 # reaches past the bins: not exact
        if best is None or (cnt, -(a + j)) > best:
            best = (cnt, -(a + j))
    if best is None:
        return None
    M = best[0]
    ok_low = a == 0 or out + int(h[:w].sum()) < M
    ok_high = top or out + int(h[n - w:].sum()) <= M
    return (-best[1], M) if ok_low and ok_high else None


def _fast_mxfp4(row):
    C = row.size
    a = min(max(_median5(row) - 1, 0), 253)
    c0, c1, c2 = (int((row == a + k).sum()) for k in range(3))
    best = None
    if c0:
        best = (c0 + c1, -a)
    if c1 and (best is None or (c1 + c2, -(a + 1)) > best):
        best = (c1 + c2, -(a + 1))
    if best is None:
        return None
    M = best[0]
    ok_low = a == 0 or C - c1 - c2 < M
    ok_high = C - c0 - c1 <= M
    return (-best[1], M) if ok_low and ok_high else None


def _oracle_bases(kind, rows):
    n, C = rows.shape
    enc = oracle.encode(kind, rows.reshape(1, n, C))
    counts = C - np.diff(enc["exc_index"].astype(np.int64))
    return enc["base"].astype(np.int64), counts


def _check(kind, rows):
    fast = _fast_nvfp4 if kind == oracle.NVFP4 else _fast_mxfp4
    base, count = _oracle_bases(kind, rows)
    fallbacks = 0
    for i, r in enumerate(rows):
        got = fast(r)
        if got is None:
            fallbacks += 1
            continue
        assert got == (base[i], count[i]), (kind, i, got, base[i], count[i], r.tolist())
    return fallbacks / len(rows)


def _adversarial(kind, C, seed, n=400):
    rng = np.random.default_rng(seed)
    w = 14 if kind == oracle.NVFP4 else 1
    probes = sorted({0, C // 4, C // 2, (3 * C) // 4, C - 1})
    rows = []
    for _ in range(n // 8):
        rows.append(rng.integers(0, 256, C))                                   # flat
        b = int(rng.integers(0, 256 - w))
        r = b + rng.integers(0, w + 1, C)
        r[probes] = (b + 128 + rng.integers(0, 60, len(probes))) % 256         # every probe an outlier
        rows.append(r)
        b1, b2 = int(rng.integers(0, 100)), int(rng.integers(140, 256 - w))
        rows.append(rng.permutation(np.concatenate([b1 + rng.integers(0, w + 1, C // 2),
                                                    b2 + rng.integers(0, w + 1, C - C // 2)])))   # twin clusters
        rows.append(np.clip(255 - rng.integers(0, w + 3, C), 0, 255))            # top of the range
        rows.append(np.clip(rng.integers(0, w + 3, C), 0, 255))                  # bottom
        m = int(rng.integers(3, 250))
        rows.append(rng.choice([m - 1, m, m + 1], C))                            # windows beside the median tie
        rows.append(np.where(rng.random(C) < 0.5, m + 2, m + 3))                 # best window above the counted ones
        k = int(rng.integers(1, 6))
        rows.append(rng.choice(rng.integers(0, 256, k), C))                      # a few values
    return np.array(rows, dtype=np.uint8)


@pytest.mark.parametrize("C", [100, 50, 7, 255])
def test_nvfp4_bound_never_accepts_a_wrong_base(C):
    _check(oracle.NVFP4, _adversarial(oracle.NVFP4, C, seed=C))


@pytest.mark.parametrize("C", [160, 100, 33, 5, 2])
def test_mxfp4_bound_never_accepts_a_wrong_base(C):
    _check(oracle.MXFP4, _adversarial(oracle.MXFP4, C, seed=1000 + C))


def test_bounds_settle_the_synthetic_stacks_fast():
    # The pages' workloads, as the synthetic stacks model them: the bound
    # settles almost every row, so the exact fallback stays rare.
    gate = synth.gate_stack(seed=0, E=8)
    down = synth.down_stack(seed=0, E=4)
    mx = synth.mxfp4_stack(seed=0, E=4)
    assert _check(oracle.NVFP4, gate.reshape(-1, gate.shape[-1])[:4000]) < 0.005
    assert _check(oracle.NVFP4, down.reshape(-1, down.shape[-1])[:4000]) < 0.02
    assert _check(oracle.MXFP4, mx.reshape(-1, mx.shape[-1])[:4000]) < 0.02

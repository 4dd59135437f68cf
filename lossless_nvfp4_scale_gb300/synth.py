"""Seeded synthetic scale stacks shaped like the pages' workloads.

This module only draws random bytes; it holds none of the codec's arithmetic
and is shared by the tests, the benchmark and the smoke check as the single
source of inputs for both the CUDA path and the CPU oracle.

Workloads (sizes and value distributions from the pages' measured stacks):
  * tiny      4 x 64 x 8     NVFP4, row base U[0x20, 0x60], offsets U{0..14},
                             3% of entries replaced by U{0..255}.
  * gate      512 x 1024 x 100 NVFP4 (52.43 MB dense), base U[0x28, 0x50],
                             offsets clip(rint(N(6, 3)), 0, 14), 2% replaced.
  * down      512 x 2048 x 50 NVFP4 (52.43 MB), base U[0x28, 0x50],
                             deviation floor(exp(N(1.303, 1))) capped at
                             255 - base: the heavy tail past 14 makes ~8%
                             exceptions.
  * mxfp4     384 x 2048 x 160 UE8M0 (125.8 MB), base U{118..126}; w.p. 0.85
                             base + Bernoulli(1/2), else uniform over
                             {0..254} minus {base, base+1}.
  * routing   8 of E experts uniform without replacement, 64 tokens: one to
                             each, the other 56 uniform among the 8; the
                             expert_start prefix is the exclusive cumsum (E+1).

Generation is chunked over experts so memory stays bounded; the chunking is
fixed, so the bytes depend on the seed only.
"""
from __future__ import annotations

import numpy as np

CHUNK_EXPERTS = 16

WORKLOADS = {
    "tiny": dict(kind=0, E=4, R=64, C=8),
    "gate": dict(kind=0, E=512, R=1024, C=100),
    "down": dict(kind=0, E=512, R=2048, C=50),
    "mxfp4": dict(kind=1, E=384, R=2048, C=160),
}


def _uniform_rows(rng, e, R, C, base_lo, base_hi, replace_p, offsets_fn):
    base = rng.integers(base_lo, base_hi + 1, size=(e, R, 1), dtype=np.int64)
    off = offsets_fn(rng, (e, R, C))
    vals = base + off
    repl_mask = rng.random((e, R, C)) < replace_p
    repl = rng.integers(0, 256, size=(e, R, C), dtype=np.int64)
    return np.where(repl_mask, repl, vals).astype(np.uint8)


def tiny_stack(seed: int = 0, E: int = 4, R: int = 64, C: int = 8,
               replace_p: float = 0.03) -> np.ndarray:
    """Base U[0x20,0x60] per row, offsets U{0..14}, replace_p random bytes."""
    rng = np.random.default_rng(seed)
    out = np.empty((E, R, C), np.uint8)
    for e0 in range(0, E, CHUNK_EXPERTS):
        e = min(CHUNK_EXPERTS, E - e0)
        out[e0:e0 + e] = _uniform_rows(
            rng, e, R, C, 0x20, 0x60, replace_p,
            lambda g, s: g.integers(0, 15, size=s, dtype=np.int64))
    return out


def gate_stack(seed: int = 0, E: int = 512, R: int = 1024, C: int = 100,
               replace_p: float = 0.02) -> np.ndarray:
    """Base U[0x28,0x50], offsets clip(rint(N(6,3)),0,14), replace_p random."""
    rng = np.random.default_rng(seed)
    out = np.empty((E, R, C), np.uint8)

    def offs(g, s):
        return np.clip(np.rint(g.normal(6.0, 3.0, size=s)), 0, 14).astype(np.int64)

    for e0 in range(0, E, CHUNK_EXPERTS):
        e = min(CHUNK_EXPERTS, E - e0)
        out[e0:e0 + e] = _uniform_rows(rng, e, R, C, 0x28, 0x50, replace_p, offs)
    return out


def down_stack(seed: int = 0, E: int = 512, R: int = 2048, C: int = 50) -> np.ndarray:
    """Base U[0x28,0x50] plus a log-normal deviation, capped at 255 - base."""
    rng = np.random.default_rng(seed)
    out = np.empty((E, R, C), np.uint8)
    for e0 in range(0, E, CHUNK_EXPERTS):
        e = min(CHUNK_EXPERTS, E - e0)
        base = rng.integers(0x28, 0x51, size=(e, R, 1), dtype=np.int64)
        dev = np.floor(np.exp(rng.normal(1.303, 1.0, size=(e, R, C)))).astype(np.int64)
        dev = np.minimum(dev, 255 - base)
        out[e0:e0 + e] = (base + dev).astype(np.uint8)
    return out


def mxfp4_stack(seed: int = 0, E: int = 384, R: int = 2048, C: int = 160) -> np.ndarray:
    """UE8M0 exponents: base U{118..126}; 85% base or base+1, rest spread."""
    rng = np.random.default_rng(seed)
    out = np.empty((E, R, C), np.uint8)
    for e0 in range(0, E, CHUNK_EXPERTS):
        e = min(CHUNK_EXPERTS, E - e0)
        base = rng.integers(118, 127, size=(e, R, 1), dtype=np.int64)
        near = base + rng.integers(0, 2, size=(e, R, C), dtype=np.int64)
        u = rng.integers(0, 253, size=(e, R, C), dtype=np.int64)
        far = np.where(u >= base, u + 2, u)
        keep = rng.random((e, R, C)) < 0.85
        out[e0:e0 + e] = np.where(keep, near, far).astype(np.uint8)
    return out


def stack(name: str, seed: int = 0) -> np.ndarray:
    return {"tiny": tiny_stack, "gate": gate_stack, "down": down_stack,
            "mxfp4": mxfp4_stack}[name](seed)


def routing(E: int = 512, active: int = 8, tokens: int = 64, seed: int = 0,
            dtype=np.int32) -> np.ndarray:
    """Grouped-routing expert_start prefix (E+1 entries) over `tokens` tokens
    routed to `active` experts drawn uniformly without replacement."""
    rng = np.random.default_rng(seed)
    experts = rng.choice(E, size=active, replace=False)
    counts = np.zeros(E, np.int64)
    counts[experts] += 1
    extra = rng.integers(0, active, size=tokens - active)
    np.add.at(counts, experts[extra], 1)
    start = np.zeros(E + 1, np.int64)
    np.cumsum(counts, out=start[1:])
    return start.astype(dtype)


def random_rows(seed: int, rows: int, C: int, spread: int = 40,
                replace_p: float = 0.05) -> np.ndarray:
    """Small mixed rows for property tests: a per-row centre, a narrow spread
    and some uniformly random bytes."""
    rng = np.random.default_rng(seed)
    centre = rng.integers(0, 256, size=(rows, 1))
    vals = (centre + rng.integers(-spread // 2, spread // 2 + 1, size=(rows, C))) % 256
    repl = rng.integers(0, 256, size=(rows, C))
    mask = rng.random((rows, C)) < replace_p
    return np.where(mask, repl, vals).astype(np.uint8)

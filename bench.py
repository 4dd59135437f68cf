"""Benchmark: CSF decode of a 512-expert NVFP4 scale stack on GB300.

One step = one full-stack decode (the whole hot path of a decode call:
expert gating, fixed-stream expand, exception pass, stores) of the
512 x 1024 x 100 gate stack (52.43 MB of dense UE4M3 scale bytes), through the
C ABI.  `value` = dense-scale GB/s, whole job (all ranks).  Also measured in
the same run (the "rows" object): routed 8-of-512 decode, paired gate+down
decode (full and routed), GPU prepare of the gate stack, and MXFP4 prepare and
decode (384 x 2048 x 160).

Timing: the steps are captured in a CUDA graph (16 launches) and replayed back
to back; CUDA events on the launching stream bracket the whole timed region,
so a step's time is the region's time divided by the steps in it (launches
overlap their ramp-up and drain the way they do in serving).  The stack and
workspace rotate over 4 copies (321 MB > 129 MB L2), so every step reads and
writes HBM.  nvidia-smi samples clocks during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun the ranks split the 512 experts into contiguous ranges, each
rank preparing and decoding its own sub-stack (strong scaling; --replicas
gives every rank a whole stack instead, weak scaling); no collective on the
data path; rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSF decode µs & dense-scale GB/s per 512-expert stack; % of HBM roofline"
WORKLOAD = "gate 512x1024x100 NVFP4-CSF full-stack decode"
FALLBACK_HBM_GBS = 6800.0
ROTATE = 4           # stack/workspace copies (working set > L2)
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (context beside the measured copy peak)


def peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples (100 ms) while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def timed_steps(torch, fn, steps, warmup, per_graph=16, hold_s=0.0):
    """Run `fn(i)` `warmup` times eagerly, capture the calls into CUDA graphs
    (`per_graph` calls each, plus one graph for the remainder) and replay them
    back to back for exactly `steps` calls, with CUDA events only around the
    whole timed region (on the launching stream).  Each graph is replayed once,
    untimed, before the region (its first launch uploads it).  With `hold_s`
    > 0 the full graph is then replayed again, untimed, for that long, so a
    clock sampler running around this call sees the same kernel under load.
    Returns (total_ms, steps)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(warmup):
            fn(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    full, rem = divmod(steps, per_graph)
    graphs = []
    for count, reps in ((per_graph, full), (rem, 1 if rem else 0)):
        if reps == 0:
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(count):
                fn(i)
        g.replay()
        graphs.append((g, reps))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for g, reps in graphs:
        for _ in range(reps):
            g.replay()
    e1.record()
    torch.cuda.synchronize()
    if hold_s > 0 and graphs:
        g = graphs[0][0]
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < hold_s:
            for _ in range(64):
                g.replay()
            torch.cuda.synchronize()
    return e0.elapsed_time(e1), steps


def single_launches(torch, fn, n, flush):
    """`n` launches of `fn`, each timed alone with CUDA events on the launching
    stream after `flush` (a buffer of twice the L2 size) is read, outside the
    events.  Reading it evicts every line, and any write-back of dirty lines
    happens before the start event, so each launch starts from a cold, clean
    L2.  The flush also keeps the stream busy while the host enqueues the
    start event and the launch, so the events bracket the kernel only.
    Returns the per-launch times in ms (three untimed launches first)."""
    out = []
    for i in range(n + 3):
        flush.sum()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(i)
        e1.record()
        out.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in out[3:]]


def reduce_max(torch, dist, value, device):
    """Maximum of a per-rank float over all ranks (the job's time is its slowest
    rank's); no data-path collective exists, this is timing only."""
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def stack_traffic(st, rows_active=None, index=True):
    """Algorithmic bytes of one decode: packed streams read (offsets, escape
    plane, bases, exception bytes and, with `index`, the per-row exception
    index) + dense bytes written.  Routed: only the active experts' share.
    The kernel itself reads the index only at the two ends of each warp
    segment; `index=False` gives that read set."""
    sb = st.stream_bytes()
    total_rows = st.E * st.R
    frac = 1.0 if rows_active is None else rows_active / total_rows
    read = (sb["offsets"] + sb["escapes"] + sb["base"] + (sb["exc_index"] if index else 0)) * frac
    exc = sb["exc_bytes"] * frac
    return read + exc + st.dense_bytes * frac


def run_own(args, rank, world, torch, dist):
    from lossless_nvfp4_scale_gb300 import build as b, shard, synth
    b.ensure_built()
    from lossless_nvfp4_scale_gb300 import csf

    dev = torch.cuda.current_device()
    hbm, peak_kind = peak_hbm()
    # N > 1: the ranks split the 512 experts of one stack into contiguous
    # ranges (expert parallel, strong scaling); --replicas gives every rank a
    # whole stack of its own instead (weak scaling).  No data-path collective.
    split = world > 1 and not args.replicas
    E_all = 512
    e0, e1 = shard.expert_range(E_all, world, rank) if split else (0, E_all)

    # ---- headline: full gate decode -------------------------------------
    full = synth.gate_stack(seed=0 if split else rank)
    gate_dense = torch.from_numpy(np.ascontiguousarray(shard.shard_dense(full, e0, e1))).cuda()
    del full
    gate = csf.prepare(gate_dense, csf.NVFP4)
    copies = [gate] + [clone_stack(torch, gate) for _ in range(ROTATE - 1)]
    wss = [torch.empty_like(gate_dense) for _ in range(ROTATE)]

    def step(i):
        k = i % ROTATE
        csf.decode(copies[k], wss[k])

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t0 = time.perf_counter()
        total_ms, steps = timed_steps(torch, step, args.steps, args.warmup, hold_s=args.clock_hold)
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    assert torch.equal(wss[0], gate_dense), "decode output differs from the dense stack"
    assert gate.errors() == 0
    if world > 1:
        total_ms = reduce_max(torch, dist, total_ms, "cuda")
    ms_per_step = total_ms / steps
    job_dense = (E_all * 1024 * 100) if split else world * gate.dense_bytes
    value = job_dense / 1e9 * steps / (total_ms / 1e3)
    alg = stack_traffic(gate)                        # with the per-row index
    alg_kernel = stack_traffic(gate, index=False)    # what the kernel reads
    achieved = alg / (ms_per_step / 1e3) / 1e9
    traffic, traffic_src = profiled_traffic()
    parallelism = (f"expert split x{world}: rank r decodes experts [{e0}, {e1}) of the 512 (no collective)"
                   if split else (f"replicas x{world} (independent stacks, no collective)" if world > 1 else "single GPU"))
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded gate-shaped stack; the pages' checkpoint streams are not available)",
        "config": {"workload": WORKLOAD, "experts": E_all, "rows": 1024, "cols": 100,
                   "experts_this_rank": e1 - e0, "dense_bytes": gate.dense_bytes, "exceptions": gate.num_exc,
                   "l2": f"inputs rotate over {ROTATE} stack+workspace copies "
                         f"({ROTATE * alg / 1e6:.0f} MB > 129 MB L2)",
                   "timing": "exactly `steps` decodes replayed from CUDA graphs (16 per graph plus a "
                             "remainder graph), CUDA events around the whole region",
                   "parallelism": parallelism},
        "us_per_stack": round(1e3 * ms_per_step, 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": peak_kind,
                     "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes": int(alg),
                     "algorithmic_bytes_definition": "offsets + bases + exception index + exception bytes "
                                                     "read, dense bytes written (per-unit figures of the "
                                                     "measurement plan, actual buffer lengths)",
                     "kernel_read_set_bytes": int(alg_kernel),
                     "frac_kernel_read_set": round(alg_kernel / (ms_per_step / 1e3) / 1e9 / hbm, 4),
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4)},
        "gpu_launches": steps,
        "wall_s": round(wall, 3),
    }
    result["clocks"] = clk.summary()
    result["clocks"]["window"] = (f"sampled every 100 ms from before the timed region through {args.clock_hold} s "
                                  "of untimed replays of the same graph right after it")
    if rank == 0 and not args.skip_rows:
        result["rows"] = measure_rows(torch, csf, synth, gate, gate_dense, hbm, args.steps)
        sl = result["rows"].get("gate_single_launch")
        if sl:
            result["roofline"]["single_launch_l2_flushed"] = {
                "median_us": sl["median_us"], "frac": sl["hbm_frac"],
                "frac_kernel_read_set": round(alg_kernel / (sl["median_us"] / 1e6) / 1e9 / hbm, 4)}
    if rank == 0:
        result["e2e"] = measure_e2e(torch, csf, gate, gate_dense)
        if not args.skip_cpu:
            result["cpu_baseline"] = cpu_baseline(synth)
    return result


def clone_stack(torch, st):
    import copy
    c = copy.copy(st)
    c.base, c.offsets, c.exc_index, c.exc_bytes = (t.clone() for t in (st.base, st.offsets, st.exc_index, st.exc_bytes))
    if st.escapes is not None:
        c.escapes = st.escapes.clone()
    c.error_word = torch.zeros_like(st.error_word)
    return c


def profiled_traffic():
    """DRAM bytes per decode launch, read from the committed ncu summary of
    the gate decode if it was taken on the current kernel source (else null).
    Returns (bytes or None, a label of where the figure comes from)."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, "lossless_nvfp4_scale_gb300", "csrc", "csf_decode.cu"), "rb").read()
        digest = hashlib.sha256(src).hexdigest()[:16]
        info = {}
        with open(os.path.join(ROOT, "profiles", "decode_gate_512x1024x100.md")) as f:
            for ln in f:
                if ": " in ln and ln.startswith("- "):
                    k, v = ln[2:].split(": ", 1)
                    info[k.strip()] = v.strip().strip("`")
        if info.get("csf_decode.cu sha256[:16]") == digest:
            return float(info["dram bytes per launch"]), (
                "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the committed profile "
                "summary taken on this kernel source (not measured in this run)")
        return None, "the committed profile summary was taken on another kernel source"
    except Exception:
        return None, "no profile summary"


def tiled_bytes(t):
    """Bytes of a tile-packed stack that a full decode reads: codes, bases,
    tile index and exception bytes."""
    return t.codes.numel() + t.bases.numel() + 4 * t.tile_index.numel() + t.num_exc


def measure_rows(torch, csf, synth, gate, gate_dense, hbm, max_steps):
    """Side figures of the other rows; each row times its default number of
    steps, fewer when the run asks for fewer (short profiling runs)."""
    rows = {}

    def n(k):
        return max(16, min(k, max_steps))

    E = 512
    start = torch.from_numpy(synth.routing(E=E, active=8, tokens=64, seed=0)).cuda()
    active = int((start[1:] > start[:-1]).sum().item())
    ws = torch.full_like(gate_dense, 0xFF)

    def rec(name, timed, alg, extra=None):
        m = timed[0] / timed[1]
        d = {"us": round(1e3 * m, 3), "algorithmic_MB": round(alg / 1e6, 3),
             "GB_s": round(alg / (m / 1e3) / 1e9, 1), "hbm_frac": round(alg / (m / 1e3) / 1e9 / hbm, 4)}
        if extra:
            d.update(extra)
        rows[name] = d

    # routed 8 of 512: latency-bound, 1.25 MB, L2-warm like the pages' warm
    # graph figure; reported next to an empty-launch floor
    durs = timed_steps(torch, lambda i: csf.decode(gate, ws, expert_start=start), n(400), 20)
    rec("routed_8of512", durs, stack_traffic(gate, rows_active=active * 1024), {"l2": "warm"})
    z = torch.zeros(1, device="cuda")
    floor = timed_steps(torch, lambda i: z.add_(1), n(400), 20)
    rows["routed_8of512"]["empty_launch_floor_us"] = round(1e3 * floor[0] / floor[1], 3)
    # the same persistent grid with no active expert: launch, routing prologue, nothing to decode
    none = torch.zeros(E + 1, dtype=start.dtype, device="cuda")
    floor = timed_steps(torch, lambda i: csf.decode(gate, ws, expert_start=none), n(400), 20)
    rows["routed_8of512"]["no_active_expert_us"] = round(1e3 * floor[0] / floor[1], 3)

    # the gate decode one launch at a time: L2 flushed (a 258 MB read) before
    # each launch (median of 50), and warm (one copy decoded back to back, so its 80 MB
    # stay largely in the 129 MB L2; may exceed the HBM bound)
    flush = torch.ones(2 * 129 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")

    def cold(name, fn, alg, extra=None):
        ts = sorted(single_launches(torch, fn, 50, flush))
        med = ts[len(ts) // 2]
        rows[name] = {"l2": "flushed (2 x L2 read before each launch)", "n": len(ts),
                      "median_us": round(1e3 * med, 3), "p10_us": round(1e3 * ts[len(ts) // 10], 3),
                      "p90_us": round(1e3 * ts[(9 * len(ts)) // 10], 3), "algorithmic_MB": round(alg / 1e6, 3),
                      "GB_s": round(alg / (med / 1e3) / 1e9, 1), "hbm_frac": round(alg / (med / 1e3) / 1e9 / hbm, 4)}
        if extra:
            rows[name].update(extra)

    alg = stack_traffic(gate)
    cold("gate_single_launch", lambda i: csf.decode(gate, ws), alg)
    cold("routed_8of512_cold", lambda i: csf.decode(gate, ws, expert_start=start),
         stack_traffic(gate, rows_active=active * 1024))
    durs = timed_steps(torch, lambda i: csf.decode(gate, ws), n(400), 20)
    rec("gate_warm", durs, alg, {"l2": "warm"})

    # gate half of every expert (rows [0, R/2): the stack read as fused
    # gate/up), rotating over 4 copies (4 x 40 MB of inputs > L2)
    hc = [gate] + [clone_stack(torch, gate) for _ in range(3)]
    hw = [torch.empty_like(gate_dense) for _ in range(4)]
    durs = timed_steps(torch, lambda i: csf.decode(hc[i % 4], hw[i % 4], rows=(0, 512)), n(400), 20)
    assert torch.equal(hw[0][:, :512], gate_dense[:, :512])
    rec("gate_half_all", durs, stack_traffic(gate, rows_active=512 * 512))
    del hc, hw

    # the gate stack decoded straight into the block-scaled GEMM scale layout,
    # rotating over 4 copies (4 x 80 MB > L2)
    bc = [gate] + [clone_stack(torch, gate) for _ in range(3)]
    bw = [torch.empty(csf.blocked_bytes(gate), dtype=torch.uint8, device="cuda") for _ in range(4)]
    durs = timed_steps(torch, lambda i: csf.decode(bc[i % 4], bw[i % 4], layout=csf.LAYOUT_BLOCKED), n(400), 20)
    rec("gate_blocked_layout", durs, stack_traffic(gate))

    # the same scales kept tile-packed (stage-readable: each 128 x 4 tile
    # decodes alone) and decoded into the same layout; the pack runs once per
    # stack at load time and is reported beside it
    tps = [csf.tiled_pack(c) for c in bc]
    durs = timed_steps(torch, lambda i: csf.tiled_decode(tps[i % 4], bw[i % 4]), n(400), 20)
    assert torch.equal(bw[0], csf.decode(gate, layout=csf.LAYOUT_BLOCKED))
    packed = tiled_bytes(tps[0])
    pk = timed_steps(torch, lambda i: csf.tiled_pack(bc[i % 4]), n(20), 3)
    rec("gate_tiled_packed", durs, packed + bw[0].numel(),
        {"packed_MB": round(packed / 1e6, 3), "pack_us": round(1e3 * pk[0] / pk[1], 1)})
    # the same tiles rebuilt per stage in shared memory only (the device
    # decoder of include/csf_tile.cuh), one 4-byte checksum per tile written
    sums = [torch.empty(tps[0].tile_index.numel() - 1, dtype=torch.int32, device="cuda") for _ in range(4)]
    durs = timed_steps(torch, lambda i: csf.tiled_checksums(tps[i % 4], sums[i % 4]), n(400), 20)
    rec("gate_tiled_stage_read", durs, packed + 4 * sums[0].numel(),
        {"written_MB": round(4 * sums[0].numel() / 1e6, 3), "decoded_to": "shared memory"})
    del bc, bw, tps, sums

    # the down stack alone (C = 50: lane chunks span up to three rows), then
    # paired with the gate
    down_dense = torch.from_numpy(synth.down_stack(seed=0)).cuda()
    down = csf.prepare(down_dense, csf.NVFP4)
    dc = [down] + [clone_stack(torch, down) for _ in range(3)]
    dw = [torch.empty_like(down_dense) for _ in range(4)]
    durs = timed_steps(torch, lambda i: csf.decode(dc[i % 4], dw[i % 4]), n(400), 20)
    assert torch.equal(dw[0], down_dense)
    rec("decode_down", durs, stack_traffic(down))
    del dc, dw
    gws, dws = torch.empty_like(gate_dense), torch.empty_like(down_dense)
    g2, d2 = clone_stack(torch, gate), clone_stack(torch, down)
    gws2, dws2 = torch.empty_like(gate_dense), torch.empty_like(down_dense)
    pairs = [(gate, down, gws, dws), (g2, d2, gws2, dws2)]
    durs = timed_steps(torch, lambda i: csf.decode_pair(*pairs[i % 2]), n(200), 10)
    assert torch.equal(gws, gate_dense) and torch.equal(dws, down_dense)
    rec("pair_full", durs, stack_traffic(gate) + stack_traffic(down))
    durs = timed_steps(torch, lambda i: csf.decode_pair(gate, down, gws, dws, expert_start=start), n(400), 20)
    pair_routed_alg = stack_traffic(gate, rows_active=active * 1024) + stack_traffic(down, rows_active=active * 2048)
    rec("pair_routed_8of512", durs, pair_routed_alg, {"l2": "warm"})
    cold("pair_routed_8of512_cold", lambda i: csf.decode_pair(gate, down, gws, dws, expert_start=start),
         pair_routed_alg)
    del flush
    del g2, d2, gws2, dws2, pairs

    # ahead-of-call expansion: the gate + down pair expanded on a side stream
    # while the launching stream runs other work of the layer, joined before
    # the step ends.  Two stand-ins for that work: a latency-bound chain of 24
    # small kernels (the GPU mostly idle), and a bf16 GEMM that fills every SM.
    ga = torch.randn(4096, 2048, device="cuda", dtype=torch.bfloat16)
    gb = torch.randn(2048, 4096, device="cuda", dtype=torch.bfloat16)
    gc = torch.empty(4096, 4096, device="cuda", dtype=torch.bfloat16)
    small = torch.ones(1 << 16, device="cuda")
    side = torch.cuda.Stream()

    def chain(i):
        for _ in range(24):
            small.mul_(1.0000001)

    def gemm(i):
        torch.matmul(ga, gb, out=gc)

    def overlapped(work):
        def f(i):
            cur = torch.cuda.current_stream()
            ready = torch.cuda.Event()
            ready.record(cur)
            ev = csf.expand_scales([(gate, gws), (down, dws)], side, after=ready)
            work(i)
            cur.wait_event(ev)
        return f

    def us(fn):
        t = timed_steps(torch, fn, n(200), 10)
        return 1e3 * t[0] / t[1]

    ue = us(lambda i: csf.expand_scales([(gate, gws), (down, dws)]))
    row = {"expand_us": round(ue, 3)}
    for name, work in (("latency_bound_chain", chain), ("gemm_bf16_4096x4096x2048", gemm)):
        uw = us(work)
        ub = us(overlapped(work))
        row[name] = {"work_us": round(uw, 3), "both_us": round(ub, 3), "hidden_frac": round((uw + ue - ub) / ue, 3)}
    assert torch.equal(gws, gate_dense) and torch.equal(dws, down_dense)
    rows["expand_side_stream"] = row
    del ga, gb, gc, small

    # GPU prepare of the gate stack (reads dense once, writes the streams)
    E_, R_, C_ = gate.shape
    psts = [csf.empty_stack(csf.NVFP4, E_, R_, C_, exc_capacity=gate.dense_bytes) for _ in range(2)]
    scrs = [csf.prepare_scratch(csf.NVFP4, E_, R_, C_) for _ in range(2)]
    dens = [gate_dense, gate_dense.clone()]                 # 2 rotating copies: 2 x 82 MB > L2
    durs = timed_steps(torch, lambda i: csf.prepare_async(dens[i % 2], psts[i % 2], scrs[i % 2]), n(100), 5)
    sb = gate.stream_bytes()
    rec("prepare_gate", durs, gate.dense_bytes + sb["offsets"] + sb["base"] + sb["exc_index"] + sb["exc_bytes"])
    del psts, scrs, dens

    # MXFP4: prepare + decode
    mx_dense = torch.from_numpy(synth.mxfp4_stack(seed=0)).cuda()
    mx = csf.prepare(mx_dense, csf.MXFP4)
    E_, R_, C_ = mx.shape
    pst = csf.empty_stack(csf.MXFP4, E_, R_, C_, exc_capacity=mx.dense_bytes)
    scr = csf.prepare_scratch(csf.MXFP4, E_, R_, C_)
    durs = timed_steps(torch, lambda i: csf.prepare_async(mx_dense, pst, scr), n(50), 5)
    sb = mx.stream_bytes()
    rec("prepare_mxfp4", durs, mx.dense_bytes + sb["offsets"] + sb["escapes"] + sb["base"] + sb["exc_index"]
        + sb["exc_bytes"], {"exception_rate": round(mx.num_exc / mx.dense_bytes, 4)})
    mx2 = clone_stack(torch, mx)
    mws = [torch.empty_like(mx_dense), torch.empty_like(mx_dense)]
    mcs = [mx, mx2]
    durs = timed_steps(torch, lambda i: csf.decode(mcs[i % 2], mws[i % 2]), n(100), 5)
    assert torch.equal(mws[0], mx_dense)
    rec("decode_mxfp4", durs, stack_traffic(mx))
    # the MXFP4 workload as one step: prepare the stack, then decode what was
    # just prepared (the bytes of both)
    pst.num_exc = mx.num_exc
    mws[0].zero_()

    def prep_dec(i):
        csf.prepare_async(mx_dense, pst, scr)
        csf.decode(pst, mws[0])

    durs = timed_steps(torch, prep_dec, n(50), 5)
    assert torch.equal(mws[0], mx_dense) and pst.errors() == 0
    rec("mxfp4_prepare_then_decode", durs, 2 * (mx.dense_bytes + sb["offsets"] + sb["escapes"] + sb["base"]
                                              + sb["exc_index"] + sb["exc_bytes"]))
    del pst, scr
    return rows


def measure_e2e(torch, csf, gate, gate_dense, steps=24):
    """Same metric end to end through the public API with HOST buffers: every
    step copies the compressed stack from pinned host memory to the device,
    decodes it, and copies the dense result back to pinned host memory.

    `value` is the pipelined throughput: steps run on three streams (copy in,
    decode, copy out) over two buffer sets, so step i's copy in overlaps
    step i-1's decode and copy out (the link is full duplex); events order
    every buffer's reuse.  `us_per_step_serial` is one step run alone, copy
    in -> decode -> copy out -> synchronise."""
    import copy
    names = ("base", "offsets", "exc_index", "exc_bytes")
    host = {}
    for name in names:
        t = getattr(gate, name)
        host[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[name].copy_(t)
    devs, wss, outs = [], [], []
    for _ in range(2):
        dev = copy.copy(gate)
        for name in names:
            setattr(dev, name, torch.empty_like(getattr(gate, name)))
        devs.append(dev)
        wss.append(torch.empty_like(gate_dense))
        outs.append(torch.empty(gate_dense.shape, dtype=torch.uint8, pin_memory=True))
    h2d = sum(t.numel() * t.element_size() for t in host.values())

    # one step alone
    times = []
    for i in range(6):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for name, t in host.items():
            getattr(devs[0], name).copy_(t, non_blocking=True)
        csf.decode(devs[0], wss[0])
        outs[0].copy_(wss[0], non_blocking=True)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(time.perf_counter() - t0)
    serial = statistics.median(times)

    # pipelined steps
    s_in, s_dec, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_dec = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_dec[b])            # step i-2's decode has read these inputs
                for name, t in host.items():
                    getattr(devs[b], name).copy_(t, non_blocking=True)
                ev_in[b].record(s_in)
            s_dec.wait_event(ev_in[b])
            if i >= 2:
                s_dec.wait_event(ev_out[b])               # step i-2's copy out has read this workspace
            csf.decode(devs[b], wss[b], stream=s_dec)
            ev_dec[b].record(s_dec)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_dec[b])
                outs[b].copy_(wss[b], non_blocking=True)
                ev_out[b].record(s_out)

    run(4)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    t = time.perf_counter() - t0
    assert torch.equal(outs[0], gate_dense.cpu()) and torch.equal(outs[1], gate_dense.cpu())
    return {"value": round(steps * gate.dense_bytes / t / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(gate.dense_bytes),
            "us_per_step": round(1e6 * t / steps, 1), "pipelined": "copy in / decode / copy out on 3 streams",
            "us_per_step_serial": round(1e6 * serial, 1)}


def cpu_baseline(synth, budget_s=8.0):
    """The CPU oracle's decode, as it stands, on a bounded sample (experts of
    the same gate stack), one thread."""
    import oracle
    E = 64
    dense = synth.gate_stack(seed=0, E=E)
    enc = oracle.encode(oracle.NVFP4, dense)
    reps, t = 0, 0.0
    while t < budget_s:
        t0 = time.perf_counter()
        out, st = oracle.decode(enc)
        t += time.perf_counter() - t0
        reps += 1
    assert st == oracle.OK and np.array_equal(out, dense)
    gbs = reps * dense.size / t / 1e9
    # Encode (the CPU counterpart of the GPU prepare), timed separately.
    ereps, et = 0, 0.0
    while et < budget_s / 4:
        t0 = time.perf_counter()
        oracle.encode(oracle.NVFP4, dense)
        et += time.perf_counter() - t0
        ereps += 1
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{E} of the 512 experts ({dense.size / 1e6:.1f} MB dense), {reps} decodes, "
                      f"{t:.1f} s, 1 thread; us per 512-expert stack = {1e6 * 512 / E * t / reps:.0f}",
            "encode_GB_s": round(ereps * dense.size / et / 1e9, 4),
            "host": {"cpu": cpu_model(), "nproc": os.cpu_count()}}


def cpu_model() -> str:
    """CPU model string of the host, from /proc/cpuinfo (x86 `model name`, Arm
    `CPU part` and implementer otherwise)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for ln in info:
            if ln.startswith(key) and ":" in ln:
                return ln.split(":", 1)[1].strip()
    parts = sorted({ln.split(":", 1)[1].strip() for ln in info if ln.startswith(("CPU implementer", "CPU part"))})
    return "arm " + " ".join(parts) if parts else "unknown"


def run_reference(args, world=1):
    """The CPU oracle as the reference arm: same metric and workload, each
    step decodes a bounded sample (16 experts) of the gate stack."""
    import oracle
    from lossless_nvfp4_scale_gb300 import synth
    E = 16
    dense = synth.gate_stack(seed=0, E=E)
    enc = oracle.encode(oracle.NVFP4, dense)
    for _ in range(args.warmup):
        oracle.decode(enc)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        out, st = oracle.decode(enc)
    t = time.perf_counter() - t0
    assert st == oracle.OK and np.array_equal(out, dense)
    value = args.steps * dense.size / t / 1e9
    sample = f"{E} of the 512 experts per step ({dense.size / 1e6:.2f} MB dense), 1 thread"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t / args.steps, 3),
            "higher_is_better": True, "scaling": "strong" if world > 1 else "weak", "vs_baseline": None,
            "dtype": "u8", "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--skip-rows", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--replicas", action="store_true",
                    help="N > 1: every rank decodes a whole stack of its own (weak scaling) instead of "
                         "its range of the 512 experts")
    ap.add_argument("--clock-hold", type=float, default=1.0,
                    help="seconds of untimed replays after the timed region, for the clock record")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    res = run_own(args, rank, world, torch, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

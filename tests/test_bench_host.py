"""CPU checks of bench.py's host-side logic (no GPU)."""
import hashlib
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profiled_traffic_matches_the_committed_summary():
    # The roofline's `traffic` comes from the committed ncu summary only when
    # that summary names the current decode source; the line format is
    # "- key: `value`" and the key itself holds a colon ("sha256[:16]").
    src = open(os.path.join(ROOT, "lossless_nvfp4_scale_gb300", "csrc", "csf_decode.cu"), "rb").read()
    digest = hashlib.sha256(src).hexdigest()[:16]
    text = open(os.path.join(ROOT, "profiles", "decode_gate_512x1024x100.md")).read()
    got, source = bench.profiled_traffic()
    if f"`{digest}`" in text:
        assert got is not None and got > 0 and "ncu" in source
    else:
        assert got is None


def test_profiled_traffic_ignores_a_stale_summary(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "lossless_nvfp4_scale_gb300" / "csrc").mkdir(parents=True)
    (tmp_path / "lossless_nvfp4_scale_gb300" / "csrc" / "csf_decode.cu").write_text("// kernel v2\n")
    summary = "- csf_decode.cu sha256[:16]: `{}`\n- dram bytes per launch: `1234`\n"
    stale = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles" / "decode_gate_512x1024x100.md").write_text(summary.format(stale))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic()[0] is None
    fresh = hashlib.sha256(b"// kernel v2\n").hexdigest()[:16]
    (tmp_path / "profiles" / "decode_gate_512x1024x100.md").write_text(summary.format(fresh))
    assert bench.profiled_traffic()[0] == 1234.0


def test_tiled_bytes_counts_every_stream_of_the_packed_gate():
    """512 x 1024 x 100 NVFP4: 102,400 tiles of 256 code bytes, 4,096 row blocks
    of 128 base bytes, a 102,401-entry u32 tile index, plus the exceptions."""
    import types
    E, R, C, exc = 512, 1024, 100, 984_000
    tiles = E * (R // 128) * (C // 4)
    t = types.SimpleNamespace(codes=types.SimpleNamespace(numel=lambda: tiles * 256),
                              bases=types.SimpleNamespace(numel=lambda: E * (R // 128) * 128),
                              tile_index=types.SimpleNamespace(numel=lambda: tiles + 1), num_exc=exc)
    assert bench.tiled_bytes(t) == tiles * 256 + E * 8 * 128 + 4 * (tiles + 1) + exc


class _FakeCuda:
    """Stand-in for torch.cuda that counts the calls a replayed graph makes."""

    def __init__(self):
        self.calls = 0
        self.capturing = None
        cuda = self

        class Graph:
            def __init__(self):
                self.n = 0

            def replay(self):
                cuda.calls += self.n

        class Ctx:
            def __init__(self, g):
                self.g = g

            def __enter__(self):
                cuda.capturing = self.g

            def __exit__(self, *a):
                cuda.capturing = None

        class Event:
            def __init__(self, enable_timing=False):
                self.at = None

            def record(self, stream=None):
                self.at = cuda.calls

            def elapsed_time(self, other):
                return float(other.at - self.at)   # "ms" = calls in between

        class Stream:
            def wait_stream(self, other):
                pass

        self.CUDAGraph = Graph
        self.graph = Ctx
        self.Event = Event
        self.Stream = Stream

    def stream(self, s):
        import contextlib
        return contextlib.nullcontext()

    def current_stream(self):
        return self.Stream()

    def synchronize(self):
        pass


def test_timed_steps_times_exactly_the_requested_steps():
    import types
    for steps in (1, 15, 16, 17, 20, 32, 50):
        cuda = _FakeCuda()
        fake = types.SimpleNamespace(cuda=cuda)

        def fn(i):
            if cuda.capturing is not None:
                cuda.capturing.n += 1
            else:
                cuda.calls += 1

        ms, done = bench.timed_steps(fake, fn, steps, warmup=3)
        assert done == steps
        assert ms == steps          # replays inside the events made exactly `steps` calls

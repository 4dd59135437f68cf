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
    got = bench.profiled_traffic()
    if f"`{digest}`" in text:
        assert got is not None and got > 0
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
    assert bench.profiled_traffic() is None
    fresh = hashlib.sha256(b"// kernel v2\n").hexdigest()[:16]
    (tmp_path / "profiles" / "decode_gate_512x1024x100.md").write_text(summary.format(fresh))
    assert bench.profiled_traffic() == 1234.0


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

"""The C ABI used from plain C, with no Python binding and no PyTorch:
tests/c_abi_roundtrip.c links libcsf.so and the CUDA runtime, prepares a
seeded stack, decodes it whole and routed, and compares bytes on the host."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_round_trip_from_c(tmp_path):
    from lossless_nvfp4_scale_gb300 import build
    lib = build.ensure_built()
    nvcc = build.nvcc()
    exe = str(tmp_path / "c_abi_roundtrip")
    libdir = os.path.dirname(lib)
    subprocess.run([nvcc, "-O2", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_roundtrip.c"),
                    "-o", exe, "-cudart", "shared", "-L", libdir, "-lcsf", "-Xlinker", f"-rpath={libdir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")

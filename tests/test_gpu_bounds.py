"""The bounds-check build (libvq3_bc.so, compiled with -DVQ3_BOUNDS_CHECK) on one call of every
kernel path, the 5120 / 17408 SwiGLU block included: no instrumented global access is out of
range, and the outputs are bit-identical to the normal build's."""

import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ("decode", "lowrank", "delta", "rotate", "prefill", "prefill_wide")


def _run(path, lib=None):
    env = dict(os.environ)
    env.pop("VQ3_LIB", None)
    if lib:
        env["VQ3_LIB"] = lib
    r = subprocess.run([sys.executable, "-m", "tests.bounds_workloads", str(path)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return np.load(path)


def test_bounds_check_build_clean_and_bit_identical(tmp_path):
    from bit_vector_lut_gb300 import build as B
    bc_lib = B.build(bounds_check=True)
    bc = _run(tmp_path / "bc.npz", bc_lib)
    assert "bounds-check build" in str(bc["version"])
    for f in FILES:
        count, site = bc[f"bounds_{f}"]
        assert count == 0, f"{f}: {count} accesses out of range, first at site {site}"
    ref = _run(tmp_path / "normal.npz")
    assert "bounds-check" not in str(ref["version"])
    names = [n for n in ref.files if n != "version"]
    assert len(names) >= 20
    for n in names:
        a, b = bc[n], ref[n]
        assert a.shape == b.shape and a.dtype == b.dtype, n
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{n}: the two builds differ"

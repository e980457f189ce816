"""The range-checked debug library (libttt_debug.so, built with
TTT_DEBUG_BOUNDS) against libttt.so.

Each library runs in a child process (the binding loads one library per
process, chosen by TTT_LIBRARY).  The self-test kernel evaluates one check
and touches no memory, so an out-of-range index is only recorded.  The
workload (tests/bounds_workload.py) must give the same results under both
libraries, and no check of the debug library may fail on it.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRIPT = os.path.join(ROOT, "tests", "bounds_workload.py")


def _run(library, *args):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if library == "debug" and not os.path.exists(os.path.join(ROOT, "long_context_lm_ttt_b300", "libttt_debug.so")):
        from long_context_lm_ttt_b300 import build
        build.build(debug_bounds=True)
    env = dict(os.environ, TTT_LIBRARY=library)
    r = subprocess.run([sys.executable, SCRIPT, *args], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return r.stdout


def test_bounds_selftest():
    """With the checks an index outside [0, limit) is recorded as the
    self-test kernel's (id 7) and reading clears the record; an index inside
    is not.  libttt.so records nothing."""
    dbg = json.loads(_run("debug", "--selftest").strip().splitlines()[-1])
    assert dbg["checked"] is True
    assert dbg["inside"] == [0, 0, 0, 0]
    assert dbg["outside"] == [2, 7, 5, 3]  # two failed checks, the first one described
    assert dbg["after"] == [0, 0, 0, 0]
    plain = json.loads(_run("normal", "--selftest").strip().splitlines()[-1])
    assert plain["checked"] is False
    assert plain["outside"] == [0, 0, 0, 0]


def test_debug_library_matches_and_passes_its_checks(tmp_path):
    """The workload's outputs agree between the two libraries (the checks
    guard accesses and change no arithmetic), and every check of the debug
    library passes on it."""
    a_path, b_path = str(tmp_path / "plain.npz"), str(tmp_path / "debug.npz")
    _run("normal", a_path)
    _run("debug", b_path)
    a, b = np.load(a_path), np.load(b_path)
    assert int(a["checked"][0]) == 0 and int(b["checked"][0]) == 1
    assert b["bounds"].tolist() == [0, 0, 0, 0], b["bounds"]
    keys = sorted(k for k in a.files if k not in ("bounds", "checked"))
    assert keys == sorted(k for k in b.files if k not in ("bounds", "checked"))
    assert any(k.startswith("attn3") for k in keys) and "ctx_decode_tokens" in keys
    for k in keys:
        x, y = a[k], b[k]
        assert x.shape == y.shape, k
        assert np.all(np.isfinite(x)), k
        if x.dtype.kind in "iu":
            assert np.array_equal(x, y), k
        else:
            scale = max(float(np.abs(x).max()), 1e-30)
            assert float(np.abs(x.astype(np.float64) - y).max()) <= 1e-6 * scale, k

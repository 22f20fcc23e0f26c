"""The debug build (libdg_debug.so, -DDG_DEBUG=1): its index checks raise no bit on in-bounds
calls of every kernel family and leave every result bit-identical to the release build; a
planted narrowing of the output rows (a test hook, no out-of-bounds access) raises DG_DEBUG_OUT
and skips exactly the stores past it; an injected producer stall (a load that is never issued, so
a bounded wait runs out) returns DG_STATUS_TIMEOUT and leaves the next call clean."""
import os
import subprocess
import sys

import numpy as np
import pytest

from moe_grouped_fp8_gb300 import DG_DEBUG_OUT, DG_STATUS_TIMEOUT, build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def run_cases(tmp_path, debug: bool) -> dict:
    path = tmp_path / ("debug.npz" if debug else "release.npz")
    env = {**os.environ, "DG_DEBUG": "1" if debug else "0",
           "PYTHONPATH": os.pathsep.join([ROOT, os.environ.get("PYTHONPATH", "")])}
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py"), str(path)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    with np.load(path) as z:
        return {k: z[k] for k in z.files}


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    build.build()
    build.build(debug=True)
    tmp = tmp_path_factory.mktemp("debug_build")
    return run_cases(tmp, False), run_cases(tmp, True)


def test_builds_identify_themselves(results):
    rel, dbg = results
    assert int(rel["debug_build"][0]) == 0 and int(dbg["debug_build"][0]) == 1


def test_in_bounds_calls_raise_no_bit_and_match_release_bitwise(results):
    rel, dbg = results
    assert int(rel["word"][0]) == 0
    assert int(dbg["word"][0]) == 0, f"debug word {int(dbg['word'][0]):#x} on in-bounds calls"
    cases = sorted(k for k in rel if "." in k)
    assert len(cases) >= 25 and cases == sorted(k for k in dbg if "." in k)
    for k in cases:
        assert np.array_equal(rel[k], dbg[k]), f"{k}: debug build differs from release"


def test_planted_row_limit_is_flagged_and_skipped(results):
    rel, dbg = results
    G, cap, N = 4, 200, 512
    # release: the hook has no effect
    assert int(rel["planted_word"][0]) == 0
    assert np.array_equal(rel["planted_out"], rel["masked_short.0"])
    # debug: the first group's rows are stored, every later row keeps the sentinel, one bit
    assert int(dbg["planted_word"][0]) == DG_DEBUG_OUT
    d = dbg["planted_out"].reshape(G, cap, N * 2)
    full = rel["masked_short.0"].reshape(G, cap, N * 2)
    assert np.array_equal(d[0], full[0])
    assert np.all(d[1:] == 0xFF)


def test_injected_producer_stall_times_out_cleanly(results):
    rel, dbg = results
    # release: the hook has no effect
    assert int(rel["stall_status"][0]) == 0
    # debug: the stalled CTA's waits ran out; the call returned and the next one is bit-identical
    assert int(dbg["stall_status"][0]) & DG_STATUS_TIMEOUT
    assert np.array_equal(dbg["after_stall.0"], rel["masked_long.0"])
    assert np.array_equal(rel["after_stall.0"], rel["masked_long.0"])

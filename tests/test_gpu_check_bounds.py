"""The W4_CHECK_BOUNDS build of the library (every data-dependent global
store of the alignment, the GEMM epilogues and the folded combine checked
against its array's extent; a failed check sets W4_DEV_OUT_OF_BOUNDS and
skips the store) on the test workloads: no check fails, and the outputs are
the normal build's bit for bit.  compute-sanitizer is not available here;
this is the range check that stands in for it."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

NAMES = ["tiny", "ragged", "layer256"]


@pytest.fixture(scope="module")
def checked_lib(tmp_path_factory):
    from w4a16_moe_expert_sync_gb300 import build
    return build.build_checked(str(tmp_path_factory.mktemp("w4chk")))


def test_checked_build_matches_and_finds_nothing(lib, checked_lib, tmp_path):
    here = os.path.dirname(os.path.abspath(__file__))
    out = str(tmp_path / "checked.npz")
    r = subprocess.run([sys.executable, os.path.join(here, "checked_build_run.py"), checked_lib,
                        out, *NAMES], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ref = str(tmp_path / "normal.npz")
    import checked_build_run
    from w4a16_moe_expert_sync_gb300 import build
    checked_build_run.run(build.LIB, NAMES, ref)
    got, want = np.load(out), np.load(ref)
    for name in NAMES:
        st = got[f"{name}_status"]
        assert not np.any(st & lib.W4_DEV_OUT_OF_BOUNDS), (name, st)
        assert np.array_equal(st, want[f"{name}_status"]), (name, st)
        assert np.array_equal(got[f"{name}_out"], want[f"{name}_out"]), name
        assert np.array_equal(got[f"{name}_out2"], want[f"{name}_out2"]), name

"""The checked library (built with MOE_CHECK: index checks in the kernels that
index with rows, slots or tokens another kernel wrote) computes exactly what
the normal one does, reports a clean status on valid calls, and reports
MOE_ERR_DEVICE_CHECK, skipping the access, when a slot is out of bounds."""
import json
import os
import subprocess
import sys

import pytest

from mixture_experts_layer_99_b300 import build as B

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def _child(*args):
    if B.stale(B.LIB_CHECK):   # missing, or built before the current sources
        B.build(check=True)
    env = dict(os.environ, MOE_B300_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py"), *args],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_matches_normal_build():
    import checked_cases
    checked = _child()
    normal = checked_cases.run_cases()
    for name, d in normal.items():
        assert d["status"] == [0, 0] and d["stage_status"] == [0, 0], name
        assert checked[name] == d, name


def test_checked_build_reports_a_slot_out_of_bounds():
    r = _child("corrupt")
    assert r["backward_status"] == [6, 55]   # MOE_ERR_DEVICE_CHECK, the backward's combine

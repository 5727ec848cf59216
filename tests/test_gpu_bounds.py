"""The bounds-checked debug build (-DLMOE_BOUNDS), the stand-in for a memory
checker: every epilogue store, scatter write and combine read checks its row
against its buffer and reports through LATENTMOE_STATUS_BOUNDS instead of
touching memory outside it. The build is made here, and the forward paths
(tiny, ragged token counts, the shared expert, the skewed workload, the
multi-round schedule, router replay with out-of-range ids, E4M3 experts) run
in a child process that loads it; each must finish with no bounds bit set
and match the oracle."""
import os
import subprocess
import sys

import pytest

from mixture_experts_layer_router_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build_runs_clean():
    lib = build.build(variant="bounds")
    env = dict(os.environ, LATENTMOE_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_child.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "bounds build: all cases clean" in r.stdout


def test_bounds_status_bit_is_declared():
    from mixture_experts_layer_router_gb300 import capi
    header = open(os.path.join(os.path.dirname(HERE), "include", "latentmoe.h")).read()
    assert "LATENTMOE_STATUS_BOUNDS = 8u" in header and capi.STATUS_BOUNDS == 8

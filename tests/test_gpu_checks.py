"""The checks build (DUALKV_CHECKS): device-side index checks before every
global access and tile-copy coordinate, and per-CTA agreement of the pipeline
roles' step counts.  A failed check records its site in the device error
word instead of trapping, so this build can run where no memory sanitizer
is available.  The test builds libdualkv_checks.so, runs the small parity
cases and the layer's GEMM through it in a child process
(tests/checks_cases.py) and requires a clean error word after every case and
the usual parity with the oracle (the GEMM: with fp64 products)."""
import json
import os
import subprocess
import sys

import pytest

from tests.parity_util import GRAD_REL_L2, LSE_MAX_ABS, OUT_REL_L2

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checks_build_runs_the_parity_cases_clean():
    from shared_prompt_exact_dualkv_gb300 import build
    build.build(checks=True)
    env = dict(os.environ, DUALKV_LIBRARY="checks")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checks_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 9, r.stdout
    for res in lines:
        assert res["status"] == 0 and res["site"] == 0, res
        for key, val in res.items():
            if key in ("case", "status", "site"):
                continue
            bound = {"out": OUT_REL_L2, "lse": LSE_MAX_ABS, "gemm": 4e-3}.get(key, GRAD_REL_L2)
            assert val <= bound, (res["case"], key, val)

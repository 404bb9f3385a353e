"""The debug build (libttemb_debug.so: every data-derived index in the kernels
checked against its bound, a violation reported as TT_ERR_BOUNDS and the access
kept in range) on small workloads and the edge cases: no check fires and the
results match the oracle.  Runs in a fresh process, which loads the debug
library (TTEMB_DEBUG=1)."""
import os
import subprocess
import sys

import pytest

import tensor_train_compressed_embeddingbag_gb300 as tt

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_small_cases_check_clean():
    tt.build(debug=True)
    env = {**os.environ, "TTEMB_DEBUG": "1"}
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_cases.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok ") == 8, r.stdout

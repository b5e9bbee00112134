"""The bounds-checked build on the GPU: tests/checked_build_run.py runs every kernel family on small,
odd shapes (ragged tiles and tails, rows cut into segments, several tiles of the prefill) with the
library compiled with -DQMM_CHECK_BOUNDS, in a process of its own, and checks each result against
the CPU oracle and that no index check fired (the device status stays QMM_OK)."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")
from block_quantized_weight_q8_gb300 import buildlib  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bounds_checked_build_runs_clean():
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    lib = buildlib.build(checked=True)
    env = dict(os.environ, QMM_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_build_run.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "checked build ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]

"""The bounds-checked variant of the library (compiled with -DQMM_CHECK_BOUNDS, where every kernel
checks the index ranges of its computed accesses and records QMM_E_BOUNDS in a device error word
instead of faulting) builds for sm_103a on the CPU and exports the same entry points as the normal
build.  Its GPU run on small, odd shapes is tests/test_gpu_checked_build.py."""
import re
import subprocess

from test_abi import declared_functions

from block_quantized_weight_q8_gb300 import buildlib


def test_checked_variant_builds_and_exports_the_boundary():
    path = buildlib.build(checked=True)
    assert path == buildlib.CHECKED_LIB
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(qmm_\w+)", out))
    assert exported == set(declared_functions()), exported ^ set(declared_functions())


def test_checks_compile_away_in_the_normal_build():
    """QMM_IN_BOUNDS is the constant true unless QMM_CHECK_BOUNDS is defined."""
    src = open(buildlib.os.path.join(buildlib.CSRC, "qmm_device.cuh")).read()
    normal = src.split("#ifdef QMM_CHECK_BOUNDS", 1)[1].split("#else", 1)[1].split("#endif", 1)[0]
    assert "#define QMM_IN_BOUNDS(err, i, n) true" in normal

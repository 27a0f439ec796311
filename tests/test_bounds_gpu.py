"""The bounds-checked build (QL_BOUNDS_CHECK): every plain global load and
store of the kernels is range-checked against its buffer's bytes, and a
violation is recorded, not trapped. Small cases over every kernel and path
run through that build in a child process: the device status must stay
clean after each, and every output must equal the product build's, bit for
bit (the checks change nothing for in-range accesses)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_clean_and_identical(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from quantised_linear_layers_gb300 import build, ops
    checked = build.build_bounds_checked()
    build.build()
    ops.load_library()
    assert ops.load_library().ql_bounds_checked() == 0
    env = dict(os.environ, QL_LIBRARY=checked, PYTHONPATH=ROOT + os.pathsep + os.path.join(ROOT, "tests"))
    npz = str(tmp_path / "checked.npz")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_cases.py"), npz], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "flag 1" in r.stdout, "the child did not load the bounds-checked build"
    got = np.load(npz)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bounds_cases
    ref = bounds_cases.run(ops)
    assert len(ref) > 60
    for name, (arrs, st) in ref.items():
        assert st == 0, f"{name}: product build status {st}"
        assert int(got[f"{name}__status"][0]) == 0, f"{name}: bounds-checked build reported {got[f'{name}__status'][0]}"
        for i, arr in enumerate(arrs):
            assert np.array_equal(got[f"{name}__{i}"], arr), f"{name}[{i}] differs in the bounds-checked build"

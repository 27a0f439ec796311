"""The package's smoke entry point (one small cast + block cast + GEMM on
cuda:0 checked against the CPU oracle) passes, so the round-end smoke run and
the test suite exercise the same path."""
import os
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_smoke_entry_point(capsys):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.smoke()
    assert "smoke ok" in capsys.readouterr().out

"""The package entry point's smoke run (forward, backward and the balanced
layer of one small shape against the oracle) as a GPU test."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_smoke_entry_point():
    sys.path.insert(0, ROOT)
    try:
        import __graft_entry__ as entry
    finally:
        sys.path.remove(ROOT)
    entry.smoke()

"""Shared helpers for the tests: build the library on demand."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def ensure_built():
    from sliding_window_gqa_swa_gb300 import build
    return build.build()

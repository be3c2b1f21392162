"""Shared pytest setup: the ``gpu`` marker and session-wide workload caches."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


_CACHE: dict = {}


def cached_inputs(name: str):
    """(weights, x, ids) of a named workload, generated once per session."""
    import workload

    if name not in _CACHE:
        _CACHE[name] = workload.make_inputs(workload.CONFIGS[name])
    return _CACHE[name]

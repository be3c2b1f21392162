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
    """(weights, x, ids) of a named workload, generated once per session;
    workloads of the same layer shape share one weight set (same seeds)."""
    import workload

    if name not in _CACHE:
        cfg = workload.CONFIGS[name]
        shape = (cfg.experts, cfg.hidden, cfg.inter)
        if shape not in _CACHE:
            _CACHE[shape] = workload.make_weights(*shape)
        x = workload.make_x(cfg.batch, cfg.hidden, outlier_fraction=cfg.outlier_fraction)
        ids = workload.make_ids(cfg.batch, cfg.experts, dist=cfg.ids, s=cfg.zipf_s)
        _CACHE[name] = (_CACHE[shape], x, ids)
    return _CACHE[name]

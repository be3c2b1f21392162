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


def floor_rule_pair_case(experts: int = 16):
    """The hand-worked pair of tests/golden/floor_rule_pair.json as inputs:
    (weights, x bits [1, H], ids [1, 16], spec). Expert 0 carries the listed
    weights; experts 1..experts-1 are all-zero codes with scale byte 127; the
    token routes to experts 0..15, so pair 0 is the worked one."""
    import json

    import numpy as np

    spec = json.load(open(os.path.join(ROOT, "tests", "golden", "floor_rule_pair.json")))
    H, I = spec["hidden"], spec["inter"]
    w13 = np.zeros((experts, 2 * I, H // 2), np.uint8)
    s13 = np.full((experts, 2 * I, H // 32), 127, np.uint8)
    w2 = np.zeros((experts, H, I // 2), np.uint8)
    s2 = np.full((experts, H, I // 32), 127, np.uint8)
    for w, s, entries, kk in ((w13, s13, spec["w13"], "k"), (w2, s2, spec["w2"], "j")):
        for ent in entries:
            r, k = ent["row"], ent[kk]
            w[0, r, k // 2] |= ent["code"] << (4 * (k % 2))  # element 2i in the low nibble
            s[0, r, k // 32] = ent["scale_byte"]
    one = 0x3F80  # BF16 1.0
    x = np.full((1, H), one, np.uint16)
    ids = np.arange(16, dtype=np.int32).reshape(1, 16)
    return (w13, s13, w2, s2), x, ids, spec

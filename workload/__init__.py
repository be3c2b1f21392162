"""Seeded synthetic workloads for the MXFP8 x MXFP4 top-16 MoE decode layer.

Shared by the tests, the oracle's callers and ``bench.py``; it imports neither
the CUDA library nor the oracle and holds none of the layer's arithmetic. It
only draws inputs:

* weights: BF16 samples of N(0, 0.02), quantized to MXFP4 (e2m1 codes, one
  E8M0 scale per 32 along K) by the OCP MX v1.0 conversion (shared exponent
  floor(log2 amax) - 2, round to nearest even on the e2m1 grid, saturate at
  6). This is data synthesis: the layer itself never quantizes weights.
  w13 [E, 2I, H/2] (rows 0..I-1 gate, I..2I-1 up), s13 [E, 2I, H/32],
  w2 [E, H, I/2], s2 [E, H, I/32]; element 2i sits in the low nibble of byte i.
* x: BF16 samples of N(0, 1), [B, H], as raw uint16 bits; optionally a
  fraction of rows (chosen by the same generator) multiplied by 50.
* ids: int32 [B, 16], 16 distinct experts per token, uniform
  (a random permutation's first 16) or Zipf(s) (p_e ~ (e + 1)^-s, drawn
  without replacement).

Every tensor has its own numpy PCG64 stream: weights per expert from
SeedSequence([seed, expert]) (w13 seed 0, w2 seed 1), x seed 2, ids seed 3,
so generation is parallel over experts and reproducible.
"""
from __future__ import annotations

import concurrent.futures as _futures
import os
from dataclasses import dataclass

import numpy as np

SLOTS = 16


@dataclass(frozen=True)
class Config:
    name: str
    experts: int
    hidden: int
    inter: int
    batch: int
    ids: str  # "uniform" or "zipf"
    outlier_fraction: float = 0.0
    zipf_s: float = 1.1

    def describe(self) -> str:
        return (f"{self.name}: E={self.experts} H={self.hidden} I={self.inter} "
                f"B={self.batch} top-16 ids={self.ids}")


#: The five workloads: a tiny correctness case, then the TP8 / TP16 shard
#: shapes of a 384-expert top-16 layer with hidden 3584.
CONFIGS = {
    "tiny": Config("tiny", 32, 256, 64, 2, "uniform"),
    "tp8_b1": Config("tp8_b1", 384, 3584, 384, 1, "uniform"),
    "tp16_b8": Config("tp16_b8", 384, 3584, 256, 8, "uniform"),
    "tp8_b64": Config("tp8_b64", 384, 3584, 384, 64, "zipf"),
    "tp8_b256": Config("tp8_b256", 384, 3584, 384, 256, "zipf", outlier_fraction=0.01),
}


# --- BF16 and MXFP4 data synthesis ----------------------------------------

def float_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    one, half = np.uint32(1), np.uint32(0x7FFF)
    rounded = (u + half + ((u >> np.uint32(16)) & one)) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_tables():
    """Code of the nearest e2m1 magnitude for a in (i/4, (i+1)/4) and for a == i/4.

    Every tie point between two grid values is a multiple of 1/4, so the
    rounding is constant inside each open quarter interval; a tie takes the
    even code.
    """
    def nearest(a):
        d = np.abs(_E2M1_GRID - a)
        best = np.flatnonzero(d == d.min())
        return int(best[0] if len(best) == 1 else best[best % 2 == 0][0])

    open_ = np.array([nearest(i / 4 + 1 / 16) for i in range(33)], np.uint8)
    exact = np.array([nearest(i / 4) for i in range(33)], np.uint8)
    open_[32] = exact[32] = 7  # a >= 8 cannot occur; saturate anyway
    return open_, exact


_E2M1_OPEN, _E2M1_EXACT = _e2m1_tables()


def mxfp4_encode(values: np.ndarray):
    """OCP MX v1.0 MXFP4 of the last axis (a multiple of 32).

    Returns (packed uint8 [..., K/2], scales uint8 [..., K/32]).
    """
    v = np.asarray(values, dtype=np.float32)
    *lead, K = v.shape
    blocks = v.reshape(*lead, K // 32, 32)
    mag = np.abs(blocks)
    amax = mag.max(axis=-1)
    _, e = np.frexp(amax)  # amax in [2^(e-1), 2^e)
    shared = np.where(amax > 0, e - 1 - 2, -127).clip(-127, 127).astype(np.int32)
    a = mag * np.ldexp(np.float32(1.0), -shared)[..., None].astype(np.float32)
    quarter = np.minimum(np.floor(a * np.float32(4.0)), np.float32(32.0)).astype(np.int32)
    code = np.where(a == quarter.astype(np.float32) * np.float32(0.25),
                    _E2M1_EXACT[quarter], _E2M1_OPEN[quarter])
    code = (code | (np.signbit(blocks).astype(np.uint8) << 3)).reshape(*lead, K)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, (shared + 127).astype(np.uint8)


def _expert_rows(seed: int, expert: int, rows: int, cols: int):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, expert])))
    w = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02)
    return mxfp4_encode(bf16_bits_to_float(float_to_bf16_bits(w)))


def make_weights(experts: int, hidden: int, inter: int, seed13: int = 0, seed2: int = 1,
                 threads: int | None = None):
    """MXFP4 expert weights (w13, s13, w2, s2) in the library's input layout."""
    w13 = np.empty((experts, 2 * inter, hidden // 2), np.uint8)
    s13 = np.empty((experts, 2 * inter, hidden // 32), np.uint8)
    w2 = np.empty((experts, hidden, inter // 2), np.uint8)
    s2 = np.empty((experts, hidden, inter // 32), np.uint8)

    def one(e):
        w13[e], s13[e] = _expert_rows(seed13, e, 2 * inter, hidden)
        w2[e], s2[e] = _expert_rows(seed2, e, hidden, inter)

    workers = threads or min(32, len(os.sched_getaffinity(0)))
    with _futures.ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(one, range(experts)))
    return w13, s13, w2, s2


def make_x(batch: int, hidden: int, seed: int = 2, outlier_fraction: float = 0.0):
    """BF16 bits [B, H] of N(0, 1); round(fraction * B) rows scaled by 50."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((batch, hidden), dtype=np.float32)
    outliers = int(round(outlier_fraction * batch))
    if outliers:
        rows = rng.choice(batch, size=outliers, replace=False)
        x[rows] *= np.float32(50.0)
    return float_to_bf16_bits(x)


def make_ids(batch: int, experts: int, seed: int = 3, dist: str = "uniform", s: float = 1.1):
    """int32 [B, 16]: 16 distinct experts per token, uniform or Zipf(s)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = np.empty((batch, SLOTS), np.int32)
    if dist == "uniform":
        for t in range(batch):
            ids[t] = rng.permutation(experts)[:SLOTS]
    elif dist == "zipf":
        p = (np.arange(experts, dtype=np.float64) + 1.0) ** (-s)
        p /= p.sum()
        for t in range(batch):
            ids[t] = rng.choice(experts, size=SLOTS, replace=False, p=p)
    else:
        raise ValueError(dist)
    return ids


def make_inputs(cfg: Config, threads: int | None = None):
    """(weights tuple, x bits, ids) for a config, from the fixed seeds."""
    weights = make_weights(cfg.experts, cfg.hidden, cfg.inter, threads=threads)
    x = make_x(cfg.batch, cfg.hidden, outlier_fraction=cfg.outlier_fraction)
    ids = make_ids(cfg.batch, cfg.experts, dist=cfg.ids, s=cfg.zipf_s)
    return weights, x, ids


def touched_experts(ids: np.ndarray) -> np.ndarray:
    return np.unique(np.asarray(ids).reshape(-1))


def expert_bytes(hidden: int, inter: int) -> int:
    """Bytes of one expert's w13 + s13 + w2 + s2 (FP4 packed, E8M0 scales)."""
    return 2 * inter * hidden // 2 + 2 * inter * hidden // 32 + hidden * inter // 2 + hidden * inter // 32

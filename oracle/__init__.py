"""CPU oracle for the MXFP8 x MXFP4 top-16 MoE decode layer (float64).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. It never imports the CUDA library and the CUDA library never imports
it; the two share no code. The arithmetic lives in ``moe_oracle.c``; this file
only marshals numpy arrays through ctypes.

What it computes (pages: ``...cutedsl.moe.experts`` and
``...cutedsl.moe.experts_runtime``): per token, MXFP8 of the BF16 row (ceil
rule); per (token, slot) pair with expert e = ids[t, s]: FC1 against e's
MXFP4 gate+up rows, SiLU(gate) * up, MXFP8 requant of the hidden row (floor
rule iff 2I == 768), FC2 against e's MXFP4 down rows, BF16 (RNE) output row
``t * 16 + s``; and the routing-weighted combine of a token's 16 rows
(ExpertsKernel.finalize). Sums are exact-order float64 loops.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

SLOTS = 16
UNIT_ROWS = 8

_lib = None


def _library():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        i16p = np.ctypeslib.ndpointer(np.int16, flags="C_CONTIGUOUS")
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        c_int, c_uint, c_double = ctypes.c_int, ctypes.c_uint, ctypes.c_double
        lib.orc_e2m1_value.argtypes, lib.orc_e2m1_value.restype = [c_uint], c_double
        lib.orc_e4m3_value.argtypes, lib.orc_e4m3_value.restype = [c_uint], c_double
        lib.orc_e8m0_value.argtypes, lib.orc_e8m0_value.restype = [c_uint], c_double
        lib.orc_bf16_value.argtypes, lib.orc_bf16_value.restype = [ctypes.c_uint16], c_double
        lib.orc_e4m3_encode.argtypes, lib.orc_e4m3_encode.restype = [c_double], ctypes.c_uint8
        lib.orc_bf16_encode.argtypes, lib.orc_bf16_encode.restype = [c_double], ctypes.c_uint16
        lib.orc_mx_exponent.argtypes, lib.orc_mx_exponent.restype = [c_double, c_int], c_int
        lib.orc_hidden_floor_rule.argtypes, lib.orc_hidden_floor_rule.restype = [c_int], c_int
        lib.orc_gated.argtypes, lib.orc_gated.restype = [c_double, c_double], c_double
        lib.orc_mxfp8_block.argtypes = [f64p, c_int, u8p, u8p]
        lib.orc_mxfp8_block.restype = None
        lib.orc_quantize_x.argtypes = [u16p, c_int, c_int, u8p, u8p]
        lib.orc_quantize_x.restype = None
        lib.orc_group.argtypes = [i32p, c_int, c_int, i32p, i16p, c_int]
        lib.orc_group.restype = c_int
        vp = ctypes.c_void_p
        lib.orc_pairs.argtypes = [u8p, u8p, u8p, u8p, c_int, c_int, c_int, u8p, u8p, i32p, i32p,
                                  c_int, u16p, vp, vp, vp, c_int]
        lib.orc_pairs.restype = None
        lib.orc_fc2_rows.argtypes = [u8p, u8p, c_int, c_int, c_int, i32p, u8p, u8p, c_int, u16p,
                                     c_int]
        lib.orc_fc2_rows.restype = None
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        lib.orc_combine.argtypes = [u16p, f32p, u8p, c_int, c_int, u16p]
        lib.orc_combine.restype = None
        _lib = lib
    return _lib


def default_threads() -> int:
    """Host threads the oracle may use: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --- element formats ------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _library().orc_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return _library().orc_e4m3_value(code)


def e8m0_value(b: int) -> float:
    return _library().orc_e8m0_value(b)


def bf16_value(bits: int) -> float:
    return _library().orc_bf16_value(bits)


def e4m3_encode(v: float) -> int:
    return int(_library().orc_e4m3_encode(float(v)))


def bf16_encode(v: float) -> int:
    return int(_library().orc_bf16_encode(float(v)))


def mx_exponent(amax: float, floor_rule: bool) -> int:
    return int(_library().orc_mx_exponent(float(amax), int(bool(floor_rule))))


def gated(gate: float, up: float) -> float:
    """SiLU(gate) * up in float64."""
    return float(_library().orc_gated(float(gate), float(up)))


def hidden_floor_rule(inter: int) -> bool:
    return bool(_library().orc_hidden_floor_rule(int(inter)))


def mxfp8_block(values, floor_rule: bool):
    """One block of 32 float64 values -> (codes uint8[32], scale byte)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    assert v.shape == (32,)
    codes = np.zeros(32, np.uint8)
    scale = np.zeros(1, np.uint8)
    _library().orc_mxfp8_block(v, int(bool(floor_rule)), codes, scale)
    return codes, int(scale[0])


# --- path steps -----------------------------------------------------------

def quantize_x(x_bf16_bits: np.ndarray):
    """x: uint16 BF16 bits [B, H] -> (codes uint8 [B, H], scales uint8 [B, H/32])."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    B, H = x.shape
    codes = np.zeros((B, H), np.uint8)
    scales = np.zeros((B, H // 32), np.uint8)
    _library().orc_quantize_x(x, B, H, codes, scales)
    return codes, scales


def group(ids: np.ndarray, experts: int):
    """ids int32 [B, 16] -> (unit_expert int32 [U], unit_rows int16 [U, 8])."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    B = ids.shape[0]
    cap = B * SLOTS
    ue = np.zeros(cap, np.int32)
    ur = np.zeros(cap * UNIT_ROWS, np.int16)
    units = _library().orc_group(ids, B, experts, ue, ur, cap)
    if units < 0:
        raise ValueError("unit table overflow")
    return ue[:units].copy(), ur[: units * UNIT_ROWS].reshape(units, UNIT_ROWS).copy()


def pairs_forward(weights, xq, xs, ids, pairs=None, want_hidden=False, want_fc1=False,
                  threads=None):
    """Run the listed pairs (t * 16 + s; default all) through their experts.

    weights = (w13, s13, w2, s2) in the user layout (uint8 arrays
    [E, 2I, H/2], [E, 2I, H/32], [E, H, I/2], [E, H, I/32]).
    Returns dict(out=uint16 [n, H], hq=[n, I], hs=[n, I/32], y=float64 [n, 2I]).
    """
    w13, s13, w2, s2 = (np.ascontiguousarray(a, dtype=np.uint8) for a in weights)
    E, rows, half_h = w13.shape
    H, inter = half_h * 2, rows // 2
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    B = ids.shape[0]
    if pairs is None:
        pairs = np.arange(B * SLOTS, dtype=np.int32)
    pairs = np.ascontiguousarray(pairs, dtype=np.int32)
    n = int(pairs.shape[0])
    out = np.zeros((n, H), np.uint16)
    hq = np.zeros((n, inter), np.uint8) if want_hidden else None
    hs = np.zeros((n, inter // 32), np.uint8) if want_hidden else None
    y = np.zeros((n, 2 * inter), np.float64) if want_fc1 else None
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    _library().orc_pairs(w13, s13, w2, s2, E, H, inter, np.ascontiguousarray(xq, np.uint8),
                         np.ascontiguousarray(xs, np.uint8), ids, pairs, n, out, ptr(hq),
                         ptr(hs), ptr(y), int(threads or default_threads()))
    return {"out": out, "hq": hq, "hs": hs, "y": y}


def fc2_rows(w2, s2, experts, hq, hs, threads=None):
    """FC2 alone: rows of given hidden codes/scales through the given experts."""
    w2 = np.ascontiguousarray(w2, np.uint8)
    s2 = np.ascontiguousarray(s2, np.uint8)
    E, H, half_i = w2.shape
    inter = half_i * 2
    experts = np.ascontiguousarray(experts, np.int32)
    n = int(experts.shape[0])
    out = np.zeros((n, H), np.uint16)
    _library().orc_fc2_rows(w2, s2, E, H, inter, experts, np.ascontiguousarray(hq, np.uint8),
                            np.ascontiguousarray(hs, np.uint8), n, out,
                            int(threads or default_threads()))
    return out


def combine(rows, weights, kept=None):
    """Routing-weighted combine: rows uint16 BF16 [B*16, H] (pair t*16+s),
    weights float32 [B, 16], kept uint8 [B*16] (default: all) -> uint16 BF16
    [B, H] = bf16(sum_s w[t, s] * row[t, s]) in float64, skipped pairs left out."""
    rows = np.ascontiguousarray(rows, np.uint16)
    weights = np.ascontiguousarray(weights, np.float32)
    B = weights.shape[0]
    H = rows.shape[1]
    assert rows.shape[0] == B * SLOTS
    kept = np.ones(B * SLOTS, np.uint8) if kept is None else np.ascontiguousarray(kept, np.uint8)
    out = np.zeros((B, H), np.uint16)
    _library().orc_combine(rows, weights.reshape(-1), kept.reshape(-1), B, H, out)
    return out

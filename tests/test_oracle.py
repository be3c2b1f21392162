"""Pins of the CPU oracle against values fixed by the number formats, the
pages' definitions and mathematics, each formulated independently of the
oracle's C code (textbook format values, hand-worked blocks, torch's BF16
rounding, numpy matmuls of decoded matrices, brute-force recounts).

Page cited throughout: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.experts
(``mx_block``, ``plan_chunk``, ``ExpertsKernel.group``, ``ExpertsKernel.store_hidden``,
``stage``) and ...moe.experts_runtime (``PersistentExperts.__init__``).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Textbook values (OCP MX v1.0), written out independently of the oracle.
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0,
                 -4.0, -6.0])


def e4m3_table():
    """All 256 e4m3 values by (sign, exponent field, mantissa), NaN at 0x7F/0xFF."""
    out = np.empty(256)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            out[code] = np.nan
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -mag if s else mag
    return out


E4M3 = e4m3_table()


# --- element formats -----------------------------------------------------

def test_e2m1_table_all_codes():
    for code in range(16):
        assert oracle.e2m1_value(code) == E2M1[code]
        assert math.copysign(1.0, oracle.e2m1_value(code)) == math.copysign(1.0, E2M1[code])


def test_e4m3_textbook_codes():
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for code, value in known.items():
        assert oracle.e4m3_value(code) == value
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    for code in range(256):
        v = oracle.e4m3_value(code)
        assert (math.isnan(v) and math.isnan(E4M3[code])) or v == E4M3[code]


def test_e8m0_textbook_values():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert oracle.e8m0_value(130) == 8.0
    assert math.isnan(oracle.e8m0_value(255))


def test_e4m3_encode_round_trips_every_finite_code():
    for code in range(256):
        if code in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(E4M3[code]) == code, hex(code)


def test_e4m3_encode_midpoints_go_to_even_and_neighbours_to_nearest():
    positive = [(E4M3[c], c) for c in range(0x7F)]  # increasing with the code
    for (a, ca), (b, cb) in zip(positive, positive[1:]):
        mid = (a + b) / 2
        even = ca if ca % 2 == 0 else cb
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(-mid) == even | 0x80
        step = (b - a) / 8
        assert oracle.e4m3_encode(mid - step) == ca
        assert oracle.e4m3_encode(mid + step) == cb


def test_e4m3_encode_saturates_and_keeps_sign():
    for v in (448.0, 448.5, 464.0, 480.0, 1e6):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00


def test_bf16_encode_matches_torch_on_float32_values():
    rng = np.random.default_rng(11)
    values = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-30).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -130], np.float32),
    ])
    expect = torch.from_numpy(values).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_encode(float(v)) for v in values], np.uint16)
    np.testing.assert_array_equal(got, expect)


def test_bf16_encode_rounds_float64_once():
    # Just above a tie: one rounding goes up; a detour through float32 would
    # first land on the tie and then round down to even.
    assert oracle.bf16_encode(1 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_encode(1 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_encode(-0.0) == 0x8000
    assert oracle.bf16_value(0x3F81) == 1 + 2.0 ** -7


# --- MXFP8 block quantization (mx_block, store_hidden) -----------------------

def test_mx_exponent_hand_worked():
    ceil = lambda a: oracle.mx_exponent(a, False)
    floor = lambda a: oracle.mx_exponent(a, True)
    assert ceil(0.0) == -127 and floor(0.0) == -127
    assert ceil(1.0) == -8  # 0.875 < 1 <= 1.75
    assert ceil(1.75) == -8
    assert ceil(1.765625) == -7
    assert ceil(448.0) == 0 and ceil(449.0) == 1
    assert ceil(1024.0) == 2
    for k in range(-100, 100, 7):
        assert ceil(2.0 ** k) == k - 8
        assert ceil(1.75 * 2.0 ** k) == k - 8
        assert ceil(1.875 * 2.0 ** k) == k - 7
    assert ceil(1e-45) == -127  # clamped at the E8M0 floor
    assert floor(1.9) == -8 and floor(1.0) == -8 and floor(0.99) == -9
    assert floor(448.0) == 0 and floor(512.0) == 1
    assert floor(1e-45) == -127


def test_mx_exponent_ceil_is_the_smallest_fitting_power():
    rng = np.random.default_rng(5)
    for a in np.exp(rng.uniform(-80, 80, 5000)):
        E = oracle.mx_exponent(a, False)
        assert a <= 448.0 * 2.0 ** E
        assert E == -127 or a > 448.0 * 2.0 ** (E - 1)


def test_golden_mx_blocks():
    blocks = json.load(open(os.path.join(GOLDEN, "mx_blocks.json")))["blocks"]
    for b in blocks:
        values = np.full(32, b["default"], np.float64)
        for i, v in b["set"].items():
            values[int(i)] = v
        codes, scale = oracle.mxfp8_block(values, b["rule"] == "floor")
        expect = np.full(32, b["default_code"], np.uint8)
        for i, c in b["codes"].items():
            expect[int(i)] = c
        assert scale == b["scale"], b["name"]
        np.testing.assert_array_equal(codes, expect, err_msg=b["name"])


def test_quantize_dequantize_identity_for_representable_blocks():
    rng = np.random.default_rng(7)
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    big = [c for c in finite if 224 < abs(E4M3[c]) <= 448]
    for _ in range(500):
        codes = rng.choice(finite, 32)
        codes[rng.integers(32)] = rng.choice(big)
        codes = np.where(codes == 0x80, 0, codes)  # -0 and +0 dequantize alike
        E = int(rng.integers(-100, 100))
        x = E4M3[codes] * 2.0 ** E
        got_codes, scale = oracle.mxfp8_block(x, False)
        assert scale == E + 127
        np.testing.assert_array_equal(got_codes, codes)
        np.testing.assert_array_equal(E4M3[got_codes] * 2.0 ** (scale - 127), x)


def test_quantize_x_rows_of_representable_values():
    rng = np.random.default_rng(9)
    B, H = 3, 256
    codes = rng.choice([c for c in range(0x7F)] + [c | 0x80 for c in range(1, 0x7F)], (B, H))
    codes[:, ::32] = 0x7E  # each block reaches 448: the ceil rule keeps the chosen exponent
    exps = rng.integers(-20, 20, (B, H // 32))
    x = E4M3[codes] * np.repeat(2.0 ** exps, 32, axis=1)
    bits = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(torch.from_numpy(bits).view(torch.bfloat16).double().numpy(), x)
    q, s = oracle.quantize_x(bits.view(np.uint16))
    np.testing.assert_array_equal(q, codes)
    np.testing.assert_array_equal(s, exps + 127)


def test_hidden_rule_follows_w13_rows():
    assert oracle.hidden_floor_rule(384)  # 2I = 768 rows: the TP8 shard
    assert not oracle.hidden_floor_rule(256)
    assert not oracle.hidden_floor_rule(64)


def test_gated_activation_closed_forms():
    assert oracle.gated(0.0, 5.0) == 0.0
    assert oracle.gated(3.0, 0.0) == 0.0
    assert oracle.gated(1.0, 1.0) == pytest.approx(0.7310585786300049, rel=1e-15)  # sigmoid(1)
    assert oracle.gated(40.0, 2.0) == pytest.approx(80.0, rel=1e-15)
    assert abs(oracle.gated(-40.0, 1.0)) < 1e-15
    assert oracle.gated(-1.0, -2.0) == pytest.approx(2 * 0.2689414213699951, rel=1e-15)


# --- grouping (ExpertsKernel.group) ----------------------------------------------

def brute_force_units(ids, experts):
    units = []
    flat = np.asarray(ids).reshape(-1)
    for e in range(experts):
        pairs = [p for p in range(flat.size) if flat[p] == e]
        for i in range(0, len(pairs), 8):
            chunk = pairs[i:i + 8]
            units.append((e, chunk + [-1] * (8 - len(chunk))))
    return units


@pytest.mark.parametrize("batch,experts,seed", [(1, 384, 0), (2, 32, 1), (37, 20, 2),
                                                (64, 384, 3), (256, 384, 4)])
def test_group_matches_brute_force(batch, experts, seed):
    rng = np.random.default_rng(seed)
    p = (np.arange(experts) + 1.0) ** -1.1
    ids = np.stack([rng.choice(experts, 16, replace=False, p=p / p.sum()) for _ in range(batch)])
    ue, ur = oracle.group(ids.astype(np.int32), experts)
    expect = brute_force_units(ids, experts)
    assert len(ue) == len(expect)
    for u, (e, rows) in enumerate(expect):
        assert ue[u] == e
        assert list(ur[u]) == rows
    # every pair exactly once; units per expert = ceil(n_e / 8)
    rows = ur[ur >= 0]
    assert sorted(rows.tolist()) == list(range(batch * 16))
    counts = np.bincount(ids.reshape(-1), minlength=experts)
    assert len(ue) == int(np.sum((counts + 7) // 8))


# --- one pair through an expert (stage, store_hidden, fc2) ------------------------

def decode_fp4(packed):
    """[..., K/2] packed -> [..., K] codes, element 2i in the low nibble of byte i."""
    lo, hi = packed & 15, packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def dequant_weights(w, s):
    return E2M1[decode_fp4(w)] * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=-1)


def random_weights(rng, E, H, I, scale_spread=3):
    w13 = rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8)
    w2 = rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8)
    s13 = (127 + rng.integers(-scale_spread, scale_spread + 1, (E, 2 * I, H // 32))).astype(np.uint8)
    s2 = (127 + rng.integers(-scale_spread, scale_spread + 1, (E, H, I // 32))).astype(np.uint8)
    return w13, s13, w2, s2


def test_nibble_order_and_every_e2m1_code_in_a_row():
    E, H, I = 1, 64, 32
    k = np.arange(H)
    row = (k % 16).astype(np.uint8)
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    w13[0, 0] = row[0::2] | (row[1::2] << 4)
    s13 = np.full((E, 2 * I, H // 32), 127, np.uint8)
    w2 = np.zeros((E, H, I // 2), np.uint8)
    s2 = np.full((E, H, I // 32), 127, np.uint8)
    for k0 in range(H):
        x = np.zeros((1, H), np.float32)
        x[0, k0] = 1.0
        bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xq, xs = oracle.quantize_x(bits)
        ids = np.zeros((1, 16), np.int32)
        res = oracle.pairs_forward((w13, s13, w2, s2), xq, xs, ids, pairs=np.array([0]),
                                   want_fc1=True, threads=1)
        assert res["y"][0, 0] == E2M1[k0 % 16]
        assert np.all(res["y"][0, 1:] == 0)


def test_fc1_with_unit_scales_is_a_matmul_of_decoded_codes():
    rng = np.random.default_rng(3)
    E, H, I, B = 3, 256, 64, 2
    w13, s13, w2, s2 = random_weights(rng, E, H, I, scale_spread=0)
    codes = rng.integers(0, 0x7F, (B, H))
    codes[:, ::32] = 0x7E
    x = E4M3[codes] * 2.0 ** -4
    bits = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    xq, xs = oracle.quantize_x(bits.view(np.uint16))
    ids = np.stack([rng.permutation(E)[:1].repeat(16) for _ in range(B)]).astype(np.int32)
    res = oracle.pairs_forward((w13, s13, w2, s2), xq, xs, ids, want_fc1=True, threads=2)
    W = E2M1[decode_fp4(w13)]  # scales are all 2^0
    for i, pair in enumerate(range(B * 16)):
        t, e = pair // 16, ids.reshape(-1)[pair]
        np.testing.assert_array_equal(res["y"][i], W[e] @ x[t])


def naive_pair(w13, s13, w2, s2, xq, xs, e, t, floor_rule):
    """Triple-loop restatement of one pair, written apart from the oracle."""
    H, I = xq.shape[1], w2.shape[2] * 2
    xv = [E4M3[xq[t, k]] * 2.0 ** (int(xs[t, k // 32]) - 127) for k in range(H)]
    y = []
    for r in range(2 * I):
        acc = 0.0
        for k in range(H):
            byte = int(w13[e, r, k // 2])
            code = (byte >> 4) if k % 2 else (byte & 15)
            acc += E2M1[code] * 2.0 ** (int(s13[e, r, k // 32]) - 127) * xv[k]
        y.append(acc)
    h = [y[j] / (1 + math.exp(-y[j])) * y[I + j] for j in range(I)]
    hq, hs = [], []
    for b in range(I // 32):
        c, s = oracle.mxfp8_block(np.array(h[32 * b:32 * b + 32]), floor_rule)
        hq += list(c)
        hs.append(s)
    hv = [E4M3[hq[j]] * 2.0 ** (hs[j // 32] - 127) for j in range(I)]
    o = []
    for n in range(H):
        acc = 0.0
        for j in range(I):
            byte = int(w2[e, n, j // 2])
            code = (byte >> 4) if j % 2 else (byte & 15)
            acc += E2M1[code] * 2.0 ** (int(s2[e, n, j // 32]) - 127) * hv[j]
        o.append(acc)
    return np.array(y), np.array(hq, np.uint8), np.array(hs, np.uint8), np.array(o)


@pytest.mark.parametrize("inter", [32, 64, 256, 384])
def test_pairs_against_naive_triple_loop(inter):
    """inter = 256 > H: FC2 rows are longer than FC1 rows. inter = 384 is the
    TP8 shard's (2I = 768): the hidden requant takes the floor rule there
    (ExpertsKernel.store_hidden, floor = tp == 8; PersistentExperts.__init__,
    tp = 8 iff w13 has 768 rows), every other inter the ceil rule. The loop
    below is told the rule from the pages' definition, not from the oracle, and
    the test checks that the other rule would have given different codes, so
    an oracle that ignored or misrouted the rule fails here."""
    rng = np.random.default_rng(inter)
    E, H, B = 16, 64, 2  # 16 distinct experts per token: 32 distinct hidden rows
    floor_rule = 2 * inter == 768
    weights = random_weights(rng, E, H, inter)
    x = rng.standard_normal((B, H)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xq, xs = oracle.quantize_x(bits)
    ids = np.stack([rng.permutation(E) for _ in range(B)]).astype(np.int32)
    # Short hidden rows have few 32-blocks: take every pair there, so that some
    # block falls between the two rules.
    pairs = np.arange(B * 16, dtype=np.int32) if inter <= 64 else np.array([0, 5, 16, 31], np.int32)
    res = oracle.pairs_forward(weights, xq, xs, ids, pairs=pairs, want_hidden=True,
                               want_fc1=True, threads=2)
    other_rule_differs = False
    for i, p in enumerate(pairs):
        y, hq, hs, o = naive_pair(*weights, xq, xs, ids.reshape(-1)[p], p // 16, floor_rule)
        np.testing.assert_allclose(res["y"][i], y, rtol=1e-12, atol=1e-300)
        np.testing.assert_array_equal(res["hq"][i], hq)
        np.testing.assert_array_equal(res["hs"][i], hs)
        # Bit for bit: o is rounded once, from float64, exactly as the oracle does.
        expect = torch.from_numpy(o).to(torch.bfloat16)
        got = torch.from_numpy(res["out"][i].view(np.int16)).view(torch.bfloat16)
        assert torch.equal(got, expect)
        _, hq2, hs2, _ = naive_pair(*weights, xq, xs, ids.reshape(-1)[p], p // 16, not floor_rule)
        other_rule_differs |= not (np.array_equal(hq2, hq) and np.array_equal(hs2, hs))
    assert other_rule_differs, "the data does not tell the two scale rules apart"


def test_floor_rule_pair_golden():
    """The hand-worked pair of golden/floor_rule_pair.json (I = 384, floor rule)
    reproduces its codes, scales and output bits through the oracle."""
    from conftest import floor_rule_pair_case

    weights, x, ids, spec = floor_rule_pair_case()
    xq, xs = oracle.quantize_x(x)
    assert (xs == spec["x_scale"]).all() and (xq == spec["x_code"]).all()
    res = oracle.pairs_forward(weights, xq, xs, ids, pairs=np.array([0], np.int32),
                               want_hidden=True, threads=1)
    I, H = spec["inter"], spec["hidden"]
    hs = np.full(I // 32, spec["hidden_scale_default"], np.uint8)
    for b, v in spec["hidden_scales"].items():
        hs[int(b)] = v
    hq = np.full(I, spec["hidden_code_default"], np.uint8)
    for j, v in spec["hidden_codes"].items():
        hq[int(j)] = v
    out = np.full(H, spec["out_bits_default"], np.uint16)
    for n, v in spec["out_bits"].items():
        out[int(n)] = v
    np.testing.assert_array_equal(res["hs"][0], hs)
    np.testing.assert_array_equal(res["hq"][0], hq)
    np.testing.assert_array_equal(res["out"][0], out)
    # The hidden block alone, under each rule, as the golden's derivation states.
    h0 = 2.125 / (1.0 + math.exp(-2.125))
    block = np.zeros(32)
    block[0] = h0
    codes, scale = oracle.mxfp8_block(block, True)
    assert (int(scale), int(codes[0])) == (spec["hidden_scales"]["0"], spec["hidden_codes"]["0"])
    codes, scale = oracle.mxfp8_block(block, False)
    alt = spec["ceil_rule_would_give"]
    assert (int(scale), int(codes[0])) == (alt["hidden_scale_0"], alt["hidden_code_0"])


def test_fc2_only_entry_reproduces_pair_outputs():
    rng = np.random.default_rng(21)
    E, H, I, B = 5, 128, 64, 3
    weights = random_weights(rng, E, H, I)
    x = rng.standard_normal((B, H)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xq, xs = oracle.quantize_x(bits)
    ids = np.stack([np.resize(rng.permutation(E), 16) for _ in range(B)]).astype(np.int32)
    res = oracle.pairs_forward(weights, xq, xs, ids, want_hidden=True, threads=2)
    out = oracle.fc2_rows(weights[2], weights[3], ids.reshape(-1), res["hq"], res["hs"], threads=2)
    np.testing.assert_array_equal(out, res["out"])


def test_fc2_with_unit_scales_is_a_matmul_of_decoded_codes():
    rng = np.random.default_rng(4)
    E, H, I = 2, 128, 64
    _, _, w2, s2 = random_weights(rng, E, H, I, scale_spread=0)
    hq = rng.integers(0, 0x7F, (E, I)).astype(np.uint8)
    hs = np.full((E, I // 32), 120, np.uint8)
    out = oracle.fc2_rows(w2, s2, np.arange(E, dtype=np.int32), hq, hs, threads=1)
    W = E2M1[decode_fp4(w2)]
    for e in range(E):
        o = W[e] @ (E4M3[hq[e]] * 2.0 ** -7)
        expect = torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16)
        assert torch.equal(torch.from_numpy(out[e].view(np.int16)).view(torch.bfloat16), expect)


# --- routing-weighted combine (ExpertsKernel.finalize, single GPU) ----------

def bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_rows(rng, B, H):
    """BF16 bits of N(0, 1) rows, with negatives and a few subnormal and huge values."""
    x = rng.standard_normal((B * 16, H)).astype(np.float32)
    x[:, :2] = np.float32(1e-39), np.float32(-3e38)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_combine_one_hot_weights_select_each_slot():
    rng = np.random.default_rng(31)
    B, H = 3, 40
    rows = random_rows(rng, B, H)
    for t in range(B):
        for s in range(16):
            w = np.zeros((B, 16), np.float32)
            w[t, s] = 1.0
            out = oracle.combine(rows, w)
            np.testing.assert_array_equal(out[t], rows[t * 16 + s])
            assert not out[np.arange(B) != t].any()  # other tokens: +0.0


def test_combine_zero_weights_and_skipped_pairs_contribute_nothing():
    rng = np.random.default_rng(32)
    B, H = 2, 24
    rows = random_rows(rng, B, H)
    assert not oracle.combine(rows, np.zeros((B, 16), np.float32)).any()
    w = np.ones((B, 16), np.float32)
    assert not oracle.combine(rows, w, kept=np.zeros(B * 16, np.uint8)).any()
    # Skipping a pair gives the sum over the others: pair 5 of token 1 carries
    # a huge row that would dominate the sum.
    rows2 = rows.copy()
    rows2[16 + 5] = bf16_bits([1e30] * H)
    kept = np.ones(B * 16, np.uint8)
    kept[16 + 5] = 0
    w = np.zeros((B, 16), np.float32)
    w[1, 3] = 1.0
    w[1, 5] = 1.0
    np.testing.assert_array_equal(oracle.combine(rows2, w, kept)[1], rows2[16 + 3])


def test_combine_power_of_two_weights_scale_exactly():
    rng = np.random.default_rng(33)
    B, H = 1, 64
    x = (rng.standard_normal((16, H)) * 4).astype(np.float32)
    rows = torch.from_numpy(x).to(torch.bfloat16)
    w = np.zeros((B, 16), np.float32)
    w[0, 9] = 0.25
    got = torch.from_numpy(oracle.combine(rows.view(torch.int16).numpy().view(np.uint16), w).view(np.int16))
    expect = (rows[9].float() * 0.25).to(torch.bfloat16)  # exact: normal values times 2^-2
    assert torch.equal(got.view(torch.bfloat16)[0], expect)


def test_combine_cancellation_and_a_worked_sum():
    rng = np.random.default_rng(34)
    H = 16
    rows = random_rows(rng, 1, H)
    rows[4] = rows[2]
    w = np.zeros((1, 16), np.float32)
    w[0, 2], w[0, 4] = 1.0, -1.0
    assert not oracle.combine(rows, w).any()
    # 0.5 * 1 + 0.25 * 2 + 0.25 * 4 = 2 exactly, on every column.
    rows = np.zeros((16, H), np.uint16)
    rows[0], rows[7], rows[15] = bf16_bits([1.0] * H), bf16_bits([2.0] * H), bf16_bits([4.0] * H)
    w = np.zeros((1, 16), np.float32)
    w[0, 0], w[0, 7], w[0, 15] = 0.5, 0.25, 0.25
    np.testing.assert_array_equal(oracle.combine(rows, w)[0], bf16_bits([2.0] * H))

"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.

Bars (pages ...cutedsl.moe.experts / ...experts_runtime as read for this
build): the MXFP8 activation plan and the unit table match bit for bit; the
output matches within relative L2 <= 1e-2 over all rows and
|err| <= 3e-2 * rms(row) for every element; hidden requant flips (codes that
differ because the GPU sums FP32 in another order than the float64 oracle) are
counted and reported, and FC2 alone is re-checked on the GPU's own hidden
codes.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workload
from conftest import cached_inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
ROW_TOL = 3e-2


@pytest.fixture(scope="module")
def moe():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    import mxfp4_weight_mxfp8_gb300 as m

    return m


_LAYERS: dict = {}


def layer_for(moe, weights):
    """One prepared layer per weight set for the session. The cache keeps the weight
    set itself too, so that its id() cannot be reused by a later weight set."""
    import torch

    w13 = weights[0]
    key = (w13.shape, id(weights))
    if key not in _LAYERS:
        dev = torch.device("cuda:0")
        _LAYERS[key] = (moe.MoeLayer(tuple(torch.from_numpy(w).to(dev) for w in weights)), weights)
    return _LAYERS[key][0]


def to_device(x_bits, ids):
    import torch

    dev = torch.device("cuda:0")
    xd = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev).view(torch.bfloat16)
    return xd, torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev)


def bf16_to_float(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_layer(moe, layer, x_bits, ids):
    import torch

    xd, idsd = to_device(x_bits, ids)
    out = layer(xd, idsd)
    status = moe.moe_sync_status(layer.handle)
    B = x_bits.shape[0]
    got = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, layer.hidden)
    return got, status


def check_rows(got_bits, ref_bits, label):
    got, ref = bf16_to_float(got_bits).astype(np.float64), bf16_to_float(ref_bits).astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    worst = np.max(np.abs(got - ref) / np.maximum(rms, 1e-300))
    print(f"[{label}] rel L2 {rel:.3e}, worst |err|/rms(row) {worst:.3e}")
    assert rel <= REL_L2, f"{label}: relative L2 {rel}"
    assert worst <= ROW_TOL, f"{label}: element error {worst} x rms(row)"
    return rel, worst


def units_of(moe, layer, batch):
    count = np.zeros(1, np.int32)
    cap = batch * 16
    experts = np.zeros(cap, np.int32)
    rows = np.zeros(cap * 8, np.int16)
    moe.moe_copy_units(layer.handle, count, experts, rows, cap)
    n = int(count[0])
    return experts[:n], rows[: n * 8].reshape(n, 8)


CONFIGS = ["tiny", "tp8_b1", "tp16_b8", "tp8_b64", "tp8_b256"]


@pytest.mark.parametrize("name", CONFIGS)
def test_quantize_plan_is_bit_exact(moe, name):
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    xd, _ = to_device(x, ids)
    B, H = x.shape
    moe.moe_quantize(layer.handle, xd, B)
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    codes = np.zeros((B, H), np.uint8)
    scales = np.zeros((B, H // 32), np.uint8)
    moe.moe_copy_plan(layer.handle, codes, scales, B)
    ref_codes, ref_scales = oracle.quantize_x(x)
    np.testing.assert_array_equal(scales, ref_scales)
    np.testing.assert_array_equal(codes, ref_codes)


def test_quantize_edge_values_are_bit_exact(moe):
    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    H = 256
    rng = np.random.default_rng(17)
    rows = []
    rows.append(np.zeros(H, np.uint16))                                   # all-zero blocks
    rows.append(np.full(H, 0x8000, np.uint16))                           # negative zeros
    rows.append(rng.integers(1, 0x80, H).astype(np.uint16))              # BF16 subnormals
    rows.append((rng.integers(1, 0x80, H) | 0x8000).astype(np.uint16))   # negative subnormals
    rows.append(np.full(H, 0x7F7F, np.uint16))                            # largest finite BF16
    big = rng.integers(0x7F00, 0x7F80, H).astype(np.uint16)
    big[::3] |= 0x8000
    rows.append(big)                                                      # huge magnitudes
    mixed = workload.float_to_bf16_bits(rng.standard_normal(H).astype(np.float32))
    mixed[::32] = workload.float_to_bf16_bits(np.float32(1.75))[()]        # the 1.75 boundary
    mixed[1::32] = workload.float_to_bf16_bits(np.float32(-1e-6))[()]
    rows.append(mixed)
    tiny_block = workload.float_to_bf16_bits((rng.standard_normal(H) * 1e-38).astype(np.float32))
    rows.append(tiny_block)
    x = np.stack(rows)
    xd, _ = to_device(x, np.zeros((len(rows), 16), np.int32))
    moe.moe_quantize(layer.handle, xd, x.shape[0])
    codes = np.zeros(x.shape, np.uint8)
    scales = np.zeros((x.shape[0], H // 32), np.uint8)
    moe.moe_copy_plan(layer.handle, codes, scales, x.shape[0])
    ref_codes, ref_scales = oracle.quantize_x(x)
    np.testing.assert_array_equal(scales, ref_scales)
    np.testing.assert_array_equal(codes, ref_codes)


@pytest.mark.parametrize("name", CONFIGS)
def test_group_matches_oracle_exactly(moe, name):
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    _, idsd = to_device(x, ids)
    B = ids.shape[0]
    moe.moe_group(layer.handle, idsd, B)
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    experts, rows = units_of(moe, layer, B)
    ref_experts, ref_rows = oracle.group(ids, layer.experts)
    np.testing.assert_array_equal(experts, ref_experts)
    np.testing.assert_array_equal(rows, ref_rows)


@pytest.mark.parametrize("batch", [16, 17])
def test_grouping_paths_at_the_small_batch_threshold(moe, batch):
    """Up to 16 tokens the grouping block takes its one-pair-per-thread path,
    above it the general one. Zipf ids over 32 experts give experts with more
    than 8 pairs, so both paths must split them into several units."""
    weights, _, _ = cached_inputs("tiny")
    x = workload.make_x(batch, 256, seed=7)
    ids = workload.make_ids(batch, 32, seed=11, dist="zipf", s=1.1)
    assert np.bincount(ids.ravel(), minlength=32).max() > 8
    layer = layer_for(moe, weights)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    experts, rows = units_of(moe, layer, batch)
    ref_experts, ref_rows = oracle.group(ids, layer.experts)
    np.testing.assert_array_equal(experts, ref_experts)
    np.testing.assert_array_equal(rows, ref_rows)
    xq, xs = oracle.quantize_x(x)
    check_rows(got, oracle.pairs_forward(weights, xq, xs, ids)["out"], f"tiny B{batch} zipf")


def oracle_pairs_for(name, weights, x, ids):
    """Every pair of the call (TP8 B256: 4,096 pairs, about 15 s of oracle time)."""
    return np.arange(ids.size, dtype=np.int32)


_ORACLE_RUNS: dict = {}


def oracle_run(name):
    """(pairs, oracle outputs with hidden codes) of a config, computed once."""
    if name not in _ORACLE_RUNS:
        weights, x, ids = cached_inputs(name)
        pairs = oracle_pairs_for(name, weights, x, ids)
        xq, xs = oracle.quantize_x(x)
        _ORACLE_RUNS[name] = (pairs, oracle.pairs_forward(weights, xq, xs, ids, pairs=pairs,
                                                          want_hidden=True))
    return _ORACLE_RUNS[name]


def routing_weights(batch, seed=5):
    """Positive float32 weights per token, summing to one (a softmax's shape)."""
    w = np.random.default_rng(seed).random((batch, 16)).astype(np.float32) + 0.1
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


def run_combined(moe, layer, x_bits, ids, rw):
    import torch

    xd, idsd = to_device(x_bits, ids)
    B = x_bits.shape[0]
    wd = torch.from_numpy(rw).to("cuda:0")
    out = torch.full((B, layer.hidden), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    moe.moe_run_combined(layer.handle, xd, idsd, wd, out, B)
    status = moe.moe_sync_status(layer.handle)
    return out.view(torch.int16).cpu().numpy().view(np.uint16), status


@pytest.mark.parametrize("name", CONFIGS)
def test_run_matches_oracle(moe, name):
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    pairs, ref = oracle_run(name)
    check_rows(got[pairs], ref["out"], name)

    # Hidden requant flips, unit row by unit row.
    experts, rows = units_of(moe, layer, x.shape[0])
    I = layer.inter
    hq = np.zeros((len(experts), 8, I), np.uint8)
    hs = np.zeros((len(experts), 8, I // 32), np.uint8)
    moe.moe_copy_hidden(layer.handle, hq, hs, len(experts))
    where = {int(p): i for i, p in enumerate(pairs)}
    gpu_hq, gpu_hs, sel = [], [], []
    for u in range(len(experts)):
        for r in range(8):
            p = int(rows[u, r])
            if p >= 0 and p in where:
                gpu_hq.append(hq[u, r])
                gpu_hs.append(hs[u, r])
                sel.append(where[p])
    gpu_hq, gpu_hs, sel = np.array(gpu_hq), np.array(gpu_hs), np.array(sel)
    code_flips = int(np.sum(gpu_hq != ref["hq"][sel]))
    scale_flips = int(np.sum(gpu_hs != ref["hs"][sel]))
    total = gpu_hq.size
    print(f"[{name}] hidden requant flips: {code_flips} / {total} codes, "
          f"{scale_flips} / {gpu_hs.size} scales")
    assert code_flips <= max(8, total // 100), "hidden codes differ far more than rounding flips"

    # FC2 alone on the GPU's own hidden codes: isolates the flips.
    fc2 = oracle.fc2_rows(weights[2], weights[3], ids.reshape(-1)[pairs[sel]], gpu_hq, gpu_hs)
    got_sel = bf16_to_float(got[pairs[sel]]).astype(np.float64)
    ref_sel = bf16_to_float(fc2).astype(np.float64)
    rel = np.linalg.norm(got_sel - ref_sel) / max(np.linalg.norm(ref_sel), 1e-300)
    print(f"[{name}] FC2 on GPU hidden codes: rel L2 {rel:.3e}")
    assert rel <= 2e-3


@pytest.mark.parametrize("batch", [1, 3, 8, 9, 17, 64, 256])
def test_ragged_batches_tiny_layer(moe, batch):
    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    x = workload.make_x(batch, 256, seed=100 + batch)
    ids = workload.make_ids(batch, 32, seed=200 + batch, dist="zipf" if batch % 2 else "uniform")
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids)
    check_rows(got, ref["out"], f"tiny B={batch}")


def test_partial_tiles_and_host_weights(moe):
    """I = 96: a gate/up tile pair with 32 padded rows and a 96-K FC2 chunk;
    H = 512; the weights are passed as host arrays."""
    E, H, I, B = 16, 512, 96, 5
    weights = workload.make_weights(E, H, I, seed13=7, seed2=8)
    layer = moe.MoeLayer(weights)
    x = workload.make_x(B, H, seed=9)
    ids = workload.make_ids(B, E, seed=10)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids)
    check_rows(got, ref["out"], "E=16 H=512 I=96")
    layer.close()


@pytest.mark.parametrize("E,H,I,B,dist", [
    (1024, 256, 64, 256, "uniform"),   # most experts, largest batch: 1,536 units
    (16, 16384, 512, 2, "uniform"),    # largest hidden and intermediate sizes
    (1024, 256, 512, 16, "zipf"),      # largest I with many experts
    (16, 16384, 64, 4, "zipf"),        # largest hidden with the smallest I
])
def test_supported_limits(moe, E, H, I, B, dist):
    """The edges of the supported shapes (include/moe.h): E <= 1024, H <= 16384,
    I <= 512, B <= 256, against the oracle on every pair."""
    weights = workload.make_weights(E, H, I, seed13=21, seed2=22)
    import torch

    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to("cuda:0") for w in weights))
    x = workload.make_x(B, H, seed=23)
    ids = workload.make_ids(B, E, seed=24, dist=dist)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids)
    check_rows(got, ref["out"], f"E={E} H={H} I={I} B={B}")
    layer.close()


SMALL_PATHS = [1, 2]  # the small-batch kernel, the cluster variant


# The widest layer the small-batch kernel serves at I = 512: its packed build (one or two
# tokens, 3-slot ring, x images 256 bytes apart) holds 32 K chunks of x in half an SM, its
# wide build (up to eight tokens, full 1 KB images) 26.
SMALL_MAX_HIDDEN = {1: 4096, 2: 4096, 8: 3328}


def small_too_wide(shape, batch):
    """Whether the small-batch kernel leaves a layer of this (H, I) to the grid kernel."""
    H, I = shape
    widest = SMALL_MAX_HIDDEN[1] if batch <= 2 else SMALL_MAX_HIDDEN[8]
    return I == 512 and H > widest


def set_path(moe, layer, path, batch, shape=None):
    """Select an experts kernel for calls of `batch` tokens and check that it serves them.
    Paths 1 and 3 both run the small-batch kernel, which leaves layers wider than
    SMALL_MAX_HIDDEN (its x images would not fit half an SM) to the grid kernel."""
    moe.moe_debug_paths(layer.handle, path)
    if path in (1, 3) and shape is not None and small_too_wide(shape, batch):
        assert moe.moe_kernel_path(layer.handle, batch) == 0
        return
    assert moe.moe_kernel_path(layer.handle, batch) == (1 if path == 3 else path)
    if path == 2:
        assert moe.moe_cluster_size(layer.handle, batch) >= 2


@pytest.mark.parametrize("path", SMALL_PATHS, ids=["small", "cluster"])
@pytest.mark.parametrize("E,H,I,B", [
    (16, 512, 96, 1),      # partial tiles (I = 96); clusters of 6
    (16, 512, 96, 2),      # two-row units; the piece layout allows only small clusters
    (8, 3584, 384, 1),     # fewer experts than slots: 8 units; clusters of 8
    (32, 3584, 384, 2),    # the TP8 shard's shape at two tokens; clusters of 4
    (1024, 256, 512, 2),   # the widest I with the smallest H
    (16, 16384, 512, 1),   # the largest H and I (the small-batch path falls back to the grid kernel)
])
def test_small_batch_path_shapes(moe, E, H, I, B, path):
    """The small-batch kernel and the cluster variant over odd shapes, against the oracle."""
    weights = workload.make_weights(E, H, I, seed13=31, seed2=32)
    import torch

    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to("cuda:0") for w in weights))
    set_path(moe, layer, path, B, shape=(H, I))
    print(f"[E={E} H={H} I={I} B={B}] path {path}, clusters of {moe.moe_cluster_size(layer.handle, B)}")
    x = workload.make_x(B, H, seed=33)
    ids = workload.make_ids(B, E, seed=34) if E >= 16 else np.stack(
        [np.random.default_rng(35 + t).permutation(16) % E for t in range(B)]).astype(np.int32)
    got, status = run_layer(moe, layer, x, ids)
    xq, xs = oracle.quantize_x(x)
    if E >= 16:
        assert status == moe.MOE_OK
        ref = oracle.pairs_forward(weights, xq, xs, ids)
        check_rows(got, ref["out"], f"path {path} E={E} H={H} I={I} B={B}")
    else:
        # 16 slots over 8 experts: each expert twice per token, the higher slot dropped.
        assert status == moe.MOE_ERR_DEVICE_IDS
        keep = np.array([t * 16 + s for t in range(B) for s in range(16)
                         if s == min(np.nonzero(ids[t] == ids[t, s])[0])], np.int32)
        ref = oracle.pairs_forward(weights, xq, xs, ids, pairs=keep)
        check_rows(got[keep], ref["out"], f"path {path} E={E} H={H} I={I} B={B}")
    layer.close()


@pytest.mark.parametrize("B", [1, 2, 8])
def test_small_batch_widest_hidden(moe, B):
    """The widest layer the small-batch kernel serves at the widest I (32 K chunks of x
    in the packed build at one or two tokens, 26 in the wide build; two CTAs per SM),
    against the oracle; two chunks more fall back."""
    E, H, I = 16, SMALL_MAX_HIDDEN[B], 512
    weights = workload.make_weights(E, H, I, seed13=36, seed2=37)
    import torch

    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to("cuda:0") for w in weights))
    set_path(moe, layer, 1 if B <= 2 else 3, B, shape=(H, I))
    x = workload.make_x(B, H, seed=38)
    ids = workload.make_ids(B, E, seed=39)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids)
    check_rows(got, ref["out"], f"small E={E} H={H} I={I} B={B}")
    layer.close()
    wider = moe.MoeLayer(tuple(torch.from_numpy(w).to("cuda:0")
                               for w in workload.make_weights(E, H + 256, I, seed13=36, seed2=37)))
    set_path(moe, wider, 1 if B <= 2 else 3, B, shape=(H + 256, I))
    wider.close()


@pytest.mark.parametrize("shape,B", [((32, 1024, 128), 3), ((32, 1024, 128), 5), ((32, 1024, 128), 8),
                                     ((16, 512, 96), 3), ((16, 512, 96), 4), ("tp16_b8", 8)])
def test_small_batch_wide_path(moe, shape, B):
    """Path 3: the small-batch kernel for calls of up to eight tokens (one FC1 segment
    holds eight token rows per tile; the hand-off lands them all), against the oracle.
    Path 1 sends the same calls to the grid kernel."""
    if shape == "tp16_b8":
        weights, _, _ = cached_inputs(shape)
    else:
        weights = workload.make_weights(*shape, seed13=42, seed2=43)
    layer = layer_for(moe, weights)
    E, H = weights[0].shape[0], layer.hidden
    x = workload.make_x(B, H, seed=44 + B)
    ids = workload.make_ids(B, E, seed=45 + B)
    try:
        moe.moe_debug_paths(layer.handle, 1)
        assert moe.moe_kernel_path(layer.handle, B) == 0
        set_path(moe, layer, 3, B)
        got, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        again, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
    finally:
        moe.moe_debug_paths(layer.handle, 1)
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids)
    check_rows(got, ref["out"], f"path 3 {shape} B={B}")
    assert np.array_equal(got, again)


@pytest.mark.parametrize("B", [5, 8])
def test_small_batch_wide_path_reads_back_and_reports_bad_ids(moe, B):
    """Path 3 at five and eight tokens over 32 experts, so most units hold several tokens'
    rows (the unit table spans several warps and the token masks): the plan and unit table
    left for read-back are the oracle's, bit for bit. A call with a repeated and two
    out-of-range ids reports them and keeps every other pair exact; the table it leaves
    drops those pairs; the next call gives the first call's bits again."""
    weights = workload.make_weights(32, 1024, 128, seed13=52, seed2=53)
    layer = layer_for(moe, weights)
    x = workload.make_x(B, 1024, seed=54 + B)
    ids = workload.make_ids(B, 32, seed=55 + B)
    xq, xs = oracle.quantize_x(x)
    try:
        set_path(moe, layer, 3, B)
        first, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        codes = np.zeros((B, 1024), np.uint8)
        scales = np.zeros((B, 1024 // 32), np.uint8)
        moe.moe_copy_plan(layer.handle, codes, scales, B)
        np.testing.assert_array_equal(codes, xq)
        np.testing.assert_array_equal(scales, xs)
        experts, rows = units_of(moe, layer, B)
        ref_e, ref_r = oracle.group(ids, 32)
        assert (ref_r >= 0).sum(axis=1).max() >= 2  # units of several rows
        np.testing.assert_array_equal(experts, ref_e)
        np.testing.assert_array_equal(rows, ref_r)
        check_rows(first, oracle.pairs_forward(weights, xq, xs, ids)["out"], f"path 3 E32 B={B}")

        bad = ids.copy()
        bad[1, 9] = bad[1, 3]   # a repeat: slot 9 is dropped
        bad[B - 1, 0] = -1      # out of range
        bad[B - 1, 15] = 32     # out of range
        dropped = {1 * 16 + 9, (B - 1) * 16, (B - 1) * 16 + 15}
        got, status = run_layer(moe, layer, x, bad)
        assert status == moe.MOE_ERR_DEVICE_IDS
        keep = np.array([p for p in range(B * 16) if p not in dropped], np.int32)
        check_rows(got[keep], oracle.pairs_forward(weights, xq, xs, bad, pairs=keep)["out"],
                   f"path 3 E32 B={B} with bad ids")
        clean = bad.copy()
        clean[1, 9] = -1
        experts, rows = units_of(moe, layer, B)
        ref_e, ref_r = oracle.group(clean, 32)
        np.testing.assert_array_equal(experts, ref_e)
        np.testing.assert_array_equal(rows, ref_r)

        again, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        np.testing.assert_array_equal(again, first)
    finally:
        moe.moe_debug_paths(layer.handle, 1)


def test_small_batch_wide_path_falls_back(moe):
    """Where three tokens' segment sums would not fit the x images' region (H = 256:
    two K chunks), path 3 leaves the call to the grid kernel; one and two tokens stay."""
    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    try:
        moe.moe_debug_paths(layer.handle, 3)
        assert [moe.moe_kernel_path(layer.handle, b) for b in (1, 2, 3, 8)] == [1, 1, 0, 0]
        with pytest.raises(moe.MoeError):
            moe.moe_debug_paths(layer.handle, 4)
    finally:
        moe.moe_debug_paths(layer.handle, 1)


@pytest.mark.parametrize("path", SMALL_PATHS, ids=["small", "cluster"])
def test_small_batch_paths_with_bad_and_repeated_ids(moe, path):
    """One token whose ids include a repeat and an out-of-range id: 14 units.
    The small-batch kernel derives the same table from the ids in the kernel;
    on the cluster variant the last two clusters find no unit and leave."""
    weights, x, ids = cached_inputs("tp8_b1")
    layer = layer_for(moe, weights)
    set_path(moe, layer, path, 1)
    bad = ids.copy()
    bad[0, 9] = bad[0, 4]   # a repeat: slot 9 is dropped
    bad[0, 12] = 384        # out of range: slot 12 is dropped
    try:
        got, status = run_layer(moe, layer, x, bad)
    finally:
        moe.moe_debug_paths(layer.handle, 1)
    assert status == moe.MOE_ERR_DEVICE_IDS
    experts, _ = units_of(moe, layer, 1)
    assert len(experts) == 14
    keep = np.array([s for s in range(16) if s not in (9, 12)], np.int32)
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, bad, pairs=keep)
    check_rows(got[keep], ref["out"], f"tp8 B1 with bad ids (path {path})")


def test_repeated_expert_is_reported_and_others_kept(moe):
    weights, x, ids = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    bad = ids.copy()
    bad[0, 7] = bad[0, 2]  # token 0 names one expert twice: one of the two pairs is dropped
    got, status = run_layer(moe, layer, x, bad)
    assert status == moe.MOE_ERR_DEVICE_IDS
    keep = np.array([p for p in range(32) if p not in (2, 7)], np.int32)
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, bad, pairs=keep)
    check_rows(got[keep], ref["out"], "tiny with a repeated id")


def test_run_host_equals_device_run(moe):
    import torch

    weights, x, ids = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    got, _ = run_layer(moe, layer, x, ids)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    idsh = torch.from_numpy(ids).pin_memory()
    outh = torch.empty((x.shape[0], 16, 256), dtype=torch.int16).pin_memory()
    moe.moe_run_host(layer.handle, xh, idsh, outh, x.shape[0])
    np.testing.assert_array_equal(outh.numpy().view(np.uint16).reshape(-1, 256), got)


def test_run_host_in_place_and_copied(moe):
    """moe_run_host on pinned buffers (used in place by the kernels) and on
    pageable arrays (copied), each against moe_run; then a bad id through the
    pinned path reports its status from the host-side status word."""
    import torch

    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    for step, batch in enumerate([8, 3, 1]):
        x = workload.make_x(batch, 256, seed=400 + step)
        ids = workload.make_ids(batch, 32, seed=500 + step)
        want, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        idsh = torch.from_numpy(ids).pin_memory()
        outh = torch.zeros((batch, 16, 256), dtype=torch.int16).pin_memory()
        moe.moe_run_host(layer.handle, xh, idsh, outh, batch)
        np.testing.assert_array_equal(outh.numpy().view(np.uint16).reshape(-1, 256), want)
        out = np.zeros((batch, 16, 256), np.uint16)
        moe.moe_run_host(layer.handle, x, ids, out, batch)
        np.testing.assert_array_equal(out.reshape(-1, 256), want)
    bad = ids.copy()
    bad[0, 0] = 99
    idsh = torch.from_numpy(bad).pin_memory()
    with pytest.raises(moe.MoeError) as err:
        moe.moe_run_host(layer.handle, xh, idsh, outh, 1)
    assert err.value.code == moe.MOE_ERR_DEVICE_IDS
    moe.moe_run_host(layer.handle, xh, torch.from_numpy(ids).pin_memory(), outh, 1)


@pytest.mark.parametrize("batch", [1, 2])
def test_run_host_on_the_packed_small_build(moe, batch):
    """One or two tokens on a layer where the small kernel's packed build (x and hidden
    images 256 bytes apart) fits: moe_run_host copies the prep grid's plan into those
    images (pinned buffers in place, pageable ones copied) and equals moe_run, which
    quantizes x in the kernel, bit for bit; moe_run matches the oracle."""
    import torch

    weights = workload.make_weights(32, 1024, 128, seed13=60, seed2=61)
    layer = layer_for(moe, weights)
    x = workload.make_x(batch, 1024, seed=62 + batch)
    ids = workload.make_ids(batch, 32, seed=63 + batch)
    assert moe.moe_kernel_path(layer.handle, batch) == moe.PATH_SMALL
    want, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    check_rows(want, oracle.pairs_forward(weights, xq, xs, ids)["out"], f"packed build B={batch}")
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    idsh = torch.from_numpy(ids).pin_memory()
    outh = torch.zeros((batch, 16, 1024), dtype=torch.int16).pin_memory()
    moe.moe_run_host(layer.handle, xh, idsh, outh, batch)
    np.testing.assert_array_equal(outh.numpy().view(np.uint16).reshape(-1, 1024), want)
    out = np.zeros((batch, 16, 1024), np.uint16)
    moe.moe_run_host(layer.handle, x, ids, out, batch)
    np.testing.assert_array_equal(out.reshape(-1, 1024), want)


@pytest.mark.parametrize("B", [4, 8, 40])
def test_grid_calls_alternating_handles_start_early(moe, B):
    """Grid-kernel calls alternating between two handles on one stream: each call after
    the other handle's starts early (its prep grid writes the handle's tables without
    waiting for the previous grid, its experts kernel streams FC1 while the previous call
    runs, and waits for it only before its first output row). Every call's rows equal the
    same call made alone, and when all calls write one output buffer it ends with the last
    call's rows."""
    import torch

    wa = workload.make_weights(64, 1024, 256, seed13=70, seed2=71)
    wb = workload.make_weights(64, 1024, 256, seed13=72, seed2=73)
    la, lb = layer_for(moe, wa), layer_for(moe, wb)
    assert moe.moe_kernel_path(la.handle, B) == moe.PATH_GRID
    n = 6
    layers = [la, lb] * (n // 2)
    xs = [workload.make_x(B, 1024, seed=80 + i) for i in range(n)]
    idss = [workload.make_ids(B, 64, seed=90 + i) for i in range(n)]
    want = []
    for layer, x, ids in zip(layers, xs, idss):
        got, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        want.append(got)
    xq, xsc = oracle.quantize_x(xs[1])
    check_rows(want[1], oracle.pairs_forward(wb, xq, xsc, idss[1])["out"], f"handle B, B={B}")
    dev = [to_device(x, ids) for x, ids in zip(xs, idss)]
    stream = torch.cuda.Stream()
    for rep in range(3):
        outs = [torch.full((B, 16, 1024), float("nan"), dtype=torch.bfloat16, device="cuda:0") for _ in range(n)]
        shared = torch.full((B, 16, 1024), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for layer, (xd, idsd), o in zip(layers, dev, outs):
                layer(xd, idsd, out=o, stream=stream.cuda_stream)
            for layer, (xd, idsd) in zip(layers, dev):
                layer(xd, idsd, out=shared, stream=stream.cuda_stream)
        stream.synchronize()
        for layer in (la, lb):
            assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
        for i, o in enumerate(outs):
            got = o.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, 1024)
            np.testing.assert_array_equal(got, want[i], err_msg=f"rep {rep} call {i}")
        got = shared.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, 1024)
        np.testing.assert_array_equal(got, want[-1], err_msg=f"rep {rep}, shared output")


def test_early_grid_calls_replayed_in_a_graph_with_new_inputs(moe):
    """Grid-kernel calls alternating between two handles, captured once in a CUDA graph
    and replayed with new routing ids and activations in the same buffers: the early-start
    flag of each call is back at rest after the call, so a replay's experts kernel reads
    the tables its own prep grid wrote, never the previous replay's."""
    import torch

    B = 8
    wa = workload.make_weights(64, 1024, 256, seed13=74, seed2=75)
    wb = workload.make_weights(64, 1024, 256, seed13=76, seed2=77)
    layers = [layer_for(moe, wa), layer_for(moe, wb)] * 2
    n = len(layers)
    xbufs = [torch.empty((B, 1024), dtype=torch.bfloat16, device="cuda:0") for _ in range(n)]
    idbufs = [torch.empty((B, 16), dtype=torch.int32, device="cuda:0") for _ in range(n)]
    outs = [torch.empty((B, 16, 1024), dtype=torch.bfloat16, device="cuda:0") for _ in range(n)]

    def fill(rep):
        inputs = []
        for i in range(n):
            x = workload.make_x(B, 1024, seed=100 + 10 * rep + i)
            ids = workload.make_ids(B, 64, seed=200 + 10 * rep + i)
            xd, idsd = to_device(x, ids)
            xbufs[i].copy_(xd)
            idbufs[i].copy_(idsd)
            inputs.append((x, ids))
        return inputs

    stream = torch.cuda.Stream()
    fill(0)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):  # warm up on the capture stream
        for layer, xb, ib, o in zip(layers, xbufs, idbufs, outs):
            layer(xb, ib, out=o, stream=stream.cuda_stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for layer, xb, ib, o in zip(layers, xbufs, idbufs, outs):
            layer(xb, ib, out=o, stream=stream.cuda_stream)
    for rep in range(1, 4):
        inputs = fill(rep)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for layer in layers[:2]:
            assert moe.moe_sync_status(layer.handle) == moe.MOE_OK, f"replay {rep}"
        for i, (layer, (x, ids)) in enumerate(zip(layers, inputs)):
            want, status = run_layer(moe, layer, x, ids)
            assert status == moe.MOE_OK
            got = outs[i].view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, 1024)
            np.testing.assert_array_equal(got, want, err_msg=f"replay {rep}, call {i}")


def test_run_host_replay_graph_follows_buffers_batch_and_settings(moe):
    """The in-place moe_run_host replays a captured graph. The same pinned
    buffers with new contents are read afresh, and a smaller batch, a
    cluster-path switch or a new timeout captures again. Each call equals
    moe_run on device copies."""
    import torch

    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    xh = torch.zeros((4, 256), dtype=torch.int16).pin_memory()
    idsh = torch.zeros((4, 16), dtype=torch.int32).pin_memory()
    outh = torch.zeros((4, 16, 256), dtype=torch.int16).pin_memory()
    steps = [(4, None), (4, None), (2, None), (2, ("paths", 0)), (4, ("timeout", 50_000_000)), (4, None)]
    try:
        for step, (batch, setting) in enumerate(steps):
            if setting and setting[0] == "paths":
                moe.moe_debug_paths(layer.handle, setting[1])
            if setting and setting[0] == "timeout":
                moe.moe_set_timeout(layer.handle, setting[1])
            x = workload.make_x(batch, 256, seed=600 + step)
            ids = workload.make_ids(batch, 32, seed=700 + step)
            want, status = run_layer(moe, layer, x, ids)
            assert status == moe.MOE_OK
            xh[:batch].copy_(torch.from_numpy(x.view(np.int16)))
            idsh[:batch].copy_(torch.from_numpy(ids))
            outh.zero_()
            moe.moe_run_host(layer.handle, xh, idsh, outh, batch)
            got = outh[:batch].numpy().view(np.uint16).reshape(-1, 256)
            np.testing.assert_array_equal(got, want, err_msg=f"step {step}")
    finally:
        moe.moe_debug_paths(layer.handle, 1)
        moe.moe_set_timeout(layer.handle, 0)


def test_quantize_group_experts_equals_run(moe):
    weights, x, ids = cached_inputs("tp16_b8")
    layer = layer_for(moe, weights)
    import torch

    got, _ = run_layer(moe, layer, x, ids)
    xd, idsd = to_device(x, ids)
    B = x.shape[0]
    out = torch.empty((B, 16, layer.hidden), dtype=torch.bfloat16, device="cuda:0")
    moe.moe_quantize(layer.handle, xd, B)
    moe.moe_group(layer.handle, idsd, B)
    moe.moe_experts(layer.handle, out, B)
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    np.testing.assert_array_equal(
        out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B * 16, -1), got)


def test_runs_are_deterministic(moe):
    weights, x, ids = cached_inputs("tp8_b64")
    layer = layer_for(moe, weights)
    a, _ = run_layer(moe, layer, x, ids)
    b, _ = run_layer(moe, layer, x, ids)
    np.testing.assert_array_equal(a, b)


def test_out_of_range_ids_are_reported_and_skipped(moe):
    weights, x, ids = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    bad = ids.copy()
    bad[0, 3] = 32   # out of range
    bad[1, 5] = -1
    got, status = run_layer(moe, layer, x, bad)
    assert status == moe.MOE_ERR_DEVICE_IDS
    keep = np.array([p for p in range(32) if p not in (3, 16 + 5)], np.int32)
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids, pairs=keep)
    check_rows(got[keep], ref["out"], "tiny with bad ids")


@pytest.mark.parametrize("name,path", [("tiny", 1), ("tiny", 2), ("tiny", 0), ("tp8_b1", 1)],
                         ids=["small", "cluster", "grid", "tp8_b1-small-packed"])
def test_bounded_wait_reports_timeout_and_context_survives(moe, name, path):
    """Unit 0's FC1 results are never published: its consumers' bounded waits run out,
    the call reports the timeout, and the next call on the handle is exact (tiny at two
    tokens runs the small kernel's wide build, TP8 at one token its packed build)."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    try:
        set_path(moe, layer, path, x.shape[0])
        moe.moe_set_timeout(layer.handle, 20_000_000)  # 20 ms
        moe.moe_debug_withhold(layer.handle, 0)        # unit 0 never publishes its hidden vector
        _, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_ERR_DEVICE_TIMEOUT
        moe.moe_debug_withhold(layer.handle, -1)
        moe.moe_set_timeout(layer.handle, 0)
        got, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
    finally:
        moe.moe_debug_withhold(layer.handle, -1)
        moe.moe_set_timeout(layer.handle, 0)
        moe.moe_debug_paths(layer.handle, 1)
    xq, xs = oracle.quantize_x(x)
    check_rows(got, oracle.pairs_forward(weights, xq, xs, ids)["out"], f"{name} after timeout")


@pytest.mark.parametrize("name,path", [("tiny", 0), ("tp16_b8", 0), ("tiny", 1), ("tp8_b1", 1)],
                         ids=["tiny-grid", "tp16_b8-grid", "tiny-small", "tp8_b1-small"])
def test_mbarrier_timeout_aborts_and_context_survives(moe, name, path):
    """The grid kernel's abort path, made to run deterministically: the
    hidden loader never hands unit 0's image to the MMA issuers, so their
    bounded mbarrier wait runs out and every CTA with a job of that unit gives
    up (the other roles stop, MMAs drain, copies settle). The call reports
    the timeout and ends; the next call is exact. On the small-batch kernel
    the epilogue never releases unit 0's hidden image to the issuers."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    try:
        set_path(moe, layer, path, x.shape[0])
        moe.moe_set_timeout(layer.handle, 20_000_000)  # 20 ms
        moe.moe_debug_withhold_image(layer.handle, 0)
        _, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_ERR_DEVICE_TIMEOUT
        moe.moe_debug_withhold_image(layer.handle, -1)
        moe.moe_set_timeout(layer.handle, 0)
        got, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
    finally:
        moe.moe_debug_withhold_image(layer.handle, -1)
        moe.moe_set_timeout(layer.handle, 0)
        moe.moe_debug_paths(layer.handle, 1)
    xq, xs = oracle.quantize_x(x)
    check_rows(got, oracle.pairs_forward(weights, xq, xs, ids)["out"], f"{name} after an abort")


@pytest.mark.parametrize("name", ["tiny", "tp8_b1"])
def test_three_paths_for_one_and_two_tokens(moe, name):
    """One- and two-token calls run on the small-batch kernel by default; the
    cluster variant and the grid kernel serve them when selected. All three
    meet the oracle's tolerances and agree with each other up to the
    rounding of their different split-K groupings."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    B = x.shape[0]
    pairs, ref = oracle_run(name)
    assert moe.moe_kernel_path(layer.handle, B) == 1
    rows = {}
    try:
        for path, label in [(1, "small"), (2, "cluster"), (0, "grid")]:
            set_path(moe, layer, path, B)
            rows[label], status = run_layer(moe, layer, x, ids)
            assert status == moe.MOE_OK
            check_rows(rows[label][pairs], ref["out"], f"{name} {label} path")
    finally:
        moe.moe_debug_paths(layer.handle, 1)
    base = bf16_to_float(rows["grid"]).astype(np.float64)
    for label in ("small", "cluster"):
        other = bf16_to_float(rows[label]).astype(np.float64)
        rel = np.linalg.norm(other - base) / max(np.linalg.norm(base), 1e-300)
        print(f"[{name}] {label} vs grid: rel L2 {rel:.3e}")
        assert rel <= 2e-3


@pytest.mark.parametrize("path", [1, 2, 0], ids=["small", "cluster", "grid"])
def test_floor_rule_pair_golden_on_the_gpu(moe, path):
    """The hand-worked pair of golden/floor_rule_pair.json (I = 384: the floor
    rule saturates its hidden block) through the kernels: its hidden codes,
    scales and output bits are the golden's, on both paths, and every other
    pair (an all-zero expert) gives +0.0 rows."""
    import torch
    from conftest import floor_rule_pair_case

    weights, x, ids, spec = floor_rule_pair_case()
    dev = torch.device("cuda:0")
    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to(dev) for w in weights))
    try:
        set_path(moe, layer, path, 1)
        got, status = run_layer(moe, layer, x, ids)
        assert status == moe.MOE_OK
        H, I = spec["hidden"], spec["inter"]
        out = np.full(H, spec["out_bits_default"], np.uint16)
        for n, v in spec["out_bits"].items():
            out[int(n)] = v
        np.testing.assert_array_equal(got[0], out)
        assert not got[1:].any()
        experts, _ = units_of(moe, layer, 1)
        hq = np.zeros((len(experts), 8, I), np.uint8)
        hs = np.zeros((len(experts), 8, I // 32), np.uint8)
        moe.moe_copy_hidden(layer.handle, hq, hs, len(experts))
        assert experts[0] == 0
        expect_hs = np.full(I // 32, spec["hidden_scale_default"], np.uint8)
        expect_hs[0] = spec["hidden_scales"]["0"]
        expect_hq = np.full(I, spec["hidden_code_default"], np.uint8)
        expect_hq[0] = spec["hidden_codes"]["0"]
        np.testing.assert_array_equal(hs[0, 0], expect_hs)
        np.testing.assert_array_equal(hq[0, 0], expect_hq)
    finally:
        layer.close()


@pytest.mark.parametrize("path", SMALL_PATHS, ids=["small", "cluster"])
def test_small_batch_paths_at_two_tokens_with_shared_experts(moe, path):
    """Two tokens routed to the same experts: every unit holds two rows, so
    each split-K piece carries two rows of partial sums."""
    weights, x, _ = cached_inputs("tp8_b1")
    rng = np.random.default_rng(11)
    x2 = np.concatenate([x, x[:1] ^ np.uint16(0x0001)], axis=0)  # a second, slightly different row
    row = rng.permutation(weights[0].shape[0])[:16].astype(np.int32)
    ids = np.stack([row, row[::-1]]).astype(np.int32)
    layer = layer_for(moe, weights)
    try:
        set_path(moe, layer, path, 2)
        got, status = run_layer(moe, layer, x2, ids)
    finally:
        moe.moe_debug_paths(layer.handle, 1)
    assert status == moe.MOE_OK
    experts, rows = units_of(moe, layer, 2)
    assert len(experts) == 16 and np.all(rows[:, 1] >= 0)
    xq, xs = oracle.quantize_x(x2)
    check_rows(got, oracle.pairs_forward(weights, xq, xs, ids)["out"], "tp8 two tokens, shared experts")


@pytest.mark.parametrize("name", CONFIGS)
def test_run_combined_matches_oracle(moe, name):
    """Routing-weighted combine (ExpertsKernel.finalize on one GPU) against the
    oracle's combine of its own per-pair rows, on every token whose 16 pairs
    the oracle ran."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    rw = routing_weights(x.shape[0])
    got, status = run_combined(moe, layer, x, ids, rw)
    assert status == moe.MOE_OK
    pairs, ref = oracle_run(name)
    tokens = pairs.reshape(-1, 16)[:, 0] // 16
    assert np.array_equal(pairs.reshape(-1, 16), tokens[:, None] * 16 + np.arange(16))
    check_rows(got[tokens], oracle.combine(ref["out"], rw[tokens]), f"{name} combined")


def test_run_combined_leaves_out_dropped_pairs(moe):
    weights, x, ids = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    bad = ids.copy()
    bad[0, 7] = bad[0, 2]  # up to 16 tokens the lower slot of a repeat is kept
    rw = routing_weights(x.shape[0], seed=9)
    got, status = run_combined(moe, layer, x, bad, rw)
    assert status == moe.MOE_ERR_DEVICE_IDS
    kept = np.ones(32, np.uint8)
    kept[7] = 0
    xq, xs = oracle.quantize_x(x)
    rows = oracle.pairs_forward(weights, xq, xs, bad)["out"]
    check_rows(got, oracle.combine(rows, rw, kept), "tiny combined with a repeated id")


@pytest.mark.parametrize("name", ["tp8_b1", "tp16_b8"])
def test_kernel_span_records_the_last_launch(moe, name):
    """The launch clock (moe_debug_kernel_span) gives a positive span for the
    last launch, on the cluster variant and on the grid kernel, leaves the rows
    unchanged, reads each launch once, and records nothing when off."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    ref, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    moe.moe_debug_kernel_span(layer.handle, 1)
    try:
        for _ in range(3):
            got, status = run_layer(moe, layer, x, ids)
            assert status == moe.MOE_OK
            np.testing.assert_array_equal(got, ref)
            span = moe.moe_read_kernel_span(layer.handle)
            assert 0 < span < 5_000_000, span
            print(f"[{name}] span {span / 1e3:.2f} us")
        with pytest.raises(moe.MoeError):
            moe.moe_read_kernel_span(layer.handle)  # read already: nothing recorded since
    finally:
        moe.moe_debug_kernel_span(layer.handle, 0)
    run_layer(moe, layer, x, ids)
    with pytest.raises(moe.MoeError):
        moe.moe_read_kernel_span(layer.handle)


@pytest.mark.parametrize("name", ["tiny", "tp8_b1"])
def test_single_launch_call_leaves_plan_and_units_for_read_back(moe, name):
    """A one- or two-token moe_run is the small-batch kernel alone (no prep
    grid): the activation plan and the unit table it leaves for read-back
    are the oracle's, bit for bit, and two runs give the same bits."""
    weights, x, ids = cached_inputs(name)
    layer = layer_for(moe, weights)
    B, H = x.shape
    assert moe.moe_kernel_path(layer.handle, B) == moe.PATH_SMALL
    first, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    codes = np.zeros((B, H), np.uint8)
    scales = np.zeros((B, H // 32), np.uint8)
    moe.moe_copy_plan(layer.handle, codes, scales, B)
    ref_codes, ref_scales = oracle.quantize_x(x)
    np.testing.assert_array_equal(scales, ref_scales)
    np.testing.assert_array_equal(codes, ref_codes)
    experts, rows = units_of(moe, layer, B)
    ref_e, ref_r = oracle.group(ids, weights[0].shape[0])
    np.testing.assert_array_equal(experts, ref_e)
    np.testing.assert_array_equal(rows, ref_r)
    again, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    np.testing.assert_array_equal(again, first)


def test_single_launch_call_after_bad_ids_is_exact(moe):
    """A call with a repeated and an out-of-range id reports them; the next
    call, on the same handle, is exact (its piece counts start from zero)."""
    weights, x, ids = cached_inputs("tp8_b1")
    layer = layer_for(moe, weights)
    bad = ids.copy()
    bad[0, 3] = bad[0, 1]
    bad[0, 7] = -1
    _, status = run_layer(moe, layer, x, bad)
    assert status == moe.MOE_ERR_DEVICE_IDS
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    check_rows(got, oracle.pairs_forward(weights, xq, xs, ids)["out"], "tp8 B1 after bad ids")


def ids_with_counts(B, E, counts, seed):
    """Routing ids where expert k is picked by the first counts[k] tokens and
    the other slots by distinct experts >= len(counts), in shuffled order."""
    rng = np.random.default_rng(seed)
    ids = np.zeros((B, 16), np.int32)
    for t in range(B):
        row = [k for k, c in enumerate(counts) if t < c]
        row += list(rng.choice(np.arange(len(counts), E), 16 - len(row), replace=False))
        row = np.array(row, np.int32)
        rng.shuffle(row)
        ids[t] = row
    return ids


@pytest.mark.parametrize("shape", [(32, 256, 64), (64, 512, 384)], ids=["tiny", "I384"])
@pytest.mark.parametrize("B,counts", [
    (12, [7, 8, 9, 12]),                          # one grouping block path (<= 256 pairs)
    (16, [7, 8, 9, 15, 16]),
    (40, [7, 8, 9, 15, 16, 17, 24, 32, 40]),      # the general grouping path
])
def test_pairs_of_units_at_unit_boundaries(moe, shape, B, counts):
    """Calls of more than 8 tokens run pairs of the table's 8-row units as
    16-row units. Experts with 7, 8, 9, 15, 16, 17, 24, 32 and 40 tokens give
    single units, full and partial pairs and odd unit counts; the output, the
    unit table and the hidden read-back (rows 8-15 of a pair land in the
    second unit's image) must hold for every pair."""
    import torch

    E, H, I = shape
    weights = workload.make_weights(E, H, I, seed13=41, seed2=42)
    layer = moe.MoeLayer(tuple(torch.from_numpy(w).to("cuda:0") for w in weights))
    x = workload.make_x(B, H, seed=43 + B)
    ids = ids_with_counts(B, E, counts, seed=44 + B)
    got, status = run_layer(moe, layer, x, ids)
    assert status == moe.MOE_OK
    xq, xs = oracle.quantize_x(x)
    ref = oracle.pairs_forward(weights, xq, xs, ids, want_hidden=True)
    check_rows(got, ref["out"], f"E={E} H={H} I={I} B={B} counts {counts}")
    experts, rows = units_of(moe, layer, B)
    ref_e, ref_r = oracle.group(ids, E)
    np.testing.assert_array_equal(experts, ref_e)
    np.testing.assert_array_equal(rows, ref_r)
    hq = np.zeros((len(experts), 8, I), np.uint8)
    hs = np.zeros((len(experts), 8, I // 32), np.uint8)
    moe.moe_copy_hidden(layer.handle, hq, hs, len(experts))
    flips = 0
    for u in range(len(experts)):
        for r in range(8):
            p = int(rows[u, r])
            if p >= 0:
                flips += int(np.sum(hq[u, r] != ref["hq"][p]))
                assert np.sum(hs[u, r] != ref["hs"][p]) <= 1, f"unit {u} row {r}: hidden scales"
    assert flips <= max(8, B * 16 * I // 100), f"{flips} hidden code flips"
    layer.close()


@pytest.mark.parametrize("batch", [1, 2, 8])
def test_stacked_combined_calls_read_the_previous_output(moe, batch):
    """Layer stacking: each moe_run_combined call takes the previous call's
    combined output as its x, queued back to back on one stream. The chained
    launches must not let a call read x before the call that writes it has
    ended: the rows equal those of the same calls with a synchronize between."""
    import torch

    weights, _, _ = cached_inputs("tiny")
    layer = layer_for(moe, weights)
    H = layer.hidden
    x0 = workload.make_x(batch, H, seed=61 + batch)
    ids = workload.make_ids(batch, weights[0].shape[0], seed=62 + batch)
    xd, idsd = to_device(x0, ids)
    wd = torch.from_numpy(routing_weights(batch, seed=63)).to("cuda:0")
    depth = 6

    def stack(sync):
        bufs = [xd] + [torch.empty((batch, H), dtype=torch.bfloat16, device="cuda:0") for _ in range(depth)]
        for i in range(depth):
            moe.moe_run_combined(layer.handle, bufs[i], idsd, wd, bufs[i + 1], batch)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
        return [b.view(torch.int16).cpu().numpy() for b in bufs[1:]]

    ref = stack(True)
    for rep in range(3):
        got = stack(False)
        for i in range(depth):
            np.testing.assert_array_equal(got[i], ref[i], err_msg=f"rep {rep} layer {i}")


@pytest.mark.parametrize("batch", [1, 2])
def test_small_calls_replayed_in_graphs(moe, batch):
    """Small-batch calls captured in CUDA graphs and replayed: handles A and B as
    A, B, A and handle C as C, C, C. Across replays a handle's calls need not
    alternate between the two halves of its segment slots and claim counters (B and
    C start each replay on the half their last call used), so each call must leave
    its half at rest. Every replayed output equals the eager call's bits."""
    import torch

    weights, _, _ = cached_inputs("tiny")
    dev = torch.device("cuda:0")
    handles = [moe.MoeLayer(tuple(torch.from_numpy(w).to(dev) for w in weights)) for _ in range(3)]
    H = handles[0].hidden
    x = workload.make_x(batch, H, seed=71 + batch)
    ids = workload.make_ids(batch, weights[0].shape[0], seed=72 + batch)
    xd, idsd = to_device(x, ids)
    ref = handles[0](xd, idsd)
    torch.cuda.synchronize()
    assert moe.moe_sync_status(handles[0].handle) == moe.MOE_OK
    want = ref.view(torch.int16).cpu().numpy()
    order = [0, 1, 0, 2, 2, 2]
    outs = [torch.empty_like(ref) for _ in order]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):  # warm up on the capture stream
        for h, o in zip(order, outs):
            handles[h](xd, idsd, out=o, stream=stream.cuda_stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for h, o in zip(order, outs):
            handles[h](xd, idsd, out=o, stream=stream.cuda_stream)
    for rep in range(3):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for h in handles:
            assert moe.moe_sync_status(h.handle) == moe.MOE_OK, f"replay {rep}"
        for i, o in enumerate(outs):
            assert np.array_equal(o.view(torch.int16).cpu().numpy(), want), f"replay {rep}, call {i}"
    # Eager calls after the replays.
    for h in handles:
        got = h(xd, idsd)
        torch.cuda.synchronize()
        assert moe.moe_sync_status(h.handle) == moe.MOE_OK
        assert np.array_equal(got.view(torch.int16).cpu().numpy(), want)
    del graph
    for h in handles:
        h.close()

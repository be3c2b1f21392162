"""moe_run_noalloc against moe_run, through the C ABI.

moe_run_noalloc takes all per-call scratch from the library's static device
buffer instead of the handle's workspace. It runs the same kernels with the
same work split as moe_run, and every sum of both (split-K pieces in CTA
order, one fixed cut per call) is deterministic, so its rows must equal
moe_run's bit for bit, on consecutive calls that share the buffer. A batch
whose scratch would not fit must be refused before any launch. The file is named so that pytest collects it last; it also passes on
its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

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


def make_layer(moe, weights):
    import torch

    dev = torch.device("cuda:0")
    return moe.MoeLayer(tuple(torch.from_numpy(w).to(dev) for w in weights))


def to_device(x_bits, ids):
    import torch

    dev = torch.device("cuda:0")
    xd = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev).view(torch.bfloat16)
    return xd, torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev)


def rows_as_float(out, batch, hidden):
    import torch

    bits = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(batch * 16, hidden)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_reference(moe, layer, xd, idsd):
    import torch

    batch = int(xd.shape[0])
    out = torch.empty((batch, 16, layer.hidden), dtype=torch.bfloat16, device=xd.device)
    rc = moe.library().moe_run(layer.handle, xd.data_ptr(), idsd.data_ptr(), out.data_ptr(),
                               batch, torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    return rows_as_float(out, batch, layer.hidden)


def run_noalloc(moe, layer, xd, idsd):
    import torch

    batch = int(xd.shape[0])
    # NaN-filled, so a row the call never writes cannot pass.
    out = torch.full((batch, 16, layer.hidden), float("nan"), dtype=torch.bfloat16, device=xd.device)
    rc = moe.library().moe_run_noalloc(layer.handle, xd.data_ptr(), idsd.data_ptr(),
                                       out.data_ptr(), batch,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK, moe.moe_last_error_detail()
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    return rows_as_float(out, batch, layer.hidden)


def check_close(got, ref, label):
    assert np.all(np.isfinite(got)), f"{label}: unwritten or non-finite rows"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    worst = float(np.max(np.abs(got - ref) / np.maximum(rms, 1e-300)))
    print(f"{label}: rel_l2 {rel:.3e} worst/rms {worst:.3e} identical {np.array_equal(got, ref)}")
    # The same kernels and split as moe_run: identical rows. (Had the paths
    # summed in different orders, the parity bars below would be the bar.)
    np.testing.assert_array_equal(got, ref, err_msg=label)
    assert rel <= REL_L2, (label, rel)
    assert worst <= ROW_TOL, (label, worst)


def test_noalloc_matches_moe_run_on_consecutive_calls_tiny(moe):
    weights, x, ids = cached_inputs("tiny")
    layer = make_layer(moe, weights)
    xd, idsd = to_device(x, ids)
    ref = run_reference(moe, layer, xd, idsd)
    for call in range(2):
        check_close(run_noalloc(moe, layer, xd, idsd), ref, f"tiny call {call}")
    layer.close()


def test_noalloc_matches_moe_run_on_consecutive_calls_tp8(moe):
    """Two calls in a row with different batches: the second finds the first
    call's leftovers (and the tiny layer's before it) in the shared buffer."""
    weights, x, ids = cached_inputs("tp8_b64")
    layer = make_layer(moe, weights)
    for call, (lo, hi) in enumerate([(0, 16), (40, 41)]):
        xd, idsd = to_device(x[lo:hi], ids[lo:hi])
        ref = run_reference(moe, layer, xd, idsd)
        check_close(run_noalloc(moe, layer, xd, idsd), ref, f"tp8 call {call} batch {hi - lo}")
    layer.close()


def test_noalloc_refuses_a_batch_beyond_the_static_buffer(moe):
    import torch

    weights, x, ids = cached_inputs("tp8_b256")  # about 9 MB of scratch
    layer = make_layer(moe, weights)
    xd, idsd = to_device(x, ids)
    out = torch.zeros((256, 16, layer.hidden), dtype=torch.bfloat16, device=xd.device)
    torch.cuda.synchronize()
    rc = moe.library().moe_run_noalloc(layer.handle, xd.data_ptr(), idsd.data_ptr(),
                                       out.data_ptr(), 256, torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_ERR_ARG
    detail = moe.moe_last_error_detail()
    assert "scratch" in detail and str(moe.MOE_NOALLOC_SCRATCH_BYTES) in detail, detail
    torch.cuda.synchronize()
    assert not torch.any(out.view(torch.int16) != 0).item(), "a refused call wrote output"
    assert moe.moe_sync_status(layer.handle) == moe.MOE_OK
    layer.close()

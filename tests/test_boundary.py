"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point include/moe.h declares, and rejects bad arguments before touching
the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|void)\s+(moe_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import mxfp4_weight_mxfp8_gb300 as moe

    return moe


def test_header_declares_the_four_calls():
    names = declared_functions()
    for call in ("moe_prepare", "moe_quantize", "moe_group", "moe_run"):
        assert call in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.library()._name)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_library_is_built_for_sm103a_only(lib):
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_moe_build_check", os.path.join(ROOT, "mxfp4_weight_mxfp8_gb300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(lib.library()._name)


def test_small_batch_build_rules_without_a_gpu(lib):
    """Which build of the small-batch kernel a call gets, from host arithmetic alone
    (the shared-memory layouts of half an SM, the landing of an item's segment sums and
    the FC2 split over 152 CTAs)."""
    b = lib.moe_small_batch_build
    P, W, N = lib.SMALL_PACKED, lib.SMALL_WIDE, lib.SMALL_NONE
    # The TP8 and TP16 shards: one or two tokens packed, more wide.
    assert [b(384, 3584, 384, n) for n in (1, 2, 3, 8)] == [P, P, W, W]
    assert [b(384, 3584, 256, n) for n in (1, 2, 8)] == [P, P, W]
    # Widest layers at I = 512: packed up to H = 4096 (32 K chunks of 256-byte images),
    # wide up to 3328 (26 K chunks of 1 KB images).
    assert [b(16, 4096, 512, n) for n in (1, 2, 3)] == [P, P, N]
    assert b(16, 4352, 512, 1) == N
    assert [b(16, 3328, 512, n) for n in (3, 8)] == [W, W]
    assert b(16, 3584, 512, 8) == N
    assert b(16, 16384, 512, 1) == N
    # H = 256: two K chunks hold one token's segment sums in the packed layout's pad,
    # two tokens' only in the wide layout's full images.
    assert [b(32, 256, 64, n) for n in (1, 2, 3)] == [P, W, N]
    # Partial tiles (I = 96): the packed build at one token, the wide one up to four.
    assert [b(16, 512, 96, n) for n in (1, 2, 4, 5)] == [P, W, W, N]
    for bad in [(0, 3584, 384, 1), (384, 3600, 384, 1), (384, 3584, 40, 1), (384, 3584, 384, 0),
                (384, 3584, 384, 9)]:
        with pytest.raises(lib.MoeError):
            b(*bad)
    with pytest.raises(lib.MoeError):
        b(384, 3584, 384, 1, grid=300)


def test_device_support_check_without_a_gpu(lib):
    """moe_prepare's device check on faked properties: sm_103 with the
    kernel's shared memory is accepted; sm_100 (no sm_103a code), other
    majors and too little shared memory are refused."""
    ok = 232448  # cudaDeviceProp::sharedMemPerBlockOptin of a GB300
    assert lib.moe_device_supported(10, 3, ok) == lib.MOE_OK
    assert lib.moe_device_supported(10, 0, ok) == lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_device_supported(12, 0, ok) == lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_device_supported(9, 0, ok) == lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_device_supported(10, 3, 100 * 1024) == lib.MOE_ERR_UNSUPPORTED


def test_error_strings(lib):
    for code in range(7):
        assert lib.moe_error_string(code)
    assert lib.moe_error_string(99) == "unknown status"


def test_prepare_rejects_bad_arguments_before_any_cuda_call(lib):
    raw = lib.library()
    handle = ctypes.c_void_p(1234)
    fake = ctypes.c_void_p(0x1000)
    assert raw.moe_prepare(None, fake, fake, fake, fake, 32, 256, 64) == lib.MOE_ERR_ARG
    bad_sizes = [(0, 256, 64), (1025, 256, 64), (32, 255, 64), (32, 384, 64), (32, 256, 48),
                 (32, 256, 16), (32, 256, 544), (32, 16640, 64)]
    for experts, hidden, inter in bad_sizes:
        rc = raw.moe_prepare(ctypes.byref(handle), fake, fake, fake, fake, experts, hidden, inter)
        assert rc == lib.MOE_ERR_ARG, (experts, hidden, inter)
        assert handle.value is None
    assert raw.moe_prepare(ctypes.byref(handle), None, fake, fake, fake, 32, 256, 64) == lib.MOE_ERR_ARG


def test_calls_reject_null_handles_and_bad_batches(lib):
    raw = lib.library()
    p = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
    assert raw.moe_run(None, p, p, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_quantize(None, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_group(None, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_run_host(None, p, p, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_experts(None, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_run_noalloc(None, p, p, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_run_combined(None, p, p, p, p, 1, None) == lib.MOE_ERR_ARG
    assert raw.moe_sync_status(None, None) == lib.MOE_ERR_ARG
    assert raw.moe_copy_plan(None, p, p, 1) == lib.MOE_ERR_ARG
    assert raw.moe_copy_units(None, p, p, p, 1) == lib.MOE_ERR_ARG
    assert raw.moe_copy_hidden(None, p, p, 1) == lib.MOE_ERR_ARG
    assert raw.moe_set_timeout(None, 5) == lib.MOE_ERR_ARG
    assert raw.moe_debug_withhold(None, 0) == lib.MOE_ERR_ARG
    assert raw.moe_debug_paths(None, 1) == lib.MOE_ERR_ARG
    assert raw.moe_cluster_size(None, 1) == -lib.MOE_ERR_ARG
    info = lib.MoeInfo()
    assert raw.moe_info(None, ctypes.byref(info)) == lib.MOE_ERR_ARG
    raw.moe_destroy(None)  # no-op


def test_python_binding_names_match_the_c_abi(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_noalloc_scratch_limit_matches_the_header(lib):
    text = open(HEADER, encoding="utf-8").read()
    m = re.search(r"#define MOE_NOALLOC_SCRATCH_BYTES \((\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == lib.MOE_NOALLOC_SCRATCH_BYTES

"""GB300 (sm_103a) MXFP8-activation x MXFP4-weight top-16 MoE decode layer.

A thin ctypes binding over the C ABI declared in ``include/moe.h``: every
function here only marshals arguments (tensor or array -> pointer, torch
stream -> cudaStream_t) and raises ``MoeError`` on a non-zero status. All of
the layer's work runs in the library's CUDA kernels; there is no other path.
Importing fails loudly when the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIBRARY

__all__ = [
    "MoeError", "MoeInfo", "MoeLayer", "library", "moe_prepare", "moe_quantize", "moe_group",
    "moe_run", "moe_experts", "moe_run_noalloc", "moe_run_combined", "moe_run_host",
    "moe_sync_status", "moe_copy_plan", "moe_copy_units", "moe_copy_hidden", "moe_set_timeout",
    "moe_debug_withhold", "moe_debug_withhold_image", "moe_debug_paths", "moe_cluster_size", "moe_info",
    "moe_destroy", "moe_error_string",
    "MOE_OK", "MOE_ERR_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA", "MOE_ERR_DEVICE_TIMEOUT", "MOE_ERR_DEVICE_IDS",
    "MOE_ERR_STATE", "TOPK", "UNIT_ROWS", "MOE_NOALLOC_SCRATCH_BYTES", "moe_last_error_detail",
    "MAX_BATCH", "moe_device_supported", "moe_small_batch_build", "SMALL_NONE", "SMALL_PACKED", "SMALL_WIDE", "moe_debug_kernel_span", "moe_read_kernel_span",
    "moe_kernel_path", "PATH_GRID", "PATH_SMALL", "PATH_CLUSTER", "PATH_SMALL_WIDE",
]

MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_IDS, MOE_ERR_STATE = 4, 5, 6
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20  # static scratch of moe_run_noalloc
TOPK, UNIT_ROWS, MAX_BATCH = 16, 8, 256


class MoeInfo(ctypes.Structure):
    _fields_ = [("experts", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
                ("hidden_floor_rule", ctypes.c_int), ("grid", ctypes.c_int),
                ("ring_stages", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("stages_per_expert", ctypes.c_int), ("unit_capacity", ctypes.c_int),
                ("hidden_image_bytes", ctypes.c_int), ("weight_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load():
    if not os.path.exists(LIBRARY):
        raise ImportError(f"CUDA library not built ({LIBRARY} missing): run "
                          "`python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIBRARY)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    signatures = {
        "moe_prepare": ([ctypes.POINTER(vp), vp, vp, vp, vp, i32, i32, i32], i32),
        "moe_quantize": ([vp, vp, i32, vp], i32),
        "moe_group": ([vp, vp, i32, vp], i32),
        "moe_run": ([vp, vp, vp, vp, i32, vp], i32),
        "moe_experts": ([vp, vp, i32, vp], i32),
        "moe_run_noalloc": ([vp, vp, vp, vp, i32, vp], i32),
        "moe_run_combined": ([vp, vp, vp, vp, vp, i32, vp], i32),
        "moe_run_host": ([vp, vp, vp, vp, i32, vp], i32),
        "moe_sync_status": ([vp, vp], i32),
        "moe_copy_plan": ([vp, vp, vp, i32], i32),
        "moe_copy_units": ([vp, vp, vp, vp, i32], i32),
        "moe_copy_hidden": ([vp, vp, vp, i32], i32),
        "moe_set_timeout": ([vp, u64], i32),
        "moe_debug_withhold": ([vp, i32], i32),
        "moe_debug_withhold_image": ([vp, i32], i32),
        "moe_debug_paths": ([vp, i32], i32),
        "moe_cluster_size": ([vp, i32], i32),
        "moe_kernel_path": ([vp, i32], i32),
        "moe_info": ([vp, ctypes.POINTER(MoeInfo)], i32),
        "moe_destroy": ([vp], None),
        "moe_error_string": ([i32], ctypes.c_char_p),
        "moe_last_error_detail": ([], ctypes.c_char_p),
        "moe_device_supported": ([i32, i32, ctypes.c_size_t], i32),
        "moe_small_batch_build": ([i32, i32, i32, i32, i32], i32),
        "moe_debug_kernel_span": ([vp, i32], i32),
        "moe_read_kernel_span": ([vp, ctypes.POINTER(u64)], i32),
    }
    for name, (args, res) in signatures.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    return lib


_lib = _load()


def library():
    """The loaded ctypes library (its path is ``library()._name``)."""
    return _lib


class MoeError(RuntimeError):
    def __init__(self, code: int, call: str):
        detail = _lib.moe_last_error_detail().decode()
        text = _lib.moe_error_string(code).decode()
        super().__init__(f"{call}: {text} (status {code}){': ' + detail if detail else ''}")
        self.code = code


def moe_last_error_detail() -> str:
    """Detail of this thread's last argument or CUDA error ("" if none)."""
    return _lib.moe_last_error_detail().decode()


def _check(code: int, call: str) -> int:
    if code != MOE_OK:
        raise MoeError(code, call)
    return code


def _ptr(obj):
    """Address of a torch tensor, numpy array or raw integer pointer."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    if hasattr(obj, "ctypes"):
        return obj.ctypes.data
    raise TypeError(f"cannot take the address of {type(obj).__name__}")


def _stream(stream):
    """cudaStream_t of a torch stream / raw handle; default: torch's current stream."""
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def moe_prepare(w13, s13, w2, s2, experts: int, hidden: int, inter: int):
    """Handle (an int) of a prepared layer; see include/moe.h."""
    handle = ctypes.c_void_p()
    _check(_lib.moe_prepare(ctypes.byref(handle), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2),
                            experts, hidden, inter), "moe_prepare")
    return handle.value


def moe_quantize(handle, x, batch: int, stream=None):
    return _check(_lib.moe_quantize(handle, _ptr(x), batch, _stream(stream)), "moe_quantize")


def moe_group(handle, ids, batch: int, stream=None):
    return _check(_lib.moe_group(handle, _ptr(ids), batch, _stream(stream)), "moe_group")


def moe_run(handle, x, ids, out, batch: int, stream=None):
    return _check(_lib.moe_run(handle, _ptr(x), _ptr(ids), _ptr(out), batch, _stream(stream)),
                  "moe_run")


def moe_experts(handle, out, batch: int, stream=None):
    return _check(_lib.moe_experts(handle, _ptr(out), batch, _stream(stream)), "moe_experts")


def moe_run_combined(handle, x, ids, weights, out, batch: int, stream=None):
    """moe_run, then out[t] = bf16(sum_s weights[t, s] * row[t, s]) (out: [B, H])."""
    return _check(_lib.moe_run_combined(handle, _ptr(x), _ptr(ids), _ptr(weights), _ptr(out),
                                        batch, _stream(stream)), "moe_run_combined")


def moe_run_noalloc(handle, x, ids, out, batch: int, stream=None):
    """moe_run with all per-call scratch in the library's static device
    buffer (for callers that cannot allocate when they run the layer)."""
    return _check(_lib.moe_run_noalloc(handle, _ptr(x), _ptr(ids), _ptr(out), batch,
                                       _stream(stream)), "moe_run_noalloc")


def moe_run_host(handle, x, ids, out, batch: int, stream=None):
    return _check(_lib.moe_run_host(handle, _ptr(x), _ptr(ids), _ptr(out), batch,
                                    _stream(stream)), "moe_run_host")


def moe_sync_status(handle, stream=None) -> int:
    """Device status of the finished calls (not raised: tests inspect it)."""
    return _lib.moe_sync_status(handle, _stream(stream))


def moe_copy_plan(handle, codes, scales, batch: int):
    return _check(_lib.moe_copy_plan(handle, _ptr(codes), _ptr(scales), batch), "moe_copy_plan")


def moe_copy_units(handle, count, experts, rows, capacity: int):
    return _check(_lib.moe_copy_units(handle, _ptr(count), _ptr(experts), _ptr(rows), capacity),
                  "moe_copy_units")


def moe_copy_hidden(handle, codes, scales, units: int):
    return _check(_lib.moe_copy_hidden(handle, _ptr(codes), _ptr(scales), units),
                  "moe_copy_hidden")


def moe_set_timeout(handle, nanoseconds: int):
    return _check(_lib.moe_set_timeout(handle, nanoseconds), "moe_set_timeout")


def moe_debug_withhold(handle, unit: int):
    return _check(_lib.moe_debug_withhold(handle, unit), "moe_debug_withhold")


def moe_debug_withhold_image(handle, unit: int):
    return _check(_lib.moe_debug_withhold_image(handle, unit), "moe_debug_withhold_image")


PATH_GRID, PATH_SMALL, PATH_CLUSTER, PATH_SMALL_WIDE = 0, 1, 2, 3


def moe_debug_paths(handle, path: int):
    """0 grid kernel, 1 small-batch kernel for 1-2 tokens (default), 2 cluster variant,
    3 small-batch kernel for up to 8 tokens."""
    return _check(_lib.moe_debug_paths(handle, path), "moe_debug_paths")


def moe_kernel_path(handle, batch: int) -> int:
    """The experts kernel a call of `batch` tokens runs on (PATH_*)."""
    n = _lib.moe_kernel_path(handle, batch)
    if n < 0:
        raise MoeError(-n, "moe_kernel_path")
    return n


def moe_debug_kernel_span(handle, enable: int):
    return _check(_lib.moe_debug_kernel_span(handle, enable), "moe_debug_kernel_span")


def moe_read_kernel_span(handle):
    """Span (ns) of the last experts-kernel launch recorded by the launch clock."""
    span = ctypes.c_uint64()
    _check(_lib.moe_read_kernel_span(handle, ctypes.byref(span)), "moe_read_kernel_span")
    return span.value


def moe_cluster_size(handle, batch: int) -> int:
    """CTAs per cluster a call of `batch` tokens runs on (0: the grid kernel)."""
    n = _lib.moe_cluster_size(handle, batch)
    if n < 0:
        raise MoeError(-n, "moe_cluster_size")
    return n


def moe_info(handle) -> MoeInfo:
    info = MoeInfo()
    _check(_lib.moe_info(handle, ctypes.byref(info)), "moe_info")
    return info


def moe_destroy(handle):
    _lib.moe_destroy(handle)


SMALL_NONE, SMALL_PACKED, SMALL_WIDE = 0, 1, 2


def moe_small_batch_build(experts: int, hidden: int, inter: int, batch: int, grid: int = 152) -> int:
    """The small-batch kernel's build for such a call (SMALL_*); no GPU needed."""
    n = _lib.moe_small_batch_build(experts, hidden, inter, batch, grid)
    if n < 0:
        raise MoeError(-n, "moe_small_batch_build")
    return n


def moe_device_supported(cc_major: int, cc_minor: int, smem_per_block_optin: int) -> int:
    """MOE_OK if a device with these properties runs the library (sm_103 with
    enough shared memory per block), else MOE_ERR_UNSUPPORTED."""
    return _lib.moe_device_supported(cc_major, cc_minor, smem_per_block_optin)


def moe_error_string(code: int) -> str:
    return _lib.moe_error_string(code).decode()


class MoeLayer:
    """One prepared layer: owns a handle and allocates outputs with torch.

    ``weights`` = (w13, s13, w2, s2) uint8 tensors or arrays in the layout of
    include/moe.h (device or host). ``layer(x, ids)`` returns the BF16
    [B, 16, H] rows on x's device, on the current torch stream.
    """

    def __init__(self, weights):
        w13, s13, w2, s2 = weights
        experts, rows, half_hidden = (int(d) for d in w13.shape)
        self.experts, self.hidden, self.inter = experts, 2 * half_hidden, rows // 2
        self._keep = weights
        self.handle = moe_prepare(w13, s13, w2, s2, self.experts, self.hidden, self.inter)
        self._keep = None

    def __call__(self, x, ids, out=None, stream=None):
        import torch

        batch = int(x.shape[0])
        if out is None:
            out = torch.empty((batch, TOPK, self.hidden), dtype=torch.bfloat16, device=x.device)
        moe_run(self.handle, x, ids, out, batch, stream)
        return out

    def info(self) -> dict:
        return moe_info(self.handle).as_dict()

    def close(self):
        if self.handle:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

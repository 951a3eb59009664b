"""ctypes binding to libgma.so (include/gma.h).  Argument marshalling only:
every step of the computation runs in the library's CUDA kernels.  There is
no fallback: if the library is missing or a call fails, an exception is
raised."""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgma.so")

GMA_F32, GMA_BF16 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_TC, PATH_TC_SINGLE_PASS = 0, 1, 2, 3

STATUS_NAMES = {
    0: "GMA_OK", 1: "GMA_ERR_INVALID_ARG", 2: "GMA_ERR_UNSUPPORTED_SHAPE",
    3: "GMA_ERR_WORKSPACE_TOO_SMALL", 4: "GMA_ERR_CUDA", 5: "GMA_ERR_TIMEOUT",
    6: "GMA_ERR_NONFINITE_PARAM",
}

# Every symbol declared in include/gma.h (checked by the CPU test-suite).
EXPORTED = ("gma_workspace_size", "gma_responsibilities", "gma_forward_bidir",
            "gma_forward_causal", "gma_last_device_status", "gma_status_string",
            "gma_selected_path", "gma_stage_count", "gma_stage_name",
            "gma_forward_bidir_noalloc", "gma_backward_workspace_size", "gma_backward_bidir",
            "gma_backward_causal", "gma_latent_memory_workspace_size", "gma_latent_memory",
            "gma_decode_workspace_size", "gma_decode_step", "gma_routing_stats_workspace_size",
            "gma_routing_stats", "gma_read_memory_workspace_size", "gma_read_memory",
            "gma_causal_carry_workspace_size", "gma_forward_causal_carry", "gma_reparameterize",
            "gma_reparameterize_backward", "gma_project_workspace_size", "gma_project_qkv",
            "gma_combine_memories", "gma_tc_partition")


class Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("chunk", ctypes.c_int), ("splits", ctypes.c_int),
                ("sync_status", ctypes.c_int), ("o_bf16", ctypes.c_int),
                ("stage_events", ctypes.POINTER(ctypes.c_void_p)),
                ("n_stage_events", ctypes.c_int), ("test_stall", ctypes.c_int)]


class GmaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libgma.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with "
                               "`python -m gaussian_mixture_latent_diag_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        opt = ctypes.POINTER(Options)
        lib.gma_workspace_size.argtypes = [i, i, i, i, i, i, i, i, opt]
        lib.gma_workspace_size.restype = sz
        lib.gma_responsibilities.argtypes = [vp, i, vp, vp, vp, vp, i, i, i, i, i, opt, vp, sz, vp]
        lib.gma_responsibilities.restype = i
        fwd = [vp, vp, vp, i, vp, vp, vp, f, vp, i, i, i, i, i, i, opt, vp, sz, vp]
        lib.gma_forward_bidir.argtypes = fwd
        lib.gma_forward_bidir.restype = i
        lib.gma_forward_causal.argtypes = fwd
        lib.gma_forward_causal.restype = i
        lib.gma_forward_bidir_noalloc.argtypes = fwd[:16] + [vp]
        lib.gma_forward_bidir_noalloc.restype = i
        lib.gma_backward_workspace_size.argtypes = [i, i, i, i, i, i, i, i, opt]
        lib.gma_backward_workspace_size.restype = sz
        lib.gma_backward_bidir.argtypes = [vp, vp, vp, i, vp, vp, vp, f] + [vp] * 7 + [i] * 6 + [opt, vp, sz, vp]
        lib.gma_backward_bidir.restype = i
        lib.gma_backward_causal.argtypes = lib.gma_backward_bidir.argtypes
        lib.gma_backward_causal.restype = i
        lib.gma_latent_memory_workspace_size.argtypes = [i, i, i, i, i, i, i, opt]
        lib.gma_latent_memory_workspace_size.restype = sz
        lib.gma_latent_memory.argtypes = [vp, vp, i, vp, vp, vp, vp, vp] + [i] * 6 + [opt, vp, sz, vp]
        lib.gma_latent_memory.restype = i
        lib.gma_decode_workspace_size.argtypes = [i, i, i]
        lib.gma_decode_workspace_size.restype = sz
        lib.gma_decode_step.argtypes = [vp, vp, vp, i, vp, vp, vp, f, vp, vp, vp] + [i] * 5 + [opt, vp, sz, vp]
        lib.gma_decode_step.restype = i
        lib.gma_routing_stats_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.gma_routing_stats_workspace_size.restype = sz
        lib.gma_routing_stats.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp] + [i] * 5 + [opt, vp, sz, vp]
        lib.gma_routing_stats.restype = i
        lib.gma_read_memory_workspace_size.argtypes = [i, i, i, i, i, i, i]
        lib.gma_read_memory_workspace_size.restype = sz
        lib.gma_read_memory.argtypes = [vp, i, vp, vp, vp, f, vp, vp, vp] + [i] * 6 + [opt, vp, sz, vp]
        lib.gma_read_memory.restype = i
        lib.gma_causal_carry_workspace_size.argtypes = [i, i, i, i, i, i, i]
        lib.gma_causal_carry_workspace_size.restype = sz
        lib.gma_forward_causal_carry.argtypes = [vp, vp, vp, i, vp, vp, vp, f, vp, vp, vp, vp, vp] + [i] * 6 + \
            [opt, vp, sz, vp]
        lib.gma_forward_causal_carry.restype = i
        lib.gma_reparameterize.argtypes = [vp, vp, i, i, i, f, vp, vp, vp]
        lib.gma_reparameterize.restype = i
        lib.gma_reparameterize_backward.argtypes = [vp, vp, vp, vp, i, i, i, vp, vp, vp]
        lib.gma_reparameterize_backward.restype = i
        lib.gma_combine_memories.argtypes = [vp, i, ctypes.c_longlong, i, vp, vp]
        lib.gma_combine_memories.restype = i
        lib.gma_project_workspace_size.argtypes = []
        lib.gma_project_workspace_size.restype = sz
        lib.gma_project_qkv.argtypes = [vp] * 7 + [i] * 7 + [opt, vp, sz, vp]
        lib.gma_project_qkv.restype = i
        lib.gma_last_device_status.argtypes = [vp, vp]
        lib.gma_last_device_status.restype = i
        lib.gma_status_string.argtypes = [i]
        lib.gma_status_string.restype = ctypes.c_char_p
        lib.gma_selected_path.argtypes = [i, i, i, i, i, i, opt]
        lib.gma_selected_path.restype = i
        ip = ctypes.POINTER(ctypes.c_int)
        lib.gma_tc_partition.argtypes = [i, i, i, ip, i, ip]
        lib.gma_tc_partition.restype = i
        lib.gma_stage_count.argtypes = [i, i]
        lib.gma_stage_count.restype = i
        lib.gma_stage_name.argtypes = [i, i, i]
        lib.gma_stage_name.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().gma_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only when the library is absent
        return STATUS_NAMES.get(status, "unknown")


def options(path: int = PATH_AUTO, chunk: int = 0, splits: int = 0, sync_status: bool = False,
            o_bf16: bool = False, stage_events=None, test_stall: bool = False):
    """gma_options; `stage_events` is a list of torch.cuda.Event (or None);
    `test_stall` is the failure-path test hook (see include/gma.h)."""
    o = Options(int(path), int(chunk), int(splits), int(bool(sync_status)), int(bool(o_bf16)),
                None, 0, int(bool(test_stall)))
    if stage_events:
        for e in stage_events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record()
        arr = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
        o.stage_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        o.n_stage_events = len(stage_events)
        o._keep = arr  # keep the array alive as long as the options
    return o


def stage_names(path: int, variant: int) -> list:
    lib = load()
    return [lib.gma_stage_name(path, variant, j).decode() for j in range(lib.gma_stage_count(path, variant))]

"""Child process of tests/test_zz_no_alloc.py: calls gma_forward_bidir_noalloc
in three CUDA contexts in a row -- the device's primary context, a second
context created on the same device (driver API), and the primary context again
after the second one is destroyed -- and prints one JSON line with, per call,
the status, the normalised error against the fp64 oracle and whether O equals
gma_forward_bidir's O (same context, caller-provided workspace) bit for bit.

It runs in its own process and drives CUDA only through the driver API
(ctypes) and libgma.so, so the test process's torch state is never involved.
Usage: python noalloc_contexts.py"""
import ctypes
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402  (CPU tensors only: the inputs)

import oracle  # noqa: E402
from gaussian_mixture_latent_diag_gb300 import _native  # noqa: E402
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs  # noqa: E402

cu = ctypes.CDLL("libcuda.so.1")
u64 = ctypes.c_uint64


def ck(r, what):
    if r != 0:
        raise RuntimeError(f"{what} failed: CUresult {r}")


def host_bytes(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    return t.numpy()


class Buffers:
    """Device copies of the inputs, O for both entry points and a workspace,
    allocated with cuMemAlloc in the context current when created."""

    def __init__(self, lib, case, inp):
        self.ptrs = {}
        for name in ("Q", "K", "V", "mu", "sigma2", "log_pi"):
            a = np.ascontiguousarray(host_bytes(inp[name]))
            self.ptrs[name] = self._alloc(a.nbytes)
            ck(cu.cuMemcpyHtoD_v2(u64(self.ptrs[name]), a.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")
        self.o_bytes = 4 * case.B * case.H * case.N * case.d_v
        self.ptrs["O_noalloc"] = self._alloc(self.o_bytes)
        self.ptrs["O_ref"] = self._alloc(self.o_bytes)
        opt = _native.options()
        self.ws_bytes = lib.gma_workspace_size(case.B, case.H, case.N, case.d_r, case.d_v, case.K,
                                               _native.GMA_BF16, 0, ctypes.byref(opt))
        self.ptrs["ws"] = self._alloc(self.ws_bytes)

    def _alloc(self, n):
        p = u64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(n, 256))), "cuMemAlloc")
        return p.value

    def fetch(self, name, shape):
        out = np.empty(shape, dtype=np.float32)
        ck(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(ctypes.c_void_p), u64(self.ptrs[name]),
                              ctypes.c_size_t(out.nbytes)), "cuMemcpyDtoH")
        return out

    def free(self):
        for p in self.ptrs.values():
            ck(cu.cuMemFree_v2(u64(p)), "cuMemFree")


def one_context(lib, case, inp, ref):
    b = Buffers(lib, case, inp)
    vp = ctypes.c_void_p
    P = b.ptrs
    opt = _native.options(sync_status=True)
    args = (vp(P["Q"]), vp(P["K"]), vp(P["V"]), _native.GMA_BF16, vp(P["mu"]), vp(P["sigma2"]),
            vp(P["log_pi"]), ctypes.c_float(case.eps))
    dims = (case.B, case.H, case.N, case.d_r, case.d_v, case.K)
    st = lib.gma_forward_bidir_noalloc(*args, vp(P["O_noalloc"]), *dims, ctypes.byref(opt), None)
    st_ref = lib.gma_forward_bidir(*args, vp(P["O_ref"]), *dims, ctypes.byref(opt), vp(P["ws"]),
                                   ctypes.c_size_t(b.ws_bytes), None)
    shape = (case.B, case.H, case.N, case.d_v)
    O, O_ref = b.fetch("O_noalloc", shape), b.fetch("O_ref", shape)
    b.free()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return {"status": int(st), "status_ref": int(st_ref),
            "err": float(np.max(np.abs(O.astype(np.float64) - ref)) / rms),
            "same_as_bidir": bool(np.array_equal(O.view(np.uint32), O_ref.view(np.uint32)))}


def main():
    lib = _native.load()
    case = Case("noalloc_ctx", False, 1, 2, 700, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=21)
    ref = oracle.forward_bidir(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"],
                               case.eps)
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    calls = [one_context(lib, case, inp, ref)]
    second = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "cuCtxCreate")  # becomes current
    calls.append(one_context(lib, case, inp, ref))
    ck(cu.cuCtxDestroy_v2(second), "cuCtxDestroy")
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    calls.append(one_context(lib, case, inp, ref))
    ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
    print(json.dumps({"calls": calls}))


if __name__ == "__main__":
    main()

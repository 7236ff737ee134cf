"""Child process of tests/test_zz_no_alloc.py: the no-alloc fused call in
several CUDA contexts of one process.

The no-alloc call's scratch is a module variable, whose device address belongs
to the module as loaded into one context.  This script drives the library
through the CUDA driver API only (PyTorch's CUDA side is never initialised, so
no caching allocator holds memory across the resets) and checks, in each
context, that lp_linear_logprob_noalloc returns the bits of lp_linear_logprob
with a workspace:

  1. the device's primary context;
  2. a second context created on the same device (made current, then
     destroyed);
  3. the primary context again;
  4. the primary context after it was reset (what cudaDeviceReset does), with
     fresh allocations.

Prints one line per step and "ok" at the end; exits non-zero on a mismatch.
"""

from __future__ import annotations

import ctypes
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from invariant_token_logprobs_gb300 import lp, synth  # noqa: E402

cu = ctypes.CDLL("libcuda.so.1")
_u64 = ctypes.c_uint64


def ck(res, what):
    if res != 0:
        raise SystemExit(f"{what} failed: CUresult {res}")


def ctx_id() -> int:
    c = ctypes.c_void_p()
    ck(cu.cuCtxGetCurrent(ctypes.byref(c)), "cuCtxGetCurrent")
    i = ctypes.c_ulonglong()
    ck(cu.cuCtxGetId(c, ctypes.byref(i)), "cuCtxGetId")
    return i.value


class Buf:
    def __init__(self, nbytes: int):
        self.p = _u64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(self.p), ctypes.c_size_t(max(nbytes, 256))), "cuMemAlloc")
        self.n = nbytes

    def put(self, a: np.ndarray):
        a = np.ascontiguousarray(a)
        ck(cu.cuMemcpyHtoD_v2(self.p, a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)),
           "cuMemcpyHtoD")

    def get(self, dtype, count) -> np.ndarray:
        out = np.empty(count, dtype=dtype)
        ck(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(ctypes.c_void_p), self.p,
                              ctypes.c_size_t(out.nbytes)), "cuMemcpyDtoH")
        return out

    def free(self):
        cu.cuMemFree_v2(self.p)


def run_step(lib, label, h, w, y, T, d, V, expect=None):
    """Upload the inputs into the current context, run the workspace call and
    the no-alloc call, compare their bits; return the no-alloc logp bits."""
    bufs = [Buf(h.nbytes), Buf(w.nbytes), Buf(y.nbytes)]
    bufs[0].put(h)
    bufs[1].put(w)
    bufs[2].put(y)
    ws_bytes = lp.lp_linear_logprob_workspace_size(T, d, V)
    ws = Buf(ws_bytes)
    outs = [Buf(4 * T) for _ in range(4)]
    H, W, Y = (b.p.value for b in bufs)
    st = lib.lp_linear_logprob(H, d, W, d, Y, T, d, V, outs[0].p.value, outs[1].p.value,
                               ws.p.value, ws_bytes, None)
    ck(st, f"{label}: lp_linear_logprob")
    for _ in range(2):  # twice: the second call finds the scratch the first left behind
        st = lib.lp_linear_logprob_noalloc(H, d, W, d, Y, T, d, V, outs[2].p.value,
                                           outs[3].p.value, None)
        ck(st, f"{label}: lp_linear_logprob_noalloc")
        ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        r = [o.get(np.int32, T) for o in outs]
        if not (np.array_equal(r[0], r[2]) and np.array_equal(r[1], r[3])):
            raise SystemExit(f"{label}: no-alloc result differs from the workspace call")
    if expect is not None and not np.array_equal(expect, r[2]):
        raise SystemExit(f"{label}: result differs from the first context's")
    print(f"{label}: context id {ctx_id()}, no-alloc == workspace call, bit for bit", flush=True)
    for b in bufs + outs + [ws]:
        b.free()
    return r[2]


def main():
    lib = lp.load(build_if_needed=False)
    x = synth.fused_inputs("fused_tiny", device="cpu", T=96, d=256, V=8192 + 5, seed=31)
    T, d = x.H.shape
    V = x.W.shape[0]
    h = x.H.contiguous().view(torch.int16).numpy()  # raw bf16 bits
    w = x.W.contiguous().view(torch.int16).numpy()
    y = x.y.numpy()

    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    id1 = ctx_id()
    ref = run_step(lib, "primary context", h, w, y, T, d, V)

    other = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(other), 0, dev), "cuCtxCreate")
    id2 = ctx_id()
    assert id2 != id1
    run_step(lib, "second context", h, w, y, T, d, V, expect=ref)
    ck(cu.cuCtxDestroy_v2(other), "cuCtxDestroy")

    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    run_step(lib, "primary context again", h, w, y, T, d, V, expect=ref)

    ck(cu.cuDevicePrimaryCtxReset_v2(dev), "cuDevicePrimaryCtxReset")
    primary2 = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary2), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxSetCurrent(primary2), "cuCtxSetCurrent")
    id3 = ctx_id()
    print(f"primary context id before reset {id1}, after {id3}", flush=True)
    if id3 in (id1, id2):
        # the library caches the scratch address per context id: a reused id
        # would hand the kernels a stale address, so stop before any launch
        raise SystemExit("the reset primary context kept an old context id")
    run_step(lib, "primary context after reset", h, w, y, T, d, V, expect=ref)
    cu.cuDevicePrimaryCtxRelease_v2(dev)
    print("ok", flush=True)


if __name__ == "__main__":
    main()

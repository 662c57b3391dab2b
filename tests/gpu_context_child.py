"""Child process of tests/test_gpu_context.py: skv_topk_static and skv_topk in two CUDA
contexts of one device, alternating (the primary context and one created with the
driver API), each call on buffers allocated in its own context.  Prints OK on success;
exits non-zero with a message otherwise.  Uses the driver API through ctypes and no
torch CUDA state."""

import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from top_sparse_kv_gb300 import binding  # noqa: E402

cu = ctypes.CDLL("libcuda.so.1")


def ck(r, what):
    if r != 0:
        print(f"FAIL {what}: CUresult {r}")
        sys.exit(2)


class Buffers:
    """scores, idx and seq_lens of one problem, allocated in the current context."""

    def __init__(self, scores, lens, k):
        self.B, self.H, self.L = scores.shape
        self.k = k
        self.p = {}
        for name, nbytes in (("scores", scores.nbytes), ("idx", self.B * self.H * k * 4), ("lens", 4 * self.B)):
            ptr = ctypes.c_uint64(0)
            ck(cu.cuMemAlloc_v2(ctypes.byref(ptr), ctypes.c_size_t(nbytes)), "cuMemAlloc")
            self.p[name] = ptr.value
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(self.p["scores"]), ctypes.c_void_p(scores.ctypes.data),
                              ctypes.c_size_t(scores.nbytes)),
           "copy scores")
        lens = np.asarray(lens, dtype=np.int32)
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(self.p["lens"]), ctypes.c_void_p(lens.ctypes.data),
                              ctypes.c_size_t(lens.nbytes)),
           "copy lens")

    def problem(self):
        return binding.CProblem(self.B, self.H, self.H, 128, 128, 128, self.H, self.L, self.k, 4, 128, 16, 0, 0,
                                0.0, 0, self.p["lens"])

    def idx(self):
        out = np.empty((self.B, self.H, self.k), dtype=np.int32)
        ck(cu.cuCtxSynchronize(), "synchronize")
        ck(cu.cuMemcpyDtoH_v2(ctypes.c_void_p(out.ctypes.data), ctypes.c_uint64(self.p["idx"]),
                              ctypes.c_size_t(out.nbytes)),
           "copy idx")
        return out

    def free(self):
        for ptr in self.p.values():
            ck(cu.cuMemFree_v2(ctypes.c_uint64(ptr)), "cuMemFree")


def expect(scores, lens, k):
    B, H, _ = scores.shape
    out = np.full((B, H, k), -1, dtype=np.int32)
    for b in range(B):
        s_end, l_start = oracle.regions(int(lens[b]), 4, 128)
        pos = np.arange(s_end, l_start)
        for h in range(H):
            sel = oracle.exact_topk(scores[b, h, pos].astype(np.float64), pos, k)
            out[b, h, : len(sel)] = sel
    return out


def run_static(buf, lib):
    cp = buf.problem()
    st = ctypes.c_void_p(0)
    r = lib.skv_topk_static(ctypes.byref(cp), ctypes.c_void_p(buf.p["scores"]), ctypes.c_void_p(buf.p["idx"]), None,
                            st)
    if r != 0:
        print(f"FAIL skv_topk_static returned {r}")
        sys.exit(3)
    return buf.idx()


def main():
    lib = binding.lib()
    lib.skv_topk_static.restype = ctypes.c_int32
    for fn in (cu.cuInit, cu.cuDeviceGet, cu.cuDevicePrimaryCtxRetain, cu.cuCtxPushCurrent_v2, cu.cuCtxCreate_v2,
               cu.cuCtxPopCurrent_v2, cu.cuCtxDestroy_v2, cu.cuCtxSynchronize, cu.cuMemAlloc_v2, cu.cuMemFree_v2,
               cu.cuMemcpyHtoD_v2, cu.cuMemcpyDtoH_v2):
        fn.restype = ctypes.c_int
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p(0)
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "retain primary")
    ck(cu.cuCtxPushCurrent_v2(primary), "push primary")
    rng = np.random.default_rng(5)
    # long rows with large k: the multi-CTA passes keep their state in the fixed array
    B, H, L, k = 1, 2, 300000, 3000
    sa = (np.round(rng.standard_normal((B, H, L)) * 3) / 3).astype(np.float32)
    sb = (np.round(rng.standard_normal((B, H, L)) * 3) / 3).astype(np.float32)
    lens = [L]
    ea, eb = expect(sa, lens, k), expect(sb, lens, k)
    in_a = Buffers(sa, lens, k)
    np.testing.assert_array_equal(run_static(in_a, lib), ea)
    other = ctypes.c_void_p(0)
    ck(cu.cuCtxCreate_v2(ctypes.byref(other), 0, dev), "create context")  # now current
    in_b = Buffers(sb, lens, k)
    np.testing.assert_array_equal(run_static(in_b, lib), eb)
    ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p(0))), "pop created")  # the primary again
    np.testing.assert_array_equal(run_static(in_a, lib), ea)
    ck(cu.cuCtxPushCurrent_v2(other), "push created")
    np.testing.assert_array_equal(run_static(in_b, lib), eb)
    in_b.free()
    ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p(0))), "pop created")
    ck(cu.cuCtxDestroy_v2(other), "destroy created")
    np.testing.assert_array_equal(run_static(in_a, lib), ea)
    in_a.free()
    print("OK")


if __name__ == "__main__":
    main()

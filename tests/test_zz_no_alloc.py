"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(plugins of a framework that owns all device memory, deployments with a fixed
memory budget).  It runs with a static scratch array inside the library
instead of a workspace.

Called through the C ABI with ctypes, twice in a row:
  * against the regular fa_bwd on the same inputs: the same kernels in the same
    order on the same values, so the gradients must be identical bit for bit;
  * against the fp64 oracle at the backward's parity tolerance (max|err| / max|ref|
    <= 1e-2 fp16, 3e-2 bf16);
  * with the device's default memory pool watched (the pool fa_bwd's
    stream-ordered allocation draws from): its high-water mark must not move,
    while fa_bwd without a workspace, the control, does move it.
This file is collected last so that a run stopping at the first failure has run
every other test first."""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_io_aware_22_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_G = {"fp16": 1e-2, "bf16": 3e-2}
SCRATCH_BYTES = 16 << 20
CU_MEMPOOL_ATTR_USED_MEM_CURRENT = 7
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _lib():
    import exact_io_aware_22_gb300 as fa
    lib = fa.load_library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, ctypes.c_float, i, vp]
    lib.fa_bwd_noalloc.restype = i
    return fa, lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(lib, q, k, v, o, lse, do, B, H, N, d, causal, scale, dtype):
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                            B, H, N, d, int(causal), scale, 0 if dtype == "fp16" else 1, _stream())
    return st, (dq, dk, dv)


class _Pool:
    """The current device's default memory pool, read through the driver API."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def _get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        """Set the high-water mark back to the bytes in use now; return those bytes."""
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(zero)) == 0
        return self._get(CU_MEMPOOL_ATTR_USED_MEM_CURRENT)

    def high(self):
        return self._get(CU_MEMPOOL_ATTR_USED_MEM_HIGH)


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (2, 4, 1000, 64, "fp16", True),
    (1, 8, 2048, 128, "bf16", True),
    (2, 2, 777, 32, "bf16", False),
])
def test_noalloc_identical_to_bwd_twice(B, H, N, d, dtype, causal):
    fa, lib = _lib()
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, dtype, seed=11)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    ref = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    for call in range(2):
        st, got = _noalloc(lib, q, k, v, o, lse, do, B, H, N, d, causal, scale, dtype)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), (call, name)


def test_noalloc_matches_oracle_twice():
    import oracle
    fa, lib = _lib()
    B, H, N, d, dtype, causal = 2, 4, 1000, 64, "fp16", True
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, dtype, seed=23)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    xd = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    refs = oracle.bwd(xd["q"], xd["k"], xd["v"], xd["do"], causal, scale)[:3]
    for call in range(2):
        st, got = _noalloc(lib, q, k, v, o, lse, do, B, H, N, d, causal, scale, dtype)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, refs):
            gn = g.double().cpu().numpy()
            assert np.isfinite(gn).all(), (call, name)
            rel = float(np.max(np.abs(gn - r))) / float(np.max(np.abs(r)))
            assert rel <= TOL_G[dtype], (call, name, rel)


def test_noalloc_allocates_nothing():
    fa, lib = _lib()
    B, H, N, d, dtype, causal = 2, 8, 1536, 128, "bf16", True
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_inputs(B, H, N, d, dtype, seed=29)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    pool = _Pool()
    used = pool.reset_high()
    for call in range(2):
        st, _ = _noalloc(lib, q, k, v, o, lse, do, B, H, N, d, causal, scale, dtype)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
    assert pool.high() <= used, "fa_bwd_noalloc drew memory from the default pool"
    # control: the same probe sees fa_bwd's own stream-ordered workspace allocation
    used = pool.reset_high()
    fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert pool.high() >= used + fa.bwd_workspace_size(B, H, N, d, causal)
    assert fa.device_status() == 0


def test_noalloc_rejects_beyond_scratch():
    fa, lib = _lib()
    # 8 x 32 heads x 16384 rows need 8 bytes per row: 32 MiB > 16 MiB
    B, H, N, d = 8, 32, 16384, 64
    assert fa.bwd_workspace_size(B, H, N, d, True) > SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    st = lib.fa_bwd_noalloc(*([fake] * 9), B, H, N, d, 1, 0.125, 0, None)
    assert st == 2   # FA_ERR_UNSUPPORTED, before any launch

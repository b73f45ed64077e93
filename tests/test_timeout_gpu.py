"""The bounded-wait timeout path of the tensor-core forward, driven on the GPU
without a fault.

A test-only build of the library (libattn_waittest.so: the same sources, the
tensor-core forward compiled with ATTN_TEST_DROP_K_LOAD and a 20 ms wait
limit) skips one K-tile load in CTA 0.  The waits for that tile can then end
only by their time limit: the waiting role records ATTN_ERR_TIMEOUT with its
role flag in the device status word and raises the CTA's abort flag, the other
roles leave, the CTA waits (bounded) for its own copies and MMAs and frees its
TMEM, and the kernel returns.  The call must come back well within a second
with that status, and the normal library must work on the same device right
after it.  No fault, trap or endless wait is involved: every wait in the
kernel is bounded.
"""
import ctypes
import math
import time

import numpy as np
import pytest
import torch

import oracle
import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import build as pkg_build
from attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROLE_FLAGS = 0x100 | 0x200 | 0x400 | 0x800  # producer, MMA issuer, softmax, epilogue


@pytest.fixture(scope="module")
def waittest_lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    attn.status()
    lib = ctypes.CDLL(pkg_build.build_wait_test_library())
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.attn_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p, i, p]
    lib.attn_fwd.restype = i
    lib.attn_status.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
    lib.attn_status.restype = i
    return lib


@pytest.mark.parametrize("D, dtype", [(64, wl.F16), (128, wl.BF16)])
def test_dropped_load_times_out_and_reports(waittest_lib, D, dtype):
    B, Hq, Hkv, L = 1, 4, 2, 512
    dev = torch.device("cuda")
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=D + 5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(B * Hq, L, device=dev)
    sm = 1.0 / math.sqrt(D)
    code = ctypes.c_int(0)
    # twice: the first call on the device also loads the test library's
    # module; the second is timed
    for rep in range(2):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rc = waittest_lib.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, Hq, Hkv, L, D, sm, 1, None,
                                   wl.dtype_code(dtype), None)
        assert rc == attn.ATTN_OK  # queued: the timeout is a device-side condition
        st = waittest_lib.attn_status(None, ctypes.byref(code))
        elapsed = time.perf_counter() - t0
        assert st == 10, (st, hex(code.value))            # ATTN_ERR_TIMEOUT
        assert code.value & 1                              # a bounded wait gave up
        assert code.value & ROLE_FLAGS                     # ... and which role waited
        assert code.value & ~(ROLE_FLAGS | 1) == 0
    assert elapsed < 1.0, elapsed
    # read-and-clear in the test library too
    assert waittest_lib.attn_status(None, ctypes.byref(code)) == attn.ATTN_OK and code.value == 0

    # the device is fine: the normal library on the same inputs matches the oracle
    o2, lse2 = attn.attn_fwd(qd, kd, vd, causal=True, sm_scale=sm)
    assert attn.status() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype),
                                          sm, causal=True)
    o2 = o2.float().cpu().numpy()
    assert np.all(np.abs(o2 - o_ref) <= 2e-3 + 1e-2 * np.abs(o_ref))
    assert np.abs(lse2.cpu().numpy() - lse_ref).max() <= 1e-4

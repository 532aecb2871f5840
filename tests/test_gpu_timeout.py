"""The bounded-wait failure path of the decode kernel, on the GPU and without a
hang.  Every wait inside the kernels gives up after HSA_WAIT_NS of wall time,
flags HSA_DEVERR_TIMEOUT in dev_err and lets the kernel return.  A test-only
variant of the library is built into a temporary directory with a 2 ms limit and a
compile-time switch under which the decode producer issues no load at all: the
consumers then wait on stages nothing will ever fill.  The call must return, flag
the timeout, and leave the context usable (the product library's decode still
matches the oracle afterwards).  No TMA is ever issued in the test build, so
nothing can be in flight when its CTAs exit."""
import ctypes

import numpy as np
import pytest
import torch

import harness
import oracle
import workload

pytestmark = pytest.mark.gpu


def test_decode_wait_expiry_flags_timeout_and_returns(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    from full_attention_kv_gb300 import binding
    from full_attention_kv_gb300 import build as libbuild
    hsa.lib()
    path = libbuild.build(out_dir=str(tmp_path),
                          defines=("HSA_WAIT_NS=2000000ull", "HSA_TEST_WITHHOLD_LOADS"))
    T = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    T.hsa_decode_attn.restype = ctypes.c_int
    T.hsa_decode_attn.argtypes = [ctypes.POINTER(binding.HsaPools), i32, vp, vp, vp, vp, i32,
                                  i32, f32, vp, vp, sz, i32, vp, vp]
    inst = workload.draw(workload.CONFIGS["tiny"])
    cfg = inst.cfg
    layers = [6, 0]  # one full layer (split across CTAs), one sliding layer
    pool = harness.make_pool(inst, layers)
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        out = torch.zeros_like(q)
        ws = hsa.decode_workspace(pool, inst.R, cfg.T)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        s = T.hsa_decode_attn(pool.ref(), i, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              cl.data_ptr(), inst.R, cfg.T, cfg.scale, out.data_ptr(),
                              ws.data_ptr(), ws.numel(), 0, err.data_ptr(), None)
        assert s == hsa.HSA_OK
        torch.cuda.synchronize()  # returns: each wait gave up after 2 ms
        assert int(err.item()) & hsa.HSA_DEVERR_TIMEOUT, "layer %d: dev_err %d" % (l, err.item())
        assert torch.isfinite(out.float()).all()
    # the context is still usable: the product library's decode gives the oracle's result
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = hsa.hsa_decode_attn(pool, i, q, k, v, cl, cfg.scale, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle.attention(window=0 if inst.full[l] else cfg.W, scale=cfg.scale,
                               **harness.oracle_case(inst, l, range(inst.R)))
        assert np.max(np.abs(out.float().cpu().numpy().reshape(ref.shape) - ref)) <= 1e-2

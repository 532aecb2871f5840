"""hsa_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers cannot hand the library a workspace: code running while a stream is
captured into a CUDA graph (cudaMalloc is refused there), plug-ins inside a host
runtime that owns all device memory, and latency-critical loops that must never
wait on an allocation.  This entry point uses a fixed scratch array inside the
library instead.  The test calls it through the C ABI twice in a row (the array
keeps the previous call's contents, so the second call checks the reset) and
compares both outputs with hsa_decode_attn's, within the parity tolerance.

Kept in its own file so that pytest collects it last.
"""
import dataclasses

import pytest
import torch

import harness
import workload

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.mark.parametrize("T", [1, 4])
def test_noalloc_matches_workspace_entry_twice(T):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=T,
                              contexts=(9000, 0, 64, 130, 3000, 20000), B=6, index=90 + T)
    inst = workload.draw(cfg)
    layers = [6, 0]  # one full layer (split across CTAs, uses the counters), one sliding
    pool = harness.make_pool(inst, layers)
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        ref = hsa.hsa_decode_attn(pool, i, q, k, v, cl, cfg.scale)
        for call in range(2):
            out = torch.full_like(q, float("nan"))
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            hsa.hsa_decode_attn_noalloc(pool, i, q, k, v, cl, cfg.scale, out, dev_err=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            diff = torch.max(torch.abs(out.float() - ref.float())).item()
            assert diff <= TOL, "layer %d call %d: %g" % (l, call, diff)


def test_noalloc_caps_ctas_on_a_wide_sliding_layer():
    """64 sequences x 4 KV heads = 256 sliding-layer units: hsa_decode_attn gives each
    its own CTA, while the fixed scratch holds partial slots for about 250 CTAs, so
    the no-workspace call caps the grid and some rings are split across CTAs and
    merged through the scratch.  Both calls must agree, twice in a row."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    ctx = tuple((37 * b) % 300 for b in range(64))  # short contexts: 0 .. 299
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=1, contexts=ctx, B=64,
                              index=97)
    inst = workload.draw(cfg)
    layers = [0]
    pool = harness.make_pool(inst, layers)
    q, k, v, cl = harness.decode_inputs(inst, 0)
    ref = hsa.hsa_decode_attn(pool, 0, q, k, v, cl, cfg.scale)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        hsa.hsa_decode_attn_noalloc(pool, 0, q, k, v, cl, cfg.scale, out, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = torch.max(torch.abs(out.float() - ref.float())).item()
        assert diff <= TOL, "call %d: %g" % (call, diff)


def test_noalloc_rejects_too_many_units():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    inst = workload.draw(workload.CONFIGS["tiny"])
    pool = harness.make_pool(inst, [6])
    B = 2049  # x 2 KV heads > 4096 units
    q = torch.zeros((B, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((B, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    cl = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn_noalloc(pool, 0, q, kv, kv, cl, 0.1, torch.empty_like(q))
    assert e.value.status in (hsa.HSA_UNSUPPORTED_SHAPE, hsa.HSA_INVALID_ARG)

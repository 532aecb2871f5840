"""Layerwise SWA-KV prefetch from a pinned host tier (hsa_swa_prefetch): rows land
bit-exactly in the device ring, and decode after a prefetch matches the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import harness
import oracle
import workload

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    return hsa


def test_prefetch_rows_bit_exact():
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4,
                              contexts=(300, 40, 1000, 129, 77), B=5, index=110)
    inst = workload.draw(cfg)
    pool = harness.make_pool(inst, [0, 6])
    before = pool.k[0].clone(), pool.v[0].clone()
    n_host = 7
    hk = workload.randn_bf16((n_host, cfg.Hkv, cfg.W, cfg.d), 1, "cpu").pin_memory()
    hv = workload.randn_bf16((n_host, cfg.Hkv, cfg.W, cfg.d), 2, "cpu").pin_memory()
    host_row = torch.tensor([6, 0, 3], dtype=torch.int32, device="cuda")
    seq = torch.tensor([2, 4, 0], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hsa.hsa_swa_prefetch(pool, 0, hk, hv, host_row, seq, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rr = inst.ring_row
    for h, s in zip(host_row.tolist(), seq.tolist()):
        assert torch.equal(pool.k[0][rr[s]].cpu(), hk[h]) and torch.equal(pool.v[0][rr[s]].cpu(), hv[h])
    for s in (1, 3):  # untouched sequences keep their rings
        assert torch.equal(pool.k[0][rr[s]], before[0][rr[s]])
        assert torch.equal(pool.v[0][rr[s]], before[1][rr[s]])


def test_decode_after_prefetch_matches_oracle():
    """SWA KV offloaded to a host tier, device rings cleared, then prefetched."""
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=4,
                              contexts=(0, 5, 127, 128, 129, 700, 4000), B=7, index=111)
    inst = workload.draw(cfg)
    layers = [0, 6]
    pool = harness.make_pool(inst, layers)
    # host tier: row b = sequence b's ring, built by the oracle's own placement
    n = inst.R
    hk = np.zeros((n, cfg.Hkv, cfg.W, cfg.d), np.uint16)
    hv = hk.copy()
    for b in range(n):
        k, v, start = workload.history(inst, 0, b, "cuda")
        if k.shape[0]:
            oracle.append(hk, hv, [0, k.shape[0]], [b], [start], k, v,
                          ring_row=np.arange(n, dtype=np.int32))
    host_k = torch.from_numpy(hk.view(np.int16)).view(torch.bfloat16).pin_memory()
    host_v = torch.from_numpy(hv.view(np.int16)).view(torch.bfloat16).pin_memory()
    pool.k[0].zero_()
    pool.v[0].zero_()
    side = torch.cuda.Stream()
    rows = torch.arange(n, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(side):
        hsa.hsa_swa_prefetch(pool, 0, host_k, host_v, rows, rows)
    done = torch.cuda.Event()
    done.record(side)
    torch.cuda.current_stream().wait_event(done)
    q, k, v, cl = harness.decode_inputs(inst, 0)
    out = hsa.hsa_decode_attn(pool, 0, q, k, v, cl, cfg.scale)
    torch.cuda.synchronize()
    c = harness.oracle_case(inst, 0, range(n))
    ref = oracle.attention(window=cfg.W, scale=cfg.scale, **c)
    assert np.max(np.abs(out.float().cpu().numpy().reshape(ref.shape) - ref)) <= TOL


def test_prefetch_argument_errors():
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    pool = harness.make_pool(inst, [0, 6])
    cfg = inst.cfg
    hk = torch.zeros((2, cfg.Hkv, cfg.W, cfg.d), dtype=torch.bfloat16).pin_memory()
    rows = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_swa_prefetch(pool, 1, hk, hk, rows, rows)      # a full layer has no ring
    assert e.value.status == hsa.HSA_INVALID_ARG
    with pytest.raises(ValueError):
        hsa.hsa_swa_prefetch(pool, 0, torch.zeros_like(hk, device="cpu"), hk, rows, rows)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([5], dtype=torch.int32, device="cuda")  # host row past the tier
    hsa.hsa_swa_prefetch(pool, 0, hk, hk, bad, rows, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hsa.HSA_DEVERR_BAD_LEN

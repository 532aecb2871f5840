"""FP8 (E4M3 and E5M2) Full KV Pool variant for decode, through the C ABI.

Pools: the codes and scales the library writes (hsa_kv_append and the fused
append of hsa_decode_attn_append) equal the oracle's quantisation of the same
rows, bit for bit, read back through the documented layout (include/hsa.h).
Attention: decode / MTP verify over an FP8 full layer against the float64 oracle
over the dequantised history (oracle.attention_fp8hist), max-abs-error <= 1e-2;
the bf16 rounding bar of the bf16 path applies, since quantisation is part of
what both sides compute.
"""
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


def _perm16(l):
    return 4 * ((l % 8) // 2) + (l % 2) + 2 * (l // 8)


_IDX = {n: np.array([16 * (c // 16) + _perm16(c % 16) for c in range(n)]) for n in (64, 128)}


def _logical(pool, i):
    """(K codes, K scales, V codes, V scales), codes as [nb, Hkv, row, dim] numpy."""
    kc, ks, vc, vs = pool.fp8_views(i)
    kc = kc.cpu().numpy()[..., _IDX[128]]
    vc = vc.cpu().numpy()[..., _IDX[64]].transpose(0, 1, 3, 2)
    return kc, ks.cpu().numpy(), vc, vs.cpu().numpy()


def _gather(inst, arr, s, n):
    """Rows of positions 0 .. n-1 of sequence s from a [nb, Hkv, page, ...] array,
    each located by the oracle's placement."""
    at = [oracle.full_place(inst.block_tables, inst.num_blocks, inst.cfg.page, s, p)
          for p in range(n)]
    blk = np.array([b for b, _ in at], np.int64)
    off = np.array([o for _, o in at], np.int64)
    return arr[blk, :, off]


FORMATS = oracle.FP8_FORMATS


def _fp8_case(inst, layer, seqs, fmt):
    c = harness.oracle_case(inst, layer, seqs)
    hk, hks = oracle.quantize_fp8(c["hist_k"], fmt)
    hv, hvs = oracle.quantize_fp8(c["hist_v"], fmt)
    return dict(cu_rows=c["cu_rows"], prefix_len=c["prefix_len"], q=c["q"], k_new=c["k_new"],
                v_new=c["v_new"], hk=hk, hks=hks, hv=hv, hvs=hvs, hist_off=c["hist_off"],
                fmt=fmt)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("name,R", [("tiny", None), ("decode", 3)])
def test_fp8_append_bit_exact(name, R, fmt):
    _cuda()
    inst = workload.draw(workload.CONFIGS[name], R=R)
    full_layer = next(l for l in range(inst.cfg.n_layers) if inst.full[l])
    pool = harness.make_pool(inst, [full_layer], fp8=fmt)
    kc, ks, vc, vs = _logical(pool, 0)
    for s in range(inst.R):
        hk, hv, st = workload.history(inst, full_layer, s, "cuda")
        assert st == 0
        n = hk.shape[0]
        ek, eks = oracle.quantize_fp8(hk.cpu(), fmt)
        ev, evs = oracle.quantize_fp8(hv.cpu(), fmt)
        assert np.array_equal(_gather(inst, kc, s, n), ek), "K codes, seq %d" % s
        assert np.array_equal(_gather(inst, ks, s, n), eks), "K scales, seq %d" % s
        assert np.array_equal(_gather(inst, vc, s, n), ev), "V codes, seq %d" % s
        assert np.array_equal(_gather(inst, vs, s, n), evs), "V scales, seq %d" % s


@pytest.mark.parametrize("fmt", FORMATS)
def test_fp8_decode_parity_tiny_all_rows(fmt):
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    l = 6
    pool = harness.make_pool(inst, [l], fp8=fmt)
    q, k, v, cl = harness.decode_inputs(inst, l)
    out = hsa.hsa_decode_attn(pool, 0, q, k, v, cl, inst.cfg.scale)
    torch.cuda.synchronize()
    ref = oracle.attention_fp8hist(scale=inst.cfg.scale,
                                   **_fp8_case(inst, l, range(inst.R), fmt))
    got = out.view(-1, inst.cfg.Hq, inst.cfg.d).float().cpu().numpy()
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL, err


def _sampled(hsa, name, R=None, seed=0, fmt="e4m3"):
    cfg = workload.CONFIGS[name]
    inst = workload.draw(cfg, R=R)
    l = 6
    pool = harness.make_pool(inst, [l], fp8=fmt)
    B, T = inst.R, cfg.T
    q, k, v, cl = harness.decode_inputs(inst, l)
    ws = hsa.decode_workspace(pool, B, T)
    err_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = hsa.hsa_decode_attn_append(pool, 0, q, k, v, cl, cfg.scale, workspace=ws,
                                     dev_err=err_t)
    torch.cuda.synchronize()
    assert int(err_t.item()) == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(200 + cfg.index + seed)
    order = np.argsort(inst.prefix)
    seqs = sorted({int(order[0]), int(order[-1])} |
                  {int(x) for x in rng.choice(B, size=min(2, B), replace=False)})
    items = np.array([(s * T + t, int(h)) for s in seqs for t in range(T)
                      for h in rng.choice(cfg.Hq, size=4, replace=False)], np.int32)
    ref = oracle.attention_fp8hist(scale=cfg.scale, items=items,
                                   **_fp8_case(inst, l, seqs, fmt))
    got = out.view(B * T, cfg.Hq, cfg.d).float().cpu().numpy()[items[:, 0], items[:, 1]]
    e = float(np.max(np.abs(got - ref)))
    assert e <= TOL, "%s: max abs err %g" % (name, e)
    # the fused append quantised the new rows into the pool, bit-exact
    kc, ks, vc, vs = _logical(pool, 0)
    pg = cfg.page
    for s in seqs:
        ek, eks = oracle.quantize_fp8(k[s].cpu(), fmt)
        ev, evs = oracle.quantize_fp8(v[s].cpu(), fmt)
        for t in range(T):
            pos = int(inst.prefix[s]) + t
            blk = int(inst.block_tables[s, pos // pg])
            assert np.array_equal(kc[blk, :, pos % pg], ek[t])
            assert np.array_equal(ks[blk, :, pos % pg], eks[t])
            assert np.array_equal(vc[blk, :, pos % pg], ev[t])
            assert np.array_equal(vs[blk, :, pos % pg], evs[t])


@pytest.mark.parametrize("fmt", FORMATS)
def test_fp8_decode_full_size_sampled(fmt):
    _sampled(_cuda(), "decode", fmt=fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_fp8_mtp_verify_sampled(fmt):
    _sampled(_cuda(), "mtp", R=8, fmt=fmt)


def test_fp8_layers_are_decode_only():
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    pool = harness.make_pool(inst, [6], fp8=True)
    q, k, v, cu, pl, seq = harness.prefill_inputs(inst, 6)
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_prefill_attn(pool, 0, q, k, v, cu, pl, seq, 4, inst.cfg.scale)
    assert e.value.status == hsa.HSA_UNSUPPORTED_SHAPE
    # a sliding layer cannot be flagged FP8: the ring (newest W tokens) stays bf16
    z = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        hsa.DualPool([False], [z], [z], pool.block_tables, pool.ring_row, 16, kv_fp8=[True],
                     Hkv=2, d=128, num_blocks=1)
    both = harness.make_pool(inst, [0, 6], fp8=True)
    assert both.kv_fp8 == [False, True]
    both._fp8[0] = 1  # forge the flag past the binding: the library refuses too
    q, k, v, cl = harness.decode_inputs(inst, 0)
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn(both, 0, q, k, v, cl, inst.cfg.scale)
    assert e.value.status == hsa.HSA_UNSUPPORTED_SHAPE
    both._fp8[0] = 0
    both._fp8[1] = 3  # no such format
    q, k, v, cl = harness.decode_inputs(inst, 6)
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn(both, 1, q, k, v, cl, inst.cfg.scale)
    assert e.value.status == hsa.HSA_INVALID_ARG


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("T,heads,max_ctas", [(1, (16, 2), 0), (2, (16, 2), 0), (4, (16, 2), 0),
                                              (1, (16, 2), 3), (1, (8, 2), 0), (1, (8, 2), 5)])
def test_fp8_ragged_contexts(T, heads, max_ctas, fmt):
    """Empty, one-token, page-edge, partial-page and multi-page contexts with 1, 2
    and 4 new tokens on an FP8 full layer, every row against the oracle; the fused
    append's codes bit-exact.  T = 1 with at most 8 query heads a KV head runs the
    eight-warp loop: 8 and 4 heads (padding columns), units split across CTAs
    (max_ctas=0: one CTA per SM) and whole units, several a CTA (max_ctas=3, 5)."""
    import dataclasses
    hsa = _cuda()
    contexts = (0, 1, 63, 64, 65, 127, 200, 1000, 4097)
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], T=T, Hq=heads[0], Hkv=heads[1],
                              contexts=contexts, B=len(contexts), index=70 + T + heads[0])
    inst = workload.draw(cfg)
    l = 6
    pool = harness.make_pool(inst, [l], fp8=fmt)
    q, k, v, cl = harness.decode_inputs(inst, l)
    ws = hsa.decode_workspace(pool, inst.R, T)
    err_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = hsa.hsa_decode_attn_append(pool, 0, q, k, v, cl, cfg.scale, workspace=ws,
                                     max_ctas=max_ctas, dev_err=err_t)
    torch.cuda.synchronize()
    assert int(err_t.item()) == 0
    ref = oracle.attention_fp8hist(scale=cfg.scale, **_fp8_case(inst, l, range(inst.R), fmt))
    got = out.view(-1, cfg.Hq, cfg.d).float().cpu().numpy()
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL, "T=%d: %g" % (T, err)
    kc, ks, vc, vs = _logical(pool, 0)
    pg = cfg.page
    for s in range(inst.R):
        ek, eks = oracle.quantize_fp8(k[s].cpu(), fmt)
        ev, evs = oracle.quantize_fp8(v[s].cpu(), fmt)
        for t in range(T):
            pos = int(inst.prefix[s]) + t
            blk = int(inst.block_tables[s, pos // pg])
            assert np.array_equal(kc[blk, :, pos % pg], ek[t])
            assert np.array_equal(vc[blk, :, pos % pg], ev[t])
            assert np.array_equal(ks[blk, :, pos % pg], eks[t])
            assert np.array_equal(vs[blk, :, pos % pg], evs[t])

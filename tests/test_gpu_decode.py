"""GPU parity of KV append and decode / MTP-verify attention against the oracle.

Every case runs through the C ABI (the ctypes binding) on seeded inputs from
workload.py; the oracle gets the generator's tensors, never anything the CUDA
path wrote.  Bars: pools bit-exact; attention max-abs-error <= 1e-2 against the
float64 oracle (bf16 inputs, fp32 accumulation, unit-scale outputs).
"""
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


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _decode_all(hsa, inst, pool, layers, **kw):
    outs = []
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        outs.append(hsa.hsa_decode_attn(pool, i, q, k, v, cl, inst.cfg.scale, **kw))
    torch.cuda.synchronize()
    return outs


def _oracle_layer(inst, l, seqs=None):
    seqs = range(inst.R) if seqs is None else seqs
    c = harness.oracle_case(inst, l, seqs)
    W = 0 if inst.full[l] else inst.cfg.W
    return oracle.attention(window=W, scale=inst.cfg.scale, **c)


def test_append_pools_bit_exact_tiny():
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    layers = list(range(inst.cfg.n_layers))
    pool = harness.make_pool(inst, layers)
    cfg = inst.cfg
    for i, l in enumerate(layers):
        k0, v0 = workload.pool_init(inst, l, "cuda")
        ek, ev = _bits(k0).copy(), _bits(v0).copy()
        for s in range(inst.R):
            hk, hv, st = workload.history(inst, l, s, "cuda")
            kw = dict(block_tables=inst.block_tables) if inst.full[l] else dict(ring_row=inst.ring_row)
            bad = oracle.append(ek, ev, [0, hk.shape[0]], [s], [st], hk, hv, **kw)
            assert bad == 0
        assert np.array_equal(_bits(pool.k[i]), ek), "K pool of layer %d" % l
        assert np.array_equal(_bits(pool.v[i]), ev), "V pool of layer %d" % l
    # one decode token per sequence on top, then compare again
    for i, l in enumerate(layers):
        _, k, v = workload.new_tokens(inst, l, "cuda")
        ek, ev = _bits(pool.k[i]).copy(), _bits(pool.v[i]).copy()
        cu = torch.arange(inst.R + 1, dtype=torch.int32, device="cuda")
        seq = torch.arange(inst.R, dtype=torch.int32, device="cuda")
        pos = torch.from_numpy(inst.prefix).cuda()
        hsa.hsa_kv_append(pool, i, k, v, cu, seq, pos)
        torch.cuda.synchronize()
        kw = dict(block_tables=inst.block_tables) if inst.full[l] else dict(ring_row=inst.ring_row)
        oracle.append(ek, ev, np.arange(inst.R + 1), np.arange(inst.R), inst.prefix, k, v, **kw)
        assert np.array_equal(_bits(pool.k[i]), ek) and np.array_equal(_bits(pool.v[i]), ev)


def test_ring_append_longer_than_window_keeps_last_w():
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], contexts=(0, 0), B=2)
    inst = workload.draw(cfg)
    pool = harness.make_pool(inst, [0])
    ek, ev = _bits(pool.k[0]).copy(), _bits(pool.v[0]).copy()
    n = [300, 77]
    k = workload.randn_bf16((sum(n), cfg.Hkv, cfg.d), 5, "cuda")
    v = workload.randn_bf16((sum(n), cfg.Hkv, cfg.d), 6, "cuda")
    cu = torch.tensor([0, n[0], sum(n)], dtype=torch.int32, device="cuda")
    seq = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, 1000], dtype=torch.int32, device="cuda")
    hsa.hsa_kv_append(pool, 0, k, v, cu, seq, pos)
    torch.cuda.synchronize()
    oracle.append(ek, ev, [0, n[0], sum(n)], [1, 0], [5, 1000], k, v, ring_row=inst.ring_row)
    assert np.array_equal(_bits(pool.k[0]), ek) and np.array_equal(_bits(pool.v[0]), ev)


def test_decode_tiny_all_layers():
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    layers = list(range(inst.cfg.n_layers))
    pool = harness.make_pool(inst, layers)
    outs = _decode_all(hsa, inst, pool, layers)
    for i, l in enumerate(layers):
        ref = _oracle_layer(inst, l)
        got = outs[i].float().cpu().numpy().reshape(ref.shape)
        err = np.max(np.abs(got - ref))
        assert err <= TOL, "layer %d (%s): max abs err %g" % (l, "full" if inst.full[l] else "swa", err)


CONTEXTS = (0, 1, 63, 64, 65, 127, 128, 129, 200, 1000, 4097)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("heads", [(32, 4), (16, 4)])
def test_decode_ragged_contexts_and_mtp(T, heads):
    hsa = _cuda()
    Hq, Hkv = heads
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=Hq, Hkv=Hkv, T=T,
                              contexts=CONTEXTS, B=len(CONTEXTS), index=50 + T)
    inst = workload.draw(cfg)
    layers = [6, 0]  # one full, one sliding
    pool = harness.make_pool(inst, layers)
    outs = _decode_all(hsa, inst, pool, layers)
    for i, l in enumerate(layers):
        ref = _oracle_layer(inst, l)
        got = outs[i].float().cpu().numpy().reshape(ref.shape)
        err = np.max(np.abs(got - ref))
        assert err <= TOL, "T=%d heads=%s layer %d: err %g" % (T, heads, l, err)


RING_T1_CONTEXTS = (0, 1, 63, 64, 100, 127, 128, 129, 191, 192, 193, 255, 256, 257, 1000, 4097)


@pytest.mark.parametrize("heads", [(16, 2), (8, 2)])
@pytest.mark.parametrize("max_ctas", [0, 40])
def test_ring_t1_whole_units(heads, max_ctas):
    """Sliding layer at T = 1 with whole (sequence, KV head) units per CTA: 96
    sequences x 2 KV heads is enough units for one CTA each (max_ctas=0), or several
    whole units and a split one per CTA (max_ctas=40).  Full rings (c >= W) take the
    path with the new token written over the slot its query no longer sees; the
    contexts put that slot at the start, middle and end of both 64-key tiles, and
    mix in rings not yet full.  8 query heads per KV head, and 4 (padding columns).
    Attention against the oracle; the fused append's rings bit-exact."""
    hsa = _cuda()
    Hq, Hkv = heads
    ctx = tuple(RING_T1_CONTEXTS[i % len(RING_T1_CONTEXTS)] + 128 * (i // len(RING_T1_CONTEXTS))
                for i in range(96))
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=Hq, Hkv=Hkv, T=1, contexts=ctx,
                              B=len(ctx), index=90 + Hq)
    inst = workload.draw(cfg)
    pool = harness.make_pool(inst, [0])
    q, k, v, cl = harness.decode_inputs(inst, 0)
    ref = _oracle_layer(inst, 0)
    out = hsa.hsa_decode_attn(pool, 0, q, k, v, cl, cfg.scale, max_ctas=max_ctas)
    torch.cuda.synchronize()
    err = np.max(np.abs(out.float().cpu().numpy().reshape(ref.shape) - ref))
    assert err <= TOL, "heads=%s max_ctas=%d: err %g" % (heads, max_ctas, err)
    ek, ev = _bits(pool.k[0]).copy(), _bits(pool.v[0]).copy()
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2 = hsa.hsa_decode_attn_append(pool, 0, q, k, v, cl, cfg.scale, max_ctas=max_ctas,
                                      dev_err=dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0
    assert torch.equal(out2, out)
    B = inst.R
    oracle.append(ek, ev, np.arange(B + 1), np.arange(B), inst.prefix,
                  k.view(B, Hkv, cfg.d), v.view(B, Hkv, cfg.d), ring_row=inst.ring_row)
    assert np.array_equal(_bits(pool.k[0]), ek) and np.array_equal(_bits(pool.v[0]), ev)


def test_split_count_and_page_permutation_invariance():
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=4,
                              contexts=(3000, 70, 0, 9000, 129), B=5, index=60)
    inst = workload.draw(cfg)
    layers = [6, 0]
    pool = harness.make_pool(inst, layers)
    base = _decode_all(hsa, inst, pool, layers)
    for mc in (1, 2, 5, 13):
        outs = _decode_all(hsa, inst, pool, layers, max_ctas=mc)
        for a, b in zip(base, outs):
            assert torch.max(torch.abs(a.float() - b.float())).item() <= TOL
    # same logical contents under another physical page permutation: identical bits
    inst2 = workload.draw(cfg, rng_seed=12345)
    inst2.prefix[:] = inst.prefix
    pool2 = harness.make_pool(inst2, layers)
    outs2 = _decode_all(hsa, inst2, pool2, layers)
    for a, b in zip(base, outs2):
        assert torch.equal(a, b)


def test_device_range_errors_flagged_not_trapped():
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], contexts=(500, 300), B=2, index=61)
    inst = workload.draw(cfg)
    pool = harness.make_pool(inst, [6, 0])
    good = _decode_all(hsa, inst, pool, [6, 0])
    bad_bt = pool.block_tables.clone()
    bad_bt[1, 2] = inst.num_blocks + 7         # sequence 1, page 2: outside the pool
    pool.block_tables.copy_(bad_bt)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, cl = harness.decode_inputs(inst, 6)
    out = hsa.hsa_decode_attn(pool, 0, q, k, v, cl, cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hsa.HSA_DEVERR_BAD_BLOCK
    assert torch.equal(out[0], good[0][0])     # the other sequence is untouched
    # append through the bad entry is skipped and flagged as well
    err.zero_()
    kk = torch.zeros((1, cfg.Hkv, cfg.d), dtype=torch.bfloat16, device="cuda")
    hsa.hsa_kv_append(pool, 0, kk, kk, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                      torch.tensor([1], dtype=torch.int32, device="cuda"),
                      torch.tensor([130], dtype=torch.int32, device="cuda"), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hsa.HSA_DEVERR_BAD_BLOCK
    # a ring row outside the ring
    err.zero_()
    pool.ring_row[0] = inst.n_ring_rows + 3
    q, k, v, cl = harness.decode_inputs(inst, 0)
    hsa.hsa_decode_attn(pool, 1, q, k, v, cl, cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & hsa.HSA_DEVERR_BAD_RING


def test_host_argument_errors():
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["tiny"])
    pool = harness.make_pool(inst, [6])
    q, k, v, cl = harness.decode_inputs(inst, 6)
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn(pool, 3, q, k, v, cl, 0.1)            # layer out of range
    assert e.value.status == hsa.HSA_INVALID_ARG
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn(pool, 0, q, k, v, cl, 0.1, workspace=ws)  # workspace too small
    assert e.value.status == hsa.HSA_INVALID_ARG
    q5 = torch.zeros((4, 5, 16, 128), dtype=torch.bfloat16, device="cuda")
    k5 = torch.zeros((4, 5, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_decode_attn(pool, 0, q5, k5, k5, cl, 0.1)         # G*T > 32
    assert e.value.status == hsa.HSA_UNSUPPORTED_SHAPE


def test_window_safe_len_matches_oracle_bit_exact():
    hsa = _cuda()
    W = 128
    match, slots, (idx, bm_len, off, live) = workload.window_cases(1000, W, seed=1004)
    got = hsa.hsa_window_safe_len(torch.from_numpy(match).cuda(), torch.from_numpy(slots).cuda(), W)
    ref = oracle.window_safe_len_ring(match, slots, W)
    assert np.array_equal(got.cpu().numpy(), ref)
    got_b = hsa.hsa_window_safe_len_bitmap(torch.from_numpy(bm_len).cuda(),
                                           torch.from_numpy(off).cuda(),
                                           torch.from_numpy(live).cuda(), W)
    ref_b = oracle.window_safe_len_bitmap(bm_len, off, live, W)
    assert np.array_equal(got_b.cpu().numpy(), ref_b)


@pytest.mark.parametrize("W", [3, 4, 31, 32, 33, 64])
def test_window_safe_len_small_windows(W):
    hsa = _cuda()
    match, slots, (idx, bm_len, off, live) = workload.window_cases(400, W, seed=W, m_hi=300)
    got = hsa.hsa_window_safe_len(torch.from_numpy(match).cuda(), torch.from_numpy(slots).cuda(), W)
    assert np.array_equal(got.cpu().numpy(), oracle.window_safe_len_ring(match, slots, W))
    got_b = hsa.hsa_window_safe_len_bitmap(torch.from_numpy(bm_len).cuda(),
                                           torch.from_numpy(off).cuda(),
                                           torch.from_numpy(live).cuda(), W)
    assert np.array_equal(got_b.cpu().numpy(), oracle.window_safe_len_bitmap(bm_len, off, live, W))


@pytest.mark.parametrize("T", [1, 4])
@pytest.mark.parametrize("max_ctas", [0, 3])
def test_fused_append_matches_attention_then_append(T, max_ctas):
    """hsa_decode_attn_append = hsa_decode_attn + appending the T new rows.

    max_ctas=3 splits units across CTAs, so the append of a ring whose unit is
    split is done by the last CTA to finish it (T = 4 would clobber live slots
    if any CTA were still reading)."""
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=T,
                              contexts=(0, 1, 63, 130, 700, 5000), B=6, index=70 + T)
    inst = workload.draw(cfg)
    layers = [6, 0]
    pool = harness.make_pool(inst, layers)
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        ref = hsa.hsa_decode_attn(pool, i, q, k, v, cl, cfg.scale, max_ctas=max_ctas)
        ek, ev = _bits(pool.k[i]).copy(), _bits(pool.v[i]).copy()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = hsa.hsa_decode_attn_append(pool, i, q, k, v, cl, cfg.scale, max_ctas=max_ctas,
                                         dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, ref)
        kw = dict(block_tables=inst.block_tables) if inst.full[l] else dict(ring_row=inst.ring_row)
        B = inst.R
        oracle.append(ek, ev, np.arange(0, B * T + 1, T), np.arange(B), inst.prefix,
                      k.view(B * T, cfg.Hkv, cfg.d), v.view(B * T, cfg.Hkv, cfg.d), **kw)
        assert np.array_equal(_bits(pool.k[i]), ek) and np.array_equal(_bits(pool.v[i]), ev)
        # and the attention it computed is the oracle's
        c = harness.oracle_case(inst, l, range(B))
        refo = oracle.attention(window=0 if inst.full[l] else cfg.W, scale=cfg.scale, **c)
        assert np.max(np.abs(out.float().cpu().numpy().reshape(refo.shape) - refo)) <= TOL


def _extended_case(inst, layer, k1, v1, q2, k2, v2, T):
    """Oracle inputs for a second decode step on `layer`: the history of every
    sequence extended by the T rows (k1, v1) the first step appended, and the second
    step's new rows.  Histories come from the generator, never from a pool."""
    c = harness.oracle_case(inst, layer, range(inst.R))
    B = inst.R
    hk, hv, off = [], [], [0]
    for s in range(B):
        a, b = int(c["hist_off"][s]), int(c["hist_off"][s + 1])
        hk.append(torch.cat([c["hist_k"][a:b], k1[s].cpu()]))
        hv.append(torch.cat([c["hist_v"][a:b], v1[s].cpu()]))
        off.append(off[-1] + hk[-1].shape[0])
    return dict(cu_rows=c["cu_rows"], prefix_len=inst.prefix + T,
                q=q2.reshape(B * T, inst.cfg.Hq, inst.cfg.d).cpu(),
                k_new=k2.reshape(B * T, inst.cfg.Hkv, inst.cfg.d).cpu(),
                v_new=v2.reshape(B * T, inst.cfg.Hkv, inst.cfg.d).cpu(),
                hist_k=torch.cat(hk), hist_v=torch.cat(hv), hist_off=np.array(off, np.int64),
                hist_start=c["hist_start"])


@pytest.mark.parametrize("T", [1, 2, 4])
def test_early_pool_read_equals_plain_and_ordering_holds(T):
    """HSA_DECODE_EARLY_POOL_READ on sliding layers.

    (1) Queued right after a fused decode + append on another sliding layer (a
    kernel that signals its dependents early and writes that layer's ring), the
    early decode of layer B gives bit for bit the result of B's decode without the
    option.  (2) The hazard the option must not be used for, checked without it: a
    fused decode + append on layer A, then at once A's next decode step (cached
    length + T) -- the second call must see the rows the first just wrote (the
    oracle's history includes them)."""
    hsa = _cuda()
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=T,
                              contexts=(0, 1, 63, 126, 127, 128, 700, 5000, 130, 255),
                              B=10, index=60 + T)
    inst = workload.draw(cfg)
    layers = [0, 1]  # both sliding
    pool = harness.make_pool(inst, layers)
    qa, ka, va, cl = harness.decode_inputs(inst, 0)
    qb, kb, vb, _ = harness.decode_inputs(inst, 1)
    ref_b = hsa.hsa_decode_attn(pool, 1, qb, kb, vb, cl, cfg.scale)
    torch.cuda.synchronize()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        # (1) ring A written just before; B read early
        hsa.hsa_decode_attn_append(pool, 0, qa, ka, va, cl, cfg.scale, dev_err=err)
        out_b = hsa.hsa_decode_attn(pool, 1, qb, kb, vb, cl, cfg.scale, dev_err=err,
                                    early_pool_read=True)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out_b, ref_b)
    # (2) A's ring now holds the appended rows at c .. c+T-1; the next step on A,
    # queued right behind a fused append on A, without the option
    pool2 = harness.make_pool(inst, layers)
    q2, k2, v2, _ = harness.decode_inputs(inst, 1)  # stand-ins for the next step's rows
    hsa.hsa_decode_attn_append(pool2, 0, qa, ka, va, cl, cfg.scale, dev_err=err)
    out2 = hsa.hsa_decode_attn(pool2, 0, q2, k2, v2, cl + T, cfg.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref2 = oracle.attention(window=cfg.W, scale=cfg.scale,
                            **_extended_case(inst, 0, ka, va, q2, k2, v2, T))
    got = out2.float().cpu().numpy().reshape(ref2.shape)
    assert np.max(np.abs(got - ref2)) <= TOL

"""GPU parity of chunked prefill on a cached prefix (tcgen05 kernel) against
the oracle, through the C ABI.  Bar: max-abs-error <= 1e-2 against float64."""
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


def _cfg(prefixes, chunks, Hq=32, Hkv=4, index=80):
    return workload.Config("prefill-case", index, "prefill", 7, Hq, Hkv, prefixes=tuple(prefixes),
                           chunks=tuple(chunks))


def _run(hsa, inst, layers, pool=None):
    pool = pool or harness.make_pool(inst, layers)
    outs = []
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i, l in enumerate(layers):
        q, k, v, cu, pl, seq = harness.prefill_inputs(inst, l)
        outs.append(hsa.hsa_prefill_attn(pool, i, q, k, v, cu, pl, seq, int(inst.new.max()),
                                         inst.cfg.scale, dev_err=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error bits %d" % int(err.item())
    return pool, outs


def _where(inst, got, ref):
    """Where the largest error sits: request, chunk row, head, dim, both values and
    the number of keys that row attends (for a failure message)."""
    idx = np.unravel_index(int(np.argmax(np.abs(got - ref))), got.shape)
    row = int(idx[0])
    r = int(np.searchsorted(inst.cu_new, row, side="right")) - 1
    i = row - int(inst.cu_new[r])
    return ("request %d (prefix %d, chunk %d) row %d head %d dim %d: got %.5f ref %.5f" %
            (r, int(inst.prefix[r]), int(inst.new[r]), i, int(idx[1]), int(idx[2]),
             float(got[idx]), float(ref[idx])))


def _check(inst, layers, outs, seqs=None):
    for i, l in enumerate(layers):
        c = harness.oracle_case(inst, l, range(inst.R) if seqs is None else seqs)
        ref = oracle.attention(window=0 if inst.full[l] else inst.cfg.W, scale=inst.cfg.scale, **c)
        got = outs[i].float().cpu().numpy()
        err = float(np.max(np.abs(got - ref)))
        assert err <= TOL, "layer %d (%s): max abs err %g at %s" % (
            l, "full" if inst.full[l] else "swa", err, _where(inst, got, ref))


@pytest.mark.parametrize("heads", [(32, 4), (16, 2)])
def test_prefill_ragged_small(heads):
    hsa = _cuda()
    inst = workload.draw(_cfg([0, 100, 300, 64, 1000], [1, 130, 257, 128, 70], *heads))
    layers = [6, 0]
    _, outs = _run(hsa, inst, layers)
    _check(inst, layers, outs)


@pytest.mark.parametrize("W,heads", [(128, (32, 4)), (64, (32, 4)), (64, (16, 4)), (64, (8, 4)),
                                     (128, (16, 4)), (256, (32, 4))])
def test_prefill_sliding_windows_and_groups(W, heads):
    """Sliding layers over windows W = 64 / 128 / 256 and GQA groups G = 8 / 4 / 2:
    prefixes shorter than, equal to and longer than W (ring partly filled, exactly
    full, wrapped; lengths on and off 16-row boundaries), chunks whose rows cross
    i = W - 1 (the last row that still sees the prefix) and end on ragged tiles."""
    hsa = _cuda()
    cfg = dataclasses.replace(
        _cfg([0, 1, 17, W - 1, W, W + 1, 1007, 1008], [300, 2 * W + 3, 40, 129, W, 16, 17, 1],
             *heads, index=84), W=W)
    inst = workload.draw(cfg)
    layers = [0, 6]
    _, outs = _run(hsa, inst, layers)
    _check(inst, layers, outs)


def test_prefill_sliding_many_tiles_per_cta():
    """Three requests of 2.5K-5K rows (about 17 sliding-kernel tiles per CTA, across
    request boundaries; one request without a prefix): every barrier phase of the
    persistent kernel's pipeline wraps several times.  Sampled rows at the window and
    tile edges of every request against the oracle, and no device error."""
    hsa = _cuda()
    cfg = _cfg([20000, 300, 0], [3000, 5000, 2500], index=85)
    inst = workload.draw(cfg)
    layers = [0]
    _, outs = _run(hsa, inst, layers)
    rows = []
    for r in range(inst.R):
        a, b = int(inst.cu_new[r]), int(inst.cu_new[r + 1])
        rows += [a + i for i in (0, 1, 15, 16, 127, 128, 129, 1500, b - a - 17, b - a - 1)]
    items = np.array([(ri, h) for ri in rows for h in (0, 7, 8, 31)], np.int32)
    c = harness.oracle_case(inst, 0, range(inst.R))
    ref = oracle.attention(window=cfg.W, scale=cfg.scale, items=items, **c)
    got = outs[0].float().cpu().numpy()[items[:, 0], items[:, 1]]
    assert float(np.max(np.abs(got - ref))) <= TOL


def test_prefill_multi_tile_prefix_and_chunk():
    hsa = _cuda()
    inst = workload.draw(_cfg([5000, 12345], [700, 1029], index=81))
    layers = [6, 0]
    _, outs = _run(hsa, inst, layers)
    _check(inst, layers, outs)


def test_prefill_then_append_matches_oracle_pools():
    """The prefill flow: attention on the cached prefix, then append the chunk."""
    hsa = _cuda()
    inst = workload.draw(_cfg([200, 0, 777], [300, 129, 64], index=82))
    layers = [6, 0]
    pool, outs = _run(hsa, inst, layers)
    _check(inst, layers, outs)
    for i, l in enumerate(layers):
        ek, ev = _bits(pool.k[i]).copy(), _bits(pool.v[i]).copy()
        q, k, v, cu, pl, seq = harness.prefill_inputs(inst, l)
        hsa.hsa_kv_append(pool, i, k, v, cu, seq, pl)
        torch.cuda.synchronize()
        kw = dict(block_tables=inst.block_tables) if inst.full[l] else dict(ring_row=inst.ring_row)
        oracle.append(ek, ev, inst.cu_new, np.arange(inst.R), inst.prefix, k, v, **kw)
        assert np.array_equal(_bits(pool.k[i]), ek) and np.array_equal(_bits(pool.v[i]), ev)


def test_prefill_equals_decode_for_single_rows():
    """A one-row chunk is a decode step: the two kernels agree within tolerance."""
    hsa = _cuda()
    ctx = (63, 64, 129, 3000)
    inst = workload.draw(_cfg(ctx, [1] * len(ctx), index=83))
    dcfg = dataclasses.replace(workload.CONFIGS["tiny"], Hq=32, Hkv=4, T=1, contexts=ctx,
                               B=len(ctx), index=83)
    dinst = workload.draw(dcfg)
    layers = [6, 0]
    pool, outs = _run(hsa, inst, layers)
    for i, l in enumerate(layers):
        q, k, v, cu, pl, seq = harness.prefill_inputs(inst, l)
        B = inst.R
        d = hsa.hsa_decode_attn(pool, i, q.view(B, 1, 32, 128), k.view(B, 1, 4, 128),
                                v.view(B, 1, 4, 128), pl, inst.cfg.scale)
        torch.cuda.synchronize()
        assert torch.max(torch.abs(d.view_as(outs[i]).float() - outs[i].float())).item() <= TOL
    assert dinst.R == inst.R


def test_prefill_full_size_sampled():
    """8 requests, prefix 16K-128K, chunk 2K-8K (one full and one sliding layer):
    every request's rows 0, 127, 128, 255, 256 and its last row (the window and tile
    edges) plus seeded random rows, a few query heads each, against the oracle."""
    hsa = _cuda()
    inst = workload.draw(workload.CONFIGS["prefill"])
    layers = [6, 0]
    _, outs = _run(hsa, inst, layers)
    rng = np.random.default_rng(2024)
    for i, l in enumerate(layers):
        seqs = list(range(inst.R))
        rows = []
        for s in seqs:
            a, b = int(inst.cu_new[s]), int(inst.cu_new[s + 1])
            rows += [a, a + 127, a + 128, a + 255, a + 256, b - 1] + rng.integers(a, b, 4).tolist()
        items = np.array([(r, int(h)) for r in rows for h in rng.integers(0, inst.cfg.Hq, 2)],
                         np.int32)
        c = harness.oracle_case(inst, l, seqs)
        ref = oracle.attention(window=0 if inst.full[l] else inst.cfg.W, scale=inst.cfg.scale,
                               items=items, **c)
        got = outs[i].float().cpu().numpy()[items[:, 0], items[:, 1]]
        err = float(np.max(np.abs(got - ref)))
        assert err <= TOL, "layer %d: max abs err %g" % (l, err)
        assert torch.isfinite(outs[i].float()).all()

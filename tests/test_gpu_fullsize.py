"""Full-size parity for the decode workloads, in the launch configuration the
benchmark times (hsa_decode_attn_append, default CTA count), on one full and one
sliding layer: sampled (sequence, token, head) outputs against the float64
oracle, plus properties that hold at any size (finite outputs, appended rows
equal to the new tokens).  Bar: max-abs-error <= 1e-2.
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


def _sample_seqs(inst, rng, k=2):
    order = np.argsort(inst.prefix)
    picks = {int(order[0]), int(order[-1])}
    picks.update(int(x) for x in rng.choice(inst.R, size=min(k, inst.R), replace=False))
    return sorted(picks)


@pytest.mark.parametrize("name", ["decode", "long", "mtp"])
def test_decode_full_size_sampled(name):
    hsa = _cuda()
    cfg = workload.CONFIGS[name]
    inst = workload.draw(cfg)
    layers = [6, 0]  # one full layer, one sliding layer
    pool = harness.make_pool(inst, layers, stale="zero")
    rng = np.random.default_rng(100 + cfg.index)
    B, T = inst.R, cfg.T
    ws = hsa.decode_workspace(pool, B, T)
    for i, l in enumerate(layers):
        q, k, v, cl = harness.decode_inputs(inst, l)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = hsa.hsa_decode_attn_append(pool, i, q, k, v, cl, cfg.scale, workspace=ws,
                                         dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.isfinite(out.float()).all()
        seqs = _sample_seqs(inst, rng)
        items = []
        for s in seqs:
            for t in range(T):
                for h in rng.choice(cfg.Hq, size=4, replace=False):
                    items.append((s * T + t, int(h)))
        items = np.array(items, np.int32)
        c = harness.oracle_case(inst, l, seqs)
        ref = oracle.attention(window=0 if inst.full[l] else cfg.W, scale=cfg.scale,
                               items=items, **c)
        got = out.view(B * T, cfg.Hq, cfg.d).float().cpu().numpy()[items[:, 0], items[:, 1]]
        e = float(np.max(np.abs(got - ref)))
        assert e <= TOL, "%s layer %d: max abs err %g" % (name, l, e)
        # the appended rows hold the new tokens (position c + t of every sequence)
        for s in seqs:
            for t in range(T):
                pos = int(inst.prefix[s]) + t
                if inst.full[l]:
                    blk, off = oracle.full_place(inst.block_tables, inst.num_blocks, cfg.page,
                                                 s, pos)
                    row_k = pool.k[i][blk, :, off]
                else:
                    row, slot = oracle.ring_place(inst.ring_row, inst.n_ring_rows, cfg.W, s, pos)
                    row_k = pool.k[i][row, :, slot]
                assert torch.equal(row_k, k[s, t])

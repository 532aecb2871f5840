"""On-device batched window-safe matching through the prefix tree: the host tree
matches a batch of requests, one GPU launch (hsa_window_safe_len, ring form) gives
every request's window-safe length; compared exactly with the float-free oracle
(brute-force model + oracle.window_safe_len_ring).  W = 128 as on the pages."""
import random

import numpy as np
import pytest
import torch

import oracle
from oracle.prefix_model import PrefixModel, ring_positions

pytestmark = pytest.mark.gpu

W = 128


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    return hsa


@pytest.mark.parametrize("seed", [5, 6])
def test_batched_window_safe_matches_oracle(seed):
    hsa = _cuda()
    rng = random.Random(seed)
    tree, model = hsa.PrefixTree(W, 512), PrefixModel(W)
    paths, slot = [], 1
    rows = list(range(512))
    for _ in range(200):
        if paths and rng.random() < 0.7:
            base = rng.choice(paths)
            toks = base[:rng.randint(0, len(base))] + \
                [rng.randint(0, 3) for _ in range(rng.randint(1, 3 * W))]
        else:
            toks = [rng.randint(0, 3) for _ in range(rng.randint(1, 5 * W))]
        full = list(range(slot, slot + len(toks)))
        slot += len(toks)
        row = rows.pop() if rows and rng.random() < 0.9 else -1
        pos = None
        if row >= 0:
            freed = [s for s in range(W) if rng.random() < 0.02]
            pos = ring_positions(len(toks), W, freed)
        _, kept = tree.insert(toks, full, row, pos)
        _, ekept = model.insert(toks, full, row, pos)
        assert kept == ekept
        if row >= 0 and not kept:
            rows.append(row)
        paths.append(toks)
    model.drop_rows(tree.evict_swa(40))  # SWA evicted independently of the Full index
    reqs = []
    for _ in range(1000):  # follow-ups, branches, exact repeats, strangers
        base = rng.choice(paths)
        u = rng.random()
        if u < 0.4:
            reqs.append(base + [rng.randint(0, 3) for _ in range(rng.randint(1, 64))])
        elif u < 0.7:
            reqs.append(base[:rng.randint(0, len(base))] + [9])
        elif u < 0.9:
            reqs.append(list(base))
        else:
            reqs.append([rng.randint(10, 12) for _ in range(rng.randint(0, 40))])
    got = tree.window_safe(reqs)
    m = np.zeros(len(reqs), np.int32)
    pos = np.full((len(reqs), W), -1, np.int32)
    for k, r in enumerate(reqs):
        em, _, _, epos = model.match(r)
        m[k] = em
        pos[k] = epos
    want = oracle.window_safe_len_ring(m, pos, W)
    assert np.array_equal(got.numpy(), want)
    # the cases the rule is for are all present
    assert (want == m).sum() > 100          # full hits (follow-up turns)
    assert ((want < m) & (m > 0)).sum() > 50  # cut back to the window boundary

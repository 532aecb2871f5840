"""Prefix tree (include/hsa_tree.h) against the brute-force model in oracle/.

Host code only (no GPU): match, insert, take, lock and both eviction policies, on
seeded multi-turn workloads.  The model knows no tree; matches are compared
exactly (match length, Full slots, ring row, slot positions, duplicate slots,
ring kept), evictions through what is unique (the freed slots, mirrored into the
model) and invariants (locked paths survive, only least-recently-used leaves go).
"""
import random

import pytest
import torch

import oracle
from oracle.prefix_model import PrefixModel, ring_positions

W = 8  # small window: paths are a few windows long, so every case is reachable


def _tree(W=W, rows=64):
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    return hsa.PrefixTree(W, rows)


def _same_match(tree, model, seqs):
    m, r, pos = tree.match_batch(seqs)
    for k, s in enumerate(seqs):
        em, eslots, er, epos = model.match(s)
        assert int(m[k]) == em, (k, s)
        assert int(r[k]) == er, (k, s)
        assert [int(x) for x in pos[k]] == epos, (k, s)
    for s in seqs[:8]:  # single match also returns the Full slots
        mm, slots, rr, pp, h = tree.match(s)
        em, eslots, er, epos = model.match(s)
        assert (mm, [int(x) for x in slots], rr) == (em, eslots, er)
        assert h == -1


class Workload:
    """Seeded conversations: each turn extends a cached path or branches off it."""

    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.next_slot = 1000
        self.free_rows = list(range(64))
        self.paths = []

    def new_slots(self, n):
        s = list(range(self.next_slot, self.next_slot + n))
        self.next_slot += n
        return s

    def request(self):
        rng = self.rng
        if self.paths and rng.random() < 0.75:
            base = list(rng.choice(self.paths))
            cut = rng.randint(0, len(base)) if rng.random() < 0.4 else len(base)
            toks = base[:cut] + [rng.randint(0, 5) for _ in range(rng.randint(1, 3 * W))]
        else:
            toks = [rng.randint(0, 5) for _ in range(rng.randint(1, 4 * W))]
        return toks


def _finish(tree, model, wl, toks, reuse):
    """A request over `toks` ends: it reused the cached Full slots of its match
    (unless `reuse` is False: then it wrote its own copies) and leaves a ring row
    with its last window (some slots freed at random)."""
    m, slots, _, _, _ = tree.match(toks)
    mine = [int(x) for x in slots] if reuse else wl.new_slots(m)
    full = mine + wl.new_slots(len(toks) - m)
    row = wl.free_rows.pop() if wl.free_rows else -1
    pos = None
    if row >= 0:
        freed = [s for s in range(W) if wl.rng.random() < 0.1]
        pos = ring_positions(len(toks), W, freed)
    dup, kept = tree.insert(toks, full, row, pos)
    edup, ekept = model.insert(toks, full, row, pos)
    assert sorted(int(x) for x in dup) == sorted(edup)
    assert kept == ekept
    if row >= 0 and not kept:
        wl.free_rows.append(row)
    wl.paths.append(toks)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_matches_model_through_inserts(seed):
    tree, model, wl = _tree(), PrefixModel(W), Workload(seed)
    for step in range(120):
        toks = wl.request()
        _finish(tree, model, wl, toks, reuse=wl.rng.random() < 0.7)
        if step % 10 == 9:
            probes = [wl.request() for _ in range(24)] + wl.paths[-6:] + [[], [9, 9]]
            _same_match(tree, model, probes)
    c, rows, _ = tree.stats()
    assert c == model.cached_tokens()
    assert rows == len(model.rows_held())


def test_take_ring_moves_ownership():
    tree, model, wl = _tree(), PrefixModel(W), Workload(7)
    for _ in range(40):
        _finish(tree, model, wl, wl.request(), reuse=True)
    for toks in wl.paths[-10:]:
        m, slots, row, pos, _ = tree.match(toks, take_ring=True)
        em, _, er, epos = model.match(toks)
        assert (m, row, [int(x) for x in pos]) == (em, er, epos)
        if row >= 0:
            model.take_ring(row)
        _same_match(tree, model, wl.paths[-12:])


def test_window_safe_cases_from_the_pages():
    """A follow-up turn that extends the cached path hits with L = m; a turn that
    branches before the cached end sees a ring written past its match: L < W."""
    tree = _tree(W=8)
    toks = list(range(20))
    tree.insert(toks, list(range(100, 120)), 3, ring_positions(20, 8))
    m, r, pos = tree.match_batch([toks + [50, 51], toks[:15] + [77]])
    assert [int(x) for x in m] == [20, 15]
    assert [int(x) for x in r] == [3, 3]
    L = oracle.window_safe_len_ring(m.numpy(), pos.numpy(), 8)
    assert int(L[0]) == 20          # all of [12, 20) live
    assert int(L[1]) < 8            # ring holds 12..19, match ends at 15
    # a ring with a freed slot inside the window gives a shorter safe length
    tree2 = _tree(W=8)
    tree2.insert(toks, list(range(100, 120)), 4, ring_positions(20, 8, freed=[17 % 8]))
    m2, _, pos2 = tree2.match_batch([toks])
    assert int(oracle.window_safe_len_ring(m2.numpy(), pos2.numpy(), 8)[0]) < 20


def test_evict_full_frees_lru_leaves_and_keeps_locks():
    tree, model, wl = _tree(), PrefixModel(W), Workload(11)
    for _ in range(60):
        _finish(tree, model, wl, wl.request(), reuse=True)
    locked = wl.paths[5]
    m0, slots0, _, _, handle = tree.match(locked, lock=True)
    assert handle > 0
    before, _, _ = tree.stats()
    freed, rows = tree.evict_full(before)  # ask for everything
    after, _, _ = tree.stats()
    assert before - after == len(freed)
    assert len(set(int(x) for x in freed)) == len(freed)
    # the locked path is intact; everything else unlocked is gone
    m1, slots1, _, _, _ = tree.match(locked)
    assert m1 == m0 and [int(x) for x in slots1] == [int(x) for x in slots0]
    assert after == m0
    model.drop_slots(freed)
    model.drop_rows(rows)
    _same_match(tree, model, wl.paths[-20:])
    tree.unlock(handle)
    freed2, _ = tree.evict_full(1 << 30)
    assert tree.stats()[0] == 0 and len(freed2) == m0


def test_evict_full_order_is_lru():
    tree = _tree()
    a, b, c = [1, 2, 3, 4], [1, 2, 7, 8], [5, 6]
    tree.insert(a, [10, 11, 12, 13])
    tree.insert(b, [10, 11, 22, 23])
    tree.insert(c, [30, 31])
    tree.match(a)                      # a is now the most recent
    freed, _ = tree.evict_full(1)
    assert sorted(int(x) for x in freed) == [22, 23]   # b's leaf (oldest)
    freed, _ = tree.evict_full(1)
    assert sorted(int(x) for x in freed) == [30, 31]   # then c
    freed, _ = tree.evict_full(1)
    assert sorted(int(x) for x in freed) == [12, 13]   # then a's leaf, then the shared part
    freed, _ = tree.evict_full(1)
    assert sorted(int(x) for x in freed) == [10, 11]


def test_evict_swa_is_independent_of_full():
    tree, model, wl = _tree(), PrefixModel(W), Workload(13)
    for _ in range(30):
        _finish(tree, model, wl, wl.request(), reuse=True)
    c0, r0, _ = tree.stats()
    rows = tree.evict_swa(r0 // 2)
    c1, r1, _ = tree.stats()
    assert c1 == c0 and r1 == r0 - len(rows) and len(rows) == r0 // 2
    model.drop_rows(rows)
    _same_match(tree, model, wl.paths)
    # SWA pool occupancy is one window per cached path end at most
    assert r1 <= len(wl.paths)


def test_locked_rows_are_not_evicted():
    tree = _tree()
    tree.insert([1, 2, 3], [5, 6, 7], 9, ring_positions(3, W))
    _, _, row, _, h = tree.match([1, 2, 3], lock=True)
    assert row == 9
    assert len(tree.evict_swa(4)) == 0
    tree.unlock(h)
    assert [int(x) for x in tree.evict_swa(4)] == [9]


def test_invalid_arguments():
    import full_attention_kv_gb300 as hsa
    tree = _tree()
    with pytest.raises(hsa.HsaError):
        tree.unlock(12345)
    with pytest.raises(hsa.HsaError):
        tree.insert([1, 2], [3, 4], ring_row=999, swa_slot_pos=[0] * W)
    tree.insert([1, 2], [3, 4])
    _, _, _, _, h = tree.match([1, 2], lock=True)
    tree.unlock(h)
    with pytest.raises(hsa.HsaError):
        tree.unlock(h)  # already released
    L = hsa.lib()
    assert L.hsa_ptree_create(0, 4, None) == hsa.HSA_INVALID_ARG


@pytest.mark.parametrize("seed", [21, 22, 23, 24])
def test_interleaved_operations_match_model(seed):
    """Inserts, locked matches, unlocks, ring hand-overs and both evictions in a
    random interleaving; after every few operations each probe's match (length,
    ring row, slot positions, Full slots) equals the model's, and every locked path
    is still cached with the slots it had when it was locked."""
    tree, model, wl = _tree(), PrefixModel(W), Workload(seed)
    rng = wl.rng
    held = []  # (handle, tokens, m, slots) of live locks
    for step in range(300):
        u = rng.random()
        if u < 0.45 or not wl.paths:
            _finish(tree, model, wl, wl.request(), reuse=rng.random() < 0.7)
        elif u < 0.6:
            toks = list(rng.choice(wl.paths))[:rng.randint(1, 3 * W)]
            m, slots, _, _, h = tree.match(toks, lock=True)
            if h > 0:
                held.append((h, toks, m, [int(x) for x in slots]))
        elif u < 0.7 and held:
            h, _, _, _ = held.pop(rng.randrange(len(held)))
            tree.unlock(h)
        elif u < 0.8:
            toks = rng.choice(wl.paths)
            _, _, row, _, _ = tree.match(toks, take_ring=True)
            if row >= 0:
                model.take_ring(row)
                wl.free_rows.append(row)
        elif u < 0.92:
            freed, rows = tree.evict_full(rng.randint(1, 4 * W))
            model.drop_slots(freed)
            model.drop_rows(rows)
            wl.free_rows.extend(int(r) for r in rows)
        else:
            rows = tree.evict_swa(rng.randint(1, 4))
            model.drop_rows(rows)
            wl.free_rows.extend(int(r) for r in rows)
        if step % 5 == 4:
            probes = [wl.request() for _ in range(12)] + wl.paths[-4:] + [[]]
            _same_match(tree, model, probes)
            c, rows_held, _ = tree.stats()
            assert c == model.cached_tokens()
            assert rows_held == len(model.rows_held())
            for _, toks, m0, slots0 in held:
                m, slots, _, _, _ = tree.match(toks)
                assert m >= m0 and [int(x) for x in slots[:m0]] == slots0
    for h, _, _, _ in held:
        tree.unlock(h)
    freed, rows = tree.evict_full(1 << 30)
    assert tree.stats()[:2] == (0, 0)


def test_evict_full_reports_a_buffer_too_small():
    import full_attention_kv_gb300 as hsa
    tree = _tree()
    tree.insert([7], [20])                   # least recently used
    tree.insert([1, 2, 3, 4], [10, 11, 12, 13])
    freed, _ = tree.evict_full(10, slot_cap=3)  # [7] fits, then the four-slot leaf does not
    assert [int(x) for x in freed] == [20] and tree.stats()[0] == 4
    with pytest.raises(hsa.HsaError) as e:
        tree.evict_full(1, slot_cap=3)       # the first leaf already does not fit
    assert e.value.status == hsa.HSA_OUT_OF_RANGE
    assert tree.stats()[0] == 4              # nothing changed


def test_ring_choice_scales_with_shared_prefixes():
    """Thousands of cached paths below one shared system prompt: a batch of
    requests matching up to the shared end each gets the preferred row (shortest
    path, then latest attached) without walking the subtree."""
    W_ = 128
    tree = _tree(W=W_, rows=4096)
    system = list(range(1000, 1000 + 2 * W_))
    for i in range(3000):
        toks = system + [i % 50, i] + [7] * (i % 5)
        tree.insert(toks, list(range(len(toks))), i, ring_positions(len(toks), W_))
    reqs = [system + [99999, k] for k in range(2000)]
    m, rows, pos = tree.match_batch(reqs)
    # shortest cached paths through the prompt end have 2 extra tokens (i % 5 == 0);
    # among them the latest attached row wins
    want = max(i for i in range(3000) if i % 5 == 0)
    assert all(int(x) == len(system) for x in m)
    assert all(int(r) == want for r in rows)
    assert list(pos[0]) == ring_positions(len(system) + 2, W_)


def test_evict_full_default_buffers_fit_any_leaf():
    """A leaf longer than any fixed buffer (a 1M-token context is one leaf) is
    evicted by the default call: the binding sizes its buffers from the tree."""
    tree = _tree()
    n = (1 << 20) + 5
    tree.insert(list(range(n)), list(range(n)))
    freed, rows = tree.evict_full(1)
    assert len(freed) == n and tree.stats()[0] == 0


def test_token_arrays_are_checked_not_wrapped():
    """Token ids past the int32 range and two-dimensional token arrays are refused
    by the binding before they reach the C ABI (a silent wrap would match the wrong
    prefix)."""
    tree = _tree()
    with pytest.raises(ValueError):
        tree.match(torch.tensor([1, 2 ** 31], dtype=torch.int64))
    with pytest.raises(ValueError):
        tree.match_batch([torch.tensor([5, -(2 ** 31) - 1], dtype=torch.int64)])
    with pytest.raises(ValueError):
        tree.match(torch.ones((2, 3), dtype=torch.int32))
    with pytest.raises(ValueError):
        tree.match([1.5, 2.0])
    m, _, _ = tree.match_batch([torch.tensor([7, 2 ** 31 - 1], dtype=torch.int64), []])
    assert m.tolist() == [0, 0]

"""Pins of the CPU oracle against facts it does not compute itself.

Each test is chosen so that a plausible slip in the oracle (a dropped scale, a
window off by one, a wrong GQA head, a leaked future token, a wrong ring slot,
a window-safe scan that stops early) fails at least one of them:

* torch's float64 scaled_dot_product_attention with an explicit boolean mask (an
  independent library routine) on tiny inputs;
* closed forms: q = 0 gives the plain mean of the visible V rows; two keys give a
  logistic weight; SWA equals full attention while the sequence fits the window;
* planted values just inside / just outside the window and in future rows;
* placement bijectivity and ring-slot reuse properties;
* an independent closed form of the window-safe length, hand-derived cases, and
  the KV-byte ratio the pages print (about 1/7).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _case(rng, prefixes, rows, Hq, Hkv, d, hist_from=None):
    """Random tiny attention case with full histories."""
    R = len(prefixes)
    cu = np.zeros(R + 1, np.int32)
    cu[1:] = np.cumsum(rows)
    n = int(cu[-1])
    q = _bf16(rng.standard_normal((n, Hq, d)))
    kn = _bf16(rng.standard_normal((n, Hkv, d)))
    vn = _bf16(rng.standard_normal((n, Hkv, d)))
    starts = [0 if hist_from is None else hist_from[r] for r in range(R)]
    lens = [prefixes[r] - starts[r] for r in range(R)]
    ho = np.zeros(R + 1, np.int64)
    ho[1:] = np.cumsum(lens)
    hk = _bf16(rng.standard_normal((int(ho[-1]), Hkv, d)))
    hv = _bf16(rng.standard_normal((int(ho[-1]), Hkv, d)))
    return dict(cu_rows=cu, prefix_len=np.array(prefixes, np.int32), q=q, k_new=kn,
                v_new=vn, hist_k=hk, hist_v=hv, hist_off=ho,
                hist_start=np.array(starts, np.int32))


def _sdpa_reference(c, window, scale):
    """Per request: whole K/V sequence, explicit mask, torch SDPA in float64."""
    outs = []
    Hq = c["q"].shape[1]
    Hkv = c["k_new"].shape[1]
    for r in range(len(c["prefix_len"])):
        P = int(c["prefix_len"][r])
        a, b = int(c["cu_rows"][r]), int(c["cu_rows"][r + 1])
        ho0, ho1 = int(c["hist_off"][r]), int(c["hist_off"][r + 1])
        K = torch.cat([c["hist_k"][ho0:ho1], c["k_new"][a:b]]).double()   # [P+n, Hkv, d]
        V = torch.cat([c["hist_v"][ho0:ho1], c["v_new"][a:b]]).double()
        Q = c["q"][a:b].double()                                              # [n, Hq, d]
        n = b - a
        pos_q = torch.arange(P, P + n)[:, None]
        pos_k = torch.arange(0, P + n)[None, :]
        mask = pos_k <= pos_q
        if window:
            mask &= pos_k > pos_q - window
        Kx = K.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)          # [Hq, P+n, d]
        Vx = V.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            Q.permute(1, 0, 2), Kx, Vx, attn_mask=mask, scale=scale)         # [Hq, n, d]
        outs.append(o.permute(1, 0, 2))
    return torch.cat(outs).numpy()


@pytest.mark.parametrize("window", [0, 8, 128])
def test_matches_torch_sdpa(window):
    rng = np.random.default_rng(7 + window)
    c = _case(rng, prefixes=[0, 5, 40, 150], rows=[1, 4, 17, 3], Hq=6, Hkv=2, d=16)
    scale = 0.37
    got = oracle.attention(window=window, scale=scale, **c)
    ref = _sdpa_reference(c, window, scale)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_item_mode_matches_full_mode():
    rng = np.random.default_rng(3)
    c = _case(rng, prefixes=[30, 70], rows=[2, 5], Hq=8, Hkv=2, d=32)
    full = oracle.attention(window=16, scale=0.2, **c)
    items = np.array([[0, 0], [6, 7], [3, 4], [1, 2]], np.int32)
    got = oracle.attention(window=16, scale=0.2, items=items, **c)
    for k, (r, h) in enumerate(items):
        assert np.array_equal(got[k], full[r, h])


def test_swa_equals_full_when_sequence_fits_window():
    """Every key is in the window while position < W: outputs are identical."""
    rng = np.random.default_rng(11)
    W = 128
    c = _case(rng, prefixes=[0, 1, 100, 124], rows=[128, 1, 28, 4], Hq=4, Hkv=1, d=24)
    a = oracle.attention(window=W, scale=0.1, **c)
    b = oracle.attention(window=0, scale=0.1, **c)
    assert np.array_equal(a, b)
    # one more row (position 128) and the window must bite
    c2 = _case(rng, prefixes=[128], rows=[1], Hq=4, Hkv=1, d=24)
    a2 = oracle.attention(window=W, scale=0.1, **c2)
    b2 = oracle.attention(window=0, scale=0.1, **c2)
    assert not np.array_equal(a2, b2)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(5)
    W = 8
    c = _case(rng, prefixes=[20], rows=[3], Hq=2, Hkv=1, d=8)
    c["q"] = _bf16(np.zeros((3, 2, 8)))
    out = oracle.attention(window=W, scale=1.0, **c)
    vals = torch.cat([c["hist_v"], c["v_new"]]).double().numpy()[:, 0, :]   # positions 0..22
    for i in range(3):
        p = 20 + i
        expect = vals[p - W + 1:p + 1].mean(axis=0)                          # W visible keys
        assert np.allclose(out[i, 0], expect, atol=1e-14)
        assert np.allclose(out[i, 1], expect, atol=1e-14)


def test_two_keys_logistic_weight_pins_scale():
    """Two keys, q.k0 = a, q.k1 = 0: out = sigmoid(scale * a) * v0 + (1 - .) * v1."""
    a, scale = 2.0, 0.75
    q = _bf16([[[a, 0.0]]])
    hk = _bf16([[[1.0, 0.0]]])
    hv = _bf16([[[1.0, 0.0]]])
    kn = _bf16([[[0.0, 0.0]]])
    vn = _bf16([[[0.0, 1.0]]])
    out = oracle.attention(cu_rows=[0, 1], prefix_len=[1], q=q, k_new=kn, v_new=vn,
                           hist_k=hk, hist_v=hv, hist_off=[0, 1], hist_start=[0],
                           window=0, scale=scale)
    w = 1.0 / (1.0 + math.exp(-scale * a))
    assert abs(out[0, 0, 0] - w) < 1e-15 and abs(out[0, 0, 1] - (1 - w)) < 1e-15


def test_window_edge_planted_values():
    """A query at p sees p-W+1 (W keys including itself) but not p-W."""
    W, d, P = 16, 4, 40
    p = P  # the single new row
    hist = np.zeros((P, 1, d))
    q = _bf16(np.zeros((1, 1, d)))
    base = dict(cu_rows=[0, 1], prefix_len=[P], q=q, k_new=_bf16(np.zeros((1, 1, d))),
                v_new=_bf16(np.zeros((1, 1, d))), hist_k=_bf16(hist), hist_off=[0, P],
                hist_start=[0], window=W, scale=1.0)
    v_out = hist.copy()
    v_out[p - W, 0, 0] = 64.0          # just outside: must not move the output
    o1 = oracle.attention(hist_v=_bf16(v_out), **base)
    assert o1[0, 0, 0] == 0.0
    v_in = hist.copy()
    v_in[p - W + 1, 0, 0] = 64.0       # just inside: mean over W keys
    o2 = oracle.attention(hist_v=_bf16(v_in), **base)
    assert o2[0, 0, 0] == 64.0 / W


def test_new_rows_are_causal_among_themselves():
    rng = np.random.default_rng(9)
    c = _case(rng, prefixes=[33], rows=[4], Hq=4, Hkv=2, d=16)
    base = oracle.attention(window=0, scale=0.3, **c)
    c2 = dict(c)
    kn = c["k_new"].clone()
    vn = c["v_new"].clone()
    kn[2:] = 5.0
    vn[2:] = -7.0
    c2["k_new"], c2["v_new"] = kn, vn
    moved = oracle.attention(window=0, scale=0.3, **c2)
    assert np.array_equal(base[:2], moved[:2])       # rows 0, 1 never see rows 2, 3
    assert not np.array_equal(base[2:], moved[2:])


def test_gqa_contiguous_grouping():
    """Query head h reads KV head h // (Hq / Hkv)."""
    Hq, Hkv, d = 8, 2, 4
    vh = np.zeros((3, Hkv, d))
    vh[:, 1, :] = 1.0
    c = dict(cu_rows=[0, 1], prefix_len=[3], q=_bf16(np.zeros((1, Hq, d))),
             k_new=_bf16(np.zeros((1, Hkv, d))), v_new=_bf16(np.zeros((1, Hkv, d)) + [[0.0], [1.0]]),
             hist_k=_bf16(np.zeros((3, Hkv, d))), hist_v=_bf16(vh), hist_off=[0, 3],
             hist_start=[0])
    out = oracle.attention(window=0, scale=1.0, **c)
    assert np.all(out[0, :4] == 0.0) and np.all(out[0, 4:] == 1.0)


def test_missing_history_is_an_error():
    rng = np.random.default_rng(1)
    c = _case(rng, prefixes=[300], rows=[1], Hq=2, Hkv=1, d=8, hist_from=[300 - 128])
    oracle.attention(window=128, scale=0.1, **c)        # the window fits the kept tail
    with pytest.raises(ValueError):
        oracle.attention(window=0, scale=0.1, **c)       # full attention needs all of it


# --------------------------------------------------------------------------- placement
def test_full_place_is_a_bijection_onto_allocated_pages():
    rng = np.random.default_rng(2)
    page, lens = 8, [13, 0, 40, 8]
    pages = [(n + page - 1) // page for n in lens]
    perm = rng.permutation(sum(pages))
    bt = np.full((len(lens), max(pages)), -1, np.int32)
    k = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[k:k + n]
        k += n
    seen = set()
    for s, n in enumerate(lens):
        prev = None
        for p in range(n):
            blk, off = oracle.full_place(bt, sum(pages), page, s, p)
            assert 0 <= off < page
            if prev is not None and p % page:
                assert blk == prev[0] and off == prev[1] + 1     # pages are contiguous
            seen.add((blk, off))
            prev = (blk, off)
    assert len(seen) == sum(lens)
    assert oracle.full_place(bt, sum(pages), page, 1, 0) is None  # unallocated page
    ident = np.arange(4, dtype=np.int32)[None, :]
    assert oracle.full_place(ident, 4, 64, 0, 200) == (3, 8)      # textbook paging


def test_ring_place_reuses_slots_every_window():
    W = 128
    rr = np.array([5, 2], np.int32)
    slots = [oracle.ring_place(rr, 8, W, 1, p) for p in range(1000, 1000 + W)]
    assert sorted(s for _, s in slots) == list(range(W))
    assert all(r == 2 for r, _ in slots)
    for p in (0, 77, 128, 5000):
        assert oracle.ring_place(rr, 8, W, 0, p) == oracle.ring_place(rr, 8, W, 0, p + W)


def _tagged(positions, Hkv, d):
    """K rows that encode their own position exactly in bf16 (integers < 256)."""
    x = np.zeros((len(positions), Hkv, d), np.float32)
    for i, p in enumerate(positions):
        x[i, :, 0] = p // 256
        x[i, :, 1] = p % 256
        x[i, :, 2] = np.arange(Hkv)
    return _bf16(x)


def _untag(bits_row):
    row = torch.from_numpy(bits_row.view(np.int16)).view(torch.bfloat16).float().numpy()
    return int(row[0]) * 256 + int(row[1])


def test_ring_append_keeps_latest_position_per_slot():
    W, Hkv, d = 16, 2, 4
    rk = np.full((3, Hkv, W, d), 0xFFFF, np.uint16)
    rv = rk.copy()
    rr = np.array([2], np.int32)
    # three calls: 5 tokens, then 23 (longer than W), then 1
    start = 0
    for n in (5, 23, 1):
        pos = list(range(start, start + n))
        t = _tagged(pos, Hkv, d)
        bad = oracle.append(rk, rv, [0, n], [0], [start], t, t, ring_row=rr)
        assert bad == 0
        start += n
    E = start
    for j in range(W):
        latest = max(p for p in range(E) if p % W == j)
        for h in range(Hkv):
            assert _untag(rk[2, h, j]) == latest
    assert np.all(rk[0] == 0xFFFF) and np.all(rk[1] == 0xFFFF)


def test_full_append_then_gather_recovers_history():
    page, Hkv, d = 8, 2, 4
    lens = [19, 6]
    bt = np.array([[4, 0, 2], [1, -1, -1]], np.int32)
    pk = np.zeros((5, Hkv, page, d), np.uint16)
    pv = pk.copy()
    for s, n in enumerate(lens):
        t = _tagged(range(n), Hkv, d)
        assert oracle.append(pk, pv, [0, n], [s], [0], t, t, block_tables=bt) == 0
    for s, n in enumerate(lens):
        for p in range(n):
            blk, off = oracle.full_place(bt, 5, page, s, p)
            assert _untag(pk[blk, 1, off]) == p
    t = _tagged([24], Hkv, d)            # page 3 of sequence 0 is not allocated
    assert oracle.append(pk, pv, [0, 1], [0], [24], t, t, block_tables=bt) == 1


# --------------------------------------------------------------------------- window-safe
def _safe_len_closed_form(m, slot_pos, W):
    """Independent route to the ring-form answer.

    Each slot holds one position, so at most W positions are live and no two share
    a residue.  A window [L-W, L) with L > W therefore fills the whole ring, which
    forces L = 1 + (largest live position).  Shorter answers L <= W need positions
    0..L-1 live, i.e. L is at most the first dead position.
    """
    if m <= 0:
        return 0
    live = set(int(x) for j, x in enumerate(slot_pos) if x >= 0 and x % W == j)
    first_dead = 0
    while first_dead in live:
        first_dead += 1
    best = min(m, first_dead)
    if live:
        q = max(live) + 1
        if W < q <= m and all((q - W + i) in live for i in range(W)):
            best = max(best, q)
    return best


def test_window_safe_ring_matches_closed_form_on_seeded_cases():
    from workload import window_cases
    W = 128
    match, slots, _ = window_cases(1000, W, seed=1004)
    got = oracle.window_safe_len_ring(match, slots, W)
    for k in range(len(match)):
        assert got[k] == _safe_len_closed_form(int(match[k]), slots[k], W), k
    assert 0 < np.count_nonzero(got) < len(got)
    assert np.any(got == match) and np.any((got > 0) & (got < match))


def test_window_safe_exhaustive_tiny_rings():
    """Every ring state of W = 3 over positions 0..7 (plus freed), every m <= 9."""
    W = 3
    choices = [-1] + list(range(8))
    for a in choices:
        for b in choices:
            for c in choices:
                sp = np.array([a, b, c], np.int32)
                ms = np.arange(10, dtype=np.int32)
                got = oracle.window_safe_len_ring(ms, np.tile(sp, (10, 1)), W)
                for m in range(10):
                    assert got[m] == _safe_len_closed_form(m, sp, W)


def test_window_safe_hand_cases():
    W = 4
    # ring holds 6,7,8,9 (slots 2,3,0,1): the whole match of 10 is safe
    assert oracle.window_safe_len_ring([10], [[8, 9, 6, 7]], W)[0] == 10
    # same ring, match of 12: positions 10, 11 were never written; trimmed to 10
    assert oracle.window_safe_len_ring([12], [[8, 9, 6, 7]], W)[0] == 10
    # same ring, match of 8: the ring ran past the match and overwrote 4, 5 -> 0
    assert oracle.window_safe_len_ring([8], [[8, 9, 6, 7]], W)[0] == 0
    # slot 0 (position 8) freed: no window of 4 survives and position 0 is dead -> 0
    assert oracle.window_safe_len_ring([10], [[-1, 9, 6, 7]], W)[0] == 0
    # a young sequence: positions 0, 1, 2 live, 3 never written, m = 3 -> 3
    assert oracle.window_safe_len_ring([3], [[0, 1, 2, -1]], W)[0] == 3
    # same ring, m = 2: trimmed to the match itself
    assert oracle.window_safe_len_ring([2], [[0, 1, 2, -1]], W)[0] == 2
    # m = 0 is always 0
    assert oracle.window_safe_len_ring([0], [[-1, -1, -1, -1]], W)[0] == 0
    # bitmap form: live 0..5, dead 6, live 7..11 (5 >= W): the tail is safe -> 12
    live = np.array([1] * 6 + [0] + [1] * 5, np.uint8)
    assert oracle.window_safe_len_bitmap([12], [0, 12], live, W)[0] == 12
    # dead 9 instead: tail run 10..11 is short; L = 9 has window 5..8 with 6 dead;
    # L = 6 has window 2..5 all live -> 6
    live = np.array([1] * 6 + [0, 1, 1, 0, 1, 1], np.uint8)
    assert oracle.window_safe_len_bitmap([12], [0, 12], live, W)[0] == 6


def test_window_safe_bitmap_agrees_with_ring_view():
    """The bitmap of a ring's live positions gives the ring-form answer."""
    from workload import window_cases
    W = 128
    match, slots, _ = window_cases(200, W, seed=77)
    ring = oracle.window_safe_len_ring(match, slots, W)
    lives, offs = [], [0]
    for k in range(len(match)):
        m = int(match[k])
        lv = np.zeros(m, np.uint8)
        for j, p in enumerate(slots[k]):
            if 0 <= p < m and p % W == j:
                lv[p] = 1
        lives.append(lv)
        offs.append(offs[-1] + m)
    bm = oracle.window_safe_len_bitmap(match, offs, np.concatenate(lives), W)
    assert np.array_equal(ring, bm)


# --------------------------------------------------------------------------- KV bytes
def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    return vals


def test_kv_ratio_reproduces_the_pages_one_seventh():
    g = _golden("pages_facts.txt")
    n_layers, n_full, W = int(g["layers"]), int(g["full_layers"]), int(g["window"])
    from workload import layer_is_full
    full = layer_is_full(n_layers)
    assert sum(full) == n_full and n_layers - sum(full) == int(g["swa_layers"])
    target = float(g["kv_ratio_num"]) / float(g["kv_ratio_den"])
    r_long = oracle.kv_ratio(full, W, 1 << 20)
    assert abs(r_long - target) < 1e-3            # "about 1/7" at 1M tokens
    for L in (1, 64, W):
        assert oracle.kv_ratio(full, W, L) == 1.0  # fits the window: nothing saved
    prev = 1.0
    for L in (W + 1, 256, 8192, 65536, 1 << 20):
        r = oracle.kv_ratio(full, W, L)
        assert target < r < prev
        prev = r
    # bytes per token per layer: K and V, 4 KV heads, d = 128, bf16
    assert oracle.kv_bytes([1], W, 1, 2 * 4 * 128 * 2) == 2048.0


# ---------------------------------------------------------------- FP8 (E4M3) KV
# hotdry.top "MiMo inference optimization, edge deployment", "KV Cache 量化策略的技术选型":
# FP8 KV; the E4M3 values follow the OCP 8-bit floating point definition (bias 7,
# 3 mantissa bits, no infinities, largest finite 448).

def test_e4m3_hand_values():
    enc = oracle.e4m3_encode
    assert enc(448.0) == 0x7E and enc(1.0) == 0x38 and enc(-2.0) == 0xC0
    assert enc(2.0 ** -9) == 0x01            # smallest subnormal
    assert enc(2.0 ** -10) == 0x00           # tie with 0 -> even code
    assert enc(1.0625) == 0x38               # tie between 1 and 1.125 -> even
    assert enc(1.1875) == 0x3A               # tie between 1.125 and 1.25 -> even
    assert enc(500.0) == 0x7E and enc(-1e9) == 0xFE   # saturating
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_round_trip_and_order():
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    for c in finite:
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)
    pos = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))   # codes 0..126 are increasing


def test_e4m3_matches_torch_cast():
    """A library routine: torch's float8_e4m3fn cast (round to nearest even)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 dtype in this torch")
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(1000) * 0.01,
                        rng.uniform(-448, 448, 1000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_quantize_rows_scale_and_extremes():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(9)
    x = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    x[3] = 0
    codes, scales = oracle.quantize_e4m3(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    assert scales[3] == 0 and not codes[3].any()
    for r in range(64):
        if r == 3:
            continue
        j = int(np.argmax(np.abs(xf[r])))
        assert codes[r, j] & 0x7F == 0x7E            # the row maximum maps to 448
        deq = np.array([oracle.e4m3_value(c) for c in codes[r]]) * scales[r]
        # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormals
        big = np.abs(xf[r]) > scales[r] * 2.0 ** -6
        assert np.all(np.abs(deq - xf[r])[big] <= np.abs(xf[r])[big] * 2.0 ** -4 + 1e-12)


def test_fp8_history_attention_equals_bf16_oracle_on_exact_values():
    """With unit scales the dequantised history is exactly the E4M3 values, all
    representable in bf16: orc_attention_fp8hist must equal orc_attention fed
    those values as bf16 (both float64)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    Hq, Hkv, d, R = 8, 2, 32, 2
    P = [13, 40]
    T = [1, 3]
    hist = sum(P)
    codes_k = rng.integers(0, 0x7F, (hist, Hkv, d)).astype(np.uint8) | \
        (rng.integers(0, 2, (hist, Hkv, d)).astype(np.uint8) << 7)
    codes_k[codes_k == 0xFF] = 0xFE
    codes_v = rng.integers(0x20, 0x50, (hist, Hkv, d)).astype(np.uint8)
    ones = np.ones((hist, Hkv), np.float32)
    val_k = np.vectorize(oracle.e4m3_value)(codes_k).astype(np.float32)
    val_v = np.vectorize(oracle.e4m3_value)(codes_v).astype(np.float32)
    bk = torch.from_numpy(val_k).to(torch.bfloat16)
    bv = torch.from_numpy(val_v).to(torch.bfloat16)
    assert np.array_equal(bk.float().numpy(), val_k)   # exactly representable
    rows = sum(T)
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(rows, Hq, d, generator=g) * 0.05).to(torch.bfloat16)
    kn = torch.randn(rows, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(rows, Hkv, d, generator=g).to(torch.bfloat16)
    cu = np.array([0, T[0], rows], np.int32)
    pl = np.array(P, np.int32)
    ho = np.array([0, P[0], hist], np.int64)
    a = oracle.attention_fp8hist(cu, pl, q, kn, vn, codes_k, ones, codes_v, ones, ho, 0.3)
    b = oracle.attention(cu, pl, q, kn, vn, bk, bv, ho, np.zeros(R, np.int32), 0, 0.3)
    assert np.max(np.abs(a - b)) == 0.0
    # doubling one row's scale doubles that key's dequantised values (exact)
    two = ones.copy()
    two[5] = 2.0
    bk2 = torch.from_numpy(val_k * two[:, :, None]).to(torch.bfloat16)
    bv2 = torch.from_numpy(val_v * two[:, :, None]).to(torch.bfloat16)
    a2 = oracle.attention_fp8hist(cu, pl, q, kn, vn, codes_k, two, codes_v, two, ho, 0.3)
    b2 = oracle.attention(cu, pl, q, kn, vn, bk2, bv2, ho, np.zeros(R, np.int32), 0, 0.3)
    assert np.max(np.abs(a2 - b2)) == 0.0


# E5M2, the second FP8 format (hotdry.top "MiMo inference optimization, edge
# deployment", "KV Cache 量化策略的技术选型"): OCP E5M2, bias 15, 2 mantissa bits.

def test_e5m2_hand_values():
    enc = oracle.e5m2_encode
    assert enc(57344.0) == 0x7B and enc(1.0) == 0x3C and enc(-2.0) == 0xC0
    assert enc(2.0 ** -16) == 0x01           # smallest subnormal
    assert enc(2.0 ** -17) == 0x00           # tie with 0 -> even code
    assert enc(2.0 ** -14) == 0x04           # smallest normal
    assert enc(1.125) == 0x3C                # tie between 1 and 1.25 -> even
    assert enc(1.375) == 0x3E                # tie between 1.25 and 1.5 -> even
    assert enc(61440.0) == 0x7B and enc(1e6) == 0x7B and enc(-1e9) == 0xFB   # saturating
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert oracle.e5m2_value(0x7B) == 57344.0 and oracle.e5m2_value(0x01) == 2.0 ** -16
    assert oracle.e5m2_value(0x7C) == math.inf and oracle.e5m2_value(0xFC) == -math.inf
    assert np.isnan(oracle.e5m2_value(0x7D)) and np.isnan(oracle.e5m2_value(0xFF))


def test_e5m2_values_are_the_top_byte_of_fp16():
    """An E5M2 code is an IEEE binary16 with its low 8 bits zero: numpy's float16
    decoding (an independent routine) gives every finite code's value."""
    for c in range(256):
        if (c & 0x7F) >= 0x7C:
            continue
        ref = float(np.array([c << 8], np.uint16).view(np.float16)[0])
        assert oracle.e5m2_value(c) == ref, hex(c)


def test_e5m2_round_trip_and_order():
    finite = [c for c in range(256) if (c & 0x7F) < 0x7C]
    for c in finite:
        assert oracle.e5m2_encode(oracle.e5m2_value(c)) == c, hex(c)
    pos = [oracle.e5m2_value(c) for c in range(0x7C)]
    assert all(a < b for a, b in zip(pos, pos[1:]))


def test_e5m2_matches_torch_cast():
    """torch's float8_e5m2 cast (round to nearest even) inside the finite range."""
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("no float8 dtype in this torch")
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(3000) * 3000, rng.standard_normal(1000) * 1e-3,
                        rng.uniform(-57344, 57344, 1000),
                        rng.standard_normal(500) * 2.0 ** -15]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    got = np.array([oracle.e5m2_encode(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_quantize_e5m2_rows_scale_and_extremes():
    g = torch.Generator().manual_seed(13)
    x = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    x[5] = 0
    codes, scales = oracle.quantize_e5m2(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, (amax / np.float32(57344.0)).astype(np.float32))
    assert scales[5] == 0 and not codes[5].any()
    c2, s2 = oracle.quantize_fp8(x, "e5m2")
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    for r in range(64):
        if r == 5:
            continue
        j = int(np.argmax(np.abs(xf[r])))
        assert codes[r, j] & 0x7F == 0x7B            # the row maximum maps to 57344
        deq = np.array([oracle.e5m2_value(c) for c in codes[r]]) * scales[r]
        # E5M2 keeps 2 mantissa bits: relative error <= 2^-3 above the subnormals
        big = np.abs(xf[r]) > scales[r] * 2.0 ** -14
        assert np.all(np.abs(deq - xf[r])[big] <= np.abs(xf[r])[big] * 2.0 ** -3 + 1e-12)


def test_e5m2_history_attention_equals_bf16_oracle_on_exact_values():
    """Every E5M2 value is exact in bf16: with unit scales the E5M2 history must
    give orc_attention fed those values, and the format switch must matter."""
    rng = np.random.default_rng(14)
    Hq, Hkv, d, R = 8, 2, 32, 2
    P, T = [9, 33], [2, 1]
    hist = sum(P)
    codes_k = (rng.integers(0x30, 0x44, (hist, Hkv, d)).astype(np.uint8) |
               (rng.integers(0, 2, (hist, Hkv, d)).astype(np.uint8) << 7))
    codes_v = rng.integers(0x28, 0x48, (hist, Hkv, d)).astype(np.uint8)
    ones = np.ones((hist, Hkv), np.float32)
    val_k = np.vectorize(oracle.e5m2_value)(codes_k).astype(np.float32)
    val_v = np.vectorize(oracle.e5m2_value)(codes_v).astype(np.float32)
    bk = torch.from_numpy(val_k).to(torch.bfloat16)
    bv = torch.from_numpy(val_v).to(torch.bfloat16)
    assert np.array_equal(bk.float().numpy(), val_k)
    rows = sum(T)
    g = torch.Generator().manual_seed(15)
    q = (torch.randn(rows, Hq, d, generator=g) * 0.05).to(torch.bfloat16)
    kn = torch.randn(rows, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(rows, Hkv, d, generator=g).to(torch.bfloat16)
    cu = np.array([0, T[0], rows], np.int32)
    pl = np.array(P, np.int32)
    ho = np.array([0, P[0], hist], np.int64)
    a = oracle.attention_fp8hist(cu, pl, q, kn, vn, codes_k, ones, codes_v, ones, ho, 0.3,
                                 fmt="e5m2")
    b = oracle.attention(cu, pl, q, kn, vn, bk, bv, ho, np.zeros(R, np.int32), 0, 0.3)
    assert np.max(np.abs(a - b)) == 0.0
    e4 = oracle.attention_fp8hist(cu, pl, q, kn, vn, codes_k, ones, codes_v, ones, ho, 0.3)
    assert np.max(np.abs(e4 - b)) > 0.1          # read as E4M3 the codes mean other values
    with pytest.raises(ValueError):
        oracle.attention_fp8hist(cu, pl, q, kn, vn, codes_k, ones, codes_v, ones, ho, 0.3,
                                 fmt="e3m4")


# ---------------------------------------------------------------- prefix model
# youleyou.com s2 "KVCache系统重构": a hit counts up to the window-safe length; the
# Full index is authoritative; SWA is kept for a finished request's last window.

def test_prefix_model_hand_cases():
    from oracle.prefix_model import PrefixModel, ring_positions
    m = PrefixModel(W=4)
    assert m.match([1, 2]) == (0, [], -1, [-1] * 4)
    dup, kept = m.insert([1, 2, 3, 4, 5, 6], [10, 11, 12, 13, 14, 15], 7, ring_positions(6, 4))
    assert dup == [] and kept
    assert ring_positions(6, 4) == [4, 5, 2, 3]           # slot s keeps the latest p = s mod 4
    # a follow-up turn: full match, the path's own ring, every window position live
    mm, slots, row, pos = m.match([1, 2, 3, 4, 5, 6, 9])
    assert (mm, slots, row) == (6, [10, 11, 12, 13, 14, 15], 7)
    assert int(oracle.window_safe_len_ring([mm], [pos], 4)[0]) == 6
    # a branch before the path's end: the ring was written past the match
    mm, _, row, pos = m.match([1, 2, 3, 8])
    assert (mm, row) == (3, 7) and int(oracle.window_safe_len_ring([mm], [pos], 4)[0]) < 4
    # a second path through the same point: the shorter path's ring is offered first
    dup, kept = m.insert([1, 2, 3, 9], [10, 11, 12, 30], 8, ring_positions(4, 4))
    assert dup == [] and kept
    assert m.match([1, 2, 3, 5])[2] == 8
    # duplicates: a request that recomputed a cached position returns its own slot
    dup, kept = m.insert([1, 2, 7], [40, 41, 42], 8, ring_positions(3, 4))
    assert dup == [40, 41] and not kept                   # row 8 is already held
    # dropping the Full slots of a suffix shortens later matches
    m.drop_slots([14, 15])
    assert m.match([1, 2, 3, 4, 5, 6])[0] == 4
    # equal path lengths through the match point: the latest attached row wins,
    # whatever its id (the most recent request's window is the freshest)
    m2 = PrefixModel(W=4)
    m2.insert([1, 2, 3, 4], [10, 11, 12, 13], 5, ring_positions(4, 4))
    m2.insert([1, 2, 3, 6], [10, 11, 12, 16], 9, ring_positions(4, 4))
    assert m2.match([1, 2, 3, 7])[2] == 9
    m2.insert([1, 2, 3, 8], [10, 11, 12, 18], 2, ring_positions(4, 4))
    assert m2.match([1, 2, 3, 7])[2] == 2
    m2.take_ring(2)
    assert m2.match([1, 2, 3, 7])[2] == 9

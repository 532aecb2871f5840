"""Grid index arithmetic of the kernels, restated on the host and checked over
random layouts: the decode kernel's stream-K split and in-kernel merge
(full_attention_kv_gb300/csrc/decode.cu, including the 1M-token extreme) and the
prefill kernel's CTA-to-tile-pair map, grid bound and key-tile schedule (csrc/prefill.cu,
csrc/api.cu), both kernels' ring-visibility formulas, and the slot and owning warp of
the new token on the sliding decode's T = 1 full-ring path.

Items (64-key tiles) of all units are laid end to end; CTA c takes items
[c N / C, (c + 1) N / C).  A unit split across CTAs leaves one partial state per
covering CTA in slot 2 c + (1 if the unit starts after the CTA's first item), and
the CTA whose arrival count reaches c_hi - c_lo merges slots c_lo .. c_hi with
c_lo = ((start + 1) C - 1) / N and c_hi = (end C - 1) / N.  The invariants: every
CTA gets at least one item, no two partial states share a slot, the covering CTAs
are exactly c_lo .. c_hi, and the arrival count the last CTA waits for is their
number minus one."""
import random


def _check(units_items, grid):
    N = sum(units_items)
    C = min(N, grid)
    starts, acc = [], 0
    for n in units_items:
        starts.append(acc)
        acc += n
    written = set()
    for cta in range(C):
        i0, i1 = cta * N // C, (cta + 1) * N // C
        assert i1 > i0
        for us, n in zip(starts, units_items):
            ue = us + n
            if ue <= i0 or us >= i1 or (us >= i0 and ue <= i1):
                continue  # not touched, or whole inside this CTA (written straight out)
            slot = 2 * cta + (1 if i0 < us else 0)
            assert slot not in written
            written.add(slot)
            c_lo, c_hi = ((us + 1) * C - 1) // N, (ue * C - 1) // N
            covering = [c for c in range(C) if c * N // C < ue and (c + 1) * N // C > us]
            assert covering == list(range(c_lo, c_hi + 1))


def test_partition_and_merge_slots():
    rng = random.Random(7)
    for _ in range(600):
        U = rng.randint(1, 40)
        items = [rng.choice([1, 2, rng.randint(1, 40), rng.randint(100, 4000)]) for _ in range(U)]
        _check(items, rng.choice([1, 2, 3, 7, 128, 152, rng.randint(1, 300)]))


def test_partition_extremes():
    _check([16384] * 16, 152)   # 4 sequences x 4 KV heads at 1M tokens, one CTA per SM
    _check([1] * 2000, 152)     # more units than CTAs, one tile each
    _check([3], 152)            # fewer items than CTAs: the grid shrinks to N


def _prefill_grid_pairs(rows, R, max_chunk):
    """Tile-pair count the prefill launch sizes its grid for (api.cu, prefill.cu)."""
    b1 = rows // 128 + R
    b2 = R * ((max_chunk + 127) // 128)
    tiles = min(b1, b2)
    return (tiles + R + 1) // 2


def test_prefill_grid_covers_every_tile_pair_once():
    """prefill.cu maps CTA x (per query head) to the x-th (request, 256-row pair)
    in request order; the grid bound computed on the host from rows, R and
    max_chunk must cover every pair, and CTAs past the last pair map to none."""
    rng = random.Random(11)
    for _ in range(3000):
        R = rng.randint(1, 12)
        C = [rng.choice([0, 1, 127, 128, 129, 255, 256, 257, rng.randint(0, 9000)])
             for _ in range(R)]
        rows = sum(C)
        if rows == 0:
            continue
        grid = _prefill_grid_pairs(rows, R, max(C))
        seen = []
        for tl in range(grid):
            acc, found = 0, None
            for r, c in enumerate(C):
                n_pairs = (c + 255) // 256
                if tl < acc + n_pairs:
                    found = (r, tl - acc)
                    break
                acc += n_pairs
            if found is not None:
                seen.append(found)
        want = [(r, q) for r, c in enumerate(C) for q in range((c + 255) // 256)]
        assert seen == want


def _ring_after(P, W):
    """Position each ring slot holds after positions 0 .. P-1 were appended (-1: none)."""
    held = [-1] * W
    for p in range(P):
        held[p % W] = p
    return held


def test_ring_visibility_formulas():
    """The kernels never build the ring's slot -> position table: decode derives a
    slot's position as c - 1 - ((c - 1 - s) mod W), prefill as P - 1 - back with
    back = r0 - s (+ W when s > r0), r0 = (P - 1) mod W, and a row sees the slot
    iff back <= P - 1 - max(0, P + i - W + 1).  Both must equal the definition:
    the slot's held position p (if any) lies in the row's window
    [max(0, q - W + 1), q] of its query position q."""
    for W in (64, 128, 256):
        for P in list(range(0, 3 * W + 2, 7)) + [1, W - 1, W, W + 1, 2 * W]:
            held = _ring_after(P, W)
            r0 = (P - 1) % W if P > 0 else 0
            for i in (0, 1, 5, W - 2, W - 1, W, W + 3):
                q = P + i
                lim = P - 1 - max(0, q - W + 1)
                for s in range(W):
                    want = held[s] >= 0 and held[s] >= max(0, q - W + 1)
                    # prefill (the ring is read only when P > 0)
                    if P > 0:
                        back = r0 - s + (W if s > r0 else 0)
                        assert (back <= lim) == want, (W, P, i, s)
                    # decode: query t = i of a T-token step on c = P cached tokens
                    pos = P - 1 - ((P - 1 - s) % W)
                    got = pos >= 0 and pos >= q - W + 1
                    assert got == want, (W, P, i, s)


def _sched(P, i0, has_b, W, ring):
    """prefill.cu make_sched: (prefix or ring tiles, first chunk tile, tile count)."""
    i_last = i0 + (256 if has_b else 128) - 1
    if not ring:
        n_fixed, m_lo = (P + 127) // 128, 0
    else:
        n_fixed = (W + 127) // 128 if (P > 0 and i0 < W - 1) else 0
        lo = i0 - W + 1
        m_lo = lo // 128 if lo > 0 else 0
    return n_fixed, m_lo, n_fixed + (i_last // 128 - m_lo + 1)


def test_prefill_schedule_covers_every_visible_key():
    """Each CTA of a request runs its prefix (or ring) tiles and the chunk tiles
    m_lo .. last row / 128; every key a row of the pair can see must lie in one."""
    for W in (64, 128, 256):
        for ring in (False, True):
            for P in (0, 1, 63, 64, 200, 5000):
                for C in (1, 100, 128, 129, 256, 257, 700):
                    for qp in range((C + 255) // 256):
                        i0 = qp * 256
                        has_b = i0 + 128 < C
                        n_fixed, m_lo, nt = _sched(P, i0, has_b, W, ring)
                        chunk_lo, chunk_hi = m_lo * 128, (m_lo + nt - n_fixed) * 128
                        for i in range(i0, min(i0 + 256, C)):
                            q = P + i
                            first = max(0, q - W + 1) if ring else 0
                            # prefix keys [first, P) need the prefix / ring tiles
                            if first < P:
                                if ring:
                                    assert n_fixed == (W + 127) // 128
                                else:
                                    assert n_fixed * 128 >= P
                            # chunk rows [max(first - P, 0), i]
                            lo_row = max(first - P, 0)
                            assert chunk_lo <= lo_row and i < chunk_hi, (W, ring, P, C, i)


# ---------------------------------------------------------------- sliding-window prefill
KV_ROWS = 160   # prefill_swa.cu: key capacity of a stage
BOX = 16        # rows per K / V TMA box


def _swa_supported(W, G):
    return 128 % G == 0 and W % BOX == 0 and W + 128 // G + BOX <= KV_ROWS


def _swa_tile(P, C, i0, W, G):
    """prefill_swa.cu producer: the tile's two key regions (ring: first position a0,
    nr keys; chunk: first chunk row z0, nc keys)."""
    ppt = 128 // G
    nr, a0 = 0, 0
    if P > 0 and i0 < W - 1:
        a0 = max(0, P + i0 - W + 1) & ~(BOX - 1)
        nr = ((P + BOX - 1) & ~(BOX - 1)) - a0
    z0 = max(0, i0 - W)
    nc = i0 + ppt - z0
    return a0, nr, z0, nc


def _swa_row_ranges(P, C, i, W, a0, nr, z0):
    """prefill_swa.cu softmax: visible columns [rlo, rhi) of the ring region and
    [clo, chi) of the chunk region for chunk row i."""
    rlo = rhi = 0
    if nr > 0:
        rlo = max(0, P + i - W + 1) - a0
        rhi = max(rlo, P - a0)
    clo = nr + max(0, i - W + 1) - z0
    chi = nr + i + 1 - z0
    return rlo, rhi, clo, chi


def test_swa_prefill_tiles_cover_each_row_window_exactly():
    """Every row of every tile sees, through its two column ranges, exactly the
    positions of its window [max(0, P + i - W + 1), P + i]; the ring region's columns
    it sees hold exactly those positions (a 16-aligned position block maps onto one
    16-slot block of the ring, and the ring -- written in position order up to P --
    holds position p in slot p mod W for every p it sees); both regions fit a stage
    and every TMA box stays inside the ring row of its (sequence, head)."""
    rng = random.Random(5)
    shapes = [(W, G) for W in (64, 128, 192, 256) for G in (1, 2, 4, 8) if _swa_supported(W, G)]
    assert (128, 8) in shapes and (64, 8) in shapes
    for W, G in shapes:
        ppt = 128 // G
        cases = [(P, C) for P in (0, 1, 15, 16, 17, W - 1, W, W + 1, 1000, 1007, 1008)
                 for C in (1, 2, 15, 16, 17, W - 1, W, W + 1, 300)]
        cases += [(rng.randint(0, 5000), rng.randint(1, 700)) for _ in range(200)]
        for P, C in cases:
            held = _ring_after(P, W)
            for i0 in range(0, C, ppt):
                a0, nr, z0, nc = _swa_tile(P, C, i0, W, G)
                assert nr % BOX == 0 and nc % BOX == 0 and nr >= 0 and nc > 0
                assert nr + nc <= KV_ROWS, (W, G, P, C, i0, nr, nc)
                assert (nr + nc) // 2 <= 128          # P columns stay below O's
                for b in range(0, nr, BOX):
                    slot = (a0 + b) % W
                    assert slot + BOX <= W            # a box never wraps the ring row
                assert z0 >= 0
                for i in range(i0, min(i0 + ppt, C)):
                    rlo, rhi, clo, chi = _swa_row_ranges(P, C, i, W, a0, nr, z0)
                    assert 0 <= rlo <= rhi <= nr and nr <= clo <= chi <= nr + nc
                    seen = []
                    for c in range(nr + nc):
                        if rlo <= c < rhi:
                            pos = a0 + c
                            assert held[pos % W] == pos, (W, P, i, c)
                            seen.append(pos)
                        elif clo <= c < chi:
                            seen.append(P + z0 + (c - nr))
                    q = P + i
                    assert seen == list(range(max(0, q - W + 1), q + 1)), (W, G, P, C, i)


def test_swa_prefill_tile_walk_matches_the_grid():
    """The persistent CTAs walk tiles t = cta + k * grid in request order (KV head
    fastest); the host grid bound Hkv (rows / ppt + R) never drops a tile, and the
    walk visits every (request, row block, head) exactly once."""
    rng = random.Random(3)
    for _ in range(500):
        G = rng.choice([2, 4, 8])
        Hkv = rng.choice([1, 2, 4])
        ppt = 128 // G
        R = rng.randint(1, 10)
        C = [rng.choice([0, 1, ppt - 1, ppt, ppt + 1, rng.randint(0, 3000)]) for _ in range(R)]
        rows = sum(C)
        tiles = [((c + ppt - 1) // ppt) * Hkv for c in C]
        total = sum(tiles)
        bound = (rows // ppt + R) * Hkv
        assert bound >= total
        grid = min(bound, rng.choice([1, 7, 152]))
        seen = []
        for cta in range(grid):
            n_my = (total - 1 - cta) // grid + 1 if cta < total else 0
            r, acc = 0, 0
            for k in range(n_my):
                t = cta + k * grid
                while t >= acc + tiles[r]:
                    acc += tiles[r]
                    r += 1
                loc = t - acc
                seen.append((r, loc // Hkv, loc % Hkv))
        want = [(r, b, h) for r, c in enumerate(C) for b in range((c + ppt - 1) // ppt)
                for h in range(Hkv)]
        assert sorted(seen) == want


def test_ring_t1_new_token_slot_and_owner():
    """Sliding-layer decode at T = 1 on a full ring (c >= W = 128, decode.cu's
    leading loop): the kernel writes the new token over the staged row of slot
    c mod W and then lets the query see all W staged keys.  Against the oracle's ring
    placement and the window definition: after positions 0 .. c-1 were appended,
    that slot holds position c - W, the one ring position outside the query's window
    (c - W, c]; every other slot holds a position inside it, so after the overwrite
    the W slots hold exactly the window.  And exactly one of the four consumer warps
    writes the row: warp 2 grp + half reads tile my_j = grp xor (k0 & 1) of the unit
    (its stage grp, k0 the unit's first item index in the CTA's range), keys
    32 half .. 32 half + 31 of it."""
    import numpy as np

    import oracle
    W = 128
    ring_row = np.array([0], np.int32)
    for c in list(range(W, 3 * W + 2)) + [1000, 4097, 65535]:
        held = [-1] * W
        for p in range(max(0, c - 2 * W), c):  # older positions are overwritten anyway
            row, slot = oracle.ring_place(ring_row, 1, W, 0, p)
            assert row == 0
            held[slot] = p
        window = set(range(c - W + 1, c + 1))
        _, new_slot = oracle.ring_place(ring_row, 1, W, 0, c)
        assert new_slot == c % W
        assert held[new_slot] == c - W and (c - W) not in window
        assert all(held[s] in window for s in range(W) if s != new_slot)
        after = list(held)
        after[new_slot] = c
        assert set(after) == window
        for k0 in (0, 1, 2, 7):
            owners = []
            for warp in range(4):
                grp, half = warp // 2, warp % 2
                my_j = grp ^ (k0 & 1)
                assert (k0 + my_j) % 2 == grp  # the stage of item k0 + my_j is grp
                if new_slot // 64 == my_j and (new_slot % 64) // 32 == half:
                    owners.append(warp)
                    assert my_j * 64 + 32 * half <= new_slot < my_j * 64 + 32 * half + 32
            assert len(owners) == 1, (c, k0, owners)

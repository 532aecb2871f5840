"""Grid index arithmetic of the kernels, restated on the host and checked over
random layouts: the decode kernel's stream-K split and in-kernel merge
(full_attention_kv_gb300/csrc/decode.cu, including the 1M-token extreme) and the
prefill kernel's CTA-to-tile-pair map, grid bound and key-tile schedule (csrc/prefill.cu,
csrc/api.cu), and both kernels' ring-visibility formulas.

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

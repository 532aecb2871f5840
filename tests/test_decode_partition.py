"""Index arithmetic of the decode kernel's stream-K split and in-kernel merge
(full_attention_kv_gb300/csrc/decode.cu), restated on the host and checked over
random unit layouts, CTA counts and the 1M-token extreme.

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

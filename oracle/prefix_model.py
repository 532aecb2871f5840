"""Brute-force model of the prefix-tree liveness semantics -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module.  It shares no code with the library's
tree and knows nothing of nodes, splits or edges: the cache is a dictionary from
every cached prefix (a token tuple) to the Full KV Pool slot of its last token,
plus a dictionary from cached paths to the SWA ring row that holds their last
window.

Semantics followed [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s2
"KVCache系统重构"; hotdry.top "MiMo-V2.5 ultra-speed inference architecture",
"Hybrid SWA"]: the Full Attention index is authoritative and maps to the SWA pool;
a hit counts only up to the window-safe length; SWA is kept for the last window of
a finished request (eviction tied to request lifetime); the Full index and the
SWA rows are evicted independently.

Readings (the pages fix no data structure): the match length m is the longest
cached prefix; the ring row offered with it belongs to a cached path whose common
prefix with the request is exactly m, the shortest such path first, then the
latest attached row, then the smallest row id; no row when m = 0.  The
window-safe length is then ``oracle.window_safe_len_ring(m, row positions, W)``.
"""


class PrefixModel:
    def __init__(self, W):
        self.W = W
        self.slot = {}    # prefix tuple -> Full slot of its last token
        self.rings = {}   # path tuple -> (ring row, positions held [W], attach order)
        self.order = 0

    # -- queries ----------------------------------------------------------------
    def match(self, tokens):
        """-> (m, Full slots of [0, m), ring row or -1, positions [W])."""
        tokens = tuple(int(t) for t in tokens)
        m = 0
        while m < len(tokens) and tokens[:m + 1] in self.slot:
            m += 1
        slots = [self.slot[tokens[:i + 1]] for i in range(m)]
        if m == 0:
            return 0, slots, -1, [-1] * self.W
        head = tokens[:m]
        cands = [(len(path), -order, row, path)
                 for path, (row, _, order) in self.rings.items() if path[:m] == head]
        if not cands:
            return m, slots, -1, [-1] * self.W
        _, _, row, path = min(cands)
        return m, slots, row, list(self.rings[path][1])

    def cached_tokens(self):
        return len(self.slot)

    def rows_held(self):
        return sorted(r for r, _, _ in self.rings.values())

    # -- updates ----------------------------------------------------------------
    def insert(self, tokens, slots, ring_row=-1, positions=None):
        """-> (request slots that duplicate cached positions, ring kept)."""
        tokens = tuple(int(t) for t in tokens)
        dup = []
        for i in range(len(tokens)):
            key = tokens[:i + 1]
            if key in self.slot:
                if self.slot[key] != int(slots[i]):
                    dup.append(int(slots[i]))
            else:
                self.slot[key] = int(slots[i])
        kept = False
        held = {r for r, _, _ in self.rings.values()}
        if ring_row >= 0 and tokens and tokens not in self.rings and ring_row not in held:
            self.order += 1
            self.rings[tokens] = (ring_row, [int(p) for p in positions], self.order)
            kept = True
        return dup, kept

    def take_ring(self, row):
        """The request that matched took ownership of `row`."""
        for path, (r, _, _) in list(self.rings.items()):
            if r == row:
                del self.rings[path]

    def drop_slots(self, freed):
        """Mirror a Full eviction: forget every prefix whose slot was freed."""
        freed = set(int(s) for s in freed)
        for key in [k for k, s in self.slot.items() if s in freed]:
            del self.slot[key]

    def drop_rows(self, rows):
        for r in rows:
            self.take_ring(int(r))


def ring_positions(length, W, freed=()):
    """Positions a ring row holds after positions 0 .. length-1 were written in
    order (slot s keeps the latest p < length with p mod W == s, else -1), with the
    slots in `freed` then marked -1."""
    pos = [-1] * W
    for p in range(length):
        pos[p % W] = p
    for s in freed:
        pos[s] = -1
    return pos

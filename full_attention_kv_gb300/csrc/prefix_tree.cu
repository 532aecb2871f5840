// prefix_tree.cu -- host-side prefix tree with a Full-index / SWA-segment liveness
// model (no device code; the window-safe lengths of a matched batch are computed
// on the GPU by hsa_window_safe_len).
//
// [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s2 "KVCache系统重构":
// the Full Attention index is the authoritative index and maps to SWA; matching is
// upgraded to the window-safe length; SWA eviction follows the request lifetime so
// the SWA pool stays at window scale; each node carries a Full Attention segment
// index and an SWA segment mapping with independent eviction.  hotdry.top
// "MiMo-V2.5 ultra-speed inference architecture", "Hybrid SWA": a node records the
// Full Attention index and the SWA window mapping; the match is cut back to the
// window boundary.]
//
// A radix tree over int32 tokens.  Node ids are stable (a split keeps the lower
// part under the old id and gives the upper part a new one), so a lock handle -- the
// id of the node where a match ended -- stays valid while the tree changes.
// Every node caches the preferred ring holder of its subtree, so choosing the ring
// row of a match costs O(1) however many paths share the match point; eviction
// takes leaves from a heap ordered as the policies state, O(log n) per victim.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/hsa_tree.h"

namespace {

struct Node {
    int32_t parent = -1;
    int64_t depth = 0;                           // position after the node's last token
    std::vector<int32_t> tok, slot;              // tokens and their Full KV Pool slots
    std::unordered_map<int32_t, int32_t> child;  // first token -> child id
    int32_t ring = -1;                           // ring row of the path ending here
    std::vector<int32_t> ring_pos;               // [W] positions held by that row
    uint64_t ring_attach = 0;                    // clock when the row was attached
    uint64_t ring_use = 0;                       // attach or last selection (SWA LRU)
    uint64_t last_use = 0;                       // last match or insert through it (Full LRU)
    int32_t lock = 0;
    int32_t best = -1;                           // preferred ring holder in the subtree
    bool alive = false;
};

struct Walk {
    int64_t m = 0;      // tokens matched
    int32_t end = 0;    // last node touched (root if m == 0)
    int32_t kin = 0;    // tokens matched inside `end`
};

}  // namespace

struct hsa_ptree {
    int32_t W = 0, n_rows = 0;
    std::vector<Node> nodes;
    std::vector<int32_t> free_ids;
    std::vector<uint8_t> row_held;  // ring row attached somewhere in the tree
    uint64_t clock = 0;
    int64_t cached = 0;
    int32_t rows_held = 0;

    int32_t new_node(int32_t parent)
    {
        int32_t id;
        if (!free_ids.empty()) {
            id = free_ids.back();
            free_ids.pop_back();
            nodes[id] = Node();
        } else {
            id = (int32_t)nodes.size();
            nodes.emplace_back();
        }
        nodes[id].parent = parent;
        nodes[id].alive = true;
        return id;
    }

    // Longest cached prefix of tokens[0..n); optionally gathers its Full slots.
    Walk walk(const int32_t *tokens, int64_t n, int32_t *slots_out) const
    {
        Walk w;
        int32_t cur = 0;
        while (w.m < n) {
            const Node &nc = nodes[cur];
            auto it = nc.child.find(tokens[w.m]);
            if (it == nc.child.end())
                break;
            const Node &c = nodes[it->second];
            int32_t k = 0;
            const int32_t len = (int32_t)c.tok.size();
            while (k < len && w.m + k < n && c.tok[k] == tokens[w.m + k])
                ++k;
            if (slots_out)
                std::memcpy(slots_out + w.m, c.slot.data(), sizeof(int32_t) * (size_t)k);
            w.m += k;
            w.end = it->second;
            w.kin = k;
            if (k < len)
                break;
            cur = it->second;
        }
        return w;
    }

    // Ring preference between two ring holders (b may be -1): the shorter path,
    // then the later attached row, then the smaller row id.  A strict total order,
    // since a row is attached at one node at most.
    bool ring_better(int32_t a, int32_t b) const
    {
        if (b < 0)
            return true;
        const Node &na = nodes[a], &nb = nodes[b];
        if (na.depth != nb.depth)
            return na.depth < nb.depth;
        if (na.ring_attach != nb.ring_attach)
            return na.ring_attach > nb.ring_attach;
        return na.ring < nb.ring;
    }

    // Recompute `best` of x and of its ancestors after a ring or a child of x
    // changed.  An ancestor's value depends only on its own ring and its children's
    // values, so the walk stops at the first node whose value is unchanged.
    void refresh_best(int32_t x)
    {
        for (; x >= 0; x = nodes[x].parent) {
            int32_t b = nodes[x].ring >= 0 ? x : -1;
            for (const auto &kv : nodes[x].child) {
                const int32_t cb = nodes[kv.second].best;
                if (cb >= 0 && ring_better(cb, b))
                    b = cb;
            }
            if (b == nodes[x].best)
                return;
            nodes[x].best = b;
        }
    }

    // Ring row for a match ending in node `end`: the preferred ring holder among the
    // path ends in its subtree (the cached paths through the match point).  -1 if
    // none or if nothing matched.
    int32_t choose_ring(const Walk &w) const { return w.m == 0 ? -1 : nodes[w.end].best; }

    void touch(int32_t x)
    {
        const uint64_t now = ++clock;
        for (; x > 0; x = nodes[x].parent)
            nodes[x].last_use = now;
    }

    // Split node c after its first k tokens (0 < k < len); returns the new upper node.
    int32_t split(int32_t c, int32_t k)
    {
        const int32_t u = new_node(nodes[c].parent);
        Node &nu = nodes[u];
        Node &nc = nodes[c];
        nu.tok.assign(nc.tok.begin(), nc.tok.begin() + k);
        nu.slot.assign(nc.slot.begin(), nc.slot.begin() + k);
        nu.depth = nc.depth - (int64_t)(nc.tok.size() - k);
        nu.lock = nc.lock;  // a lock on the old node covered this part too
        nu.last_use = nc.last_use;
        nc.tok.erase(nc.tok.begin(), nc.tok.begin() + k);
        nc.slot.erase(nc.slot.begin(), nc.slot.begin() + k);
        nodes[nu.parent].child[nu.tok[0]] = u;
        nu.child[nc.tok[0]] = c;
        nc.parent = u;
        refresh_best(u);  // u inherits c's value; the parent's is unchanged
        return u;
    }

    // Detach x's ring row (the caller refreshes `best` from x or its parent).
    void detach_ring(int32_t x)
    {
        Node &nx = nodes[x];
        row_held[nx.ring] = 0;
        nx.ring = -1;
        nx.ring_pos.clear();
        --rows_held;
    }
};

extern "C" {

hsa_status hsa_ptree_create(int32_t W, int32_t n_ring_rows, hsa_ptree **out)
{
    if (!out || W <= 0 || n_ring_rows < 0)
        return HSA_INVALID_ARG;
    hsa_ptree *t = new (std::nothrow) hsa_ptree();
    if (!t)
        return HSA_INVALID_ARG;
    t->W = W;
    t->n_rows = n_ring_rows;
    t->row_held.assign((size_t)n_ring_rows, 0);
    t->new_node(-1);  // root: id 0, no tokens
    *out = t;
    return HSA_OK;
}

void hsa_ptree_destroy(hsa_ptree *t) { delete t; }

hsa_status hsa_ptree_match(hsa_ptree *t, const int32_t *tokens, int32_t n, int32_t lock,
                           int32_t take_ring, int32_t *match_len, int32_t *full_slots,
                           int32_t *ring_row, int32_t *swa_slot_pos, int64_t *lock_handle)
{
    if (!t || n < 0 || (n > 0 && (!tokens || !full_slots)) || !match_len || !ring_row ||
        !swa_slot_pos || !lock_handle)
        return HSA_INVALID_ARG;
    const Walk w = t->walk(tokens, n, full_slots);
    *match_len = (int32_t)w.m;
    const int32_t x = t->choose_ring(w);
    if (x >= 0) {
        Node &nx = t->nodes[x];
        *ring_row = nx.ring;
        std::memcpy(swa_slot_pos, nx.ring_pos.data(), sizeof(int32_t) * (size_t)t->W);
        nx.ring_use = ++t->clock;
        if (take_ring) {
            t->detach_ring(x);
            t->refresh_best(x);
        }
    } else {
        *ring_row = -1;
        for (int32_t s = 0; s < t->W; ++s)
            swa_slot_pos[s] = -1;
    }
    *lock_handle = -1;
    if (w.m > 0) {
        t->touch(w.end);
        if (lock) {
            for (int32_t y = w.end; y > 0; y = t->nodes[y].parent)
                ++t->nodes[y].lock;
            *lock_handle = w.end;
        }
    }
    return HSA_OK;
}

hsa_status hsa_ptree_match_batch(hsa_ptree *t, const int32_t *tokens, const int64_t *tok_off,
                                 int32_t n, int32_t *match_len, int32_t *ring_row,
                                 int32_t *swa_slot_pos)
{
    if (!t || n < 0 || (n > 0 && (!tok_off || !match_len || !ring_row || !swa_slot_pos)))
        return HSA_INVALID_ARG;
    for (int32_t k = 0; k < n; ++k) {
        const int64_t len = tok_off[k + 1] - tok_off[k];
        if (tok_off[k] < 0 || len < 0 || (len > 0 && !tokens))
            return HSA_INVALID_ARG;
    }
    for (int32_t k = 0; k < n; ++k) {
        const int64_t len = tok_off[k + 1] - tok_off[k];
        const Walk w = t->walk(tokens + tok_off[k], len, nullptr);
        match_len[k] = (int32_t)w.m;
        const int32_t x = t->choose_ring(w);
        int32_t *pos = swa_slot_pos + (int64_t)k * t->W;
        if (x >= 0) {
            ring_row[k] = t->nodes[x].ring;
            std::memcpy(pos, t->nodes[x].ring_pos.data(), sizeof(int32_t) * (size_t)t->W);
        } else {
            ring_row[k] = -1;
            for (int32_t s = 0; s < t->W; ++s)
                pos[s] = -1;
        }
    }
    return HSA_OK;
}

hsa_status hsa_ptree_insert(hsa_ptree *t, const int32_t *tokens, const int32_t *full_slots,
                            int32_t len, int32_t ring_row, const int32_t *swa_slot_pos,
                            int32_t *dup_slots, int32_t *n_dup, int32_t *ring_kept)
{
    if (!t || len < 0 || (len > 0 && (!tokens || !full_slots || !dup_slots)) || !n_dup ||
        !ring_kept || ring_row < -1 || ring_row >= t->n_rows || (ring_row >= 0 && !swa_slot_pos))
        return HSA_INVALID_ARG;
    *n_dup = 0;
    *ring_kept = 0;
    int32_t cur = 0;
    int64_t pos = 0;
    while (pos < len) {
        auto it = t->nodes[cur].child.find(tokens[pos]);
        if (it == t->nodes[cur].child.end()) {
            const int32_t leaf = t->new_node(cur);
            Node &nl = t->nodes[leaf];
            nl.tok.assign(tokens + pos, tokens + len);
            nl.slot.assign(full_slots + pos, full_slots + len);
            nl.depth = len;
            t->nodes[cur].child[tokens[pos]] = leaf;
            t->cached += len - pos;
            cur = leaf;
            pos = len;
            break;
        }
        const int32_t c = it->second;
        int32_t k = 0;
        {
            const Node &nc = t->nodes[c];
            const int32_t clen = (int32_t)nc.tok.size();
            while (k < clen && pos + k < len && nc.tok[k] == tokens[pos + k]) {
                if (nc.slot[k] != full_slots[pos + k])
                    dup_slots[(*n_dup)++] = full_slots[pos + k];
                ++k;
            }
            if (k == clen) {
                pos += k;
                cur = c;
                continue;
            }
        }
        cur = t->split(c, k);
        pos += k;
    }
    if (len > 0)
        t->touch(cur);
    if (ring_row >= 0 && len > 0 && t->nodes[cur].ring < 0 && !t->row_held[ring_row]) {
        Node &nx = t->nodes[cur];
        nx.ring = ring_row;
        nx.ring_pos.assign(swa_slot_pos, swa_slot_pos + t->W);
        nx.ring_attach = nx.ring_use = ++t->clock;
        t->row_held[ring_row] = 1;
        ++t->rows_held;
        *ring_kept = 1;
        t->refresh_best(cur);
    }
    return HSA_OK;
}

hsa_status hsa_ptree_unlock(hsa_ptree *t, int64_t lock_handle)
{
    if (!t || lock_handle <= 0 || lock_handle >= (int64_t)t->nodes.size() ||
        !t->nodes[lock_handle].alive)
        return HSA_INVALID_ARG;
    for (int32_t y = (int32_t)lock_handle; y > 0; y = t->nodes[y].parent)
        if (t->nodes[y].lock <= 0)
            return HSA_INVALID_ARG;
    for (int32_t y = (int32_t)lock_handle; y > 0; y = t->nodes[y].parent)
        --t->nodes[y].lock;
    return HSA_OK;
}

hsa_status hsa_ptree_evict_full(hsa_ptree *t, int32_t n_tokens, int32_t *freed_slots,
                                int32_t slot_cap, int32_t *n_slots, int32_t *freed_rows,
                                int32_t row_cap, int32_t *n_rows)
{
    if (!t || n_tokens < 0 || slot_cap < 0 || row_cap < 0 || !n_slots || !n_rows ||
        (slot_cap > 0 && !freed_slots) || (row_cap > 0 && !freed_rows))
        return HSA_INVALID_ARG;
    *n_slots = 0;
    *n_rows = 0;
    // Evictable leaves, least recently used first (ties: smaller id).  Evicting a
    // leaf changes no other node's stamp or lock, so the keys stay valid; a parent
    // left without children joins the heap.
    typedef std::pair<uint64_t, int32_t> Key;
    std::priority_queue<Key, std::vector<Key>, std::greater<Key>> heap;
    if (n_tokens > 0)
        for (int32_t x = 1; x < (int32_t)t->nodes.size(); ++x) {
            const Node &nx = t->nodes[x];
            if (nx.alive && nx.lock <= 0 && nx.child.empty())
                heap.push(Key(nx.last_use, x));
        }
    while (*n_slots < n_tokens && !heap.empty()) {
        const int32_t victim = heap.top().second;
        heap.pop();
        Node &nv = t->nodes[victim];
        const int32_t need_rows = nv.ring >= 0 ? 1 : 0;
        if (*n_slots + (int32_t)nv.slot.size() > slot_cap || *n_rows + need_rows > row_cap)
            return *n_slots == 0 && *n_rows == 0 ? HSA_OUT_OF_RANGE : HSA_OK;
        std::memcpy(freed_slots + *n_slots, nv.slot.data(), sizeof(int32_t) * nv.slot.size());
        *n_slots += (int32_t)nv.slot.size();
        if (need_rows) {
            freed_rows[(*n_rows)++] = nv.ring;
            t->detach_ring(victim);
        }
        t->cached -= (int64_t)nv.slot.size();
        const int32_t parent = nv.parent;
        t->nodes[parent].child.erase(nv.tok[0]);
        nv = Node();
        t->free_ids.push_back(victim);
        t->refresh_best(parent);
        const Node &np = t->nodes[parent];
        if (parent > 0 && np.lock <= 0 && np.child.empty())
            heap.push(Key(np.last_use, parent));
    }
    return HSA_OK;
}

hsa_status hsa_ptree_evict_swa(hsa_ptree *t, int32_t n_rows, int32_t *freed_rows,
                               int32_t *n_freed)
{
    if (!t || n_rows < 0 || !n_freed || (n_rows > 0 && !freed_rows))
        return HSA_INVALID_ARG;
    *n_freed = 0;
    if (n_rows == 0)
        return HSA_OK;
    // Rows of unlocked nodes, least recently used first (ties: smaller row id);
    // detaching one changes no other row's stamp.
    std::vector<std::pair<uint64_t, int32_t>> cand;  // (ring_use, ring row) ...
    std::vector<int32_t> holder(t->row_held.size(), -1);
    for (int32_t x = 1; x < (int32_t)t->nodes.size(); ++x) {
        const Node &nx = t->nodes[x];
        if (nx.alive && nx.lock <= 0 && nx.ring >= 0) {
            cand.push_back(std::make_pair(nx.ring_use, nx.ring));
            holder[nx.ring] = x;
        }
    }
    const size_t take = std::min(cand.size(), (size_t)n_rows);
    std::partial_sort(cand.begin(), cand.begin() + take, cand.end());
    for (size_t i = 0; i < take; ++i) {
        const int32_t x = holder[cand[i].second];
        freed_rows[(*n_freed)++] = cand[i].second;
        t->detach_ring(x);
        t->refresh_best(x);
    }
    return HSA_OK;
}

hsa_status hsa_ptree_stats(const hsa_ptree *t, int64_t *cached_tokens, int32_t *rows_held,
                           int32_t *nodes)
{
    if (!t || !cached_tokens || !rows_held || !nodes)
        return HSA_INVALID_ARG;
    *cached_tokens = t->cached;
    *rows_held = t->rows_held;
    *nodes = (int32_t)(t->nodes.size() - t->free_ids.size());
    return HSA_OK;
}

}  // extern "C"

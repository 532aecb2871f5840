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
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
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

    // Ring row for a match ending in node `end`: among the path ends in its subtree
    // (the cached paths through the match point), the shortest path, then the
    // latest attached row, then the smallest row id.  -1 if none.
    int32_t choose_ring(const Walk &w) const
    {
        if (w.m == 0)
            return -1;
        int32_t best = -1;
        std::vector<int32_t> stack(1, w.end);
        while (!stack.empty()) {
            const int32_t x = stack.back();
            stack.pop_back();
            const Node &nx = nodes[x];
            if (nx.ring >= 0) {
                if (best < 0) {
                    best = x;
                } else {
                    const Node &nb = nodes[best];
                    if (nx.depth < nb.depth ||
                        (nx.depth == nb.depth &&
                         (nx.ring_attach > nb.ring_attach ||
                          (nx.ring_attach == nb.ring_attach && nx.ring < nb.ring))))
                        best = x;
                }
            }
            for (const auto &kv : nx.child)
                stack.push_back(kv.second);
        }
        return best;
    }

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
        return u;
    }

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
        if (take_ring)
            t->detach_ring(x);
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
        if (len < 0 || (len > 0 && !tokens))
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
    while (*n_slots < n_tokens) {
        int32_t victim = -1;
        for (int32_t x = 1; x < (int32_t)t->nodes.size(); ++x) {
            const Node &nx = t->nodes[x];
            if (!nx.alive || nx.lock > 0 || !nx.child.empty())
                continue;
            if (victim < 0 || nx.last_use < t->nodes[victim].last_use)
                victim = x;
        }
        if (victim < 0)
            break;
        Node &nv = t->nodes[victim];
        const int32_t need_rows = nv.ring >= 0 ? 1 : 0;
        if (*n_slots + (int32_t)nv.slot.size() > slot_cap || *n_rows + need_rows > row_cap)
            break;
        std::memcpy(freed_slots + *n_slots, nv.slot.data(), sizeof(int32_t) * nv.slot.size());
        *n_slots += (int32_t)nv.slot.size();
        if (need_rows) {
            freed_rows[(*n_rows)++] = nv.ring;
            t->detach_ring(victim);
        }
        t->cached -= (int64_t)nv.slot.size();
        t->nodes[nv.parent].child.erase(nv.tok[0]);
        nv = Node();
        t->free_ids.push_back(victim);
    }
    return HSA_OK;
}

hsa_status hsa_ptree_evict_swa(hsa_ptree *t, int32_t n_rows, int32_t *freed_rows,
                               int32_t *n_freed)
{
    if (!t || n_rows < 0 || !n_freed || (n_rows > 0 && !freed_rows))
        return HSA_INVALID_ARG;
    *n_freed = 0;
    while (*n_freed < n_rows) {
        int32_t victim = -1;
        for (int32_t x = 1; x < (int32_t)t->nodes.size(); ++x) {
            const Node &nx = t->nodes[x];
            if (!nx.alive || nx.lock > 0 || nx.ring < 0)
                continue;
            const Node *nb = victim >= 0 ? &t->nodes[victim] : nullptr;
            if (!nb || nx.ring_use < nb->ring_use ||
                (nx.ring_use == nb->ring_use && nx.ring < nb->ring))
                victim = x;
        }
        if (victim < 0)
            break;
        freed_rows[(*n_freed)++] = t->nodes[victim].ring;
        t->detach_ring(victim);
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

/*
 * hsa_tree.h -- prefix tree with a Full-index / SWA-segment liveness model.
 *
 * What it models [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%",
 * s2 "KVCache系统重构"; hotdry.top "MiMo-V2.5 ultra-speed inference architecture",
 * "Hybrid SWA"]: the scheduler and the prefix tree see one sequence view in which
 * the Full Attention index is authoritative and carries a mapping to the SWA
 * pool; a prefix hit counts only up to the window-safe length (the last W tokens
 * before it still hold valid SWA slots); SWA eviction is tied to the request
 * lifetime, so the SWA pool holds about one window per cached path; every node
 * carries its Full Attention segment index and SWA mapping, and the two are
 * evicted by independent policies.
 *
 * Readings (the pages give the semantics, not the data structure):
 *  - A node holds a run of tokens and, per token, its slot in the Full KV Pool
 *    (physical page * page size + offset).  Those slots are authoritative.
 *  - SWA KV lives in ring rows of W slots (slot = position mod W).  When a request
 *    ends, its ring row holds its last W positions; the row is attached to the
 *    node where its path ends (one row per path end at most).  The row's
 *    swa_slot_pos[W] (position held by each slot, -1 = freed) is kept with it.
 *  - match(T): m = the longest cached prefix of T.  Its ring candidates are the
 *    rows attached at the ends of cached paths that pass through the match point
 *    (their common prefix with T is exactly m).  The chosen row has the shortest
 *    path (ties: the latest attached, then the smallest row id); none when m = 0.
 *    The window-safe length then follows from (m, that row's swa_slot_pos) by the
 *    ring-form rule of hsa_window_safe_len, computed for a whole batch on the GPU.
 *  - Eviction: evict_full removes least-recently-used unlocked leaf nodes (their
 *    Full slots, and their ring row if any, are returned to the caller);
 *    evict_swa detaches least-recently-used ring rows from unlocked nodes and
 *    leaves the Full index in place.
 *
 * Ownership: the tree is host memory owned by the library between create and
 * destroy; every buffer passed in is caller-owned host memory, read or written
 * only during the call.  The tree is not thread-safe: one caller at a time.
 * Errors: HSA_INVALID_ARG for a null handle or pointer, a negative length or
 * offset, or a ring row outside [0, n_ring_rows); HSA_OUT_OF_RANGE from
 * hsa_ptree_evict_full when the first leaf to evict does not fit the caller's
 * buffers (the call then changes nothing).  Output arrays sized by the stated
 * rule ("room for n") are the caller's contract and are not checked.
 * Cost: match O(matched tokens) plus O(1) for the ring choice; insert O(len);
 * the evictions O(nodes + victims * log nodes).
 */
#ifndef HSA_TREE_H
#define HSA_TREE_H

#include <stdint.h>

#include "hsa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hsa_ptree hsa_ptree;

/* A tree for window W and ring rows [0, n_ring_rows).  *out receives the handle. */
hsa_status hsa_ptree_create(int32_t W, int32_t n_ring_rows, hsa_ptree **out);
void hsa_ptree_destroy(hsa_ptree *t);

/*
 * Match one request tokens[0..n).  Writes match_len (m), full_slots[0..m) (the
 * caller passes room for n), ring_row (-1 if none) and swa_slot_pos[0..W) (all -1
 * if no row).  lock != 0 pins the matched path against eviction until
 * hsa_ptree_unlock(*lock_handle) (-1 when nothing was locked).  take_ring != 0
 * detaches the chosen row from the tree: its ownership passes to the caller.
 * The path's last-use stamp is refreshed.
 */
hsa_status hsa_ptree_match(hsa_ptree *t, const int32_t *tokens, int32_t n, int32_t lock,
                           int32_t take_ring, int32_t *match_len, int32_t *full_slots,
                           int32_t *ring_row, int32_t *swa_slot_pos, int64_t *lock_handle);

/*
 * Match a batch without locking or detaching: request k is
 * tokens[tok_off[k] .. tok_off[k+1]).  Writes match_len[n], ring_row[n] and
 * swa_slot_pos[n * W] -- the inputs of hsa_window_safe_len (ring form), which the
 * caller copies to the device to get every request's window-safe length in one
 * launch.
 */
hsa_status hsa_ptree_match_batch(hsa_ptree *t, const int32_t *tokens, const int64_t *tok_off,
                                 int32_t n, int32_t *match_len, int32_t *ring_row,
                                 int32_t *swa_slot_pos);

/*
 * Insert a finished request: tokens[0..len) with their Full slots, and the ring
 * row holding its last window (-1: none) with that row's swa_slot_pos[W].
 * Positions already cached keep the tree's slot; the request's own slot for such
 * a position, when different, is returned in dup_slots (room for len) for the
 * caller to free, *n_dup their count.  *ring_kept = 1 if the row was attached,
 * 0 if the path end already held one (the caller frees the row).
 */
hsa_status hsa_ptree_insert(hsa_ptree *t, const int32_t *tokens, const int32_t *full_slots,
                            int32_t len, int32_t ring_row, const int32_t *swa_slot_pos,
                            int32_t *dup_slots, int32_t *n_dup, int32_t *ring_kept);

/* Release a lock taken by hsa_ptree_match. */
hsa_status hsa_ptree_unlock(hsa_ptree *t, int64_t lock_handle);

/*
 * Evict least-recently-used unlocked leaves until at least n_tokens Full slots
 * are freed or none is evictable.  Freed slots go to freed_slots (room for
 * slot_cap), freed ring rows to freed_rows (room for row_cap); the call stops
 * before a leaf whose slots or row would not fit (HSA_OUT_OF_RANGE if that is the
 * first leaf).  Ties in last use go to the smaller node id.
 */
hsa_status hsa_ptree_evict_full(hsa_ptree *t, int32_t n_tokens, int32_t *freed_slots,
                                int32_t slot_cap, int32_t *n_slots, int32_t *freed_rows,
                                int32_t row_cap, int32_t *n_rows);

/* Detach up to n_rows least-recently-used ring rows of unlocked nodes (last use:
 * attach or last selection by a match; ties go to the smaller row id). */
hsa_status hsa_ptree_evict_swa(hsa_ptree *t, int32_t n_rows, int32_t *freed_rows,
                               int32_t *n_freed);

/* Cached tokens (Full slots held), ring rows held, live nodes (root included). */
hsa_status hsa_ptree_stats(const hsa_ptree *t, int64_t *cached_tokens, int32_t *rows_held,
                           int32_t *nodes);

#ifdef __cplusplus
}
#endif

#endif /* HSA_TREE_H */

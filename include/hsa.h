/*
 * hsa.h -- C ABI of the Hybrid-SWA dual-KV-pool attention library (libhsa.so).
 *
 * The model interleaves sliding-window layers (window W = 128) with full-attention
 * layers (60 : 10 in a 70-layer stack, 6:1).  Full layers keep every token in a
 * paged Full KV Pool that grows on demand; sliding layers keep only the last W
 * tokens of each sequence in a ring-buffer SWA KV Pool (slot = pos mod W), so
 * their storage is O(W).  One unified sequence view: the block table (full index)
 * is authoritative, and the ring row is the mapping into the SWA pool.
 * Sources: youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s1
 * "为什么选择 Hybrid SWA 架构" and s2 "KVCache系统重构"; hotdry.top "MiMo-V2.5
 * ultra-speed inference architecture", "Hybrid SWA" and "三层 KVCache 系统".
 *
 * Conventions shared by every entry point
 *  - All tensors are caller-owned DEVICE memory unless a parameter says "host".
 *    The library never allocates, frees or synchronises; every kernel is queued on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and the call returns
 *    once it is queued.
 *  - bf16 tensors are little-endian IEEE bfloat16, densely packed, row-major, with
 *    the shapes given below; every device pointer must be 16-byte aligned.
 *  - Host-detectable errors are returned synchronously and nothing is launched.
 *    Range errors that only the device can see (a block-table entry outside the
 *    pool, a position past the block table, a ring row outside the ring) are
 *    OR-ed into *dev_err (device int32, caller zeroes it) as HSA_DEVERR_* bits;
 *    the offending item is skipped or its keys treated as absent, never trapped.
 *  - Attention calls never modify the pools; only hsa_kv_append does.
 *  - Attention reads pool positions < cached/prefix length only; the current
 *    step's new tokens are read from k_new/v_new.  For several new tokens on a
 *    sliding layer (MTP verify, prefill chunks) call append AFTER attention:
 *    appending first would overwrite ring slots the earlier queries still need.
 *  - Query head h uses KV head h / (Hq / Hkv).  A sliding-window query at
 *    position p attends positions max(0, p-W+1) .. p (W keys including itself).
 *  - One device per process: the kernels' shared-memory opt-in is set once, on the
 *    device current at a kernel's first call.  In a process that drives several
 *    GPUs a call on another device may be refused with HSA_CUDA_ERROR (the launch
 *    fails; nothing runs).
 */
#ifndef HSA_H
#define HSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int hsa_status;
#define HSA_OK 0
#define HSA_INVALID_ARG 1        /* null pointer, negative size, bad layer index */
#define HSA_UNSUPPORTED_SHAPE 2  /* head_dim != 128, page != 64, W not a multiple of 64, ... */
#define HSA_CUDA_ERROR 3         /* a CUDA runtime call failed (launch, attribute, ...) */
#define HSA_OUT_OF_RANGE 4       /* a caller buffer is too small for the result (host calls) */

/* bits OR-ed into *dev_err by the kernels */
#define HSA_DEVERR_BAD_BLOCK 1   /* block-table entry outside [0, num_blocks) */
#define HSA_DEVERR_BAD_PAGE 2    /* position needs a logical page >= max_blocks */
#define HSA_DEVERR_BAD_SEQ 4     /* sequence index outside [0, batch) */
#define HSA_DEVERR_BAD_RING 8    /* ring row outside [0, n_ring_rows) */
#define HSA_DEVERR_BAD_LEN 16    /* negative length or offsets out of order */
#define HSA_DEVERR_TIMEOUT 32    /* a bounded wait inside a kernel (2 s) gave up: the kernel
                                    stopped early and its outputs are incomplete */

/* FP8 formats of a Full KV Pool layer (hsa_pools.layer_kv_fp8). */
#define HSA_KV_E4M3 1
#define HSA_KV_E5M2 2

/*
 * The dual KV pool of one model (host struct of device pointers).
 *  layer_is_full[l]  host uint8: 1 = full layer (Full KV Pool), 0 = sliding layer.
 *  k[l], v[l]        host arrays of device pointers, one K and one V tensor per layer:
 *                    full layer:    [num_blocks, Hkv, page_size, d] bf16
 *                                   (a block holds page_size consecutive positions;
 *                                   each (block, head) tile is contiguous)
 *                    sliding layer: [n_ring_rows, Hkv, W, d] bf16, slot = pos mod W
 *  block_tables      device int32 [batch, max_blocks]: logical page -> physical block,
 *                    shared by every full layer; entries past a sequence's
 *                    allocation are never read.
 *  ring_row          device int32 [batch]: the SWA ring row of each sequence,
 *                    shared by every sliding layer.
 *  layer_kv_fp8      host uint8 [n_layers] or NULL: HSA_KV_E4M3 (1) or HSA_KV_E5M2
 *                    (2) = this full layer is an FP8 Full KV Pool layer of that
 *                    format, 0 = bf16, any other value HSA_INVALID_ARG
 *                    [hotdry.top "MiMo inference optimization, edge deployment",
 *                    "KV Cache 量化策略的技术选型": FP8 KV (E4M3 / E5M2), quantisation
 *                    groups aligned to the window; "边缘部署的工程权衡与参数清单": the
 *                    newest 128 tokens at the original precision -- a sliding
 *                    layer's ring, which holds exactly those, stays bf16].  Then k[l]
 *                    and v[l] each point to num_blocks * Hkv * 64 * (d + 4) bytes:
 *                    FP8 codes, then one fp32 scale per (block, head, row):
 *                      codes  [num_blocks * Hkv * 64 * d] bytes, then
 *                      scales [num_blocks * Hkv * 64] fp32, index (block*Hkv + h)*64 + row
 *                    K codes: page (block, h) = 64 rows of d bytes; dimension c of a
 *                    row at byte 16*(c/16) + perm16(c%16).  V codes (transposed):
 *                    page (block, h) = d rows of 64 bytes; key row r of dimension c at
 *                    byte 16*(r/16) + perm16(r%16) of row c.
 *                    perm16(l) = 4*((l%8)/2) + (l%2) + 2*(l/8).
 *                    scale = amax / F of the row's d values (fp32 division), F = 448
 *                    (E4M3) or 57344 (E5M2), the format's largest finite magnitude;
 *                    code = FP8 of value / scale (round to nearest even, saturating);
 *                    an all-zero row stores scale 0.  hsa_kv_append and
 *                    hsa_decode_attn_append quantise on write; decode reads such
 *                    layers; prefill rejects them (HSA_UNSUPPORTED_SHAPE), as does a
 *                    sliding layer flagged FP8.  Decode multiplies in fp16 there:
 *                    q, the new rows and |v| * 256 / 448 (E4M3) or |v| * 256 / 57344
 *                    (E5M2) must stay within fp16 range.
 * Supported shape: d = 128, page_size = 64, W a multiple of 64 in [64, 256],
 * Hq a multiple of Hkv with Hq / Hkv in {1, 2, 4, 8}.
 */
typedef struct hsa_pools {
    int32_t n_layers;
    const uint8_t *layer_is_full;
    void *const *k;
    void *const *v;
    int32_t num_blocks;
    int32_t page_size;
    const int32_t *block_tables;
    int32_t max_blocks;
    const int32_t *ring_row;
    int32_t n_ring_rows;
    int32_t batch;
    int32_t W;
    int32_t Hq;
    int32_t Hkv;
    int32_t d;
    const uint8_t *layer_kv_fp8;
} hsa_pools;

/*
 * KV append [youleyou s2 "KVCache系统重构": Full KV Pool grows on demand; SWA KV
 * Pool is a ring buffer of W slots per sequence].
 * Request r appends rows cu_tokens[r] .. cu_tokens[r+1]-1 of k_new / v_new
 * ([ntok, Hkv, d] bf16) to sequence seq_idx[r] at positions start_pos[r] + i.
 *  full layer:    K/V row -> pool[block_tables[seq][pos / page]][h][pos % page]
 *  sliding layer: K/V row -> ring[ring_row[seq]][h][pos % W]; of a request longer
 *                 than W only its last W tokens are written (each slot once),
 *                 which equals appending every token in position order.
 * cu_tokens, seq_idx, start_pos are device int32 arrays; cu_tokens[R] == ntok.
 * A sequence may appear in at most one request per call.
 */
hsa_status hsa_kv_append(const hsa_pools *pools, int32_t layer, const void *k_new,
                         const void *v_new, const int32_t *cu_tokens, const int32_t *seq_idx,
                         const int32_t *start_pos, int32_t R, int32_t ntok,
                         int32_t *dev_err, void *stream);

/*
 * Decode / MTP-verify attention [youleyou s1: decode latency tracks the KV bytes
 * read; s2 "Decode加速与多模态优化": 3-layer MTP, several candidate tokens verified
 * per step].  Sequence b (row b of block_tables / ring_row) has cached_len[b]
 * tokens in the pools and T new tokens at positions cached_len[b] + t, causal
 * among themselves.
 *  q      [B, T, Hq, d] bf16      k_new, v_new [B, T, Hkv, d] bf16
 *  out    [B, T, Hq, d] bf16      cached_len   device int32 [B]
 *  T in 1..4 (else HSA_UNSUPPORTED_SHAPE).  Full layers attend positions 0 .. cached_len+t; sliding layers
 *  attend the last W positions, the cached part read from the ring.
 *  Full layers split each sequence's pages across all SMs (flash-decoding) and
 *  merge the partial softmax states in the same kernel; that needs `workspace`
 *  of at least hsa_decode_workspace_bytes() bytes, ZERO-FILLED ONCE after
 *  allocation (every call leaves it zeroed again).  Calls sharing one workspace
 *  must not run concurrently.  After a call that set any bit in *dev_err, zero
 *  the workspace again before reusing it.
 *  max_ctas: 0 = one persistent CTA per SM (the default); > 0 caps the CTA count
 *  (results do not depend on it beyond rounding).
 */
size_t hsa_decode_workspace_bytes(const hsa_pools *pools, int32_t B, int32_t T);

hsa_status hsa_decode_attn(const hsa_pools *pools, int32_t layer, const void *q,
                           const void *k_new, const void *v_new, const int32_t *cached_len,
                           int32_t B, int32_t T, float scale, void *out, void *workspace,
                           size_t ws_bytes, int32_t max_ctas, int32_t *dev_err, void *stream);

/*
 * Decode attention fused with the append of the step's new tokens (the usual
 * decode step: attend, then keep the new K/V).  Same arguments and outputs as
 * hsa_decode_attn; in addition the T new rows of every sequence are written to
 * this layer's pool at positions cached_len[b] + t (Full KV Pool page through the
 * block table, or ring slot (cached_len[b] + t) mod W), exactly what hsa_kv_append
 * with one request per sequence would write.  Each (sequence, KV head) is appended
 * by the CTA that finishes its attention, after every read of it, so T > 1 on a
 * sliding layer is safe.  For MTP verify where only some drafts are accepted, use
 * hsa_decode_attn and then hsa_kv_append with the accepted tokens instead.
 */
hsa_status hsa_decode_attn_append(const hsa_pools *pools, int32_t layer, const void *q,
                                  const void *k_new, const void *v_new,
                                  const int32_t *cached_len, int32_t B, int32_t T, float scale,
                                  void *out, void *workspace, size_t ws_bytes, int32_t max_ctas,
                                  int32_t *dev_err, void *stream);

/*
 * Decode attention with options (a bit mask; other bits give HSA_INVALID_ARG):
 *  HSA_DECODE_APPEND           append the new rows as hsa_decode_attn_append does.
 *  HSA_DECODE_EARLY_POOL_READ  sliding layers: the kernel starts reading cached_len,
 *      ring_row and this layer's ring before the kernel queued just before it on
 *      `stream` has finished.  The decode kernels are launched with programmatic
 *      dependent launch: they may start once the previous kernel signals its
 *      dependents (this library's decode kernels signal at their start), and they
 *      read q, k_new, v_new and write out / the pools only after it has completed.
 *      With this option the caller guarantees that the kernel just before does not
 *      write cached_len, ring_row or this layer's ring: in a model that kernel is the
 *      layer's QKV projection (it writes q, k_new, v_new only); in a run of decode
 *      calls layer after layer it is the previous layer's attention.  A kernel that
 *      does not signal its dependents early (hsa_kv_append, for one) has completed
 *      before this one starts, so it may write anything.  The option lets the next
 *      layer's ring loads overlap the current layer's kernel (two sliding-layer CTAs
 *      fit on an SM for T <= 2).  Results are those of the same call without it.
 *      Full layers ignore it.
 * Same arguments and results as hsa_decode_attn otherwise.
 */
#define HSA_DECODE_APPEND 1
#define HSA_DECODE_EARLY_POOL_READ 2
hsa_status hsa_decode_attn_ex(const hsa_pools *pools, int32_t layer, const void *q,
                              const void *k_new, const void *v_new, const int32_t *cached_len,
                              int32_t B, int32_t T, float scale, void *out, void *workspace,
                              size_t ws_bytes, int32_t max_ctas, int32_t options,
                              int32_t *dev_err, void *stream);

/*
 * hsa_decode_attn without a caller workspace.  The pages have no counterpart: this
 * is a convenience of this library for callers that cannot allocate device memory
 * where they run decode (while a stream is being captured, inside a host runtime
 * that owns every allocation, or in a loop that must never wait on cudaMalloc).
 * Same arguments and results as hsa_decode_attn minus `workspace` / `ws_bytes`.
 * The scratch is a fixed 8 MiB device array inside libhsa, held by every GPU that
 * loads the library until the process exits; it covers any batch with
 * B * Hkv <= 4096 (larger returns HSA_UNSUPPORTED_SHAPE) and caps the CTA count
 * at what fits (about 250).  This call allocates and frees nothing.
 *  - The first call on a device looks up the array's device address (and may load
 *    the library's device code): make that first call before any stream capture.
 *    The address is kept until the process exits: do not call this again after
 *    cudaDeviceReset (or another teardown of the device's primary context).
 *  - Each call zeroes the counter part of the array on `stream`, then launches.
 *  - All calls share the one array, so calls whose kernels could overlap on the
 *    GPU (different streams, or different host threads) race; serialise them.
 */
hsa_status hsa_decode_attn_noalloc(const hsa_pools *pools, int32_t layer, const void *q,
                                   const void *k_new, const void *v_new,
                                   const int32_t *cached_len, int32_t B, int32_t T, float scale,
                                   void *out, int32_t max_ctas, int32_t *dev_err, void *stream);

/*
 * Chunked prefill on a cached prefix [youleyou s1: SWA cuts prefill compute to
 * the window; hotdry.top "PD 分离与长度分桶": chunked prefill].
 * Request r has prefix_len[r] tokens in the pools of sequence seq_idx[r] and new
 * rows cu_rows[r] .. cu_rows[r+1]-1 at positions prefix_len[r] + i.
 *  q  [rows, Hq, d] bf16     k_new, v_new [rows, Hkv, d] bf16    out [rows, Hq, d] bf16
 *  cu_rows [R+1], prefix_len [R], seq_idx [R]: device int32.
 *  max_chunk: host upper bound on any request's row count (sizes the grid); rows of a
 *  request past the bound it implies are left unwritten, so it must not understate.
 * A sliding layer needs the ring to hold the prefix's last W positions.
 */
hsa_status hsa_prefill_attn(const hsa_pools *pools, int32_t layer, const void *q,
                            const void *k_new, const void *v_new, const int32_t *cu_rows,
                            const int32_t *prefix_len, const int32_t *seq_idx, int32_t R,
                            int32_t rows, int32_t max_chunk, float scale, void *out,
                            int32_t *dev_err, void *stream);

/*
 * Layerwise SWA-KV prefetch [youleyou s2 "KVCache系统重构": the SWA layers' KV is
 * prefetched layer by layer, overlapped with compute, so reading the cache costs
 * almost nothing; hotdry.top "三层 KVCache 系统": host-to-device KV loads overlap the
 * compute stream].  Copies ring rows of sliding layer `layer` from a host tier into
 * the device SWA KV Pool: entry i moves row host_row[i] of host_k / host_v
 * ([n_host_rows, Hkv, W, d] bf16 in PINNED host memory, which the GPU reads
 * directly) into ring row ring_row[seq_idx[i]] of the layer.
 *  host_row, seq_idx: device int32 [n].  Full layers are rejected (HSA_INVALID_ARG),
 *  as is host memory that is not pinned.  Launch it on a side stream ahead of the
 *  attention that reads the layer and order the two with an event.
 */
hsa_status hsa_swa_prefetch(const hsa_pools *pools, int32_t layer, const void *host_k,
                            const void *host_v, int32_t n_host_rows, const int32_t *host_row,
                            const int32_t *seq_idx, int32_t n, int32_t *dev_err, void *stream);

/*
 * Window-safe prefix length [youleyou s2 "KVCache系统重构": a prefix match counts
 * only while the last W tokens still hold valid SWA slots; hotdry.top "Hybrid
 * SWA": the match length is cut back to the window boundary].
 * out_len[k] = the largest L in [0, match_len[k]] such that every position in
 * [max(0, L-W), L) is live.  The full-pool KV is taken as live on [0, match_len).
 *  ring form:   swa_slot_pos [n, W] device int32, the position each ring slot holds
 *               (-1 = freed); position p is live iff swa_slot_pos[p mod W] == p.
 *  bitmap form: live [live_off[n]] device uint8, live_off [n+1] device int64;
 *               position p of case k is live iff live[live_off[k] + p] != 0.
 * match_len, out_len: device int32 [n].  Negative match_len gives 0.
 */
hsa_status hsa_window_safe_len(const int32_t *match_len, const int32_t *swa_slot_pos,
                               int32_t n, int32_t W, int32_t *out_len, void *stream);

hsa_status hsa_window_safe_len_bitmap(const int32_t *match_len, const int64_t *live_off,
                                      const uint8_t *live, int32_t n, int32_t W,
                                      int32_t *out_len, void *stream);

/* Human-readable name of a status code (static string). */
const char *hsa_status_string(hsa_status s);

#ifdef __cplusplus
}
#endif

#endif /* HSA_H */

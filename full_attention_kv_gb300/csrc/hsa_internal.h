// hsa_internal.h -- launch interfaces between the C-ABI layer (api.cu) and the
// kernels.  Host/device shared structs only; no kernel code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/hsa.h"

struct __nv_bfloat16;

namespace hsa {

// The decode parameter struct is passed by value and kept at <= 128 bytes: on
// sm_103a the decode kernel measured 19% slower with the same code when this
// struct grew from 128 to 136 bytes (a different code generation of the hot loop).
struct DecodeParams {
    const __nv_bfloat16 *q;      // [B, T, Hq, d]
    const __nv_bfloat16 *k_new;  // [B, T, Hkv, d]
    const __nv_bfloat16 *v_new;
    const int32_t *cached_len;   // [B]
    const int32_t *block_tables; // [batch, max_blocks]
    const int32_t *ring_row;     // [batch]
    __nv_bfloat16 *out;          // [B, T, Hq, d]
    uint8_t *ws;                 // workspace: arrival counters, then partial softmax states
    int32_t *dev_err;
    uint4 *k_dst;                // this layer's K pool / ring (append only)
    uint4 *v_dst;
    int32_t max_blocks, num_blocks, n_ring_rows;
    int32_t B, Hkv, W;
    int16_t T, G;                // query tokens per sequence; query heads per KV head
    int32_t flags;               // kDecode* bits below
    float scale_log2;            // softmax scale * log2(e)
};
constexpr int32_t kDecodeRing = 1;    // sliding layer: read the SWA ring
constexpr int32_t kDecodeAppend = 2;  // append the T new rows (hsa_decode_attn_append)
constexpr int32_t kDecodeFp8 = 4;     // full layer stored as FP8 codes + scales (fp8_kv.cuh)
constexpr int32_t kDecodeEarly = 8;   // sliding layer: walk and load the ring before the
                                      // grid-dependency wait (HSA_DECODE_EARLY_POOL_READ)
constexpr int32_t kDecodeE5M2 = 16;   // with kDecodeFp8: the codes are E5M2 (else E4M3)
static_assert(sizeof(DecodeParams) <= 128, "keep the decode parameter struct <= 128 bytes");

// Bytes of the arrival-counter region at the start of a decode workspace.
__host__ __device__ inline size_t decode_counter_bytes(int B, int Hkv)
{
    return ((size_t)B * Hkv * sizeof(int32_t) + 255) & ~size_t(255);
}

size_t decode_workspace_bytes(int num_sms, int B, int Hkv);
// Every host-side check of a decode call except the workspace's (api.cu); HSA_OK
// with *done = true means there is nothing to do (B = 0).
hsa_status decode_host_check(const hsa_pools *pools, int32_t layer, const void *q,
                             const void *k_new, const void *v_new, const int32_t *cached_len,
                             int32_t B, int32_t T, const void *out, int32_t max_ctas, bool *done);
cudaError_t launch_decode(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                          int ctas, cudaStream_t stream);

struct AppendParams {
    const uint4 *k_new;          // [ntok, Hkv, d] as 16-byte chunks
    const uint4 *v_new;
    const int32_t *cu_tokens;    // [R+1]
    const int32_t *seq_idx;      // [R]
    const int32_t *start_pos;    // [R]
    uint4 *k_dst;                // layer's K pool / ring
    uint4 *v_dst;
    const int32_t *block_tables;
    const int32_t *ring_row;
    int32_t *dev_err;
    int32_t R, ntok, Hkv, chunks_per_row;  // chunks_per_row = d * 2 / 16
    int32_t batch, max_blocks, num_blocks, page_size, n_ring_rows, W;
    int32_t ring_mode;
    int32_t fp8;                 // full layer stored as FP8 codes + scales (fp8_kv.cuh):
                                 // 0 bf16, 1 E4M3, 2 E5M2
};

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);

// Prefill keeps its larger by-value struct: promoted into registers (<= 128
// bytes) it raised the prefill kernel's spills from 76 to 252 bytes.
struct PrefillParams {
    const __nv_bfloat16 *q;      // [rows, Hq, d]
    const __nv_bfloat16 *k_new;  // [rows, Hkv, d]
    const __nv_bfloat16 *v_new;
    const int32_t *cu_rows;      // [R+1]
    const int32_t *prefix_len;   // [R]
    const int32_t *seq_idx;      // [R]
    const int32_t *block_tables;
    const int32_t *ring_row;
    __nv_bfloat16 *out;          // [rows, Hq, d]
    int32_t *dev_err;
    int32_t R, rows, Hq, Hkv, G, W;
    int32_t batch, max_blocks, num_blocks, n_ring_rows;
    int32_t ring_mode;
    int32_t tiles_per_req_bound; // host upper bound on the total number of 128-row tiles
    float scale_log2;
};

size_t prefill_smem_bytes();
cudaError_t launch_prefill(const CUtensorMap &tmPoolK, const CUtensorMap &tmPoolV,
                           const CUtensorMap &tmNewK, const CUtensorMap &tmNewV,
                           const CUtensorMap &tmQ, const PrefillParams &p, cudaStream_t stream);

// Sliding layers whose window and GQA group fit one key tile (W + 128 / G + 16 <=
// 160 keys: W = 64 or 128 at G = 8, W = 64 at G = 2 or 4) run the persistent
// sliding-window prefill kernel
// (prefill_swa.cu); other sliding shapes run prefill_kernel in ring mode.
bool prefill_swa_supported(int W, int G);
cudaError_t launch_prefill_swa(const CUtensorMap &tmQ, const CUtensorMap &tmNewK,
                               const CUtensorMap &tmNewV, const CUtensorMap &tmRingK,
                               const CUtensorMap &tmRingV, const PrefillParams &p, int sms,
                               cudaStream_t stream);

struct SwaPrefetchParams {
    const uint4 *host_k;         // pinned host ring rows [n_host_rows, Hkv, W, d] (device-visible)
    const uint4 *host_v;
    uint4 *dev_k;                // the layer's device ring [n_ring_rows, Hkv, W, d]
    uint4 *dev_v;
    const int32_t *host_row;     // [n]
    const int32_t *seq_idx;      // [n]
    const int32_t *ring_row;     // [batch]
    int32_t *dev_err;
    int32_t n, n_host_rows, n_ring_rows, batch, Hkv, W, chunks_per_row;
};

cudaError_t launch_swa_prefetch(const SwaPrefetchParams &p, cudaStream_t stream);

cudaError_t launch_window_safe_ring(const int32_t *match_len, const int32_t *slot_pos, int32_t n,
                                    int32_t W, int32_t *out, cudaStream_t stream);
cudaError_t launch_window_safe_bitmap(const int32_t *match_len, const int64_t *live_off,
                                      const uint8_t *live, int32_t n, int32_t W, int32_t *out,
                                      cudaStream_t stream);

}  // namespace hsa

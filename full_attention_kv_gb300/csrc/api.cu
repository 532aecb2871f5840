// api.cu -- the C ABI of libhsa (declared in include/hsa.h).
//
// Host side only: validates arguments, encodes TMA tensor maps for the layer's
// pool tensors, sizes grids and queues kernels on the caller's stream.  It never
// allocates device memory and never synchronises.
#include <algorithm>
#include <mutex>

#include "hsa_internal.h"

namespace {

using hsa::DecodeParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over `rows` rows of `cols` elements with a row pitch of
// `pitch_elems`; box = box_cols x box_rows; 128-byte swizzle.
bool encode_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
               uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over a packed [d2][d1][d0] tensor (d0 = 128 elements);
// box = box0 x box1 x box2; 128-byte swizzle.
bool encode_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t box0, uint32_t box2, uint32_t box1 = 1)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor map (E4M3 codes): rows of `cols` bytes, row pitch `cols`.
bool encode_2d_u8(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                  uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// FP8 format of a layer: 0 bf16, HSA_KV_E4M3, HSA_KV_E5M2 (other values are
// rejected by check_pools)
int layer_fp8(const hsa_pools *p, int32_t layer)
{
    return p->layer_kv_fp8 ? p->layer_kv_fp8[layer] : 0;
}

int device_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

hsa_status check_pools(const hsa_pools *p, int32_t layer)
{
    if (!p || !p->layer_is_full || !p->k || !p->v)
        return HSA_INVALID_ARG;
    if (layer < 0 || layer >= p->n_layers)
        return HSA_INVALID_ARG;
    if (p->d != 128 || p->page_size != 64 || p->W < 64 || p->W > 256 || p->W % 64 != 0)
        return HSA_UNSUPPORTED_SHAPE;
    if (p->Hkv <= 0 || p->Hq <= 0 || p->Hq % p->Hkv != 0)
        return HSA_UNSUPPORTED_SHAPE;
    const int G = p->Hq / p->Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return HSA_UNSUPPORTED_SHAPE;
    if (p->batch < 0 || p->num_blocks < 0 || p->max_blocks < 0 || p->n_ring_rows < 0)
        return HSA_INVALID_ARG;
    if (!p->k[layer] || !p->v[layer] || !aligned16(p->k[layer]) || !aligned16(p->v[layer]))
        return HSA_INVALID_ARG;
    const int fmt = layer_fp8(p, layer);
    if (fmt != 0 && fmt != HSA_KV_E4M3 && fmt != HSA_KV_E5M2)
        return HSA_INVALID_ARG;
    if (fmt && !p->layer_is_full[layer])
        return HSA_UNSUPPORTED_SHAPE;  // the ring (newest W tokens) stays bf16
    if (p->layer_is_full[layer]) {
        if (!p->block_tables || p->num_blocks <= 0 || p->max_blocks <= 0)
            return HSA_INVALID_ARG;
    } else {
        if (!p->ring_row || p->n_ring_rows <= 0)
            return HSA_INVALID_ARG;
    }
    return HSA_OK;
}

}  // namespace

extern "C" {

const char *hsa_status_string(hsa_status s)
{
    switch (s) {
    case HSA_OK:
        return "ok";
    case HSA_INVALID_ARG:
        return "invalid argument";
    case HSA_UNSUPPORTED_SHAPE:
        return "unsupported shape";
    case HSA_CUDA_ERROR:
        return "CUDA error";
    case HSA_OUT_OF_RANGE:
        return "buffer too small";
    default:
        return "unknown status";
    }
}

hsa_status hsa_kv_append(const hsa_pools *pools, int32_t layer, const void *k_new,
                         const void *v_new, const int32_t *cu_tokens, const int32_t *seq_idx,
                         const int32_t *start_pos, int32_t R, int32_t ntok, int32_t *dev_err,
                         void *stream)
{
    hsa_status st = check_pools(pools, layer);
    if (st != HSA_OK)
        return st;
    if (R < 0 || ntok < 0)
        return HSA_INVALID_ARG;
    if (ntok == 0 || R == 0)
        return HSA_OK;
    if (!k_new || !v_new || !cu_tokens || !seq_idx || !start_pos || !aligned16(k_new) ||
        !aligned16(v_new))
        return HSA_INVALID_ARG;
    hsa::AppendParams a{};
    a.k_new = static_cast<const uint4 *>(k_new);
    a.v_new = static_cast<const uint4 *>(v_new);
    a.cu_tokens = cu_tokens;
    a.seq_idx = seq_idx;
    a.start_pos = start_pos;
    a.k_dst = static_cast<uint4 *>(pools->k[layer]);
    a.v_dst = static_cast<uint4 *>(pools->v[layer]);
    a.block_tables = pools->block_tables;
    a.ring_row = pools->ring_row;
    a.dev_err = dev_err;
    a.R = R;
    a.ntok = ntok;
    a.Hkv = pools->Hkv;
    a.chunks_per_row = pools->d * 2 / 16;
    a.batch = pools->batch;
    a.max_blocks = pools->max_blocks;
    a.num_blocks = pools->num_blocks;
    a.page_size = pools->page_size;
    a.n_ring_rows = pools->n_ring_rows;
    a.W = pools->W;
    a.ring_mode = pools->layer_is_full[layer] ? 0 : 1;
    a.fp8 = layer_fp8(pools, layer) == HSA_KV_E5M2 ? 2 : layer_fp8(pools, layer) ? 1 : 0;
    return hsa::launch_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? HSA_OK
                                                                                  : HSA_CUDA_ERROR;
}

size_t hsa_decode_workspace_bytes(const hsa_pools *pools, int32_t B, int32_t T)
{
    (void)T;
    // partial slots for the largest CTA count hsa_decode_attn picks: one per SM
    // (full layers) or one per (sequence, KV head) (sliding layers)
    const int sms = device_sms();
    const int hkv = pools ? pools->Hkv : 0;
    if (B < 0 || hkv <= 0)
        return 0;
    return hsa::decode_workspace_bytes(std::max(sms > 0 ? sms : 1, B * hkv), B, hkv);
}

}  // extern "C"

namespace hsa {

hsa_status decode_host_check(const hsa_pools *pools, int32_t layer, const void *q,
                             const void *k_new, const void *v_new, const int32_t *cached_len,
                             int32_t B, int32_t T, const void *out, int32_t max_ctas, bool *done)
{
    *done = false;
    hsa_status st = check_pools(pools, layer);
    if (st != HSA_OK)
        return st;
    if (B < 0 || T < 1 || max_ctas < 0)
        return HSA_INVALID_ARG;
    const int G = pools->Hq / pools->Hkv;
    if (T > 4 || G * T > 32)
        return HSA_UNSUPPORTED_SHAPE;
    if (B > pools->batch)
        return HSA_INVALID_ARG;
    if (B == 0) {
        *done = true;
        return HSA_OK;
    }
    if (!q || !k_new || !v_new || !cached_len || !out || !aligned16(q) || !aligned16(k_new) ||
        !aligned16(v_new) || !aligned16(out))
        return HSA_INVALID_ARG;
    return HSA_OK;
}

}  // namespace hsa

namespace {

hsa_status decode_common(const hsa_pools *pools, int32_t layer, const void *q, const void *k_new,
                         const void *v_new, const int32_t *cached_len, int32_t B, int32_t T,
                         float scale, void *out, void *workspace, size_t ws_bytes,
                         int32_t max_ctas, int32_t *dev_err, void *stream, int32_t options)
{
    if (options & ~(HSA_DECODE_APPEND | HSA_DECODE_EARLY_POOL_READ))
        return HSA_INVALID_ARG;
    const bool append = (options & HSA_DECODE_APPEND) != 0;
    bool done = false;
    const hsa_status st = hsa::decode_host_check(pools, layer, q, k_new, v_new, cached_len, B, T,
                                                 out, max_ctas, &done);
    if (st != HSA_OK || done)
        return st;
    const int G = pools->Hq / pools->Hkv;
    const bool full = pools->layer_is_full[layer] != 0;
    const int sms = device_sms();
    if (sms <= 0)
        return HSA_CUDA_ERROR;
    int ctas;
    const int units = B * pools->Hkv;
    if (full) {
        ctas = sms;
    } else {
        // one CTA per (sequence, KV head) when that fills the GPU, else split rings
        ctas = units >= sms / 2 ? units : std::min(units * (pools->W / 64), sms);
    }
    if (max_ctas > 0 && ctas > max_ctas)
        ctas = max_ctas;
    const size_t need = hsa::decode_workspace_bytes(ctas, B, pools->Hkv);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return HSA_INVALID_ARG;

    CUtensorMap tmK, tmV;
    const int fmt = layer_fp8(pools, layer);
    const bool fp8 = fmt != 0;
    const uint64_t rows = full ? (uint64_t)pools->num_blocks * pools->Hkv * pools->page_size
                               : (uint64_t)pools->n_ring_rows * pools->Hkv * pools->W;
    if (fp8) {
        // K codes: rows of 128 bytes, a page = box of 64 rows (128-byte swizzle);
        // V codes: transposed pages, rows of 64 bytes, box of 128 rows (64-byte swizzle)
        if (!encode_2d_u8(&tmK, pools->k[layer], 128, rows, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d_u8(&tmV, pools->v[layer], 64, rows * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B))
            return HSA_CUDA_ERROR;
    } else if (!encode_2d(&tmK, pools->k[layer], 128, rows, 128, 64, 64) ||
               !encode_2d(&tmV, pools->v[layer], 128, rows, 128, 64, 64)) {
        return HSA_CUDA_ERROR;
    }

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.cached_len = cached_len;
    p.block_tables = pools->block_tables;
    p.ring_row = pools->ring_row;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.ws = static_cast<uint8_t *>(workspace);
    p.dev_err = dev_err;
    p.k_dst = static_cast<uint4 *>(pools->k[layer]);
    p.v_dst = static_cast<uint4 *>(pools->v[layer]);
    p.max_blocks = pools->max_blocks;
    p.num_blocks = pools->num_blocks;
    p.n_ring_rows = pools->n_ring_rows;
    p.B = B;
    p.Hkv = pools->Hkv;
    p.W = pools->W;
    p.T = (int16_t)T;
    p.G = (int16_t)G;
    p.flags = (full ? 0 : hsa::kDecodeRing) | (append ? hsa::kDecodeAppend : 0) |
              (fp8 ? hsa::kDecodeFp8 : 0) | (fmt == HSA_KV_E5M2 ? hsa::kDecodeE5M2 : 0) |
              ((!full && (options & HSA_DECODE_EARLY_POOL_READ)) ? hsa::kDecodeEarly : 0);
    p.scale_log2 = scale * 1.4426950408889634f;
    return hsa::launch_decode(tmK, tmV, p, ctas, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HSA_OK
               : HSA_CUDA_ERROR;
}

}  // namespace

extern "C" {

hsa_status hsa_decode_attn(const hsa_pools *pools, int32_t layer, const void *q,
                           const void *k_new, const void *v_new, const int32_t *cached_len,
                           int32_t B, int32_t T, float scale, void *out, void *workspace,
                           size_t ws_bytes, int32_t max_ctas, int32_t *dev_err, void *stream)
{
    return decode_common(pools, layer, q, k_new, v_new, cached_len, B, T, scale, out, workspace,
                         ws_bytes, max_ctas, dev_err, stream, 0);
}

hsa_status hsa_decode_attn_append(const hsa_pools *pools, int32_t layer, const void *q,
                                  const void *k_new, const void *v_new,
                                  const int32_t *cached_len, int32_t B, int32_t T, float scale,
                                  void *out, void *workspace, size_t ws_bytes, int32_t max_ctas,
                                  int32_t *dev_err, void *stream)
{
    return decode_common(pools, layer, q, k_new, v_new, cached_len, B, T, scale, out, workspace,
                         ws_bytes, max_ctas, dev_err, stream, HSA_DECODE_APPEND);
}

hsa_status hsa_decode_attn_ex(const hsa_pools *pools, int32_t layer, const void *q,
                              const void *k_new, const void *v_new, const int32_t *cached_len,
                              int32_t B, int32_t T, float scale, void *out, void *workspace,
                              size_t ws_bytes, int32_t max_ctas, int32_t options,
                              int32_t *dev_err, void *stream)
{
    return decode_common(pools, layer, q, k_new, v_new, cached_len, B, T, scale, out, workspace,
                         ws_bytes, max_ctas, dev_err, stream, options);
}

hsa_status hsa_prefill_attn(const hsa_pools *pools, int32_t layer, const void *q,
                            const void *k_new, const void *v_new, const int32_t *cu_rows,
                            const int32_t *prefix_len, const int32_t *seq_idx, int32_t R,
                            int32_t rows, int32_t max_chunk, float scale, void *out,
                            int32_t *dev_err, void *stream)
{
    hsa_status st = check_pools(pools, layer);
    if (st != HSA_OK)
        return st;
    if (layer_fp8(pools, layer))
        return HSA_UNSUPPORTED_SHAPE;  // FP8 pool layers are a decode variant
    if (R < 0 || rows < 0 || max_chunk < 0)
        return HSA_INVALID_ARG;
    if (R == 0 || rows == 0 || max_chunk == 0)
        return HSA_OK;
    if (!q || !k_new || !v_new || !cu_rows || !prefix_len || !seq_idx || !out ||
        !aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return HSA_INVALID_ARG;
    const bool full = pools->layer_is_full[layer] != 0;
    const int G = pools->Hq / pools->Hkv;
    CUtensorMap tmPK, tmPV, tmNK, tmNV, tmQ;
    const uint64_t prow = full ? (uint64_t)pools->num_blocks * pools->Hkv * pools->page_size
                               : (uint64_t)pools->n_ring_rows * pools->Hkv * pools->W;
    const bool swa_kernel = !full && hsa::prefill_swa_supported(pools->W, G);
    if (swa_kernel) {
        // q boxes of 128 / G positions x the G heads of one KV head; K / V boxes of
        // 16 rows (chunk rows, or 16 slots of a ring)
        if (!encode_2d(&tmPK, pools->k[layer], 128, prow, 128, 64, 16) ||
            !encode_2d(&tmPV, pools->v[layer], 128, prow, 128, 64, 16) ||
            !encode_3d(&tmNK, k_new, 128, pools->Hkv, rows, 64, 16) ||
            !encode_3d(&tmNV, v_new, 128, pools->Hkv, rows, 64, 16) ||
            !encode_3d(&tmQ, q, 128, pools->Hq, rows, 64, 128 / G, G))
            return HSA_CUDA_ERROR;
    } else if (!encode_2d(&tmPK, pools->k[layer], 128, prow, 128, 64, 64) ||
        !encode_2d(&tmPV, pools->v[layer], 128, prow, 128, 64, 64) ||
        !encode_3d(&tmNK, k_new, 128, pools->Hkv, rows, 64, 128) ||
        !encode_3d(&tmNV, v_new, 128, pools->Hkv, rows, 64, 128) ||
        !encode_3d(&tmQ, q, 128, pools->Hq, rows, 64, 128))
        return HSA_CUDA_ERROR;
    hsa::PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.cu_rows = cu_rows;
    p.prefix_len = prefix_len;
    p.seq_idx = seq_idx;
    p.block_tables = pools->block_tables;
    p.ring_row = pools->ring_row;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.dev_err = dev_err;
    p.R = R;
    p.rows = rows;
    p.Hq = pools->Hq;
    p.Hkv = pools->Hkv;
    p.G = G;
    p.W = pools->W;
    p.batch = pools->batch;
    p.max_blocks = pools->max_blocks;
    p.num_blocks = pools->num_blocks;
    p.n_ring_rows = pools->n_ring_rows;
    p.ring_mode = full ? 0 : 1;
    // upper bound on sum_r ceil(C_r / 128): CTAs past the real count exit at once
    const int64_t b1 = (int64_t)rows / 128 + R;
    const int64_t b2 = (int64_t)R * ((max_chunk + 127) / 128);
    p.tiles_per_req_bound = (int32_t)std::min(b1, b2);
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaError_t e;
    if (swa_kernel) {
        const int sms = device_sms();
        if (sms <= 0)
            return HSA_CUDA_ERROR;
        e = hsa::launch_prefill_swa(tmQ, tmNK, tmNV, tmPK, tmPV, p, sms,
                                    static_cast<cudaStream_t>(stream));
    } else {
        e = hsa::launch_prefill(tmPK, tmPV, tmNK, tmNV, tmQ, p, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? HSA_OK : HSA_CUDA_ERROR;
}

hsa_status hsa_swa_prefetch(const hsa_pools *pools, int32_t layer, const void *host_k,
                            const void *host_v, int32_t n_host_rows, const int32_t *host_row,
                            const int32_t *seq_idx, int32_t n, int32_t *dev_err, void *stream)
{
    hsa_status st = check_pools(pools, layer);
    if (st != HSA_OK)
        return st;
    if (pools->layer_is_full[layer])
        return HSA_INVALID_ARG;  // only sliding layers have a ring to prefetch
    if (n < 0 || n_host_rows < 0)
        return HSA_INVALID_ARG;
    if (n == 0)
        return HSA_OK;
    if (!host_k || !host_v || !host_row || !seq_idx || !aligned16(host_k) || !aligned16(host_v))
        return HSA_INVALID_ARG;
    // the host tier must be pinned (page-locked) host memory the GPU can address
    void *dk = nullptr, *dv = nullptr;
    if (cudaHostGetDevicePointer(&dk, const_cast<void *>(host_k), 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&dv, const_cast<void *>(host_v), 0) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error the failed query recorded
        return HSA_INVALID_ARG;
    }
    hsa::SwaPrefetchParams p{};
    p.host_k = static_cast<const uint4 *>(dk);
    p.host_v = static_cast<const uint4 *>(dv);
    p.dev_k = static_cast<uint4 *>(pools->k[layer]);
    p.dev_v = static_cast<uint4 *>(pools->v[layer]);
    p.host_row = host_row;
    p.seq_idx = seq_idx;
    p.ring_row = pools->ring_row;
    p.dev_err = dev_err;
    p.n = n;
    p.n_host_rows = n_host_rows;
    p.n_ring_rows = pools->n_ring_rows;
    p.batch = pools->batch;
    p.Hkv = pools->Hkv;
    p.W = pools->W;
    p.chunks_per_row = pools->d * 2 / 16;
    return hsa::launch_swa_prefetch(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HSA_OK
               : HSA_CUDA_ERROR;
}

hsa_status hsa_window_safe_len(const int32_t *match_len, const int32_t *swa_slot_pos, int32_t n,
                               int32_t W, int32_t *out_len, void *stream)
{
    if (n < 0 || W <= 0)
        return HSA_INVALID_ARG;
    if (n == 0)
        return HSA_OK;
    if (!match_len || !swa_slot_pos || !out_len)
        return HSA_INVALID_ARG;
    return hsa::launch_window_safe_ring(match_len, swa_slot_pos, n, W, out_len,
                                        static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HSA_OK
               : HSA_CUDA_ERROR;
}

hsa_status hsa_window_safe_len_bitmap(const int32_t *match_len, const int64_t *live_off,
                                      const uint8_t *live, int32_t n, int32_t W,
                                      int32_t *out_len, void *stream)
{
    if (n < 0 || W <= 0)
        return HSA_INVALID_ARG;
    if (n == 0)
        return HSA_OK;
    if (!match_len || !live_off || !live || !out_len)
        return HSA_INVALID_ARG;
    return hsa::launch_window_safe_bitmap(match_len, live_off, live, n, W, out_len,
                                          static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HSA_OK
               : HSA_CUDA_ERROR;
}

}  // extern "C"

// append.cu -- KV append into the dual pool (sm_103a).
//
// [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s2 "KVCache系统重构"]:
// the Full KV Pool grows on demand (paged: block = block_tables[seq][pos / page],
// row = pos % page) and keeps every token; the SWA KV Pool is a ring of W slots per
// sequence (slot = pos mod W) whose storage never exceeds O(W).
//
// One thread moves one 16-byte chunk of one (token, KV head) row of K and of V, so
// a warp writes two whole 256-byte rows: fully coalesced 16-byte loads and stores.
// For the ring only a request's last W tokens are written, so every slot is
// written once per call (deterministic, race-free) and the result equals
// appending the tokens one by one in position order.
// An FP8 full layer (fp8_kv.cuh) is written by append_fp8_kernel instead: one warp
// per (token, KV head, K or V) row quantises the row to E4M3 or E5M2 codes plus one
// fp32 scale (amax / 448 or amax / 57344, the amax found by a warp reduction) and
// stores them in the page layout.
#include "fp8_kv.cuh"
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p)
{
    const int64_t total = (int64_t)p.ntok * p.Hkv * p.chunks_per_row;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int chunk = (int)(e % p.chunks_per_row);
        const int64_t th = e / p.chunks_per_row;
        const int h = (int)(th % p.Hkv);
        const int tok = (int)(th / p.Hkv);
        // request owning this token: binary search in cu_tokens
        int lo = 0, hi = p.R;  // invariant: cu[lo] <= tok < cu[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.cu_tokens + mid) <= tok)
                lo = mid;
            else
                hi = mid;
        }
        const int r = lo;
        const int first = __ldg(p.cu_tokens + r), last = __ldg(p.cu_tokens + r + 1);
        if (tok < first || tok >= last) {
            set_err(p.dev_err, HSA_DEVERR_BAD_LEN);
            continue;
        }
        const int seq = __ldg(p.seq_idx + r);
        if (seq < 0 || seq >= p.batch) {
            set_err(p.dev_err, HSA_DEVERR_BAD_SEQ);
            continue;
        }
        const int i = tok - first;
        const int64_t pos = (int64_t)__ldg(p.start_pos + r) + i;
        if (pos < 0) {
            set_err(p.dev_err, HSA_DEVERR_BAD_LEN);
            continue;
        }
        int64_t dst_row;  // row index in units of d elements
        if (p.ring_mode) {
            if (i < (last - first) - p.W)
                continue;  // overwritten later in this same request
            const int rr = __ldg(p.ring_row + seq);
            if (rr < 0 || rr >= p.n_ring_rows) {
                set_err(p.dev_err, HSA_DEVERR_BAD_RING);
                continue;
            }
            dst_row = ((int64_t)rr * p.Hkv + h) * p.W + (pos % p.W);
        } else {
            const int64_t page = pos / p.page_size;
            if (page >= p.max_blocks) {
                set_err(p.dev_err, HSA_DEVERR_BAD_PAGE);
                continue;
            }
            const int blk = __ldg(p.block_tables + (int64_t)seq * p.max_blocks + page);
            if (blk < 0 || blk >= p.num_blocks) {
                set_err(p.dev_err, HSA_DEVERR_BAD_BLOCK);
                continue;
            }
            dst_row = ((int64_t)blk * p.Hkv + h) * p.page_size + (pos % p.page_size);
        }
        const int64_t src = ((int64_t)tok * p.Hkv + h) * p.chunks_per_row + chunk;
        const int64_t dst = dst_row * p.chunks_per_row + chunk;
        p.k_dst[dst] = __ldg(p.k_new + src);
        p.v_dst[dst] = __ldg(p.v_new + src);
    }
}

// FP8 Full KV Pool layer: one warp per (token, KV head, K or V) row, quantised
// into the layer's E4M3 or E5M2 codes (fp8_kv.cuh).
__global__ void __launch_bounds__(256) append_fp8_kernel(const AppendParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t total = (int64_t)p.ntok * p.Hkv * 2;
    uint8_t *const kc = reinterpret_cast<uint8_t *>(p.k_dst);
    uint8_t *const vc = reinterpret_cast<uint8_t *>(p.v_dst);
    const int64_t cb = fp8_codes_bytes(p.num_blocks, p.Hkv);
    float *const ks = reinterpret_cast<float *>(kc + cb);
    float *const vs = reinterpret_cast<float *>(vc + cb);
    for (int64_t e = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); e < total;
         e += warps) {
        const int kv = (int)(e & 1);
        const int64_t th = e >> 1;
        const int h = (int)(th % p.Hkv);
        const int tok = (int)(th / p.Hkv);
        int lo = 0, hi = p.R;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.cu_tokens + mid) <= tok)
                lo = mid;
            else
                hi = mid;
        }
        const int first = __ldg(p.cu_tokens + lo), last = __ldg(p.cu_tokens + lo + 1);
        const int seq = __ldg(p.seq_idx + lo);
        const int64_t pos = (int64_t)__ldg(p.start_pos + lo) + (tok - first);
        int err = 0, blk = 0;
        if (tok < first || tok >= last || pos < 0) {
            err = HSA_DEVERR_BAD_LEN;
        } else if (seq < 0 || seq >= p.batch) {
            err = HSA_DEVERR_BAD_SEQ;
        } else if (pos / p.page_size >= p.max_blocks) {
            err = HSA_DEVERR_BAD_PAGE;
        } else {
            blk = __ldg(p.block_tables + (int64_t)seq * p.max_blocks + pos / p.page_size);
            if (blk < 0 || blk >= p.num_blocks)
                err = HSA_DEVERR_BAD_BLOCK;
        }
        if (err) {  // uniform across the warp
            if (lane == 0)
                set_err(p.dev_err, err);
            continue;
        }
        const __nv_bfloat16 *src =
            reinterpret_cast<const __nv_bfloat16 *>(kv ? p.v_new : p.k_new) + ((int64_t)tok * p.Hkv + h) * 128;
        fp8_store_row(src, kv ? vc : kc, kv ? vs : ks, blk, h, p.Hkv, (int)(pos % p.page_size), kv,
                      lane, p.fp8 == 2);
    }
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (p.fp8) {
        const int64_t warps = (int64_t)p.ntok * p.Hkv * 2;
        if (warps == 0)
            return cudaSuccess;
        int64_t blocks = (warps + 7) / 8;
        const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
        if (blocks > cap)
            blocks = cap;
        append_fp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const int64_t total = (int64_t)p.ntok * p.Hkv * p.chunks_per_row;
    if (total == 0)
        return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
    if (blocks > cap)
        blocks = cap;
    append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace hsa

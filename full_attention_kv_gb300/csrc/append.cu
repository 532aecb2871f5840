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

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream)
{
    const int64_t total = (int64_t)p.ntok * p.Hkv * p.chunks_per_row;
    if (total == 0)
        return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
    if (blocks > cap)
        blocks = cap;
    append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace hsa

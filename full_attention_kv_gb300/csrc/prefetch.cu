// prefetch.cu -- layerwise prefetch of SWA KV rings from host memory (sm_103a).
//
// [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s2 "KVCache系统重构":
// the SWA layers' KV can be prefetched layer by layer, fully overlapped with
// compute, so reading the cache costs almost nothing; hotdry.top "MiMo-V2.5
// ultra-speed inference architecture", "三层 KVCache 系统": host-to-device KV loads
// overlap the compute stream.]
//
// A sequence whose SWA KV was moved to host memory keeps, per sliding layer, its
// ring row there ([n_host_rows, Hkv, W, d] bf16, pinned).  Bringing it back for
// layer l is one gather kernel: every thread moves one 16-byte chunk, reading the
// pinned host row directly over NVLink-C2C (no staging copy) and writing the
// device ring row of the destination sequence, with four loads in flight per
// thread.  The caller launches it on a side stream one or more layers ahead of the
// attention that needs it; it keeps to a small grid and no shared memory, so it
// runs beside the attention kernels.
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kUnroll = 4;  // independent 16-byte host loads in flight per thread

__global__ void __launch_bounds__(256) swa_prefetch_kernel(const SwaPrefetchParams p)
{
    const int64_t per_row = (int64_t)p.Hkv * p.W * p.chunks_per_row;  // 16-B chunks per K row
    const int64_t total = (int64_t)p.n * 2 * per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e0 < total;
         e0 += stride * kUnroll) {
        uint4 v[kUnroll];
        int64_t dst[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t e = e0 + u * stride;
            ok[u] = false;
            if (e >= total)
                continue;
            const int64_t within = e % per_row;
            const int kv = (int)((e / per_row) & 1);
            const int i = (int)(e / (2 * per_row));
            const int hr = __ldg(p.host_row + i);
            const int seq = __ldg(p.seq_idx + i);
            if (hr < 0 || hr >= p.n_host_rows || seq < 0 || seq >= p.batch) {
                if (within == 0 && kv == 0)
                    set_err(p.dev_err, hr < 0 || hr >= p.n_host_rows ? HSA_DEVERR_BAD_LEN
                                                                     : HSA_DEVERR_BAD_SEQ);
                continue;
            }
            const int rr = __ldg(p.ring_row + seq);
            if (rr < 0 || rr >= p.n_ring_rows) {
                if (within == 0 && kv == 0)
                    set_err(p.dev_err, HSA_DEVERR_BAD_RING);
                continue;
            }
            const uint4 *src = kv ? p.host_v : p.host_k;
            v[u] = src[(int64_t)hr * per_row + within];
            dst[u] = ((int64_t)rr * per_row + within) * 2 + kv;  // row index, K/V bit
            ok[u] = true;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (ok[u])
                (dst[u] & 1 ? p.dev_v : p.dev_k)[dst[u] >> 1] = v[u];
    }
}

}  // namespace

cudaError_t launch_swa_prefetch(const SwaPrefetchParams &p, cudaStream_t stream)
{
    const int64_t total = (int64_t)p.n * 2 * p.Hkv * p.W * p.chunks_per_row;
    if (total == 0)
        return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about 0.4 CTAs of 8 warps an SM: enough 16-byte loads in flight to fill the host
    // link (~190 GB/s, reached from 64 CTAs up), few enough to leave the attention
    // kernels running beside it their SMs (an all-rings decode step took 6.60 ms with
    // 64 CTAs, 6.84 ms with two an SM; more loads a thread did not help)
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 2 / 5;
    if (blocks > cap)
        blocks = cap;
    swa_prefetch_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace hsa

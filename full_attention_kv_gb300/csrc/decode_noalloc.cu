// decode_noalloc.cu -- hsa_decode_attn_noalloc: decode attention whose scratch
// memory lives in a fixed, library-owned device array instead of a caller buffer.
//
// Why it exists: hsa_decode_attn needs a workspace (split-softmax partials and
// per-unit arrival counters) that the caller allocates.  Some callers cannot
// allocate device memory at the point where they run decode: code that runs while
// a CUDA stream is being captured into a graph (cudaMalloc is not allowed during
// capture), plug-ins hosted by a runtime that owns every device allocation and
// exposes no allocator, and latency-critical loops that must not risk an
// allocation failure or the device-wide synchronisation cudaMalloc may cause.
// For them this entry point uses a file-scope device array, sized once at build
// time, that every GPU loading the library keeps until the process exits.
#include <algorithm>
#include <mutex>

#include "hsa_internal.h"

namespace {

// 8 MiB: arrival counters for every (sequence, KV head) unit plus two partial
// softmax slots per CTA.  At B * Hkv = 4096 units the counters take 16 KiB and the
// rest holds partials for 250 CTAs (a full GB300 uses 152 on full layers).
constexpr size_t kScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per
// device (the first call on a device may load this module's device code).  The
// address is kept for the life of the process: it stays valid while the device's
// context lives, so the entry point must not be called again after cudaDeviceReset
// (or any teardown of the primary context) in the same process.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" hsa_status hsa_decode_attn_noalloc(const hsa_pools *pools, int32_t layer,
                                              const void *q, const void *k_new,
                                              const void *v_new, const int32_t *cached_len,
                                              int32_t B, int32_t T, float scale, void *out,
                                              int32_t max_ctas, int32_t *dev_err, void *stream)
{
    // every host argument check first: a call refused for its arguments queues
    // nothing, not even the memset (a CUDA failure further on -- the symbol lookup,
    // tensor-map encoding or the launch -- may leave the counter reset queued, which
    // only zeroes counters)
    bool done = false;
    const hsa_status st = hsa::decode_host_check(pools, layer, q, k_new, v_new, cached_len, B, T,
                                                 out, max_ctas, &done);
    if (st != HSA_OK || done)
        return st;
    // CTA cap so that the counters and every CTA's partial slots fit the array
    if ((int64_t)B * pools->Hkv > 4096)
        return HSA_UNSUPPORTED_SHAPE;  // more units than the fixed scratch is sized for
    const size_t base = hsa::decode_workspace_bytes(0, B, pools->Hkv);
    const size_t per_cta = hsa::decode_workspace_bytes(1, B, pools->Hkv) - base;
    const int64_t cap = (int64_t)((kScratchBytes - base) / per_cta);
    int32_t ctas = max_ctas > 0 ? max_ctas : (int32_t)std::min<int64_t>(cap, 1 << 30);
    if (ctas > cap)
        ctas = (int32_t)cap;

    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return HSA_CUDA_ERROR;
    // the counters must start at zero; the array keeps whatever the last call left
    const size_t cnt_bytes = hsa::decode_counter_bytes(B, pools->Hkv);
    if (cudaMemsetAsync(scratch, 0, cnt_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HSA_CUDA_ERROR;
    return hsa_decode_attn(pools, layer, q, k_new, v_new, cached_len, B, T, scale, out, scratch,
                           kScratchBytes, ctas, dev_err, stream);
}

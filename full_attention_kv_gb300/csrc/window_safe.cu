// window_safe.cu -- window-safe prefix length (sm_103a).
//
// [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s2 "KVCache系统重构":
// a prefix match is reusable only while the last W tokens still hold valid SWA
// slots; hotdry.top "MiMo-V2.5 ultra-speed inference architecture", "Hybrid SWA":
// the match length is cut back to the window boundary.]
// Answer for a case: the largest L in [0, m] with every position of
// [max(0, L-W), L) live.
//
// One warp per case walks down from m in 32-position chunks (one ballot each).
// It keeps `top`, the best candidate so far (m, then the lowest dead position
// seen), and `run`, the number of live positions directly below `top`.  `top`
// is safe as soon as run reaches W or the walk passes position 0.  Within a chunk
// only the highest and lowest dead positions matter when W > 32 (no run of W fits
// between two dead positions of one chunk); for W <= 32 every dead position of the
// chunk is visited.  The ring form needs at most W positions of work near the top
// because everything outside the ring's W positions is dead: the walk jumps from
// m straight to the newest ring position.
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

template <typename Live>
__device__ int32_t safe_len_warp(int32_t m, int32_t W, int64_t floor_dead, Live live)
{
    // floor_dead: every position in [floor_dead, m) is known dead (or -1 = unknown)
    const int lane = threadIdx.x & 31;
    if (m <= 0)
        return 0;
    int64_t top = m;
    int64_t run = 0;
    int64_t hi = m;  // positions [0, hi) not yet examined
    if (floor_dead >= 0 && floor_dead < m) {
        // positions floor_dead .. m-1 are all dead: the lowest of them is the candidate
        top = floor_dead;
        hi = floor_dead;
    }
    while (hi > 0) {
        const int64_t base = hi >= 32 ? hi - 32 : 0;
        const int n = (int)(hi - base);
        const int64_t pos = base + lane;
        const bool dead = lane < n && !live(pos);
        const uint32_t dm = __ballot_sync(0xffffffffu, dead);  // bit i = position base + i
        if (dm == 0) {
            if (run + n >= W)
                return (int32_t)top;
            run += n;
        } else if (W > 32) {
            const int hb = 31 - __clz(dm);  // highest dead bit
            if (run + (n - 1 - hb) >= W)
                return (int32_t)top;
            const int lb = __ffs(dm) - 1;   // lowest dead bit
            top = base + lb;
            run = lb;
        } else {
            uint32_t rest = dm;
            int above = n;  // bits below `above` not yet consumed
            while (rest) {
                const int hb = 31 - __clz(rest);
                if (run + (above - 1 - hb) >= W)
                    return (int32_t)top;
                top = base + hb;
                run = 0;
                above = hb;
                rest &= ~(1u << hb);
            }
            run = above;
            if (run >= W)
                return (int32_t)top;
        }
        hi = base;
    }
    return (int32_t)top;  // the walk passed position 0: [0, top) is all live
}

__global__ void window_safe_ring_kernel(const int32_t *match_len, const int32_t *slot_pos,
                                        int32_t n, int32_t W, int32_t *out)
{
    const int warps = blockDim.x >> 5;
    const int64_t k = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    if (k >= n)
        return;
    const int lane = threadIdx.x & 31;
    const int32_t *sp = slot_pos + k * W;
    const int32_t m = match_len[k];
    // newest position the ring holds: everything at or above newest+1 is dead
    int32_t newest = -1;
    for (int j = lane; j < W; j += 32) {
        const int32_t v = __ldg(sp + j);
        if (v >= 0 && v % W == j && v > newest)
            newest = v;
    }
    for (int o = 16; o > 0; o >>= 1)
        newest = max(newest, __shfl_xor_sync(0xffffffffu, newest, o));
    auto live = [&](int64_t p) -> bool { return __ldg(sp + (p % W)) == p; };
    const int32_t L = safe_len_warp(m, W, (int64_t)newest + 1, live);
    if (lane == 0)
        out[k] = L;
}

__global__ void window_safe_bitmap_kernel(const int32_t *match_len, const int64_t *live_off,
                                          const uint8_t *live_bytes, int32_t n, int32_t W,
                                          int32_t *out)
{
    const int warps = blockDim.x >> 5;
    const int64_t k = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    if (k >= n)
        return;
    const uint8_t *lv = live_bytes + live_off[k];
    const int64_t have = live_off[k + 1] - live_off[k];  // positions past the bitmap: dead
    auto live = [&](int64_t p) -> bool { return p < have && __ldg(lv + p) != 0; };
    const int32_t L = safe_len_warp(match_len[k], W, -1, live);
    if ((threadIdx.x & 31) == 0)
        out[k] = L;
}

}  // namespace

cudaError_t launch_window_safe_ring(const int32_t *match_len, const int32_t *slot_pos, int32_t n,
                                    int32_t W, int32_t *out, cudaStream_t stream)
{
    if (n == 0)
        return cudaSuccess;
    const int warps = 8;
    window_safe_ring_kernel<<<(n + warps - 1) / warps, warps * 32, 0, stream>>>(match_len,
                                                                                 slot_pos, n, W, out);
    return cudaGetLastError();
}

cudaError_t launch_window_safe_bitmap(const int32_t *match_len, const int64_t *live_off,
                                      const uint8_t *live, int32_t n, int32_t W, int32_t *out,
                                      cudaStream_t stream)
{
    if (n == 0)
        return cudaSuccess;
    const int warps = 8;
    window_safe_bitmap_kernel<<<(n + warps - 1) / warps, warps * 32, 0, stream>>>(
        match_len, live_off, live, n, W, out);
    return cudaGetLastError();
}

}  // namespace hsa

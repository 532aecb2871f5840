// decode.cu -- decode / MTP-verify attention over the dual KV pool (sm_103a).
//
// What it computes [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s1
// "为什么选择 Hybrid SWA 架构": decode latency tracks the KV bytes read; s2
// "KVCache系统重构": Full KV Pool paged and growing, SWA KV Pool a W-slot ring; s2
// "Decode加速与多模态优化": MTP verifies several candidate tokens per step]:
// for sequence b, KV head h and query row (t, hh) at position c_b + t,
//   o = softmax(scale * q . K^T) V over the visible keys,
// full layers: positions 0 .. c_b + t; sliding layers: c_b + t - W + 1 .. c_b + t.
// Cached keys come from the pool (block table or ring row), the T new keys from
// k_new / v_new.
//
// Design (one kernel per layer, persistent, one CTA per SM):
//  * Work items are 64-key tiles: one page of the Full KV Pool, or one half of a
//    128-slot ring row.  Items of all (sequence, KV head) units are laid end to
//    end and cut into equal contiguous ranges, one per CTA (flash-decoding with
//    perfect balance whatever the length mix).
//  * A producer warp streams each tile's K and V (2 x 16 KB bf16; FP8 codes plus
//    their scales for an FP8 full layer) into a shared-memory stage ring with TMA
//    (128-byte swizzle), mbarrier-tracked; 4 stages bf16, 8 FP8.  It flags per stage
//    whether a tile was loaded and reads the next block-table entry before waiting
//    for a free stage (FP8 layers: 32 entries at a time, one per lane, a batch ahead).
//  * Four consumer warps (eight in the FP8 loop below) run tiles on tensor cores
//    (mma.sync m16n8k16, fp32 accumulate).  GQA packing: the G query heads x T
//    tokens that share a KV head form the M dimension (row = t * G + hh), so each KV
//    byte is read once for all of them; MT = 1 (T <= 2) or 2 (T = 3, 4) 16-row
//    m-tiles.  Full layers: 4 / MT
//    groups of MT warps, a group taking every (4 / MT)-th tile with all 64 keys, so
//    several tiles are in flight.  Rings: two groups, one per tile of a unit.  Online
//    softmax in registers (exp2, quad shuffles).
//  * T = 1 special cases with the operands swapped (keys on the MMA's M side, the
//    unit's <= 8 query heads on N): a sliding layer's whole unit with a full ring
//    (the new token overwrites the staged row of the one slot its query no longer
//    sees, so no mask and no new-token tile remain), and FP8 full layers (eight
//    consumer warps, a 64-key tile each, the new token merged as one more key).
//  * At the end of a unit the warps merge their softmax states through shared
//    memory.  A unit covered by one CTA is written straight to `out`; a unit split
//    across CTAs leaves (m, l, o) partials in the workspace and the last CTA to
//    finish it (atomic counter, no waiting) merges them and resets the counter.
//  * Optionally (hsa_decode_attn_append) the CTA that completes a unit also appends
//    the unit's new K/V rows to the pool or ring: every read of that unit is done
//    by then, so even a T > 1 ring write cannot clobber a slot still being read.
//    (The T = 1 full-ring path appends as soon as its tile is staged: the slot it
//    writes holds a position no query of the step sees.)
//  * Launched with programmatic dependent launch: nothing global is read before
//    griddepcontrol.wait (except, with kDecodeEarly, a sliding layer's item walk and
//    ring loads), so the launch and prologue overlap the previous kernel.
#include "fp8_kv.cuh"
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kTileKeys = 64;
constexpr int kD = 128;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
// FP8 full layers at T = 1 with at most 8 query heads a KV head run eight consumer
// warps (operands swapped, fewer registers a thread: see the consumer loop)
constexpr int kSwWarps = 8;
constexpr int kMaxThreads = (kSwWarps + 1) * 32;
constexpr int kTileBytes = kTileKeys * kD * 2;  // 16 KB: one K or V tile
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kMaxRows = 32;                    // G * T
constexpr int kNewRows = 16;                    // new-token tile (T <= 4 used)
constexpr int kCombFloats = 16 + 16 + 16 * kD;  // per warp: m, l, o[16][128]
constexpr int kHs = kD + 4;                     // swapped layouts: o[head][dim] row stride
constexpr int kSwFloats = 16 + 8 * kHs;         // swapped layouts, per warp: m[8], l[8], o[8][132]
constexpr int kCombStride = (kSwWarps * kSwFloats + kConsumerWarps - 1) / kConsumerWarps;
static_assert(kCombStride >= kCombFloats && kCombStride % 4 == 0, "merge buffer layout");
constexpr int kPartFloats = kMaxRows * (kD + 2);
// FP8 full layers (fp8_kv.cuh): a stage holds the tile's E4M3 K (64 x 128 B,
// 128-byte swizzle), transposed V (128 x 64 B, 64-byte swizzle) and the two rows
// of 64 fp32 scales; half the bytes of a bf16 stage, so more stages fit in the
// same shared memory and as many bytes stay in flight.
constexpr int kFp8Stages = 8;
constexpr int kFp8StageStride = 17408;  // 16.5 KB rounded up to 1 KB (swizzle alignment)
constexpr int kFp8TileBytes = kTileKeys * kD;  // 8 KB
constexpr int kMaxStages = 8;
// One stage region serves both layouts.  Tile-parallel consumer groups (group g
// runs items k = g mod groups) need a stage count that is a multiple of the group
// count, so that stage k mod S always belongs to the same group: a group that
// skips ahead must never wait on a stage whose earlier phase another group has not
// consumed yet (the mbarrier parity bit cannot tell two phases apart).
constexpr int kStageRegion = kFp8Stages * kFp8StageStride > kStages * kStageBytes
                                 ? kFp8Stages * kFp8StageStride
                                 : kStages * kStageBytes;
// Sliding layers (a unit is at most the ring's two 64-key tiles) run a kernel of
// their own with two stages: ~107 KB of shared memory and (T <= 2) <= 168 registers
// a thread, so two CTAs fit on an SM and the next layer's CTAs can be resident --
// and load their rings -- while this layer's run.
constexpr int kRingStages = 2;
constexpr int kRingStageRegion = kRingStages * kStageBytes;

template <int kRegion>
struct SharedStorageT {
    alignas(1024) uint8_t stage[kRegion];  // bf16: [K lo|K hi|V lo|V hi] per stage
    alignas(16) uint8_t new_k[kNewRows * kD * 2];
    alignas(16) uint8_t new_v[kNewRows * kD * 2];
    alignas(16) float comb[kConsumerWarps][kCombStride];  // also kSwWarps x kSwFloats
    float mscale[kMaxRows][kConsumerWarps];  // merge: each slice's weight per row
    float mrow[kMaxRows][2];                 // merge: each row's combined max and sum
    alignas(8) uint64_t full[kMaxStages];
    alignas(8) uint64_t empty[kMaxStages];
    int32_t tile_ok[kMaxStages];  // the producer loaded the stage's tile (else: masked)
    int32_t scan[kMaxThreads];
    int32_t first_b;
    int32_t first_items_before;  // items of all units of sequences < first_b (per KV head)
    int32_t total_items;         // per KV head sum
    int32_t is_last;
};

struct Walk {
    // position in the flattened item space: sequence b, head h, tile j of n
    int b, h, j, n, c;
};

__device__ __forceinline__ int clamp_len(int c) { return c < 0 ? 0 : c; }

__device__ __forceinline__ int items_of(const DecodeParams &p, int b)
{
    int c = clamp_len(__ldg(p.cached_len + b));
    int keys = (p.flags & kDecodeRing) ? min(c, p.W) : c;
    int n = (keys + kTileKeys - 1) / kTileKeys;
    return n > 0 ? n : 1;
}

__device__ __forceinline__ void walk_load(const DecodeParams &p, Walk &w)
{
    w.c = clamp_len(__ldg(p.cached_len + w.b));
    int keys = (p.flags & kDecodeRing) ? min(w.c, p.W) : w.c;
    int n = (keys + kTileKeys - 1) / kTileKeys;
    w.n = n > 0 ? n : 1;
}

__device__ __forceinline__ void walk_next(const DecodeParams &p, Walk &w)
{
    if (++w.j == w.n) {
        w.j = 0;
        if (++w.h == p.Hkv) {
            w.h = 0;
            ++w.b;
            if (w.b < p.B)
                walk_load(p, w);
        }
    }
}

// TMA row coordinate of tile (b, h, j), or -1 if the tile holds no cached keys or
// its address is out of range (flagged in dev_err by the producer only).
__device__ __forceinline__ int64_t tile_row(const DecodeParams &p, const Walk &w, bool report)
{
    if (w.c == 0)
        return -1;
    if (p.flags & kDecodeRing) {
        int rr = __ldg(p.ring_row + w.b);
        if (rr < 0 || rr >= p.n_ring_rows) {
            if (report)
                set_err(p.dev_err, HSA_DEVERR_BAD_RING);
            return -1;
        }
        return ((int64_t)rr * p.Hkv + w.h) * p.W + (int64_t)w.j * kTileKeys;
    }
    if (w.j >= p.max_blocks) {
        if (report)
            set_err(p.dev_err, HSA_DEVERR_BAD_PAGE);
        return -1;
    }
    int blk = __ldg(p.block_tables + (int64_t)w.b * p.max_blocks + w.j);
    if (blk < 0 || blk >= p.num_blocks) {
        if (report)
            set_err(p.dev_err, HSA_DEVERR_BAD_BLOCK);
        return -1;
    }
    return ((int64_t)blk * p.Hkv + w.h) * kTileKeys;
}

// Per-warp attention state for one m-tile of 16 query rows.
struct RowState {
    float o[kD / 8][4];
    float m[2];
    float l[2];
};

// Running max may lag the true one by up to this much (log2 units) before O is
// rescaled: P then stays below 2^8, exact enough in bf16, and most tiles skip the
// 64-register rescale of O.
constexpr float kRescaleSlack = 8.0f;

// m16n8k16 MMA and operand packing in bf16, or fp16 when F16 is set.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    if (F16)
        mma_f16_16816(d, a, b0, b1);
    else
        mma_bf16_16816(d, a, b0, b1);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi)
{
    return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}

// One key tile on tensor cores.  NT = n-tiles of 8 keys this warp owns inside the
// tile (keys key0 .. key0 + 8 NT - 1), rows = the tile's row count in shared
// memory (for the swizzle), vis(row, key) = key visible to that query row; when
// all_vis is set every key of the tile is visible to every valid row and only rows
// past G T (padding) are masked.
// F16: the operands (Q fragments and the tile in shared memory) are fp16 instead
// of bf16 (the FP8 kernel's new-token tile).
template <int NT, bool F16 = false, typename Vis>
__device__ __forceinline__ void run_tile(RowState &st, const uint32_t (&qa)[kD / 16][4],
                                         uint32_t sK, uint32_t sV, int tile_rows, int key0,
                                         float scale_log2, bool all_vis, bool row0_ok,
                                         bool row1_ok, Vis vis)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;

    // S = Q K^T: B fragments via ldmatrix (rows = keys, cols = dims)
    {
        const int mi = lane >> 3, r = lane & 7;
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const int key = key0 + np * 16 + (mi >> 1) * 8 + r;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const int dim = ks * 16 + (mi & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(sK + swz128_offset(key, dim, tile_rows), b0, b1, b2, b3);
                mma16816<F16>(s[2 * np], qa[ks], b0, b1);
                mma16816<F16>(s[2 * np + 1], qa[ks], b2, b3);
            }
        }
    }

    // mask (raw scores; the scale is positive and folded into the exponent below)
    if (!all_vis) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = key0 + nt * 8 + 2 * tq + e;
                if (!vis(g, key))
                    s[nt][e] = -INFINITY;
                if (!vis(g + 8, key))
                    s[nt][2 + e] = -INFINITY;
            }
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (!row0_ok)
                s[nt][0] = s[nt][1] = -INFINITY;
            if (!row1_ok)
                s[nt][2] = s[nt][3] = -INFINITY;
        }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    mx0 *= scale_log2;
    mx1 *= scale_log2;
    // running max, raised lazily (the quad shares a row, so its decision is uniform)
    const bool up0 = mx0 != -INFINITY && (st.m[0] == -INFINITY || mx0 > st.m[0] + kRescaleSlack);
    const bool up1 = mx1 != -INFINITY && (st.m[1] == -INFINITY || mx1 > st.m[1] + kRescaleSlack);
    if (__any_sync(0xffffffffu, up0 || up1)) {
        const float a0 = up0 ? fast_exp2(st.m[0] - mx0) : 1.f;  // m = -inf: O is still 0
        const float a1 = up1 ? fast_exp2(st.m[1] - mx1) : 1.f;
        if (up0)
            st.m[0] = mx0;
        if (up1)
            st.m[1] = mx1;
        st.l[0] *= a0;
        st.l[1] *= a1;
#pragma unroll
        for (int n = 0; n < kD / 8; ++n) {
            st.o[n][0] *= a0;
            st.o[n][1] *= a0;
            st.o[n][2] *= a1;
            st.o[n][3] *= a1;
        }
    }
    const float base0 = st.m[0] == -INFINITY ? 0.f : st.m[0];
    const float base1 = st.m[1] == -INFINITY ? 0.f : st.m[1];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = fast_exp2(fmaf(s[nt][0], scale_log2, -base0));
        s[nt][1] = fast_exp2(fmaf(s[nt][1], scale_log2, -base0));
        s[nt][2] = fast_exp2(fmaf(s[nt][2], scale_log2, -base1));
        s[nt][3] = fast_exp2(fmaf(s[nt][3], scale_log2, -base1));
    }

    // O += P V: P from the S accumulators, V fragments via ldmatrix.trans.  The row
    // sums take the same bf16-rounded P the MMA uses, so O / l is an exact convex
    // combination of V rows (no scale error proportional to |O|).
    const int mi = lane >> 3, r = lane & 7;
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < NT / 2; ++ks) {
        uint32_t pa[4];
        pa[0] = pack16<F16>(s[2 * ks][0], s[2 * ks][1]);
        pa[1] = pack16<F16>(s[2 * ks][2], s[2 * ks][3]);
        pa[2] = pack16<F16>(s[2 * ks + 1][0], s[2 * ks + 1][1]);
        pa[3] = pack16<F16>(s[2 * ks + 1][2], s[2 * ks + 1][3]);
        if constexpr (F16) {
            sum0 += f16_lo(pa[0]) + f16_hi(pa[0]) + f16_lo(pa[2]) + f16_hi(pa[2]);
            sum1 += f16_lo(pa[1]) + f16_hi(pa[1]) + f16_lo(pa[3]) + f16_hi(pa[3]);
        } else {
            sum0 += bf16_lo(pa[0]) + bf16_hi(pa[0]) + bf16_lo(pa[2]) + bf16_hi(pa[2]);
            sum1 += bf16_lo(pa[1]) + bf16_hi(pa[1]) + bf16_lo(pa[3]) + bf16_hi(pa[3]);
        }
        const int key = key0 + ks * 16 + (mi & 1) * 8 + r;
#pragma unroll
        for (int np = 0; np < kD / 16; ++np) {
            const int dim = np * 16 + (mi >> 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(sV + swz128_offset(key, dim, tile_rows), b0, b1, b2, b3);
            mma16816<F16>(st.o[2 * np], pa, b0, b1);
            mma16816<F16>(st.o[2 * np + 1], pa, b2, b3);
        }
    }
    st.l[0] += sum0;
    st.l[1] += sum1;
}

// One key tile of an FP8 full layer (fp8_kv.cuh layout) on tensor cores, fp16
// MMAs.  K: one 32-bit shared load per (key, 16-dim step) holds a thread's four
// codes of the B fragment, converted exactly to fp16 (E4M3: cvt; E5M2: a byte
// permute, an E5M2 code being the high byte of its fp16); the key's scale is then
// applied to its S column.  V (stored transposed): one 32-bit load per (dimension,
// 16-key step); each key's scale is folded into P, while the row sum takes P
// itself.  An E5M2 scale (amax / 57344) is folded in times 256, so that the fp16 P
// stays clear of fp16's subnormals; the accumulator then holds 256 O, which the
// kernel divides out at the end of the unit.  qa holds fp16 Q fragments.
template <int NT, bool E5M2, typename Vis>
__device__ __forceinline__ void run_tile_fp8(RowState &st, const uint32_t (&qa)[kD / 16][4],
                                             const uint8_t *sK, const uint8_t *sV,
                                             const float *k_scale, const float *v_scale, int key0,
                                             float scale_log2, bool all_vis, bool row0_ok,
                                             bool row1_ok, Vis vis)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    // plain shared-memory loads (ordered after the stage's barrier wait, free to be
    // scheduled early within the tile); two accumulator chains per n-tile (even and
    // odd k-steps) halve the dependent MMA chain
    float s[NT][4], s2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int key = key0 + nt * 8 + g;
        const uint8_t *row = sK + key * 128 + 4 * tq;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(row + ((ks ^ (key & 7)) << 4));
            mma_f16_16816((ks & 1) ? s2[nt] : s[nt], qa[ks], fp8x2_lo<E5M2>(w), fp8x2_hi<E5M2>(w));
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            s[nt][e] += s2[nt][e];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float ksc = k_scale[key0 + nt * 8 + 2 * tq + e];
            s[nt][e] *= ksc;
            s[nt][2 + e] *= ksc;
        }
    }
    if (!all_vis) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = key0 + nt * 8 + 2 * tq + e;
                if (!vis(g, key))
                    s[nt][e] = -INFINITY;
                if (!vis(g + 8, key))
                    s[nt][2 + e] = -INFINITY;
            }
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (!row0_ok)
                s[nt][0] = s[nt][1] = -INFINITY;
            if (!row1_ok)
                s[nt][2] = s[nt][3] = -INFINITY;
        }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    mx0 *= scale_log2;
    mx1 *= scale_log2;
    const bool up0 = mx0 != -INFINITY && (st.m[0] == -INFINITY || mx0 > st.m[0] + kRescaleSlack);
    const bool up1 = mx1 != -INFINITY && (st.m[1] == -INFINITY || mx1 > st.m[1] + kRescaleSlack);
    if (__any_sync(0xffffffffu, up0 || up1)) {
        const float a0 = up0 ? fast_exp2(st.m[0] - mx0) : 1.f;
        const float a1 = up1 ? fast_exp2(st.m[1] - mx1) : 1.f;
        if (up0)
            st.m[0] = mx0;
        if (up1)
            st.m[1] = mx1;
        st.l[0] *= a0;
        st.l[1] *= a1;
#pragma unroll
        for (int n = 0; n < kD / 8; ++n) {
            st.o[n][0] *= a0;
            st.o[n][1] *= a0;
            st.o[n][2] *= a1;
            st.o[n][3] *= a1;
        }
    }
    const float base0 = st.m[0] == -INFINITY ? 0.f : st.m[0];
    const float base1 = st.m[1] == -INFINITY ? 0.f : st.m[1];
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = fast_exp2(fmaf(s[nt][0], scale_log2, -base0));
        s[nt][1] = fast_exp2(fmaf(s[nt][1], scale_log2, -base0));
        s[nt][2] = fast_exp2(fmaf(s[nt][2], scale_log2, -base1));
        s[nt][3] = fast_exp2(fmaf(s[nt][3], scale_log2, -base1));
        sum0 += s[nt][0] + s[nt][1];
        sum1 += s[nt][2] + s[nt][3];
    }
#pragma unroll
    for (int ks = 0; ks < NT / 2; ++ks) {
        const int kb = key0 + ks * 16 + 2 * tq;
        constexpr float f = E5M2 ? 256.f : 1.f;
        const float va0 = v_scale[kb] * f, va1 = v_scale[kb + 1] * f;
        const float vb0 = v_scale[kb + 8] * f, vb1 = v_scale[kb + 9] * f;
        uint32_t pa[4];
        pa[0] = pack_f16(s[2 * ks][0] * va0, s[2 * ks][1] * va1);
        pa[1] = pack_f16(s[2 * ks][2] * va0, s[2 * ks][3] * va1);
        pa[2] = pack_f16(s[2 * ks + 1][0] * vb0, s[2 * ks + 1][1] * vb1);
        pa[3] = pack_f16(s[2 * ks + 1][2] * vb0, s[2 * ks + 1][3] * vb1);
        const int grp = (key0 >> 4) + ks;  // 16-key group: the 16-byte chunk of a V row
#pragma unroll
        for (int n = 0; n < kD / 8; ++n) {
            const int dim = n * 8 + g;
            const uint32_t w = *reinterpret_cast<const uint32_t *>(
                sV + dim * 64 + ((grp ^ ((dim >> 1) & 3)) << 4) + 4 * tq);
            mma_f16_16816(st.o[n], pa, fp8x2_lo<E5M2>(w), fp8x2_hi<E5M2>(w));
        }
    }
    st.l[0] += sum0;
    st.l[1] += sum1;
}

// KM keys (KM / 16 m-tiles) of a 64-key page of an FP8 full layer at T = 1, from
// key0, with the operands swapped: S^T = K Q^T with the keys on the MMA's M side and
// the unit's query heads on its N side (column n = head g, heads past G are zero),
// then O^T += V^T P^T with the output dimensions on M (eight m-tiles).  The
// shared-memory words are the ones run_tile_fp8 reads (K: four codes of one key, V
// transposed: four codes of one dimension), now taken for two keys / two dimensions
// an MMA.  P reaches the B operand of the second product through an 8x8 transpose.
// State per thread: heads 2 tq and 2 tq + 1 (m, l in log2 units) and oT[dt] = O^T
// rows dt * 16 + g, + 8.  Keys of the page >= `valid` are masked (a partly filled
// last page).
template <int KM, bool E5M2>
__device__ __forceinline__ void tile_fp8_sw(float (&m)[2], float (&l)[2], float (&oT)[kD / 16][4],
                                            const uint32_t (&qb)[kD / 16][2], const uint8_t *sK,
                                            const uint8_t *sV, const float *k_scale,
                                            const float *v_scale, int key0, int valid,
                                            float scale_log2)
{
    constexpr int MTS = KM / 16;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    float s[MTS][4], s2[MTS][4];
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
        s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = s2[mt][0] = s2[mt][1] = s2[mt][2] = s2[mt][3] = 0.f;
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt) {
        // keys key0 + mt * 16 + g and + 8 share (key & 7) = g, so one swizzle serves both
        const uint8_t *ra = sK + (key0 + mt * 16 + g) * 128 + 4 * tq;
        const uint8_t *rb = ra + 8 * 128;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const int off = (ks ^ g) << 4;
            const uint32_t wa = *reinterpret_cast<const uint32_t *>(ra + off);
            const uint32_t wb = *reinterpret_cast<const uint32_t *>(rb + off);
            const uint32_t a[4] = {fp8x2_lo<E5M2>(wa), fp8x2_lo<E5M2>(wb), fp8x2_hi<E5M2>(wa),
                                   fp8x2_hi<E5M2>(wb)};
            mma_f16_16816((ks & 1) ? s2[mt] : s[mt], a, qb[ks][0], qb[ks][1]);
        }
    }
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt) {
        const int ka = key0 + mt * 16 + g, kb = ka + 8;
        const float sa = ka < valid ? k_scale[ka] : 0.f, sb = kb < valid ? k_scale[kb] : 0.f;
        s[mt][0] = ka < valid ? (s[mt][0] + s2[mt][0]) * sa : -INFINITY;
        s[mt][1] = ka < valid ? (s[mt][1] + s2[mt][1]) * sa : -INFINITY;
        s[mt][2] = kb < valid ? (s[mt][2] + s2[mt][2]) * sb : -INFINITY;
        s[mt][3] = kb < valid ? (s[mt][3] + s2[mt][3]) * sb : -INFINITY;
        x0 = fmaxf(x0, fmaxf(s[mt][0], s[mt][2]));
        x1 = fmaxf(x1, fmaxf(s[mt][1], s[mt][3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
    }
    x0 *= scale_log2;
    x1 *= scale_log2;
    // running max raised lazily, as in run_tile (the lanes of a column agree)
    const bool up0 = x0 != -INFINITY && (m[0] == -INFINITY || x0 > m[0] + kRescaleSlack);
    const bool up1 = x1 != -INFINITY && (m[1] == -INFINITY || x1 > m[1] + kRescaleSlack);
    if (__any_sync(0xffffffffu, up0 || up1)) {
        const float a0 = up0 ? fast_exp2(m[0] - x0) : 1.f;
        const float a1 = up1 ? fast_exp2(m[1] - x1) : 1.f;
        if (up0)
            m[0] = x0;
        if (up1)
            m[1] = x1;
        l[0] *= a0;
        l[1] *= a1;
#pragma unroll
        for (int dt = 0; dt < kD / 16; ++dt) {
            oT[dt][0] *= a0;
            oT[dt][1] *= a1;
            oT[dt][2] *= a0;
            oT[dt][3] *= a1;
        }
    }
    const float base0 = m[0] == -INFINITY ? 0.f : m[0];
    const float base1 = m[1] == -INFINITY ? 0.f : m[1];
    constexpr float f = E5M2 ? 256.f : 1.f;  // an E5M2 V scale is folded in times 256
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < MTS; ++ks) {
        const int ka = key0 + ks * 16 + g, kb = ka + 8;
        const int grp = (key0 >> 4) + ks;  // 16-key group: the 16-byte chunk of a V row
        const float p0 = fast_exp2(fmaf(s[ks][0], scale_log2, -base0));
        const float p1 = fast_exp2(fmaf(s[ks][1], scale_log2, -base1));
        const float p2 = fast_exp2(fmaf(s[ks][2], scale_log2, -base0));
        const float p3 = fast_exp2(fmaf(s[ks][3], scale_log2, -base1));
        sum0 += p0 + p2;
        sum1 += p1 + p3;
        const float va = (ka < valid ? v_scale[ka] : 0.f) * f;
        const float vb = (kb < valid ? v_scale[kb] : 0.f) * f;
        // P^T rows ka (keys 0-7 of the 16) and kb (8-15), columns heads 2 tq, +1
        const uint32_t b0 = movmatrix_trans(pack_f16(p0 * va, p1 * va));
        const uint32_t b1 = movmatrix_trans(pack_f16(p2 * vb, p3 * vb));
#pragma unroll
        for (int dt = 0; dt < kD / 16; ++dt) {
            const int da = dt * 16 + g, db = da + 8;
            const uint32_t wa = *reinterpret_cast<const uint32_t *>(
                sV + da * 64 + ((grp ^ ((da >> 1) & 3)) << 4) + 4 * tq);
            const uint32_t wb = *reinterpret_cast<const uint32_t *>(
                sV + db * 64 + ((grp ^ ((db >> 1) & 3)) << 4) + 4 * tq);
            const uint32_t a[4] = {fp8x2_lo<E5M2>(wa), fp8x2_lo<E5M2>(wb), fp8x2_hi<E5M2>(wa),
                                   fp8x2_hi<E5M2>(wb)};
            mma_f16_16816(oT[dt], a, b0, b1);
        }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        sum0 += __shfl_xor_sync(0xffffffffu, sum0, o);
        sum1 += __shfl_xor_sync(0xffffffffu, sum1, o);
    }
    l[0] += sum0;
    l[1] += sum1;
}

// Append of unit (b, h) into an FP8 full layer: one warp per new K or V row.
__device__ __forceinline__ void append_unit_fp8(const DecodeParams &p, int b, int h, int c, int warp,
                                                int lane, int nwarps, bool e5m2)
{
    uint8_t *const kc = reinterpret_cast<uint8_t *>(p.k_dst);
    uint8_t *const vc = reinterpret_cast<uint8_t *>(p.v_dst);
    const int64_t cb = fp8_codes_bytes(p.num_blocks, p.Hkv);
    for (int e = warp; e < 2 * p.T; e += nwarps) {
        const int kv = e & 1, t = e >> 1;
        const int64_t pos = (int64_t)c + t;
        const int64_t page = pos / kTileKeys;
        if (page >= p.max_blocks) {
            if (lane == 0)
                set_err(p.dev_err, HSA_DEVERR_BAD_PAGE);
            continue;
        }
        const int blk = __ldg(p.block_tables + (int64_t)b * p.max_blocks + page);
        if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0)
                set_err(p.dev_err, HSA_DEVERR_BAD_BLOCK);
            continue;
        }
        const __nv_bfloat16 *src = (kv ? p.v_new : p.k_new) + ((int64_t)(b * p.T + t) * p.Hkv + h) * kD;
        uint8_t *codes = kv ? vc : kc;
        fp8_store_row(src, codes, reinterpret_cast<float *>(codes + cb), blk, h, p.Hkv,
                      (int)(pos % kTileKeys), kv, lane, e5m2);
    }
}

// Append the T new K/V rows of unit (b, h) to this layer's pool or ring.  Called by
// the CTA that completes the unit, after every read of the unit has finished.  With
// new_k / new_v (the rows this CTA staged in shared memory, bf16, 128-byte swizzle)
// the rows are copied from there instead of being read again from k_new / v_new.
__device__ __forceinline__ void append_unit(const DecodeParams &p, int b, int h, int c, int tid,
                                            int nthreads, const uint8_t *new_k = nullptr,
                                            const uint8_t *new_v = nullptr)
{
    constexpr int kChunks = kD * 2 / 16;  // 16-byte chunks per row
    const int total = 2 * p.T * kChunks;
    const bool ring = (p.flags & kDecodeRing) != 0;
    int rr = 0;
    if (ring) {
        rr = __ldg(p.ring_row + b);
        if (rr < 0 || rr >= p.n_ring_rows) {
            if (tid == 0)
                set_err(p.dev_err, HSA_DEVERR_BAD_RING);
            return;
        }
    }
    for (int e = tid; e < total; e += nthreads) {
        const int kv = e / (p.T * kChunks);
        const int t = (e / kChunks) % p.T;
        const int ch = e % kChunks;
        const int64_t pos = (int64_t)c + t;
        int64_t dst_row;
        if (ring) {
            dst_row = ((int64_t)rr * p.Hkv + h) * p.W + pos % p.W;
        } else {
            const int64_t page = pos / kTileKeys;
            if (page >= p.max_blocks) {
                set_err(p.dev_err, HSA_DEVERR_BAD_PAGE);
                continue;
            }
            const int blk = __ldg(p.block_tables + (int64_t)b * p.max_blocks + page);
            if (blk < 0 || blk >= p.num_blocks) {
                set_err(p.dev_err, HSA_DEVERR_BAD_BLOCK);
                continue;
            }
            dst_row = ((int64_t)blk * p.Hkv + h) * kTileKeys + pos % kTileKeys;
        }
        uint4 *to = kv ? p.v_dst : p.k_dst;
        if (new_k) {
            to[dst_row * kChunks + ch] = *reinterpret_cast<const uint4 *>(
                (kv ? new_v : new_k) + swz128_offset(t, ch * 8, kNewRows));
        } else {
            const int64_t src = ((int64_t)(b * p.T + t) * p.Hkv + h) * kChunks + ch;
            const uint4 *from = reinterpret_cast<const uint4 *>(kv ? p.v_new : p.k_new);
            to[dst_row * kChunks + ch] = __ldg(from + src);
        }
    }
}

// A unit split across CTAs: count this CTA's part in (its (m, l, o) partial is in
// the workspace already); the last CTA to arrive (atomic counter, no waiting)
// merges every part into `out`, appends the unit's new rows and resets the counter.
// Called by the nwarps consumer warps of the CTA, named barrier 1.
template <int FP8>
__device__ __forceinline__ void finish_split_unit(const DecodeParams &p, int32_t &is_last,
                                                  const Walk &cur, int64_t unit_start,
                                                  int64_t unit_end, int64_t N, int64_t C, int tid,
                                                  int warp, int lane, int nwarps)
{
    int32_t *const ws_cnt = reinterpret_cast<int32_t *>(p.ws);
    const float *const ws_part =
        reinterpret_cast<const float *>(p.ws + decode_counter_bytes(p.B, p.Hkv));
    const int nthreads = nwarps * 32;
    const int Hq = p.G * p.Hkv;
    const int unit = cur.b * p.Hkv + cur.h;
    const int64_t c_lo = ((unit_start + 1) * C - 1) / N;
    const int64_t c_hi = (unit_end * C - 1) / N;
    named_bar_sync(1, nthreads);
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(ws_cnt + unit, 1);
        is_last = (prev == (int)(c_hi - c_lo));
    }
    named_bar_sync(1, nthreads);
    if (!is_last)
        return;
    __threadfence();
    for (int e = tid; e < p.G * p.T * kD; e += nthreads) {
        const int rr = e / kD, dim = e % kD;
        float M = -INFINITY;
        for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
            const int64_t start_cc = cc * N / C;
            const int sl = 2 * (int)cc + (start_cc < unit_start ? 1 : 0);
            M = fmaxf(M, __ldcg(ws_part + (int64_t)sl * kPartFloats + rr));
        }
        const float base = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
        for (int64_t cc = c_lo; cc <= c_hi; ++cc) {
            const int64_t start_cc = cc * N / C;
            const int sl = 2 * (int)cc + (start_cc < unit_start ? 1 : 0);
            const float *pp = ws_part + (int64_t)sl * kPartFloats;
            const float a = fast_exp2(__ldcg(pp + rr) - base);
            L += __ldcg(pp + kMaxRows + rr) * a;
            O += __ldcg(pp + 2 * kMaxRows + rr * kD + dim) * a;
        }
        const int t = rr / p.G, hh = rr % p.G;
        p.out[((int64_t)(cur.b * p.T + t) * Hq + cur.h * p.G + hh) * kD + dim] =
            __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
    }
    if (p.flags & kDecodeAppend) {
        if constexpr (FP8)
            append_unit_fp8(p, cur.b, cur.h, cur.c, warp, lane, nwarps, FP8 == 2);
        else
            append_unit(p, cur.b, cur.h, cur.c, tid, nthreads);
    }
    if (tid == 0)
        ws_cnt[unit] = 0;
}

template <bool RING>
using SharedStorage = SharedStorageT<RING ? kRingStageRegion : kStageRegion>;

// MT: 16-row m-tiles of query rows (1: T <= 2, 2: T = 3, 4); FP8: an FP8 full
// layer; RING: a sliding layer (its own instantiation with two stages; at MT = 1 it
// is held to 168 registers so that two CTAs fit on an SM -- at MT = 2 that limit
// spilled ~170 bytes a thread, so MTP rings keep one CTA an SM).
// CW: consumer warps (kConsumerWarps, or kSwWarps for the swapped FP8 loop).
template <int MT, int FP8, bool RING, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, (RING && MT == 1) ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    static_assert(!(FP8 && RING), "the rings stay bf16");
    static_assert(CW == kConsumerWarps || (CW == kSwWarps && FP8 && MT == 1 && !RING),
                  "eight consumer warps: FP8 full layers at T = 1 only");
    constexpr int kThr = (CW + 1) * 32;
    constexpr int NS = RING ? kRingStages : (FP8 ? kFp8Stages : kStages);
    extern __shared__ uint8_t smem_raw[];
    SharedStorage<RING> &sh = *reinterpret_cast<SharedStorage<RING> *>(
        align_smem_1024(smem_raw));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sh.full[s], 1);
            // released by the warps of the stage's owning group: MT (full layers), 2 (rings)
            mbar_init(&sh.empty[s], RING ? 2 : MT);
        }
        fence_barrier_init();
    }
    if (warp == CW && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // Everything above touches no global memory that an earlier kernel writes.  With
    // kDecodeEarly (sliding layers) the item walk and the producer's ring loads below
    // also run before the wait -- they read cached_len, ring_row and this layer's ring,
    // which the caller guarantees the kernel just before does not write -- and only
    // the consumers wait, before they read q / k_new / v_new or write anything.
    const bool early = RING && (p.flags & kDecodeEarly) != 0;
    if (!early) {
        grid_dependency_wait();
        grid_launch_dependents();
    }

    // ---- locate this CTA's contiguous range of items ------------------------
    {
        const int per = (p.B + kThr - 1) / kThr;
        const int b_lo = min(p.B, tid * per), b_hi = min(p.B, b_lo + per);
        int local = 0;
        for (int b = b_lo; b < b_hi; ++b)
            local += items_of(p, b);
        sh.scan[tid] = local;
        __syncthreads();
        if (warp == 0) {
            // exclusive scan of kThr entries: kThr / 32 consecutive entries per lane
            constexpr int kPer = kThr / 32;
            int v[kPer];
            int sum = 0;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                v[j] = sh.scan[lane * kPer + j];
                sum += v[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += u;
            }
            int acc = incl - sum;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                sh.scan[lane * kPer + j] = acc;
                acc += v[j];
            }
            if (lane == 31)
                sh.total_items = incl;
        }
        __syncthreads();
    }
    const int64_t N = (int64_t)sh.total_items * p.Hkv;
    const int64_t C = N < (int64_t)gridDim.x ? N : (int64_t)gridDim.x;
    if ((int64_t)blockIdx.x >= C) {
        if (early)
            grid_dependency_wait();  // every CTA's exit stays ordered after the previous grid
        return;
    }
    const int64_t i0 = (int64_t)blockIdx.x * N / C;
    const int64_t i1 = ((int64_t)blockIdx.x + 1) * N / C;
    {
        // the thread whose chunk of sequences holds item i0 records it
        const int per = (p.B + kThr - 1) / kThr;
        const int b_lo = min(p.B, tid * per), b_hi = min(p.B, b_lo + per);
        int before = sh.scan[tid];
        for (int b = b_lo; b < b_hi; ++b) {
            int n = items_of(p, b);
            if ((int64_t)(before + n) * p.Hkv > i0 && (int64_t)before * p.Hkv <= i0) {
                sh.first_b = b;
                sh.first_items_before = before;
            }
            before += n;
        }
        __syncthreads();
    }
    Walk w0;
    w0.b = sh.first_b;
    walk_load(p, w0);
    {
        const int64_t off = i0 - (int64_t)sh.first_items_before * p.Hkv;
        w0.h = (int)(off / w0.n);
        w0.j = (int)(off % w0.n);
    }
    const int64_t w0_unit_start = i0 - w0.j;  // item index of tile 0 of the first unit

    if (warp == CW) {
        // ---------------------------------------------------------------- producer
#ifdef HSA_TEST_WITHHOLD_LOADS
        // Test-only builds (never the product library): the producer issues no load
        // and no arrival, so every consumer's first stage wait runs out after
        // HSA_WAIT_NS and the kernel must flag HSA_DEVERR_TIMEOUT and return.
        return;
#endif
        const uint64_t pol = policy_evict_first();
        const int64_t fp8_cb = fp8_codes_bytes(p.num_blocks, p.Hkv);
        // Lane 0: stage k gets item (b, h, j) whose TMA row is r (< 0: nothing to
        // load; its consumers skip it).  false = the stage never came free.
        auto issue = [&](int64_t k, int64_t r, int b, int h, int j, bool first) -> bool {
            if (early && (j == 0 || first)) {
                // before the grid-dependency wait: pull the unit's q rows and new K / V
                // rows towards L2 (a hint; the consumers read them after it)
                const int Hq = p.G * p.Hkv;
                for (int t = 0; t < p.T; ++t) {
                    const int64_t rq = (int64_t)b * p.T + t;
                    prefetch_l2(p.q + (rq * Hq + (int64_t)h * p.G) * kD, p.G * kD * 2);
                    prefetch_l2(p.k_new + (rq * p.Hkv + h) * kD, kD * 2);
                    prefetch_l2(p.v_new + (rq * p.Hkv + h) * kD, kD * 2);
                }
            }
            const int st = (int)(k % NS);
            const uint32_t ph = (uint32_t)((k / NS) & 1);
            if (!mbar_wait(&sh.empty[st], ph ^ 1)) {
                set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
                return false;
            }
            // read by the stage's consumers after the full barrier (whose arrive below
            // releases this write)
            sh.tile_ok[st] = r >= 0 ? 1 : 0;
            if (FP8 && r >= 0) {
                // E4M3 K page (64 rows x 128 B), transposed V page (128 rows x 64 B), and
                // the page's 64 K and 64 V scales
                mbar_arrive_expect_tx(&sh.full[st], 2 * kFp8TileBytes + 2 * 256);
                uint8_t *dst = sh.stage + st * kFp8StageStride;
                tma_load_2d(dst, &tmK, &sh.full[st], 0, (int32_t)r, pol);
                tma_load_2d(dst + kFp8TileBytes, &tmV, &sh.full[st], 0, (int32_t)(2 * r), pol);
                const uint8_t *kb = reinterpret_cast<const uint8_t *>(p.k_dst) + fp8_cb;
                const uint8_t *vb = reinterpret_cast<const uint8_t *>(p.v_dst) + fp8_cb;
                bulk_load(dst + 2 * kFp8TileBytes, kb + r * 4, 256, &sh.full[st], pol);
                bulk_load(dst + 2 * kFp8TileBytes + 256, vb + r * 4, 256, &sh.full[st], pol);
            } else if (r >= 0) {
                mbar_arrive_expect_tx(&sh.full[st], kStageBytes);
                uint8_t *dst = sh.stage + st * kStageBytes;
                tma_load_2d(dst, &tmK, &sh.full[st], 0, (int32_t)r, pol);
                tma_load_2d(dst + kTileBytes / 2, &tmK, &sh.full[st], 64, (int32_t)r, pol);
                tma_load_2d(dst + kTileBytes, &tmV, &sh.full[st], 0, (int32_t)r, pol);
                tma_load_2d(dst + kTileBytes + kTileBytes / 2, &tmV, &sh.full[st], 64, (int32_t)r,
                            pol);
            } else {
                mbar_arrive(&sh.full[st]);
            }
            return true;
        };
        int64_t k = 0;
        if constexpr (FP8 != 0) {
            // FP8 pages are half the bytes of bf16 ones, and reading the block table one
            // entry at a time (a dependent L2 access, ~0.5 us, on the producer's path
            // between stages) bounded the layer.  The rows are read 32 items at a time,
            // lane l taking item start + l, one batch ahead of the stages they feed; lane
            // 0 issues the stages, the rows and walk positions reaching it by shuffles.
            // A lane walks only to items of the CTA's range (past it a walk can cross
            // many short units, each a dependent read of cached_len).  (Measured on bf16
            // layers, the same scheme was ~2% slower, so they keep the loop below.)
            Walk wl = w0;
            int64_t row = -1;
            if (i0 + lane < i1) {
                for (int e = 0; e < lane; ++e)
                    walk_next(p, wl);
                row = tile_row(p, wl, true);
            }
            for (int64_t ib = i0; ib < i1; ib += 32) {
                Walk wn = wl;  // this lane's item of the next batch
                int64_t nrow = -1;
                if (ib + 32 + lane < i1) {
                    for (int e = 0; e < 32; ++e)
                        walk_next(p, wn);
                    nrow = tile_row(p, wn, true);
                }
                const int cnt = (int)(i1 - ib < 32 ? i1 - ib : 32);
                bool stop = false;
                for (int e = 0; e < cnt; ++e, ++k) {
                    const int64_t r = __shfl_sync(0xffffffffu, row, e);
                    const int eb = __shfl_sync(0xffffffffu, wl.b, e);
                    const int eh = __shfl_sync(0xffffffffu, wl.h, e);
                    const int ej = __shfl_sync(0xffffffffu, wl.j, e);
                    int ok = 1;
                    if (lane == 0)
                        ok = issue(k, r, eb, eh, ej, ib + e == i0) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        stop = true;
                        break;
                    }
                }
                if (stop)
                    break;
                row = nrow;
                wl = wn;
            }
        } else if (lane == 0) {
            // the block-table read of the next tile is issued before waiting for its
            // stage, so its latency hides behind the wait
            Walk w = w0;
            int64_t row = i0 < i1 ? tile_row(p, w, true) : -1;
            for (int64_t i = i0; i < i1; ++i, ++k) {
                if (!issue(k, row, w.b, w.h, w.j, i == i0))
                    break;
                walk_next(p, w);
                row = i + 1 < i1 ? tile_row(p, w, true) : -1;
            }
        }
        if (lane == 0) {
            // drain: no TMA write may still be in flight when the CTA exits
            for (int64_t s = 0; s < NS && s < k; ++s) {
                const int64_t last = s + ((k - 1 - s) / NS) * NS;
                mbar_wait(&sh.full[s], (uint32_t)((last / NS) & 1));
            }
        }
        return;
    }

    if constexpr (CW == kSwWarps) {
        // ------------------------------------------ consumers: FP8 full layer, T = 1
        // Eight warps; warp w runs the tiles k = w mod 8 of the CTA's range (stage k
        // mod 8) with tile_fp8_sw.  At the end of a unit the warps' states merge
        // through shared memory, warp h taking query head h and each lane four output
        // dimensions; the CTA that owns the unit's last tile adds the new token there
        // as one more key (its score q . k_new from the bf16 rows, weight and value
        // exact).  Split units go through the workspace as in the general loop.
        constexpr bool kE5 = FP8 == 2;
        const int g = lane >> 2, tq = lane & 3;
        const int Hq = p.G * p.Hkv;
        float *const ws_part = reinterpret_cast<float *>(p.ws + decode_counter_bytes(p.B, p.Hkv));
        float *const comb = &sh.comb[0][0];
        uint32_t qb[kD / 16][2];
        float m[2], l[2], oT[kD / 16][4];
        Walk w = w0;
        int64_t unit_start = w0_unit_start;
        bool fresh = true, timed_out = false;
        for (int64_t i = i0, k = 0; i < i1; ++i, ++k) {
            if (fresh) {
                fresh = false;
                m[0] = m[1] = -INFINITY;
                l[0] = l[1] = 0.f;
#pragma unroll
                for (int dt = 0; dt < kD / 16; ++dt)
                    oT[dt][0] = oT[dt][1] = oT[dt][2] = oT[dt][3] = 0.f;
                // B operand of S^T = K Q^T in fp16: column g = query head g of the unit
                const bool ok = g < p.G;
                const __nv_bfloat16 *qg = p.q + ((int64_t)w.b * Hq + w.h * p.G + (ok ? g : 0)) * kD;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qg + ks * 16 + 2 * tq);
                    qb[ks][0] = ok ? bf16x2_to_f16x2(__ldg(q32)) : 0u;
                    qb[ks][1] = ok ? bf16x2_to_f16x2(__ldg(q32 + 4)) : 0u;
                }
            }
            if ((int)(k % kSwWarps) == warp) {
                const int stg = (int)(k % NS);
                if (!timed_out && !mbar_wait(&sh.full[stg], (uint32_t)((k / NS) & 1))) {
                    set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
                    timed_out = true;
                }
                const int valid = w.c - w.j * kTileKeys;  // cached keys on this page
                if (!timed_out && sh.tile_ok[stg] != 0 && valid > 0) {
                    const uint8_t *base = sh.stage + stg * kFp8StageStride;
                    const float *ksc = reinterpret_cast<const float *>(base + 2 * kFp8TileBytes);
                    tile_fp8_sw<kTileKeys, kE5>(m, l, oT, qb, base, base + kFp8TileBytes, ksc,
                                                ksc + 64, 0, valid < kTileKeys ? valid : kTileKeys,
                                                p.scale_log2);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sh.empty[stg]);
            }
            const bool unit_last_tile = (w.j == w.n - 1);
            const Walk cur = w;
            walk_next(p, w);
            if (!(unit_last_tile || i == i1 - 1))
                continue;

            // ---- end of this CTA's share of unit (cur.b, cur.h) --------------
            const int64_t unit_end = unit_start + cur.n;
            if constexpr (kE5) {  // the E5M2 tiles accumulate 256 O
#pragma unroll
                for (int dt = 0; dt < kD / 16; ++dt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        oT[dt][e] *= 1.f / 256.f;
            }
            {
                float *cb = comb + warp * kSwFloats;
                if (g == 0) {
                    cb[2 * tq] = m[0];
                    cb[2 * tq + 1] = m[1];
                    cb[8 + 2 * tq] = l[0];
                    cb[8 + 2 * tq + 1] = l[1];
                }
                float *co = cb + 16;
#pragma unroll
                for (int dt = 0; dt < kD / 16; ++dt) {
                    co[(2 * tq) * kHs + dt * 16 + g] = oT[dt][0];
                    co[(2 * tq + 1) * kHs + dt * 16 + g] = oT[dt][1];
                    co[(2 * tq) * kHs + dt * 16 + g + 8] = oT[dt][2];
                    co[(2 * tq + 1) * kHs + dt * 16 + g + 8] = oT[dt][3];
                }
            }
            named_bar_sync(1, kSwWarps * 32);
            const bool whole = unit_start >= i0 && unit_end <= i1;
            const bool has_new = unit_end <= i1;  // this CTA owns the unit's last tile
            const int head = warp;
            if (head < p.G) {
                const int d0 = lane * 4;
                float sn = -INFINITY, vn[4] = {0.f, 0.f, 0.f, 0.f};
                if (has_new) {
                    const uint2 qv = __ldg(reinterpret_cast<const uint2 *>(
                        p.q + ((int64_t)cur.b * Hq + cur.h * p.G + head) * kD + d0));
                    const int64_t rk = ((int64_t)cur.b * p.Hkv + cur.h) * kD + d0;
                    const uint2 kv = __ldg(reinterpret_cast<const uint2 *>(p.k_new + rk));
                    const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(p.v_new + rk));
                    float dot = bf16_lo(qv.x) * bf16_lo(kv.x) + bf16_hi(qv.x) * bf16_hi(kv.x) +
                                bf16_lo(qv.y) * bf16_lo(kv.y) + bf16_hi(qv.y) * bf16_hi(kv.y);
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1)
                        dot += __shfl_xor_sync(0xffffffffu, dot, o);
                    sn = dot * p.scale_log2;
                    vn[0] = bf16_lo(vv.x);
                    vn[1] = bf16_hi(vv.x);
                    vn[2] = bf16_lo(vv.y);
                    vn[3] = bf16_hi(vv.y);
                }
                float M = sn;
#pragma unroll
                for (int s = 0; s < kSwWarps; ++s)
                    M = fmaxf(M, comb[s * kSwFloats + head]);
                const float base = M == -INFINITY ? 0.f : M;
                const float an = has_new ? fast_exp2(sn - base) : 0.f;
                float L = an;
                float o[4] = {an * vn[0], an * vn[1], an * vn[2], an * vn[3]};
#pragma unroll
                for (int s = 0; s < kSwWarps; ++s) {
                    const float *cs = comb + s * kSwFloats;
                    const float a = fast_exp2(cs[head] - base);
                    L += cs[8 + head] * a;
                    const float4 x = *reinterpret_cast<const float4 *>(cs + 16 + head * kHs + d0);
                    o[0] += x.x * a;
                    o[1] += x.y * a;
                    o[2] += x.z * a;
                    o[3] += x.w * a;
                }
                if (whole) {
                    const float norm = L > 0.f ? 1.f / L : 0.f;
                    *reinterpret_cast<uint2 *>(
                        p.out + ((int64_t)cur.b * Hq + cur.h * p.G + head) * kD + d0) =
                        make_uint2(pack_bf16(o[0] * norm, o[1] * norm),
                                   pack_bf16(o[2] * norm, o[3] * norm));
                } else {
                    const int slot = 2 * (int)blockIdx.x + (i0 < unit_start ? 1 : 0);
                    float *part = ws_part + (int64_t)slot * kPartFloats;
                    if (lane == 0) {
                        __stcg(part + head, M);
                        __stcg(part + kMaxRows + head, L);
                    }
                    __stcg(reinterpret_cast<float4 *>(part + 2 * kMaxRows + head * kD + d0),
                           make_float4(o[0], o[1], o[2], o[3]));
                }
            }
            if (whole && (p.flags & kDecodeAppend))
                append_unit_fp8(p, cur.b, cur.h, cur.c, warp, lane, kSwWarps, kE5);
            if (!whole)
                finish_split_unit<FP8>(p, sh.is_last, cur, unit_start, unit_end, N, C, tid, warp,
                                       lane, kSwWarps);
            named_bar_sync(1, kSwWarps * 32);  // merge buffer free again
            unit_start = unit_end;
            fresh = true;
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int mt = warp % MT;
    const int slice = warp / MT;
    // Full layers (long units of pages): tile-parallel groups -- the MT warps of group
    // `slice` (one per 16-row m-tile) run every (4 / MT)-th tile of the CTA's range
    // with all 64 keys (eight independent MMA chains per warp), 4 / MT tiles in
    // flight.  Rings (a unit is two tiles): two groups, one per tile of a unit, so the
    // two run side by side -- MT = 1: two warps per tile, 32 keys each; MT = 2: one
    // warp per m-tile with all 64 keys.
    constexpr int kGroups = kConsumerWarps / MT;
    static_assert(RING ? NS % 2 == 0 : (NS % kGroups == 0 && NS % 2 == 0),
                  "each stage belongs to one group");
    constexpr bool ring = RING;
    constexpr int wt = (ring && MT == 1) ? 2 : 1;  // warps per m-tile sharing a tile
    constexpr int groups = ring ? 2 : kGroups;
    if (early) {
        // the consumers read q / k_new / v_new, which the previous kernel writes
        grid_dependency_wait();
        grid_launch_dependents();
    }
    const int key0 = (slice % wt) * (kTileKeys / wt);
    const int g = lane >> 2, tq = lane & 3;
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const int t0 = r0 / p.G, t1 = r1 / p.G;
    const int rows_valid = p.G * p.T;
    const int Hq = p.G * p.Hkv;
    float *const ws_part = reinterpret_cast<float *>(p.ws + decode_counter_bytes(p.B, p.Hkv));

    RowState st;
    uint32_t qa[kD / 16][4];
    Walk w = w0;
    int64_t unit_start = w0_unit_start;
    bool fresh = true;
    bool timed_out = false;

    // the unit's new tokens (staged in new_k / new_v): positions c .. c+T-1, causal
    // among themselves
    auto run_new_tile = [&]() {
        const int T = p.T;
        auto vis_new = [&](int rr, int key) -> bool {
            const int t = rr == g ? t0 : t1;
            return t < T && key <= t;
        };
        run_tile<2, (FP8 != 0)>(st, qa, smem_u32(sh.new_k), smem_u32(sh.new_v), kNewRows, 0,
                                p.scale_log2, false, t0 < T, t1 < T, vis_new);
    };

    // Sliding layers at T = 1 with a full ring (c >= W = 128): the new token replaces
    // the one slot its query no longer sees (position c - W, slot c mod W), so once
    // that row of the staged tile is overwritten with the new K / V, every one of the
    // tile pair's 128 keys is visible and no mask or separate new-token tile remains.
    // Each warp takes 32 keys with the operands swapped -- keys on the MMA's M side,
    // the unit's (at most 8) query heads on its N side -- which halves the MMAs and
    // the accumulator registers of the 16-row form; P goes from the S accumulators to
    // the B operand of P V through an 8x8 transpose.  The warp holding the new slot
    // also appends the new row, and one shared-memory pass merges the four warps.
    const bool fold_ok = RING && MT == 1 && p.T == 1 && p.G <= 8 && p.W == 2 * kTileKeys;
    auto ring_unit_t1 = [&](int64_t k_first, bool last_unit) {
        const int grp = slice / wt;                    // tile-pair half this warp reads
        const int my_j = grp ^ (int)(k_first & 1);     // the unit's tile in stage grp
        const int64_t kk = k_first + my_j;
        const int c = w.c;
        const int slot_new = c % p.W;
        const bool patcher = slot_new / kTileKeys == my_j && (slot_new % kTileKeys) / 32 == slice % wt;
        // B operand of S^T = K Q^T: column n = query head g of the unit (zero past G)
        uint32_t qb[kD / 16][2];
        {
            const bool ok = g < p.G;
            const __nv_bfloat16 *qg = p.q + ((int64_t)w.b * Hq + w.h * p.G + (ok ? g : 0)) * kD;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                qb[ks][0] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qg + ks * 16 + 2 * tq)) : 0u;
                qb[ks][1] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qg + ks * 16 + 8 + 2 * tq)) : 0u;
            }
        }
        // the new row: lanes 0-15 hold K's sixteen 16-byte chunks, lanes 16-31 V's
        const int ch = lane & 15;
        uint4 nrow = make_uint4(0, 0, 0, 0);
        int rr = -1;
        if (patcher) {
            const uint4 *src = reinterpret_cast<const uint4 *>(lane < 16 ? p.k_new : p.v_new);
            nrow = __ldg(src + ((int64_t)w.b * p.Hkv + w.h) * (kD / 8) + ch);
            if (p.flags & kDecodeAppend)
                rr = __ldg(p.ring_row + w.b);
        }
        const uint32_t ph = (uint32_t)((kk / NS) & 1);
        if (!timed_out && !mbar_wait(&sh.full[grp], ph)) {
            set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
            timed_out = true;
        }
        const bool loaded = !timed_out && sh.tile_ok[grp] != 0;
        const uint32_t sK = smem_u32(sh.stage + grp * kStageBytes);
        const uint32_t sV = sK + kTileBytes;
        if (patcher && loaded) {
            const int row = slot_new % kTileKeys;
            *reinterpret_cast<uint4 *>(sh.stage + grp * kStageBytes + (lane < 16 ? 0 : kTileBytes) +
                                       swz128_offset(row, ch * 8, kTileKeys)) = nrow;
            if (p.flags & kDecodeAppend) {
                if (rr >= 0 && rr < p.n_ring_rows) {
                    const int64_t dst_row = ((int64_t)rr * p.Hkv + w.h) * p.W + slot_new;
                    (lane < 16 ? p.k_dst : p.v_dst)[dst_row * (kD / 8) + ch] = nrow;
                } else if (lane == 0) {
                    set_err(p.dev_err, HSA_DEVERR_BAD_RING);
                }
            }
        }
        __syncwarp();
        // this warp's 32 keys: S^T (keys x heads), softmax per head column, O^T += V^T P^T
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2 tq, 2 tq + 1
        float oT[kD / 16][4];
#pragma unroll
        for (int dt = 0; dt < kD / 16; ++dt)
            oT[dt][0] = oT[dt][1] = oT[dt][2] = oT[dt][3] = 0.f;
        if (loaded) {
            const int kb = (slice % wt) * 32;
            const int mi = lane >> 3, r8 = lane & 7;
            float sc[2][4];
#pragma unroll
            for (int mt2 = 0; mt2 < 2; ++mt2) {
                sc[mt2][0] = sc[mt2][1] = sc[mt2][2] = sc[mt2][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    uint32_t a[4];
                    ldmatrix_x4(sK + swz128_offset(kb + mt2 * 16 + (mi & 1) * 8 + r8,
                                                   ks * 16 + (mi >> 1) * 8, kTileKeys),
                                a[0], a[1], a[2], a[3]);
                    mma_bf16_16816(sc[mt2], a, qb[ks][0], qb[ks][1]);
                }
            }
            float x0 = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
            float x1 = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
            }
            m0 = x0 * p.scale_log2;
            m1 = x1 * p.scale_log2;
            uint32_t pb[2][2];
#pragma unroll
            for (int mt2 = 0; mt2 < 2; ++mt2) {
                const uint32_t lo = pack_bf16(fast_exp2(fmaf(sc[mt2][0], p.scale_log2, -m0)),
                                              fast_exp2(fmaf(sc[mt2][1], p.scale_log2, -m1)));
                const uint32_t hi = pack_bf16(fast_exp2(fmaf(sc[mt2][2], p.scale_log2, -m0)),
                                              fast_exp2(fmaf(sc[mt2][3], p.scale_log2, -m1)));
                // the sums take the bf16-rounded P the MMA uses
                l0 += bf16_lo(lo) + bf16_lo(hi);
                l1 += bf16_hi(lo) + bf16_hi(hi);
                pb[mt2][0] = movmatrix_trans(lo);  // keys 0-7 of the 16: B rows 2 tq, +1
                pb[mt2][1] = movmatrix_trans(hi);  // keys 8-15
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                for (int dt = 0; dt < kD / 16; ++dt) {
                    uint32_t a[4];
                    ldmatrix_x4_trans(sV + swz128_offset(kb + ks * 16 + (mi >> 1) * 8 + r8,
                                                         dt * 16 + (mi & 1) * 8, kTileKeys),
                                      a[0], a[1], a[2], a[3]);
                    mma_bf16_16816(oT[dt], a, pb[ks][0], pb[ks][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sh.empty[grp]);
        // merge: per warp m[8], l[8], then O as [head][dim] with a 132-float head stride
        float *cb = sh.comb[warp];
        if (g == 0) {
            cb[2 * tq] = m0;
            cb[2 * tq + 1] = m1;
            cb[8 + 2 * tq] = l0;
            cb[8 + 2 * tq + 1] = l1;
        }
        float *co = cb + 16;
#pragma unroll
        for (int dt = 0; dt < kD / 16; ++dt) {
            co[(2 * tq) * kHs + dt * 16 + g] = oT[dt][0];
            co[(2 * tq + 1) * kHs + dt * 16 + g] = oT[dt][1];
            co[(2 * tq) * kHs + dt * 16 + g + 8] = oT[dt][2];
            co[(2 * tq + 1) * kHs + dt * 16 + g + 8] = oT[dt][3];
        }
        named_bar_sync(1, kConsumerWarps * 32);
        {
            const int head = tid >> 4, d0 = (tid & 15) * 8;
            if (head < p.G) {
                float M = -INFINITY;
#pragma unroll
                for (int s = 0; s < kConsumerWarps; ++s)
                    M = fmaxf(M, sh.comb[s][head]);
                const float base = M == -INFINITY ? 0.f : M;
                float a[kConsumerWarps], L = 0.f;
#pragma unroll
                for (int s = 0; s < kConsumerWarps; ++s) {
                    a[s] = fast_exp2(sh.comb[s][head] - base);
                    L += sh.comb[s][8 + head] * a[s];
                }
                const float norm = L > 0.f ? 1.f / L : 0.f;
                float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < kConsumerWarps; ++s) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(&sh.comb[s][16 + head * kHs + d0]);
                    const float4 x = src[0], y = src[1];
                    const float wgt = a[s] * norm;
                    o[0] += x.x * wgt;
                    o[1] += x.y * wgt;
                    o[2] += x.z * wgt;
                    o[3] += x.w * wgt;
                    o[4] += y.x * wgt;
                    o[5] += y.y * wgt;
                    o[6] += y.z * wgt;
                    o[7] += y.w * wgt;
                }
                uint4 v;
                v.x = pack_bf16(o[0], o[1]);
                v.y = pack_bf16(o[2], o[3]);
                v.z = pack_bf16(o[4], o[5]);
                v.w = pack_bf16(o[6], o[7]);
                *reinterpret_cast<uint4 *>(p.out + ((int64_t)w.b * Hq + w.h * p.G + head) * kD + d0) = v;
            }
        }
        if (!last_unit)
            named_bar_sync(1, kConsumerWarps * 32);  // comb free again
    };

    int64_t i = i0, k = 0;
    if constexpr (RING && MT == 1) {
        // the CTA's leading whole units with a full ring take the path above; from the
        // first unit that does not (a partial unit, a ring not yet full) the general
        // loop below takes the rest
        while (fold_ok && i < i1 && w.j == 0 && w.c >= p.W && unit_start + w.n <= i1) {
            const int n = w.n;
            ring_unit_t1(k, unit_start + n == i1);
            i += n;
            k += n;
            unit_start += n;
            for (int e = 0; e < n; ++e)
                walk_next(p, w);
        }
    }
    for (; i < i1; ++i, ++k) {
        if (fresh) {
            fresh = false;
            st.m[0] = st.m[1] = -INFINITY;
            st.l[0] = st.l[1] = 0.f;
#pragma unroll
            for (int n = 0; n < kD / 8; ++n)
                st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
            const __nv_bfloat16 *q0 =
                p.q + ((int64_t)(w.b * p.T + t0) * Hq + w.h * p.G + r0 % p.G) * kD;
            const __nv_bfloat16 *q1 =
                p.q + ((int64_t)(w.b * p.T + t1) * Hq + w.h * p.G + r1 % p.G) * kD;
            const bool v0 = t0 < p.T, v1 = t1 < p.T;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const int c0 = ks * 16 + 2 * tq;
                qa[ks][0] = v0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c0)) : 0u;
                qa[ks][1] = v1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c0)) : 0u;
                qa[ks][2] = v0 ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c0 + 8)) : 0u;
                qa[ks][3] = v1 ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c0 + 8)) : 0u;
                if (FP8) {  // the FP8 kernel multiplies in fp16
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        qa[ks][e] = bf16x2_to_f16x2(qa[ks][e]);
                }
            }
            // when this CTA owns the unit's last tile, stage the unit's new rows (rows
            // >= T zero).  Rings (a unit is two tiles): the slice-0 warps (one per
            // m-tile) stage them and run them as a 16-key tile now, while the other
            // warps wait for their stage (the online softmax takes tiles in any
            // order).  Full layers: every consumer warp stages, and the slice-0 warps
            // run the tile at the end of the unit, so that no group starts late.
            if (unit_start + w.n <= i1 && (!RING || slice == 0)) {
                constexpr int kStagers = (RING ? MT : kConsumerWarps) * 32;
                for (int e = tid; e < kNewRows * kD / 8; e += kStagers) {
                    const int rr = e / (kD / 8), col = (e % (kD / 8)) * 8;
                    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
                    if (rr < p.T) {
                        const int64_t src =
                            ((int64_t)(w.b * p.T + rr) * p.Hkv + w.h) * kD + col;
                        kv = __ldg(reinterpret_cast<const uint4 *>(p.k_new + src));
                        vv = __ldg(reinterpret_cast<const uint4 *>(p.v_new + src));
                        if (FP8) {
                            kv = make_uint4(bf16x2_to_f16x2(kv.x), bf16x2_to_f16x2(kv.y),
                                            bf16x2_to_f16x2(kv.z), bf16x2_to_f16x2(kv.w));
                            vv = make_uint4(bf16x2_to_f16x2(vv.x), bf16x2_to_f16x2(vv.y),
                                            bf16x2_to_f16x2(vv.z), bf16x2_to_f16x2(vv.w));
                        }
                    }
                    *reinterpret_cast<uint4 *>(sh.new_k + swz128_offset(rr, col, kNewRows)) = kv;
                    *reinterpret_cast<uint4 *>(sh.new_v + swz128_offset(rr, col, kNewRows)) = vv;
                }
                if constexpr (RING) {
                    if (MT == 1)
                        __syncwarp();
                    else
                        named_bar_sync(2, MT * 32);
                    run_new_tile();
                }
            }
        }
        const int stg = (int)(k % NS);
        const uint32_t ph = (uint32_t)((k / NS) & 1);
        const bool mine = (int)(k % groups) == slice / wt;
        if (mine && !timed_out && !mbar_wait(&sh.full[stg], ph)) {
            set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
            timed_out = true;
        }
        const bool loaded = mine && !timed_out && sh.tile_ok[stg] != 0;
        const int c = w.c;
        const int j = w.j;
        bool any = loaded;
        if (loaded && !ring)
            any = key0 < c - j * kTileKeys;  // this warp's keys hold a cached position
        if (any) {
            const uint32_t sK = smem_u32(sh.stage + stg * kStageBytes);
            const uint32_t sV = sK + kTileBytes;
            const int W = p.W, T = p.T;
            // ring slot s holds position c - 1 - back(s), back(s) = (r0 - s) mod W with
            // r0 = (c - 1) mod W (one modulo a tile, not one a key); query row t sees it
            // iff back(s) <= c - 1 - max(0, c + t - W + 1)
            const int r0 = ring ? (c - 1) % W : 0;
            auto vis = [&](int rr, int key) -> bool {
                const int t = rr == g ? t0 : t1;
                if (t >= T)
                    return false;
                const int slot = j * kTileKeys + key;
                if (!ring)
                    return slot < c;
                const int back = r0 - slot + (slot > r0 ? W : 0);
                return back <= c - 1 - max(0, c + t - W + 1);
            };
            // full layers: every key of a complete page is visible to every query
            const bool all_vis = !ring && (j + 1) * kTileKeys <= c;
            if constexpr (FP8) {  // full layers only: tile-parallel
                const uint8_t *base = sh.stage + stg * kFp8StageStride;
                const float *ksc = reinterpret_cast<const float *>(base + 2 * kFp8TileBytes);
                run_tile_fp8<kTileKeys / 8, FP8 == 2>(st, qa, base, base + kFp8TileBytes, ksc,
                                                      ksc + 64, key0, p.scale_log2, all_vis,
                                                      t0 < T, t1 < T, vis);
            } else if (wt == 1) {
                run_tile<kTileKeys / 8>(st, qa, sK, sV, kTileKeys, key0, p.scale_log2, all_vis,
                                        t0 < T, t1 < T, vis);
            } else {
                run_tile<kTileKeys / 16>(st, qa, sK, sV, kTileKeys, key0, p.scale_log2, all_vis,
                                         t0 < T, t1 < T, vis);
            }
        }
        __syncwarp();
        if (mine && lane == 0)
            mbar_arrive(&sh.empty[stg]);

        const bool unit_last_tile = (j == w.n - 1);
        const Walk cur = w;
        walk_next(p, w);
        if (!(unit_last_tile || i == i1 - 1))
            continue;

        // ---- end of this CTA's share of unit (cur.b, cur.h) ------------------
        const int64_t unit_end = unit_start + cur.n;  // one past its last item
        if constexpr (FP8 == 2) {  // the E5M2 tiles accumulate 256 O
#pragma unroll
            for (int n = 0; n < kD / 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    st.o[n][e] *= 1.f / 256.f;
        }
        if (!RING && unit_last_tile) {
            named_bar_sync(1, kConsumerWarps * 32);  // new rows staged by every warp
            if (slice == 0)
                run_new_tile();
        }
        // merge the warps' states (same m-tile, different key slices)
        {
            float l0 = st.l[0], l1 = st.l[1];
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            float *cb = sh.comb[warp];
            if (tq == 0) {
                cb[g] = st.m[0];
                cb[g + 8] = st.m[1];
                cb[16 + g] = l0;
                cb[16 + g + 8] = l1;
            }
            float *co = cb + 32;
#pragma unroll
            for (int n = 0; n < kD / 8; ++n) {
                *reinterpret_cast<float2 *>(co + g * kD + n * 8 + 2 * tq) =
                    make_float2(st.o[n][0], st.o[n][1]);
                *reinterpret_cast<float2 *>(co + (g + 8) * kD + n * 8 + 2 * tq) =
                    make_float2(st.o[n][2], st.o[n][3]);
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);

        const bool whole = unit_start >= i0 && unit_end <= i1;
        int32_t slot = -1;
        if (!whole)
            slot = 2 * (int)blockIdx.x + (i0 < unit_start ? 1 : 0);  // 1 = CTA's last unit
        constexpr int kSlices = kConsumerWarps / MT;
        float *part = ws_part + (int64_t)(slot < 0 ? 0 : slot) * kPartFloats;
        // (a) per row: the combined max M, sum L and each slice's weight 2^(m_s - M)
        // (with 1 / L folded in for a unit written straight to out)
        for (int rr = tid; rr < MT * 16; rr += kConsumerWarps * 32) {
            const int m_t = rr / 16, rl = rr % 16;
            float M = -INFINITY;
#pragma unroll
            for (int s = 0; s < kSlices; ++s)
                M = fmaxf(M, sh.comb[m_t + MT * s][rl]);
            const float base = M == -INFINITY ? 0.f : M;
            float a[kSlices], L = 0.f;
#pragma unroll
            for (int s = 0; s < kSlices; ++s) {
                a[s] = fast_exp2(sh.comb[m_t + MT * s][rl] - base);
                L += sh.comb[m_t + MT * s][16 + rl] * a[s];
            }
            const float norm = whole ? (L > 0.f ? 1.f / L : 0.f) : 1.f;
#pragma unroll
            for (int s = 0; s < kSlices; ++s)
                sh.mscale[rr][s] = a[s] * norm;
            sh.mrow[rr][0] = M;
            sh.mrow[rr][1] = L;
        }
        named_bar_sync(1, kConsumerWarps * 32);
        // (b) eight output dimensions a thread: O = sum_s o_s * weight_s, written as
        // 16 bytes of bf16 (a whole unit) or two 16-byte fp32 partials (a split one)
        for (int e = tid; e < MT * 16 * (kD / 8); e += kConsumerWarps * 32) {
            const int rr = e / (kD / 8), d0 = (e % (kD / 8)) * 8;
            if (rr >= rows_valid)
                continue;
            const int m_t = rr / 16, rl = rr % 16;
            float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < kSlices; ++s) {
                const float w = sh.mscale[rr][s];
                const float4 *src =
                    reinterpret_cast<const float4 *>(&sh.comb[m_t + MT * s][32 + rl * kD + d0]);
                const float4 x = src[0], y = src[1];
                o[0] += x.x * w;
                o[1] += x.y * w;
                o[2] += x.z * w;
                o[3] += x.w * w;
                o[4] += y.x * w;
                o[5] += y.y * w;
                o[6] += y.z * w;
                o[7] += y.w * w;
            }
            if (whole) {
                const int t = rr / p.G, hh = rr % p.G;
                uint4 v;
                v.x = pack_bf16(o[0], o[1]);
                v.y = pack_bf16(o[2], o[3]);
                v.z = pack_bf16(o[4], o[5]);
                v.w = pack_bf16(o[6], o[7]);
                *reinterpret_cast<uint4 *>(
                    p.out + ((int64_t)(cur.b * p.T + t) * Hq + cur.h * p.G + hh) * kD + d0) = v;
            } else {
                if (d0 == 0) {
                    __stcg(part + rr, sh.mrow[rr][0]);
                    __stcg(part + kMaxRows + rr, sh.mrow[rr][1]);
                }
                float4 *dst = reinterpret_cast<float4 *>(part + 2 * kMaxRows + rr * kD + d0);
                __stcg(dst, make_float4(o[0], o[1], o[2], o[3]));
                __stcg(dst + 1, make_float4(o[4], o[5], o[6], o[7]));
            }
        }
        if (whole && (p.flags & kDecodeAppend)) {
            // a whole unit's new rows were staged by this CTA (it owns the last tile)
            if constexpr (FP8)
                append_unit_fp8(p, cur.b, cur.h, cur.c, warp, lane, kConsumerWarps, FP8 == 2);
            else
                append_unit(p, cur.b, cur.h, cur.c, tid, kConsumerWarps * 32, sh.new_k, sh.new_v);
        }
        if (!whole)
            finish_split_unit<FP8>(p, sh.is_last, cur, unit_start, unit_end, N, C, tid, warp, lane,
                                   kConsumerWarps);
        named_bar_sync(1, kConsumerWarps * 32);  // comb / new-token buffers free again
        unit_start = unit_end;
        fresh = true;
    }
}

}  // namespace

size_t decode_workspace_bytes(int num_sms, int B, int Hkv)
{
    size_t cnt = decode_counter_bytes(B, Hkv);
    size_t part = (size_t)2 * num_sms * kPartFloats * sizeof(float);
    return cnt + part;
}

cudaError_t launch_decode(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                          int ctas, cudaStream_t stream)
{
    const int MT = (p.G * p.T + 15) / 16;
    const bool fp8 = (p.flags & kDecodeFp8) != 0;
    const bool ring = (p.flags & kDecodeRing) != 0;
    const size_t smem = (ring ? sizeof(SharedStorage<true>) : sizeof(SharedStorage<false>)) + 1024;
    // the opt-in shared-memory size is set once per process (the API is not a stream
    // operation, but setting it once keeps graph capture free of extra calls)
    static bool attr_set[10] = {false, false, false, false, false,
                                false, false, false, false, false};
    void (*kern)(CUtensorMap, CUtensorMap, DecodeParams);
    int which;
    constexpr int C4 = kConsumerWarps;
    // FP8 full layers at T = 1 with <= 8 query heads a KV head: the eight-warp loop
    const bool sw = fp8 && !ring && p.T == 1 && p.G <= 8;
    if (ring) {
        kern = MT == 1 ? decode_kernel<1, 0, true, C4> : decode_kernel<2, 0, true, C4>;
        which = 4 + MT - 1;
    } else if (sw) {
        kern = (p.flags & kDecodeE5M2) ? decode_kernel<1, 2, false, kSwWarps>
                                       : decode_kernel<1, 1, false, kSwWarps>;
        which = (p.flags & kDecodeE5M2) ? 9 : 8;
    } else if (fp8 && (p.flags & kDecodeE5M2)) {
        kern = MT == 1 ? decode_kernel<1, 2, false, C4> : decode_kernel<2, 2, false, C4>;
        which = 6 + MT - 1;
    } else if (fp8) {
        kern = MT == 1 ? decode_kernel<1, 1, false, C4> : decode_kernel<2, 1, false, C4>;
        which = 2 + MT - 1;
    } else {
        kern = MT == 1 ? decode_kernel<1, 0, false, C4> : decode_kernel<2, 0, false, C4>;
        which = MT - 1;
    }
    if (!attr_set[which]) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set[which] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(((sw ? kSwWarps : kConsumerWarps) + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmK, tmV, p);
}

}  // namespace hsa

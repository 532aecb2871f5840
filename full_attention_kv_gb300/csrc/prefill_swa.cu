// prefill_swa.cu -- chunked prefill attention of a sliding-window layer (sm_103a,
// tcgen05).
//
// What it computes [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s1
// "为什么选择 Hybrid SWA 架构": an SWA layer attends only the last 128 tokens, so its
// prefill work is set by the window, not the context; s2 "KVCache系统重构": the SWA KV
// Pool is a ring of W slots per sequence]: request r has P cached tokens and C new
// rows at positions P + i; row i attends positions max(0, P + i - W + 1) .. P + i,
// those below P read from the sequence's ring (slot = position mod W), the others
// from the chunk's own k_new / v_new.
//
// Why a kernel of its own: a row of a sliding layer attends at most W keys, so per
// chunk row the launch does 4 d W Hq flops (2.1 MFLOP at W = 128, Hq = 32) while it
// reads the row's q and writes its output (16 KB) plus the row's new K / V (2 KB):
// about 115 flops per byte, below the ~270 per byte at which GB300's tensor cores
// and HBM balance.  HBM bounds it.  So q and out stream through once, every K / V
// byte loaded serves all G query heads that share it, and a row's tensor work is one
// S tile and one PV tile.
//
// Design (persistent, one CTA per SM, tiles dealt round-robin):
//  * A tile is one KV head h and 128 / G consecutive chunk rows i0 .. of one request.
//    Its M = 128 query rows are those positions times the G query heads sharing h
//    (row = position * G + head): one TMA box of q gives them.
//  * Its keys are two regions in shared memory, loaded by TMA in 16-row boxes:
//      ring region   prefix positions a0 .. ceil16(P) - 1 (a0 = the first position a
//                    row of the tile sees, rounded down to 16) read from ring slots
//                    position mod W -- 16-aligned blocks never wrap the ring;
//      chunk region  chunk rows max(0, i0 - W) .. i0 + 128/G - 1.
//    At most W + 128/G + 16 keys (160 for W = 128, G = 8), so S = Q K^T is one MMA
//    chain of N <= 160 columns and each row's softmax is exact: the row maximum is
//    known before any exponential, no running max, no rescale of O.
//  * Two shared-memory stages (q + K, and V, of one tile, each freed as soon as the
//    MMA that reads it has run), two TMEM S slots (S, then P over it) and one O
//    region; tile n uses stage and slot n mod 2.  Warp 0 = TMA producer; warp 1 = TMEM owner and
//    single-thread MMA issuer (S(n), then PV(n-1)); warps 2-9 = softmax and epilogue,
//    two warps per TMEM lane quarter (TMEM lane = query row), each taking half of
//    the row's key columns and half of its output columns, so that every SM
//    sub-partition has two softmax warps to interleave: the softmax of tile n reads
//    the half-row's scores from TMEM once and keeps them in registers for both
//    passes, the pair combines the row max and sum through TMEM, then the epilogue
//    of tile n - 1 reads O, after which PV(n) runs while the softmax of tile n + 1
//    does -- whose S the tensor cores computed during tile n's softmax.
//  * TMEM: S slots at columns [0, N) and [192, 192 + N), P as bf16 pairs over the
//    slot's first N/2 columns, O at [384, 512), written by PV(n) once the epilogue
//    of tile n - 1 has read it.  The epilogue divides O by the row sum (of the bf16 P
//    the MMA used) and writes bf16.
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kBM = 128;                   // query rows per tile (positions x heads)
constexpr int kD = 128;
constexpr int kKvRows = 160;               // key capacity of a stage
constexpr int kBox = 16;                   // rows per K / V TMA box
constexpr int kQHalf = kBM * 128;          // 128 rows x 64 bf16 (one swizzle column block)
constexpr int kKvHalf = kKvRows * 128;
constexpr int kThreads = 320;
// TMEM: two S slots of kKvRows columns (tile n in slot n mod 2; P as bf16 pairs over
// S's first columns) 192 columns apart, and one O region that every tile's PV
// accumulates into in turn: S(n + 2) can then run while the epilogue of tile n
// still reads O -- only PV(n + 1) waits for it.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlotCols = 192;
constexpr uint32_t kColO = 2 * kSlotCols;
static_assert(kColO + 128 <= kTmemCols, "two S slots and O fit in TMEM");
// Columns of an S slot past S (never written by an MMA) through which the two
// halves of a row pass values (per lane, so per row): the halves' maxima of the
// slot's tile, then their row sums, read by the tile's epilogue.
constexpr uint32_t kColMax = kKvRows;         // + half
constexpr uint32_t kColSum = kKvRows + 2;     // + half
static_assert(kColSum + 2 <= kSlotCols, "exchange columns inside the slot");

struct TileInfo {
    int32_t valid;     // 0: a bad request -- nothing loaded, nothing written
    int32_t i0;        // first chunk row of the tile
    int32_t C, P;      // chunk rows and prefix length of the request
    int32_t row_base;  // the request's first row in q / k_new / out
    int32_t h;         // KV head
    int32_t nr, nc;    // keys in the ring and chunk regions (multiples of 16)
    int32_t a0, z0;    // first position of the ring region, first chunk row
};

struct SwaSmem {
    alignas(1024) uint8_t q[2][2 * kQHalf];
    alignas(1024) uint8_t k[2][2 * kKvHalf];
    alignas(1024) uint8_t v[2][2 * kKvHalf];
    // stage s: q + K loaded / free (free once S has read them), V loaded / free
    alignas(8) uint64_t full_qk[2], empty_qk[2], full_v[2], empty_v[2];
    uint64_t s_full[2], p_full[2];  // per S slot
    uint64_t o_full, o_free;        // O holds PV(n) / O read by the epilogue of tile n
    // description of tile k in info[k mod 4], published by info_full[k mod 4]: the
    // producer writes tile k + 4's once stage k mod 2 frees for it, i.e. after
    // S(k + 2), which the MMA thread issues after PV(k), which waits for every
    // softmax warp's P of tile k -- so no slot is overwritten while its tile's warps
    // may still read it, and its barrier cannot complete the next phase before they
    // have waited on this one.  (The softmax warps must not wait on
    // full_qk for this: that barrier completes again for tile k + 2 as soon as S(k)
    // has read stage k mod 2, possibly before a late waiter looks, and a parity wait
    // cannot tell two completions from none.)
    TileInfo info[4];
    uint64_t info_full[4];
    uint32_t tmem_base;
    int32_t total;
    int32_t red[kThreads / 32];
};

__device__ __forceinline__ int chunk_rows(const PrefillParams &p, int r)
{
    return __ldg(p.cu_rows + r + 1) - __ldg(p.cu_rows + r);
}

__device__ __forceinline__ int tiles_of(const PrefillParams &p, int r, int ppt)
{
    const int C = chunk_rows(p, r);
    return C > 0 ? ((C + ppt - 1) / ppt) * p.Hkv : 0;
}

// Bit c set iff column c0 + c lies in [lo, hi).
__device__ __forceinline__ uint32_t range_mask(int c0, int lo, int hi)
{
    const int a = min(max(lo - c0, 0), 32), b = min(max(hi - c0, 0), 32);
    if (b <= a)
        return 0u;
    const uint32_t below_b = b == 32 ? 0xffffffffu : (1u << b) - 1u;
    return below_b & ~((1u << a) - 1u);  // a < b <= 32, so a < 32
}

// Scores of the 16 columns whose bit in vm is clear become -inf; skipped when every
// lane of the warp sees the whole chunk (the common case inside a tile).
__device__ __forceinline__ void mask_chunk16(uint32_t (&r)[16], uint32_t vm)
{
    if (__all_sync(0xffffffffu, (vm & 0xffffu) == 0xffffu))
        return;
#pragma unroll
    for (int c = 0; c < 16; ++c)
        if (!(vm & (1u << c)))
            r[c] = __float_as_uint(-INFINITY);
}

// Request cursor of the producer's tile walk (tiles are dealt in request order).
struct Cursor {
    int r, acc, tr;  // request, tiles of requests < r, tiles of request r
};

// Describe tile t (the cursor only moves forward): its request, rows and the two key
// regions; reports a bad request once (on its first tile) and marks it invalid.
__device__ __forceinline__ void describe(const PrefillParams &p, int ppt, int t, Cursor &cur,
                                         TileInfo &inf, int &rr, bool may_report)
{
    while (t >= cur.acc + cur.tr) {
        cur.acc += cur.tr;
        ++cur.r;
        cur.tr = tiles_of(p, cur.r, ppt);
    }
    const int r = cur.r;
    const int loc = t - cur.acc;
    const int blk = loc / p.Hkv;
    inf.h = loc % p.Hkv;
    inf.i0 = blk * ppt;
    inf.row_base = __ldg(p.cu_rows + r);
    inf.C = __ldg(p.cu_rows + r + 1) - inf.row_base;
    inf.P = __ldg(p.prefix_len + r);
    const int seq = __ldg(p.seq_idx + r);
    const bool report = may_report && inf.h == 0 && blk == 0;  // one report per request
    inf.valid = 1;
    if (inf.row_base < 0 || inf.row_base + inf.C > p.rows) {
        if (report)
            set_err(p.dev_err, HSA_DEVERR_BAD_LEN);  // rows outside q / out
        inf.valid = 0;
    } else if (seq < 0 || seq >= p.batch) {
        if (report)
            set_err(p.dev_err, HSA_DEVERR_BAD_SEQ);
        inf.valid = 0;
    } else if (inf.P < 0) {
        if (report)
            set_err(p.dev_err, HSA_DEVERR_BAD_LEN);
        inf.valid = 0;
    }
    rr = 0;
    inf.nr = 0;
    inf.a0 = 0;
    if (inf.valid && inf.P > 0 && inf.i0 < p.W - 1) {
        // some row of the tile still sees the prefix
        rr = __ldg(p.ring_row + seq);
        if (rr < 0 || rr >= p.n_ring_rows) {
            if (report)
                set_err(p.dev_err, HSA_DEVERR_BAD_RING);  // prefix keys absent
        } else {
            inf.a0 = max(0, inf.P + inf.i0 - p.W + 1) & ~(kBox - 1);
            inf.nr = ((inf.P + kBox - 1) & ~(kBox - 1)) - inf.a0;
        }
    }
    inf.z0 = max(0, inf.i0 - p.W);
    inf.nc = inf.i0 + ppt - inf.z0;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_swa_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmNK,
                       const __grid_constant__ CUtensorMap tmNV, const __grid_constant__ CUtensorMap tmRK,
                       const __grid_constant__ CUtensorMap tmRV, const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    SwaSmem &sh = *reinterpret_cast<SwaSmem *>(
        align_smem_1024(smem_raw));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ppt = kBM / p.G;  // positions per tile

    // ---- tiles of the launch: Hkv x sum_r ceil(C_r / ppt) ------------------------
    {
        int local = 0;
        for (int r = tid; r < p.R; r += kThreads)
            local += tiles_of(p, r, ppt);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            local += __shfl_xor_sync(0xffffffffu, local, o);
        if (lane == 0)
            sh.red[warp] = local;
        __syncthreads();
        if (tid == 0) {
            int t = 0;
            for (int w = 0; w < kThreads / 32; ++w)
                t += sh.red[w];
            sh.total = t;
        }
        __syncthreads();
    }
    const int total = sh.total;
    const int n_my = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (n_my == 0)
        return;  // the whole CTA, before any barrier or TMEM is set up

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.full_qk[s], 1);
            mbar_init(&sh.empty_qk[s], 1);
            mbar_init(&sh.full_v[s], 1);
            mbar_init(&sh.empty_v[s], 1);
            mbar_init(&sh.s_full[s], 1);
            mbar_init(&sh.p_full[s], 8 * 32);
        }
        mbar_init(&sh.o_full, 1);
        mbar_init(&sh.o_free, 8 * 32);
        for (int j = 0; j < 4; ++j)
            mbar_init(&sh.info_full[j], 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ================================================================ producer
        // The whole warp: lane 0 waits for a stage and arms its barrier, then every
        // lane issues one TMA box (a tile's q + K or V is up to 22 boxes of 16 rows x
        // 64 columns: 16-row blocks never wrap the ring), so no single thread walks
        // the boxes one by one.
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmNK);
            tma_prefetch_desc(&tmNV);
            tma_prefetch_desc(&tmRK);
            tma_prefetch_desc(&tmRV);
        }
        const uint64_t pol_q = policy_evict_first();  // q is read once
        const uint64_t pol_kv = policy_evict_last();  // a key serves ~W / ppt tiles
        // Loads go out in the order their stages free up: q + K of tile k (stage k mod
        // 2 is free once S(k-2) has read it), then V of tile k-1 (free once PV(k-3)
        // has); a tile's description is read one tile ahead (by every lane, so that
        // each knows the boxes), its global loads overlapping the waits.
        Cursor cur{0, 0, tiles_of(p, 0, ppt)};
        TileInfo inf_next, inf_prev{};
        int rr_next = 0, rr_prev = 0;
        describe(p, ppt, (int)blockIdx.x, cur, inf_next, rr_next, lane == 0);
        // box e of a K or V region: e & 1 = 64-column half, e >> 1 = 16-row block
        // (ring blocks first, then chunk blocks)
        auto issue_kv = [&](uint8_t *dst, const TileInfo &inf, int rr, const CUtensorMap *ring,
                            const CUtensorMap *chunk, uint64_t *bar, int e) {
            const int half = e & 1, b = (e >> 1) * kBox;
            uint8_t *d = dst + half * kKvHalf + b * 128;
            if (b < inf.nr) {
                const int y = (rr * p.Hkv + inf.h) * p.W + (inf.a0 + b) % p.W;
                tma_load_2d(d, ring, bar, half * 64, y, pol_kv);
            } else {
                const int z = inf.row_base + inf.z0 + (b - inf.nr);
                tma_load_3d(d, chunk, bar, half * 64, inf.h, z, pol_kv);
            }
        };
        auto load_v = [&](int j, const TileInfo &inf, int rr) -> bool {
            const int s = j & 1;
            int ok_w = 1;
            if (lane == 0) {
                ok_w = mbar_wait_sleep(&sh.empty_v[s], ((j >> 1) & 1) ^ 1);
                if (ok_w) {
                    if (inf.valid)
                        mbar_arrive_expect_tx(&sh.full_v[s], (inf.nr + inf.nc) * 256);
                    else
                        mbar_arrive(&sh.full_v[s]);
                }
            }
            ok_w = __shfl_sync(0xffffffffu, ok_w, 0);  // also orders the copies after the arm
            if (ok_w && inf.valid && lane < 2 * (inf.nr + inf.nc) / kBox)
                issue_kv(sh.v[s], inf, rr, &tmRV, &tmNV, &sh.full_v[s], lane);
            return ok_w != 0;
        };
        bool ok = true;
        for (int k = 0; k < n_my; ++k) {
            const TileInfo inf = inf_next;
            const int rr = rr_next;
            if (k + 1 < n_my)
                describe(p, ppt, (int)blockIdx.x + (k + 1) * (int)gridDim.x, cur, inf_next, rr_next,
                         lane == 0);
            const int s = k & 1;
            uint64_t *bar = &sh.full_qk[s];
            int ok_w = 1;
            if (lane == 0) {
                ok_w = mbar_wait_sleep(&sh.empty_qk[s], ((k >> 1) & 1) ^ 1);
                if (ok_w) {
                    sh.info[k & 3] = inf;
                    mbar_arrive(&sh.info_full[k & 3]);  // publishes it to the softmax warps
                    if (inf.valid)
                        mbar_arrive_expect_tx(bar, 2 * kQHalf + (inf.nr + inf.nc) * 256);
                    else
                        mbar_arrive(bar);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok_w, 0)) {
                ok = false;
                break;
            }
            if (inf.valid) {
                const int nk = 2 * (inf.nr + inf.nc) / kBox;  // K boxes, <= 20
                if (lane < nk) {
                    issue_kv(sh.k[s], inf, rr, &tmRK, &tmNK, bar, lane);
                } else if (lane < nk + 2) {
                    // q: ppt positions x the G query heads of KV head h (rows past the
                    // request are masked; rows past the tensor are zero-filled)
                    const int half = lane - nk;
                    tma_load_3d(sh.q[s] + half * kQHalf, &tmQ, bar, half * 64, inf.h * p.G,
                                inf.row_base + inf.i0, pol_q);
                }
            }
            if (k > 0 && !load_v(k - 1, inf_prev, rr_prev)) {
                ok = false;
                break;
            }
            inf_prev = inf;
            rr_prev = rr;
        }
        if (ok && !load_v(n_my - 1, inf_prev, rr_prev))
            ok = false;
        if (lane == 0) {
            if (!ok)
                set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
            // drain: no TMA write may still be in flight when the CTA exits
            for (int j = max(0, n_my - 2); j < n_my; ++j) {
                mbar_wait_sleep(&sh.full_qk[j & 1], (j >> 1) & 1);
                mbar_wait_sleep(&sh.full_v[j & 1], (j >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t dhi = smem_desc_sw128_hi(1024);
            const uint32_t id_pv = idesc_bf16_f32(kBM, kD, 0, 1);
            uint32_t q_lo[2], k_lo[2], v_lo[2];
            for (int s = 0; s < 2; ++s) {
                q_lo[s] = smem_desc_sw128_lo(smem_u32(sh.q[s]), 16);
                k_lo[s] = smem_desc_sw128_lo(smem_u32(sh.k[s]), 16);
                v_lo[s] = smem_desc_sw128_lo(smem_u32(sh.v[s]), kKvHalf);
            }
            int n_prev = 0;  // keys of the previous tile (0: invalid, no PV)
            // O = P V over n keys: P from TMEM over S of slot s (k-step ks: 16 keys =
            // 8 columns of bf16 pairs), V the MN-major tile (16 key rows = 2048 bytes)
            auto issue_pv = [&](int s, int n) {
                const uint32_t base = tmem + s * kSlotCols;
                if (n > 0) {
                    tc_mma_ts_k<0>(tmem + kColO, base, desc_join(v_lo[s], dhi), id_pv);
                    for (int ks = 1; ks < n / 16; ++ks)
                        tc_mma_ts_k<1>(tmem + kColO, base + ks * 8,
                                       desc_join(v_lo[s] + ks * (2048 >> 4), dhi), id_pv);
                }
                tc_commit(&sh.o_full);
                tc_commit(&sh.empty_v[s]);
            };
            // PV(j) waits for its P, its V and the epilogue of tile j - 1 (O free)
            auto wait_pv = [&](int j) -> bool {
                const int sp = j & 1;
                const uint32_t php = (j >> 1) & 1;
                return mbar_wait_sleep(&sh.p_full[sp], php) && mbar_wait_sleep(&sh.full_v[sp], php) &&
                       mbar_wait_sleep(&sh.o_free, (j & 1) ^ 1);
            };
            bool ok = true;
            for (int k = 0; k < n_my && ok; ++k) {
                const int s = k & 1;
                const uint32_t ph = (k >> 1) & 1;
                // slot s last held tile k - 2, whose P PV(k - 2) -- issued earlier by
                // this thread, so run earlier -- has read
                if (!mbar_wait_sleep(&sh.full_qk[s], ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const TileInfo &inf = sh.info[k & 3];
                const int n = inf.valid ? inf.nr + inf.nc : 0;
                if (n > 0) {
                    // S = Q K^T over d = 128 in 8 k-steps of 16 (32 bytes inside a
                    // 128-byte swizzle row; steps 4-7 in the second 64-column block)
                    const uint32_t id_s = idesc_bf16_f32(kBM, n, 0, 0);
                    const uint32_t d = tmem + s * kSlotCols;
                    tc_mma_ss_k<0>(d, desc_join(q_lo[s], dhi), desc_join(k_lo[s], dhi), id_s);
#pragma unroll
                    for (int ks = 1; ks < kD / 16; ++ks) {
                        const uint32_t oq = (ks >> 2) * (kQHalf >> 4) + (ks & 3) * 2;
                        const uint32_t okv = (ks >> 2) * (kKvHalf >> 4) + (ks & 3) * 2;
                        tc_mma_ss_k<1>(d, desc_join(q_lo[s] + oq, dhi), desc_join(k_lo[s] + okv, dhi),
                                       id_s);
                    }
                }
                tc_commit(&sh.s_full[s]);
                tc_commit(&sh.empty_qk[s]);  // q and K of stage s are free once S has run
                if (k > 0) {
                    if (!wait_pv(k - 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv((k - 1) & 1, n_prev);
                }
                n_prev = n;
            }
            if (ok) {
                if (wait_pv(n_my - 1)) {
                    tc_fence_after();
                    issue_pv((n_my - 1) & 1, n_prev);
                } else {
                    ok = false;
                }
            }
            if (!ok)
                set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
        }
    } else {
        // ================================================================ softmax + epilogue
        // Warps 2-9: two per TMEM lane quarter, one query row per pair of threads.
        // Half 0 (warps 2-5) takes key columns [0, 80) and output columns [0, 64),
        // half 1 (warps 6-9) key columns [80, 160) and output columns [64, 128); the
        // two warps of a quarter meet at a 64-thread barrier of their own to combine
        // the row max (every tile) and the row sum (for the epilogue).  Every tile in
        // turn: the softmax of tile k, then the epilogue of tile k - 1, which frees O
        // for PV(k).
        const int wq = warp & 3;             // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;    // key / output column half
        const int m = wq * 32 + lane;        // query row of the tile: position m / G, head m % G
        const int u = m / p.G, g = m % p.G;
        const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t pair_bar = 1 + wq;    // named barrier of the quarter's two warps
        TileInfo prev{};
        // A wait that gives up never leaves one warp of a pair behind at a barrier:
        // `ok` (this warp's waits so far) goes into the pair barrier of the next tile,
        // which both warps reach and leave with the same answer.
        bool ok = true;
        for (int k = 0; k <= n_my; ++k) {
            TileInfo inf{};
            const int s = k & 1;
            const uint32_t base = lane_addr + s * kSlotCols;
            bool w_ok = ok;
            if (k < n_my && w_ok)
                w_ok = mbar_wait_sleep(&sh.info_full[k & 3], (k >> 2) & 1) &&
                       mbar_wait_sleep(&sh.s_full[s], (k >> 1) & 1);
            w_ok = __all_sync(0xffffffffu, w_ok);  // the TMEM reads below are warp-wide
            // This half's <= 80 scores: one TMEM read of each 16-column chunk, one
            // wait, kept in registers for both passes.  Invisible scores become -inf
            // (skipped for a chunk every row of the warp sees whole).
            constexpr int kChunks = kKvRows / 32;  // 16-column chunks per half
            const int c_base = half * kChunks * 16;
            uint32_t sr[kChunks][16];
            int n = 0;
            if (k < n_my && w_ok) {
                tc_fence_after();
                inf = sh.info[k & 3];
                const int i = inf.i0 + u;
                const bool row_ok = inf.valid && i < inf.C;
                n = inf.valid ? inf.nr + inf.nc : 0;
                // visible key columns: ring region [rlo, rhi), chunk region [clo, chi)
                int rlo = 0, rhi = 0, clo = 0, chi = 0;
                if (row_ok) {
                    if (inf.nr > 0) {
                        rlo = max(0, inf.P + i - p.W + 1) - inf.a0;
                        rhi = max(rlo, inf.P - inf.a0);
                    }
                    clo = inf.nr + max(0, i - p.W + 1) - inf.z0;
                    chi = inf.nr + i + 1 - inf.z0;
                }
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci)
                    if (c_base + ci * 16 < n)
                        tmem_ld16(base + c_base + ci * 16, sr[ci]);
                tmem_wait_ld();
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci) {
                    const int c0 = c_base + ci * 16;
                    if (c0 < n) {
                        mask_chunk16(sr[ci], range_mask(c0, rlo, rhi) | range_mask(c0, clo, chi));
#pragma unroll
                        for (int c = 0; c < 16; c += 8) {
                            m4[0] = fmax3(m4[0], __uint_as_float(sr[ci][c + 0]), __uint_as_float(sr[ci][c + 1]));
                            m4[1] = fmax3(m4[1], __uint_as_float(sr[ci][c + 2]), __uint_as_float(sr[ci][c + 3]));
                            m4[2] = fmax3(m4[2], __uint_as_float(sr[ci][c + 4]), __uint_as_float(sr[ci][c + 5]));
                            m4[3] = fmax3(m4[3], __uint_as_float(sr[ci][c + 6]), __uint_as_float(sr[ci][c + 7]));
                        }
                    }
                }
                tmem_st1(base + kColMax + half,
                         __float_as_uint(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]))));
                tmem_wait_st();
            }
            // the pair meets: both halves' maxima (and, for the epilogue below, the
            // other half's row sum of tile k - 1) are in TMEM, and both have read
            // their S before either writes P over S's first columns
            tc_fence_before();
            if (!named_bar_and(pair_bar, 64, w_ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (k < n_my) {
                if (n > 0) {
                    uint32_t m0, m1;
                    tmem_ld2(base + kColMax, m0, m1);
                    tmem_wait_ld();
                    const float mx = fmaxf(__uint_as_float(m0), __uint_as_float(m1));
                    const float mb = mx == -INFINITY ? 0.f : mx * p.scale_log2;
                    // P = 2^(s scale log2e - max) as bf16 pairs: key column c goes to P
                    // column c / 2 (chunk ci to columns c_base / 2 + 8 ci .. + 7; a
                    // masked score gives 2^-inf = 0).  The row sum takes the rounded P
                    // the PV MMA uses, in two independent f32x2 accumulators.
                    const uint64_t sc2 = f2_make(p.scale_log2, p.scale_log2);
                    const uint64_t nb2 = f2_make(-mb, -mb);
                    uint64_t acc2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
                    for (int ci = 0; ci < kChunks; ++ci) {
                        if (c_base + ci * 16 < n) {
                            uint32_t pk[8];
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const uint64_t x2 = f2_fma(f2_make(__uint_as_float(sr[ci][2 * c]),
                                                                   __uint_as_float(sr[ci][2 * c + 1])),
                                                           sc2, nb2);
                                float x0, x1;
                                f2_split(x2, x0, x1);
                                pk[c] = pack_bf16(fast_exp2(x0), fast_exp2(x1));
                                acc2[c & 1] = f2_add(acc2[c & 1], f2_make(bf16_lo(pk[c]), bf16_hi(pk[c])));
                            }
                            tmem_st8(base + c_base / 2 + ci * 8, pk);
                        }
                    }
                    float a0, a1, b0, b1;
                    f2_split(acc2[0], a0, a1);
                    f2_split(acc2[1], b0, b1);
                    tmem_st1(base + kColSum + half, __float_as_uint((a0 + a1) + (b0 + b1)));
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&sh.p_full[s]);
            }
            // ---- epilogue of tile k - 1: O / l -> bf16, this half's 64 columns ----
            // (the other half's row sum of tile k - 1 was written before it reached
            // this iteration's pair barrier)
            if (k > 0) {
                const int j = k - 1;
                const int s = j & 1;
                if (!__all_sync(0xffffffffu, mbar_wait_sleep(&sh.o_full, j & 1))) {
                    ok = false;  // left at the next pair barrier, by both warps
                    continue;
                }
                tc_fence_after();
                if (prev.valid) {
                    const int i = prev.i0 + u;
                    const bool row_ok = i < prev.C;
                    uint32_t l0, l1;
                    tmem_ld2(lane_addr + s * kSlotCols + kColSum, l0, l1);
                    tmem_wait_ld();
                    const float l = __uint_as_float(l0) + __uint_as_float(l1);
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    const uint32_t base = lane_addr + kColO + half * 64;
                    __nv_bfloat16 *dst =
                        p.out + ((int64_t)(prev.row_base + i) * p.Hq + prev.h * p.G + g) * kD +
                        half * 64;
                    uint32_t o32[2][32];
                    tmem_ld32(base, o32[0]);
                    tmem_ld32(base + 32, o32[1]);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
                            for (int c = 0; c < 32; c += 8) {
                                uint4 w;
                                w.x = pack_bf16(__uint_as_float(o32[c2][c + 0]) * inv, __uint_as_float(o32[c2][c + 1]) * inv);
                                w.y = pack_bf16(__uint_as_float(o32[c2][c + 2]) * inv, __uint_as_float(o32[c2][c + 3]) * inv);
                                w.z = pack_bf16(__uint_as_float(o32[c2][c + 4]) * inv, __uint_as_float(o32[c2][c + 5]) * inv);
                                w.w = pack_bf16(__uint_as_float(o32[c2][c + 6]) * inv, __uint_as_float(o32[c2][c + 7]) * inv);
                                *reinterpret_cast<uint4 *>(dst + c2 * 32 + c) = w;
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sh.o_free);
            }
            prev = inf;
        }
        if (!ok)
            set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool prefill_swa_supported(int W, int G)
{
    return G >= 1 && G <= 8 && kBM % G == 0 && W % kBox == 0 && W + kBM / G + kBox <= kKvRows;
}

cudaError_t launch_prefill_swa(const CUtensorMap &tmQ, const CUtensorMap &tmNK, const CUtensorMap &tmNV,
                               const CUtensorMap &tmRK, const CUtensorMap &tmRV, const PrefillParams &p,
                               int sms, cudaStream_t stream)
{
    const size_t smem = sizeof(SwaSmem) + 1024;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_swa_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    // tiles_per_req_bound bounds sum_r ceil(C_r / 128); a tile here holds 128 / G rows
    const int64_t tiles = ((int64_t)p.rows / (kBM / p.G) + p.R) * p.Hkv;
    const int64_t ctas = tiles < sms ? tiles : sms;
    if (ctas <= 0)
        return cudaSuccess;
    prefill_swa_kernel<<<(unsigned)ctas, kThreads, smem, stream>>>(tmQ, tmNK, tmNV, tmRK, tmRV, p);
    return cudaGetLastError();
}

}  // namespace hsa

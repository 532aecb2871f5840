// prefill.cu -- chunked prefill attention on a cached prefix (sm_103a, tcgen05).
//
// What it computes [youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s1
// "为什么选择 Hybrid SWA 架构": SWA layers attend only the last 128 tokens, so their
// prefill compute falls to the window; hotdry.top "MiMo-V2.5 ultra-speed inference
// architecture", "PD 分离与长度分桶": chunked prefill]: request r has P cached
// tokens and C new rows at positions P + i.  Row i attends
//   full layers:    positions 0 .. P + i
//   sliding layers: positions P + i - W + 1 .. P + i
// with positions < P read from the pools (Full KV Pool pages through the block
// table, or the SWA ring) and positions >= P from the chunk's own k_new / v_new.
//
// Design: one CTA per (request, pair of 128-row query tiles A and B, query head);
// both tiles share every 128-key K / V tile.  Ten warps:
//   warp 0    TMA producer: Q_A and Q_B once, then K and V tiles into a 2-stage
//             ring (128-byte swizzle; a prefix tile is two 64-token pages)
//   warp 1    TMEM owner (S_A, S_B, O_A, O_B: 4 x 128 columns) and MMA issuer
//             (one thread): S = Q K^T, O += P V with P read from TMEM
//   warps 2-5 softmax of tile A, warps 6-9 softmax of tile B, one query row per
//             thread (TMEM lane = row): masks, running max raised lazily (O is
//             rescaled in TMEM only when the max grows by more than 2^8), P written
//             back over S as bf16
// The MMA thread issues PV_A(n), then S_A(n+1), then PV_B(n), then S_B(n+1), so
// the tensor cores work on one tile while the other tile's warps run softmax, and
// each SM sub-partition holds two independent softmax warps.  Every key tile is
// run for both query tiles (a tile a row cannot see is simply masked: at most one
// extra 128-key tile per CTA).  The epilogue divides O by the row sum and writes
// bf16.
#include "hsa_device.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kD = 128;
constexpr int kHalfBytes = 128 * 128;      // 128 rows x 64 bf16 (one swizzle column block)
constexpr int kTileBytes = 2 * kHalfBytes; // 32 KB
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;            // S_A, S_B at 0 / 128; O_A, O_B at 256 / 384
constexpr float kRescaleSlack = 8.0f;      // log2 units: P may reach 2^8 before a rescale

struct PrefillSmem {
    alignas(1024) uint8_t q[2][kTileBytes];
    alignas(1024) uint8_t k[2][kTileBytes];
    alignas(1024) uint8_t v[2][kTileBytes];
    alignas(8) uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2], o_full;  // s_full / p_full per query tile
    uint32_t tmem_base;
    int32_t r, qp, P, C, seq, row0;
};

struct Sched {
    int nt;          // key tiles (union over both query tiles)
    int n_fixed;     // prefix tiles (full) or ring tiles (sliding) before the chunk tiles
    int m_lo;        // first chunk tile
};

// Key tiles of the CTA whose query tiles start at rows i0 (A) and i0 + 128 (B, if
// has_b): full layers read every prefix tile and chunk tiles 0 .. last row / 128;
// sliding layers read the ring if a row still sees the prefix, and the chunk tiles
// inside the window.
__device__ __forceinline__ Sched make_sched(const PrefillParams &p, int P, int i0, bool has_b)
{
    const int i_last = i0 + (has_b ? 2 * kBM : kBM) - 1;  // last row of the CTA (may pad)
    Sched s;
    if (!p.ring_mode) {
        s.n_fixed = (P + kBN - 1) / kBN;
        s.m_lo = 0;
    } else {
        s.n_fixed = (P > 0 && i0 < p.W - 1) ? (p.W + kBN - 1) / kBN : 0;
        const int lo = i0 - p.W + 1;
        s.m_lo = lo > 0 ? lo / kBN : 0;
    }
    s.nt = s.n_fixed + (i_last / kBN - s.m_lo + 1);
    return s;
}

__device__ __forceinline__ bool page_ok(const PrefillParams &p, int seq, int page, int *blk)
{
    if (page >= p.max_blocks)
        return false;
    const int b = __ldg(p.block_tables + (int64_t)seq * p.max_blocks + page);
    if (b < 0 || b >= p.num_blocks)
        return false;
    *blk = b;
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmPK, const __grid_constant__ CUtensorMap tmPV,
                   const __grid_constant__ CUtensorMap tmNK, const __grid_constant__ CUtensorMap tmNV,
                   const __grid_constant__ CUtensorMap tmQ, const PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem &sh = *reinterpret_cast<PrefillSmem *>(
        align_smem_1024(smem_raw));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int hq = blockIdx.x % p.Hq;
    const int h = hq / p.G;

    // ---- which (request, pair of query tiles) this CTA owns -----------------
    if (tid == 0) {
        const int tl = blockIdx.x / p.Hq;
        int acc = 0, found = -1, qp = 0;
        for (int r = 0; r < p.R; ++r) {
            const int C = __ldg(p.cu_rows + r + 1) - __ldg(p.cu_rows + r);
            const int np = C > 0 ? (C + 2 * kBM - 1) / (2 * kBM) : 0;
            if (tl < acc + np) {
                found = r;
                qp = tl - acc;
                break;
            }
            acc += np;
        }
        sh.r = found;
        if (found >= 0) {
            sh.qp = qp;
            sh.P = __ldg(p.prefix_len + found);
            sh.C = __ldg(p.cu_rows + found + 1) - __ldg(p.cu_rows + found);
            sh.seq = __ldg(p.seq_idx + found);
            sh.row0 = __ldg(p.cu_rows + found) + qp * 2 * kBM;
            if (sh.seq < 0 || sh.seq >= p.batch) {
                if (hq == 0)
                    set_err(p.dev_err, HSA_DEVERR_BAD_SEQ);
                sh.r = -1;
            } else if (sh.P < 0) {
                if (hq == 0)
                    set_err(p.dev_err, HSA_DEVERR_BAD_LEN);
                sh.r = -1;
            }
        }
    }
    __syncthreads();
    if (sh.r < 0)
        return;  // past the last tile pair (grid is an upper bound) or a bad request
    const int P = sh.P, C = sh.C, seq = sh.seq, i0 = sh.qp * 2 * kBM, row0 = sh.row0;
    const bool has_b = i0 + kBM < C;
    const Sched sc = make_sched(p, P, i0, has_b);

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.v_empty[s], 1);
            mbar_init(&sh.s_full[s], 1);
            mbar_init(&sh.p_full[s], 4 * 32);
        }
        mbar_init(&sh.o_full, 1);
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
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmPK);
            tma_prefetch_desc(&tmPV);
            tma_prefetch_desc(&tmNK);
            tma_prefetch_desc(&tmNV);
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            mbar_arrive_expect_tx(&sh.q_full, (has_b ? 2 : 1) * kTileBytes);
            for (int t = 0; t < (has_b ? 2 : 1); ++t) {
                tma_load_3d(sh.q[t], &tmQ, &sh.q_full, 0, hq, row0 + t * kBM, pol_stream);
                tma_load_3d(sh.q[t] + kHalfBytes, &tmQ, &sh.q_full, 64, hq, row0 + t * kBM,
                            pol_stream);
            }
            int ring_row = 0;
            if (p.ring_mode) {
                ring_row = __ldg(p.ring_row + seq);
                if (ring_row < 0 || ring_row >= p.n_ring_rows) {
                    if (hq == 0 && sh.qp == 0)
                        set_err(p.dev_err, HSA_DEVERR_BAD_RING);
                    ring_row = 0;
                }
            }
            bool ok = true;
            for (int n = 0; n < sc.nt && ok; ++n) {
                const int s = n & 1;
                const uint32_t ph = (n >> 1) & 1;
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    uint64_t *empty = kv ? &sh.v_empty[s] : &sh.k_empty[s];
                    uint64_t *full = kv ? &sh.v_full[s] : &sh.k_full[s];
                    uint8_t *dst = kv ? sh.v[s] : sh.k[s];
                    const CUtensorMap *pool = kv ? &tmPV : &tmPK;
                    const CUtensorMap *nw = kv ? &tmNV : &tmNK;
                    if (!mbar_wait_sleep(empty, ph ^ 1)) {
                        set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full, kTileBytes);
                    if (n < sc.n_fixed) {
                        // two 64-key blocks: pool pages (full) or ring slot blocks (sliding)
                        for (int pg = 0; pg < 2; ++pg) {
                            int32_t y;
                            if (!p.ring_mode) {
                                int page = 2 * n + pg;
                                if (page * 64 >= P)
                                    page = 2 * n;  // past the prefix: reload, masked
                                int blk = 0;
                                if (!page_ok(p, seq, page, &blk)) {
                                    if (kv == 0)
                                        set_err(p.dev_err, HSA_DEVERR_BAD_BLOCK);
                                    blk = 0;  // finite stand-in, masked by the softmax warps
                                }
                                y = (blk * p.Hkv + h) * 64;
                            } else {
                                int sb = 2 * n + pg;
                                if (sb * 64 >= p.W)
                                    sb = 2 * n;
                                y = (ring_row * p.Hkv + h) * p.W + sb * 64;
                            }
                            tma_load_2d(dst + pg * 8192, pool, full, 0, y, pol_keep);
                            tma_load_2d(dst + kHalfBytes + pg * 8192, pool, full, 64, y, pol_keep);
                        }
                    } else {
                        const int m = sc.m_lo + (n - sc.n_fixed);
                        const int z = row0 - i0 + m * kBN;  // chunk row of key tile m
                        tma_load_3d(dst, nw, full, 0, h, z, pol_keep);
                        tma_load_3d(dst + kHalfBytes, nw, full, 64, h, z, pol_keep);
                    }
                }
            }
            // drain: no TMA write may still be in flight when the CTA exits
            for (int s = 0; s < 2 && sc.nt > s; ++s) {
                const int last = s + ((sc.nt - 1 - s) / 2) * 2;
                const uint32_t ph = (last >> 1) & 1;
                mbar_wait_sleep(&sh.k_full[s], ph);
                mbar_wait_sleep(&sh.v_full[s], ph);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            const uint32_t id_pv = idesc_bf16_f32(kBM, kD, 0, 1);
            const int ntile = has_b ? 2 : 1;
            bool ok = mbar_wait_sleep(&sh.q_full, 0);
            // Descriptor low words of every operand tile (the high word is common:
            // SBO 1024, version 1, 128-byte swizzle); a k-step adds a constant to the
            // low word, so each MMA costs the issuing thread one or two integer adds
            const uint32_t dhi = smem_desc_sw128_hi(1024);
            const uint32_t q_lo[2] = {smem_desc_sw128_lo(smem_u32(sh.q[0]), 16),
                                      smem_desc_sw128_lo(smem_u32(sh.q[1]), 16)};
            const uint32_t k_lo[2] = {smem_desc_sw128_lo(smem_u32(sh.k[0]), 16),
                                      smem_desc_sw128_lo(smem_u32(sh.k[1]), 16)};
            const uint32_t v_lo[2] = {smem_desc_sw128_lo(smem_u32(sh.v[0]), kHalfBytes),
                                      smem_desc_sw128_lo(smem_u32(sh.v[1]), kHalfBytes)};
            // S_t = Q_t K_n^T into TMEM columns t * 128 (k-step ks: 16 d-columns, i.e.
            // 32 bytes inside a 128-byte swizzle row, 64 columns per 16 KB block)
            auto issue_s = [&](int t, int n) {
                const uint32_t qa = t ? q_lo[1] : q_lo[0];
                const uint32_t kb = (n & 1) ? k_lo[1] : k_lo[0];
                const uint32_t d = tmem + t * 128;
                tc_mma_ss_k<0>(d, desc_join(qa, dhi), desc_join(kb, dhi), id_s);
#pragma unroll
                for (int ks = 1; ks < kD / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * (kHalfBytes >> 4) + (ks & 3) * 2;
                    tc_mma_ss_k<1>(d, desc_join(qa + off, dhi), desc_join(kb + off, dhi), id_s);
                }
                tc_commit(&sh.s_full[t]);
            };
            // O_t += P_t V_n, P_t read from TMEM over S_t (k-step ks: 16 keys = 8 TMEM
            // columns of bf16 pairs, and 16 rows = 2048 bytes of the MN-major V tile)
            auto issue_pv = [&](int t, int n) {
                const uint32_t vb = (n & 1) ? v_lo[1] : v_lo[0];
                const uint32_t d = tmem + kColO + t * 128, a = tmem + t * 128;
                if (n > 0)
                    tc_mma_ts_k<1>(d, a, desc_join(vb, dhi), id_pv);
                else
                    tc_mma_ts_k<0>(d, a, desc_join(vb, dhi), id_pv);
#pragma unroll
                for (int ks = 1; ks < kBN / 16; ++ks)
                    tc_mma_ts_k<1>(d, a + ks * 8, desc_join(vb + ks * (2048 >> 4), dhi), id_pv);
            };
            if (ok && (ok = mbar_wait_sleep(&sh.k_full[0], 0))) {
                tc_fence_after();
                for (int t = 0; t < ntile; ++t)
                    issue_s(t, 0);
                tc_commit(&sh.k_empty[0]);
            }
            for (int n = 0; n < sc.nt && ok; ++n) {
                const int s = n & 1;
                const bool more = n + 1 < sc.nt;
                if (more && !mbar_wait_sleep(&sh.k_full[(n + 1) & 1], ((n + 1) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < ntile; ++t) {
                    // tile t's P of key tile n is in TMEM once its softmax warps arrive;
                    // S_t(n+1) is issued behind PV_t(n) (tcgen05 MMAs from one thread run
                    // in issue order, so PV reads P before S overwrites it)
                    if (!mbar_wait_sleep(&sh.p_full[t], n & 1) ||
                        (t == 0 && !mbar_wait_sleep(&sh.v_full[s], (n >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(t, n);
                    if (more)
                        issue_s(t, n + 1);
                }
                if (!ok)
                    break;
                if (more)
                    tc_commit(&sh.k_empty[(n + 1) & 1]);
                tc_commit(&sh.v_empty[s]);
            }
            if (ok) {
                tc_commit(&sh.o_full);
                mbar_wait_sleep(&sh.o_full, 0);  // every MMA done before TMEM is released
            } else {
                set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
            }
        }
    } else {
        // ================================================================ softmax
        const int t = (warp - 2) >> 2;  // query tile: 0 = A (warps 2-5), 1 = B (warps 6-9)
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int i = i0 + t * kBM + row;
        const bool tile_ok = t == 0 || has_b;
        const bool row_ok = tile_ok && i < C;
        const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t col_s = t * 128, col_o = kColO + t * 128;
        float m_used = -INFINITY, l = 0.f;
        // Full layers let the running max lag by up to 2^8 (few O rescales over long
        // rows).  Ring mode raises it exactly: its rows see at most W keys, some only
        // a handful, and then the dominant weight must stay exactly 1 (a lagging max
        // rounds it to bf16 like the rest, which at |o| ~ 2 costs a bf16 output ulp).
        const float slack = p.ring_mode ? 0.f : kRescaleSlack;
        int ring_row_ok = 1;
        if (p.ring_mode) {
            const int rr = __ldg(p.ring_row + seq);
            ring_row_ok = rr >= 0 && rr < p.n_ring_rows;
        }
        bool ok = true;
        for (int n = 0; n < sc.nt && tile_ok; ++n) {
            if (!mbar_wait_sleep(&sh.s_full[t], n & 1)) {
                set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
                ok = false;
                break;
            }
            // S_t(n) complete implies every earlier MMA (PV_t(n-1) included) completed
            tc_fence_after();
            // ---- visibility of the 128 keys of tile n for query row i ----------
            int lo = 0, hi = 0;
            bool ok0 = true, ok1 = true, ring = false;
            if (n < sc.n_fixed) {
                if (!p.ring_mode) {
                    hi = min(kBN, P - n * kBN);
                    int blk;
                    ok0 = page_ok(p, seq, 2 * n, &blk);
                    ok1 = (2 * n + 1) * 64 >= P || page_ok(p, seq, 2 * n + 1, &blk);
                } else {
                    ring = true;
                }
            } else {
                const int m = sc.m_lo + (n - sc.n_fixed);
                const int kb = m * kBN;
                hi = min(kBN, min(i, C - 1) - kb + 1);
                if (p.ring_mode)
                    lo = max(0, i - p.W + 1 - kb);
            }
            if (!row_ok)
                hi = 0;
            const bool whole_tile = !ring && lo == 0 && hi == kBN && ok0 && ok1;
            // ring slot s holds the latest prefix position below P congruent to s mod W,
            // P - 1 - back(s) with back(s) = (r0 - s) mod W and r0 = (P - 1) mod W; the
            // row sees it iff that position is >= max(0, P + i - W + 1), i.e. back <= lim
            const int r0 = ring ? (P - 1) % p.W : 0;
            const int lim = (row_ok && ring_row_ok) ? P - 1 - max(0, P + i - p.W + 1) : -1;
            auto vis = [&](int key) -> bool {
                if (ring) {
                    const int slot = n * kBN + key;
                    const int back = r0 - slot + (slot > r0 ? p.W : 0);
                    return slot < p.W && back <= lim;
                }
                return key >= lo && key < hi && (key < 64 ? ok0 : ok1);
            };
            // ---- the row's 128 scores: one TMEM read, kept in registers ------------
            uint32_t r32[4][32];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                tmem_ld32(lane_addr + col_s + c4 * 32, r32[c4]);
            tmem_wait_ld();
            if (!whole_tile) {
                // keys the row cannot see become -inf: 2^-inf = 0 in the P pass below
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (!vis(c4 * 32 + c))
                            r32[c4][c] = __float_as_uint(-INFINITY);
            }
            // ---- row max (three-input max, four chains) ---------------------------
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    m4[0] = fmax3(m4[0], __uint_as_float(r32[c4][c + 0]), __uint_as_float(r32[c4][c + 1]));
                    m4[1] = fmax3(m4[1], __uint_as_float(r32[c4][c + 2]), __uint_as_float(r32[c4][c + 3]));
                    m4[2] = fmax3(m4[2], __uint_as_float(r32[c4][c + 4]), __uint_as_float(r32[c4][c + 5]));
                    m4[3] = fmax3(m4[3], __uint_as_float(r32[c4][c + 6]), __uint_as_float(r32[c4][c + 7]));
                }
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
            // ---- running max, lazily raised (O is rescaled below when it moves) ----
            float m_new = m_used;
            if (mx != -INFINITY && (m_used == -INFINITY || mx > m_used + slack))
                m_new = mx;
            const bool resc = m_used != -INFINITY && m_new != m_used;
            const float alpha = resc ? fast_exp2(m_used - m_new) : 1.0f;
            m_used = m_new;
            const float base = m_used == -INFINITY ? 0.f : m_used;
            // ---- P = 2^(s scale log2e - m) as bf16 pairs, from the registers ------
            // group c4's 16 P columns land on S columns 16 c4 .. 16 c4 + 15, all read
            // above.  On whole tiles the row sum takes the unrounded P (128 keys: the
            // bf16 rounding averages out, relative error ~2^-12.5); on partial tiles
            // it takes the bf16-rounded P the PV MMA uses, so rows with few keys get
            // no scale error proportional to |O|.
            const uint64_t sc2 = f2_make(p.scale_log2, p.scale_log2);
            const uint64_t nb2 = f2_make(-base, -base);
            uint64_t acc2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
            float accr = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint64_t x2 = f2_fma(f2_make(__uint_as_float(r32[c4][2 * c]),
                                                       __uint_as_float(r32[c4][2 * c + 1])),
                                               sc2, nb2);
                    float x0, x1;
                    f2_split(x2, x0, x1);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    pk[c] = pack_bf16(p0, p1);
                    if (whole_tile)
                        acc2[c & 1] = f2_add(acc2[c & 1], f2_make(p0, p1));
                    else
                        accr += bf16_lo(pk[c]) + bf16_hi(pk[c]);
                }
                tmem_st16(lane_addr + col_s + c4 * 16, pk);
            }
            // O (read by PV_t(n), which waits for this warp) is rescaled after the P
            // pass, once the score registers are free
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o32[32];
                    tmem_ld32(lane_addr + col_o + c4 * 32, o32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o32[c] = __float_as_uint(__uint_as_float(o32[c]) * alpha);
                    tmem_st32(lane_addr + col_o + c4 * 32, o32);
                }
            }
            {
                float a0, a1;
                f2_split(f2_add(acc2[0], acc2[1]), a0, a1);
                l = l * alpha + ((a0 + a1) + accr);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sh.p_full[t]);
        }
        // ---- epilogue: O / l -> bf16 ------------------------------------------
        if (tile_ok && ok && mbar_wait_sleep(&sh.o_full, 0)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = p.out + ((int64_t)(row0 + t * kBM + row) * p.Hq + hq) * kD;
            uint32_t o32[32];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                tmem_ld32(lane_addr + col_o + c4 * 32, o32);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o32[c + 0]) * inv, __uint_as_float(o32[c + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(o32[c + 2]) * inv, __uint_as_float(o32[c + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(o32[c + 4]) * inv, __uint_as_float(o32[c + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(o32[c + 6]) * inv, __uint_as_float(o32[c + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c4 * 32 + c) = w;
                    }
                }
            }
        } else if (tile_ok && ok) {
            set_err(p.dev_err, HSA_DEVERR_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t prefill_smem_bytes() { return sizeof(PrefillSmem) + 1024; }

cudaError_t launch_prefill(const CUtensorMap &tmPK, const CUtensorMap &tmPV,
                           const CUtensorMap &tmNK, const CUtensorMap &tmNV,
                           const CUtensorMap &tmQ, const PrefillParams &p, cudaStream_t stream)
{
    const size_t smem = prefill_smem_bytes();
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    // tiles_per_req_bound bounds the number of 128-row tiles; a CTA takes a pair of
    // them, and each request may end on an odd tile
    const int64_t pairs = ((int64_t)p.tiles_per_req_bound + p.R + 1) / 2;
    const int64_t ctas = pairs * p.Hq;
    if (ctas <= 0)
        return cudaSuccess;
    prefill_kernel<<<(unsigned)ctas, kThreads, smem, stream>>>(tmPK, tmPV, tmNK, tmNV, tmQ, p);
    return cudaGetLastError();
}

}  // namespace hsa

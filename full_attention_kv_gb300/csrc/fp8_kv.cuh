// fp8_kv.cuh -- layout of an FP8 (E4M3 or E5M2) Full KV Pool layer and the warp
// routine that quantises one (token, KV head) row into it.
//
// [hotdry.top "MiMo inference optimization, edge deployment", "KV Cache 量化策略的
// 技术选型": FP8 KV, with quantisation groups aligned to the window so that no
// group straddles a window boundary; "边缘部署的工程权衡与参数清单": FP8 as the
// baseline KV format, the newest 128 tokens kept at the original precision.]
// Here a group is one (position, KV head) row of d = 128 values with one fp32
// scale = amax / F, code = FP8(x / scale) (round to nearest even, saturating), F
// the format's largest finite magnitude: 448 for E4M3 (4 exponent, 3 mantissa
// bits), 57344 for E5M2 (5 exponent, 2 mantissa bits; the section weighs the
// range of one against the precision of the other).  An all-zero row stores scale
// 0 and zero codes.  Only full layers use FP8: a sliding layer's ring holds
// exactly the newest W = 128 tokens and stays bf16.  Both formats share the layout.
//
// Layer buffer for K (and, separately, for V) of num_blocks pages:
//   codes  [num_blocks * Hkv * 64 * 128] bytes, then
//   scales [num_blocks * Hkv * 64] fp32 (index (block * Hkv + h) * 64 + row).
//  K codes: page (block, h) is 64 rows of 128 bytes; row r's value of dimension c
//           sits at byte 16 (c / 16) + perm16(c mod 16) of the row.
//  V codes: page (block, h) is 128 rows (one per dimension) of 64 bytes; the value
//           of key row r in dimension c sits at byte 16 (r / 16) + perm16(r mod 16)
//           of row c (V is stored transposed).
//  perm16(l) = 4 ((l mod 8) / 2) + (l mod 2) + 2 (l / 8) puts the four values a
//  thread needs for one 16-wide step of an m16n8k16 MMA fragment (l = 2q, 2q + 1,
//  2q + 8, 2q + 9) in four consecutive bytes, so one 32-bit shared load feeds both
//  fragment registers.
#pragma once

#include "hsa_device.cuh"

namespace hsa {

__host__ __device__ constexpr int perm16(int l) { return 4 * ((l & 7) >> 1) + (l & 1) + 2 * (l >> 3); }

__host__ __device__ inline int64_t fp8_codes_bytes(int64_t num_blocks, int Hkv)
{
    return num_blocks * Hkv * 64 * 128;
}

// Quantise one row of 128 bf16 values (src) into page (blk, h), row `off`, of an
// FP8 layer (codes base `codes`, scales base `scales`).  Called by a full warp;
// kv = 0 writes the K layout, 1 the V layout; e5m2 picks the format (else E4M3).
__device__ __forceinline__ void fp8_store_row(const __nv_bfloat16 *src, uint8_t *codes,
                                              float *scales, int64_t blk, int h, int Hkv, int off,
                                              int kv, int lane, bool e5m2)
{
    float x[4];
    if (kv == 0) {
        // lane L fills stored bytes 4L .. 4L+3 = dims 16 (L / 4) + 2 (L mod 4) + {0, 1, 8, 9}
        const int d0 = 16 * (lane >> 2) + 2 * (lane & 3);
        const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t *>(src + d0));
        const uint32_t w1 = __ldg(reinterpret_cast<const uint32_t *>(src + d0 + 8));
        x[0] = bf16_lo(w0);
        x[1] = bf16_hi(w0);
        x[2] = bf16_lo(w1);
        x[3] = bf16_hi(w1);
    } else {
        // lane L covers dims 4L .. 4L+3
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(src + 4 * lane));
        x[0] = bf16_lo(w.x);
        x[1] = bf16_hi(w.x);
        x[2] = bf16_lo(w.y);
        x[3] = bf16_hi(w.y);
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, e5m2 ? 57344.0f : 448.0f);
    uint32_t c01 = 0, c23 = 0;
    if (amax > 0.f) {
        const float y0 = __fdiv_rn(x[0], scale), y1 = __fdiv_rn(x[1], scale);
        const float y2 = __fdiv_rn(x[2], scale), y3 = __fdiv_rn(x[3], scale);
        c01 = e5m2 ? f32x2_to_e5m2x2(y0, y1) : f32x2_to_e4m3x2(y0, y1);
        c23 = e5m2 ? f32x2_to_e5m2x2(y2, y3) : f32x2_to_e4m3x2(y2, y3);
    }
    const int64_t page = blk * Hkv + h;
    if (kv == 0) {
        *reinterpret_cast<uint32_t *>(codes + (page * 64 + off) * 128 + 4 * lane) = c01 | (c23 << 16);
    } else {
        const int kb = 16 * (off >> 4) + perm16(off & 15);
        const uint32_t c = c01 | (c23 << 16);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            codes[(page * 128 + 4 * lane + j) * 64 + kb] = (uint8_t)(c >> (8 * j));
    }
    if (lane == 0)
        scales[page * 64 + off] = amax > 0.f ? scale : 0.f;
}

}  // namespace hsa

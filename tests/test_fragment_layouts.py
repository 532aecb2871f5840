"""Operand layouts of the decode kernel's swapped-operand tiles, restated on the host.

At T = 1 two paths of full_attention_kv_gb300/csrc/decode.cu put the keys on the M
side of `mma.sync.m16n8k16` and the unit's (at most 8) query heads on its N side:
tile_fp8_sw (FP8 full layers) and the sliding layers' full-ring path.  Each lane
builds its A and B fragments from shared-memory words or ldmatrix results, and P
reaches the B operand of P V through `movmatrix.trans`.  This file models the
PTX fragment layouts of those instructions (lane l = 4 g + tq holds A rows g, g + 8
at columns 2 tq, 2 tq + 1 (+ 8), B rows 2 tq, 2 tq + 1 (+ 8) at column g, and C
rows g, g + 8 at columns 2 tq, 2 tq + 1), feeds them the kernels' address formulas
on the pages' stored layouts (FP8: the perm16 byte order of fp8_kv.cuh under the
TMA swizzles; bf16: the 128-byte swizzle of two 64-column boxes), and checks that
the products are exactly S^T = K Q^T and O^T = V^T P^T.  Values stand in for codes
and bf16 bits, so the check is exact.
"""
import numpy as np

D = 128


def perm16(l):
    return 4 * ((l & 7) >> 1) + (l & 1) + 2 * (l >> 3)


def mma(c, a, b):
    """c[lane] (4) += A (16 x 16) B (16 x 8), A from a[lane] = 4 pairs, B from b[lane] =
    2 pairs, in the m16n8k16 fragment layout."""
    A = np.zeros((16, 16))
    B = np.zeros((16, 8))
    for lane in range(32):
        g, tq = lane >> 2, lane & 3
        for e in range(2):
            A[g, 2 * tq + e] = a[lane][0][e]
            A[g + 8, 2 * tq + e] = a[lane][1][e]
            A[g, 2 * tq + 8 + e] = a[lane][2][e]
            A[g + 8, 2 * tq + 8 + e] = a[lane][3][e]
            B[2 * tq + e, g] = b[lane][0][e]
            B[2 * tq + 8 + e, g] = b[lane][1][e]
    C = A @ B
    for lane in range(32):
        g, tq = lane >> 2, lane & 3
        c[lane] += np.array([C[g, 2 * tq], C[g, 2 * tq + 1], C[g + 8, 2 * tq], C[g + 8, 2 * tq + 1]])


def movmatrix_trans(x):
    """x[lane] = (M[g][2 tq], M[g][2 tq + 1]) of an 8 x 8 matrix -> the same for M^T."""
    M = np.zeros((8, 8))
    for lane in range(32):
        g, tq = lane >> 2, lane & 3
        M[g, 2 * tq], M[g, 2 * tq + 1] = x[lane]
    return [(M[2 * (l & 3), l >> 2], M[2 * (l & 3) + 1, l >> 2]) for l in range(32)]


def word(smem, off):
    """A 32-bit shared load of four one-byte values: lo pair bytes 0-1, hi pair 2-3."""
    return (smem[off], smem[off + 1]), (smem[off + 2], smem[off + 3])


def test_fp8_swapped_tile_layout():
    rng = np.random.default_rng(7)
    K = rng.integers(-8, 8, (64, D)).astype(float)   # keys x dims
    V = rng.integers(-8, 8, (64, D)).astype(float)
    Q = rng.integers(-8, 8, (8, D)).astype(float)    # heads x dims
    P = rng.integers(-8, 8, (64, 8)).astype(float)   # keys x heads (P^T)
    # K page as staged: row r (key), logical 16-byte chunk q at chunk q ^ (r mod 8)
    # (128-byte swizzle), byte 16 (c / 16) + perm16(c mod 16) of the row = dim c
    sK = np.zeros(64 * 128)
    for r in range(64):
        for c in range(D):
            b = 16 * (c // 16) + perm16(c % 16)
            sK[r * 128 + (((b >> 4) ^ (r & 7)) << 4) + (b & 15)] = K[r, c]
    # V page as staged: row c (dim) of 64 bytes, key r at byte 16 (r / 16) + perm16(r mod
    # 16), the 16-byte chunk q at chunk q ^ ((c / 2) mod 4) (64-byte swizzle)
    sV = np.zeros(D * 64)
    for c in range(D):
        for r in range(64):
            b = 16 * (r // 16) + perm16(r % 16)
            sV[c * 64 + (((b >> 4) ^ ((c >> 1) & 3)) << 4) + (b & 15)] = V[r, c]
    # B operand of S^T = K Q^T: column g = head g, rows = dims
    qb = [[((Q[l >> 2, 16 * ks + 2 * (l & 3)], Q[l >> 2, 16 * ks + 2 * (l & 3) + 1]),
            (Q[l >> 2, 16 * ks + 8 + 2 * (l & 3)], Q[l >> 2, 16 * ks + 9 + 2 * (l & 3)]))
           for ks in range(D // 16)] for l in range(32)]
    for key0, km in ((0, 64), (0, 32), (32, 32)):
        mts = km // 16
        s = [[np.zeros(4) for _ in range(32)] for _ in range(mts)]
        for mt in range(mts):
            for ks in range(D // 16):
                a = []
                for l in range(32):
                    g, tq = l >> 2, l & 3
                    ra = (key0 + mt * 16 + g) * 128 + 4 * tq
                    rb = ra + 8 * 128
                    off = (ks ^ g) << 4
                    (alo, ahi), (blo, bhi) = word(sK, ra + off), word(sK, rb + off)
                    a.append((alo, blo, ahi, bhi))
                mma(s[mt], a, [qb[l][ks] for l in range(32)])
        for mt in range(mts):
            for l in range(32):
                g, tq = l >> 2, l & 3
                ka, kb = key0 + mt * 16 + g, key0 + mt * 16 + g + 8
                want = [K[ka] @ Q[2 * tq], K[ka] @ Q[2 * tq + 1], K[kb] @ Q[2 * tq], K[kb] @ Q[2 * tq + 1]]
                assert np.array_equal(s[mt][l], want)
        # O^T += V^T P^T over the same keys
        o = [[np.zeros(4) for _ in range(32)] for _ in range(D // 16)]
        for ks in range(mts):
            grp = (key0 >> 4) + ks
            lo = [(P[key0 + ks * 16 + (l >> 2), 2 * (l & 3)], P[key0 + ks * 16 + (l >> 2), 2 * (l & 3) + 1])
                  for l in range(32)]
            hi = [(P[key0 + ks * 16 + 8 + (l >> 2), 2 * (l & 3)],
                   P[key0 + ks * 16 + 8 + (l >> 2), 2 * (l & 3) + 1]) for l in range(32)]
            b0, b1 = movmatrix_trans(lo), movmatrix_trans(hi)
            bfr = [(b0[l], b1[l]) for l in range(32)]
            for dt in range(D // 16):
                a = []
                for l in range(32):
                    g, tq = l >> 2, l & 3
                    da, db = dt * 16 + g, dt * 16 + g + 8
                    (alo, ahi) = word(sV, da * 64 + ((grp ^ ((da >> 1) & 3)) << 4) + 4 * tq)
                    (blo, bhi) = word(sV, db * 64 + ((grp ^ ((db >> 1) & 3)) << 4) + 4 * tq)
                    a.append((alo, blo, ahi, bhi))
                mma(o[dt], a, bfr)
        OT = V[key0:key0 + km].T @ P[key0:key0 + km]   # dims x heads
        for dt in range(D // 16):
            for l in range(32):
                g, tq = l >> 2, l & 3
                want = [OT[dt * 16 + g, 2 * tq], OT[dt * 16 + g, 2 * tq + 1],
                        OT[dt * 16 + g + 8, 2 * tq], OT[dt * 16 + g + 8, 2 * tq + 1]]
                assert np.array_equal(o[dt][l], want)


def swz128(row, col, rows):
    """Element offset (in bf16 units) of (row, col) in a tile of 64-column boxes written
    with the 128-byte swizzle (hsa_device.cuh swz128_offset, divided by 2)."""
    box, c = col >> 6, col & 63
    return box * rows * 64 + row * 64 + ((((c >> 3) ^ (row & 7)) << 4) + ((c & 7) << 1)) // 2


def ldmatrix_x4(smem, addr, trans=False):
    """ldmatrix.x4 (.trans): lanes 8 i .. 8 i + 7 give the row addresses of matrix i."""
    out = [[None] * 4 for _ in range(32)]
    for i in range(4):
        M = np.array([smem[addr[8 * i + r]:addr[8 * i + r] + 8] for r in range(8)])
        if trans:
            M = M.T
        for l in range(32):
            out[l][i] = (M[l >> 2, 2 * (l & 3)], M[l >> 2, 2 * (l & 3) + 1])
    return out


def test_ring_t1_swapped_tile_layout():
    rng = np.random.default_rng(11)
    K = rng.integers(-8, 8, (64, D)).astype(float)
    V = rng.integers(-8, 8, (64, D)).astype(float)
    Q = rng.integers(-8, 8, (8, D)).astype(float)
    P = rng.integers(-8, 8, (64, 8)).astype(float)
    sK = np.zeros(64 * D)
    sV = np.zeros(64 * D)
    for r in range(64):
        for c in range(D):
            sK[swz128(r, c, 64)] = K[r, c]
            sV[swz128(r, c, 64)] = V[r, c]
    qb = [[((Q[l >> 2, 16 * ks + 2 * (l & 3)], Q[l >> 2, 16 * ks + 2 * (l & 3) + 1]),
            (Q[l >> 2, 16 * ks + 8 + 2 * (l & 3)], Q[l >> 2, 16 * ks + 9 + 2 * (l & 3)]))
           for ks in range(D // 16)] for l in range(32)]
    for kb in (0, 32):  # the warp's 32 keys of the tile
        sc = [[np.zeros(4) for _ in range(32)] for _ in range(2)]
        for mt2 in range(2):
            for ks in range(D // 16):
                addr = [swz128(kb + mt2 * 16 + ((l >> 3) & 1) * 8 + (l & 7),
                               ks * 16 + (l >> 4) * 8, 64) for l in range(32)]
                a = ldmatrix_x4(sK, addr)
                mma(sc[mt2], a, [qb[l][ks] for l in range(32)])
        for mt2 in range(2):
            for l in range(32):
                g, tq = l >> 2, l & 3
                ka, kk = kb + mt2 * 16 + g, kb + mt2 * 16 + g + 8
                assert np.array_equal(sc[mt2][l], [K[ka] @ Q[2 * tq], K[ka] @ Q[2 * tq + 1],
                                                   K[kk] @ Q[2 * tq], K[kk] @ Q[2 * tq + 1]])
        o = [[np.zeros(4) for _ in range(32)] for _ in range(D // 16)]
        for ks in range(2):
            lo = [(P[kb + ks * 16 + (l >> 2), 2 * (l & 3)], P[kb + ks * 16 + (l >> 2), 2 * (l & 3) + 1])
                  for l in range(32)]
            hi = [(P[kb + ks * 16 + 8 + (l >> 2), 2 * (l & 3)],
                   P[kb + ks * 16 + 8 + (l >> 2), 2 * (l & 3) + 1]) for l in range(32)]
            b0, b1 = movmatrix_trans(lo), movmatrix_trans(hi)
            bfr = [(b0[l], b1[l]) for l in range(32)]
            for dt in range(D // 16):
                addr = [swz128(kb + ks * 16 + (l >> 4) * 8 + (l & 7),
                               dt * 16 + ((l >> 3) & 1) * 8, 64) for l in range(32)]
                a = ldmatrix_x4(sV, addr, trans=True)
                mma(o[dt], a, bfr)
        OT = V[kb:kb + 32].T @ P[kb:kb + 32]
        for dt in range(D // 16):
            for l in range(32):
                g, tq = l >> 2, l & 3
                assert np.array_equal(o[dt][l], [OT[dt * 16 + g, 2 * tq], OT[dt * 16 + g, 2 * tq + 1],
                                                 OT[dt * 16 + g + 8, 2 * tq],
                                                 OT[dt * 16 + g + 8, 2 * tq + 1]])

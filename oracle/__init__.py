"""CPU oracle for Hybrid-SWA dual-KV-pool attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.

All arithmetic lives in ``hsa_oracle.c`` (plain loops, double precision); this
module only marshals numpy arrays through ctypes.  bf16 tensors are passed as
their raw uint16 bit patterns.

Sources: youleyou.com "小米MiMo首次公开模型推理系统全链路优化降价99%", s1 "为什么选择
Hybrid SWA 架构" (window 128, 60 SWA + 10 full layers, KV ~1/7) and s2
"KVCache系统重构" (Full KV Pool, ring-buffer SWA KV Pool, window-safe length);
hotdry.top "MiMo-V2.5 ultra-speed inference architecture", "Hybrid SWA" section
(6:1 interleave, match length cut to the window boundary).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        dp = ctypes.POINTER(ctypes.c_double)
        L.orc_attention.restype = ctypes.c_int
        L.orc_attention.argtypes = [
            ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, u16p, u16p, u16p, u16p, u16p, i64p, i32p,
            ctypes.c_int64, i32p, i32p, dp, ctypes.c_int]
        L.orc_full_place.restype = ctypes.c_int
        L.orc_full_place.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int64, i32p, i32p]
        L.orc_ring_place.restype = ctypes.c_int
        L.orc_ring_place.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int64, i32p, i32p]
        L.orc_append.restype = ctypes.c_int64
        L.orc_append.argtypes = [
            ctypes.c_int, u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, i32p, ctypes.c_int, i32p, ctypes.c_int, i32p, i32p, i32p,
            u16p, u16p]
        L.orc_window_safe_len_ring.restype = None
        L.orc_window_safe_len_ring.argtypes = [ctypes.c_int, ctypes.c_int, i32p, i32p, i32p]
        L.orc_window_safe_len_bitmap.restype = None
        L.orc_window_safe_len_bitmap.argtypes = [ctypes.c_int, ctypes.c_int, i32p, i64p,
                                                 u8p, i32p]
        L.orc_kv_bytes.restype = ctypes.c_double
        L.orc_kv_bytes.argtypes = [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_double]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_num_threads.argtypes = []
        fp = ctypes.POINTER(ctypes.c_float)
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_quantize_e4m3.restype = None
        L.orc_quantize_e4m3.argtypes = [ctypes.c_int64, ctypes.c_int, u16p, u8p, fp]
        L.orc_e5m2_value.restype = ctypes.c_double
        L.orc_e5m2_value.argtypes = [ctypes.c_uint8]
        L.orc_e5m2_encode.restype = ctypes.c_uint8
        L.orc_e5m2_encode.argtypes = [ctypes.c_float]
        L.orc_quantize_e5m2.restype = None
        L.orc_quantize_e5m2.argtypes = [ctypes.c_int64, ctypes.c_int, u16p, u8p, fp]
        L.orc_attention_fp8hist_fmt.restype = ctypes.c_int
        L.orc_attention_fp8hist_fmt.argtypes = [
            ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            u16p, u16p, u16p, u8p, fp, u8p, fp, i64p, ctypes.c_int64, i32p, i32p, dp,
            ctypes.c_int, ctypes.c_int]
        _lib = L
    return _lib


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_bits(t):
    """Raw uint16 bit patterns of a bf16 torch tensor (or pass a uint16 array)."""
    if isinstance(t, np.ndarray):
        return _c(t, np.uint16)
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def num_threads():
    return int(lib().orc_num_threads())


def attention(cu_rows, prefix_len, q, k_new, v_new, hist_k, hist_v, hist_off, hist_start,
              window, scale, items=None, nthreads=None):
    """Masked softmax attention of new rows over (history ++ new rows), float64.

    q: [rows, Hq, d] bf16; k_new/v_new: [rows, Hkv, d] bf16; request r owns rows
    cu_rows[r]:cu_rows[r+1] at positions prefix_len[r] + i.  hist_k/hist_v:
    [sum_r n_r, Hkv, d] bf16 with request r's rows hist_off[r]:hist_off[r+1] holding
    positions hist_start[r] .. prefix_len[r]-1.  window 0 = full causal.
    items: None (all rows x heads -> [rows, Hq, d]) or an int array [n, 2] of
    (row, head) -> [n, d].
    """
    L = lib()
    qb, kb, vb = bf16_bits(q), bf16_bits(k_new), bf16_bits(v_new)
    hk, hv = bf16_bits(hist_k), bf16_bits(hist_v)
    rows, Hq, d = qb.shape
    Hkv = kb.shape[1]
    cu = _c(cu_rows, np.int32)
    pl = _c(prefix_len, np.int32)
    ho = _c(hist_off, np.int64)
    hs = _c(hist_start, np.int32)
    R = len(pl)
    assert cu.shape == (R + 1,) and ho.shape == (R + 1,) and hs.shape == (R,)
    assert int(cu[-1]) == rows
    if hk.size == 0:  # keep valid pointers for empty histories
        hk = np.zeros((1, Hkv, d), np.uint16)
        hv = np.zeros((1, Hkv, d), np.uint16)
    if items is None:
        n = -1
        out = np.zeros((rows, Hq, d), np.float64)
        ir = np.zeros(1, np.int32)
        ih = np.zeros(1, np.int32)
    else:
        it = _c(items, np.int32).reshape(-1, 2)
        n = it.shape[0]
        out = np.zeros((n, d), np.float64)
        ir = _c(it[:, 0], np.int32)
        ih = _c(it[:, 1], np.int32)
        if n == 0:
            return out
    nt = num_threads() if nthreads is None else int(nthreads)
    rc = L.orc_attention(
        R, _p(cu, ctypes.c_int32), _p(pl, ctypes.c_int32), Hq, Hkv, d, int(window),
        float(scale), _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16),
        _p(vb, ctypes.c_uint16), _p(hk, ctypes.c_uint16), _p(hv, ctypes.c_uint16),
        _p(ho, ctypes.c_int64), _p(hs, ctypes.c_int32), n, _p(ir, ctypes.c_int32),
        _p(ih, ctypes.c_int32), _p(out, ctypes.c_double), nt)
    if rc != 0:
        raise ValueError("oracle attention failed: %d" % rc)
    return out


def full_place(block_tables, num_blocks, page_size, seq, pos):
    """(block, offset) of position pos of sequence seq in the Full KV Pool."""
    bt = _c(block_tables, np.int32)
    b = ctypes.c_int32()
    o = ctypes.c_int32()
    rc = lib().orc_full_place(_p(bt, ctypes.c_int32), bt.shape[1], num_blocks, page_size,
                              seq, pos, ctypes.byref(b), ctypes.byref(o))
    return None if rc else (b.value, o.value)


def ring_place(ring_row, n_rows, W, seq, pos):
    """(ring row, slot) of position pos of sequence seq in the SWA KV Pool."""
    rr = _c(ring_row, np.int32)
    r = ctypes.c_int32()
    s = ctypes.c_int32()
    rc = lib().orc_ring_place(_p(rr, ctypes.c_int32), n_rows, W, seq, pos,
                              ctypes.byref(r), ctypes.byref(s))
    return None if rc else (r.value, s.value)


def append(pool_k, pool_v, cu_rows, seq_idx, start_pos, k_new, v_new, *,
           block_tables=None, ring_row=None):
    """Apply one append call to uint16 host pool images, in place.

    Full pool: pool [num_blocks, Hkv, page, d] with block_tables [B, max_blocks].
    Ring:      pool [n_rows, Hkv, W, d] with ring_row [B].
    Returns the number of tokens that could not be placed.
    """
    assert pool_k.dtype == np.uint16 and pool_k.flags.c_contiguous
    assert pool_v.dtype == np.uint16 and pool_v.flags.c_contiguous
    nb, Hkv, page, d = pool_k.shape
    kb, vb = bf16_bits(k_new), bf16_bits(v_new)
    cu = _c(cu_rows, np.int32)
    si = _c(seq_idx, np.int32)
    sp = _c(start_pos, np.int32)
    is_ring = ring_row is not None
    bt = _c(block_tables if not is_ring else np.zeros((1, 1)), np.int32)
    rr = _c(ring_row if is_ring else np.zeros(1), np.int32)
    return int(lib().orc_append(
        int(is_ring), _p(pool_k, ctypes.c_uint16), _p(pool_v, ctypes.c_uint16), nb, Hkv,
        page, d, _p(bt, ctypes.c_int32), bt.shape[1] if bt.ndim == 2 else 1,
        _p(rr, ctypes.c_int32), len(si), _p(cu, ctypes.c_int32), _p(si, ctypes.c_int32),
        _p(sp, ctypes.c_int32), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16)))


def window_safe_len_ring(match_len, slot_pos, W):
    m = _c(match_len, np.int32)
    sp = _c(slot_pos, np.int32).reshape(len(m), W)
    out = np.zeros(len(m), np.int32)
    lib().orc_window_safe_len_ring(len(m), W, _p(m, ctypes.c_int32), _p(sp, ctypes.c_int32),
                                   _p(out, ctypes.c_int32))
    return out


def window_safe_len_bitmap(match_len, live_off, live, W):
    m = _c(match_len, np.int32)
    off = _c(live_off, np.int64)
    lv = _c(live, np.uint8)
    if lv.size == 0:
        lv = np.zeros(1, np.uint8)
    out = np.zeros(len(m), np.int32)
    lib().orc_window_safe_len_bitmap(len(m), W, _p(m, ctypes.c_int32), _p(off, ctypes.c_int64),
                                     _p(lv, ctypes.c_uint8), _p(out, ctypes.c_int32))
    return out


def kv_bytes(layer_is_full, W, L, bytes_per_token):
    f = _c(layer_is_full, np.uint8)
    return float(lib().orc_kv_bytes(len(f), _p(f, ctypes.c_uint8), W, int(L),
                                    float(bytes_per_token)))


def kv_ratio(layer_is_full, W, L):
    """KV bytes of the hybrid stack over an all-full stack of the same depth."""
    n = len(layer_is_full)
    return kv_bytes(layer_is_full, W, L, 1.0) / kv_bytes([1] * n, W, L, 1.0)


# ---------------------------------------------------------------- FP8 KV (E4M3, E5M2)
# hotdry.top "MiMo inference optimization, edge deployment": FP8 KV with
# quantisation groups aligned to the window; one fp32 scale per (position, KV
# head) row here.  Arithmetic in hsa_oracle.c.

def e4m3_value(code):
    """Value of one E4M3 code (OCP 8-bit float, bias 7, no infinities)."""
    return float(lib().orc_e4m3_value(int(code) & 0xFF))


def e4m3_encode(x):
    """Nearest finite E4M3 code of a float32 value (ties to even, saturating)."""
    return int(lib().orc_e4m3_encode(float(np.float32(x))))


def e5m2_value(code):
    """Value of one E5M2 code (OCP 8-bit float, bias 15, infinities at 0x7C / 0xFC)."""
    return float(lib().orc_e5m2_value(int(code) & 0xFF))


def e5m2_encode(x):
    """Nearest finite E5M2 code of a float32 value (ties to even, saturating)."""
    return int(lib().orc_e5m2_encode(float(np.float32(x))))


FP8_FORMATS = ("e4m3", "e5m2")


def fp8_value(code, fmt="e4m3"):
    """Value of one code of an FP8 format ("e4m3" or "e5m2")."""
    return e5m2_value(code) if fmt == "e5m2" else e4m3_value(code)


def quantize_e5m2(rows):
    """bf16 rows [..., d] -> (E5M2 codes uint8 [..., d], scales float32 [...]):
    scale = amax / 57344 per row."""
    return _quantize(rows, lib().orc_quantize_e5m2)


def quantize_fp8(rows, fmt="e4m3"):
    """quantize_e4m3 or quantize_e5m2 by format name."""
    if fmt not in FP8_FORMATS:
        raise ValueError("unknown FP8 format %r" % (fmt,))
    return quantize_e5m2(rows) if fmt == "e5m2" else quantize_e4m3(rows)


def quantize_e4m3(rows):
    """bf16 rows [..., d] -> (codes uint8 [..., d], scales float32 [...])."""
    return _quantize(rows, lib().orc_quantize_e4m3)


def _quantize(rows, fn):
    xb = bf16_bits(rows)
    shape = xb.shape
    d = shape[-1]
    flat = _c(xb.reshape(-1, d), np.uint16)
    n = flat.shape[0]
    codes = np.zeros((max(n, 1), d), np.uint8)
    scales = np.zeros(max(n, 1), np.float32)
    if n:
        fn(n, d, _p(flat, ctypes.c_uint16), _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_float))
    return codes[:n].reshape(shape), scales[:n].reshape(shape[:-1])


def attention_fp8hist(cu_rows, prefix_len, q, k_new, v_new, hk, hks, hv, hvs, hist_off, scale,
                      items=None, nthreads=None, fmt="e4m3"):
    """Full causal attention of new rows over an FP8 history (codes + scales,
    dequantised exactly in float64) followed by the bf16 new rows.  History of
    request r: rows hist_off[r]:hist_off[r+1] = positions 0 .. prefix_len[r]-1.
    fmt names the codes' format ("e4m3" or "e5m2")."""
    if fmt not in FP8_FORMATS:
        raise ValueError("unknown FP8 format %r" % (fmt,))
    L = lib()
    qb, kb, vb = bf16_bits(q), bf16_bits(k_new), bf16_bits(v_new)
    rows, Hq, d = qb.shape
    Hkv = kb.shape[1]
    cu, pl, ho = _c(cu_rows, np.int32), _c(prefix_len, np.int32), _c(hist_off, np.int64)
    R = len(pl)
    hk, hv = _c(hk, np.uint8), _c(hv, np.uint8)
    hks, hvs = _c(hks, np.float32), _c(hvs, np.float32)
    if hk.size == 0:
        hk = np.zeros((1, Hkv, d), np.uint8)
        hv = np.zeros((1, Hkv, d), np.uint8)
        hks = np.zeros((1, Hkv), np.float32)
        hvs = np.zeros((1, Hkv), np.float32)
    if items is None:
        n = -1
        out = np.zeros((rows, Hq, d), np.float64)
        ir = ih = np.zeros(1, np.int32)
    else:
        it = _c(items, np.int32).reshape(-1, 2)
        n = it.shape[0]
        out = np.zeros((n, d), np.float64)
        ir, ih = _c(it[:, 0], np.int32), _c(it[:, 1], np.int32)
        if n == 0:
            return out
    nt = num_threads() if nthreads is None else int(nthreads)
    fp = ctypes.c_float
    rc = L.orc_attention_fp8hist_fmt(
        R, _p(cu, ctypes.c_int32), _p(pl, ctypes.c_int32), Hq, Hkv, d, float(scale),
        _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
        _p(hk, ctypes.c_uint8), _p(hks, fp), _p(hv, ctypes.c_uint8), _p(hvs, fp),
        _p(ho, ctypes.c_int64), n, _p(ir, ctypes.c_int32), _p(ih, ctypes.c_int32),
        _p(out, ctypes.c_double), 1 if fmt == "e5m2" else 0, nt)
    if rc != 0:
        raise ValueError("oracle fp8 attention failed: %d" % rc)
    return out

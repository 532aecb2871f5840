"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/hsa.h declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header="hsa.h"):
    src = open(os.path.join(ROOT, "include", header), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hsa_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from full_attention_kv_gb300 import build as b
    path = b.build()
    L = ctypes.CDLL(path)
    names = _declared()
    assert "hsa_decode_attn" in names and "hsa_kv_append" in names
    for n in names:
        assert hasattr(L, n), n


def test_library_exports_the_tree_header():
    import full_attention_kv_gb300 as hsa
    L = ctypes.CDLL(hsa.build.build() if hasattr(hsa, "build") else hsa.binding.LIB_PATH)
    names = _declared("hsa_tree.h")
    assert "hsa_ptree_match_batch" in names
    for n in names:
        assert hasattr(L, n), n
    assert sorted(hsa.TREE_EXPORTS) == names


def test_binding_covers_the_header():
    import full_attention_kv_gb300 as hsa
    assert sorted(hsa.EXPORTS) == _declared()
    L = hsa.lib()
    assert hsa.status_string(hsa.HSA_OK) == "ok"
    assert hsa.status_string(hsa.HSA_UNSUPPORTED_SHAPE) == "unsupported shape"
    assert L.hsa_status_string(99) == b"unknown status"


def test_host_validation_rejects_without_launching():
    """Null / malformed arguments are refused on the host before any CUDA call."""
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    assert L.hsa_decode_attn(None, 0, None, None, None, None, 1, 1, 1.0, None, None, 0, 0,
                             None, None) == hsa.HSA_INVALID_ARG
    assert L.hsa_kv_append(None, 0, None, None, None, None, None, 1, 1, None, None) == \
        hsa.HSA_INVALID_ARG
    assert L.hsa_window_safe_len(None, None, -1, 128, None, None) == hsa.HSA_INVALID_ARG
    assert L.hsa_window_safe_len(None, None, 0, 128, None, None) == hsa.HSA_OK
    k = (ctypes.c_void_p * 1)(16)
    full = (ctypes.c_uint8 * 1)(1)
    pools = hsa.HsaPools(n_layers=1, layer_is_full=ctypes.cast(full, ctypes.POINTER(ctypes.c_uint8)),
                         k=ctypes.cast(k, ctypes.POINTER(ctypes.c_void_p)),
                         v=ctypes.cast(k, ctypes.POINTER(ctypes.c_void_p)), num_blocks=1,
                         page_size=64, block_tables=16, max_blocks=1, ring_row=16, n_ring_rows=1,
                         batch=1, W=128, Hq=32, Hkv=4, d=64)
    assert L.hsa_decode_attn(ctypes.byref(pools), 0, None, None, None, None, 1, 1, 1.0, None,
                             None, 0, 0, None, None) == hsa.HSA_UNSUPPORTED_SHAPE
    pools.d = 128
    pools.W = 96
    assert L.hsa_kv_append(ctypes.byref(pools), 0, None, None, None, None, None, 1, 1, None,
                           None) == hsa.HSA_UNSUPPORTED_SHAPE


def test_binding_constants_match_the_headers():
    """Every HSA_* status and device-error bit the headers define has the same value
    in the binding (the binding reads dev_err with these)."""
    import full_attention_kv_gb300 as hsa
    for header in ("hsa.h", "hsa_tree.h"):
        src = open(os.path.join(ROOT, "include", header), encoding="utf-8").read()
        for name, val in re.findall(r"#define\s+(HSA_[A-Z0-9_]+)\s+(\d+)", src):
            assert getattr(hsa, name) == int(val), name


def test_decode_rejects_more_than_four_new_tokens():
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    k = (ctypes.c_void_p * 1)(16)
    full = (ctypes.c_uint8 * 1)(1)
    pools = hsa.HsaPools(n_layers=1, layer_is_full=ctypes.cast(full, ctypes.POINTER(ctypes.c_uint8)),
                         k=ctypes.cast(k, ctypes.POINTER(ctypes.c_void_p)),
                         v=ctypes.cast(k, ctypes.POINTER(ctypes.c_void_p)), num_blocks=1,
                         page_size=64, block_tables=16, max_blocks=1, ring_row=16, n_ring_rows=1,
                         batch=1, W=128, Hq=4, Hkv=4, d=128)
    for T in (5, 16):  # G = 1 leaves G * T within 32: only the documented T <= 4 refuses
        assert L.hsa_decode_attn(ctypes.byref(pools), 0, None, None, None, None, 1, T, 1.0, None,
                                 None, 0, 0, None, None) == hsa.HSA_UNSUPPORTED_SHAPE
    assert L.hsa_decode_attn(ctypes.byref(pools), 0, None, None, None, None, 1, 0, 1.0, None,
                             None, 0, 0, None, None) == hsa.HSA_INVALID_ARG


def _pools(hsa, **kw):
    """A host struct that passes every host check unless `kw` breaks one.  Pointer
    values are never dereferenced by the checks (no CUDA call is reached)."""
    n = kw.pop("n_layers", 2)
    full = (ctypes.c_uint8 * n)(*kw.pop("full", [0, 1]))
    fp8 = kw.pop("fp8", None)
    fp8a = (ctypes.c_uint8 * n)(*fp8) if fp8 is not None else None
    ptr = kw.pop("ptr", 256)
    kv = (ctypes.c_void_p * n)(*([ptr] * n))
    args = dict(n_layers=n, layer_is_full=ctypes.cast(full, ctypes.POINTER(ctypes.c_uint8)),
                k=ctypes.cast(kv, ctypes.POINTER(ctypes.c_void_p)),
                v=ctypes.cast(kv, ctypes.POINTER(ctypes.c_void_p)), num_blocks=8, page_size=64,
                block_tables=256, max_blocks=4, ring_row=256, n_ring_rows=2, batch=2, W=128,
                Hq=32, Hkv=4, d=128,
                layer_kv_fp8=ctypes.cast(fp8a, ctypes.POINTER(ctypes.c_uint8)) if fp8a else None)
    args.update(kw)
    p = hsa.HsaPools(**args)
    p._keep = (full, kv, fp8a)
    return p


_BAD_POOLS = [
    # (change, layer, expected status name)
    (dict(d=64), 1, "HSA_UNSUPPORTED_SHAPE"),
    (dict(page_size=32), 1, "HSA_UNSUPPORTED_SHAPE"),
    (dict(W=96), 0, "HSA_UNSUPPORTED_SHAPE"),
    (dict(W=320), 0, "HSA_UNSUPPORTED_SHAPE"),
    (dict(Hq=24), 1, "HSA_UNSUPPORTED_SHAPE"),      # group of 6
    (dict(Hq=30), 1, "HSA_UNSUPPORTED_SHAPE"),      # Hq not a multiple of Hkv
    (dict(Hq=64), 1, "HSA_UNSUPPORTED_SHAPE"),      # group of 16
    (dict(Hkv=0), 1, "HSA_UNSUPPORTED_SHAPE"),
    (dict(batch=-1), 1, "HSA_INVALID_ARG"),
    (dict(ptr=264), 1, "HSA_INVALID_ARG"),          # pool not 16-byte aligned
    (dict(ptr=0), 1, "HSA_INVALID_ARG"),
    (dict(block_tables=None), 1, "HSA_INVALID_ARG"),  # full layer without block tables
    (dict(num_blocks=0), 1, "HSA_INVALID_ARG"),
    (dict(ring_row=None), 0, "HSA_INVALID_ARG"),    # sliding layer without ring rows
    (dict(n_ring_rows=0), 0, "HSA_INVALID_ARG"),
    (dict(fp8=[1, 0]), 0, "HSA_UNSUPPORTED_SHAPE"),  # a sliding layer flagged FP8
    (dict(fp8=[2, 0]), 0, "HSA_UNSUPPORTED_SHAPE"),  # ... flagged E5M2
    (dict(fp8=[0, 3]), 1, "HSA_INVALID_ARG"),        # no FP8 format 3
    (dict(), 2, "HSA_INVALID_ARG"),                 # layer index past n_layers
    (dict(), -1, "HSA_INVALID_ARG"),
]


@pytest.mark.parametrize("change,layer,status", _BAD_POOLS)
def test_pool_checks_refuse_on_the_host(change, layer, status):
    """Every entry point taking the pools refuses a malformed struct with the
    documented status and launches nothing (this runs without a GPU)."""
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    want = getattr(hsa, status)
    p = ctypes.byref(_pools(hsa, **change))
    assert L.hsa_kv_append(p, layer, 256, 256, 256, 256, 256, 1, 1, None, None) == want
    assert L.hsa_decode_attn(p, layer, 256, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20, 0,
                             None, None) == want
    assert L.hsa_decode_attn_append(p, layer, 256, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20,
                                    0, None, None) == want
    if change.get("fp8") is None:
        assert L.hsa_prefill_attn(p, layer, 256, 256, 256, 256, 256, 256, 1, 1, 1, 0.1, 256,
                                  None, None) == want


def test_call_argument_checks_refuse_on_the_host():
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    p = ctypes.byref(_pools(hsa))
    INV, UNS, OK = hsa.HSA_INVALID_ARG, hsa.HSA_UNSUPPORTED_SHAPE, hsa.HSA_OK
    # append: negative sizes, null or unaligned rows; nothing to do is OK
    assert L.hsa_kv_append(p, 1, 256, 256, 256, 256, 256, -1, 1, None, None) == INV
    assert L.hsa_kv_append(p, 1, 256, 256, 256, 256, 256, 1, -1, None, None) == INV
    assert L.hsa_kv_append(p, 1, None, 256, 256, 256, 256, 1, 1, None, None) == INV
    assert L.hsa_kv_append(p, 1, 264, 256, 256, 256, 256, 1, 1, None, None) == INV
    assert L.hsa_kv_append(p, 1, None, None, None, None, None, 0, 0, None, None) == OK
    # decode: T out of range, B past the pool's batch, null / unaligned buffers, B = 0 is OK
    dec = L.hsa_decode_attn
    assert dec(p, 1, 256, 256, 256, 256, 1, 0, 0.1, 256, 256, 1 << 20, 0, None, None) == INV
    assert dec(p, 1, 256, 256, 256, 256, 1, 5, 0.1, 256, 256, 1 << 20, 0, None, None) == UNS
    assert dec(p, 1, 256, 256, 256, 256, 3, 1, 0.1, 256, 256, 1 << 20, 0, None, None) == INV
    assert dec(p, 1, 256, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20, -1, None, None) == INV
    assert dec(p, 1, 264, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20, 0, None, None) == INV
    assert dec(p, 1, 256, 256, 256, None, 1, 1, 0.1, 256, 256, 1 << 20, 0, None, None) == INV
    assert dec(p, 1, None, None, None, None, 0, 1, 0.1, None, None, 0, 0, None, None) == OK
    # prefill: negative sizes, null buffers; an empty call is OK; FP8 layers refused
    pre = L.hsa_prefill_attn
    assert pre(p, 1, 256, 256, 256, 256, 256, 256, -1, 1, 1, 0.1, 256, None, None) == INV
    assert pre(p, 1, 256, 256, 256, 256, 256, 256, 1, 1, -1, 0.1, 256, None, None) == INV
    assert pre(p, 1, 256, 256, 256, None, 256, 256, 1, 1, 1, 0.1, 256, None, None) == INV
    assert pre(p, 1, None, None, None, None, None, None, 0, 0, 0, 0.1, None, None, None) == OK
    p8 = ctypes.byref(_pools(hsa, fp8=[0, 1]))
    assert pre(p8, 1, 256, 256, 256, 256, 256, 256, 1, 1, 1, 0.1, 256, None, None) == UNS
    # prefetch: full layers have no ring; negative counts; n = 0 is OK
    pf = L.hsa_swa_prefetch
    assert pf(p, 1, 256, 256, 1, 256, 256, 1, None, None) == INV
    assert pf(p, 0, 256, 256, 1, 256, 256, -1, None, None) == INV
    assert pf(p, 0, None, None, 0, None, None, 0, None, None) == OK
    # window-safe: bad W or n, null buffers
    assert L.hsa_window_safe_len(256, 256, 1, 0, 256, None) == INV
    assert L.hsa_window_safe_len(None, 256, 1, 128, 256, None) == INV
    assert L.hsa_window_safe_len_bitmap(256, 256, 256, -1, 128, 256, None) == INV
    assert L.hsa_window_safe_len_bitmap(256, None, 256, 1, 128, 256, None) == INV
    assert L.hsa_decode_workspace_bytes(None, 1, 1) == 0
    assert L.hsa_decode_workspace_bytes(p, -1, 1) == 0


def test_noalloc_refuses_before_touching_its_scratch():
    """The no-workspace decode applies every host check before it queues anything
    (its scratch reset included): without a GPU a malformed call still gets the
    argument error, not a CUDA error from the scratch lookup."""
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    p = ctypes.byref(_pools(hsa))
    na = L.hsa_decode_attn_noalloc
    assert na(p, 5, 256, 256, 256, 256, 1, 1, 0.1, 256, 0, None, None) == hsa.HSA_INVALID_ARG
    assert na(p, 1, 256, 256, 256, 256, 1, 5, 0.1, 256, 0, None, None) == \
        hsa.HSA_UNSUPPORTED_SHAPE
    assert na(p, 1, 256, 256, 256, None, 1, 1, 0.1, 256, 0, None, None) == hsa.HSA_INVALID_ARG
    assert na(p, 1, 256, 256, 256, 256, 3, 1, 0.1, 256, 0, None, None) == hsa.HSA_INVALID_ARG
    assert na(p, 1, None, None, None, None, 0, 1, 0.1, None, 0, None, None) == hsa.HSA_OK
    bad = ctypes.byref(_pools(hsa, W=96))
    assert na(bad, 0, 256, 256, 256, 256, 1, 1, 0.1, 256, 0, None, None) == \
        hsa.HSA_UNSUPPORTED_SHAPE


def test_noalloc_unit_cap_is_refused_on_the_host():
    """The no-workspace decode holds arrival counters for at most 4096 (sequence, KV
    head) units in its fixed scratch: a batch of 1025 sequences x 4 KV heads (4100
    units) inside a pool that has room for it is refused with HSA_UNSUPPORTED_SHAPE
    on either kind of layer.  (No call here passes the host checks: the pointers are
    placeholders that no kernel may ever receive.)"""
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    na = L.hsa_decode_attn_noalloc
    p = ctypes.byref(_pools(hsa, batch=2048, Hkv=4, Hq=32))
    assert na(p, 1, 256, 256, 256, 256, 1025, 1, 0.1, 256, 0, None, None) == \
        hsa.HSA_UNSUPPORTED_SHAPE
    assert na(p, 0, 256, 256, 256, 256, 1025, 1, 0.1, 256, 0, None, None) == \
        hsa.HSA_UNSUPPORTED_SHAPE


def test_decode_ex_options_are_checked_on_the_host():
    """hsa_decode_attn_ex accepts only the documented option bits (append, early
    pool read); any other bit, and every malformed pool or argument the other decode
    entry points refuse, is refused before any CUDA call."""
    import full_attention_kv_gb300 as hsa
    L = hsa.lib()
    ex = L.hsa_decode_attn_ex
    p = ctypes.byref(_pools(hsa))
    for bad in (4, 8, 1 << 30, -1):
        assert ex(p, 0, 256, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20, 0, bad, None,
                  None) == hsa.HSA_INVALID_ARG
    for opts in (0, hsa.HSA_DECODE_APPEND, hsa.HSA_DECODE_EARLY_POOL_READ, 3):
        assert ex(p, 0, 256, 256, 256, 256, 1, 5, 0.1, 256, 256, 1 << 20, 0, opts, None,
                  None) == hsa.HSA_UNSUPPORTED_SHAPE
        assert ex(p, 0, None, None, None, None, 0, 1, 0.1, None, None, 0, 0, opts, None,
                  None) == hsa.HSA_OK
    bad = ctypes.byref(_pools(hsa, W=96))
    assert ex(bad, 0, 256, 256, 256, 256, 1, 1, 0.1, 256, 256, 1 << 20, 0, 2, None,
              None) == hsa.HSA_UNSUPPORTED_SHAPE

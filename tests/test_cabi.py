"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/hsa.h declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

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

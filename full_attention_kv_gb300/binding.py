"""Thin ctypes binding of libhsa (include/hsa.h), same entry-point names.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If libhsa.so has not been
built, every call raises; there is no fallback of any kind.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libhsa.so")

HSA_OK = 0
HSA_INVALID_ARG = 1
HSA_UNSUPPORTED_SHAPE = 2
HSA_CUDA_ERROR = 3
HSA_OUT_OF_RANGE = 4

HSA_DECODE_APPEND = 1
HSA_DECODE_EARLY_POOL_READ = 2

HSA_DEVERR_BAD_BLOCK = 1
HSA_DEVERR_BAD_PAGE = 2
HSA_DEVERR_BAD_SEQ = 4
HSA_DEVERR_BAD_RING = 8
HSA_DEVERR_BAD_LEN = 16
HSA_DEVERR_TIMEOUT = 32

# every symbol include/hsa.h declares
EXPORTS = ("hsa_kv_append", "hsa_decode_workspace_bytes", "hsa_decode_attn",
           "hsa_decode_attn_append", "hsa_decode_attn_ex", "hsa_decode_attn_noalloc",
           "hsa_prefill_attn",
           "hsa_swa_prefetch",
           "hsa_window_safe_len", "hsa_window_safe_len_bitmap", "hsa_status_string")
# every symbol include/hsa_tree.h declares
TREE_EXPORTS = ("hsa_ptree_create", "hsa_ptree_destroy", "hsa_ptree_match",
                "hsa_ptree_match_batch", "hsa_ptree_insert", "hsa_ptree_unlock",
                "hsa_ptree_evict_full", "hsa_ptree_evict_swa", "hsa_ptree_stats")


class HsaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))


class HsaPools(ctypes.Structure):
    """Mirror of the C struct hsa_pools."""
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("layer_is_full", ctypes.POINTER(ctypes.c_uint8)),
        ("k", ctypes.POINTER(ctypes.c_void_p)),
        ("v", ctypes.POINTER(ctypes.c_void_p)),
        ("num_blocks", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("block_tables", ctypes.c_void_p),
        ("max_blocks", ctypes.c_int32),
        ("ring_row", ctypes.c_void_p),
        ("n_ring_rows", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("W", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("layer_kv_fp8", ctypes.POINTER(ctypes.c_uint8)),
    ]


_lib = None


def lib():
    """Load libhsa.so (raises if it was not built: the CUDA path is the only path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libhsa.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        pp = ctypes.POINTER(HsaPools)
        L.hsa_kv_append.restype = ctypes.c_int
        L.hsa_kv_append.argtypes = [pp, i32, vp, vp, vp, vp, vp, i32, i32, vp, vp]
        L.hsa_decode_workspace_bytes.restype = sz
        L.hsa_decode_workspace_bytes.argtypes = [pp, i32, i32]
        L.hsa_decode_attn.restype = ctypes.c_int
        L.hsa_decode_attn.argtypes = [pp, i32, vp, vp, vp, vp, i32, i32, f32, vp, vp, sz, i32,
                                      vp, vp]
        L.hsa_decode_attn_append.restype = ctypes.c_int
        L.hsa_decode_attn_append.argtypes = [pp, i32, vp, vp, vp, vp, i32, i32, f32, vp, vp, sz,
                                             i32, vp, vp]
        L.hsa_decode_attn_ex.restype = ctypes.c_int
        L.hsa_decode_attn_ex.argtypes = [pp, i32, vp, vp, vp, vp, i32, i32, f32, vp, vp, sz,
                                         i32, i32, vp, vp]
        L.hsa_decode_attn_noalloc.restype = ctypes.c_int
        L.hsa_decode_attn_noalloc.argtypes = [pp, i32, vp, vp, vp, vp, i32, i32, f32, vp, i32,
                                              vp, vp]
        L.hsa_prefill_attn.restype = ctypes.c_int
        L.hsa_prefill_attn.argtypes = [pp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, vp,
                                       vp, vp]
        L.hsa_swa_prefetch.restype = ctypes.c_int
        L.hsa_swa_prefetch.argtypes = [pp, i32, vp, vp, i32, vp, vp, i32, vp, vp]
        L.hsa_window_safe_len.restype = ctypes.c_int
        L.hsa_window_safe_len.argtypes = [vp, vp, i32, i32, vp, vp]
        L.hsa_window_safe_len_bitmap.restype = ctypes.c_int
        L.hsa_window_safe_len_bitmap.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.hsa_status_string.restype = ctypes.c_char_p
        L.hsa_status_string.argtypes = [ctypes.c_int]
        i64, pi32 = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32)
        L.hsa_ptree_create.restype = ctypes.c_int
        L.hsa_ptree_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        L.hsa_ptree_destroy.restype = None
        L.hsa_ptree_destroy.argtypes = [vp]
        L.hsa_ptree_match.restype = ctypes.c_int
        L.hsa_ptree_match.argtypes = [vp, vp, i32, i32, i32, pi32, vp, pi32, vp,
                                      ctypes.POINTER(i64)]
        L.hsa_ptree_match_batch.restype = ctypes.c_int
        L.hsa_ptree_match_batch.argtypes = [vp, vp, vp, i32, vp, vp, vp]
        L.hsa_ptree_insert.restype = ctypes.c_int
        L.hsa_ptree_insert.argtypes = [vp, vp, vp, i32, i32, vp, vp, pi32, pi32]
        L.hsa_ptree_unlock.restype = ctypes.c_int
        L.hsa_ptree_unlock.argtypes = [vp, i64]
        L.hsa_ptree_evict_full.restype = ctypes.c_int
        L.hsa_ptree_evict_full.argtypes = [vp, i32, vp, i32, pi32, vp, i32, pi32]
        L.hsa_ptree_evict_swa.restype = ctypes.c_int
        L.hsa_ptree_evict_swa.argtypes = [vp, i32, vp, pi32]
        L.hsa_ptree_stats.restype = ctypes.c_int
        L.hsa_ptree_stats.argtypes = [vp, ctypes.POINTER(i64), pi32, pi32]
        _lib = L
    return _lib


def status_string(s):
    return lib().hsa_status_string(int(s)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t, name, dtype, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims, got %d" % (name, ndim, t.dim()))


def _shape(t, name, shape):
    """The library takes plain pointers: sizes the pool implies are checked here."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _same_device(ref, *ts):
    for t in ts:
        if t is not None and t.device != ref.device:
            raise ValueError("all device tensors must be on %s" % ref.device)


def _need_err(dev_err):
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
        if dev_err.numel() < 1:
            raise ValueError("dev_err must hold one int32")


def _check(fn, status):
    if status != HSA_OK:
        raise HsaError(fn, status)


HSA_KV_E4M3 = 1
HSA_KV_E5M2 = 2


def fp8_code(fmt):
    """layer_kv_fp8 value of a format: False / None / 0 -> 0 (bf16), True / 1 / "e4m3"
    -> HSA_KV_E4M3, 2 / "e5m2" -> HSA_KV_E5M2."""
    if fmt is None or fmt is False or (isinstance(fmt, int) and not isinstance(fmt, bool)
                                       and fmt == 0):
        return 0
    if fmt is True or fmt == "e4m3" or (isinstance(fmt, int) and fmt == HSA_KV_E4M3):
        return HSA_KV_E4M3
    if fmt == "e5m2" or (isinstance(fmt, int) and fmt == HSA_KV_E5M2):
        return HSA_KV_E5M2
    raise ValueError("unknown FP8 format %r" % (fmt,))


class DualPool:
    """The dual KV pool of one model: the C struct plus the tensors it points at.

    Full layers own K/V tensors [num_blocks, Hkv, page, d]; sliding layers own
    rings [n_ring_rows, Hkv, W, d]; block_tables [batch, max_blocks] and ring_row
    [batch] (int32) are shared by every layer of their kind.
    """

    def __init__(self, layer_is_full, k, v, block_tables, ring_row, Hq, W=128, page=64,
                 kv_fp8=None, Hkv=None, d=None, num_blocks=None):
        """kv_fp8[l] marks an FP8 full layer (True or "e4m3": E4M3 codes; "e5m2":
        E5M2 codes; False / None: bf16): k[l], v[l] are then flat uint8 buffers of
        num_blocks * Hkv * page * (d + 4) bytes (codes, then fp32 scales;
        include/hsa.h gives the layout), and Hkv, d, num_blocks must be passed."""
        self.layer_is_full = [bool(x) for x in layer_is_full]
        self.k, self.v = list(k), list(v)
        self.block_tables, self.ring_row = block_tables, ring_row
        n = len(self.layer_is_full)
        assert len(self.k) == n and len(self.v) == n
        self.kv_fp8 = [fp8_code(x) for x in kv_fp8] if kv_fp8 is not None else [0] * n
        assert len(self.kv_fp8) == n
        _need(block_tables, "block_tables", torch.int32, ndim=2)
        _need(ring_row, "ring_row", torch.int32, ndim=1)
        n_rows = None
        for l in range(n):
            if self.kv_fp8[l]:
                if not self.layer_is_full[l]:
                    raise ValueError("layer %d: only full layers can be FP8" % l)
                if Hkv is None or d is None or num_blocks is None:
                    raise ValueError("FP8 layers need Hkv, d and num_blocks")
                for t, nm in ((self.k[l], "k"), (self.v[l], "v")):
                    _need(t, "%s[%d]" % (nm, l), torch.uint8, ndim=1)
                    if t.numel() != num_blocks * Hkv * page * (d + 4):
                        raise ValueError("%s[%d]: wrong FP8 layer size" % (nm, l))
                continue
            _need(self.k[l], "k[%d]" % l, torch.bfloat16, ndim=4)
            _need(self.v[l], "v[%d]" % l, torch.bfloat16, ndim=4)
            if self.k[l].shape != self.v[l].shape:
                raise ValueError("k[%d] and v[%d] differ in shape" % (l, l))
            nb, hk, rows, dd = self.k[l].shape
            if self.layer_is_full[l]:
                if rows != page:
                    raise ValueError("full layer %d: rows per block %d != page %d" % (l, rows, page))
                num_blocks = nb if num_blocks is None else num_blocks
                if nb != num_blocks:
                    raise ValueError("full layers disagree on num_blocks")
            else:
                if rows != W:
                    raise ValueError("sliding layer %d: ring slots %d != W %d" % (l, rows, W))
                n_rows = nb if n_rows is None else n_rows
                if nb != n_rows:
                    raise ValueError("sliding layers disagree on ring rows")
            Hkv = hk if Hkv is None else Hkv
            d = dd if d is None else d
            if hk != Hkv or dd != d:
                raise ValueError("layers disagree on Hkv / d")
        self._full = (ctypes.c_uint8 * n)(*[1 if f else 0 for f in self.layer_is_full])
        self._fp8 = (ctypes.c_uint8 * n)(*self.kv_fp8)
        self._k = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.k])
        self._v = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.v])
        self.c = HsaPools(
            n_layers=n, layer_is_full=ctypes.cast(self._full, ctypes.POINTER(ctypes.c_uint8)),
            k=ctypes.cast(self._k, ctypes.POINTER(ctypes.c_void_p)),
            v=ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p)),
            num_blocks=num_blocks or 0, page_size=page, block_tables=block_tables.data_ptr(),
            max_blocks=block_tables.shape[1], ring_row=ring_row.data_ptr(),
            n_ring_rows=n_rows or 0, batch=block_tables.shape[0], W=W, Hq=Hq, Hkv=Hkv or 0,
            d=d or 0, layer_kv_fp8=ctypes.cast(self._fp8, ctypes.POINTER(ctypes.c_uint8)))
        self.Hq, self.Hkv, self.d, self.W, self.page = Hq, Hkv, d, W, page
        self.num_blocks = num_blocks or 0

    def fp8_views(self, layer):
        """Views of an FP8 layer: (K codes [nb, Hkv, page, d] in stored byte order,
        K scales [nb, Hkv, page] fp32, V codes [nb, Hkv, d, page] (transposed, stored
        key order), V scales [nb, Hkv, page] fp32)."""
        if not self.kv_fp8[layer]:
            raise ValueError("layer %d is not FP8" % layer)
        nb, hk, pg, dd = self.num_blocks, self.Hkv, self.page, self.d
        cb = nb * hk * pg * dd
        out = []
        for buf, shape in ((self.k[layer], (nb, hk, pg, dd)), (self.v[layer], (nb, hk, dd, pg))):
            out.append(buf[:cb].view(shape))
            out.append(buf[cb:].view(torch.float32).view(nb, hk, pg))
        return tuple(out)

    @classmethod
    def allocate(cls, layer_is_full, num_blocks, n_ring_rows, block_tables, ring_row, Hq, Hkv,
                 d=128, W=128, page=64, device="cuda", kv_fp8=False):
        """Zero-filled pools (rows past a sequence's length must hold finite values).
        kv_fp8=True / "e4m3" / "e5m2" stores every full layer as an FP8 layer of that
        format (sliding rings stay bf16)."""
        k, v = [], []
        fp8 = [fp8_code(kv_fp8) if f else 0 for f in layer_is_full]
        for f, q8 in zip(layer_is_full, fp8):
            if q8:
                nbytes = num_blocks * Hkv * page * (d + 4)
                k.append(torch.zeros(nbytes, dtype=torch.uint8, device=device))
                v.append(torch.zeros(nbytes, dtype=torch.uint8, device=device))
                continue
            shape = (num_blocks, Hkv, page, d) if f else (n_ring_rows, Hkv, W, d)
            k.append(torch.zeros(shape, dtype=torch.bfloat16, device=device))
            v.append(torch.zeros(shape, dtype=torch.bfloat16, device=device))
        return cls(layer_is_full, k, v, block_tables, ring_row, Hq, W=W, page=page, kv_fp8=fp8,
                   Hkv=Hkv, d=d, num_blocks=num_blocks)

    def ref(self):
        return ctypes.byref(self.c)


def hsa_kv_append(pool, layer, k_new, v_new, cu_tokens, seq_idx, start_pos, dev_err=None,
                  stream=None):
    _need(k_new, "k_new", torch.bfloat16, ndim=3)
    _need(v_new, "v_new", torch.bfloat16, ndim=3)
    for n, t in (("cu_tokens", cu_tokens), ("seq_idx", seq_idx), ("start_pos", start_pos)):
        _need(t, n, torch.int32, ndim=1)
    R = seq_idx.shape[0]
    if cu_tokens.shape[0] != R + 1 or start_pos.shape[0] != R:
        raise ValueError("cu_tokens must be [R+1] and start_pos [R]")
    _shape(k_new, "k_new", (k_new.shape[0], pool.Hkv, pool.d))
    _shape(v_new, "v_new", k_new.shape)
    _need_err(dev_err)
    _same_device(k_new, v_new, cu_tokens, seq_idx, start_pos, dev_err)
    s = lib().hsa_kv_append(pool.ref(), int(layer), _ptr(k_new), _ptr(v_new), _ptr(cu_tokens),
                            _ptr(seq_idx), _ptr(start_pos), R, k_new.shape[0], _ptr(dev_err),
                            _stream(stream))
    _check("hsa_kv_append", s)


def hsa_decode_workspace_bytes(pool, B, T):
    return int(lib().hsa_decode_workspace_bytes(pool.ref(), int(B), int(T)))


def decode_workspace(pool, B, T, device="cuda"):
    """Zero-filled workspace for hsa_decode_attn (allocate once, reuse)."""
    n = hsa_decode_workspace_bytes(pool, B, T)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def _decode_shapes(pool, q, k_new, v_new, cached_len):
    B, T = q.shape[0], q.shape[1]
    _shape(q, "q", (B, T, pool.Hq, pool.d))
    _shape(k_new, "k_new", (B, T, pool.Hkv, pool.d))
    _shape(v_new, "v_new", (B, T, pool.Hkv, pool.d))
    _shape(cached_len, "cached_len", (B,))
    _same_device(q, k_new, v_new, cached_len)


def hsa_decode_attn(pool, layer, q, k_new, v_new, cached_len, scale, out=None, workspace=None,
                    max_ctas=0, dev_err=None, stream=None, append=False, early_pool_read=False):
    """Decode attention (hsa_decode_attn; with append=True hsa_decode_attn_append).
    early_pool_read=True calls hsa_decode_attn_ex with HSA_DECODE_EARLY_POOL_READ: the
    caller guarantees that the kernel queued just before on the stream does not write
    cached_len, ring_row or this layer's ring."""
    _need(q, "q", torch.bfloat16, ndim=4)
    _need(k_new, "k_new", torch.bfloat16, ndim=4)
    _need(v_new, "v_new", torch.bfloat16, ndim=4)
    _need(cached_len, "cached_len", torch.int32, ndim=1)
    B, T = q.shape[0], q.shape[1]
    _decode_shapes(pool, q, k_new, v_new, cached_len)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, ndim=4)
    _shape(out, "out", q.shape)
    if workspace is None:
        workspace = decode_workspace(pool, B, T, device=q.device)
    _need(workspace, "workspace", torch.uint8)
    _need_err(dev_err)
    _same_device(q, out, workspace, dev_err)
    args = (pool.ref(), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cached_len), B, T,
            float(scale), _ptr(out), _ptr(workspace), workspace.numel(), int(max_ctas))
    if early_pool_read:
        opts = HSA_DECODE_EARLY_POOL_READ | (HSA_DECODE_APPEND if append else 0)
        name = "hsa_decode_attn_ex"
        s = lib().hsa_decode_attn_ex(*args, opts, _ptr(dev_err), _stream(stream))
    else:
        name = "hsa_decode_attn_append" if append else "hsa_decode_attn"
        s = getattr(lib(), name)(*args, _ptr(dev_err), _stream(stream))
    _check(name, s)
    return out


def hsa_decode_attn_append(pool, layer, q, k_new, v_new, cached_len, scale, out=None,
                           workspace=None, max_ctas=0, dev_err=None, stream=None,
                           early_pool_read=False):
    """Decode attention, then the T new K/V rows of every sequence appended."""
    return hsa_decode_attn(pool, layer, q, k_new, v_new, cached_len, scale, out=out,
                           workspace=workspace, max_ctas=max_ctas, dev_err=dev_err,
                           stream=stream, append=True, early_pool_read=early_pool_read)


def hsa_decode_attn_noalloc(pool, layer, q, k_new, v_new, cached_len, scale, out, max_ctas=0,
                            dev_err=None, stream=None):
    """hsa_decode_attn with the library's own fixed device scratch: for callers that
    cannot allocate device memory where they run decode (no workspace argument).
    `out` must be supplied; the call itself allocates nothing.  The first call on a
    device should come before any stream capture; calls that could overlap on the
    GPU share one scratch array and must be serialised."""
    _need(q, "q", torch.bfloat16, ndim=4)
    _need(k_new, "k_new", torch.bfloat16, ndim=4)
    _need(v_new, "v_new", torch.bfloat16, ndim=4)
    _need(cached_len, "cached_len", torch.int32, ndim=1)
    _need(out, "out", torch.bfloat16, ndim=4)
    _decode_shapes(pool, q, k_new, v_new, cached_len)
    _shape(out, "out", q.shape)
    _need_err(dev_err)
    _same_device(q, out, dev_err)
    B, T = q.shape[0], q.shape[1]
    s = lib().hsa_decode_attn_noalloc(pool.ref(), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new),
                                      _ptr(cached_len), B, T, float(scale), _ptr(out),
                                      int(max_ctas), _ptr(dev_err), _stream(stream))
    _check("hsa_decode_attn_noalloc", s)
    return out


def hsa_prefill_attn(pool, layer, q, k_new, v_new, cu_rows, prefix_len, seq_idx, max_chunk,
                     scale, out=None, dev_err=None, stream=None):
    _need(q, "q", torch.bfloat16, ndim=3)
    _need(k_new, "k_new", torch.bfloat16, ndim=3)
    _need(v_new, "v_new", torch.bfloat16, ndim=3)
    for n, t in (("cu_rows", cu_rows), ("prefix_len", prefix_len), ("seq_idx", seq_idx)):
        _need(t, n, torch.int32, ndim=1)
    R = seq_idx.shape[0]
    rows = q.shape[0]
    _shape(q, "q", (rows, pool.Hq, pool.d))
    _shape(k_new, "k_new", (rows, pool.Hkv, pool.d))
    _shape(v_new, "v_new", (rows, pool.Hkv, pool.d))
    _shape(cu_rows, "cu_rows", (R + 1,))
    _shape(prefix_len, "prefix_len", (R,))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, ndim=3)
    _shape(out, "out", q.shape)
    _need_err(dev_err)
    _same_device(q, k_new, v_new, cu_rows, prefix_len, seq_idx, out, dev_err)
    s = lib().hsa_prefill_attn(pool.ref(), int(layer), _ptr(q), _ptr(k_new), _ptr(v_new),
                               _ptr(cu_rows), _ptr(prefix_len), _ptr(seq_idx), R, q.shape[0],
                               int(max_chunk), float(scale), _ptr(out), _ptr(dev_err),
                               _stream(stream))
    _check("hsa_prefill_attn", s)
    return out


def hsa_swa_prefetch(pool, layer, host_k, host_v, host_row, seq_idx, dev_err=None, stream=None):
    """Copy SWA ring rows of one sliding layer from pinned host memory into the
    device ring pool (row host_row[i] -> ring row of sequence seq_idx[i])."""
    for n, t in (("host_k", host_k), ("host_v", host_v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.is_cuda:
            raise TypeError("%s must be a bf16 host tensor" % n)
        if not t.is_pinned() or not t.is_contiguous():
            raise ValueError("%s must be pinned and contiguous" % n)
    if host_k.shape != host_v.shape or host_k.dim() != 4 or \
            tuple(host_k.shape[1:]) != (pool.Hkv, pool.W, pool.d):
        raise ValueError("host_k / host_v must be [n_host_rows, Hkv, W, d]")
    _need(host_row, "host_row", torch.int32, ndim=1)
    _need(seq_idx, "seq_idx", torch.int32, ndim=1)
    if host_row.shape != seq_idx.shape:
        raise ValueError("host_row and seq_idx must have the same length")
    _need_err(dev_err)
    _same_device(host_row, seq_idx, dev_err)
    s = lib().hsa_swa_prefetch(pool.ref(), int(layer), ctypes.c_void_p(host_k.data_ptr()),
                               ctypes.c_void_p(host_v.data_ptr()), host_k.shape[0],
                               _ptr(host_row), _ptr(seq_idx), host_row.shape[0], _ptr(dev_err),
                               _stream(stream))
    _check("hsa_swa_prefetch", s)


def hsa_window_safe_len(match_len, swa_slot_pos, W, out=None, stream=None):
    _need(match_len, "match_len", torch.int32, ndim=1)
    _need(swa_slot_pos, "swa_slot_pos", torch.int32, ndim=2)
    n = match_len.shape[0]
    if swa_slot_pos.shape != (n, W):
        raise ValueError("swa_slot_pos must be [n, W]")
    if out is None:
        out = torch.empty_like(match_len)
    _need(out, "out", torch.int32)
    _shape(out, "out", match_len.shape)
    _same_device(match_len, swa_slot_pos, out)
    s = lib().hsa_window_safe_len(_ptr(match_len), _ptr(swa_slot_pos), n, int(W), _ptr(out),
                                  _stream(stream))
    _check("hsa_window_safe_len", s)
    return out


def hsa_window_safe_len_bitmap(match_len, live_off, live, W, out=None, stream=None):
    _need(match_len, "match_len", torch.int32, ndim=1)
    _need(live_off, "live_off", torch.int64, ndim=1)
    _need(live, "live", torch.uint8, ndim=1)
    n = match_len.shape[0]
    if live_off.shape[0] != n + 1:
        raise ValueError("live_off must be [n+1]")
    if out is None:
        out = torch.empty_like(match_len)
    _need(out, "out", torch.int32)
    _shape(out, "out", match_len.shape)
    _same_device(match_len, live_off, live, out)
    s = lib().hsa_window_safe_len_bitmap(_ptr(match_len), _ptr(live_off), _ptr(live), n, int(W),
                                         _ptr(out), _stream(stream))
    _check("hsa_window_safe_len_bitmap", s)
    return out


def _i32_host(a, name):
    """A contiguous host int32 tensor of a one-dimensional sequence of ints (or a
    tensor).  Values outside the int32 range are refused, not wrapped."""
    t = a if isinstance(a, torch.Tensor) else torch.as_tensor(a)
    if t.is_cuda:
        raise ValueError("%s must be host memory" % name)
    if t.dim() > 1:
        raise ValueError("%s must be one-dimensional, got shape %s" % (name, tuple(t.shape)))
    if t.numel() == 0:
        return torch.zeros(0, dtype=torch.int32)
    if t.is_floating_point() or t.is_complex():
        raise ValueError("%s must hold integers, got %s" % (name, t.dtype))
    if t.dtype != torch.int32:
        lo, hi = int(t.min()), int(t.max())
        if lo < -2 ** 31 or hi > 2 ** 31 - 1:
            raise ValueError("%s holds values outside the int32 range" % name)
    return t.to(torch.int32).contiguous().view(-1)


class PrefixTree:
    """Host prefix tree of include/hsa_tree.h (Full index + SWA ring liveness).

    Methods mirror the C calls; token and slot arrays are host int32.
    ``window_safe(...)`` matches a batch on the host and computes every request's
    window-safe length on the GPU with hsa_window_safe_len.
    """

    def __init__(self, W, n_ring_rows):
        self.W = int(W)
        h = ctypes.c_void_p()
        _check("hsa_ptree_create", lib().hsa_ptree_create(self.W, int(n_ring_rows),
                                                           ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h is not None and self._h.value:
            lib().hsa_ptree_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens, lock=False, take_ring=False):
        """-> (match_len, full_slots[match_len], ring_row, swa_slot_pos[W], lock_handle)."""
        tok = _i32_host(tokens, "tokens")
        n = tok.numel()
        slots = torch.empty(max(n, 1), dtype=torch.int32)
        pos = torch.empty(self.W, dtype=torch.int32)
        m, r, hnd = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        _check("hsa_ptree_match", lib().hsa_ptree_match(
            self._h, ctypes.c_void_p(tok.data_ptr()), n, int(bool(lock)), int(bool(take_ring)),
            ctypes.byref(m), ctypes.c_void_p(slots.data_ptr()), ctypes.byref(r),
            ctypes.c_void_p(pos.data_ptr()), ctypes.byref(hnd)))
        return m.value, slots[:m.value].clone(), r.value, pos, hnd.value

    def match_batch(self, seqs):
        """-> (match_len [n], ring_row [n], swa_slot_pos [n, W]) host int32, read-only."""
        parts = [_i32_host(x, "tokens") for x in seqs]
        off = torch.zeros(len(seqs) + 1, dtype=torch.int64)
        if seqs:
            off[1:] = torch.cumsum(torch.tensor([t.numel() for t in parts], dtype=torch.int64), 0)
        flat = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32)
        n = len(seqs)
        m = torch.empty(max(n, 1), dtype=torch.int32)
        r = torch.empty(max(n, 1), dtype=torch.int32)
        pos = torch.empty(max(n, 1), self.W, dtype=torch.int32)
        _check("hsa_ptree_match_batch", lib().hsa_ptree_match_batch(
            self._h, ctypes.c_void_p(flat.data_ptr()) if flat.numel() else None,
            ctypes.c_void_p(off.data_ptr()), n, ctypes.c_void_p(m.data_ptr()),
            ctypes.c_void_p(r.data_ptr()), ctypes.c_void_p(pos.data_ptr())))
        return m[:n], r[:n], pos[:n]

    def window_safe(self, seqs, device="cuda", stream=None):
        """Window-safe length of each request: host match, one GPU launch."""
        m, r, pos = self.match_batch(seqs)
        if m.numel() == 0:
            return m
        out = hsa_window_safe_len(m.to(device), pos.to(device), self.W, stream=stream)
        return out.cpu()

    def insert(self, tokens, full_slots, ring_row=-1, swa_slot_pos=None):
        """-> (dup_slots to free, ring_kept)."""
        tok = _i32_host(tokens, "tokens")
        sl = _i32_host(full_slots, "full_slots")
        if tok.numel() != sl.numel():
            raise ValueError("tokens and full_slots differ in length")
        n = tok.numel()
        pos = None
        if ring_row >= 0:
            pos = _i32_host(swa_slot_pos, "swa_slot_pos")
            if pos.numel() != self.W:
                raise ValueError("swa_slot_pos must hold W entries")
        dup = torch.empty(max(n, 1), dtype=torch.int32)
        nd, kept = ctypes.c_int32(), ctypes.c_int32()
        _check("hsa_ptree_insert", lib().hsa_ptree_insert(
            self._h, ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(sl.data_ptr()), n,
            int(ring_row), None if pos is None else ctypes.c_void_p(pos.data_ptr()),
            ctypes.c_void_p(dup.data_ptr()), ctypes.byref(nd), ctypes.byref(kept)))
        return dup[:nd.value].clone(), bool(kept.value)

    def unlock(self, handle):
        _check("hsa_ptree_unlock", lib().hsa_ptree_unlock(self._h, int(handle)))

    def evict_full(self, n_tokens, slot_cap=None, row_cap=None):
        """-> (freed Full slots, freed ring rows).  The default capacities are what the
        tree holds, so every evictable leaf fits."""
        if slot_cap is None or row_cap is None:
            cached, rows, _ = self.stats()
            slot_cap = min(max(cached, 1), (1 << 31) - 1) if slot_cap is None else slot_cap
            row_cap = max(rows, 1) if row_cap is None else row_cap
        fs = torch.empty(max(slot_cap, 1), dtype=torch.int32)
        fr = torch.empty(max(row_cap, 1), dtype=torch.int32)
        ns, nr = ctypes.c_int32(), ctypes.c_int32()
        _check("hsa_ptree_evict_full", lib().hsa_ptree_evict_full(
            self._h, int(n_tokens), ctypes.c_void_p(fs.data_ptr()), int(slot_cap),
            ctypes.byref(ns), ctypes.c_void_p(fr.data_ptr()), int(row_cap), ctypes.byref(nr)))
        return fs[:ns.value].clone(), fr[:nr.value].clone()

    def evict_swa(self, n_rows):
        fr = torch.empty(max(int(n_rows), 1), dtype=torch.int32)
        nf = ctypes.c_int32()
        _check("hsa_ptree_evict_swa", lib().hsa_ptree_evict_swa(
            self._h, int(n_rows), ctypes.c_void_p(fr.data_ptr()), ctypes.byref(nf)))
        return fr[:nf.value].clone()

    def stats(self):
        """-> (cached tokens, ring rows held, nodes)."""
        c, rh, nn = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check("hsa_ptree_stats", lib().hsa_ptree_stats(self._h, ctypes.byref(c),
                                                        ctypes.byref(rh), ctypes.byref(nn)))
        return c.value, rh.value, nn.value

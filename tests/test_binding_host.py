"""Host-side marshalling of the Python binding, without a GPU: the library is
replaced by a recorder and the device check relaxed, so that the shape checks the
binding makes before handing plain pointers to the C ABI run on CPU tensors.

Every entry point must refuse a tensor whose size disagrees with the pool (the C
ABI cannot see sizes) and pass a well-formed call through with the sizes it was
given."""
import ctypes
import types

import pytest
import torch

from full_attention_kv_gb300 import binding

Hq, Hkv, d, W, PAGE = 16, 2, 128, 128, 64


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "hsa_decode_workspace_bytes":
            return lambda *a: 64
        if name == "hsa_status_string":
            return lambda s: b"fake"

        def fn(*args):
            self.calls.append((name, args))
            return binding.HSA_OK
        return fn


@pytest.fixture
def fake(monkeypatch):
    def need(t, name, dtype, device=None, ndim=None):
        if not isinstance(t, torch.Tensor):
            raise TypeError(name)
        if t.dtype != dtype:
            raise TypeError(name)
        if not t.is_contiguous():
            raise ValueError(name)
        if ndim is not None and t.dim() != ndim:
            raise ValueError(name)

    rec = _Recorder()
    monkeypatch.setattr(binding, "_need", need)
    monkeypatch.setattr(binding, "lib", lambda: rec)
    return rec


def _pool():
    bt = torch.zeros((4, 8), dtype=torch.int32)
    rr = torch.arange(4, dtype=torch.int32)
    full = torch.zeros((8, Hkv, PAGE, d), dtype=torch.bfloat16)
    ring = torch.zeros((4, Hkv, W, d), dtype=torch.bfloat16)
    return binding.DualPool([False, True], [ring, full], [ring.clone(), full.clone()], bt, rr, Hq)


def _bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def test_decode_shapes(fake):
    pool = _pool()
    B, T = 3, 2
    q, k, v, cl = _bf(B, T, Hq, d), _bf(B, T, Hkv, d), _bf(B, T, Hkv, d), _i32(B)
    binding.hsa_decode_attn(pool, 1, q, k, v, cl, 0.1, stream=0)
    name, args = fake.calls[-1]
    assert name == "hsa_decode_attn" and args[6:8] == (B, T)
    binding.hsa_decode_attn_append(pool, 1, q, k, v, cl, 0.1, stream=0)
    assert fake.calls[-1][0] == "hsa_decode_attn_append"
    binding.hsa_decode_attn_noalloc(pool, 1, q, k, v, cl, 0.1, torch.empty_like(q), stream=0)
    assert fake.calls[-1][0] == "hsa_decode_attn_noalloc"
    n = len(fake.calls)
    bad = [
        (_bf(B, T, Hq + 1, d), k, v, cl),      # query heads
        (q, _bf(B, T, Hkv * 2, d), v, cl),     # KV heads
        (q, k, _bf(B, T + 1, Hkv, d), cl),     # tokens
        (q, k, v, _i32(B - 1)),                # cached_len
        (_bf(B, T, Hq, 64), k, v, cl),         # head dim
    ]
    for args in bad:
        with pytest.raises(ValueError):
            binding.hsa_decode_attn(pool, 1, *args, 0.1, stream=0)
        with pytest.raises(ValueError):
            binding.hsa_decode_attn_noalloc(pool, 1, *args, 0.1, torch.empty_like(args[0]),
                                            stream=0)
    with pytest.raises(ValueError):
        binding.hsa_decode_attn(pool, 1, q, k, v, cl, 0.1, out=_bf(B, T, Hq, d - 8), stream=0)
    with pytest.raises(ValueError):
        binding.hsa_decode_attn(pool, 1, q, k, v, cl, 0.1, dev_err=_i32(0), stream=0)
    assert len(fake.calls) == n  # nothing reached the library


def test_prefill_shapes(fake):
    pool = _pool()
    R, rows = 2, 300
    q, k, v = _bf(rows, Hq, d), _bf(rows, Hkv, d), _bf(rows, Hkv, d)
    cu, pl, seq = _i32(R + 1), _i32(R), _i32(R)
    binding.hsa_prefill_attn(pool, 1, q, k, v, cu, pl, seq, 200, 0.1, stream=0)
    name, args = fake.calls[-1]
    assert name == "hsa_prefill_attn" and args[8:11] == (R, rows, 200)
    n = len(fake.calls)
    for args in [(q, _bf(rows - 1, Hkv, d), v, cu, pl, seq),
                 (q, k, _bf(rows, Hq, d), cu, pl, seq),
                 (q, k, v, _i32(R), pl, seq),
                 (q, k, v, cu, _i32(R + 1), seq)]:
        with pytest.raises(ValueError):
            binding.hsa_prefill_attn(pool, 1, *args, 200, 0.1, stream=0)
    assert len(fake.calls) == n


def test_append_shapes(fake):
    pool = _pool()
    k = _bf(5, Hkv, d)
    binding.hsa_kv_append(pool, 0, k, k.clone(), _i32(3), _i32(2), _i32(2), stream=0)
    name, args = fake.calls[-1]
    assert name == "hsa_kv_append" and args[7:9] == (2, 5)
    for kk, vv in [(_bf(5, Hkv + 1, d), _bf(5, Hkv + 1, d)), (k, _bf(4, Hkv, d))]:
        with pytest.raises(ValueError):
            binding.hsa_kv_append(pool, 0, kk, vv, _i32(3), _i32(2), _i32(2), stream=0)


def test_window_safe_shapes(fake):
    m, pos = _i32(7), _i32(7, W)
    binding.hsa_window_safe_len(m, pos, W, stream=0)
    assert fake.calls[-1][0] == "hsa_window_safe_len"
    with pytest.raises(ValueError):
        binding.hsa_window_safe_len(m, pos, W, out=_i32(6), stream=0)
    with pytest.raises(ValueError):
        binding.hsa_window_safe_len(m, _i32(7, W - 1), W, stream=0)
    off = torch.zeros(8, dtype=torch.int64)
    live = torch.zeros(1, dtype=torch.uint8)
    binding.hsa_window_safe_len_bitmap(m, off, live, W, stream=0)
    with pytest.raises(ValueError):
        binding.hsa_window_safe_len_bitmap(m, off[:7], live, W, stream=0)


def test_pool_struct_mirrors_the_tensors(fake):
    pool = _pool()
    c = pool.c
    assert (c.n_layers, c.num_blocks, c.page_size, c.max_blocks, c.n_ring_rows, c.batch) == \
        (2, 8, PAGE, 8, 4, 4)
    assert (c.W, c.Hq, c.Hkv, c.d) == (W, Hq, Hkv, d)
    assert [c.layer_is_full[i] for i in range(2)] == [0, 1]
    assert [c.layer_kv_fp8[i] for i in range(2)] == [0, 0]
    assert c.k[1] == pool.k[1].data_ptr() and c.v[0] == pool.v[0].data_ptr()
    assert ctypes.sizeof(binding.HsaPools) >= 16 * 4


def test_usage_flow_passes_the_binding(fake, monkeypatch):
    """The documented flow of a decode step -- allocate the dual pool, fill it with
    hsa_kv_append, then one fused decode step -- on CPU tensors against the recorder:
    every call is well formed and reaches the library."""
    monkeypatch.setattr(binding.torch.cuda, "current_stream",
                        lambda: types.SimpleNamespace(cuda_stream=0))
    dev = "cpu"
    full = [False, True]                                   # one sliding, one full layer
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32)  # 2 sequences x 2 pages
    rr = torch.tensor([1, 0], dtype=torch.int32)
    pool = binding.DualPool.allocate(full, num_blocks=4, n_ring_rows=2, block_tables=bt,
                                     ring_row=rr, Hq=32, Hkv=4, device=dev)
    for layer in range(2):
        k = torch.zeros((70, 4, 128), dtype=torch.bfloat16)
        v = torch.zeros_like(k)
        cu = torch.tensor([0, 30, 70], dtype=torch.int32)
        seq = torch.tensor([0, 1], dtype=torch.int32)
        start = torch.tensor([0, 0], dtype=torch.int32)
        binding.hsa_kv_append(pool, layer, k, v, cu, seq, start)
    q = torch.zeros((2, 1, 32, 128), dtype=torch.bfloat16)
    kn = torch.zeros((2, 1, 4, 128), dtype=torch.bfloat16)
    cl = torch.tensor([30, 40], dtype=torch.int32)
    ws = binding.decode_workspace(pool, 2, 1, dev)
    out = binding.hsa_decode_attn_append(pool, 1, q, kn, kn.clone(), cl, 128 ** -0.5,
                                         workspace=ws)
    names = [c[0] for c in fake.calls]
    assert names.count("hsa_kv_append") == 2 and names[-1] == "hsa_decode_attn_append"
    assert tuple(out.shape) == (2, 1, 32, 128)

"""Device-side setup of a drawn workload through the library's own calls.

Allocates the dual KV pool for a sub-stack of layers, writes every sequence's
cached prefix into it with ``hsa_kv_append`` (the cached prefix is "already
resident in the pools" when a step starts), and collects the host-side copies of
the generator's tensors that the oracle needs.  No attention or placement
arithmetic here: placement is done on the device by the library.
"""
import numpy as np
import torch

import full_attention_kv_gb300 as hsa
import workload


def make_pool(inst, layers=None, device="cuda", stale="random", max_bytes=1 << 31, fp8=False):
    """DualPool holding the cached prefix of every sequence for `layers`.

    Pool layer i is model layer layers[i].  `stale` = "random" fills unwritten pool
    rows with random bf16 (so that reading them would show), "zero" zero-fills.
    fp8=True / "e4m3" / "e5m2" stores the full layers as FP8 layers of that format
    (zero-filled, quantised on append by the library); sliding rings stay bf16.
    """
    cfg = inst.cfg
    layers = list(range(cfg.n_layers)) if layers is None else list(layers)
    full = [inst.full[l] for l in layers]
    if fp8:
        bt = torch.from_numpy(inst.block_tables).to(device)
        rr = torch.from_numpy(inst.ring_row).to(device)
        pool = hsa.DualPool.allocate(full, inst.num_blocks, inst.n_ring_rows, bt, rr, cfg.Hq,
                                     cfg.Hkv, d=cfg.d, W=cfg.W, page=cfg.page, device=device,
                                     kv_fp8=fp8)
        for i, l in enumerate(layers):
            fill_layer(inst, pool, i, l, device, max_bytes=max_bytes)
        return pool
    ks, vs = [], []
    for l in layers:
        if stale == "random":
            k, v = workload.pool_init(inst, l, device)
        else:
            shape = ((inst.num_blocks, cfg.Hkv, cfg.page, cfg.d) if inst.full[l]
                     else (inst.n_ring_rows, cfg.Hkv, cfg.W, cfg.d))
            k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        ks.append(k)
        vs.append(v)
    bt = torch.from_numpy(inst.block_tables).to(device)
    rr = torch.from_numpy(inst.ring_row).to(device)
    pool = hsa.DualPool(full, ks, vs, bt, rr, cfg.Hq, W=cfg.W, page=cfg.page)
    for i, l in enumerate(layers):
        fill_layer(inst, pool, i, l, device, max_bytes=max_bytes)
    return pool


def fill_layer(inst, pool, pool_layer, layer, device="cuda", max_bytes=1 << 31):
    """Append every sequence's cached history of `layer`, batching sequences."""
    cfg = inst.cfg
    row_bytes = cfg.Hkv * cfg.d * 2 * 2
    batch = []
    size = 0

    def flush():
        if not batch:
            return
        k = torch.cat([b[1] for b in batch])
        v = torch.cat([b[2] for b in batch])
        counts = [b[1].shape[0] for b in batch]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32,
                          device=device)
        seq = torch.tensor([b[0] for b in batch], dtype=torch.int32, device=device)
        start = torch.tensor([b[3] for b in batch], dtype=torch.int32, device=device)
        hsa.hsa_kv_append(pool, pool_layer, k.contiguous(), v.contiguous(), cu, seq, start)
        batch.clear()

    for s in range(inst.R):
        k, v, start = workload.history(inst, layer, s, device)
        if k.shape[0] == 0:
            continue
        batch.append((s, k, v, start))
        size += k.shape[0] * row_bytes
        if size >= max_bytes:
            flush()
            size = 0
    flush()
    torch.cuda.synchronize()


def decode_inputs(inst, layer, device="cuda"):
    """(q [B,T,Hq,d], k_new [B,T,Hkv,d], v_new, cached_len [B]) for one layer."""
    cfg = inst.cfg
    q, k, v = workload.new_tokens(inst, layer, device)
    B, T = inst.R, cfg.T
    cl = torch.from_numpy(inst.prefix).to(device)
    return (q.view(B, T, cfg.Hq, cfg.d), k.view(B, T, cfg.Hkv, cfg.d),
            v.view(B, T, cfg.Hkv, cfg.d), cl)


def prefill_inputs(inst, layer, device="cuda"):
    """(q [rows,Hq,d], k_new [rows,Hkv,d], v_new, cu_rows, prefix_len, seq_idx)."""
    q, k, v = workload.new_tokens(inst, layer, device)
    cu = torch.from_numpy(inst.cu_new).to(device)
    pl = torch.from_numpy(inst.prefix).to(device)
    seq = torch.arange(inst.R, dtype=torch.int32, device=device)
    return q, k, v, cu, pl, seq


def oracle_case(inst, layer, seqs, device="cuda"):
    """Host copies of everything the oracle needs for `seqs` of one layer.

    Histories are regenerated from the generator (never read back from a pool).
    Requests not in `seqs` get empty histories (their rows must not be asked for).
    """
    cfg = inst.cfg
    q, k, v = workload.new_tokens(inst, layer, device)
    hk, hv, off, start = [], [], [0], []
    want = set(int(s) for s in seqs)
    for s in range(inst.R):
        if s in want:
            a, b, st = workload.history(inst, layer, s, device)
            hk.append(a.cpu())
            hv.append(b.cpu())
            off.append(off[-1] + a.shape[0])
            start.append(st)
        else:
            off.append(off[-1])
            start.append(int(inst.prefix[s]))
    empty = torch.zeros((0, cfg.Hkv, cfg.d), dtype=torch.bfloat16)
    return dict(cu_rows=inst.cu_new, prefix_len=inst.prefix, q=q.cpu(), k_new=k.cpu(),
                v_new=v.cpu(), hist_k=torch.cat(hk) if hk else empty,
                hist_v=torch.cat(hv) if hv else empty, hist_off=np.array(off, np.int64),
                hist_start=np.array(start, np.int32))


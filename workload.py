"""Seeded synthetic inputs for the Hybrid-SWA dual-KV-pool attention path.

This module is shared by the tests, the benchmark and the oracle checks.  It only
draws inputs (lengths, page allocations, ring rows, bf16 tensors, window-safe
cases); it holds none of the attention, placement or window-safe arithmetic.

Workload shapes follow the pages: a 70-layer stack with 60 sliding-window layers
(W = 128) and 10 full layers interleaved 6:1 (youleyou.com "小米MiMo首次公开模型推理
系统全链路优化降价99%", s1; hotdry.top "MiMo-V2.5 ultra-speed inference
architecture", "Hybrid SWA"), context buckets 0-64K / 64K-256K / 256K-1M (same
pages, s2 "调度与Prefill优化" / "PD 分离与长度分桶"), 3 MTP draft tokens (s2
"Decode加速与多模态优化").  Reading: the full layers are those with
layer % 7 == 6.  The pages measure on production traffic; these seeded draws
stand in for it.

Tensors are bf16 N(0, 1) from torch.Generator; lengths come from random.Random.
Every history tensor of (layer, sequence) has its own derived seed, so any
sample can be regenerated on its own.
"""
import math
import random
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np
import torch

PAGE = 64
WINDOW = 128


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    kind: str                 # "decode" or "prefill"
    n_layers: int
    Hq: int
    Hkv: int
    d: int = 128
    W: int = WINDOW
    page: int = PAGE
    B: int = 0                # decode: sequences
    T: int = 1                # decode: query tokens per sequence (1 + MTP drafts)
    contexts: tuple = ()      # decode: fixed contexts, else drawn
    ctx_lo: int = 0
    ctx_hi: int = 0
    buckets: tuple = ()       # ((lo, hi, weight), ...)
    R: int = 0                # prefill: requests
    prefixes: tuple = ()      # prefill: fixed cached lengths, else drawn
    chunks: tuple = ()        # prefill: fixed chunk lengths, else drawn
    prefix_lo: int = 0
    prefix_hi: int = 0
    chunk_lo: int = 0
    chunk_hi: int = 0
    n_window_cases: int = 0

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


CONFIGS = {
    "tiny": Config("tiny", 0, "decode", 7, 16, 2, B=4, T=1, contexts=(100, 128, 300, 512)),
    "decode": Config("decode", 1, "decode", 70, 32, 4, B=32, T=1, ctx_lo=8192, ctx_hi=65536),
    "prefill": Config("prefill", 2, "prefill", 70, 32, 4, R=8, prefix_lo=16384,
                      prefix_hi=131072, chunk_lo=2048, chunk_hi=8192),
    "long": Config("long", 3, "decode", 70, 32, 4, B=4, T=1, ctx_lo=262144, ctx_hi=1048576),
    "mtp": Config("mtp", 4, "decode", 70, 32, 4, B=48, T=4,
                  buckets=((0, 65536, 0.7), (65536, 262144, 0.2), (262144, 1048576, 0.1)),
                  n_window_cases=1000),
}


def layer_is_full(n_layers: int) -> List[bool]:
    """6:1 interleave: layers 6, 13, 20, ... are full; the rest slide."""
    return [(l % 7) == 6 for l in range(n_layers)]


@dataclass
class Instance:
    """One drawn workload: lengths, page allocation and ring rows (host arrays)."""
    cfg: Config
    prefix: np.ndarray          # int32 [R]: cached tokens per sequence/request
    new: np.ndarray             # int32 [R]: new tokens per sequence/request
    cu_new: np.ndarray          # int32 [R+1]: offsets of new rows
    block_tables: np.ndarray    # int32 [R, max_blocks], -1 = unallocated
    num_blocks: int
    ring_row: np.ndarray        # int32 [R]
    n_ring_rows: int
    full: List[bool] = field(default_factory=list)

    @property
    def R(self) -> int:
        return len(self.prefix)

    @property
    def rows(self) -> int:
        return int(self.cu_new[-1])


def _pages(n_tokens: int, page: int) -> int:
    return (n_tokens + page - 1) // page


def draw(cfg: Config, *, R: Optional[int] = None, rng_seed: Optional[int] = None) -> Instance:
    """Draw lengths, a randomly permuted page allocation and ring rows.

    Pages cover prefix + new tokens so that the new tokens can be appended.
    ``R`` truncates the draw to its first R sequences (same values).
    """
    rng = random.Random(cfg.seed if rng_seed is None else rng_seed)
    if cfg.kind == "decode":
        n = cfg.B
        if cfg.contexts:
            prefix = list(cfg.contexts)
        elif cfg.buckets:
            prefix = []
            for _ in range(n):
                u = rng.random()
                acc = 0.0
                for lo, hi, w in cfg.buckets:
                    acc += w
                    if u < acc:
                        break
                prefix.append(rng.randint(lo, hi))
        else:
            prefix = [rng.randint(cfg.ctx_lo, cfg.ctx_hi) for _ in range(n)]
        new = [cfg.T] * n
    elif cfg.prefixes:
        n = len(cfg.prefixes)
        prefix, new = list(cfg.prefixes), list(cfg.chunks)
    else:
        n = cfg.R
        prefix = [rng.randint(cfg.prefix_lo, cfg.prefix_hi) for _ in range(n)]
        new = [rng.randint(cfg.chunk_lo, cfg.chunk_hi) for _ in range(n)]
    if R is not None:
        prefix, new = prefix[:R], new[:R]
        n = R
    pages = [_pages(p + t, cfg.page) for p, t in zip(prefix, new)]
    total = sum(pages)
    perm = list(range(total))
    rng.shuffle(perm)
    max_blocks = max(pages) if pages else 1
    bt = np.full((n, max(max_blocks, 1)), -1, np.int32)
    k = 0
    for s, np_ in enumerate(pages):
        bt[s, :np_] = perm[k:k + np_]
        k += np_
    rows = list(range(n))
    rng.shuffle(rows)
    cu = np.zeros(n + 1, np.int32)
    cu[1:] = np.cumsum(new)
    return Instance(cfg, np.array(prefix, np.int32), np.array(new, np.int32), cu, bt,
                    max(total, 1), np.array(rows, np.int32), max(n, 1),
                    layer_is_full(cfg.n_layers))


def shard(cfg: Config, rank: int) -> Config:
    """Rank `rank`'s share of a data-parallel global batch: rank 0 draws exactly the
    single-GPU workload; every other rank draws its own seeded batch of the same
    shape (sequences are independent, so ranks never exchange data)."""
    if rank == 0:
        return cfg
    return replace(cfg, index=cfg.index + 1000 * rank)


def _seed(cfg: Config, *parts: int) -> int:
    s = cfg.seed
    for p in parts:
        s = (s * 1000003 + p + 1) % (2 ** 61 - 1)
    return s


def randn_bf16(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def history(inst: Instance, layer: int, seq: int, device="cpu"):
    """Cached K/V of one sequence in one layer: ([n, Hkv, d], [n, Hkv, d], start).

    Full layers hold every cached position 0 .. prefix-1.  Sliding layers hold
    only the positions the SWA KV Pool still keeps, max(0, prefix-W) .. prefix-1.
    """
    cfg = inst.cfg
    P = int(inst.prefix[seq])
    start = 0 if inst.full[layer] else max(0, P - cfg.W)
    n = P - start
    k = randn_bf16((n, cfg.Hkv, cfg.d), _seed(cfg, 1, layer, seq, 0), device)
    v = randn_bf16((n, cfg.Hkv, cfg.d), _seed(cfg, 1, layer, seq, 1), device)
    return k, v, start


def new_tokens(inst: Instance, layer: int, device="cpu"):
    """Per-layer query and new K/V rows: q [rows, Hq, d], k/v [rows, Hkv, d].

    Decode rows are ordered (sequence, token), i.e. q viewed as [B, T, Hq, d].
    """
    cfg = inst.cfg
    rows = inst.rows
    q = randn_bf16((rows, cfg.Hq, cfg.d), _seed(cfg, 2, layer, 0), device)
    k = randn_bf16((rows, cfg.Hkv, cfg.d), _seed(cfg, 2, layer, 1), device)
    v = randn_bf16((rows, cfg.Hkv, cfg.d), _seed(cfg, 2, layer, 2), device)
    return q, k, v


def pool_init(inst: Instance, layer: int, device="cpu"):
    """Initial (stale) pool contents of one layer before any append: random bf16.

    Full layers: [num_blocks, Hkv, page, d]; sliding layers: [n_ring_rows, Hkv, W, d].
    Stale rows are never attended; a random fill makes that visible in tests.
    """
    cfg = inst.cfg
    if inst.full[layer]:
        shape = (inst.num_blocks, cfg.Hkv, cfg.page, cfg.d)
    else:
        shape = (inst.n_ring_rows, cfg.Hkv, cfg.W, cfg.d)
    k = randn_bf16(shape, _seed(cfg, 3, layer, 0), device)
    v = randn_bf16(shape, _seed(cfg, 3, layer, 1), device)
    return k, v


def window_cases(n: int, W: int, seed: int, m_hi: int = 4096):
    """Seeded prefix-match cases for the window-safe length rule.

    Ring form: m ~ U[0, m_hi]; the ring was filled by appending positions 0 .. q-1
    with q = m (probability 0.5) or q = m + U[1, 256] (the ring ran past the
    match); each slot then holds the most recent position of its residue below q.
    Afterwards every slot is freed (-1) with probability e ~ U[0, 0.2], and with
    probability 0.1 the whole ring is freed.
    Bitmap form (prefix-tree view): every other case also gets a live byte per
    position 0 .. m-1 with a few random freed intervals.
    Returns (match_len [n], slot_pos [n, W], bitmap cases (idx, match_len, off, live)).
    """
    rng = random.Random(seed)
    match = np.zeros(n, np.int32)
    slots = np.full((n, W), -1, np.int32)
    for k in range(n):
        m = rng.randint(0, m_hi)
        q = m if rng.random() < 0.5 else m + rng.randint(1, 256)
        match[k] = m
        # the ring was written in position order: positions 0 .. q-1, each into slot
        # p mod W over whatever it held (only the last W writes survive)
        for p in range(max(0, q - W), q):
            slots[k, p % W] = p
        e = rng.uniform(0.0, 0.2)
        for j in range(W):
            if rng.random() < e:
                slots[k, j] = -1
        if rng.random() < 0.1:
            slots[k, :] = -1
    idx, bm_len, lives = [], [], []
    for k in range(0, n, 2):
        m = int(match[k])
        live = np.ones(m, np.uint8)
        if rng.random() < 0.3 and m > 0:
            live[:rng.randint(0, m)] = 0          # old SWA KV already evicted
        for _ in range(rng.randint(0, 3)):
            if m == 0:
                break
            a = rng.randint(0, m - 1)
            live[a:a + rng.randint(1, 300)] = 0
        idx.append(k)
        bm_len.append(m)
        lives.append(live)
    off = np.zeros(len(lives) + 1, np.int64)
    off[1:] = np.cumsum([len(x) for x in lives])
    live_all = np.concatenate(lives) if lives else np.zeros(0, np.uint8)
    return match, slots, (np.array(idx, np.int32), np.array(bm_len, np.int32), off, live_all)

"""Host-side arithmetic of bench.py: the algorithmic bytes and flops the roofline
divides by, and the code digest that keys a traffic capture to a kernel.

The byte and flop counts are checked against hand counts and brute-force key
enumeration on small cases: each query row of a full layer sees every position up
to its own, a sliding-layer row the newest W of them [hotdry.top "MiMo-V2.5
ultra-speed inference architecture", "Hybrid SWA"]."""
import dataclasses

import numpy as np

import bench
import workload


def test_decode_bytes_by_hand():
    inst = workload.draw(workload.CONFIGS["tiny"])  # contexts 100, 128, 300, 512; T = 1
    per_tok = 2 * 2 * 128 * 2        # K and V, Hkv = 2, d = 128, bf16
    qo = 2 * 4 * 1 * 16 * 128 * 2    # q read + out written: R x T x Hq x d, bf16
    assert bench.decode_bytes(inst, True) == (101 + 129 + 301 + 513) * per_tok + qo
    assert bench.decode_bytes(inst, False) == (101 + 128 + 128 + 128) * per_tok + qo
    # FP8 full layer: cached rows as codes + one fp32 scale per (token, head), new rows bf16
    fp8_tok = 2 * 2 * (128 + 4)
    assert bench.decode_bytes(inst, True, fp8=True) == 1040 * fp8_tok + 4 * per_tok + qo


def test_decode_bytes_mtp_sliding_window():
    """T = 4: the oldest of the four new rows still sees W keys, the newest W + 3
    distinct keys are read in all."""
    cfg = dataclasses.replace(workload.CONFIGS["tiny"], T=4, contexts=(0, 5, 200), B=3)
    inst = workload.draw(cfg)
    per_tok = 2 * cfg.Hkv * cfg.d * 2
    qo = 2 * 3 * 4 * cfg.Hq * cfg.d * 2
    assert bench.decode_bytes(inst, False) == (4 + 9 + 131) * per_tok + qo


def _brute_keys(P, C, W, full):
    n = 0
    for i in range(C):
        q = P + i
        n += sum(1 for k in range(q + 1) if full or q - k < W)
    return n


def test_prefill_flops_against_enumeration():
    cfg = dataclasses.replace(workload.CONFIGS["prefill"], prefixes=(0, 3, 130, 257),
                              chunks=(5, 128, 1, 300), R=4)
    inst = workload.draw(cfg)
    for full in (True, False):
        keys = sum(_brute_keys(int(P), int(C), cfg.W, full)
                   for P, C in zip(inst.prefix, inst.new))
        assert bench.prefill_flops(inst, full) == 4 * cfg.d * cfg.Hq * keys
        assert int(bench.keys_per_row(inst, full).sum()) == keys


def test_code_digest_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int *p) {\n  p[0] = 1;  // one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("/* other\n   header */\n\n__global__ void k(int *p) {\n  p[0] = 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("__global__ void k(int *p) {\n  p[0] = 2;\n}\n")
    assert bench.code_digest(a) == bench.code_digest(b)
    assert bench.code_digest(a) != bench.code_digest(c)


def test_pool_allocation_realises_the_kv_byte_ratio():
    """The dual pool's allocation for a drawn workload over an all-full stack's
    equals the pages' KV-byte ratio (oracle.kv_bytes, pinned to "about 1/7") summed
    over the sequences, up to the rounding of each sequence to whole 64-token pages."""
    import oracle
    for name in ("decode", "long", "mtp"):
        inst = workload.draw(workload.CONFIGS[name])
        cfg = inst.cfg
        per_tok = 2 * cfg.Hkv * cfg.d * 2
        lens = [int(L) for L in inst.prefix + inst.new]
        hyb = sum(oracle.kv_bytes(inst.full, cfg.W, L, per_tok) for L in lens)
        full = sum(oracle.kv_bytes([1] * cfg.n_layers, cfg.W, L, per_tok) for L in lens)
        got = bench.pool_ratio(inst)
        assert abs(got - hyb / full) / (hyb / full) < 0.02, (name, got, hyb / full)
    inst = workload.draw(workload.CONFIGS["decode"])
    assert 1 / 7 < bench.pool_ratio(inst) < 0.16


def test_workload_config_names_the_workload():
    """Both arms report this object: JSON-serialisable, the workload named by what
    it is with its sizes, the whole-job batch over the ranks."""
    import json
    for name, cfg in workload.CONFIGS.items():
        inst = workload.draw(cfg)
        c = bench.workload_config(inst, 2)
        json.dumps(c)
        assert c["workload"].startswith(name + ": 70-layer" if cfg.n_layers == 70 else name)
        assert c["global_batch"] == 2 * inst.R and c["T"] == cfg.T
        assert c["parallelism"] == "replicas x2"
        assert 0 < c["kv_pool_vs_all_full"] <= 1


def test_prefill_sliding_bytes_against_enumeration():
    """Sliding-layer prefill moves q in, out back, the chunk's new K/V in, and each
    prefix position that some chunk row still sees (brute force over the rows)."""
    cfg = dataclasses.replace(workload.CONFIGS["prefill"], prefixes=(0, 3, 130, 257, 127),
                              chunks=(5, 128, 1, 300, 2), R=5)
    inst = workload.draw(cfg)
    per_tok = 2 * cfg.Hkv * cfg.d * 2
    ring = 0
    for P, C in zip(inst.prefix, inst.new):
        seen = set()
        for i in range(int(C)):
            q = int(P) + i
            seen.update(k for k in range(int(P)) if q - k < cfg.W)
        ring += len(seen) * per_tok
    rows = inst.rows
    want = 2 * rows * cfg.Hq * cfg.d * 2 + 2 * rows * cfg.Hkv * cfg.d * 2 + ring
    assert bench.prefill_swa_bytes(inst) == want


def test_traffic_is_dropped_once_the_kernel_source_changes(tmp_path, monkeypatch):
    """A capture's DRAM figure is reported only while the kernel's source (comments
    aside) still matches the digest it was taken on."""
    src = tmp_path / "full_attention_kv_gb300" / "csrc"
    src.mkdir(parents=True)
    f = src / "k.cu"
    f.write_text("__global__ void k(int *p) { p[0] = 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC", {("w", "full"): ("k.cu", bench.code_digest(f), 123)})
    assert bench._traffic("w", "full") == 123
    assert bench._traffic("w", "sliding") is None
    f.write_text("// a comment\n__global__ void k(int *p) { p[0] = 1; }\n")
    assert bench._traffic("w", "full") == 123
    f.write_text("__global__ void k(int *p) { p[0] = 2; }\n")
    assert bench._traffic("w", "full") is None

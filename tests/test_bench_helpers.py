"""Host-side helpers of bench.py, on CPU: the profiled-traffic lookup (rows
count only for the digest of the current kernel sources) and the oracle CPU
baseline timer for each kind of step it times (decode, decode over fp8
pools, windowed decode, several new tokens per sequence)."""
import dataclasses

import numpy as np
import pytest
import torch

import bench
from paged_kv_cache_123_gb300 import workloads


def test_traffic_rows_need_the_current_digest(tmp_path, monkeypatch):
    dig = bench.kernel_sources_digest()
    assert len(dig) == 16
    f = tmp_path / "traffic.txt"
    f.write_text(f"cfg_a {dig} 1234\ncfg_b 0123456789abcdef 99\nmalformed line here too\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    assert bench.profiled_traffic("cfg_a") == 1234
    assert bench.profiled_traffic("cfg_b") is None       # taken on other sources
    assert bench.profiled_traffic("cfg_c") is None       # never taken
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.txt"))
    assert bench.profiled_traffic("cfg_a") is None


def test_digest_follows_every_kernel_source(tmp_path, monkeypatch):
    for name, body in (("a.cu", "x"), ("b.cuh", "y"), ("c.h", "z"), ("notes.txt", "w")):
        (tmp_path / name).write_text(body)
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    d0 = bench.kernel_sources_digest()
    (tmp_path / "notes.txt").write_text("changed")        # not a source
    assert bench.kernel_sources_digest() == d0
    (tmp_path / "b.cuh").write_text("y2")                 # a header counts
    assert bench.kernel_sources_digest() != d0


@pytest.mark.parametrize("kind,window,N", [("decode", 0, 1), ("decode", 300, 1),
                                           ("fp8", 0, 1), ("fp8", 300, 1), ("mq", 0, 3)])
def test_oracle_timer_each_kind(kind, window, N):
    base = workloads.CONFIGS["gqa72b"]
    cfg = dataclasses.replace(base, num_seqs=3, name="gqa72b_s3", ctx_lo=200, ctx_hi=600)
    inp = workloads.make_decode_inputs(cfg, seed=cfg.seed)
    arr = bench.oracle_arrays(inp)
    if kind == "fp8":
        codes = (inp.key_cache.float() * 48).clamp(-448, 448).to(torch.float8_e4m3fn)
        arr["kc"] = arr["vc"] = codes.view(torch.uint8).numpy()
    if kind == "mq":
        arr["q"] = np.repeat(arr["q"], N, axis=0)
    timer = bench.OracleTimer(arr, cfg, inp.scale, 2, kind=kind, window=window, ks=1 / 48,
                              vs=1 / 48, N=N)
    try:
        timer.size_sample(0.05)
        gbs, tps, desc, dt = timer.measure()
    finally:
        timer.close()
    assert gbs > 0 and tps > 0 and dt > 0
    lens = inp.seq_lens.tolist()
    if kind == "mq":
        # (sequence, KV head) units; every unit of the small batch is sampled
        assert len(timer.units) == 3 * cfg.num_kv_heads
        assert "(sequence, KV head) units" in desc
    else:
        att = [min(L, window) if window else L for L in lens]
        assert timer.unit_tok == att
        assert (f"window {window}" in desc) == bool(window)
    assert (kind == "fp8") == ("fp8" in desc)


def test_block_scale_bytes_count_every_attended_block():
    # brute force: the set of blocks that hold an attended token
    rng = np.random.default_rng(3)
    for _ in range(200):
        B = int(rng.choice([1, 4, 16, 64]))
        lens = rng.integers(0, 300, size=5).tolist()
        W = int(rng.choice([0, 1, 7, 64, 250, 400]))
        want = 0
        for L in lens:
            lo = L - W if 0 < W < L else 0
            want += len({j // B for j in range(lo, L)})
        assert bench.block_scale_bytes(lens, W, B, 3) == want * 3 * 2 * 4, (lens, W, B)

"""Sliding-window decode through the C ABI against the fp64 oracle: every
dtype, group size and block size of the decode kernels, windows shorter and
longer than a tile and a partition, skipped blocks released (table entries
-1, never read), fp8 pools, and a multi-step decode loop in which the host
pool frees blocks as the window slides."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [0, 1, 15, 63, 64, 65, 200, 700, 2000]


def _oracle(inp, cfg, window, tables=None):
    return oracle.decode_attention(
        np_(inp.q), np_(inp.key_cache), np_(inp.value_cache),
        inp.block_tables.numpy() if tables is None else tables, inp.seq_lens.numpy(),
        inp.scale, cfg.num_kv_heads, cfg.block_size, cfg.dtype, window=window)


def _gpu(inp, window, tables=None, partition=0, out=None):
    g = inp.block_tables if tables is None else torch.from_numpy(tables)
    return pa.pa_decode_attention_window(
        inp.q.to(DEV), inp.key_cache.to(DEV), inp.value_cache.to(DEV), g.to(DEV),
        inp.seq_lens.to(DEV), inp.scale, inp.key_cache.shape[1], window,
        max_seq_len=inp.max_seq_len, partition_size=partition)


def _released(inp, window, B):
    """Block table with the skipped blocks' entries replaced by -1."""
    tab = inp.block_tables.numpy().copy()
    for s, L in enumerate(inp.seq_lens.tolist()):
        tab[s, :oracle.skipped_blocks(L, window, B)] = -1
    return tab


CASES = [(dt, G, 16, W, 0) for dt in ("f32", "f16", "bf16") for G in (1, 8)
         for W in (1, 64, 100)]
CASES += [("bf16", G, B, W, 0) for G in (2, 4) for B in (8, 64) for W in (5, 130)]
CASES += [("f16", 1, 1, 37, 0), ("bf16", 8, 128, 70, 0), ("bf16", 8, 128, 300, 0),
          ("f16", 4, 16, 150, 64), ("bf16", 8, 16, 1000, 128), ("f32", 1, 32, 3000, 0)]


@pytest.mark.parametrize("dtype,G,B,W,partition", CASES)
def test_window_matches_oracle_with_skipped_blocks_released(dtype, G, B, W, partition):
    Hkv = 2
    cfg = workloads.DecodeConfig("win", len(LENS), Hkv * G, Hkv, 128, B, dtype,
                                 seed=31 + G + B + W)
    inp = workloads.make_decode_inputs(cfg, context_lens=[max(L - 1, 0) for L in LENS])
    inp.seq_lens[0] = 0
    want = _oracle(inp, cfg, W)
    tab = _released(inp, W, B)
    out = _gpu(inp, W, tab, partition)
    torch.cuda.synchronize()
    err = max_abs_err(out, want)
    assert err <= TOL[dtype], err
    assert pa.pa_get_device_error() == 0        # no -1 entry was looked up
    # the released entries change nothing
    again = _gpu(inp, W, None, partition)
    torch.cuda.synchronize()
    assert torch.equal(again, out)


@pytest.mark.parametrize("dtype,G,B", [("f16", 1, 16), ("bf16", 8, 16), ("bf16", 4, 128)])
def test_window_covering_every_sequence_is_plain_decode(dtype, G, B):
    cfg = workloads.DecodeConfig("wfull", len(LENS), 2 * G, 2, 128, B, dtype, seed=5)
    inp = workloads.make_decode_inputs(cfg, context_lens=[max(L - 1, 0) for L in LENS])
    plain = pa.pa_decode_attention(inp.q.to(DEV), inp.key_cache.to(DEV),
                                   inp.value_cache.to(DEV), inp.block_tables.to(DEV),
                                   inp.seq_lens.to(DEV), inp.scale, 2,
                                   max_seq_len=inp.max_seq_len)
    for W in (0, inp.max_seq_len, inp.max_seq_len + 77):
        out = _gpu(inp, W)
        torch.cuda.synchronize()
        assert torch.equal(out, plain), W


def test_window_of_one_returns_the_new_value():
    cfg = workloads.DecodeConfig("w1", len(LENS), 16, 2, 128, 16, "bf16", seed=8)
    inp = workloads.make_decode_inputs(cfg, context_lens=[max(L - 1, 1) for L in LENS])
    out = _gpu(inp, 1, _released(inp, 1, 16)).cpu()
    for s, L in enumerate(inp.seq_lens.tolist()):
        blk = int(inp.block_tables[s, (L - 1) // 16])
        for h in range(16):
            assert torch.equal(out[s, h], inp.value_cache[blk, h // 8, (L - 1) % 16])


def test_window_workspace_and_argument_errors():
    n_full = pa.pa_decode_workspace_bytes(64, 64, 8, 128, 16, 32768, 0)
    n_win = pa.pa_decode_window_workspace_bytes(64, 64, 8, 128, 16, 32768, 4096, 0)
    assert 0 <= n_win < n_full
    assert pa.pa_decode_window_workspace_bytes(64, 64, 8, 128, 16, 32768, 0, 0) == n_full
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode_window_workspace_bytes(64, 64, 8, 128, 16, 32768, -1, 0)
    # a window shorter than the longest sequence: one wave of resident CTAs
    # (two per SM for this tensor-core shape), partitions of >= 256 tokens
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits, tok = pa.pa_decode_window_partitioning(16, 32, 8, 16, 32768, 4096, 0)
    assert 16 * 8 * splits <= 2 * sms and splits * tok >= 4096 + 63 and tok % 64 == 0
    assert (splits - 1) * tok < 4096 + 63
    # these partitions give 16 x 8 x 2 items for 2 x SMs slots, close enough
    # to one item per slot that the 16-bit call keeps them (no even schedule)
    assert pa.pa_decode_even_ctas(16, 32, 8, 128, 16, torch.bfloat16, "16bit", 32768, 4096) == 0
    assert pa.pa_decode_window_workspace_bytes(16, 32, 8, 128, 16, 32768, 4096, 0) == (
        0 if splits == 1 else 16 * 32 * splits * (128 * 4 + 8))
    # no window, or one covering every sequence: the unwindowed partitioning
    for W in (0, 32768, 40000):
        assert pa.pa_decode_window_partitioning(16, 32, 8, 16, 32768, W, 0) == \
            pa.pa_decode_partitioning(16, 32, 8, 16, 32768, 0)
    assert pa.pa_decode_window_partitioning(16, 32, 8, 16, 32768, 4096, 1000) == (5, 1024)
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode_window_partitioning(16, 32, 8, 16, 32768, -1, 0)
    cfg = workloads.DecodeConfig("we", 2, 8, 2, 128, 16, "bf16", seed=1)
    inp = workloads.make_decode_inputs(cfg, context_lens=[10, 20])
    with pytest.raises(pa.PagedAttnError):
        _gpu(inp, -3)


@pytest.mark.parametrize("dtype,G,B,W", [("bf16", 8, 16, 100), ("f16", 1, 16, 70),
                                         ("bf16", 4, 64, 1), ("f32", 2, 8, 513)])
def test_fp8_window_matches_oracle(dtype, G, B, W):
    Hkv = 2
    cfg = workloads.DecodeConfig("w8", len(LENS), Hkv * G, Hkv, 128, B, dtype, seed=3 + G + W)
    inp = workloads.make_decode_inputs(cfg, context_lens=[max(L - 1, 0) for L in LENS])
    gen = torch.Generator().manual_seed(B + W)
    ks, vs = 1 / 48, 1 / 40

    def pool(scale):
        x = torch.randn((inp.num_blocks, Hkv, B, 128), generator=gen) / scale
        return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)

    kc, vc = pool(ks), pool(vs)
    want = oracle.decode_attention_fp8(np_(inp.q), kc.numpy(), vc.numpy(),
                                       inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                       inp.scale, Hkv, B, dtype, ks, vs, window=W)
    tab = torch.from_numpy(_released(inp, W, B))
    out = pa.pa_decode_attention_fp8_window(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), tab.to(DEV),
                                            inp.seq_lens.to(DEV), inp.scale, Hkv, ks, vs, W,
                                            max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0


def test_sliding_decode_loop_with_host_pool():
    """Twelve decode steps: the host pool appends a slot per sequence and
    frees the blocks that slide out of the window; freed blocks are reused by
    later appends; each step's output matches the oracle."""
    B, Hkv, G, D, W, S = 8, 2, 4, 128, 20, 4
    NB = 64
    gen = torch.Generator().manual_seed(12)
    pool = pa.BlockPool(NB, B)
    start = [17, 30, 5, 41]
    for s in range(S):
        pool.add_sequence(s, start[s])
        pool.release_skipped(s, W)
    kc = torch.randn((NB, Hkv, B, D), generator=gen).to(torch.bfloat16)
    vc = torch.randn((NB, Hkv, B, D), generator=gen).to(torch.bfloat16)
    kd, vd = kc.to(DEV), vc.to(DEV)
    kh, vh = np_(kc), np_(vc)                  # the oracle's copies of the pools
    for step in range(12):
        pos, pairs = pool.prepare_decode_step(list(range(S)))
        assert pairs == []
        for s in range(S):
            pool.release_skipped(s, W)
        tab = pool.table_rows(list(range(S)), width=16)
        qsl = torch.arange(S + 1, dtype=torch.int32)
        q = torch.randn((S, Hkv * G, D), generator=gen).to(torch.bfloat16)
        k_new = torch.randn((S, Hkv, D), generator=gen).to(torch.bfloat16)
        v_new = torch.randn((S, Hkv, D), generator=gen).to(torch.bfloat16)
        slots = pa.pa_compute_slot_mapping(qsl.to(DEV), torch.from_numpy(pos).to(DEV),
                                           torch.from_numpy(tab).to(DEV), B)
        pa.pa_reshape_and_cache(k_new.to(DEV), v_new.to(DEV), slots, kd, vd)
        want_slots = oracle.slot_mapping(qsl.numpy(), pos, tab, B)
        assert np.array_equal(slots.cpu().numpy(), want_slots)
        oracle.reshape_and_cache(np_(k_new), np_(v_new), want_slots, kh, vh, B)
        lens = torch.from_numpy(pos + 1).to(torch.int32)
        out = pa.pa_decode_attention_window(q.to(DEV), kd, vd, torch.from_numpy(tab).to(DEV),
                                            lens.to(DEV), 0.088, Hkv, W,
                                            max_seq_len=int(lens.max()))
        want = oracle.decode_attention(np_(q), kh, vh, tab, lens.numpy(), 0.088, Hkv, B,
                                       "bf16", window=W)
        torch.cuda.synchronize()
        assert max_abs_err(out, want) <= TOL["bf16"], step
        assert pa.pa_get_device_error() == 0
    # the window holds at most ceil(W / B) + 1 blocks per sequence
    assert NB - pool.num_free() <= S * (-(-W // B) + 1)


@pytest.mark.parametrize("name,W", [("longctx_B16", 4096), ("gqa72b", 1000),
                                    ("llama7b", 333)])
def test_full_size_window_sampled(name, W):
    """Full-size batches with automatic partitioning; skipped blocks released
    on the device table; sampled (sequence, head) pairs against the oracle."""
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs(name, device=DEV)
    cfg = inp.cfg
    tab = _released(type("I", (), {"block_tables": inp.block_tables.cpu(),
                                    "seq_lens": inp.seq_lens.cpu()}), W, cfg.block_size)
    out = pa.pa_decode_attention_window(inp.q, inp.key_cache, inp.value_cache,
                                        torch.from_numpy(tab).to(DEV), inp.seq_lens.to(DEV),
                                        inp.scale, cfg.num_kv_heads, W,
                                        max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    lens = inp.seq_lens.cpu().numpy()
    rng = np.random.default_rng(1)
    seqs = sorted({int(lens.argmax()), int(lens.argmin()),
                   *rng.choice(cfg.num_seqs, size=min(3, cfg.num_seqs), replace=False).tolist()})
    heads = sorted({0, cfg.num_q_heads - 1})
    want = oracle.decode_attention(np_(inp.q), np_(inp.key_cache), np_(inp.value_cache), tab,
                                   lens, inp.scale, cfg.num_kv_heads, cfg.block_size,
                                   cfg.dtype, seqs, heads, window=W)
    assert max_abs_err(out, want, seqs, heads) <= TOL[cfg.dtype]
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("dtype,G,S", [("bf16", 8, 600), ("f16", 4, 700), ("bf16", 2, 640)])
def test_window_many_items_per_cta(dtype, G, S):
    """More (sequence, KV head) items than resident CTAs with a window: each
    CTA of the tensor-core kernel walks several items. Ragged lengths (some
    shorter than the window, some empty), released blocks, every output
    against the oracle."""
    Hkv, B, W = 2, 16, 200
    cfg = workloads.DecodeConfig("wmany", S, Hkv * G, Hkv, 128, B, dtype, seed=40 + G)
    rng = np.random.default_rng(G)
    ctx = rng.integers(0, 900, S).tolist()
    inp = workloads.make_decode_inputs(cfg, context_lens=ctx)
    inp.seq_lens[::97] = 0
    tab = _released(inp, W, B)
    want = _oracle(inp, cfg, W, tab)
    out = _gpu(inp, W, tab)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_abs_err(out, want) <= TOL[dtype]
    splits, _ = pa.pa_decode_window_partitioning(S, Hkv * G, Hkv, B, inp.max_seq_len, W, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert splits * Hkv * S > 2 * sms          # more items than resident CTAs


"""Pins for the oracle's sliding-window decode attention and skipped-block
count: the window of one token returns the new token's value exactly, a
window at least as long as the sequence is plain decode, equal keys give the
mean of the last W values, torch's fp64 scaled_dot_product_attention with a
boolean mask over an independent whole-block gather, brute-force counting of
skippable blocks, and independence from the table entries of skipped
blocks."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_123_gb300 import workloads


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _inputs(dtype="f32", B=4, lens=(1, 5, 9, 17, 40), hq=4, hkv=2, D=64, seed=3):
    cfg = workloads.DecodeConfig("w", len(lens), hq, hkv, D, B, dtype, seed=seed)
    return cfg, workloads.make_decode_inputs(cfg, context_lens=[L - 1 for L in lens])


def _run(inp, cfg, window, tables=None):
    return oracle.decode_attention(
        _np(inp.q), _np(inp.key_cache), _np(inp.value_cache),
        inp.block_tables.numpy() if tables is None else tables, inp.seq_lens.numpy(),
        inp.scale, cfg.num_kv_heads, cfg.block_size, cfg.dtype, window=window)


def test_window_start_reading():
    assert oracle.window_start(10, 0) == 0        # no window
    assert oracle.window_start(10, 10) == 0
    assert oracle.window_start(10, 11) == 0
    assert oracle.window_start(10, 4) == 6        # tokens 6..9
    assert oracle.window_start(10, 1) == 9        # the new token alone


@pytest.mark.parametrize("B", [1, 2, 4, 16])
def test_skipped_blocks_brute_force(B):
    for L in range(0, 70):
        for W in range(0, 75):
            lo = oracle.window_start(L, W)
            # leading blocks every token of which lies before the window
            want = 0
            while (want + 1) * B <= lo:
                want += 1
            assert oracle.skipped_blocks(L, W, B) == want, (L, W, B)


def test_window_of_one_is_the_new_value():
    cfg, inp = _inputs()
    out = _run(inp, cfg, 1)
    vc = oracle.upcast(_np(inp.value_cache), cfg.dtype)
    g = cfg.num_q_heads // cfg.num_kv_heads
    for s, L in enumerate(inp.seq_lens.tolist()):
        blk = int(inp.block_tables[s, (L - 1) // cfg.block_size])
        for h in range(cfg.num_q_heads):
            assert np.array_equal(out[s, h], vc[blk, h // g, (L - 1) % cfg.block_size])


def test_window_covering_the_sequence_is_plain_decode():
    cfg, inp = _inputs(dtype="bf16", B=8)
    full = _run(inp, cfg, 0)
    assert np.array_equal(_run(inp, cfg, 40), full)
    assert np.array_equal(_run(inp, cfg, 10_000), full)
    assert not np.array_equal(_run(inp, cfg, 39), full)   # drops token 0 of the last seq


def test_equal_keys_give_mean_of_last_w_values():
    cfg, inp = _inputs(lens=(23,), hq=2, hkv=1)
    kc = _np(inp.key_cache).copy()
    kc[:] = kc[int(inp.block_tables[0, 0]), 0, 0]          # one key everywhere
    vc64 = oracle.upcast(_np(inp.value_cache), "f32")
    for W in (1, 2, 5, 7, 22, 23):
        out = oracle.decode_attention(_np(inp.q), kc, _np(inp.value_cache),
                                      inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                      inp.scale, 1, cfg.block_size, "f32", window=W)
        rows = [vc64[int(inp.block_tables[0, j // 4]), 0, j % 4] for j in range(23 - W, 23)]
        want = np.mean(rows, axis=0)
        assert np.allclose(out[0, 0], want, atol=1e-14, rtol=0), W


@pytest.mark.parametrize("dtype,B,W", [("f32", 4, 3), ("f16", 8, 9), ("bf16", 16, 16),
                                       ("bf16", 2, 30)])
def test_window_matches_masked_sdpa(dtype, B, W):
    cfg, inp = _inputs(dtype=dtype, B=B)
    got = _run(inp, cfg, W)
    kc = oracle.upcast(_np(inp.key_cache), dtype)
    vc = oracle.upcast(_np(inp.value_cache), dtype)
    q = oracle.upcast(_np(inp.q), dtype)
    g = cfg.num_q_heads // cfg.num_kv_heads
    for s, L in enumerate(inp.seq_lens.tolist()):
        n = -(-L // B)
        row = inp.block_tables[s, :n].tolist()
        for kvh in range(cfg.num_kv_heads):
            K = np.concatenate([kc[b, kvh] for b in row], 0)[:L]
            V = np.concatenate([vc[b, kvh] for b in row], 0)[:L]
            mask = torch.arange(L) >= L - W                    # the last W tokens
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[s, kvh * g:(kvh + 1) * g])[None],
                torch.from_numpy(K)[None], torch.from_numpy(V)[None],
                attn_mask=mask[None, None, :], scale=inp.scale)
            assert np.allclose(got[s, kvh * g:(kvh + 1) * g], o[0].numpy(), atol=1e-12, rtol=0)


def test_skipped_table_entries_are_never_read():
    cfg, inp = _inputs(dtype="f16", B=4, lens=(3, 12, 13, 40))
    W = 6
    want = _run(inp, cfg, W)
    tab = inp.block_tables.numpy().copy()
    for s, L in enumerate(inp.seq_lens.tolist()):
        tab[s, :oracle.skipped_blocks(L, W, 4)] = -1
    assert (tab == -1).sum() > 0
    assert np.array_equal(_run(inp, cfg, W, tab), want)


def test_fp8_window_matches_masked_sdpa():
    gen = torch.Generator().manual_seed(4)
    S, Hkv, g, D, B, NB = 3, 2, 4, 128, 8, 40
    kc = (torch.randn(NB, Hkv, B, D, generator=gen) * 40).clamp(-448, 448)
    kc = kc.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vc = (torch.randn(NB, Hkv, B, D, generator=gen) * 40).clamp(-448, 448)
    vc = vc.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    q = torch.randn(S, Hkv * g, D, generator=gen).numpy()
    lens = np.array([7, 33, 80], dtype=np.int32)
    tab = np.random.default_rng(0).permutation(NB)[:30].reshape(3, 10).astype(np.int32)
    ks, vs, W = 1 / 40, 1 / 50, 21
    got = oracle.decode_attention_fp8(q, kc, vc, tab, lens, 0.088, Hkv, B, "f32", ks, vs,
                                      window=W)
    for s, L in enumerate(lens.tolist()):
        for kvh in range(Hkv):
            j = np.arange(L)
            K = oracle.e4m3_decode(kc[tab[s, j // B], kvh, j % B]) * np.float64(np.float32(ks))
            V = oracle.e4m3_decode(vc[tab[s, j // B], kvh, j % B]) * np.float64(np.float32(vs))
            mask = torch.arange(L) >= L - W
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[s, kvh * g:(kvh + 1) * g].astype(np.float64))[None],
                torch.from_numpy(K)[None], torch.from_numpy(V)[None],
                attn_mask=mask[None, None, :], scale=0.088)
            assert np.allclose(got[s, kvh * g:(kvh + 1) * g], o[0].numpy(), atol=1e-12, rtol=0)


def test_manager_releases_only_blocks_wholly_before_the_window():
    # B = 4, one sequence of 10 tokens in blocks 5, 2, 7 (free order fixed so
    # the ids are known). Window 7 starts at token 3 (block 0 still holds an
    # attended token): nothing goes. Window 6 starts at token 4: block 0 (id
    # 5) goes to the tail of the free queue and its entry is cleared. Window
    # 1 starts at token 9: block 1 (id 2) goes too, block 2 stays.
    m = oracle.OracleBlockManager(8, 4, free_order=[5, 2, 7, 0, 1, 3, 4, 6])
    assert m.allocate("a", 10) == [5, 2, 7]
    assert m.remove_skipped("a", 7) == []
    assert m.remove_skipped("a", 6) == [5]
    assert m.tables["a"] == [None, 2, 7] and m.ref[5] == 0 and list(m.free)[-1] == 5
    assert m.remove_skipped("a", 1) == [2]
    assert m.tables["a"] == [None, None, 7] and list(m.free)[-2:] == [5, 2]
    assert m.remove_skipped("a", 1) == []                 # already released
    # a block another sequence still references loses one reference only
    m2 = oracle.OracleBlockManager(8, 4)
    m2.allocate("p", 9)                                   # blocks 0, 1, 2
    m2.fork("p", "c")
    free_before = list(m2.free)
    assert m2.remove_skipped("c", 1) == [0, 1]
    assert m2.ref[:3] == [1, 1, 2] and list(m2.free) == free_before
    assert m2.tables["p"] == [0, 1, 2] and m2.tables["c"] == [None, None, 2]
    m2.free_seq("p")
    assert list(m2.free)[-2:] == [0, 1] and m2.ref[:3] == [0, 0, 1]

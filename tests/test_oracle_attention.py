"""Pins for the oracle's attention: special cases with closed forms, a pure
Python brute force, an independent library routine (torch's fp64
scaled_dot_product_attention on a block-concatenation gather), exact
invariance under relabelling of physical blocks, and exact dtype widening."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_123_gb300 import workloads


def _np(t):
    """Storage-typed numpy view of a CPU tensor (bf16 as uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _block_concat(cache64, table_row, L, kvh):
    """Independent gather: concatenate whole physical blocks in table order,
    then keep the first L rows."""
    B = cache64.shape[2]
    n = -(-L // B)
    return np.concatenate([cache64[int(b), kvh] for b in table_row[:n]], 0)[:L]


def test_bf16_upcast_is_exact():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000], dtype=np.uint16)
    got = oracle.upcast(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0078125


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(0)
    q = rng.standard_normal(64)
    K = rng.standard_normal((1, 64))
    V = rng.standard_normal((1, 64))
    assert np.array_equal(oracle.decode_attention_one(q, K, V, 0.125), V[0])


def test_equal_keys_give_the_mean_value():
    rng = np.random.default_rng(1)
    k = rng.standard_normal(32)
    K = np.tile(k, (37, 1))
    V = rng.standard_normal((37, 32))
    o = oracle.decode_attention_one(rng.standard_normal(32), K, V, 0.3)
    assert np.allclose(o, V.mean(0), atol=1e-14, rtol=0)


def test_dominant_logit_selects_its_value_without_overflow():
    rng = np.random.default_rng(2)
    D = 16
    K = rng.standard_normal((9, D))
    q = 1e4 * K[5] / np.linalg.norm(K[5])       # logit ~1e4 >> others
    K[5] *= 10.0
    V = rng.standard_normal((9, D))
    o = oracle.decode_attention_one(q, K, V, 1.0)
    assert np.all(np.isfinite(o))
    assert np.allclose(o, V[5], atol=1e-12, rtol=0)


def test_empty_context_gives_zeros():
    o = oracle.decode_attention_one(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert np.array_equal(o, np.zeros(8))


@pytest.mark.parametrize("L,D", [(1, 4), (3, 5), (7, 8)])
def test_pure_python_brute_force(L, D):
    rng = np.random.default_rng(L * 10 + D)
    q = rng.standard_normal(D)
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    scale = 1 / math.sqrt(D)
    want = _brute_force(q.tolist(), K.tolist(), V.tolist(), scale)
    got = oracle.decode_attention_one(q, K, V, scale)
    assert np.allclose(got, want, atol=1e-13, rtol=0)


def _brute_force(q_vec, K_rows, V_rows, scale):
    """Pure-Python loops with math.exp (brute force on tiny inputs)."""
    xs = [scale * sum(a * b for a, b in zip(q_vec, k)) for k in K_rows]
    m = max(xs)
    ps = [math.exp(x - m) for x in xs]
    den = sum(ps)
    return [sum(p * v[d] for p, v in zip(ps, V_rows)) / den
            for d in range(len(V_rows[0]))]


def _sdpa_reference(inp, seqs=None):
    """torch fp64 SDPA per (sequence, KV head) on the block-concatenation
    gather, query heads of a group stacked as separate queries."""
    cfg = inp.cfg
    g = cfg.num_q_heads // cfg.num_kv_heads
    dt = cfg.dtype
    kc64 = oracle.upcast(_np(inp.key_cache), dt)
    vc64 = oracle.upcast(_np(inp.value_cache), dt)
    q64 = oracle.upcast(_np(inp.q), dt)
    S = cfg.num_seqs
    out = np.zeros((S, cfg.num_q_heads, cfg.head_size))
    for s in (range(S) if seqs is None else seqs):
        L = int(inp.seq_lens[s])
        row = inp.block_tables[s].numpy()
        for kvh in range(cfg.num_kv_heads):
            K = torch.from_numpy(_block_concat(kc64, row, L, kvh))[None]
            V = torch.from_numpy(_block_concat(vc64, row, L, kvh))[None]
            Q = torch.from_numpy(q64[s, kvh * g:(kvh + 1) * g])[None]
            o = torch.nn.functional.scaled_dot_product_attention(
                Q, K, V, scale=inp.scale)
            out[s, kvh * g:(kvh + 1) * g] = o[0].numpy()
    return out


@pytest.mark.parametrize("name,dtype,hq,hkv,B", [
    ("tiny", "f32", 4, 4, 4),
    ("gqa_small", "bf16", 8, 2, 8),
    ("fp16_small", "f16", 4, 1, 16),
])
def test_oracle_matches_sdpa_fp64(name, dtype, hq, hkv, B):
    if name == "tiny":
        cfg = workloads.CONFIGS["tiny"]
    else:
        cfg = workloads.DecodeConfig(name, 3, hq, hkv, 64, B, dtype,
                                     ctx_lo=1, ctx_hi=50, seed=5)
    inp = workloads.make_decode_inputs(cfg)
    got = oracle.decode_attention(_np(inp.q), _np(inp.key_cache), _np(inp.value_cache),
                                  inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                  inp.scale, cfg.num_kv_heads, cfg.block_size, cfg.dtype)
    want = _sdpa_reference(inp)
    assert np.allclose(got, want, atol=1e-12, rtol=0)


def test_oracle_is_invariant_under_block_relabelling():
    cfg = workloads.DecodeConfig("perm", 4, 4, 2, 64, 4, "f16", ctx_lo=1,
                                 ctx_hi=40, seed=11)
    inp = workloads.make_decode_inputs(cfg)
    args = dict(scale=inp.scale, num_kv_heads=2, block_size=4, dtype="f16")
    a = oracle.decode_attention(_np(inp.q), _np(inp.key_cache), _np(inp.value_cache),
                                inp.block_tables.numpy(), inp.seq_lens.numpy(), **args)
    perm = np.random.default_rng(3).permutation(inp.num_blocks)
    kc = np.empty_like(_np(inp.key_cache))
    vc = np.empty_like(kc)
    kc[perm] = _np(inp.key_cache)
    vc[perm] = _np(inp.value_cache)
    tab = inp.block_tables.numpy().copy()
    tab[tab >= 0] = perm[tab[tab >= 0]]
    b = oracle.decode_attention(_np(inp.q), kc, vc, tab, inp.seq_lens.numpy(), **args)
    assert np.array_equal(a, b)


def test_decode_step_attends_to_the_new_token():
    """After the step, the new token is part of the attended context: with a
    query pointing hard at the new key, the output is the new value."""
    cfg = workloads.CONFIGS["tiny"]
    inp = workloads.make_decode_inputs(cfg)
    q = _np(inp.q).copy()
    kn = _np(inp.k_new)
    q[:, :, :] = 1e3 * kn[:, :, :] / np.linalg.norm(kn, axis=-1, keepdims=True)
    kc, vc = _np(inp.key_cache).copy(), _np(inp.value_cache).copy()
    slots, out = oracle.decode_step(q, kn, _np(inp.v_new), kc, vc,
                                    inp.block_tables.numpy(), inp.context_lens.numpy(),
                                    1.0, cfg.num_kv_heads, cfg.block_size, "f32")
    # context 7 -> token at position 7 lands in logical block 1, row 3
    assert slots[0] % 4 == 3 and slots[0] // 4 == inp.block_tables[0, 1]
    assert np.allclose(out, oracle.upcast(_np(inp.v_new), "f32"), atol=1e-9)


def test_gqa_query_head_reads_its_group_kv_head():
    """Each KV head gets a distinct constant value row; query head h must
    return the value of KV head h // g (equal keys -> mean of values)."""
    S, Hq, Hkv, D, B = 1, 8, 2, 8, 4
    g = Hq // Hkv
    kc = np.zeros((2, Hkv, B, D), np.float32)
    vc = np.zeros((2, Hkv, B, D), np.float32)
    for h in range(Hkv):
        vc[:, h] = h + 1.0
    q = np.random.default_rng(0).standard_normal((S, Hq, D)).astype(np.float32)
    out = oracle.decode_attention(q, kc, vc, np.array([[1, 0]]), np.array([6]),
                                  1.0, Hkv, B, "f32")
    for h in range(Hq):
        assert np.all(out[0, h] == h // g + 1.0)


def _mq_inputs(dtype, n_new, ctx, hq, hkv, B, seed):
    cfg = workloads.DecodeConfig("mq", len(ctx), hq, hkv, 64, B, dtype, seed=seed)
    lens = [c + n for c, n in zip(ctx, n_new)]
    inp = workloads.make_decode_inputs(cfg, context_lens=[L - 1 for L in lens])
    qsl = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int64)
    gen = torch.Generator().manual_seed(seed + 1)
    q = torch.empty(int(qsl[-1]), hq, 64, dtype=workloads.DTYPES[dtype])
    workloads.randn_into(q, gen)
    return inp, q, qsl, np.array(lens)


def test_multi_query_with_one_new_token_is_decode():
    inp, q, qsl, lens = _mq_inputs("bf16", [1, 1, 1], [5, 17, 40], 8, 2, 8, 3)
    a = oracle.multi_query_attention(_np(q), _np(inp.key_cache), _np(inp.value_cache),
                                     inp.block_tables.numpy(), qsl, lens, 0.125, 2, 8, "bf16")
    b = oracle.decode_attention(_np(q), _np(inp.key_cache), _np(inp.value_cache),
                                inp.block_tables.numpy(), lens, 0.125, 2, 8, "bf16")
    assert np.array_equal(a, b)


def test_multi_query_matches_sdpa_with_causal_offset_mask():
    n_new, ctx = [3, 0, 6, 1], [4, 9, 0, 30]
    inp, q, qsl, lens = _mq_inputs("f16", n_new, ctx, 8, 2, 4, 9)
    got = oracle.multi_query_attention(_np(q), _np(inp.key_cache), _np(inp.value_cache),
                                       inp.block_tables.numpy(), qsl, lens, 0.2, 2, 4, "f16")
    kc64 = oracle.upcast(_np(inp.key_cache), "f16")
    vc64 = oracle.upcast(_np(inp.value_cache), "f16")
    q64 = oracle.upcast(_np(q), "f16")
    for s, (n, L) in enumerate(zip(n_new, lens)):
        if n == 0:
            continue
        row = inp.block_tables[s].numpy()
        # query i may see key j iff j <= L - n + i
        mask = torch.from_numpy(np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None])
        for kvh in range(2):
            K = torch.from_numpy(_block_concat(kc64, row, L, kvh))
            V = torch.from_numpy(_block_concat(vc64, row, L, kvh))
            for h in range(kvh * 4, kvh * 4 + 4):
                Q = torch.from_numpy(q64[qsl[s]:qsl[s] + n, h])
                o = torch.nn.functional.scaled_dot_product_attention(
                    Q[None], K[None], V[None], attn_mask=mask[None], scale=0.2)[0]
                assert np.allclose(got[qsl[s]:qsl[s] + n, h], o.numpy(), atol=1e-12, rtol=0)

"""Full-size steps in the launch configurations bench.py times, not covered
by the other full-size tests: 2, 4 and 8 speculative tokens per sequence of
the GQA-72B batch (the multi-query kernels with automatic partitioning), the
GQA-72B, Llama-7B and long-context steps over fp8 blocks that carry their
own scales (the scale-fixing write and the scaled attention), and the
Llama-7B (group 1 on the tensor-core kernel) and long-context steps over fp8
pools with one scale per pool. The batches are built the way bench.py builds
them; every written slot, code and scale is checked in full and sampled
outputs one by one against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, bytes_equal, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("N", [2, 4, 8])
def test_speculative_tokens_gqa72b_full(N):
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs("gqa72b", device=DEV)
    cfg = inp.cfg
    S, B, Hkv, D, Hq = cfg.num_seqs, cfg.block_size, cfg.num_kv_heads, cfg.head_size, \
        cfg.num_q_heads
    gen = torch.Generator(device=DEV).manual_seed(cfg.seed + 77)
    g = {}
    for k, h in (("q", Hq), ("k_new", Hkv), ("v_new", Hkv)):
        g[k] = torch.empty((S * N, h, D), dtype=inp.q.dtype, device=DEV)
        workloads.randn_into(g[k], gen)
    qsl = torch.arange(S + 1, dtype=torch.int32, device=DEV) * N
    pos = (inp.seq_lens.to(torch.int64)[:, None] - N +
           torch.arange(N, device=DEV)[None, :]).reshape(-1).contiguous()
    kc_h, vc_h = np_(inp.key_cache), np_(inp.value_cache)
    tables = inp.block_tables
    slots = pa.pa_compute_slot_mapping(qsl, pos, tables, B)
    pa.pa_reshape_and_cache(g["k_new"], g["v_new"], slots, inp.key_cache, inp.value_cache)
    out = pa.pa_multi_query_attention(g["q"], qsl, inp.key_cache, inp.value_cache, tables,
                                      inp.seq_lens, inp.scale, Hkv, max_query_len=N,
                                      max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    slots_o = oracle.slot_mapping(qsl.cpu().numpy(), pos.cpu().numpy(), tables.cpu().numpy(), B)
    assert np.array_equal(slots.cpu().numpy(), slots_o)
    oracle.reshape_and_cache(np_(g["k_new"]), np_(g["v_new"]), slots_o, kc_h, vc_h, B)
    assert bytes_equal(inp.key_cache, kc_h) and bytes_equal(inp.value_cache, vc_h)
    q = np_(g["q"])
    lens = inp.seq_lens.cpu().numpy()
    tab = tables.cpu().numpy()
    rng = np.random.default_rng(N)
    worst = 0.0
    for s in (int(lens.argmax()), int(lens.argmin()), int(rng.integers(S))):
        for i in sorted({0, N - 1, int(rng.integers(N))}):
            t = s * N + i
            Ls = int(lens[s]) - N + i + 1          # the causal limit of new token i
            for h in (0, 9, Hq - 1):
                K = oracle.gather_kv(kc_h, tab[s], Ls, h // (Hq // Hkv), B, cfg.dtype)
                V = oracle.gather_kv(vc_h, tab[s], Ls, h // (Hq // Hkv), B, cfg.dtype)
                want = oracle.decode_attention_one(oracle.upcast(q[t, h], cfg.dtype), K, V,
                                                   inp.scale)
                worst = max(worst, float(np.abs(out[t, h].double().cpu().numpy() - want).max()))
    assert worst <= TOL[cfg.dtype], worst
    assert torch.isfinite(out.float()).all()


def _block_scaled(x):
    # bench.py's pools: the same N(0,1) draws, each (block, KV head) at the
    # power-of-two scale its write would fix had one call filled it
    amax = x.float().abs().amax(dim=(2, 3)).clamp_(min=2.0 ** -119)
    s_ = torch.exp2(torch.ceil(torch.log2(amax)) - 7)
    c_ = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    for b0 in range(0, x.shape[0], 4096):
        c_[b0:b0 + 4096] = (x[b0:b0 + 4096].float() / s_[b0:b0 + 4096, :, None, None]
                            ).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    return c_, s_.contiguous()


@pytest.mark.parametrize("name", ["gqa72b", "llama7b", "longctx_B16"])
def test_fp8_block_scales_step_full(name):
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs(name, device=DEV)
    cfg = inp.cfg
    kc, ks = _block_scaled(inp.key_cache)
    vc, vs = _block_scaled(inp.value_cache)
    del inp.key_cache, inp.value_cache
    torch.cuda.empty_cache()
    kc_h, vc_h, ks_h, vs_h = kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), \
        vs.cpu().numpy()
    slots = pa.pa_compute_slot_mapping(inp.query_start_loc, inp.positions, inp.block_tables,
                                       cfg.block_size)
    pa.pa_reshape_and_cache_fp8_scaled(inp.k_new, inp.v_new, slots, kc, vc, ks, vs)
    out = pa.pa_decode_attention_fp8_scaled(inp.q, kc, vc, ks, vs, inp.block_tables,
                                            inp.seq_lens, inp.scale, cfg.num_kv_heads,
                                            max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    slots_o = slots.cpu().numpy()
    oracle.reshape_and_cache_fp8_block_scaled(np_(inp.k_new), np_(inp.v_new), slots_o, kc_h,
                                              vc_h, ks_h, vs_h, cfg.block_size, cfg.dtype)
    assert np.array_equal(ks.cpu().numpy(), ks_h) and np.array_equal(vs.cpu().numpy(), vs_h)
    assert np.array_equal(kc.cpu().numpy(), kc_h) and np.array_equal(vc.cpu().numpy(), vc_h)
    lens = inp.seq_lens.cpu().numpy()
    seqs = sorted({int(lens.argmax()), int(lens.argmin()), 5 % cfg.num_seqs,
                   90 % cfg.num_seqs})
    heads = [0, 21 % cfg.num_q_heads, cfg.num_q_heads - 1]
    want = oracle.decode_attention_fp8_block_scaled(
        np_(inp.q), kc_h, vc_h, ks_h, vs_h, inp.block_tables.cpu().numpy(), lens, inp.scale,
        cfg.num_kv_heads, cfg.block_size, cfg.dtype, seqs=seqs, heads=heads)
    got = out.double().cpu().numpy()
    err = np.abs(got[np.ix_(seqs, heads)] - want[np.ix_(seqs, heads)]).max()
    assert err <= TOL[cfg.dtype], err
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["llama7b", "longctx_B16", "longctx_B128"])
def test_fp8_step_full(name):
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs(name, device=DEV)
    cfg = inp.cfg
    ks = vs = 1.0 / 48
    kc = (inp.key_cache.float() / ks).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (inp.value_cache.float() / vs).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    del inp.key_cache, inp.value_cache
    torch.cuda.empty_cache()
    kc_h, vc_h = kc.cpu().numpy(), vc.cpu().numpy()
    slots = pa.pa_compute_slot_mapping(inp.query_start_loc, inp.positions, inp.block_tables,
                                       cfg.block_size)
    pa.pa_reshape_and_cache_fp8(inp.k_new, inp.v_new, slots, kc, vc, ks, vs)
    out = pa.pa_decode_attention_fp8(inp.q, kc, vc, inp.block_tables, inp.seq_lens, inp.scale,
                                     cfg.num_kv_heads, ks, vs, max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    oracle.reshape_and_cache_fp8(np_(inp.k_new), np_(inp.v_new), slots.cpu().numpy(), kc_h,
                                 vc_h, cfg.block_size, cfg.dtype, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), kc_h) and np.array_equal(vc.cpu().numpy(), vc_h)
    lens = inp.seq_lens.cpu().numpy()
    seqs = sorted({int(lens.argmax()), int(lens.argmin()), 7 % cfg.num_seqs,
                   40 % cfg.num_seqs})
    heads = [0, 17 % cfg.num_q_heads, cfg.num_q_heads - 1]
    want = oracle.decode_attention_fp8(np_(inp.q), kc_h, vc_h, inp.block_tables.cpu().numpy(),
                                       lens, inp.scale, cfg.num_kv_heads, cfg.block_size,
                                       cfg.dtype, ks, vs, seqs=seqs, heads=heads)
    got = out.double().cpu().numpy()
    err = np.abs(got[np.ix_(seqs, heads)] - want[np.ix_(seqs, heads)]).max()
    assert err <= TOL[cfg.dtype], err
    assert torch.isfinite(out.float()).all()

"""Parity in the launch configurations bench.py times for the next rows: the
prefill steps (8 GQA-72B sequences x 512 new tokens, 4 long-context
sequences x 256 new tokens; automatic partitioning, tcgen05 kernel) and the
full GQA-72B decode step over fp8 pools. The batches are built the way bench.py builds them; sampled outputs
are checked one by one against the oracle, every written slot and cache
byte in full."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, bytes_equal, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name,S,N", [("gqa72b", 8, 512), ("longctx_B16", 4, 256)])
def test_prefill_step(name, S, N):
    base = workloads.CONFIGS[name]
    cfg = dataclasses.replace(base, num_seqs=S, name=f"{base.name}_s{S}",
                              ctx_fixed=None if base.ctx_fixed is None else base.ctx_fixed[:S])
    inp = workloads.make_decode_inputs(cfg, device=DEV, seed=cfg.seed)
    B, Hkv, D, Hq = cfg.block_size, cfg.num_kv_heads, cfg.head_size, cfg.num_q_heads
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
    rng = np.random.default_rng(2)
    worst = 0.0
    for s in (0, int(lens.argmax()), int(rng.integers(S))):
        for i in sorted({0, 127, 128, N // 2 + 44, N - 1}):
            t = s * N + i
            Ls = int(lens[s]) - N + i + 1
            for h in (0, 9, Hq - 1):
                K = oracle.gather_kv(kc_h, tab[s], Ls, h // (Hq // Hkv), B, cfg.dtype)
                V = oracle.gather_kv(vc_h, tab[s], Ls, h // (Hq // Hkv), B, cfg.dtype)
                want = oracle.decode_attention_one(oracle.upcast(q[t, h], cfg.dtype), K, V,
                                                   inp.scale)
                got = out[t, h].double().cpu().numpy()
                worst = max(worst, float(np.abs(got - want).max()))
    assert worst <= TOL[cfg.dtype], worst
    assert torch.isfinite(out.float()).all()


def test_fp8_decode_step_gqa72b_full():
    inp = workloads.make_decode_inputs("gqa72b", device=DEV)
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
    slots_o = slots.cpu().numpy()
    oracle.reshape_and_cache_fp8(np_(inp.k_new), np_(inp.v_new), slots_o, kc_h, vc_h,
                                 cfg.block_size, cfg.dtype, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), kc_h) and np.array_equal(vc.cpu().numpy(), vc_h)
    lens = inp.seq_lens.cpu().numpy()
    seqs = sorted({int(lens.argmax()), int(lens.argmin()), 3, 77})
    heads = [0, 13, cfg.num_q_heads - 1]
    want = oracle.decode_attention_fp8(np_(inp.q), kc_h, vc_h, inp.block_tables.cpu().numpy(),
                                       lens, inp.scale, cfg.num_kv_heads, cfg.block_size,
                                       cfg.dtype, ks, vs, seqs=seqs, heads=heads)
    got = out.double().cpu().numpy()
    err = np.abs(got[np.ix_(seqs, heads)] - want[np.ix_(seqs, heads)]).max()
    assert err <= TOL[cfg.dtype], err
    assert torch.isfinite(out.float()).all()

"""Full-size windowed workloads in the launch configuration the benchmark
times (automatic partitioning), with the table entries of the blocks wholly
before the window released to -1 as the host pool does: the even schedule
(GQA-72B batch, 1000-token window, fp8 pools with one scale per pool and
with per-block scales), the strided multi-item walk (the same window over
16-bit pools; the Llama-7B batch with a 333-token window over fp8 pools),
fixed partitions (long-context batch, 4096-token window) and the CUDA-core
kernel (the Llama-7B batch with a 333-token window over 16-bit pools). Attention is
checked element by element against the oracle on sampled (sequence, head)
pairs that it computes one by one."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"
FORMAT = {"16bit": "16bit", "fp8": "fp8", "fp8b": "fp8_block_scales"}
# (workload, window, KV format, the schedule: even CTAs > 0, or 0)
CASES = [("gqa72b", 1000, "fp8", True), ("gqa72b", 1000, "fp8b", True),
         ("gqa72b", 1000, "16bit", False), ("llama7b", 333, "fp8", False),
         ("longctx_B16", 4096, "16bit", False), ("longctx_B16", 4096, "fp8", False),
         ("llama7b", 333, "16bit", False)]


def _codes(x, scale):
    # E4M3 codes of x / scale (scale broadcast per block and KV head or per pool)
    return (x / scale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("name,W,fmt,even", CASES)
def test_full_size_window(name, W, fmt, even):
    pa.pa_get_device_error()
    inp = workloads.make_decode_inputs(name, device=DEV)
    cfg = inp.cfg
    B, Hkv, L = cfg.block_size, cfg.num_kv_heads, inp.max_seq_len
    lens = inp.seq_lens.cpu().numpy()
    tab = inp.block_tables.cpu().numpy().copy()
    for s, n in enumerate(lens.tolist()):
        tab[s, :oracle.skipped_blocks(n, W, B)] = -1
    tab_d = torch.from_numpy(tab).to(DEV)
    C = pa.pa_decode_even_ctas(cfg.num_seqs, cfg.num_q_heads, Hkv, cfg.head_size, B,
                               inp.q.dtype, FORMAT[fmt], L, W)
    assert (C > 0) == even
    rng = np.random.default_rng(1)
    seqs = sorted({int(lens.argmax()), int(lens.argmin()),
                   *rng.choice(cfg.num_seqs, size=4, replace=False).tolist()})
    heads = sorted({0, cfg.num_q_heads - 1,
                    *rng.choice(cfg.num_q_heads, size=2, replace=False).tolist()})
    q = np_(inp.q)
    gen = torch.Generator(device=DEV).manual_seed(11)
    if fmt == "16bit":
        out = pa.pa_decode_attention_window(inp.q, inp.key_cache, inp.value_cache, tab_d,
                                            inp.seq_lens, inp.scale, Hkv, W, max_seq_len=L)
        torch.cuda.synchronize()
        want = oracle.decode_attention(q, np_(inp.key_cache), np_(inp.value_cache), tab, lens,
                                       inp.scale, Hkv, B, cfg.dtype, seqs, heads, window=W)
    elif fmt == "fp8":
        ks, vs = 1 / 48, 1 / 40
        shape = inp.key_cache.shape
        kc = _codes(torch.randn(shape, generator=gen, device=DEV), ks)
        vc = _codes(torch.randn(shape, generator=gen, device=DEV), vs)
        out = pa.pa_decode_attention_fp8_window(inp.q, kc, vc, tab_d, inp.seq_lens, inp.scale,
                                                Hkv, ks, vs, W, max_seq_len=L)
        torch.cuda.synchronize()
        want = oracle.decode_attention_fp8(q, kc.cpu().numpy(), vc.cpu().numpy(), tab, lens,
                                           inp.scale, Hkv, B, cfg.dtype, ks, vs, seqs, heads,
                                           window=W)
    else:
        # values ~ N(0, 1) * 2^e with e drawn per (block, KV head): K within
        # 2^-4 .. 1, V within 2^-14 .. 1; each block's scale 2^(e - 5)
        NB, shape = inp.num_blocks, inp.key_cache.shape
        pools = []
        for lo_e in (-4, -14):
            e = torch.randint(lo_e, 1, (NB, Hkv), generator=gen, device=DEV).float()
            x = torch.randn(shape, generator=gen, device=DEV) * torch.exp2(e)[:, :, None, None]
            sc = torch.exp2(e - 5)
            pools.append((_codes(x, sc[:, :, None, None]), sc))
            del x
        (kc, ksc), (vc, vsc) = pools
        out = pa.pa_decode_attention_fp8_scaled(inp.q, kc, vc, ksc, vsc, tab_d, inp.seq_lens,
                                                inp.scale, Hkv, max_seq_len=L, window=W)
        torch.cuda.synchronize()
        want = oracle.decode_attention_fp8_block_scaled(
            q, kc.cpu().numpy(), vc.cpu().numpy(), ksc.cpu().numpy(), vsc.cpu().numpy(), tab,
            lens, inp.scale, Hkv, B, cfg.dtype, seqs, heads, window=W)
    assert pa.pa_get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    err = max_abs_err(out, want, seqs, heads)
    assert err <= TOL[cfg.dtype], err

"""fp8 (E4M3) KV pools through the C ABI: the quantising KV write must give
the oracle's codes bit for bit; decode attention over the codes must match the
oracle's fp64 attention on the dequantised values."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def fp8_pool(shape, scale, gen):
    x = torch.randn(shape, generator=gen) / scale
    return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (1 / 64, 0.037), (3.3, 0.002)])
def test_quantising_kv_write_bit_exact(dtype, k_scale, v_scale):
    cfg = workloads.DecodeConfig("q8", 30, 8, 4, 128, 16, dtype, ctx_lo=0, ctx_hi=100, seed=9)
    inp = workloads.make_decode_inputs(cfg)
    gen = torch.Generator().manual_seed(3)
    kc = fp8_pool((inp.num_blocks, 4, 16, 128), 1 / 64, gen)
    vc = fp8_pool((inp.num_blocks, 4, 16, 128), 1 / 64, gen)
    # include saturating inputs and exact zeros
    k = inp.k_new.clone()
    k[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).to(k.dtype)
    slots = oracle.slot_mapping(inp.query_start_loc.numpy(), inp.positions.numpy(),
                                inp.block_tables.numpy(), 16)
    slots[3] = -1
    ko, vo = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache_fp8(np_(k), np_(inp.v_new), slots, ko, vo, 16, dtype,
                                 k_scale, v_scale)
    kd, vd = kc.to(DEV), vc.to(DEV)
    pa.pa_reshape_and_cache_fp8(k.to(DEV), inp.v_new.to(DEV), torch.from_numpy(slots).to(DEV),
                                kd, vd, k_scale, v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), ko)
    assert np.array_equal(vd.cpu().numpy(), vo)
    assert pa.pa_get_device_error() == 0


CASES = [(dt, G, 16, 0) for dt in ("f32", "f16", "bf16") for G in (1, 2, 4, 8)]
CASES += [("bf16", 8, 1, 0), ("bf16", 8, 128, 0), ("f16", 1, 64, 192), ("bf16", 4, 16, 64),
          ("bf16", 1, 8, 0), ("f16", 1, 128, 0), ("bf16", 1, 4, 0)]


@pytest.mark.parametrize("dtype,G,B,partition", CASES)
def test_fp8_decode_matches_oracle(dtype, G, B, partition):
    Hkv = 2
    cfg = workloads.DecodeConfig("a8", 5, Hkv * G, Hkv, 128, B, dtype, seed=17 + G + B)
    inp = workloads.make_decode_inputs(cfg, context_lens=[0, 15, 63, 200, 700])
    gen = torch.Generator().manual_seed(G * 7 + B)
    ks, vs = 1 / 48, 1 / 40
    kc = fp8_pool((inp.num_blocks, Hkv, B, 128), ks, gen)
    vc = fp8_pool((inp.num_blocks, Hkv, B, 128), vs, gen)
    want = oracle.decode_attention_fp8(np_(inp.q), kc.numpy(), vc.numpy(),
                                       inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                       inp.scale, Hkv, B, dtype, ks, vs)
    out = pa.pa_decode_attention_fp8(inp.q.to(DEV), kc.to(DEV), vc.to(DEV),
                                     inp.block_tables.to(DEV), inp.seq_lens.to(DEV), inp.scale,
                                     Hkv, ks, vs, max_seq_len=inp.max_seq_len,
                                     partition_size=partition)
    torch.cuda.synchronize()
    err = max_abs_err(out, want)
    assert err <= TOL[dtype], err
    assert pa.pa_get_device_error() == 0


def test_fp8_full_step_against_oracle():
    """slot mapping, quantising write of the new token, fp8 attention that
    includes it."""
    cfg = workloads.DecodeConfig("s8", 6, 32, 8, 128, 16, "bf16", ctx_lo=1, ctx_hi=3000, seed=23)
    inp = workloads.make_decode_inputs(cfg)
    gen = torch.Generator().manual_seed(5)
    ks, vs = 1 / 50, 1 / 50
    kc = fp8_pool((inp.num_blocks, 8, 16, 128), ks, gen)
    vc = fp8_pool((inp.num_blocks, 8, 16, 128), vs, gen)
    ko, vo = kc.numpy().copy(), vc.numpy().copy()
    slots_o = oracle.slot_mapping(inp.query_start_loc.numpy(), inp.positions.numpy(),
                                  inp.block_tables.numpy(), 16)
    oracle.reshape_and_cache_fp8(np_(inp.k_new), np_(inp.v_new), slots_o, ko, vo, 16, "bf16",
                                 ks, vs)
    want = oracle.decode_attention_fp8(np_(inp.q), ko, vo, inp.block_tables.numpy(),
                                       inp.seq_lens.numpy(), inp.scale, 8, 16, "bf16", ks, vs)
    g = {k: getattr(inp, k).to(DEV) for k in ("q", "k_new", "v_new", "block_tables", "seq_lens",
                                              "positions", "query_start_loc")}
    kd, vd = kc.to(DEV), vc.to(DEV)
    slots = pa.pa_compute_slot_mapping(g["query_start_loc"], g["positions"], g["block_tables"], 16)
    pa.pa_reshape_and_cache_fp8(g["k_new"], g["v_new"], slots, kd, vd, ks, vs)
    out = pa.pa_decode_attention_fp8(g["q"], kd, vd, g["block_tables"], g["seq_lens"], inp.scale,
                                     8, ks, vs, max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(vd.cpu().numpy(), vo)
    assert max_abs_err(out, want) <= TOL["bf16"]


def test_fp8_partitioning_query():
    """Tensor-core fp8 calls take the tensor-core partition sizes for every
    group size (group 1 included), and windowed ones sized for one wave of
    three CTAs per SM, or the even schedule; pa_decode_fp8_workspace_bytes
    sizes the scratch for exactly the partitioning pa_decode_fp8_partitioning
    reports and for the even schedule of either fp8 call where it runs."""
    bf = torch.bfloat16
    # Llama-7B shape over fp8 pools: one partition per sequence
    assert pa.pa_decode_fp8_partitioning(64, 32, 32, 128, 16, bf, 2000) == (1, 2048)
    assert pa.pa_decode_partitioning(64, 32, 32, 16, 2000)[0] > 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for args in [(64, 32, 32, 128, 16), (128, 64, 8, 128, 16), (16, 32, 8, 128, 64),
                 (8, 8, 8, 64, 16), (8, 8, 8, 128, 4)]:
        S, Hq, Hkv, D, B = args
        for dt in (bf, torch.float16, torch.float32):
            for L, W in ((2049, 0), (8193, 0), (32768, 4096), (5000, 333)):
                splits, ptoks = pa.pa_decode_fp8_partitioning(S, Hq, Hkv, D, B, dt, L, W)
                covered = min(L, W + 63) if 0 < W < L else L
                assert splits == -(-covered // ptoks) and ptoks % max(64, B) == 0
                ws = pa.pa_decode_fp8_workspace_bytes(S, Hq, Hkv, D, B, dt, L, W)
                fixed = 0 if splits == 1 else (-(-S * Hq * splits * D * 4 // 256) * 256 +
                                               S * Hq * splits * 8)
                need = fixed
                for fmt, per in (("fp8", 3), ("fp8_block_scales", 3)):
                    C = pa.pa_decode_even_ctas(S, Hq, Hkv, D, B, dt, fmt, L, W)
                    if dt == torch.float32 or D != 128 or B < 8 or not 0 < W < L:
                        assert C == 0
                    assert 0 <= C <= per * sms
                    if C:      # the even schedule: partials, maxima and sums, records
                        G = Hq // Hkv
                        need = max(need, -(-C * 2 * G * D * 4 // 256) * 256 +
                                   -(-C * 2 * G * 2 * 4 // 256) * 256 + C * 8)
                assert ws == need
                if dt != torch.float32 and D == 128 and B >= 8 and 0 < W < L:
                    # windowed tensor-core fp8: as many splits as fill one
                    # wave of three CTAs per SM, never more
                    assert splits == 1 or splits * S * Hkv <= 3 * sms
    # the CUDA-core cases (fp32 queries, head size 64, blocks below 8) keep
    # the 16-bit call's partitioning
    assert pa.pa_decode_fp8_partitioning(64, 32, 32, 128, 16, torch.float32, 2049) == \
        pa.pa_decode_partitioning(64, 32, 32, 16, 2049)
    assert pa.pa_decode_fp8_partitioning(64, 32, 32, 128, 4, bf, 2049) == \
        pa.pa_decode_partitioning(64, 32, 32, 4, 2049)
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode_fp8_partitioning(64, 32, 32, 128, 16, bf, 2049, -1)


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("qmul,smul,window", [(1e6, 1.0, 0), (1e6, 1.0, 300), (1e-5, 1e5, 0),
                                              (3e30, 1e-30, 0), (1e-30, 1e30, 0)])
def test_fp8_decode_bf16_queries_over_their_whole_range(G, qmul, smul, window):
    # bf16 queries far outside fp16's range (1e6, 3e30: the products run in
    # fp16 on the tensor-core path) and far below its normal range (1e-5,
    # 1e-30), with the softmax scale adjusted so the logits stay meaningful
    # (smul) or become one-hot (1e6); windowed and not
    Hkv = 2
    cfg = workloads.DecodeConfig("r8", 5, Hkv * G, Hkv, 128, 16, "bf16", seed=31 + G)
    inp = workloads.make_decode_inputs(cfg, context_lens=[0, 15, 63, 400, 900])
    q = (inp.q.float() * qmul).to(torch.bfloat16)
    scale = inp.scale * smul
    gen = torch.Generator().manual_seed(77 + G)
    ks, vs = 1 / 48, 1 / 40
    kc = fp8_pool((inp.num_blocks, Hkv, 16, 128), ks, gen)
    vc = fp8_pool((inp.num_blocks, Hkv, 16, 128), vs, gen)
    want = oracle.decode_attention_fp8(np_(q), kc.numpy(), vc.numpy(), inp.block_tables.numpy(),
                                       inp.seq_lens.numpy(), scale, Hkv, 16, "bf16", ks, vs,
                                       window=window)
    args = (q.to(DEV), kc.to(DEV), vc.to(DEV), inp.block_tables.to(DEV), inp.seq_lens.to(DEV),
            scale, Hkv, ks, vs)
    if window:
        out = pa.pa_decode_attention_fp8_window(*args, window, max_seq_len=inp.max_seq_len)
    else:
        out = pa.pa_decode_attention_fp8(*args, max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert max_abs_err(out, want) <= TOL["bf16"]
    assert pa.pa_get_device_error() == 0

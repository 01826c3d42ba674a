"""The even schedule of the tensor-core decode kernel (windowed calls with
automatic partitioning): the batch's 64-token tiles, pair after pair, cut
into equal runs over one wave of CTAs, and the pairs cut between CTAs merged
by a second launch. Checked through the C ABI against the fp64 oracle over
16-bit pools, fp8 pools with one scale per pool and with per-block scales,
every group size, blocks smaller and larger than a tile, and the shapes that
stress the cuts: one pair spread over dozens of CTAs (its merge reads more
than 32 records), many short pairs per CTA, more CTAs than tiles, batches
with empty and invalid sequences, and a batch with no tiles at all."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _clear_device_error():
    if torch.cuda.is_available():
        pa.pa_get_device_error()
    yield


def _inputs(name, lens, Hkv, G, B, dtype, seed, max_seq_len=None):
    """Inputs with exactly these lengths, and the max_seq_len the calls
    take (at least the longest)."""
    cfg = workloads.DecodeConfig(name, len(lens), Hkv * G, Hkv, 128, B, dtype, seed=seed)
    inp = workloads.make_decode_inputs(cfg, context_lens=[max(L - 1, 0) for L in lens])
    for s, L in enumerate(lens):
        inp.seq_lens[s] = L
    msl = max(lens) if max_seq_len is None else max_seq_len
    width = -(-msl // B)               # the table must be able to hold msl tokens
    if inp.block_tables.shape[1] < width:
        pad = torch.full((len(lens), width - inp.block_tables.shape[1]), -1, dtype=torch.int32)
        inp.block_tables = torch.cat([inp.block_tables, pad], 1)
    return cfg, inp, msl


def _released(inp, window, B):
    tab = inp.block_tables.numpy().copy()
    for s, L in enumerate(inp.seq_lens.tolist()):
        tab[s, :oracle.skipped_blocks(max(L, 0), window, B)] = -1
    return tab


def _run16(inp, cfg, W, msl):
    tab = torch.from_numpy(_released(inp, W, cfg.block_size))
    return pa.pa_decode_attention_window(
        inp.q.to(DEV), inp.key_cache.to(DEV), inp.value_cache.to(DEV), tab.to(DEV),
        inp.seq_lens.to(DEV), inp.scale, cfg.num_kv_heads, W, max_seq_len=msl)


def _want16(inp, cfg, W):
    return oracle.decode_attention(np_(inp.q), np_(inp.key_cache), np_(inp.value_cache),
                                   inp.block_tables.numpy(), inp.seq_lens.numpy(), inp.scale,
                                   cfg.num_kv_heads, cfg.block_size, cfg.dtype, window=W)


def _ctas(inp, cfg, W, kv_format, msl):
    return pa.pa_decode_even_ctas(len(inp.seq_lens), cfg.num_q_heads, cfg.num_kv_heads, 128,
                                  cfg.block_size, TORCH_DT[cfg.dtype], kv_format, msl, W)


LENS = [0, 1, 40, 64, 65, 130, 999, 1000, 1001, 1063, 1100, 2500, 4000]
CASES16 = [(dt, G, B, W) for dt in ("f16", "bf16") for G in (2, 4, 8) for B, W in
           ((16, 1000), (8, 100))]
CASES16 += [("bf16", 8, 128, 1000), ("bf16", 4, 256, 333), ("f16", 2, 32, 64),
            ("bf16", 8, 64, 1)]


@pytest.mark.parametrize("dtype,G,B,W", CASES16)
def test_even_16bit_matches_oracle(dtype, G, B, W):
    cfg, inp, msl = _inputs("ev16", LENS, 2, G, B, dtype, seed=3 * G + B + W)
    assert _ctas(inp, cfg, W, "16bit", msl) > 0
    want = _want16(inp, cfg, W)
    out = _run16(inp, cfg, W, msl)
    again = _run16(inp, cfg, W, msl)
    torch.cuda.synchronize()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert torch.equal(out, again)            # same schedule, same bits
    assert pa.pa_get_device_error() == 0


def test_one_pair_over_dozens_of_ctas():
    # one sequence, one KV head: 65 tiles in the window, one per CTA; the
    # merge of its 65 pieces reads more than 32 records
    cfg, inp, msl = _inputs("ev1", [9000], 1, 8, 16, "bf16", seed=11)
    assert _ctas(inp, cfg, 4096, "16bit", msl) == 65
    out = _run16(inp, cfg, 4096, msl)
    torch.cuda.synchronize()
    assert max_abs_err(out, _want16(inp, cfg, 4096)) <= TOL["bf16"]
    assert pa.pa_get_device_error() == 0


def _short_pairs(num_seqs, seed):
    # pairs of 0..4 tiles under a 150-token window (lengths 0..199)
    gen = np.random.default_rng(seed)
    lens = gen.integers(0, 200, num_seqs).tolist()
    lens[7] = 0
    return _inputs("evm", lens, 4, 2, 16, "f16", seed=seed, max_seq_len=400)


def test_many_short_pairs_per_cta():
    # about 3.1 items per slot (4 KV heads, 2 CTAs per SM): whole items would
    # leave the busiest CTA 4 / 3.1 = 1.29 times the mean work, so the even
    # schedule runs, each CTA walking several short pairs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cfg, inp, msl = _short_pairs(-(-31 * 2 * sms // 40), 12)
    assert _ctas(inp, cfg, 150, "16bit", msl) == 2 * sms
    out = _run16(inp, cfg, 150, msl)
    torch.cuda.synchronize()
    assert max_abs_err(out, _want16(inp, cfg, 150)) <= TOL["f16"]
    assert pa.pa_get_device_error() == 0


def test_strided_items_when_they_divide_evenly():
    # 2,400 items for 2 x SMs slots: whole items per CTA are nearly balanced,
    # so the call keeps the strided walk over its partitions (no merge launch)
    cfg, inp, msl = _short_pairs(600, 13)
    assert _ctas(inp, cfg, 150, "16bit", msl) == 0
    out = _run16(inp, cfg, 150, msl)
    torch.cuda.synchronize()
    assert max_abs_err(out, _want16(inp, cfg, 150)) <= TOL["f16"]
    assert pa.pa_get_device_error() == 0


def test_no_tiles_at_all_gives_zeros():
    cfg, inp, msl = _inputs("ev0", [0, 0, 0], 2, 4, 16, "bf16", seed=13, max_seq_len=500)
    assert _ctas(inp, cfg, 100, "16bit", msl) > 0
    out = _run16(inp, cfg, 100, msl)
    torch.cuda.synchronize()
    assert torch.equal(out.float().cpu(), torch.zeros(out.shape))
    assert pa.pa_get_device_error() == 0


def test_invalid_length_is_reported_and_the_rest_is_right():
    # sequence 2 claims more tokens than max_seq_len: it has no tiles, its
    # outputs are zeros and PA_ERR_OUT_OF_RANGE is latched; the others are
    # unaffected
    lens = [300, 1200, 900, 50, 2000]
    cfg, inp, msl = _inputs("evbad", lens, 2, 8, 16, "bf16", seed=14)
    want = _want16(inp, cfg, 500)
    inp.seq_lens[2] = msl + 5
    out = _run16(inp, cfg, 500, msl)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == -5
    assert torch.equal(out[2].float().cpu(), torch.zeros(out[2].shape))
    keep = [0, 1, 3, 4]
    assert max_abs_err(out, want, seqs=keep) <= TOL["bf16"]


def _fp8_pool(shape, scale, gen):
    x = torch.randn(shape, generator=gen) / scale
    return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("dtype,G,B,W", [("bf16", 1, 16, 1000), ("f16", 2, 16, 100),
                                         ("bf16", 4, 8, 333), ("bf16", 8, 16, 1000),
                                         ("f16", 8, 128, 64)])
def test_even_fp8_matches_oracle(dtype, G, B, W):
    Hkv = 2
    cfg, inp, msl = _inputs("ev8", LENS, Hkv, G, B, dtype, seed=5 * G + B + W)
    assert _ctas(inp, cfg, W, "fp8", msl) > 0
    gen = torch.Generator().manual_seed(G + B)
    ks, vs = 1 / 48, 1 / 40
    kc = _fp8_pool((inp.num_blocks, Hkv, B, 128), ks, gen)
    vc = _fp8_pool((inp.num_blocks, Hkv, B, 128), vs, gen)
    want = oracle.decode_attention_fp8(np_(inp.q), kc.numpy(), vc.numpy(),
                                       inp.block_tables.numpy(), inp.seq_lens.numpy(),
                                       inp.scale, Hkv, B, dtype, ks, vs, window=W)
    tab = torch.from_numpy(_released(inp, W, B))
    out = pa.pa_decode_attention_fp8_window(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), tab.to(DEV),
                                            inp.seq_lens.to(DEV), inp.scale, Hkv, ks, vs, W,
                                            max_seq_len=msl)
    torch.cuda.synchronize()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype,G,B,W", [("bf16", 8, 16, 1000), ("f16", 1, 16, 300),
                                         ("bf16", 4, 64, 100)])
def test_even_fp8_block_scales_match_oracle(dtype, G, B, W):
    Hkv = 2
    cfg, inp, msl = _inputs("ev8b", LENS, Hkv, G, B, dtype, seed=7 * G + B + W)
    assert _ctas(inp, cfg, W, "fp8_block_scales", msl) > 0
    gen = torch.Generator().manual_seed(3 * G + B)
    NB = inp.num_blocks
    ek = torch.randint(-4, 1, (NB, Hkv), generator=gen).float()
    ev = torch.randint(-14, 1, (NB, Hkv), generator=gen).float()
    pools = []
    for e in (ek, ev):
        x = torch.randn(NB, Hkv, B, 128, generator=gen) * torch.exp2(e)[:, :, None, None]
        s = torch.exp2(e - 5)
        c = (x / s[:, :, None, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
        pools.append((c.view(torch.uint8), s))
    (kc, ks), (vc, vs) = pools
    want = oracle.decode_attention_fp8_block_scaled(np_(inp.q), kc.numpy(), vc.numpy(),
                                                    ks.numpy(), vs.numpy(),
                                                    inp.block_tables.numpy(),
                                                    inp.seq_lens.numpy(), inp.scale, Hkv, B,
                                                    dtype, window=W)
    out = pa.pa_decode_attention_fp8_scaled(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), ks.to(DEV),
                                            vs.to(DEV), inp.block_tables.to(DEV),
                                            inp.seq_lens.to(DEV), inp.scale, Hkv,
                                            max_seq_len=msl, window=W)
    torch.cuda.synchronize()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert pa.pa_get_device_error() == 0


def _even_bytes(C, G, D):
    return -(-C * 2 * G * D * 4 // 256) * 256 + -(-C * 2 * G * 2 * 4 // 256) * 256 + C * 8


def test_even_schedule_choice_and_sizes():
    """The even schedule runs when whole items would leave the busiest CTA
    more than 1.25 times the mean work, over one wave (2 CTAs per SM for
    16-bit pools, 3 for fp8 pools, never more CTAs than tiles at the longest
    window); the workspace queries cover it."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bf = torch.bfloat16
    for fmt, per in (("16bit", 2), ("fp8", 3), ("fp8_block_scales", 3)):
        # one long pair: its 65 tiles over 65 CTAs
        assert pa.pa_decode_even_ctas(1, 8, 1, 128, 16, bf, fmt, 9000, 4096) == 65
        assert pa.pa_decode_even_ctas(128, 64, 8, 128, 16, bf, fmt, 4096, 0) == 0
        assert pa.pa_decode_even_ctas(128, 64, 8, 128, 16, bf, fmt, 4096, 1000, 256) == 0
        # pairs for 1.1 / 2.2 waves of whole items: imbalance 1.8 / 1.36
        for waves in (1.1, 2.2):
            S = int(waves * per * sms / 8)
            items = S * 8
            busiest = -(-items // (per * sms)) * per * sms / items
            assert busiest > 1.25
            assert pa.pa_decode_even_ctas(S, 64, 8, 128, 16, bf, fmt, 4096, 1000) == per * sms
        # exactly 4 waves of whole items: balanced, no even schedule
        assert pa.pa_decode_even_ctas(per * sms // 2, 64, 8, 128, 16, bf, fmt, 4096, 1000) == 0
    S = int(2.2 * 2 * sms / 8)
    assert pa.pa_decode_window_workspace_bytes(S, 64, 8, 128, 16, 4096, 1000) >= \
        _even_bytes(2 * sms, 8, 128)
    S = int(2.2 * 3 * sms / 8)
    assert pa.pa_decode_fp8_workspace_bytes(S, 64, 8, 128, 16, bf, 4096, 1000) >= \
        _even_bytes(3 * sms, 8, 128)

"""fp8 blocks that carry their own scales, through the C ABI: the scale-fixing
KV write must give the oracle's codes and scales bit for bit (decode steps,
ragged prefill chunks whose runs fill whole blocks, PAD and out-of-pool
slots); decode attention must match the oracle's fp64 attention on the
dequantised values on both kernels (tensor-core and CUDA-core), with and
without a window and split partitions; a block's scales travel with it
through pa_copy_blocks; a whole step (slot mapping, write, attention)
matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clear_device_error():
    if torch.cuda.is_available():
        pa.pa_get_device_error()
    yield


def _codes(shape, gen):
    c = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38          # no NaN codes
    return c


def _pow2_scales(shape, gen, lo=-12, hi=-4):
    e = torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)
    return torch.exp2(e)


def _scaled_pool(NB, Hkv, B, D, gen, elo, ehi):
    """Codes and power-of-two scales for values ~ N(0, 1) * 2^e, e drawn per
    (block, head) in [elo, ehi]: blocks of very different magnitude."""
    e = torch.randint(elo, ehi + 1, (NB, Hkv), generator=gen).float()
    x = torch.randn(NB, Hkv, B, D, generator=gen) * torch.exp2(e)[:, :, None, None]
    s = torch.exp2(e - 5)
    c = (x / s[:, :, None, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    return c, s


def _store(x, dtype):
    return x.to({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype])


def _check_write(k, v, slots, NB, Hkv, B, D, dtype, gen):
    kc = _codes((NB, Hkv, B, D), gen)
    vc = _codes((NB, Hkv, B, D), gen)
    ks = _pow2_scales((NB, Hkv), gen)
    vs = _pow2_scales((NB, Hkv), gen)
    ko, vo, kso, vso = kc.numpy().copy(), vc.numpy().copy(), ks.numpy().copy(), vs.numpy().copy()
    oracle.reshape_and_cache_fp8_block_scaled(np_(k), np_(v), slots, ko, vo, kso, vso, B, dtype)
    kd, vd, ksd, vsd = kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV)
    pa.pa_reshape_and_cache_fp8_scaled(k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV),
                                       kd, vd, ksd, vsd)
    torch.cuda.synchronize()
    assert np.array_equal(ksd.cpu().numpy(), kso) and np.array_equal(vsd.cpu().numpy(), vso)
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(vd.cpu().numpy(), vo)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_scaled_write_decode_step_bit_exact(dtype, B):
    # one new token per sequence; about 1/B of them start a block
    gen = torch.Generator().manual_seed(50 + B)
    cfg = workloads.DecodeConfig("ws", 64, 8, 4, 128, B, dtype, ctx_lo=0, ctx_hi=300, seed=B)
    inp = workloads.make_decode_inputs(cfg)
    k = _store(torch.randn(64, 4, 128, generator=gen) * 3, dtype)
    v = _store(torch.randn(64, 4, 128, generator=gen) * 0.01, dtype)
    k[5, 1, :8] = _store(torch.tensor([1e4, -1e4, 0.0, -0.0, 3e-7, 1.0, 2.0, 0.5]), dtype)
    slots = oracle.slot_mapping(inp.query_start_loc.numpy(), inp.positions.numpy(),
                                inp.block_tables.numpy(), B)
    slots[::9] = -1
    _check_write(k, v, slots, inp.num_blocks, 4, B, 128, dtype, gen)
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("dtype,B,D", [("bf16", 16, 128), ("f16", 8, 64), ("f32", 4, 16),
                                       ("bf16", 64, 128), ("bf16", 3, 32)])
def test_scaled_write_prefill_chunks_bit_exact(dtype, B, D):
    # ragged multi-token requests: runs that fill whole blocks, runs that
    # start mid-block (no scale fixed), runs cut by the end of a request
    gen = torch.Generator().manual_seed(70 + B)
    NB = 4096
    qsl, pos, table = workloads.make_random_prefill_batch(
        num_reqs=23, max_tokens_per_req=3 * B + 7, block_size=B, num_blocks=NB, seed=B)
    slots = oracle.slot_mapping(qsl.numpy(), pos.numpy(), table.numpy(), B)
    T = len(slots)
    Hkv = 2
    k = _store(torch.randn(T, Hkv, D, generator=gen) * torch.exp2(
        torch.randint(-6, 6, (T, Hkv, 1), generator=gen).float()), dtype)
    v = _store(torch.randn(T, Hkv, D, generator=gen), dtype)
    _check_write(k, v, slots, NB, Hkv, B, D, dtype, gen)
    assert pa.pa_get_device_error() == 0


def test_scaled_write_out_of_pool_slot_is_skipped_and_reported():
    gen = torch.Generator().manual_seed(3)
    NB, Hkv, B, D = 8, 2, 4, 32
    k = torch.randn(4, Hkv, D, generator=gen).to(torch.bfloat16)
    slots = np.array([4, 5, NB * B, NB * B + 4], dtype=np.int64)   # the last two are past the pool
    kc, vc = _codes((NB, Hkv, B, D), gen), _codes((NB, Hkv, B, D), gen)
    ks = _pow2_scales((NB, Hkv), gen)
    ko, vo, kso, vso = kc.numpy().copy(), vc.numpy().copy(), ks.numpy().copy(), ks.numpy().copy()
    oracle.reshape_and_cache_fp8_block_scaled(np_(k[:2]), np_(k[:2]), slots[:2], ko, vo, kso,
                                              vso, B, "bf16")
    kd, vd, ksd, vsd = kc.to(DEV), vc.to(DEV), ks.to(DEV), ks.clone().to(DEV)
    pa.pa_reshape_and_cache_fp8_scaled(k.to(DEV), k.to(DEV), torch.from_numpy(slots).to(DEV),
                                       kd, vd, ksd, vsd)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == -5
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(ksd.cpu().numpy(), kso)


CASES = [(dt, G, 16, 0, 0) for dt in ("f16", "bf16") for G in (1, 2, 4, 8)]
CASES += [("f32", 4, 16, 0, 0), ("bf16", 8, 8, 0, 0), ("bf16", 8, 128, 0, 0),
          ("f16", 1, 64, 192, 0), ("bf16", 4, 16, 64, 0), ("bf16", 2, 4, 0, 0),
          ("bf16", 8, 16, 0, 300), ("f16", 1, 16, 0, 70), ("f32", 1, 8, 128, 100)]


@pytest.mark.parametrize("dtype,G,B,partition,window", CASES)
def test_scaled_decode_matches_oracle(dtype, G, B, partition, window):
    Hkv = 2
    D = 64 if dtype == "f32" else 128
    cfg = workloads.DecodeConfig("sd", 6, Hkv * G, Hkv, D, B, dtype, seed=91 + G + B)
    inp = workloads.make_decode_inputs(cfg, context_lens=[0, 15, 63, 200, 700, 1500])
    gen = torch.Generator().manual_seed(G * 11 + B)
    # V magnitudes 2^-14 .. 2^0 apart from block to block, K 2^-4 .. 2^0
    kc, ks = _scaled_pool(inp.num_blocks, Hkv, B, D, gen, -4, 0)
    vc, vs = _scaled_pool(inp.num_blocks, Hkv, B, D, gen, -14, 0)
    want = oracle.decode_attention_fp8_block_scaled(np_(inp.q), kc.numpy(), vc.numpy(),
                                                    ks.numpy(), vs.numpy(),
                                                    inp.block_tables.numpy(),
                                                    inp.seq_lens.numpy(), inp.scale, Hkv, B,
                                                    dtype, window=window)
    out = pa.pa_decode_attention_fp8_scaled(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), ks.to(DEV),
                                            vs.to(DEV), inp.block_tables.to(DEV),
                                            inp.seq_lens.to(DEV), inp.scale, Hkv,
                                            max_seq_len=inp.max_seq_len, window=window,
                                            partition_size=partition)
    torch.cuda.synchronize()
    assert max_abs_err(out, want) <= TOL[dtype]
    assert torch.isfinite(out.float()).all()
    assert pa.pa_get_device_error() == 0


def test_scaled_decode_with_equal_scales_matches_the_per_pool_call():
    # every block at the same scale is the per-pool format: same codes, same
    # result within the tolerance
    Hkv, G, B = 8, 8, 16
    cfg = workloads.DecodeConfig("eq", 16, Hkv * G, Hkv, 128, B, "bf16", ctx_lo=100,
                                 ctx_hi=3000, seed=5)
    inp = workloads.make_decode_inputs(cfg)
    gen = torch.Generator().manual_seed(6)
    kc = (torch.randn(inp.num_blocks, Hkv, B, 128, generator=gen) * 2 ** 5).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).to(DEV)
    vc = (torch.randn(inp.num_blocks, Hkv, B, 128, generator=gen) * 2 ** 5).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).to(DEV)
    ks = torch.full((inp.num_blocks, Hkv), 2.0 ** -5, device=DEV)
    vs = torch.full((inp.num_blocks, Hkv), 2.0 ** -5, device=DEV)
    args = (inp.block_tables.to(DEV), inp.seq_lens.to(DEV), inp.scale, Hkv)
    a = pa.pa_decode_attention_fp8_scaled(inp.q.to(DEV), kc, vc, ks, vs, *args,
                                          max_seq_len=inp.max_seq_len)
    b = pa.pa_decode_attention_fp8(inp.q.to(DEV), kc, vc, *args, 2.0 ** -5, 2.0 ** -5,
                                   max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert (a.float() - b.float()).abs().max().item() <= TOL["bf16"]


def test_scaled_decode_is_bit_identical_under_block_relabelling():
    Hkv, G, B = 4, 8, 16
    cfg = workloads.DecodeConfig("rl", 8, Hkv * G, Hkv, 128, B, "bf16", ctx_lo=10,
                                 ctx_hi=2000, seed=8)
    inp = workloads.make_decode_inputs(cfg)
    gen = torch.Generator().manual_seed(9)
    NB = inp.num_blocks
    kc, ks = _scaled_pool(NB, Hkv, B, 128, gen, -4, 0)
    vc, vs = _scaled_pool(NB, Hkv, B, 128, gen, -14, 0)
    perm = torch.randperm(NB, generator=gen)           # new id of block b
    inv = torch.argsort(perm)
    tables = inp.block_tables.clone().long()
    moved_tables = torch.where(tables >= 0, perm[tables.clamp(min=0)], tables).to(torch.int32)

    def run(kc_, vc_, ks_, vs_, tab):
        return pa.pa_decode_attention_fp8_scaled(
            inp.q.to(DEV), kc_.to(DEV), vc_.to(DEV), ks_.to(DEV), vs_.to(DEV), tab.to(DEV),
            inp.seq_lens.to(DEV), inp.scale, Hkv, max_seq_len=inp.max_seq_len)

    a = run(kc, vc, ks, vs, inp.block_tables)
    b = run(kc[inv], vc[inv], ks[inv], vs[inv], moved_tables)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_copy_on_write_moves_the_scales_with_the_block():
    gen = torch.Generator().manual_seed(12)
    L, NB, Hkv, B, D = 3, 40, 2, 16, 128
    kcs = [_codes((NB, Hkv, B, D), gen).to(DEV) for _ in range(L)]
    vcs = [_codes((NB, Hkv, B, D), gen).to(DEV) for _ in range(L)]
    kss = [_pow2_scales((NB, Hkv), gen).to(DEV) for _ in range(L)]
    vss = [_pow2_scales((NB, Hkv), gen).to(DEV) for _ in range(L)]
    pairs = torch.tensor([[3, 17], [5, 30], [0, 39]], dtype=torch.int64)
    want_k = [x.cpu().numpy().copy() for x in kss]
    want_v = [x.cpu().numpy().copy() for x in vss]
    oracle.copy_blocks(want_k, want_v, pairs.numpy())
    pa.pa_copy_blocks(kcs, vcs, pairs.to(DEV), pairs)
    pa.pa_copy_blocks(kss, vss, pairs.to(DEV), pairs)    # block_bytes = Hkv * 4 = 8
    torch.cuda.synchronize()
    for layer in range(L):
        assert np.array_equal(kss[layer].cpu().numpy(), want_k[layer])
        assert np.array_equal(vss[layer].cpu().numpy(), want_v[layer])
        assert torch.equal(kcs[layer][17], kcs[layer][3])
    assert pa.pa_get_device_error() == 0


def test_scaled_full_step_against_oracle():
    """slot mapping, the scale-fixing write of the new tokens (some start a
    block), then attention that includes them."""
    Hkv, G, B = 8, 8, 16
    cfg = workloads.DecodeConfig("fs", 32, Hkv * G, Hkv, 128, B, "bf16", ctx_lo=1, ctx_hi=3000,
                                 seed=29)
    inp = workloads.make_decode_inputs(cfg)
    gen = torch.Generator().manual_seed(30)
    NB = inp.num_blocks
    kc, ks = _scaled_pool(NB, Hkv, B, 128, gen, -4, 0)
    vc, vs = _scaled_pool(NB, Hkv, B, 128, gen, -6, 0)
    ko, vo, kso, vso = kc.numpy().copy(), vc.numpy().copy(), ks.numpy().copy(), vs.numpy().copy()
    slots_o = oracle.slot_mapping(inp.query_start_loc.numpy(), inp.positions.numpy(),
                                  inp.block_tables.numpy(), B)
    oracle.reshape_and_cache_fp8_block_scaled(np_(inp.k_new), np_(inp.v_new), slots_o, ko, vo,
                                              kso, vso, B, "bf16")
    want = oracle.decode_attention_fp8_block_scaled(np_(inp.q), ko, vo, kso, vso,
                                                    inp.block_tables.numpy(),
                                                    inp.seq_lens.numpy(), inp.scale, Hkv, B,
                                                    "bf16")
    g = {n: getattr(inp, n).to(DEV) for n in ("q", "k_new", "v_new", "block_tables", "seq_lens",
                                              "positions", "query_start_loc")}
    kd, vd, ksd, vsd = kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV)
    slots = pa.pa_compute_slot_mapping(g["query_start_loc"], g["positions"], g["block_tables"], B)
    pa.pa_reshape_and_cache_fp8_scaled(g["k_new"], g["v_new"], slots, kd, vd, ksd, vsd)
    out = pa.pa_decode_attention_fp8_scaled(g["q"], kd, vd, ksd, vsd, g["block_tables"],
                                            g["seq_lens"], inp.scale, Hkv,
                                            max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(ksd.cpu().numpy(), kso)
    assert max_abs_err(out, want) <= TOL["bf16"]
    assert pa.pa_get_device_error() == 0

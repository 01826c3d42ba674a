"""Paged decode attention through the C ABI against the fp64 oracle, element
by element, on seeded inputs that span several tiles and ragged tails; plus
the method's invariances and degenerate cases."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import TOL, bytes_equal, max_abs_err, np_, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clear_device_error():
    if torch.cuda.is_available():
        pa.pa_get_device_error()
    yield


def run_step(inp, partition_size=0, g=None):
    """One decode step on the GPU: slot mapping, KV write, attention."""
    cfg = inp.cfg
    g = g or to_dev(inp)
    slots = pa.pa_compute_slot_mapping(g["query_start_loc"], g["positions"],
                                       g["block_tables"], cfg.block_size)
    pa.pa_reshape_and_cache(g["k_new"], g["v_new"], slots, g["key_cache"], g["value_cache"])
    out = pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                                 g["seq_lens"], inp.scale, cfg.num_kv_heads,
                                 max_seq_len=inp.max_seq_len, partition_size=partition_size)
    torch.cuda.synchronize()
    return slots, out, g


def oracle_step(inp, seqs=None, heads=None):
    cfg = inp.cfg
    kc, vc = np_(inp.key_cache), np_(inp.value_cache)
    slots, out = oracle.decode_step(np_(inp.q), np_(inp.k_new), np_(inp.v_new), kc, vc,
                                    np_(inp.block_tables), inp.context_lens.numpy(), inp.scale,
                                    cfg.num_kv_heads, cfg.block_size, cfg.dtype, seqs, heads)
    return slots, out, kc, vc


def test_tiny_config_full_step():
    inp = workloads.make_decode_inputs("tiny")
    slots_o, out_o, kc_o, vc_o = oracle_step(inp)
    slots, out, g = run_step(inp)
    assert np.array_equal(slots.cpu().numpy(), slots_o)
    assert bytes_equal(g["key_cache"], kc_o) and bytes_equal(g["value_cache"], vc_o)
    assert max_abs_err(out, out_o) <= TOL["f32"]
    assert pa.pa_get_device_error() == 0


SWEEP = []
for dtype in ("f32", "f16", "bf16"):
    for D in (64, 128):
        for G in (1, 2, 4, 8):
            SWEEP.append((dtype, D, G, 16))
for B in (1, 2, 4, 8, 32, 64, 128, 256):
    SWEEP.append(("bf16", 128, 8, B))
    SWEEP.append(("f16", 128, 1, B))


@pytest.mark.parametrize("dtype,D,G,B", SWEEP)
def test_decode_sweep(dtype, D, G, B):
    Hkv = 2
    cfg = workloads.DecodeConfig(f"sw_{dtype}_{D}_{G}_{B}", 5, Hkv * G, Hkv, D, B, dtype,
                                 ctx_lo=0, ctx_hi=700,
                                 seed=3000 + 1000 * ["f32", "f16", "bf16"].index(dtype)
                                 + 17 * D + 7 * G + B)
    # lengths include 1, a ragged tail and several 64-token tiles
    ctx = [0, 62, 63, 64 * 3 + 5, 699]
    inp = workloads.make_decode_inputs(cfg, context_lens=ctx)
    slots_o, out_o, _, _ = oracle_step(inp)
    slots, out, _ = run_step(inp)
    assert np.array_equal(slots.cpu().numpy(), slots_o)
    err = max_abs_err(out, out_o)
    assert err <= TOL[dtype], err
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("partition", [64, 128, 192, 448, 4096])
@pytest.mark.parametrize("dtype,G", [("bf16", 8), ("f16", 1), ("f32", 4)])
def test_forced_partitions(partition, dtype, G):
    """Split-K over block ranges with the log-sum-exp combine: 1, 2, 3, 7 or
    many partitions per sequence, all within tolerance of the oracle."""
    cfg = workloads.DecodeConfig("split", 4, 2 * G, 2, 128, 16, dtype, seed=77)
    inp = workloads.make_decode_inputs(cfg, context_lens=[447, 1, 130, 900])
    _, out_o, _, _ = oracle_step(inp)
    _, out, _ = run_step(inp, partition_size=partition)
    splits, ptoks = pa.pa_decode_partitioning(4, 2 * G, 2, 16, inp.max_seq_len, partition)
    assert ptoks % 64 == 0 and splits == math.ceil(inp.max_seq_len / ptoks)
    assert max_abs_err(out, out_o) <= TOL[dtype]


def test_partition_count_does_not_change_result_beyond_rounding():
    cfg = workloads.DecodeConfig("inv", 3, 16, 2, 128, 16, "bf16", seed=5)
    inp = workloads.make_decode_inputs(cfg, context_lens=[2000, 1500, 31])
    outs = []
    for p in (64, 320, 0, 4096):
        _, out, _ = run_step(inp, partition_size=p)
        outs.append(out.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2 * TOL["bf16"]


def test_output_is_bit_identical_under_block_relabelling():
    """Physical placement is invisible to the result ("Infra: PagedAttention",
    block table figure): relabel every block, rewrite the tables, and the
    output bits must not move."""
    cfg = workloads.DecodeConfig("perm", 6, 16, 2, 128, 16, "bf16", ctx_lo=100, ctx_hi=3000,
                                 seed=21)
    inp = workloads.make_decode_inputs(cfg)
    _, out_a, _ = run_step(inp, partition_size=512)
    perm = torch.randperm(inp.num_blocks, generator=torch.Generator().manual_seed(9))
    kc = torch.empty_like(inp.key_cache)
    vc = torch.empty_like(inp.value_cache)
    kc[perm] = inp.key_cache
    vc[perm] = inp.value_cache
    tab = inp.block_tables.clone()
    m = tab >= 0
    tab[m] = perm[tab[m].long()].to(torch.int32)
    inp.key_cache, inp.value_cache, inp.block_tables = kc, vc, tab
    _, out_b, _ = run_step(inp, partition_size=512)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_single_token_returns_its_value_exactly():
    for dtype in ("f32", "f16", "bf16"):
        cfg = workloads.DecodeConfig("one", 3, 8, 2, 128, 16, dtype, seed=2)
        inp = workloads.make_decode_inputs(cfg, context_lens=[0, 0, 0])
        _, out, _ = run_step(inp)
        want = inp.v_new.repeat_interleave(4, dim=1)
        assert torch.equal(out.cpu(), want), dtype


def test_zero_length_gives_zeros_and_bad_length_latches_error():
    cfg = workloads.DecodeConfig("z", 3, 4, 4, 64, 4, "f16", seed=3)
    inp = workloads.make_decode_inputs(cfg, context_lens=[5, 5, 5])
    g = to_dev(inp)
    g["seq_lens"] = torch.tensor([0, 6, 6], dtype=torch.int32, device=DEV)
    out = pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                                 g["seq_lens"], inp.scale, 4, max_seq_len=6)
    assert out[0].eq(0).all()
    assert pa.pa_get_device_error() == 0
    g["seq_lens"] = torch.tensor([6, 7, 6], dtype=torch.int32, device=DEV)  # 7 > max_seq_len
    out = pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                                 g["seq_lens"], inp.scale, 4, max_seq_len=6)
    assert out[1].eq(0).all()
    assert pa.pa_get_device_error() == -5


def test_bad_block_id_is_skipped_and_latched():
    cfg = workloads.DecodeConfig("bb", 2, 4, 4, 64, 4, "f32", seed=4)
    inp = workloads.make_decode_inputs(cfg, context_lens=[7, 7])
    g = to_dev(inp)
    g["block_tables"][1, 0] = inp.num_blocks + 5          # outside the pool
    pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                           g["seq_lens"], inp.scale, 4, max_seq_len=8)
    assert pa.pa_get_device_error() == -5


def test_workspace_too_small_is_rejected():
    cfg = workloads.DecodeConfig("ws", 2, 8, 2, 128, 16, "bf16", seed=6)
    inp = workloads.make_decode_inputs(cfg, context_lens=[3000, 100])
    g = to_dev(inp)
    need = pa.pa_decode_workspace_bytes(2, 8, 2, 128, 16, inp.max_seq_len, 256)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                               g["seq_lens"], inp.scale, 2, max_seq_len=inp.max_seq_len,
                               partition_size=256, workspace=small)
    assert e.value.status == -4


@pytest.mark.parametrize("dtype,G", [("bf16", 8), ("f16", 4), ("f16", 1), ("f32", 2)])
def test_garbage_outside_the_sequence_never_reaches_the_output(dtype, G):
    """Pool rows that belong to no token (the tail of each last block, and
    every unassigned block) hold NaN; the result must still match the oracle,
    which reads only the rows the block tables name."""
    cfg = workloads.DecodeConfig("nan", 5, 2 * G, 2, 128, 16, dtype, seed=31)
    inp = workloads.make_decode_inputs(cfg, context_lens=[0, 5, 70, 200, 333])
    nan = float("nan")
    used = torch.zeros(inp.num_blocks, 16, dtype=torch.bool)
    for s, L in enumerate(inp.seq_lens.tolist()):
        for j in range(L):
            used[int(inp.block_tables[s, j // 16]), j % 16] = True
    # the new token's row is written by the step itself, so it counts as used
    for cache in (inp.key_cache, inp.value_cache):
        c = cache.permute(0, 2, 1, 3)            # [NB, B, Hkv, D] view
        c[~used] = nan
    _, out_o, _, _ = oracle_step(inp)
    _, out, _ = run_step(inp, partition_size=64)
    assert torch.isfinite(out.float()).all()
    assert max_abs_err(out, out_o) <= TOL[dtype]


def test_tensor_core_path_edge_rows():
    """Group-of-8 bf16 (tensor-core kernel): a zero-length sequence gives
    zeros, a sequence with a block id outside the pool latches the error, and
    the other sequences are unaffected."""
    cfg = workloads.DecodeConfig("edge", 3, 16, 2, 128, 16, "bf16", seed=8)
    inp = workloads.make_decode_inputs(cfg, context_lens=[40, 40, 40])
    _, out_o, _, _ = oracle_step(inp)
    g = to_dev(inp)
    slots = pa.pa_compute_slot_mapping(g["query_start_loc"], g["positions"], g["block_tables"], 16)
    pa.pa_reshape_and_cache(g["k_new"], g["v_new"], slots, g["key_cache"], g["value_cache"])
    g["seq_lens"][0] = 0
    g["block_tables"][1, 1] = inp.num_blocks + 3
    out = pa.pa_decode_attention(g["q"], g["key_cache"], g["value_cache"], g["block_tables"],
                                 g["seq_lens"], inp.scale, 2, max_seq_len=41)
    assert pa.pa_get_device_error() == -5
    assert out[0].eq(0).all()
    assert max_abs_err(out[2:], out_o[2:]) <= TOL["bf16"]

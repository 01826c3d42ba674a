"""Slot mapping, KV write and block copy through the C ABI, bit for bit
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import workloads
from tests.helpers import bytes_equal, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clear_device_error():
    if torch.cuda.is_available():
        pa.pa_get_device_error()
    yield


@pytest.mark.parametrize("B", [1, 3, 4, 16, 64, 128])
@pytest.mark.parametrize("seed", [0, 1])
def test_slot_mapping_ragged_batches(B, seed):
    qsl, pos, table = workloads.make_random_prefill_batch(
        num_reqs=37, max_tokens_per_req=3 * B + 5, block_size=B, num_blocks=4096, seed=seed)
    want = oracle.slot_mapping(qsl.numpy(), pos.numpy(), table.numpy(), B)
    got = pa.pa_compute_slot_mapping(qsl.to(DEV), pos.to(DEV), table.to(DEV), B)
    assert np.array_equal(got.cpu().numpy(), want)
    assert pa.pa_get_device_error() == 0


def test_slot_mapping_pages_example():
    # block table [3, 0, 4], B = 4, positions 0..8 ("Infra: PagedAttention")
    table = torch.tensor([[3, 0, 4]], dtype=torch.int32, device=DEV)
    qsl = torch.tensor([0, 9], dtype=torch.int32, device=DEV)
    pos = torch.arange(9, dtype=torch.int64, device=DEV)
    got = pa.pa_compute_slot_mapping(qsl, pos, table, 4).cpu().numpy()
    assert np.array_equal(got, oracle.slot_mapping([0, 9], np.arange(9), table.cpu().numpy(), 4))
    assert got[8] == 16


def test_slot_mapping_pad_and_empty():
    table = torch.tensor([[5, 2], [0, 1]], dtype=torch.int32, device=DEV)
    qsl = torch.tensor([0, 0, 2], dtype=torch.int32, device=DEV)
    pos = torch.tensor([1, 5, 0], dtype=torch.int64, device=DEV)
    got = pa.pa_compute_slot_mapping(qsl, pos, table, 4).cpu().numpy()
    assert got.tolist() == oracle.slot_mapping([0, 0, 2], [1, 5, 0], table.cpu().numpy(), 4,
                                               num_tokens=3).tolist()
    assert pa.pa_get_device_error() == 0
    empty = pa.pa_compute_slot_mapping(qsl, pos[:0], table, 4)
    assert empty.numel() == 0


def test_slot_mapping_bad_rows_give_pad_and_latch_error():
    table = torch.tensor([[3, -1]], dtype=torch.int32, device=DEV)
    qsl = torch.tensor([0, 3], dtype=torch.int32, device=DEV)
    pos = torch.tensor([4, 8, -2], dtype=torch.int64, device=DEV)  # unassigned, past row, negative
    got = pa.pa_compute_slot_mapping(qsl, pos, table, 4).cpu().numpy()
    assert got.tolist() == [-1, -1, -1]
    assert pa.pa_get_device_error() == -5
    assert pa.pa_get_device_error() == 0   # cleared by the read


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("f16", 128), ("bf16", 128), ("bf16", 64)])
def test_reshape_and_cache_bit_exact(dtype, D):
    cfg = workloads.DecodeConfig("w", 40, 8, 4, D, 16, dtype, ctx_lo=0, ctx_hi=200, seed=3)
    inp = workloads.make_decode_inputs(cfg)
    kc_o, vc_o = np_(inp.key_cache), np_(inp.value_cache)
    slots = oracle.slot_mapping(inp.query_start_loc.numpy(), inp.positions.numpy(),
                                inp.block_tables.numpy(), 16)
    slots[::7] = -1                       # some PAD tokens are skipped
    oracle.reshape_and_cache(np_(inp.k_new), np_(inp.v_new), slots, kc_o, vc_o, 16)
    kc, vc = inp.key_cache.to(DEV), inp.value_cache.to(DEV)
    pa.pa_reshape_and_cache(inp.k_new.to(DEV), inp.v_new.to(DEV),
                            torch.from_numpy(slots).to(DEV), kc, vc)
    torch.cuda.synchronize()
    assert bytes_equal(kc, kc_o) and bytes_equal(vc, vc_o)
    assert pa.pa_get_device_error() == 0


def test_reshape_and_cache_out_of_pool_slot_is_skipped():
    kc = torch.zeros(4, 2, 4, 64, dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones(2, 2, 64, dtype=torch.float16, device=DEV)
    slots = torch.tensor([3, 16], dtype=torch.int64, device=DEV)   # 16 = 4 blocks * 4
    pa.pa_reshape_and_cache(k, k, slots, kc, vc)
    assert pa.pa_get_device_error() == -5
    assert kc[0, :, 3].eq(1).all() and kc.sum().item() == 2 * 64


@pytest.mark.parametrize("layers", [1, 3, 70])
def test_copy_blocks_bit_exact(layers):
    gen = torch.Generator().manual_seed(layers)
    NB, Hkv, B, D = 24, 4, 16, 128
    kcs = [torch.randn(NB, Hkv, B, D, generator=gen).to(torch.bfloat16) for _ in range(layers)]
    vcs = [torch.randn(NB, Hkv, B, D, generator=gen).to(torch.bfloat16) for _ in range(layers)]
    pairs = np.array([[0, 5], [7, 3], [7, 9], [11, 23]], dtype=np.int64)
    ko, vo = [np_(t) for t in kcs], [np_(t) for t in vcs]
    oracle.copy_blocks(ko, vo, pairs)
    kd, vd = [t.to(DEV) for t in kcs], [t.to(DEV) for t in vcs]
    tp = torch.from_numpy(pairs)
    pa.pa_copy_blocks(kd, vd, tp.to(DEV), tp)
    torch.cuda.synchronize()
    for a, b in zip(kd, ko):
        assert bytes_equal(a, b)
    for a, b in zip(vd, vo):
        assert bytes_equal(a, b)
    assert pa.pa_get_device_error() == 0


def test_copy_blocks_rejects_alias_before_launch():
    kc = torch.zeros(8, 1, 4, 64, dtype=torch.float16, device=DEV)
    pairs = torch.tensor([[0, 1], [1, 2]], dtype=torch.int64)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_copy_blocks([kc], [kc.clone()], pairs.to(DEV), pairs)
    assert e.value.status == -7


def test_copy_blocks_out_of_range_pair_is_skipped_on_device():
    kc = torch.arange(8 * 64, dtype=torch.float32, device=DEV).reshape(8, 1, 1, 64)
    vc = kc.clone()
    ref = kc.clone()
    pairs = torch.tensor([[0, 1], [2, 99]], dtype=torch.int64, device=DEV)
    pa.pa_copy_blocks([kc], [vc], pairs)           # no host copy: device range check
    assert pa.pa_get_device_error() == -5
    ref[1] = ref[0]
    assert torch.equal(kc, ref) and torch.equal(vc, ref)

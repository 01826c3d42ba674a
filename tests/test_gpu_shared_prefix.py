"""Shared-prefix parallel sampling: 8 samples share a 1027-token prompt (64
full blocks of 16 and a 3-token tail); the first decode step copies the shared
tail for 7 samples (block-level copy-on-write) and the 8th writes in place;
then 256 decode steps each append one token per sample. The GPU path (host
BlockPool + the C ABI) is mirrored by the oracle's own bookkeeping and
arithmetic, step by step."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_123_gb300 as pa
from paged_kv_cache_123_gb300 import BlockPool, workloads
from tests.helpers import TOL, bytes_equal, max_abs_err, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_shared_prefix_parallel_sampling():
    pa.pa_get_device_error()
    S, Hkv, D, B, P0, STEPS = 8, 32, 128, 16, 1027, 256
    NB = 256
    dt = torch.bfloat16
    gen = torch.Generator().manual_seed(1003)
    order = torch.randperm(NB, generator=gen).tolist()
    kc = torch.empty(NB, Hkv, B, D, dtype=dt)
    vc = torch.empty(NB, Hkv, B, D, dtype=dt)
    workloads.randn_into(kc, gen)
    workloads.randn_into(vc, gen)
    k_prompt = torch.empty(P0, Hkv, D, dtype=dt)
    v_prompt = torch.empty(P0, Hkv, D, dtype=dt)
    workloads.randn_into(k_prompt, gen)
    workloads.randn_into(v_prompt, gen)

    pool, orc = BlockPool(NB, B, order), oracle.OracleBlockManager(NB, B, order)
    kco, vco = np_(kc), np_(vc)
    kcd, vcd = kc.to(DEV), vc.to(DEV)
    MB = (P0 + STEPS + B - 1) // B

    # prompt written once through the shared blocks
    pool.add_sequence(0, P0)
    orc.allocate(0, P0)
    row = torch.from_numpy(pool.table_rows([0], MB))
    qsl = torch.tensor([0, P0], dtype=torch.int32)
    pos = torch.arange(P0, dtype=torch.int64)
    slots = pa.pa_compute_slot_mapping(qsl.to(DEV), pos.to(DEV), row.to(DEV), B)
    pa.pa_reshape_and_cache(k_prompt.to(DEV), v_prompt.to(DEV), slots, kcd, vcd)
    oslots = oracle.slot_mapping([0, P0], np.arange(P0), np.array([orc.tables[0]]), B)
    oracle.reshape_and_cache(np_(k_prompt), np_(v_prompt), oslots, kco, vco, B)
    for s in range(1, S):
        pool.fork(0, s)
        orc.fork(0, s)
    seqs = list(range(S))
    scale = D ** -0.5
    check_steps = {0, 1, 13, 128, STEPS - 1}
    n_copies = 0
    for step in range(STEPS):
        q = torch.empty(S, Hkv, D, dtype=dt)
        kn = torch.empty(S, Hkv, D, dtype=dt)
        vn = torch.empty(S, Hkv, D, dtype=dt)
        for t in (q, kn, vn):
            workloads.randn_into(t, gen)
        positions, pairs = pool.prepare_decode_step(seqs)
        if pairs:
            tp = torch.tensor(pairs, dtype=torch.int64)
            pa.pa_copy_blocks([kcd], [vcd], tp.to(DEV), tp)
            n_copies += len(pairs)
        tables = torch.from_numpy(pool.table_rows(seqs, MB)).to(DEV)
        slots = pa.pa_compute_slot_mapping(torch.arange(S + 1, dtype=torch.int32, device=DEV),
                                           torch.from_numpy(positions).to(DEV), tables, B)
        pa.pa_reshape_and_cache(kn.to(DEV), vn.to(DEV), slots, kcd, vcd)
        lens = torch.from_numpy(positions + 1).to(torch.int32).to(DEV)
        out = pa.pa_decode_attention(q.to(DEV), kcd, vcd, tables, lens, scale, Hkv,
                                     max_seq_len=int(positions.max()) + 1)
        # oracle mirror
        o_pairs, o_slots = [], []
        for s in seqs:
            sl, cow = orc.append_slot(s)
            o_slots.append(sl)
            if cow is not None:
                o_pairs.append(cow)
        assert [tuple(p) for p in pairs] == o_pairs
        if o_pairs:
            oracle.copy_blocks([kco], [vco], np.array(o_pairs))
        assert np.array_equal(slots.cpu().numpy(), np.array(o_slots))
        oracle.reshape_and_cache(np_(kn), np_(vn), o_slots, kco, vco, B)
        if step in check_steps:
            otab = -np.ones((S, MB), dtype=np.int64)
            for i, s in enumerate(seqs):
                otab[i, :len(orc.tables[s])] = orc.tables[s]
            want = oracle.decode_attention(np_(q), kco, vco, otab, positions + 1, scale, Hkv, B,
                                           "bf16")
            err = max_abs_err(out, want)
            assert err <= TOL["bf16"], (step, err)
    torch.cuda.synchronize()
    assert n_copies == 7
    assert bytes_equal(kcd, kco) and bytes_equal(vcd, vco)
    assert NB - pool.num_free() == 64 + 8 * 17
    assert pa.pa_get_device_error() == 0

"""The product's host block bookkeeping (paged_kv_cache_123_gb300.BlockPool)
against the oracle's (oracle.OracleBlockManager) and the pages' examples."""
import json
import os

import numpy as np
import pytest

from oracle import OracleBlockManager
from paged_kv_cache_123_gb300.block_pool import BlockPool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_fig8_copy_on_write_example():
    g = json.load(open(os.path.join(GOLDEN, "p2_fig8_cow_simulator.json")))
    head = g["free_order_head"]
    pool = BlockPool(8, g["block_size"], head + [b for b in range(8) if b not in head])
    pool.add_sequence("A", g["prompt_tokens"])
    pool.fork("A", "B")
    assert round(100 * pool.saving(), 1) == g["saving_shared_pct"]
    pos, pairs = pool.prepare_decode_step(["A", "B"])
    assert pos.tolist() == [7, 7]
    assert pairs == [tuple(g["after_first_token"]["copy"])]
    assert pool.blocks["A"] == g["after_first_token"]["A"]
    assert pool.blocks["B"] == g["after_first_token"]["B"]
    assert round(100 * pool.saving(), 1) == g["after_first_token"]["saving_pct"]
    pool.prepare_decode_step(["A", "B"])
    assert pool.blocks["A"] == g["after_second_token"]["A"]
    assert pool.blocks["B"] == g["after_second_token"]["B"]
    assert round(100 * pool.saving(), 1) == g["after_second_token"]["saving_pct"]


def test_shared_prefix_parallel_sampling_counts():
    """8 samples of a 1027-token prompt, B=16: the tail block is copied by 7
    samples at the first step and written in place by the last; after 256
    steps 64 shared + 8 x 17 private blocks are in use."""
    pool = BlockPool(1024, 16)
    pool.add_sequence(0, 1027)
    for s in range(1, 8):
        pool.fork(0, s)
    seqs = list(range(8))
    _, pairs = pool.prepare_decode_step(seqs)
    assert len(pairs) == 7
    assert len({d for _, d in pairs}) == 7 and len({s for s, _ in pairs}) == 1
    for _ in range(255):
        _, pr = pool.prepare_decode_step(seqs)
        assert pr == []
    used = 1024 - pool.num_free()
    assert used == 64 + 8 * 17
    assert all(pool.num_tokens[s] == 1027 + 256 for s in seqs)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_oracle_on_random_operation_sequences(seed):
    rng = np.random.default_rng(seed)
    B, NB = 4, 96
    order = rng.permutation(NB).tolist()
    pool = BlockPool(NB, B, order)
    orc = OracleBlockManager(NB, B, order)
    pool.add_sequence(0, 9)
    orc.allocate(0, 9)
    live, nxt = [0], 1
    for _ in range(400):
        op = rng.integers(0, 12)
        if op == 0 and len(live) < 8:
            par = live[rng.integers(len(live))]
            pool.fork(par, nxt)
            orc.fork(par, nxt)
            live.append(nxt)
            nxt += 1
        elif op == 1 and len(live) > 1:
            s = live.pop(rng.integers(len(live)))
            pool.release(s)
            orc.free_seq(s)
        elif op == 3:
            s = live[rng.integers(len(live))]
            W = int(rng.integers(1, 14))
            assert pool.release_skipped(s, W) == orc.remove_skipped(s, W)
        elif op == 2 and len(live) < 8 and pool.num_free() > 4:
            n = int(rng.integers(1, 12))
            pool.add_sequence(nxt, n)
            orc.allocate(nxt, n)
            live.append(nxt)
            nxt += 1
        else:
            k = int(rng.integers(1, len(live) + 1))
            batch = [live[i] for i in rng.permutation(len(live))[:k]]
            if pool.num_free() < len(batch):
                continue
            pos, pairs = pool.prepare_decode_step(batch)
            want_pairs = []
            for i, s in enumerate(batch):
                want_pos = orc.lens[s]
                slot, cow = orc.append_slot(s)
                assert pos[i] == want_pos
                if cow is not None:
                    want_pairs.append(cow)
            assert pairs == want_pairs
        assert pool.refcount.tolist() == orc.ref
        assert {s: pool.blocks[s] for s in live} == {
            s: [-1 if b is None else b for b in orc.tables[s]] for s in live}
        assert list(pool._free) == list(orc.free)


def test_release_skipped_frees_only_whole_blocks_before_the_window():
    pool = BlockPool(16, 4)
    pool.add_sequence("a", 10)                  # blocks 0, 1, 2 hold tokens 0..9
    pool.fork("a", "b")
    assert pool.release_skipped("a", 7) == []   # window 3..9 touches block 0
    assert pool.release_skipped("a", 6) == [0]  # window 4..9
    assert pool.blocks["a"] == [-1, 1, 2]
    assert pool.refcount[0] == 1 and 0 not in pool._free   # still held by "b"
    assert pool.release_skipped("b", 1) == [0, 1]          # window 9..9
    assert list(pool._free)[-1] == 0 and pool.refcount[1] == 1   # 1 still held by "a"
    pool.release("a")
    pool.release("b")
    assert pool.num_free() == 16 and not pool.refcount.any()

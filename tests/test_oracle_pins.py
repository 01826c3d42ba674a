"""Pins for the oracle's integer side: slot mapping, block counts, the host
block bookkeeping and copy-on-write, each checked against worked examples the
pages print (fixtures under tests/golden/, each naming its page and section)
and against brute-force properties on small inputs."""
import json
import os
from itertools import product

import numpy as np
import pytest

import oracle
from oracle import OracleBlockManager

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- slot mapping
def test_p4_block_table_example():
    g = load("p4_block_table_example.json")
    B = g["block_size"]
    table = np.array([g["block_table"]], dtype=np.int32)
    T = g["num_tokens"]
    slots = oracle.slot_mapping([0, T], np.arange(T), table, B)
    for tok, (phys, row) in g["token_to_physical"].items():
        s = int(slots[int(tok)])
        assert (s // B, s % B) == (phys, row), tok
    assert oracle.blocks_needed(T, B) == g["blocks"]
    assert oracle.slots_allocated(T, B) == g["slots"]
    assert oracle.slots_allocated(T, B) - T == g["empty_slots"]


def test_p2_seven_token_prompt_on_demand_append():
    g = load("p2_seven_token_prompt.json")
    B = g["block_size"]
    head = g["free_order_head"]
    rest = [b for b in range(8) if b not in head]
    bm = OracleBlockManager(8, B, free_order=head + rest)
    assert bm.allocate("A", g["prompt_tokens"]) == g["table_after_prompt"]
    fills = [min(B, g["prompt_tokens"] - i * B)
             for i in range(len(g["table_after_prompt"]))]
    assert fills == g["tokens_in_logical_blocks"]
    for step in ("first_decode", "second_decode"):
        want = g[step]
        slot, cow = bm.append_slot("A")
        assert cow is None
        assert (slot // B, slot % B) == (want["physical_block"], want["row"])
        assert bm.tables["A"] == want["table"]
        # the same slot from the slot-mapping formula with the new table
        tab = np.array([bm.tables["A"]], dtype=np.int32)
        assert oracle.slot_mapping([0, 1], [want["position"]], tab, B)[0] == slot


def test_p2_fig8_copy_on_write_and_savings():
    g = load("p2_fig8_cow_simulator.json")
    B = g["block_size"]
    head = g["free_order_head"]
    rest = [b for b in range(8) if b not in head]
    bm = OracleBlockManager(8, B, free_order=head + rest)
    bm.allocate("A", g["prompt_tokens"])
    bm.fork("A", "B")
    assert bm.tables["A"] == bm.tables["B"] == g["shared_table"]
    assert all(bm.ref[b] == g["shared_refcount"] for b in g["shared_table"])
    assert round(100 * oracle.sharing_saving(bm.tables.values()), 1) == g["saving_shared_pct"]
    _, cow_a = bm.append_slot("A")
    _, cow_b = bm.append_slot("B")
    s1 = g["after_first_token"]
    assert list(cow_a) == s1["copy"] and cow_b is None
    assert bm.tables["A"] == s1["A"] and bm.tables["B"] == s1["B"]
    assert round(100 * oracle.sharing_saving(bm.tables.values()), 1) == s1["saving_pct"]
    bm.append_slot("A")
    bm.append_slot("B")
    s2 = g["after_second_token"]
    assert bm.tables["A"] == s2["A"] and bm.tables["B"] == s2["B"]
    assert round(100 * oracle.sharing_saving(bm.tables.values()), 1) == s2["saving_pct"]


def test_p4_cow_figure_tables_refcounts_and_data():
    g = load("p4_cow_figure.json")
    B = g["block_size"]
    head = g["free_order_head"]
    rest = [b for b in range(8) if b not in head]
    bm = OracleBlockManager(8, B, free_order=head + rest)
    bm.allocate("A", g["prefix_tokens"])
    bm.fork("A", "B")
    assert bm.tables["A"] == g["shared_table"]
    # a one-head, width-1 pool whose row value encodes the token position
    kc = np.full((8, 1, B, 1), -1.0, dtype=np.float32)
    vc = kc.copy()
    slots = oracle.slot_mapping([0, 6], np.arange(6), np.array([bm.tables["A"]]), B)
    pos = np.arange(6, dtype=np.float32).reshape(6, 1, 1)
    oracle.reshape_and_cache(pos, pos, slots, kc, vc, B)
    sa, cow_a = bm.append_slot("A")
    sb, cow_b = bm.append_slot("B")
    assert list(cow_a) == g["copy"] and cow_b is None
    oracle.copy_blocks([kc], [vc], np.array([cow_a]))
    a_val = np.array([[[100.0]]], dtype=np.float32)   # stands for token 'a'
    b_val = np.array([[[200.0]]], dtype=np.float32)   # stands for token 'b'
    oracle.reshape_and_cache(a_val, a_val, [sa], kc, vc, B)
    oracle.reshape_and_cache(b_val, b_val, [sb], kc, vc, B)
    assert bm.tables["A"] == g["A"]["table"] and bm.tables["B"] == g["B"]["table"]
    assert (sa // B, sa % B) == (g["A"]["new_token_block"], g["A"]["new_token_row"])
    assert (sb // B, sb % B) == (g["B"]["new_token_block"], g["B"]["new_token_row"])
    for blk, cnt in g["refcounts"].items():
        assert bm.ref[int(blk)] == cnt
    sym = {"a": 100.0, "b": 200.0}
    for blk, key in ((4, "P4_rows_hold_positions"), (0, "P0_rows_hold_positions")):
        want = [sym.get(x, x) for x in g[key]]
        assert list(kc[blk, 0, :3, 0]) == want
        assert list(vc[blk, 0, :3, 0]) == want
    # the fully shared prefix block P3 is untouched and still holds 0..3
    assert list(kc[3, 0, :, 0]) == [0, 1, 2, 3]


def test_p2_fragmentation():
    g = load("p2_fragmentation.json")
    for key, B in (("B16", 16), ("B64", 64)):
        want = g[key]
        for L, (blk, slots, empty) in zip(g["lengths"], want["per_seq"]):
            assert oracle.blocks_needed(L, B) == blk
            assert oracle.slots_allocated(L, B) == slots
            assert slots - L == empty
        blocks, slots, empty, rate = oracle.fragmentation(g["lengths"], B)
        assert (blocks, slots, empty) == (want["blocks"], want["slots"], want["empty"])
        assert round(100 * rate, 1) == want["rate_pct"]


def test_p1_scenario_block_counts():
    g = load("p1_scenario_blocks.json")
    B = g["block_size"]
    for T, n in g["tokens_to_blocks"].items():
        assert oracle.blocks_needed(int(T), B) == n
    sc = g["scenario2"]
    total = sc["shared_prefix_blocks"] + sc["requests"] * sc["private_blocks"]
    assert total == sc["total_blocks"]
    reserved = sc["requests"] * sc["reserved_slots_per_request"]
    assert round(100 * (reserved - total * B) / reserved) == sc["saving_pct"]


def test_kv_bytes_per_token_examples():
    g = load("kv_bytes_per_token.json")
    opt, qwen, llama = g["cases"]
    b = oracle.kv_bytes_per_token(opt["layers"], opt["kv_heads"], opt["head_size"], opt["dtype_bytes"])
    assert round(b / 1024) == opt["approx_kib_per_token"]
    assert round(b * opt["tokens"] / 2**30, 1) == opt["approx_gib_total"]
    b = oracle.kv_bytes_per_token(qwen["layers"], qwen["kv_heads"], qwen["head_size"], qwen["dtype_bytes"])
    assert b == qwen["exact_bytes_per_token"]
    assert b * qwen["tokens"] / 2**30 == qwen["approx_gib_total"]
    b = oracle.kv_bytes_per_token(llama["layers"], llama["kv_heads"], llama["head_size"], llama["dtype_bytes"])
    for T, gib in llama["gib_by_tokens"].items():
        assert b * int(T) == gib * 2**30


# ------------------------------------------------------- brute-force properties
@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16])
def test_slot_mapping_is_a_bijection_onto_owned_rows(B):
    """Brute force: for a few requests with shuffled tables, every position
    < T maps to a distinct slot inside a block of that request's table, at
    row pos mod B, and the block order follows the logical order."""
    rng = np.random.default_rng(B)
    lens = [1, B, B + 1, 3 * B + 1]
    nblk = [oracle.blocks_needed(L, B) for L in lens]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb)
    mb = max(nblk)
    table = -np.ones((len(lens), mb), dtype=np.int32)
    off = 0
    for r, n in enumerate(nblk):
        table[r, :n] = perm[off:off + n]
        off += n
    qsl = np.concatenate([[0], np.cumsum(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    slots = oracle.slot_mapping(qsl, pos, table, B)
    assert len(set(slots.tolist())) == len(slots)          # no slot reused
    for r, L in enumerate(lens):
        for p in range(L):
            s = slots[qsl[r] + p]
            assert s // B == table[r, p // B]
            assert s % B == p % B
            assert s // B in set(table[r, :nblk[r]].tolist())


def test_slot_mapping_ragged_and_pad():
    table = np.array([[5, 2], [0, 1]], dtype=np.int32)
    # request 0 has no token, request 1 has two; token 2 belongs to nobody
    slots = oracle.slot_mapping([0, 0, 2], [1, 5], table, 4, num_tokens=3)
    assert slots.tolist() == [0 * 4 + 1, 1 * 4 + 1, -1]


def test_slot_mapping_rejects_bad_rows():
    t = np.array([[3, -1]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.slot_mapping([0, 1], [4], t, 4)     # unassigned entry
    with pytest.raises(ValueError):
        oracle.slot_mapping([0, 1], [8], t, 4)     # past the row
    with pytest.raises(ValueError):
        oracle.slot_mapping([0, 1], [-1], t, 4)


def test_copy_blocks_rejects_aliasing():
    kc = np.zeros((4, 1, 2, 1), np.float32)
    with pytest.raises(ValueError):
        oracle.copy_blocks([kc], [kc.copy()], np.array([[0, 1], [2, 1]]))
    with pytest.raises(ValueError):
        oracle.copy_blocks([kc], [kc.copy()], np.array([[0, 1], [1, 2]]))


def test_block_manager_invariants_random_walk():
    """Random fork/append/free sequence: reference counts equal the number of
    table entries naming each block, free blocks are exactly those with
    count 0, and every appended slot is the slot-mapping formula applied to
    the writer's own table."""
    rng = np.random.default_rng(7)
    B, NB = 4, 64
    bm = OracleBlockManager(NB, B)
    bm.allocate(0, 5)
    live = [0]
    nxt = 1
    for _ in range(300):
        op = rng.integers(0, 10)
        if op < 2 and len(live) < 6:
            bm.fork(live[rng.integers(len(live))], nxt)
            live.append(nxt)
            nxt += 1
        elif op < 3 and len(live) > 1:
            s = live.pop(rng.integers(len(live)))
            bm.free_seq(s)
        else:
            s = live[rng.integers(len(live))]
            pos = bm.lens[s]
            try:
                slot, cow = bm.append_slot(s)
            except ValueError:
                continue
            tab = np.array([bm.tables[s]], dtype=np.int32)
            assert oracle.slot_mapping([0, 1], [pos], tab, B)[0] == slot
            if cow is not None:
                assert bm.ref[cow[1]] == 1
        counts = np.zeros(NB, dtype=int)
        for t in bm.tables.values():
            for b in t:
                counts[b] += 1
        assert counts.tolist() == bm.ref
        assert sorted(bm.free) == [b for b in range(NB) if counts[b] == 0]
        for s, t in bm.tables.items():
            assert len(t) == oracle.blocks_needed(bm.lens[s], B)


def test_p1_map_to_kernel_blocks_example():
    g = load("p1_map_to_kernel_blocks.json")
    r = g["blocks_per_kv_block"]
    assert r == g["manager_block_tokens"] // g["kernel_block_tokens"]
    assert oracle.map_to_kernel_blocks(g["manager_ids"], r).tolist() == g["kernel_ids"]
    for k, ids in g["per_manager_block"].items():
        assert oracle.map_to_kernel_blocks([int(k)], r).tolist() == ids


def test_map_to_kernel_blocks_preserves_token_addresses():
    """Brute force: a token at position p of a sequence whose manager table
    uses blocks of B*r tokens lands at the same (kernel block, row) whether
    addressed through the expanded kernel table with block size B, or as
    row p % (B*r) of manager block k split into r kernel blocks."""
    rng = np.random.default_rng(5)
    for r in (1, 2, 4):
        B = 4
        mids = rng.permutation(10)[:4]
        kt = oracle.map_to_kernel_blocks(mids, r)
        for p in range(4 * B * r):
            k = mids[p // (B * r)]
            off = p % (B * r)
            want = (k * r + off // B, off % B)
            s = oracle.slot_mapping([0, 1], [p], kt.reshape(1, -1), B)[0]
            assert (s // B, s % B) == want

"""Planted mistakes: each mutant below is a plausible slip in the oracle (a
dropped term, a wrong index, a transposed operand, floor for ceil, a missed
reference-count update). The pins in test_oracle_pins.py and
test_oracle_attention.py must catch every one of them. Mutants are planted in
the oracle on the CPU only, through monkeypatching."""
import numpy as np
import pytest

import oracle
import oracle.paged_attention as opa
import oracle.block_manager as obm
import tests.test_oracle_attention as ta
import tests.test_oracle_block_scales as tb
import tests.test_oracle_fp8 as tf
import tests.test_oracle_pins as tp
import tests.test_oracle_window as tw


def _slot_no_subtract(qsl, pos, tab, B, num_tokens=None):
    tab = np.asarray(tab)
    out = np.full(len(pos) if num_tokens is None else num_tokens, -1, np.int64)
    for r in range(len(qsl) - 1):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            p = int(pos[t])
            out[t] = int(tab[r, p // B]) * B + p          # offset not reduced
    return out


def _slot_offset_swapped(qsl, pos, tab, B, num_tokens=None):
    tab = np.asarray(tab)
    out = np.full(len(pos) if num_tokens is None else num_tokens, -1, np.int64)
    for r in range(len(qsl) - 1):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            p = int(pos[t])
            out[t] = int(tab[r, p % B if p % B < tab.shape[1] else 0]) * B + p // B
    return out


def _blocks_floor(T, B):
    return T // B


def _attn_no_max(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    p = np.exp(scale * (K @ q))
    return (p @ V) / p.sum()


def _attn_no_scale(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    x = K @ q
    p = np.exp(x - x.max())
    return (p @ V) / p.sum()


def _attn_no_normalise(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    x = scale * (K @ q)
    return np.exp(x - x.max()) @ V


def _attn_keys_as_values(q, K, V, scale):
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    x = scale * (K @ q)
    p = np.exp(x - x.max())
    return (p @ K) / p.sum()


def _gather_head_modulo(cache, table_row, L, kv_head, B, dtype, start=0):
    # wrong row inside the block: j // B instead of j % B
    j = np.arange(start, L)
    blk = np.asarray(table_row)[j // B]
    return opa.upcast(np.ascontiguousarray(cache[blk, kv_head, (j // B) % B, :]), dtype)


def _upcast_bf16_wrong_shift(a, dtype):
    if dtype == "bf16":
        bits = a.view(np.uint16).astype(np.uint32) << np.uint32(15)
        return bits.view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _decode_gqa_modulo(q, kc, vc, tables, lens, scale, Hkv, B, dtype, seqs=None, heads=None,
                       window=0):
    S, Hq, D = q.shape
    out = np.zeros((S, Hq, D))
    q64 = opa.upcast(q, dtype)
    for s in range(S):
        for h in range(Hq):
            kvh = h % Hkv                                  # wrong group map
            lo = opa.window_start(int(lens[s]), window)
            K = opa.gather_kv(kc, tables[s], int(lens[s]), kvh, B, dtype, lo)
            V = opa.gather_kv(vc, tables[s], int(lens[s]), kvh, B, dtype, lo)
            out[s, h] = opa.decode_attention_one(q64[s, h], K, V, scale)
    return out


def _mq_sees_one_future_token(q, kc, vc, tables, qsl, lens, scale, Hkv, B, dtype):
    T, Hq, D = q.shape
    g = Hq // Hkv
    q64 = opa.upcast(q, dtype)
    out = np.zeros((T, Hq, D))
    for s in range(len(qsl) - 1):
        n, L = int(qsl[s + 1] - qsl[s]), int(lens[s])
        for kvh in range(Hkv):
            K = opa.gather_kv(kc, tables[s], L, kvh, B, dtype)
            V = opa.gather_kv(vc, tables[s], L, kvh, B, dtype)
            for i in range(n):
                last = min(L - 1, L - n + i + 1)           # one token too far
                for h in range(kvh * g, (kvh + 1) * g):
                    out[qsl[s] + i, h] = opa.decode_attention_one(q64[qsl[s] + i, h],
                                                                  K[:last + 1], V[:last + 1],
                                                                  scale)
    return out


def _window_one_late(L, W):
    return L - W + 1 if 0 < W < L else 0               # window one token short


def _window_one_early(L, W):
    return max(L - W - 1, 0) if 0 < W < L else 0       # one token too many


def _skipped_ceil(L, W, B):
    return -(-opa.window_start(L, W) // B)             # frees a partly used block


def _quant_multiply(x, dtype, scale):
    x32 = opa.upcast(x, dtype).astype(np.float32)
    return opa.e4m3_encode(x32 * np.float32(scale))         # multiplies by the scale


def _quant_fp64(x, dtype, scale):
    # divides and rounds in fp64: the nearest code of the unrounded quotient
    q = opa.upcast(x, dtype) / np.float64(np.float32(scale))
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = opa.e4m3_decode(finite)
    out = np.zeros(q.shape, dtype=np.uint8)
    for i, v in enumerate(q.reshape(-1)):
        d = np.abs(vals - v)
        cand = finite[d == d.min()]
        if len(cand) > 1:
            cand = cand[(cand & 1) == 0]
        if v < 0 and (cand & 0x80).all() == 0:
            cand = cand | 0x80
        out.reshape(-1)[i] = cand[0]
    return out


def _quant_scale_f64(x, dtype, scale):
    # the scale is not rounded to fp32 first
    q = opa.upcast(x, dtype) / float(scale)
    return opa.e4m3_encode(q.astype(np.float32))


def _bs_floor(amax):
    a = float(amax)
    if a == 0.0:
        return 1.0
    if np.isinf(a):
        return 2.0 ** 127
    k = min(max(int(np.floor(np.log2(a))) - 7, -126), 127)   # amax lands in [128, 256)
    return 2.0 ** k


def _bs_write(first_only=False, one_pass=False):
    def write(k, v, slots, kc8, vc8, ks, vs, B, dtype):
        slots = np.asarray(slots, dtype=np.int64)
        T, Hkv = len(slots), kc8.shape[1]

        def fix(t):
            s0 = int(slots[t])
            n = 1
            while not first_only and n < B and t + n < T and int(slots[t + n]) == s0 + n:
                n += 1
            for h in range(Hkv):
                for src, dst in ((k, ks), (v, vs)):
                    run = np.abs(opa.upcast(np.ascontiguousarray(src[t:t + n, h]), dtype))
                    dst[s0 // B, h] = opa.block_scale_e4m3(float(run.max()))

        def put(t):
            s = int(slots[t])
            for h in range(Hkv):
                kc8[s // B, h, s % B] = opa.quantize_e4m3(k[t, h], dtype, float(ks[s // B, h]))
                vc8[s // B, h, s % B] = opa.quantize_e4m3(v[t, h], dtype, float(vs[s // B, h]))

        if one_pass:                                   # fixes and writes in call order
            for t in range(T):
                if slots[t] >= 0 and slots[t] % B == 0:
                    fix(t)
                if slots[t] >= 0:
                    put(t)
            return
        for t in range(T):
            if slots[t] >= 0 and slots[t] % B == 0:
                fix(t)
        for t in range(T):
            if slots[t] >= 0:
                put(t)
    return write


def _bs_attn(logical_index=False, k_for_v=False):
    def attn(q, kc8, vc8, ks, vs, tables, lens, scale, Hkv, B, dtype, seqs=None, heads=None,
             window=0):
        S, Hq, D = q.shape
        g = Hq // Hkv
        q64 = opa.upcast(q, dtype)
        out = np.zeros((S, Hq, D))
        for s in range(S):
            L = int(lens[s])
            j = np.arange(opa.window_start(L, window), L)
            blk = np.asarray(tables[s], dtype=np.int64)[j // B]
            sidx = j // B if logical_index else blk           # scale of the wrong block
            for h in range(Hq):
                kvh = h // g
                K = opa.e4m3_decode(kc8[blk, kvh, j % B]) * np.float64(ks)[sidx, kvh][:, None]
                vsrc = ks if k_for_v else vs
                V = opa.e4m3_decode(vc8[blk, kvh, j % B]) * np.float64(vsrc)[sidx, kvh][:, None]
                out[s, h] = opa.decode_attention_one(q64[s, h], K, V, scale)
        return out
    return attn


class _RemoveSkippedCeil(obm.OracleBlockManager):
    def remove_skipped(self, seq, window):
        lo = opa.window_start(self.lens[seq], window)
        table, gone = self.tables[seq], []
        for i in range(-(-lo // self.block_size)):               # a partly used block too
            if table[i] is not None:
                gone.append(table[i])
                self._release(table[i])
                table[i] = None
        return gone


class _RemoveSkippedFreesShared(obm.OracleBlockManager):
    def remove_skipped(self, seq, window):
        table, gone = self.tables[seq], []
        for i in range(opa.skipped_blocks(self.lens[seq], window, self.block_size)):
            if table[i] is not None:
                gone.append(table[i])
                self.ref[table[i]] = 0                           # ignores other holders
                self.free.append(table[i])
                table[i] = None
        return gone


class _NoDecrementOnCow(obm.OracleBlockManager):
    def _release(self, b):
        pass


class _CowAlways(obm.OracleBlockManager):
    def append_slot(self, seq):
        B = self.block_size
        L = self.lens[seq]
        table = self.tables[seq]
        lb = L // B
        cow = None
        if lb == len(table):
            table.append(self._take())
        elif self.ref[table[lb]] >= 1:                     # copies even when sole holder
            src, dst = table[lb], self._take()
            self._release(src)
            table[lb] = dst
            cow = (src, dst)
        self.lens[seq] = L + 1
        return table[lb] * B + (L - lb * B), cow


PIN_TESTS = [
    tp.test_p4_block_table_example,
    tp.test_p2_seven_token_prompt_on_demand_append,
    tp.test_p2_fig8_copy_on_write_and_savings,
    tp.test_p4_cow_figure_tables_refcounts_and_data,
    tp.test_p2_fragmentation,
    tp.test_p1_scenario_block_counts,
    tp.test_kv_bytes_per_token_examples,
    lambda: tp.test_slot_mapping_is_a_bijection_onto_owned_rows(4),
    ta.test_bf16_upcast_is_exact,
    ta.test_single_token_returns_its_value_exactly,
    ta.test_equal_keys_give_the_mean_value,
    ta.test_dominant_logit_selects_its_value_without_overflow,
    lambda: ta.test_pure_python_brute_force(7, 8),
    lambda: ta.test_oracle_matches_sdpa_fp64("gqa_small", "bf16", 8, 2, 8),
    ta.test_decode_step_attends_to_the_new_token,
    ta.test_gqa_query_head_reads_its_group_kv_head,
    ta.test_multi_query_with_one_new_token_is_decode,
    ta.test_multi_query_matches_sdpa_with_causal_offset_mask,
    tw.test_window_start_reading,
    lambda: tw.test_skipped_blocks_brute_force(4),
    tw.test_window_of_one_is_the_new_value,
    tw.test_equal_keys_give_mean_of_last_w_values,
    lambda: tw.test_window_matches_masked_sdpa("f16", 8, 9),
    tw.test_manager_releases_only_blocks_wholly_before_the_window,
    tf.test_quantize_divides_by_the_scale,
    tf.test_quantize_largest_code_for_448_scales,
    tf.test_quantize_rounds_the_quotient_to_fp32_before_encoding,
    tf.test_quantize_rounds_the_scale_to_fp32,
    tb.test_block_scale_closed_forms,
    tb.test_block_scale_is_the_smallest_power_of_two_that_fits_128,
    tb.test_decode_write_fixes_the_scale_at_row_0_and_reuses_it_later,
    tb.test_a_run_of_consecutive_slots_fixes_the_scale_from_its_largest_value,
    tb.test_the_run_ends_at_a_gap_and_scales_are_fixed_before_any_token_is_written,
    lambda: tb.test_values_on_the_code_grid_round_trip_exactly("bf16"),
    tb.test_block_scaled_attention_matches_brute_force,
    tb.test_equal_block_scales_reduce_to_the_per_pool_scale,
    tb.test_block_scaled_attention_is_invariant_under_relabelling,
]

MUTANTS = {
    "slot_no_subtract": [("slot_mapping", _slot_no_subtract)],
    "slot_offset_swapped": [("slot_mapping", _slot_offset_swapped)],
    "blocks_floor": [("blocks_needed", _blocks_floor)],
    "attn_no_max": [("decode_attention_one", _attn_no_max)],
    "attn_no_scale": [("decode_attention_one", _attn_no_scale)],
    "attn_no_normalise": [("decode_attention_one", _attn_no_normalise)],
    "attn_keys_as_values": [("decode_attention_one", _attn_keys_as_values)],
    "gather_wrong_row": [("gather_kv", _gather_head_modulo)],
    "bf16_wrong_shift": [("upcast", _upcast_bf16_wrong_shift)],
    "gqa_modulo": [("decode_attention", _decode_gqa_modulo)],
    "cow_no_decrement": [("OracleBlockManager", _NoDecrementOnCow)],
    "cow_always": [("OracleBlockManager", _CowAlways)],
    "mq_future_token": [("multi_query_attention", _mq_sees_one_future_token)],
    "window_one_late": [("window_start", _window_one_late)],
    "window_one_early": [("window_start", _window_one_early)],
    "skipped_ceil": [("skipped_blocks", _skipped_ceil)],
    "quant_multiply": [("quantize_e4m3", _quant_multiply)],
    "quant_fp64": [("quantize_e4m3", _quant_fp64)],
    "quant_scale_f64": [("quantize_e4m3", _quant_scale_f64)],
    "remove_skipped_ceil": [("OracleBlockManager", _RemoveSkippedCeil)],
    "remove_skipped_frees_shared": [("OracleBlockManager", _RemoveSkippedFreesShared)],
    "block_scale_floor": [("block_scale_e4m3", _bs_floor)],
    "block_scale_first_token_only": [("reshape_and_cache_fp8_block_scaled",
                                      _bs_write(first_only=True))],
    "block_scale_one_pass": [("reshape_and_cache_fp8_block_scaled", _bs_write(one_pass=True))],
    "block_scale_of_logical_block": [("decode_attention_fp8_block_scaled",
                                      _bs_attn(logical_index=True))],
    "block_scale_k_for_v": [("decode_attention_fp8_block_scaled", _bs_attn(k_for_v=True))],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    for attr, fn in MUTANTS[name]:
        for mod in (oracle, opa, obm, tp, tw, tf, tb):
            if hasattr(mod, attr):
                monkeypatch.setattr(mod, attr, fn)
    caught = []
    with np.errstate(all="ignore"):
        for t in PIN_TESTS:
            try:
                t()
            except Exception:
                caught.append(getattr(t, "__name__", "lambda"))
    assert caught, f"mutant {name} survived every pin"

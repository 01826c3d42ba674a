"""Pins for the oracle's fp8 blocks with their own scales (one power-of-two
scale per (physical block, KV head), fixed by the write that stores the
block's first row): the scale's closed form and a brute-force search for it,
worked write examples whose codes follow from the E4M3 definition by hand,
the run of consecutive slots that fixes a scale, the two-pass order, exact
round trips, and attention on the dequantised values against brute force,
a per-pool scale and block relabelling."""
import math

import numpy as np
import pytest

import oracle


def test_block_scale_closed_forms():
    f = oracle.block_scale_e4m3
    assert f(1.0) == 2.0 ** -7           # ceil(log2 1) = 0: 1 -> 128
    assert f(1.5) == 2.0 ** -6           # 1.5 -> 96
    assert f(3.0) == 2.0 ** -5           # 3 -> 96
    assert f(128.0) == 1.0               # exactly 128 stays 128
    assert f(129.0) == 2.0               # 129 -> 64.5
    assert f(0.0) == 1.0                 # nothing to scale
    assert f(float("inf")) == 2.0 ** 127
    assert f(1e-45) == 2.0 ** -126       # clamped to the smallest normal
    assert f(3e38) == 2.0 ** 121


def test_block_scale_is_the_smallest_power_of_two_that_fits_128():
    rng = np.random.default_rng(4)
    amaxes = np.concatenate([np.exp2(rng.uniform(-118, 126, 3000)),
                             np.exp2(rng.integers(-118, 126, 200).astype(np.float64))])
    for a in amaxes.astype(np.float32).astype(np.float64):
        # brute force: walk k upward from the smallest exponent
        k = -126
        while a > 128.0 * 2.0 ** k:
            k += 1
        s = oracle.block_scale_e4m3(a)
        assert s == 2.0 ** k, a
        assert 64.0 < a / s <= 128.0, a
        assert math.frexp(s)[0] == 0.5                   # a power of two


def _pools(NB=6, Hkv=2, B=4, D=16):
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.zeros((NB, Hkv, B, D), np.uint8)
    ks = np.full((NB, Hkv), 0.25, np.float32)
    vs = np.full((NB, Hkv), 0.25, np.float32)
    return kc, vc, ks, vs


def test_decode_write_fixes_the_scale_at_row_0_and_reuses_it_later():
    kc, vc, ks, vs = _pools()
    k = np.zeros((2, 2, 16), np.float32)
    v = np.zeros((2, 2, 16), np.float32)
    k[0, 0, 3] = -3.0          # token 0 -> slot 12 = block 3, row 0
    k[0, 0, 4] = 1.5
    k[0, 1, 0] = 0.75          # head 1: amax 0.75 -> 2^-7 (0.75 -> 96)
    v[0, :, 0] = 100.0         # -> 2^0: 100 stays 100
    k[1, 0, 0] = 1.0           # token 1 -> slot 6 = block 1, row 2: stored scale 0.25
    v[1, 0, 0] = 500.0         # 500 / 0.25 = 2000 saturates
    oracle.reshape_and_cache_fp8_block_scaled(k, v, [12, 6], kc, vc, ks, vs, 4, "f32")
    assert ks[3].tolist() == [2.0 ** -5, 2.0 ** -7] and vs[3].tolist() == [1.0, 1.0]
    assert ks[1].tolist() == [0.25, 0.25] and vs[1].tolist() == [0.25, 0.25]
    # -3 / 2^-5 = -96 = -1.5 * 2^6 -> sign | (13 << 3) | 4; 1.5 / 2^-5 = 48 -> (12 << 3) | 4
    assert kc[3, 0, 0, 3] == 0xEC and kc[3, 0, 0, 4] == 0x64
    assert kc[3, 1, 0, 0] == 0x6C                       # 0.75 / 2^-7 = 96
    # 100 lies halfway between the codes 96 (0x6C) and 104 (0x6D): the even one
    assert vc[3, 0, 0, 0] == 0x6C and vc[3, 1, 0, 0] == 0x6C
    assert kc[1, 0, 2, 0] == 0x48                        # 1.0 / 0.25 = 4 = 1.0 * 2^2
    assert vc[1, 0, 2, 0] == 0x7E                        # saturated to 448
    assert not kc[3, :, 1:].any() and not kc[0].any()    # nothing else written


def test_a_run_of_consecutive_slots_fixes_the_scale_from_its_largest_value():
    # 6 tokens of one request in slots 8..13 (B = 4): the run 8..11 fixes
    # block 2 from all four tokens (the largest, 6.0, is the third); the
    # run 12..13 fixes block 3 from its two tokens
    kc, vc, ks, vs = _pools()
    k = np.full((6, 2, 16), 0.5, np.float32)
    v = np.full((6, 2, 16), 0.5, np.float32)
    k[2, 0, 7] = 6.0                                       # -> 2^-4 (6 -> 96)
    k[5, 1, 1] = -40.0                                     # -> 2^-1 (40 -> 80)
    oracle.reshape_and_cache_fp8_block_scaled(k, v, list(range(8, 14)), kc, vc, ks, vs, 4, "f32")
    assert ks[2].tolist() == [2.0 ** -4, 2.0 ** -8]        # head 1: 0.5 -> 128
    assert ks[3].tolist() == [2.0 ** -8, 2.0 ** -1]
    assert vs[2].tolist() == [2.0 ** -8] * 2 and vs[3].tolist() == [2.0 ** -8] * 2
    assert kc[2, 0, 0, 0] == 0x50 and kc[2, 0, 2, 7] == 0x6C   # 8 = 2^3; 96
    assert (kc[2, 1] == 0x70).all()                        # 0.5 / 2^-8 = 128 = 2^7
    assert kc[3, 1, 1, 1] == 0xEA and kc[3, 1, 0, 0] == 0x38   # -80; 0.5 / 0.5 = 1
    assert (vc[2] == 0x70).all() and (vc[3, :, :2] == 0x70).all() and not vc[3, :, 2:].any()


def test_the_run_ends_at_a_gap_and_scales_are_fixed_before_any_token_is_written():
    # slots [9, 8, 21, 10]: token 0 (row 1 of block 2) comes before the
    # row-0 token 1 in the call; token 2 jumps to another block, so token 1's
    # run is token 1 alone; token 3 (row 2 of block 2) is outside the run but
    # is still quantised with the scale token 1 fixed, and saturates; token 0
    # too uses that new scale although it comes first
    kc, vc, ks, vs = _pools()
    k = np.zeros((4, 2, 16), np.float32)
    v = np.zeros((4, 2, 16), np.float32)
    k[0, :, 0] = 2.0
    k[1, :, 0] = 1.0            # the run: amax 1 -> 2^-7
    k[2, :, 0] = 1.0
    k[3, :, 0] = 8.0            # 8 / 2^-7 = 1024: past 448
    oracle.reshape_and_cache_fp8_block_scaled(k, v, [9, 8, 21, 10], kc, vc, ks, vs, 4, "f32")
    assert ks[2].tolist() == [2.0 ** -7] * 2 and vs[2].tolist() == [1.0, 1.0]
    assert ks[5].tolist() == [0.25, 0.25]                  # slot 21 is row 1: not fixed
    assert kc[2, 0, 1, 0] == 0x78                          # 2 / 2^-7 = 256 = 2^8
    assert kc[2, 0, 0, 0] == 0x70                          # 128 = 2^7
    assert kc[2, 0, 2, 0] == 0x7E                          # saturated
    assert kc[5, 0, 1, 0] == 0x48                          # 1 / 0.25 = 4 = 2^2


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_values_on_the_code_grid_round_trip_exactly(dtype):
    # every token of a full block written in one call: values that are an
    # E4M3 value times the block's scale come back exactly
    rng = np.random.default_rng(8)
    upto128 = np.array([c for c in range(256) if (c & 0x7F) <= 0x70], np.uint8)
    codes = rng.choice(upto128, size=(4, 2, 16))
    codes[0, :, 0] = 0x70                                  # 128: fixes the scale at 2^k
    k_exp = np.array([-3, 5])
    vals = oracle.e4m3_decode(codes) * np.exp2(k_exp)[None, :, None]
    x32 = vals.astype(np.float32)
    if dtype == "f16":
        x = x32.astype(np.float16)
    elif dtype == "bf16":
        x = (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    else:
        x = x32
    assert np.array_equal(oracle.upcast(x, dtype), vals)   # exactly representable
    kc, vc, ks, vs = _pools()
    oracle.reshape_and_cache_fp8_block_scaled(x, x, [16, 17, 18, 19], kc, vc, ks, vs, 4, dtype)
    assert ks[4].tolist() == [2.0 ** -3, 2.0 ** 5] and vs[4].tolist() == ks[4].tolist()
    back = oracle.e4m3_decode(kc[4].transpose(1, 0, 2)) * np.exp2(k_exp)[None, :, None]
    assert np.array_equal(np.where(back == 0, 0.0, back), np.where(vals == 0, 0.0, vals))


def _brute_attention(q, kc, vc, ks, vs, tables, lens, scale, Hkv, B):
    S, Hq, D = q.shape
    g = Hq // Hkv
    out = np.zeros((S, Hq, D))
    for s in range(S):
        for h in range(Hq):
            kvh = h // g
            logits, rows = [], []
            for j in range(int(lens[s])):
                blk, r = int(tables[s][j // B]), j % B
                kj = [float(oracle.e4m3_decode([kc[blk, kvh, r, d]])[0]) * float(ks[blk, kvh])
                      for d in range(D)]
                vj = [float(oracle.e4m3_decode([vc[blk, kvh, r, d]])[0]) * float(vs[blk, kvh])
                      for d in range(D)]
                logits.append(scale * sum(float(q[s, h, d]) * kj[d] for d in range(D)))
                rows.append(vj)
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            for d in range(D):
                out[s, h, d] = sum(wi * r[d] for wi, r in zip(w, rows)) / sum(w)
    return out


def _random_fp8_case(seed, NB=7, Hkv=2, B=4, D=8):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 256, size=(NB, Hkv, B, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, B, D)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38
    vc[(vc & 0x7F) == 0x7F] = 0x30
    ks = np.exp2(rng.integers(-12, -4, size=(NB, Hkv))).astype(np.float32)
    vs = np.exp2(rng.integers(-12, -4, size=(NB, Hkv))).astype(np.float32)
    q = rng.standard_normal((2, 4, D)).astype(np.float32)
    tables = np.array([[3, 1, 0], [5, 2, 6]])
    lens = np.array([9, 11])
    return q, kc, vc, ks, vs, tables, lens


def test_block_scaled_attention_matches_brute_force():
    q, kc, vc, ks, vs, tables, lens = _random_fp8_case(2)
    got = oracle.decode_attention_fp8_block_scaled(q, kc, vc, ks, vs, tables, lens, 0.3, 2, 4,
                                                   "f32")
    want = _brute_attention(q, kc, vc, ks, vs, tables, lens, 0.3, 2, 4)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_equal_block_scales_reduce_to_the_per_pool_scale():
    q, kc, vc, ks, vs, tables, lens = _random_fp8_case(3)
    ks[:] = 0.125
    vs[:] = 2.0 ** -9
    got = oracle.decode_attention_fp8_block_scaled(q, kc, vc, ks, vs, tables, lens, 0.3, 2, 4,
                                                   "f32", window=5)
    want = oracle.decode_attention_fp8(q, kc, vc, tables, lens, 0.3, 2, 4, "f32", 0.125,
                                       2.0 ** -9, window=5)
    assert np.array_equal(got, want)


def test_block_scaled_attention_is_invariant_under_relabelling():
    # a block's scales travel with it: permute the pool, its scales and the
    # tables together and nothing changes
    q, kc, vc, ks, vs, tables, lens = _random_fp8_case(4)
    perm = np.random.default_rng(5).permutation(kc.shape[0])    # new id of block b
    inv = np.argsort(perm)
    got = oracle.decode_attention_fp8_block_scaled(q, kc, vc, ks, vs, tables, lens, 0.3, 2, 4,
                                                   "f32")
    moved = oracle.decode_attention_fp8_block_scaled(q, kc[inv], vc[inv], ks[inv], vs[inv],
                                                     perm[tables], lens, 0.3, 2, 4, "f32")
    assert np.array_equal(got, moved)

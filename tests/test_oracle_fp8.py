"""Pins for the oracle's fp8 (E4M3) KV codes: the value of every code, the
nearest-value rounding with ties to even and saturation, against torch's
float8_e4m3fn type and brute force over all finite codes."""
import numpy as np
import torch

import oracle


def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])


def test_known_codes():
    enc = oracle.e4m3_encode
    assert oracle.e4m3_decode([0x38, 0x7E, 0x01, 0x08, 0xFE])[:4].tolist() == \
        [1.0, 448.0, 2.0 ** -9, 2.0 ** -6]
    assert enc(np.float32([1.0, 448.0, 500.0, -500.0, 1e30]))[:5].tolist() == \
        [0x38, 0x7E, 0x7E, 0xFE, 0x7E]
    # ties to even: 2^-10 lies halfway between 0 and 2^-9 -> 0; 3*2^-10 between
    # codes 1 and 2 -> 2; 1.0625 between 1.0 (0x38) and 1.125 (0x39) -> 0x38
    assert enc(np.float32([2.0 ** -10, 3 * 2.0 ** -10, 1.0625]))[:3].tolist() == [0, 2, 0x38]
    assert enc(np.float32([np.nan]))[0] == 0x7F


def test_encode_matches_torch_in_range():
    x = (np.random.default_rng(0).standard_normal(5000) * 40).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_encode_is_the_nearest_code_brute_force():
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(finite)
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 400), rng.uniform(-0.05, 0.05, 400)])
    x = x.astype(np.float32)
    codes = oracle.e4m3_encode(x)
    for xi, ci in zip(x.astype(np.float64), codes):
        d = np.abs(vals - xi)
        best = d.min()
        cand = finite[d == best]
        if len(cand) > 1:                      # a tie: the even mantissa wins
            cand = cand[(cand & 1) == 0]
            if xi == 0.0:
                cand = cand[(cand & 0x80) == (0x80 if np.signbit(xi) else 0)]
        assert ci in set(cand.tolist()), (xi, ci, cand)


def test_round_trip_of_finite_codes():
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(finite).astype(np.float32))
    assert np.array_equal(back, finite)


def test_fp8_attention_is_attention_on_dequantised_values():
    rng = np.random.default_rng(2)
    NB, Hkv, B, D = 6, 2, 4, 8
    kc = rng.integers(0, 256, size=(NB, Hkv, B, D)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(NB, Hkv, B, D)).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x38                  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x30
    q = rng.standard_normal((2, 4, D)).astype(np.float32)
    tables = np.array([[3, 1, 0], [5, 2, 4]])
    lens = np.array([9, 11])
    got = oracle.decode_attention_fp8(q, kc, vc, tables, lens, 0.3, Hkv, B, "f32", 0.5, 2.0)
    Kf = (oracle.e4m3_decode(kc) * 0.5).astype(np.float64)
    Vf = (oracle.e4m3_decode(vc) * 2.0).astype(np.float64)
    want = oracle.decode_attention(q, Kf.astype(np.float32), Vf.astype(np.float32), tables,
                                   lens, 0.3, Hkv, B, "f32")
    assert np.allclose(got, want, atol=1e-12, rtol=0)

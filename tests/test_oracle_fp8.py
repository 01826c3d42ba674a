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


# --------------------------------------------------------------------------
# The quantising step: code = e4m3(RN_fp32(x / RN_fp32(scale))). These pins
# fix each rounding of that definition independently of the oracle's own
# encoder: an exact rational model (IEEE round-to-nearest-even to fp32 done
# in integer arithmetic, then the nearest finite E4M3 value by brute force
# with ties to the even code), and hand-picked cases where each rounding
# decides the code.
# --------------------------------------------------------------------------
from fractions import Fraction


def _bits_f32(u):
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


def _rn_f32(q: Fraction) -> Fraction:
    """Round a nonzero rational to the nearest fp32 value (ties to even),
    normal range only."""
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    r = n - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def _e4m3_value(c: int) -> Fraction:
    """Value of a finite E4M3 code from the format's definition."""
    s = -1 if c & 0x80 else 1
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0:
        return s * Fraction(m, 8) * Fraction(2) ** -6
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


_MAGNITUDES = list(range(0x7F))          # the finite non-negative codes


def _nearest_code(q: Fraction) -> int:
    """Nearest finite code to q, ties to the even code; the sign bit is q's
    sign (a negative value that rounds to zero gives the negative zero)."""
    a = abs(q)
    best = min(abs(_e4m3_value(c) - a) for c in _MAGNITUDES)
    cand = [c for c in _MAGNITUDES if abs(_e4m3_value(c) - a) == best]
    if len(cand) > 1:
        cand = [c for c in cand if (c & 1) == 0]
    return cand[0] | (0x80 if q < 0 else 0)


def _exact_quantize(x: float, scale: float) -> int:
    """The definition, in exact arithmetic: fp32 scale, fp32 quotient, then
    the nearest E4M3 code (values past 448 are nearest to 448: saturation)."""
    if x == 0.0:
        return 0x80 if np.signbit(x) else 0
    s32 = Fraction(float(np.float32(scale)))
    return _nearest_code(_rn_f32(Fraction(x) / s32))


def test_quantize_divides_by_the_scale():
    q = oracle.quantize_e4m3
    # 1 / 0.5 = 2 -> 0x40; -3 / 2 = -1.5 -> 0xBC; 0.75 / 0.25 = 3 -> 0x44
    assert q(np.float32([1.0]), "f32", 0.5)[0] == 0x40
    assert q(np.float32([-3.0]), "f32", 2.0)[0] == 0xBC
    assert q(np.float16([0.75]), "f16", 0.25)[0] == 0x44


def test_quantize_largest_code_for_448_scales():
    # x = 448 * s exactly (s a power of two, or s with a short mantissa so the
    # product is an fp32 value) lands on the largest finite code; 416 * s on
    # the one below it; a little past 448 * s saturates
    for s in (0.5, 0.0078125, 3.0, 0.375, 1.25, 7.0):
        x = np.float32([448.0 * s, 416.0 * s, 460.0 * s, -448.0 * s])
        assert float(x[0]) == 448.0 * s
        assert oracle.quantize_e4m3(x, "f32", s).tolist() == [0x7E, 0x7D, 0x7E, 0xFE], s


def test_quantize_rounds_the_quotient_to_fp32_before_encoding():
    # exact x / s lies just above an E4M3 tie point (1.0625 between 0x38 and
    # 0x39, 1.5625 between 0x3C and 0x3D) by less than half an fp32 ulp, so
    # the fp32 quotient is the tie itself and goes to the even code; an
    # encoder fed the unrounded quotient would pick the odd one
    for xb, sb, tie, even, odd in ((0x3FACB0E5, 0x3FA2885F, Fraction(17, 16), 0x38, 0x39),
                                   (0x402CF31D, 0x3FDD6025, Fraction(25, 16), 0x3C, 0x3D)):
        x, s = _bits_f32(xb), _bits_f32(sb)
        exact = Fraction(float(x)) / Fraction(float(s))
        assert exact > tie and _rn_f32(exact) == tie
        assert _nearest_code(exact) == odd
        assert oracle.quantize_e4m3(np.float32([x]), "f32", float(s))[0] == even
        assert oracle.quantize_e4m3(np.float32([-x]), "f32", float(s))[0] == even | 0x80


def test_quantize_rounds_the_scale_to_fp32():
    # the scale the kernel sees is an fp32 value; with s = 0.15578555507423250
    # (not an fp32 value) x / RN32(s) rounds just below the 4.75 tie (-> 0x49)
    # while x / s would round onto it (-> 0x4A)
    s = 0.1557855550742325
    x = _bits_f32(0x3F3D6F6B)
    assert _rn_f32(Fraction(float(x)) / Fraction(s)) == Fraction(19, 4)
    assert _exact_quantize(float(x), s) == 0x49
    assert oracle.quantize_e4m3(np.float32([x]), "f32", s)[0] == 0x49


def test_quantize_matches_the_exact_definition_on_random_inputs():
    rng = np.random.default_rng(11)
    for dtype in ("f32", "f16", "bf16"):
        x32 = (rng.standard_normal(300) * rng.choice([0.01, 1.0, 30.0], 300)).astype(np.float32)
        if dtype == "f16":
            stored = x32.astype(np.float16)
            vals = stored.astype(np.float64)
        elif dtype == "bf16":
            stored = (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
            vals = (stored.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        else:
            stored, vals = x32, x32.astype(np.float64)
        for scale in (float(rng.uniform(0.002, 0.2)), float(rng.uniform(0.5, 4.0))):
            got = oracle.quantize_e4m3(stored, dtype, scale)
            want = [_exact_quantize(float(v), scale) for v in vals]
            assert got.tolist() == want, (dtype, scale)

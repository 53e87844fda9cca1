"""Pins for the oracle's 8-bit (OCP FP8 E4M3) cache: the code table, the rounding
of the scatter, and decode attention over dequantised values.

The 8-bit cache is not on the pages; the format is the published OCP FP8 E4M3
definition (sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
S.1111.111 = NaN, largest finite 448). Each pin below is fixed by that
definition, by arithmetic, or by an independent library routine (torch's
float8_e4m3fn casts), never by re-running the oracle's own formula.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- code table

# (code, value) fixed by the format definition, worked by hand:
#   exponent field 0 -> subnormal m/8 * 2^-6; otherwise (1 + m/8) * 2^(e-7).
CLOSED_FORMS = [
    (0x00, 0.0),
    (0x01, 2.0 ** -9),             # smallest subnormal: 1/8 * 2^-6
    (0x04, 2.0 ** -7),             # 4/8 * 2^-6
    (0x07, 7 * 2.0 ** -9),         # largest subnormal
    (0x08, 2.0 ** -6),             # smallest normal
    (0x30, 0.5),                   # e = 6
    (0x38, 1.0),                   # e = 7 (the bias)
    (0x39, 1.125),
    (0x3C, 1.5),
    (0x40, 2.0),
    (0x77, 240.0),                 # e = 14, m = 7: 1.875 * 2^7
    (0x78, 256.0),                 # e = 15, m = 0
    (0x7E, 448.0),                 # e = 15, m = 6: largest finite
    (0xB8, -1.0),
    (0xFE, -448.0),
]


@pytest.mark.parametrize("code,value", CLOSED_FORMS)
def test_e4m3_closed_forms(code, value):
    got = float(oracle.e4m3_to_float64([code])[0])
    assert got == value
    if value == 0.0:
        assert math.copysign(1.0, got) == 1.0


def test_e4m3_nan_codes_and_negative_zero():
    v = oracle.e4m3_to_float64([0x7F, 0xFF, 0x80])
    assert math.isnan(v[0]) and math.isnan(v[1])
    assert v[2] == 0.0 and math.copysign(1.0, v[2]) == -1.0


def test_e4m3_order_and_symmetry():
    pos = oracle.e4m3_to_float64(np.arange(0x00, 0x7F, dtype=np.uint8))
    neg = oracle.e4m3_to_float64(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0), "finite codes must increase with magnitude"
    np.testing.assert_array_equal(neg, -pos)
    # 126 positive finite values, spacing 2^-9 through the subnormals and the first binade
    np.testing.assert_array_equal(np.diff(pos[:16]), np.full(15, 2.0 ** -9))


def test_e4m3_decode_matches_torch():
    """torch's float8_e4m3fn -> float32 cast is an independent decoder."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_float64(codes.numpy())
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- rounding

def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_float64(codes).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_from_float32(vals), codes)


def test_e4m3_midpoints_tie_to_even_and_neighbours():
    pos = oracle.e4m3_to_float64(np.arange(0x00, 0x7F, dtype=np.uint8))
    for c in range(0x7E):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)       # exact: at most 5 significant bits
        assert float(mid) == (pos[c] + pos[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        up = np.nextafter(mid, np.float32(np.inf))
        down = np.nextafter(mid, np.float32(0))
        got = oracle.e4m3_from_float32(np.array([mid, up, down, -mid], dtype=np.float32))
        assert list(got) == [even, c + 1, c, 0x80 | even], c


def test_e4m3_saturation_and_specials():
    x = np.array([448.0, 463.99, 464.0, 1e6, np.inf, -np.inf, -1e30, np.nan], dtype=np.float32)
    got = oracle.e4m3_from_float32(x)
    assert list(got[:7]) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[7] == 0x7F


def test_e4m3_below_smallest_subnormal():
    half = np.float32(2.0 ** -10)                       # midpoint of 0 and 2^-9
    tiny = np.array([half, np.nextafter(half, np.float32(1)), -half, np.float32(1e-30),
                     np.float32(-1e-30), np.float32(2.0 ** -149)], dtype=np.float32)
    got = oracle.e4m3_from_float32(tiny)
    # tie -> even code 0; just above -> 0x01; sign kept on zero results
    assert list(got) == [0x00, 0x01, 0x80, 0x00, 0x80, 0x00]


def test_e4m3_encode_matches_torch_in_range():
    """torch's float32 -> float8_e4m3fn cast (round to nearest even) is an
    independent encoder for finite magnitudes below 448."""
    rng = np.random.default_rng(8101)
    mag = np.exp2(rng.uniform(-14.0, math.log2(447.9), size=40000)).astype(np.float32)
    sign = np.where(rng.random(40000) < 0.5, -1.0, 1.0).astype(np.float32)
    pos = oracle.e4m3_to_float64(np.arange(0x00, 0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([mag * sign, mids, -mids, np.float32([0.0, -0.0])])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_from_float32(x), ref)


# ---------------------------------------------------------------- scatter

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_kv_write_fp8_places_quotient_codes():
    """Each written byte is the code of the float32 quotient x / scale (numpy's
    float32 division is IEEE), at block slot // bs, offset slot % bs; slot -1 and
    untouched slots keep their bytes."""
    rng = np.random.default_rng(8102)
    T, Hk, D, bs, NB = 6, 2, 16, 4, 5
    k = rng.normal(size=(T, Hk, D)).astype(np.float32) * 3
    v = rng.normal(size=(T, Hk, D)).astype(np.float32)
    slots = np.array([7, -1, 0, 19, 12, 5], dtype=np.int32)
    kc = np.full((NB, bs, Hk, D), 0x5A, dtype=np.uint8)
    vc = np.full((NB, bs, Hk, D), 0xA5, dtype=np.uint8)
    ks, vs = np.float32(0.0371), np.float32(0.0059)
    bad = oracle.kv_write_fp8(k, v, slots, kc, vc, float(ks), float(vs), "f32")
    assert bad == 0
    ref_k = oracle.e4m3_from_float32(k / ks)
    ref_v = oracle.e4m3_from_float32(v / vs)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(kc[s // bs, s % bs], ref_k[t])
        np.testing.assert_array_equal(vc[s // bs, s % bs], ref_v[t])
    written = {int(s) for s in slots if s >= 0}
    for s in range(NB * bs):
        if s not in written:
            assert np.all(kc[s // bs, s % bs] == 0x5A) and np.all(vc[s // bs, s % bs] == 0xA5)


def test_kv_write_fp8_bf16_source_and_bad_slot():
    rng = np.random.default_rng(8103)
    T, Hk, D, bs, NB = 3, 1, 8, 2, 2
    k = _bf16_bits(rng.normal(size=(T, Hk, D)))
    v = _bf16_bits(rng.normal(size=(T, Hk, D)))
    kc = np.zeros((NB, bs, Hk, D), dtype=np.uint8)
    vc = np.zeros((NB, bs, Hk, D), dtype=np.uint8)
    bad = oracle.kv_write_fp8(k, v, np.array([0, 4, 3], dtype=np.int32), kc, vc, 0.25, 0.5, "bf16")
    assert bad == 1                       # slot 4 is past NB * bs = 4
    kf = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(kc[0, 0], oracle.e4m3_from_float32(kf[0] / np.float32(0.25)))
    np.testing.assert_array_equal(kc[1, 1], oracle.e4m3_from_float32(kf[2] / np.float32(0.25)))


# ---------------------------------------------------------------- attention

def _finite_codes(rng, shape):
    """Random E4M3 codes with exponent fields 0..11 (no NaN), both signs."""
    e = rng.integers(0, 12, size=shape)
    m = rng.integers(0, 8, size=shape)
    s = rng.integers(0, 2, size=shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def test_attention_fp8_matches_dense_numpy():
    """Dequantise with torch's float8 decoder, gather through the block table in
    the test, and take softmax(q K^T scale) V densely in float64."""
    rng = np.random.default_rng(8104)
    B, H, Hk, D, bs, NB = 3, 4, 2, 16, 4, 24
    ctx = np.array([1, 9, 22], dtype=np.int32)
    MB = 6
    perm = rng.permutation(NB)
    bt = np.full((B, MB), -1, dtype=np.int32)
    used = 0
    for b in range(B):
        n = -(-int(ctx[b]) // bs)
        bt[b, :n] = perm[used:used + n]
        used += n
    kc = _finite_codes(rng, (NB, bs, Hk, D))
    vc = _finite_codes(rng, (NB, bs, Hk, D))
    q = rng.normal(size=(B, H, D)).astype(np.float32)
    ks, vs, scale = 0.0123, 0.0456, 0.25
    got = oracle.paged_attention_fp8(q, kc, vc, bt, ctx, scale, ks, vs, "f32")

    dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    Kf = dec(kc) * np.float64(np.float32(ks))
    Vf = dec(vc) * np.float64(np.float32(vs))
    G = H // Hk
    for b in range(B):
        pos = np.arange(ctx[b])
        blk = bt[b, pos // bs]
        for h in range(H):
            K = Kf[blk, pos % bs, h // G]
            V = Vf[blk, pos % bs, h // G]
            s = scale * (K @ q[b, h].astype(np.float64))
            w = np.exp(s - s.max())
            w /= w.sum()
            np.testing.assert_allclose(got[b, h], w @ V, rtol=0, atol=1e-12)


def test_attention_fp8_equals_float_cache_attention_for_power_of_two_scales():
    """With power-of-two scales every dequantised element is exact in float32, so
    the fp8 attention must equal the float attention over those float32 values
    bit for bit (same summation order)."""
    rng = np.random.default_rng(8105)
    B, H, Hk, D, bs, NB = 2, 8, 2, 32, 8, 10
    ctx = np.array([13, 40], dtype=np.int32)
    bt = rng.permutation(NB)[: 2 * 5].reshape(2, 5).astype(np.int32)
    kc = _finite_codes(rng, (NB, bs, Hk, D))
    vc = _finite_codes(rng, (NB, bs, Hk, D))
    q = rng.normal(size=(B, H, D)).astype(np.float32)
    ks, vs = 2.0 ** -5, 2.0 ** -3
    got = oracle.paged_attention_fp8(q, kc, vc, bt, ctx, 0.125, ks, vs, "f32")
    kf = (oracle.e4m3_to_float64(kc) * ks).astype(np.float32)
    vf = (oracle.e4m3_to_float64(vc) * vs).astype(np.float32)
    ref = oracle.paged_attention(q, kf, vf, bt, ctx, 0.125, "f32")
    np.testing.assert_array_equal(got, ref)


def test_attention_fp8_single_token_is_dequantised_v():
    rng = np.random.default_rng(8106)
    kc = _finite_codes(rng, (2, 4, 1, 8))
    vc = _finite_codes(rng, (2, 4, 1, 8))
    q = rng.normal(size=(1, 2, 8)).astype(np.float32)
    got = oracle.paged_attention_fp8(q, kc, vc, np.array([[1, 0]], np.int32), np.array([1], np.int32),
                                     1.0, 0.5, 0.75, "f32")
    want = oracle.e4m3_to_float64(vc[1, 0, 0]) * 0.75
    np.testing.assert_array_equal(got[0, 0], want)
    np.testing.assert_array_equal(got[0, 1], want)

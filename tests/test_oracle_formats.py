"""Pins for oracle.formats: the narrow-format encoders and decoders.

Each check below is independent of the encoder under test: code-table
round trips, hand-listed rounding ties, a second encoder built on a different
method (nearest decoded value), and torch's own float8 conversions.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F

FMTS = ["e4m3", "e5m2", "e2m1"]


def _finite_codes(fmt):
    p = F.FORMATS[fmt]
    nb = p["nbits"]
    codes = np.arange(1 << nb)
    vals = F.decode(codes, fmt)
    return codes[np.isfinite(vals)], vals[np.isfinite(vals)]


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_known_values(fmt):
    # largest finite, smallest subnormal, and 1.0 for each format (OFP8 / OCP MX tables)
    expect = {
        "e4m3": {0x7E: 448.0, 0x01: 2.0 ** -9, 0x38: 1.0, 0x08: 2.0 ** -6, 0x78: 256.0, 0xFE: -448.0},
        "e5m2": {0x7B: 57344.0, 0x01: 2.0 ** -16, 0x3C: 1.0, 0x04: 2.0 ** -14},
        "e2m1": {0x1: 0.5, 0x2: 1.0, 0x3: 1.5, 0x4: 2.0, 0x5: 3.0, 0x6: 4.0, 0x7: 6.0, 0xF: -6.0},
    }[fmt]
    for c, v in expect.items():
        assert F.decode(np.array([c]), fmt)[0] == v, (fmt, hex(c))
    if fmt == "e4m3":
        assert np.isnan(F.decode(np.array([0x7F, 0xFF]), fmt)).all()
    if fmt == "e5m2":
        assert F.decode(np.array([0x7C]), fmt)[0] == np.inf
        assert np.isnan(F.decode(np.array([0x7D, 0x7E, 0x7F]), fmt)).all()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("enc", [F.encode, F.encode_table])
def test_roundtrip_every_code(fmt, enc):
    codes, vals = _finite_codes(fmt)
    got = enc(vals.astype(np.float32), fmt)
    np.testing.assert_array_equal(got, codes.astype(np.uint8))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("enc", [F.encode, F.encode_table])
def test_every_midpoint_ties_to_even_and_neighbours(fmt, enc):
    p = F.FORMATS[fmt]
    codes = np.arange(p["max_code"] + 1)
    vals = F.decode(codes, fmt)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)  # midpoints exact in fp32
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    np.testing.assert_array_equal(enc(mids, fmt), even.astype(np.uint8))
    below = np.nextafter(mids, np.float32(-np.inf))
    above = np.nextafter(mids, np.float32(np.inf))
    np.testing.assert_array_equal(enc(below, fmt), codes[:-1].astype(np.uint8))
    np.testing.assert_array_equal(enc(above, fmt), codes[1:].astype(np.uint8))
    sign = 1 << (p["nbits"] - 1)
    np.testing.assert_array_equal(enc(-mids, fmt), (even | sign).astype(np.uint8))


def test_hand_listed_cases():
    e = lambda v, f: int(F.encode(np.array([v], dtype=np.float32), f)[0])  # noqa: E731
    # E4M3: saturation, infinities, NaN, signed zero, subnormal ties
    assert e(448.0, "e4m3") == 0x7E
    assert e(464.0, "e4m3") == 0x7E          # midpoint 448|480 -> even mantissa 110 = 448
    assert e(1e30, "e4m3") == 0x7E
    assert e(np.inf, "e4m3") == 0x7E and e(-np.inf, "e4m3") == 0xFE
    assert e(np.nan, "e4m3") == 0x7F
    assert e(-0.0, "e4m3") == 0x80 and e(0.0, "e4m3") == 0x00
    assert e(2.0 ** -9, "e4m3") == 0x01
    assert e(2.0 ** -10, "e4m3") == 0x00      # half of the smallest subnormal ties to 0
    assert e(np.nextafter(np.float32(2.0 ** -10), np.float32(1)), "e4m3") == 0x01
    assert e(3 * 2.0 ** -10, "e4m3") == 0x02  # 1.5 quanta ties to 2 quanta (even)
    assert e(1e-30, "e4m3") == 0x00 and e(-1e-30, "e4m3") == 0x80
    # E5M2
    assert e(57344.0, "e5m2") == 0x7B
    assert e(61440.0, "e5m2") == 0x7B         # tie towards 65536 (even) then saturate
    assert e(np.inf, "e5m2") == 0x7B
    assert e(2.0 ** -17, "e5m2") == 0x00 and e(2.0 ** -16, "e5m2") == 0x01
    # E2M1 ties: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    for v, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (7.0, 7),
                 (100.0, 7), (-5.0, 0xE), (-0.0, 0x8), (0.2, 0), (0.26, 1)]:
        assert e(v, "e2m1") == c, (v, c)


def _structured_inputs(seed=0):
    """Every sign x fp32 exponent x top-12 mantissa bits, with 4 patterns of the low 11 bits.

    For these formats the rounding decision only depends on the sign, the
    exponent, the mantissa bits down to the round bit (at most 12 bits deep,
    reached by the deepest subnormal of E4M3) and whether any lower bit is set,
    so this set exercises every distinct decision.
    """
    s = np.arange(2, dtype=np.uint32)[:, None, None, None]
    e = np.arange(256, dtype=np.uint32)[None, :, None, None]
    m = np.arange(4096, dtype=np.uint32)[None, None, :, None]
    low = np.array([0, 1, 0x2AA, 0x7FF], dtype=np.uint32)[None, None, None, :]
    bits = (s << 31) | (e << 23) | (m << 11) | low
    bits = bits.reshape(-1)
    rng = np.random.default_rng(seed)
    rnd = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([bits, rnd]).view(np.float32)


@pytest.mark.parametrize("fmt", FMTS)
def test_bit_method_equals_table_method(fmt):
    x = _structured_inputs()
    if fmt == "e2m1":
        x = x[~np.isnan(x)]  # NaN is outside the E2M1 contract
    a = F.encode(x, fmt)
    b = F.encode_table(x, fmt)
    bad = np.nonzero(a != b)[0]
    assert bad.size == 0, [(float(x[i]), hex(x[i:i+1].view(np.uint32)[0]), int(a[i]), int(b[i])) for i in bad[:5]]


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_matches_torch_float8_in_range(fmt, tdt):
    x = _structured_inputs(1)
    x = x[np.isfinite(x) & (np.abs(x) <= F.FMAX[fmt])]
    ours = F.encode(x, fmt)
    theirs = torch.from_numpy(x.copy()).to(tdt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, theirs)


def test_ue4m3_and_e8m0():
    assert int(F.encode_ue4m3(np.array([448.0], np.float32))[0]) == 0x7E
    assert int(F.encode_ue4m3(np.array([1000.0], np.float32))[0]) == 0x7E
    assert F.decode_ue4m3(np.array([0x38]))[0] == 1.0
    np.testing.assert_array_equal(F.decode_e8m0(np.array([0, 127, 254])), [2.0 ** -127, 1.0, 2.0 ** 127])
    assert np.isnan(F.decode_e8m0(np.array([255]))[0])
    with pytest.raises(AssertionError):
        F.encode_ue4m3(np.array([-1.0], np.float32))


def test_floor_log2_exact():
    vals = np.array([1.0, 1.5, 2.0, 3.999, 4.0, 2.0 ** -126, 2.0 ** -149, 3.0 * 2.0 ** -140, 3.4e38], np.float32)
    exp = [0, 0, 1, 1, 2, -126, -149, -139, 127]
    np.testing.assert_array_equal(F.floor_log2(vals), exp)


def test_bf16_helpers():
    x = torch.tensor([1.0, -2.5, 3.140625, 1e-40, 65280.0], dtype=torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(F.bf16_bits_to_f32(bits), x.float().numpy())
    y = np.array([1.0, 1.00390625, 1.01171875, -3.3], np.float64)
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(F.f64_to_bf16_bits(y), ref)

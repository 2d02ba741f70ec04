"""Pins of the oracle's element formats (E2M1, E4M3, E8M0, MX block scaling).

Each check compares the oracle with something other than itself: the bit-field definition of a
format, a brute-force nearest-value search over all codes, exact round trips, or values worked out
by hand.  Formats follow the OCP Microscaling (MX) v1.0 definitions named by the pages' "MXFP4 with
per-32 E8M0 scales" (TensorSharp page, "Getting a drafter"; model card glossary).
"""
import math

import numpy as np
import pytest

import oracle


def _e2m1_bits(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def _e4m3_bits(b):
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return math.nan
    v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e2m1_decode_all_codes():
    for c in range(16):
        assert oracle.e2m1_value(c) == _e2m1_bits(c)
    assert [oracle.e2m1_value(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_decode_all_codes():
    for b in range(256):
        want = _e4m3_bits(b)
        got = oracle.e4m3_value(b)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want, b
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e8m0_decode():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))


def _nearest_even(v, values_by_code, max_mag):
    """Brute-force round-to-nearest over every non-negative finite code; ties go to the code with
    an even mantissa (code LSB 0); magnitudes at or beyond the largest finite value saturate."""
    a = abs(v)
    if a >= max_mag:
        return [c for c, val in values_by_code if val == max_mag][0]
    cands = [(abs(val - a), c) for c, val in values_by_code if val >= 0]
    best = min(dist for dist, _ in cands)
    tied = [c for dist, c in cands if dist == best]
    if len(tied) > 1:
        tied = [c for c in tied if c % 2 == 0]
    assert len(tied) == 1
    return tied[0]


def test_e4m3_encode_matches_brute_force():
    finite = [(b, _e4m3_bits(b)) for b in range(128) if not math.isnan(_e4m3_bits(b))]
    vals = sorted(set(v for _, v in finite))
    probes = set()
    for i in range(len(vals) - 1):
        lo, hi = vals[i], vals[i + 1]
        probes.update([lo, hi, (lo + hi) / 2, lo + (hi - lo) * 0.25, lo + (hi - lo) * 0.75,
                       math.nextafter((lo + hi) / 2, 0), math.nextafter((lo + hi) / 2, 1e9)])
    rng = np.random.default_rng(1)
    probes.update(float(v) for v in rng.uniform(0, 500, 2000))
    probes.update([448.0, 460.0, 464.0, 480.0, 1e6, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11])
    probes = sorted(probes)
    got = oracle.e4m3_encode(np.array(probes + [-p for p in probes]))
    for i, p in enumerate(probes):
        want = _nearest_even(p, finite, 448.0)
        assert got[i] == want, (p, got[i], want)
        neg = got[len(probes) + i]
        assert neg == (want | 0x80), (p, neg)


def test_e4m3_encode_signed_zero_and_saturation():
    out = oracle.e4m3_encode(np.array([0.0, -0.0, -2.0 ** -12, 2.0 ** -12, 1e30, -1e30]))
    assert list(out) == [0x00, 0x80, 0x80, 0x00, 0x7E, 0xFE]


def test_e2m1_encode_matches_brute_force_and_listed_ties():
    finite = [(c, _e2m1_bits(c)) for c in range(8)]
    grid = [v for _, v in finite]
    probes = set(grid)
    for i in range(len(grid) - 1):
        lo, hi = grid[i], grid[i + 1]
        probes.update([(lo + hi) / 2, math.nextafter((lo + hi) / 2, 0), math.nextafter((lo + hi) / 2, 9), lo + (hi - lo) / 3])
    probes.update([6.5, 7.0, 100.0])
    for p in sorted(probes):
        assert oracle.e2m1_encode(p) == _nearest_even(p, finite, 6.0), p
        assert oracle.e2m1_encode(-p) == (_nearest_even(p, finite, 6.0) | 8), p
    # ties in round-to-nearest-even: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    for v, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0), (5.0, 4.0)]:
        assert oracle.e2m1_value(oracle.e2m1_encode(v)) == want


def test_mx_scale_exponent():
    # floor(log2 amax) - emax, clamped to [-127, 127]; all-zero block -> -127
    assert oracle.mx_scale_exp(0.0, 8) == -127
    for j in range(-20, 21):
        assert oracle.mx_scale_exp(2.0 ** j, 8) == j - 8
        assert oracle.mx_scale_exp(2.0 ** j * 1.999, 2) == j - 2
        assert oracle.mx_scale_exp(math.nextafter(2.0 ** j, 0), 8) == j - 9
    assert oracle.mx_scale_exp(2.0 ** -140, 8) == -127
    assert oracle.mx_scale_exp(1e300, 2) == 127


def test_mxfp8_block_hand_worked():
    # block amax 3.0 -> floor(log2 3) = 1 -> exponent 1 - 8 = -7 (byte 120); elements times 2^7:
    # 3.0 -> 384 (E4M3 exact: 1.5 * 2^8); 1.1 -> 140.8 -> quantum 16 in [128, 256): 8.8 -> 9 -> 144;
    # -0.01 -> -1.28 -> quantum 0.125 in [1, 2): 10.24 -> 10 -> -1.25; 0 -> 0.
    v = np.zeros(32)
    v[:4] = [3.0, 1.1, -0.01, 0.0]
    q, s = oracle.mxfp8_quantize(v)
    assert s[0] == 120
    deq = oracle.mxfp8_dequantize(q, s)
    assert list(deq[:4] * 2 ** 7) == [384.0, 144.0, -1.25, 0.0]
    assert q[0] == ((8 + 7) << 3) | 4  # 384 = 1.5 * 2^8


def test_mxfp8_relative_error_bound():
    # E4M3 has 3 mantissa bits: inside a block, every value between 2^-6 and 448 times the block
    # scale keeps relative error <= 2^-4; values above 448 times the scale (possible because the
    # block maximum lies in [256, 512) times the scale) saturate to exactly +-448 times the scale.
    rng = np.random.default_rng(7)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    q, s = oracle.mxfp8_quantize(v)
    deq = oracle.mxfp8_dequantize(q, s)
    scale = np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    amax = np.repeat(np.abs(v).reshape(64, 8, 32).max(axis=2), 32, axis=1)
    assert np.all((amax >= 256 * scale) & (amax < 512 * scale))
    sat = np.abs(v) > 448 * scale
    mid = (np.abs(v) >= 2.0 ** -6 * scale) & ~sat
    rel = np.abs(deq - v)[mid] / np.abs(v)[mid]
    assert rel.max() <= 2.0 ** -4 + 1e-15
    assert sat.any() and np.array_equal(deq[sat], np.sign(v[sat]) * 448 * scale[sat])


def test_mxfp4_round_trip():
    rng = np.random.default_rng(3)
    n_blocks = 4096
    codes = rng.integers(0, 256, (n_blocks, 16), dtype=np.uint8)
    # make every block's maximum magnitude 4 or 6, the only maxima for which the scale is recovered
    top = rng.choice(np.array([0x6, 0x7, 0xE, 0xF], dtype=np.uint8), n_blocks)
    codes[:, 0] = (codes[:, 0] & 0xF0) | top
    scales = rng.integers(100, 150, (n_blocks, 1), dtype=np.uint8)
    v = oracle.mxfp4_dequantize(codes.reshape(1, -1), scales.reshape(1, -1)).reshape(n_blocks, 32)
    c2, s2 = oracle.mxfp4_quantize(v)
    # -0 and +0 decode equal; compare values, then codes modulo the sign of zero
    assert np.array_equal(s2, scales)
    v2 = oracle.mxfp4_dequantize(c2.reshape(1, -1), s2.reshape(1, -1)).reshape(n_blocks, 32)
    assert np.array_equal(v2, v)
    lo_a, hi_a = codes & 15, codes >> 4
    lo_b, hi_b = c2 & 15, c2 >> 4
    norm = lambda c: np.where(c == 8, 0, c)
    assert np.array_equal(norm(lo_a), norm(lo_b)) and np.array_equal(norm(hi_a), norm(hi_b))


def test_mxfp4_values_already_on_grid_are_unchanged():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, (1, 512), dtype=np.uint8)
    scales = rng.integers(110, 140, (1, 32), dtype=np.uint8)
    v = oracle.mxfp4_dequantize(codes, scales)
    c2, s2 = oracle.mxfp4_quantize(v)
    assert np.array_equal(oracle.mxfp4_dequantize(c2, s2), v)


@pytest.mark.parametrize("h", [0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049])
def test_bf16_decode(h):
    import struct
    assert oracle.bf16_value(h) == struct.unpack("<f", struct.pack("<I", h << 16))[0]


def test_bf16_encode_round_trip_and_ties():
    h = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):  # the NaN patterns
        v = (h << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(v)
    enc = oracle.bf16_encode(v[finite])
    # every finite bf16 value encodes to itself (-0 too)
    assert np.array_equal(enc, h[finite].astype(np.uint16))
    # half-way between consecutive positive normals: ties go to the even mantissa
    lo = np.arange(0x0080, 0x7F7F, dtype=np.uint32)
    a = (lo << 16).view(np.float32).astype(np.float64)
    b = ((lo + 1) << 16).view(np.float32).astype(np.float64)
    mid = (a + b) / 2  # exact in fp64
    got = oracle.bf16_encode(mid)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, want)
    # just above / below the midpoint
    assert np.array_equal(oracle.bf16_encode(mid + (b - a) * 1e-6), (lo + 1).astype(np.uint16))
    assert np.array_equal(oracle.bf16_encode(mid - (b - a) * 1e-6), lo.astype(np.uint16))
    # negative values mirror positive ones
    assert np.array_equal(oracle.bf16_encode(-mid), want | 0x8000)


def test_stack_step_adds_then_rounds_once():
    x = oracle.bf16_encode(np.array([1.0, -2.0, 3.5]))
    # bf16 spacing at 1 is 2^-7: 1 + 2^-8 lies half-way between 1 and 1 + 2^-7 and ties to the even 1
    y = np.array([2.0 ** -8, 0.25, -3.5])
    got = oracle.stack_step(x, y)
    assert np.array_equal(got, oracle.bf16_encode(np.array([1.0 + 2.0 ** -8, -1.75, 0.0])))
    assert got[0] == 0x3F80 and got[2] == 0


def _block(scale, elems, split):
    """A 17-byte block from 32 element codes, written element by element (test helper)."""
    q = np.zeros(16, dtype=np.uint8)
    for e, c in enumerate(elems):
        byte, high = (e % 16, e >= 16) if split else (e // 2, e % 2 == 1)
        q[byte] |= (c & 0xF) << (4 if high else 0)
    return np.concatenate([[scale], q]).astype(np.uint8)


@pytest.mark.parametrize("split", [False, True])
def test_mx_blocks_unpack_places_every_element(split):
    rng = np.random.default_rng(3)
    elems = rng.integers(0, 16, size=(5, 32))
    scales = rng.integers(0, 256, size=5)
    blocks = np.stack([_block(s, e, split) for s, e in zip(scales, elems)])
    codes, sc = oracle.mx_blocks_unpack(blocks, split)
    assert np.array_equal(sc, scales.astype(np.uint8))
    # canonical: element 2i in the low nibble of byte i
    assert np.array_equal(codes & 0xF, elems[:, 0::2]) and np.array_equal(codes >> 4, elems[:, 1::2])
    # the values the codes stand for: E2M1 table times 2^(scale - 127)
    v = oracle.mxfp4_dequantize(codes, sc[:, None])
    want = np.array([[oracle.e2m1_value(int(c)) for c in row] for row in elems]) * 2.0 ** (scales[:, None] - 127.0)
    assert np.array_equal(v, want)


def test_mx_blocks_unpack_hand_worked():
    # one block, scale 2^1: elements 0..31 = codes 0..15, 0..15; split order puts element i and i+16 in byte i
    elems = list(range(16)) * 2
    blk = _block(128, elems, True)
    assert blk[1] == 0x00 and blk[2] == 0x11 and blk[16] == 0xFF
    codes, sc = oracle.mx_blocks_unpack(blk[None], True)
    assert sc[0] == 128 and codes[0, 0] == 0x10 and codes[0, 7] == 0xFE and codes[0, 8] == 0x10

"""Pins of the oracle's scalar conversions against definitions and libraries.

BF16 and E4M3 rounding are checked against PyTorch's own casts (independent
implementations of the same IEEE/OCP definitions); the UE8M0 scale against
its defining property; the 128x4 layout against hand-worked offsets and a
bijection check.
"""
import numpy as np
import pytest
import torch

from conftest import golden_lines


def test_bf16_widening_is_exact_all_patterns(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    keep = ~np.isnan(ref)                      # NaN payloads are not compared
    ours = np.array([oracle_lib.bf16_to_f32(b) for b in bits[keep]], np.float32)
    assert np.array_equal(ours.view(np.uint32), ref[keep].view(np.uint32))


def test_bf16_rounding_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    words = rng.integers(0, 1 << 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    # add every tie pattern and carries into the exponent / into inf
    ties = (rng.integers(0, 1 << 16, 20000, dtype=np.uint32) << 16) | 0x8000
    edge = np.array([0x7f7fffff, 0x7f7f8000, 0x3f80ffff, 0x3f818000, 0x3f808000,
                     0x00008000, 0x00018000, 0x80000000, 0x00000000, 0x7f800000],
                    np.uint32)
    words = np.concatenate([words, ties, edge])
    vals = words.view(np.float32)
    finite = np.isfinite(vals)
    vals = vals[finite]
    ours = oracle_lib.f32_to_bf16_array(vals)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_decode_all_codes(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle_lib.e4m3_to_f64(c) for c in codes])
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    # every finite BF16 value times every power of two a UE8M0 inverse scale
    # can take, restricted to the E4M3 range (torch turns overflow into NaN,
    # the MXFP8 reading saturates instead: tested separately).
    bits = np.arange(1 << 16, dtype=np.uint32)
    base = (bits << 16).view(np.float32)
    base = base[np.isfinite(base)]
    chunks = []
    for e in range(0, 255, 1):
        v = np.clip(base.astype(np.float64) * 2.0 ** (127 - e), -1e30, 1e30).astype(np.float32)
        chunks.append(v[np.abs(v) <= 448.0])
    vals = np.unique(np.concatenate(chunks))
    ours = oracle_lib.f32_to_e4m3_array(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref), int((ours != ref).sum())


def test_e4m3_ties_go_to_even(oracle_lib):
    codes = np.arange(0, 0x7e, dtype=np.uint8)
    vals = np.array([oracle_lib.e4m3_to_f64(c) for c in codes])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)
    got = oracle_lib.f32_to_e4m3_array(mids)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, even)


def test_e4m3_saturates(oracle_lib):
    for v, code in ((449.0, 0x7e), (464.0, 0x7e), (1e30, 0x7e), (float("inf"), 0x7e),
                    (-500.0, 0xfe), (-0.0, 0x80), (2.0 ** -11, 0x00), (2.0 ** -10 * 1.01, 0x01)):
        assert oracle_lib.f32_to_e4m3(v) == code, v


def test_ue8m0_is_smallest_power_of_two_at_or_above(oracle_lib):
    from fractions import Fraction
    rng = np.random.default_rng(2)
    amax = np.concatenate([
        (rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)),
        448.0 * 2.0 ** np.arange(-120, 120), [1.0, 448.0, 450.0, 1e-38, 3.3e38]])
    inv448 = Fraction(float(np.float32(1.0) / np.float32(448.0)))
    for a in np.abs(amax).astype(np.float32):
        if a == 0:
            continue
        s = Fraction(float(np.float32(a) * np.float32(inv448)))
        e = oracle_lib.ue8m0_of_amax(float(a))
        assert 0 <= e <= 254
        assert Fraction(2) ** (e - 127) >= s or e == 254
        assert e == 0 or Fraction(2) ** (e - 128) < s
    assert oracle_lib.ue8m0_of_amax(0.0) == 0


def test_scaled_block_max_lands_in_upper_half_of_e4m3(oracle_lib):
    # With the scale rounded up, the block maximum maps into (224, 448]: the
    # scale is never so large that the top binade of E4M3 goes unused.
    rng = np.random.default_rng(3)
    for a in np.abs(rng.standard_normal(2000) * 10.0 ** rng.integers(-20, 20, 2000)):
        a = float(np.float32(a))
        if a < 1e-30:
            continue
        e = oracle_lib.ue8m0_of_amax(a)
        scaled = a * 2.0 ** (127 - e)
        assert 224.0 < scaled <= 448.0 * (1 + 2 ** -20), (a, e, scaled)


def test_swizzle_golden(oracle_lib):
    for lhs, rhs in golden_lines("swizzle_128x4.txt"):
        row, col, cols = map(int, lhs)
        assert oracle_lib.swizzle_128x4(row, col, cols) == int(rhs), lhs


@pytest.mark.parametrize("m,hidden", [(256, 6144), (300, 128), (1, 256), (129, 512)])
def test_swizzle_is_a_bijection(oracle_lib, m, hidden):
    cols = hidden // 32
    rows = (m + 127) // 128 * 128
    size = oracle_lib.mxfp8_scale_bytes(m, hidden)
    assert size == rows * ((cols + 3) // 4 * 4)
    seen = np.zeros(size, np.int32)
    for r in range(rows):
        for c in range((cols + 3) // 4 * 4):
            seen[oracle_lib.swizzle_128x4(r, c, cols)] += 1
    assert (seen == 1).all()

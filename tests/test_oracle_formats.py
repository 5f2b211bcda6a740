"""Pins of the oracle's storage-format conversions against library routines and the format
definitions (bfloat16, IEEE binary16, OCP OFP8 E4M3).

Every rounding the oracle performs goes through these conversions, so a wrong tie rule,
a dropped subnormal range or a wrong overflow threshold shows up here first.
"""
import numpy as np
import pytest
import torch


def _edge_floats():
    g = np.random.default_rng(7)
    mags = g.standard_normal(200_000).astype(np.float32)
    scales = np.float32(2.0) ** g.integers(-149, 128, 200_000).astype(np.float32)
    with np.errstate(over="ignore"):
        vals = (mags * scales).astype(np.float32)
    # every binary32 tie and near-tie pattern for a 16-bit target: low bits around the
    # half-way point of the dropped part
    base = g.integers(0, 2**31, 20_000, dtype=np.uint64).astype(np.uint32)
    ties16 = (base & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    near16 = np.concatenate([ties16, ties16 + 1, ties16 - 1])
    ties13 = (base & np.uint32(0xFFFFE000)) | np.uint32(0x1000)
    near13 = np.concatenate([ties13, ties13 + 1, ties13 - 1])
    specials = np.array([0.0, -0.0, 1.0, -1.0, 65504, 65519.99, 65520, 65536, 6.1e-5, 6.0e-8,
                         5.96e-8, 2.98e-8, 1e-45, 3.3895e38, 3.4028235e38, np.inf, -np.inf],
                        dtype=np.float32)
    return np.concatenate([vals, near16.view(np.float32), near13.view(np.float32), specials])


def test_bf16_rounding_matches_torch(orc):
    f = _edge_floats()
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bits(f, "bf16")
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"first mismatch at {f[bad[0]]!r}: {got[bad[0]]:#06x} vs {ref[bad[0]]:#06x}"


def test_fp16_rounding_matches_numpy(orc):
    f = _edge_floats()
    f = f[~np.isnan(f)]
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = orc.f32_to_bits(f, "fp16")
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"first mismatch at {f[bad[0]]!r}: {got[bad[0]]:#06x} vs {ref[bad[0]]:#06x}"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_16bit_decode_exhaustive(orc, dtype):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    ref = torch.from_numpy(allbits.view(np.int16)).view(tdt).float().numpy()
    got = orc.bits_to_f32(allbits, dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f64_to_16bit_rounds_once(orc):
    # 1 + 2^-8 is the bf16 tie between 1 and 1 + 2^-7; a binary64 value just above it must
    # round up.  Going through binary32 first would land exactly on the tie and round to 1.
    x = 1.0 + 2.0**-8 + 2.0**-40
    assert orc.f64_to_bits(x, "bf16") == 0x3F81
    assert orc.f64_to_bits(1.0 + 2.0**-8, "bf16") == 0x3F80          # exact tie -> even
    assert orc.f64_to_bits(1.0 + 3 * 2.0**-8, "bf16") == 0x3F82      # tie -> even (up)
    # binary16: tie between 1 and 1 + 2^-10 is 1 + 2^-11
    assert orc.f64_to_bits(1.0 + 2.0**-11 + 2.0**-40, "fp16") == 0x3C01
    assert orc.f64_to_bits(1.0 + 2.0**-11, "fp16") == 0x3C00


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = orc.e4m3_to_f32(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0**-9            # smallest subnormal
    assert got[0x08] == 2.0**-6            # smallest normal


def test_e4m3_round_trip_every_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = orc.e4m3_to_f32(codes)
    back = orc.f32_to_e4m3(vals)
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch_in_range(orc):
    # torch's e4m3fn cast rounds to nearest even and only differs from the saturating form
    # above 464 (where it returns NaN); below that both must agree everywhere, including
    # every midpoint between neighbouring codes.
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    grid = orc.e4m3_to_f32(codes).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    g = np.random.default_rng(3)
    rnd = np.abs(g.standard_normal(300_000) * 2.0 ** g.integers(-12, 9, 300_000))
    cand = np.concatenate([grid, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), rnd,
                           [448.0, 450.0, 463.99, 464.0]]).astype(np.float32)
    cand = cand[cand <= 464.0]
    cand = np.concatenate([cand, -cand])
    ref = torch.from_numpy(cand).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.f32_to_e4m3(cand)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"first mismatch at {cand[bad[0]]!r}: {got[bad[0]]:#04x} vs {ref[bad[0]]:#04x}"


def test_e4m3_saturates(orc):
    big = np.array([448 * (1 + 2**-4), 464.0001, 480, 1e6, 3e38, np.inf], np.float32)
    assert (orc.f32_to_e4m3(big) == 0x7E).all()
    assert (orc.f32_to_e4m3(-big) == 0xFE).all()
    assert orc.f32_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    # below half the smallest subnormal flushes to zero; the half-way point ties to 0
    assert list(orc.f32_to_e4m3(np.array([2.0**-11, 2.0**-10, 2.0**-10 * 1.01], np.float32))) == [0, 0, 1]

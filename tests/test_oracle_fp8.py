"""Pins for the oracle's FP8-E4M3 codec (T2 tier), against things other than itself:
torch's float8_e4m3fn dtype (a library routine), hand-worked codes from the format
definition (tests/golden/fp8_e4m3_cases.txt) and the format's rounding bound."""
import os

import numpy as np
import pytest
import torch

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_e4m3_cases.txt")


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_table_matches_library():
    ref = torch_decode_all()
    ours = fp8.DECODE_TABLE
    nan_ref, nan_ours = np.isnan(ref), np.isnan(ours)
    assert np.array_equal(nan_ref, nan_ours)
    assert sorted(np.nonzero(nan_ours)[0].tolist()) == [0x7F, 0xFF]
    assert np.array_equal(ref[~nan_ref], ours[~nan_ours])
    # signed zero is kept
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_golden_codes():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    vals = np.array([float(r[0]) for r in rows], dtype=np.float32)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    assert np.array_equal(fp8.encode(vals), want)


def test_encode_matches_library_on_all_midpoints_and_codes():
    pos = fp8.DECODE_TABLE[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2.0           # exactly representable in fp32
    vals = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                           [464.0]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(vals), ref)


def test_encode_matches_library_on_random_values():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-464, 464, 20000),
                           rng.standard_normal(20000) * 0.01,
                           rng.standard_normal(20000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(vals), ref)


def test_saturation_beyond_max():
    vals = np.array([465.0, 480.0, 1e6, 3.0e38, -465.0, -1e30], dtype=np.float32)
    assert fp8.encode(vals).tolist() == [0x7E] * 4 + [0xFE] * 2


def test_encode_rejects_nonfinite():
    with pytest.raises(ValueError):
        fp8.encode(np.array([np.inf], dtype=np.float32))


def test_quantise_row_amax_maps_to_448_and_error_bound():
    rng = np.random.default_rng(2)
    for d in (64, 128):
        for trial in range(50):
            x = torch.from_numpy(rng.standard_normal(d).astype(np.float32) *
                                 (20.0 if trial % 3 == 0 else 1.0)).to(torch.bfloat16).float().numpy()
            codes, scale = fp8.quantise_row(x)
            assert scale.dtype == np.float32
            amax = np.float32(np.abs(x).max())
            assert scale == np.float32(amax / np.float32(448.0))
            j = int(np.argmax(np.abs(x)))
            assert codes[j] & 0x7F == 0x7E              # amax lands on +-448 exactly
            deq = fp8.dequantise_row(codes, scale)
            # round-to-nearest in E4M3: relative error <= 2^-4 for normal codes,
            # absolute error <= 2^-10 * scale in the subnormal range, plus the fp32
            # rounding of x/scale (<= 2^-24 relative).
            y = np.abs(x / np.float64(scale))
            bound = np.where(y >= 2.0 ** -6, y * (2.0 ** -4), 2.0 ** -10) * (1 + 2.0 ** -20)
            assert np.all(np.abs(x / np.float64(scale) - deq / np.float64(scale)) <= bound + 1e-12)


def test_quantise_zero_row():
    codes, scale = fp8.quantise_row(np.zeros(64, dtype=np.float32))
    assert scale == np.float32(1.0) and not codes.any()
    assert not fp8.dequantise_row(codes, scale).any()

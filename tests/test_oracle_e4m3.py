"""Oracle pins: the E4M3 codec against PyTorch's float8_e4m3fn and the format's
closed-form values."""
import numpy as np
import torch

from oracle import e4m3


def test_decode_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3.decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_closed_form_values():
    assert e4m3.decode_code(0x7E) == 448.0            # largest finite
    assert e4m3.decode_code(0x01) == 2.0 ** -9        # smallest subnormal
    assert e4m3.decode_code(0x08) == 2.0 ** -6        # smallest normal
    assert e4m3.decode_code(0x38) == 1.0              # exponent 7 = bias
    assert e4m3.decode_code(0xB8) == -1.0
    assert np.isnan(e4m3.decode_code(0x7F)) and np.isnan(e4m3.decode_code(0xFF))
    assert np.sum(np.isnan(e4m3.DECODE_TABLE)) == 2   # no infinities, two NaNs


def _all_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    return bits.view(np.float32)


def _f64(x):
    with np.errstate(invalid="ignore"):   # signalling-NaN payloads
        return x.astype(np.float64)


def test_encode_every_bf16_value_matches_torch_in_range():
    x = _all_bf16_as_f32()
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3.encode(_f64(x))
    # torch turns magnitudes above 464 (the tie point between 448 and the
    # next binade) into NaN; the cache saturates them to 448 instead.
    finite_in_range = np.isfinite(x) & (np.abs(x) <= 464.0)
    assert np.array_equal(got[finite_in_range], ref[finite_in_range])
    big = np.isfinite(x) & (np.abs(x) > 464.0)
    assert np.all((got[big] & 0x7F) == 0x7E)
    assert np.all(got[np.isnan(x)] == e4m3.NAN_CODE)
    assert np.all((got[np.isinf(x)] & 0x7F) == 0x7E)


def test_encode_random_fp32_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200_000).astype(np.float32) * s
                        for s in (1e-3, 1e-1, 1.0, 30.0, 300.0)])
    x = x[np.abs(x) <= 464.0]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x.astype(np.float64)), ref)


def test_round_trip_and_ties_to_even():
    vals = e4m3.DECODE_TABLE[~np.isnan(e4m3.DECODE_TABLE)]
    codes = e4m3.encode(vals)
    assert np.array_equal(e4m3.decode(codes), vals)
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39)
    assert e4m3.encode(np.array([1.0625]))[0] == 0x38
    # 1.125 + 1/16 lies halfway between 0x39 (odd) and 1.25 (0x3A, even)
    assert e4m3.encode(np.array([1.1875]))[0] == 0x3A


def test_quantize_uses_fp32_product():
    x = np.array([1.0, -2.5, 3.0e-3], dtype=np.float32)
    inv = np.float32(1.0) / np.float32(0.0137)
    prod = x * inv
    assert np.array_equal(e4m3.quantize_fp32(x, float(inv)), e4m3.encode(prod.astype(np.float64)))

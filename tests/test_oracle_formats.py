"""Pins of the oracle's number formats (bf16, E4M3, E8M0, MXFP8 blocks).

E4M3 and E8M0 follow the OCP 8-bit floating point / Microscaling (MX) definitions named by the
pages' "MXFP8" mode ("Cursor Open-Sources Mixture-of-Kittens (MoK) ...", English summary; the
"Mixture-of-Kittens (MoK)" project card, "Key concepts": weights pre-quantised with
ops.mxfp8_quantize).  The oracle's encoder is a brute-force nearest-value search; it is pinned
here against torch's CPU float8_e4m3fn conversion (a library routine), closed-form cases and
numpy's frexp for the shared exponent.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_bf16_value_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    for b in (0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x8000):
        assert oracle.bf16_value(b) == got[b] or (math.isnan(got[b]))


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
            if ref[c] == 0.0:
                assert math.copysign(1.0, v) == math.copysign(1.0, ref[c])


@pytest.mark.parametrize("v,code", [
    (448.0, 0x7E),            # largest finite: 1.75 * 2^8
    (1.0, 0x38),              # exponent field 7 (bias 7), mantissa 0
    (0.5, 0x30),
    (2.0 ** -9, 0x01),        # smallest subnormal: 1/8 * 2^-6
    (2.0 ** -10, 0x00),       # halfway between 0 and 2^-9: tie -> even (0)
    (3 * 2.0 ** -10, 0x02),   # halfway between 2^-9 (odd code) and 2^-8 (even code)
    (1.0625, 0x38),           # halfway between 1.0 and 1.125: tie -> even mantissa
    (1.1875, 0x3A),           # halfway between 1.125 and 1.25: tie -> even mantissa
    (500.0, 0x7E),            # saturates (satfinite reading)
    (-500.0, 0xFE),
    (1e30, 0x7E),
    (-0.0, 0x80),
    (-(2.0 ** -12), 0x80),    # rounds to negative zero
    (0.001953125 * 1.5, 0x02),
])
def test_e4m3_encode_closed_forms(v, code):
    assert oracle.e4m3_encode(v) == code


def test_e4m3_encode_nan():
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    # every bf16 value, scaled into the E4M3 range by a few powers of two; fp32-exact inputs
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    rng = np.random.default_rng(0)
    sel = vals[np.isfinite(vals)]
    sel = sel[(np.abs(sel) < 464.0)]
    sel = rng.choice(sel, size=6000, replace=False)
    extra = np.concatenate([np.linspace(-463.9, 463.9, 2001), [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10]])
    cand = np.concatenate([sel, extra]).astype(np.float32)
    ref = torch.from_numpy(cand).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in cand], np.uint8)
    # torch keeps the sign of zero; so does the oracle
    assert np.array_equal(got, ref)


def test_e8m0_values():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))


def _rand_bf16(rng, shape, scale=1.0):
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_mxfp8_scale_matches_frexp_and_elements_match_torch():
    rng = np.random.default_rng(1)
    rows, cols = 64, 256
    x = _rand_bf16(rng, (rows, cols))
    # per-row magnitude sweep, including tiny (subnormal bf16) and huge blocks
    scales = 2.0 ** rng.integers(-140, 120, size=(rows, 1))
    xv = oracle.bf16_to_f64(x) * scales
    x = torch.from_numpy(xv.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xv = oracle.bf16_to_f64(x)
    q, sc = oracle.mxfp8_quantize(x)
    blocks = xv.reshape(rows, cols // 32, 32)
    amax = np.abs(blocks).max(axis=2)
    m, ex = np.frexp(amax)
    shared = np.where(amax == 0, -127, np.clip(ex - 1 - 8, -127, 127))
    assert np.array_equal(sc.astype(np.int64), shared + 127)
    # elements: torch's RNE conversion of v / 2^shared where it is in range, else saturation
    scaled = blocks / (2.0 ** shared)[:, :, None]
    f32 = scaled.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), scaled)  # the scaling is exact
    ref = torch.from_numpy(f32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inr = np.abs(scaled) < 464.0
    got = q.reshape(rows, cols // 32, 32)
    assert np.array_equal(got[inr], ref[inr])
    sat = ~inr
    assert np.all((got[sat] & 0x7F) == 0x7E)


def test_mxfp8_special_blocks():
    x = np.zeros((3, 64), np.uint16)
    x[1, :32] = 0x3F80           # all ones -> amax 1 -> shared -8 -> scale 119, elements 1*2^8 = 256
    x[1, 32:] = 0x8000           # negative zeros
    x[2, 5] = 0x7FC0             # NaN in block 0 of row 2
    x[2, 40] = 0x7F80            # +Inf in block 1 of row 2
    q, sc = oracle.mxfp8_quantize(x)
    assert sc[0].tolist() == [0, 0] and not q[0].any()
    assert sc[1, 0] == 119 and oracle.e4m3_value(int(q[1, 0])) == 256.0
    assert sc[1, 1] == 0 and np.all(q[1, 32:] == 0x80)
    assert sc[2].tolist() == [0xFF, 0xFF] and np.all(q[2] == 0x7F)


def test_mxfp8_round_trip_exact_on_grid():
    # values already on the E4M3 grid times a per-block power of two survive exactly
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 0x7F, size=(16, 128)).astype(np.uint8)
    codes[:, ::32] = 0x7E  # make each block's amax the top code so the block exponent is known
    sign = rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    codes = codes | sign
    grid = np.array([oracle.e4m3_value(int(c)) for c in codes.ravel()]).reshape(codes.shape)
    k = rng.integers(-20, 20, size=(16, 4))
    vals = grid * np.repeat(2.0 ** k, 32, axis=1)
    x = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(x.double().numpy(), vals)  # E4M3 values are bf16-exact
    q, sc = oracle.mxfp8_quantize(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(oracle.mxfp8_dequantize(q, sc), vals)
    assert np.array_equal(sc.astype(np.int64), k + 127)


def test_mxfp8_rejects_ragged_cols():
    with pytest.raises(ValueError):
        oracle.mxfp8_quantize(np.zeros((2, 48), np.uint16))

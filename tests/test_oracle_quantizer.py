"""Pins for the oracle's MXFP4 quantiser (CPU only).

What fixes the answers here is not the oracle itself:
  * the E2M1 element format's definition (1 sign bit, 2 exponent bits with bias 1,
    1 mantissa bit; exponent field 0 is subnormal), from which the value table is
    rebuilt below from bit fields;
  * the rounding rule (nearest, ties to the code with an even mantissa bit) at every
    midpoint of the grid;
  * the block-scale rule (the smallest power of two 2^e with amax <= 6 * 2^e),
    checked by direct comparison in exact binary floating point;
  * closed forms: data already on the grid round-trips exactly, and the quantisation
    error of an element never exceeds half the grid spacing at its magnitude.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def e2m1_from_bits(code: int) -> float:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m / 2.0) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def test_e2m1_table_matches_format_definition():
    for code in range(16):
        assert oracle.e2m1_value(code) == e2m1_from_bits(code), code
    mags = sorted({abs(e2m1_from_bits(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.mark.parametrize("y, code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),   # midpoints: even code wins
    (0.0, 0), (0.5, 1), (1.0, 2), (1.5, 3), (2.0, 4), (3.0, 5), (4.0, 6), (6.0, 7),  # grid points
    (0.2499, 0), (0.2501, 1), (5.0001, 7), (4.9999, 6), (6.5, 7),
])
def test_e2m1_rounding_points(y, code):
    assert oracle.e2m1_round(y) == code


def test_e2m1_rounding_is_nearest_with_even_ties():
    grid = np.array([abs(e2m1_from_bits(c)) for c in range(8)])
    rng = synth.Rng(11)
    ys = np.concatenate([rng.uniform(4000) * 6.0, (grid[:-1] + grid[1:]) / 2])
    for y in ys:
        c = oracle.e2m1_round(float(y))
        d = np.abs(grid - y)
        best = np.flatnonzero(d == d.min())
        if len(best) == 1:
            assert c == best[0]
        else:  # a tie: the code with mantissa bit 0
            assert c in best and c % 2 == 0


def test_block_exponent_definition():
    rng = synth.Rng(12)
    amaxes = np.concatenate([np.exp(rng.normal(3000) * 8.0), [6.0, 3.0, 6.0 * 2 ** -5, 1e-30, 1e30]])
    for a in amaxes:
        e = oracle.block_exponent(float(a))
        assert a <= 6.0 * 2.0 ** e
        assert not (a <= 6.0 * 2.0 ** (e - 1))
    # closed forms: amax = 6 * 2^e gives exactly e; the next float up gives e + 1
    for e in range(-20, 21):
        a = 6.0 * 2.0 ** e
        assert oracle.block_exponent(a) == e
        assert oracle.block_exponent(math.nextafter(a, math.inf)) == e + 1
    assert oracle.block_exponent(0.0) == -127


def _bf16(x):
    return synth.bf16_bits(np.asarray(x, np.float32))


def test_on_grid_vectors_round_trip_exactly():
    rng = synth.Rng(13)
    n = 200
    codes = rng.integers(0, 15, n * 128).reshape(n, 128)
    grid = np.array([e2m1_from_bits(c) for c in range(16)])
    vals = grid[codes]
    # force one +-6 per block so the block exponent is pinned to the drawn one
    for g in range(4):
        vals[:, 32 * g] = np.where(rng.uniform(n) < 0.5, 6.0, -6.0)
    exps = rng.integers(-10, 10, n * 4).reshape(n, 4)
    x = vals * np.repeat(2.0 ** exps, 32, axis=1)
    xb = _bf16(x)
    assert np.array_equal(synth.bf16_to_f32(xb).astype(np.float64), x)  # grid*2^e is exact in bf16
    packed, scales = oracle.quantize_plain(xb)
    assert np.array_equal(scales.astype(np.int64) - 127, exps)
    back = oracle.dequantize_plain(packed, scales)
    assert np.array_equal(back, x)


def test_quantisation_error_bound_and_scale_rule():
    case_rng = synth.Rng(14)
    x = synth.qk_bf16(case_rng, (500,))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    packed, scales = oracle.quantize_plain(x)
    back = oracle.dequantize_plain(packed, scales)
    e = scales.astype(np.int64) - 127
    for g in range(4):
        blk = xf[:, 32 * g:32 * g + 32]
        amax = np.abs(blk).max(axis=1)
        assert np.all(amax <= 6.0 * 2.0 ** e[:, g])
        assert np.all(amax > 3.0 * 2.0 ** e[:, g])
        y = np.abs(blk) * 2.0 ** (-e[:, g:g + 1])
        spacing = np.where(y <= 2.0, 0.5, np.where(y <= 4.0, 1.0, 2.0))
        err = np.abs(back[:, 32 * g:32 * g + 32] - blk) * 2.0 ** (-e[:, g:g + 1])
        assert np.all(err <= spacing / 2 + 1e-12)


def test_sign_and_zero_readings():
    # R2: a negative value that rounds to zero keeps the sign bit (code 8)
    x = np.zeros(128, np.float32)
    x[0] = 6.0
    x[1] = -0.1
    packed, scales = oracle.quantize_plain(_bf16(x)[None])
    assert scales[0, 0] == 127
    assert packed[0, 0] == (0x7 | (0x8 << 4))  # R1: element 0 in the low nibble
    # R3: an all-zero block takes scale byte 0 and zero codes
    assert scales[0, 1] == 0 and np.all(packed[0, 16:32] == 0)


def test_nibble_order_low_is_even_dim():
    x = np.zeros(128, np.float32)
    x[2] = 1.0   # dim 2 -> byte 1, low nibble
    x[3] = -6.0  # dim 3 -> byte 1, high nibble; sets the scale to 2^0
    packed, scales = oracle.quantize_plain(_bf16(x)[None])
    assert scales[0, 0] == 127
    assert packed[0, 1] == (0x2 | (0xF << 4))
    assert np.all(np.delete(packed[0, :16], 1) == 0)

"""Pins of the oracle's weight-only 8-bit block quantisation and its GEMV.

The talker of "audio.cpp Rockchip NPU build notes" streams Q8_0 weights (section "The
talker is the only DRAM-bound candidate, and it is not at the ceiling"); the layout is
read as 32-weight blocks along K with one half-precision scale d = max|w| / 127 and
codes round(w / d).  Pinned here: the half conversion against numpy's float16 (every
half exhaustively one way, edge cases the other), codes on blocks whose scale is
exact, the rounding of ties away from zero, the zero block, the error bound, and the
GEMV against numpy's float64 product with the dequantised matrix.
"""
import numpy as np
import pytest

import oracle as O


def test_half_from_float_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.normal(size=4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 5, size=4000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                  2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf],
                 np.float32)])
    with np.errstate(over="ignore"):                         # the overflow cases round to infinity
        want = vals.astype(np.float16).view(np.uint16)
    for v, h in zip(vals, want):
        assert O.f32_to_f16(v) == int(h), v


def test_float_from_every_half_matches_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([O.f16_to_f32(int(x)) for x in h], np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(got[~finite]) == np.isnan(ref[~finite]))


def test_codes_of_blocks_with_an_exact_scale():
    k = np.arange(-127, 128, dtype=np.float32)
    k = k[np.random.default_rng(1).permutation(255)[:64]]   # 64 distinct integers in [-127, 127]
    k[0], k[40] = 127.0, -127.0                             # each block's extremes: d exactly 0.5
    w = (k * np.float32(0.5)).reshape(2, 32)
    codes, scales = O.quantize_q8(w)
    assert np.array_equal(codes.astype(np.float32), k.reshape(2, 32))
    assert np.all(scales == O.f32_to_f16(0.5))


def test_ties_round_away_from_zero_and_zero_blocks():
    d = np.float32(0.25)
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = 127 * d                                        # sets d = 0.25 for block 0
    w[0, 1], w[0, 2], w[0, 3], w[0, 4] = 1.5 * d, -1.5 * d, 2.5 * d, -0.5 * d
    codes, scales = O.quantize_q8(w)
    assert list(codes[0, :5]) == [127, 2, -2, 3, -1]
    assert np.all(codes[0, 32:] == 0) and scales[0, 1] == 0


def test_error_bound_and_extremes():
    rng = np.random.default_rng(2)
    w = rng.normal(0, 0.02, size=(64, 256)).astype(np.float32)
    codes, scales = O.quantize_q8(w)
    blocks = w.reshape(64, 8, 32)
    amax = np.abs(blocks).max(axis=2)
    d = (amax / np.float32(127.0)).astype(np.float32)
    deq32 = codes.reshape(64, 8, 32).astype(np.float64) * d[..., None]
    assert np.all(np.abs(blocks - deq32) <= d[..., None] / 2 * (1 + 1e-6))
    at = np.argmax(np.abs(blocks), axis=2)
    picked = np.take_along_axis(codes.reshape(64, 8, 32), at[..., None], axis=2)[..., 0]
    assert np.all(np.abs(picked) == 127)
    dh = scales.view(np.float16).astype(np.float64)
    assert np.all(np.abs(dh - d) <= d * 2.0 ** -11 + 2.0 ** -25)


def test_gemv_is_the_dequantised_matvec():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.02, size=(300, 512)).astype(np.float32)
    x = rng.normal(size=512).astype(np.float32)
    codes, scales = O.quantize_q8(w)
    deq = codes.astype(np.float32) * np.repeat(scales.view(np.float16).astype(np.float32), 32, axis=1)
    ref = (deq.astype(np.float64) @ x.astype(np.float64))
    y = O.gemv_q8(codes, scales, x)
    assert np.max(np.abs(y - ref)) <= 1e-6 * np.max(np.abs(ref))
    # and close to the unquantised product, within the quantisation error
    exact = w.astype(np.float64) @ x.astype(np.float64)
    assert np.max(np.abs(y - exact)) < 0.02 * np.max(np.abs(exact))


def test_bad_shapes():
    with pytest.raises(O.OracleError):
        O.quantize_q8(np.zeros((2, 48), np.float32))


def test_dequantized_rows_reproduce_the_gemv():
    """dequantize_q8 (numpy) against the oracle's own 8-bit GEMV (C): the product of the
    dequantised matrix in float64 is within the GEMV's fp32 accumulation bound."""
    rng = np.random.default_rng(5)
    w = rng.normal(0.0, 0.02, size=(37, 256)).astype(np.float32)
    w[3, 32:64] = 0.0
    codes, scales = O.quantize_q8(w)
    deq = O.dequantize_q8(codes, scales)
    assert deq.dtype == np.float32 and deq.shape == w.shape
    assert np.all(deq[3, 32:64] == 0.0)
    assert np.max(np.abs(deq - w)) <= np.max(np.abs(w)) / 127 * 0.5 * (1 + 2.0 ** -10) + 1e-12
    x = rng.normal(size=256).astype(np.float32)
    ref = deq.astype(np.float64) @ x.astype(np.float64)
    mag = np.abs(deq.astype(np.float64)) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(O.gemv_q8(codes, scales, x) - ref) <= 2 * 256 * 2.0 ** -24 * mag + 1e-30)


def test_q8_model_weights_replace_only_the_matrices():
    import workloads as W
    s = W.scaled(W.ASR, n_layers=1, name="asr1q")
    w = W.model_weights(s)
    q = O.q8_model_weights(s, w)
    assert set(q) == set(w)
    as_f32 = lambda v: (v.astype(np.uint32) << 16).view(np.float32)
    for k in ("embed", "final_norm", "layers.0.attn_norm", "layers.0.mlp_norm"):
        assert np.array_equal(q[k], as_f32(w[k]))
    for k in ("layers.0.wq", "layers.0.wd", "lm_head.0"):
        assert not np.array_equal(q[k], as_f32(w[k]))
        assert np.array_equal(q[k], O.dequantize_q8(*O.quantize_q8(as_f32(w[k]))))

"""Pins of the oracle's Q4_K super-block quantisation and its GEMV.

"audio.cpp Rockchip NPU build notes", section "The talker is the only DRAM-bound
candidate, and it is not at the ceiling", measures the talker's matrices as Q4_K (251 MB
per token against 471 MB as Q8_0).  The format is read as the k-quant layout: 256
weights in 8 sub-blocks of 32, a half scale d and half min dm per super-block, 6-bit
scale sc_j and min m_j per sub-block, 4-bit codes, weight = d sc_j q - dm m_j, 144 bytes
per 256 weights.  Pinned here with a numpy unpacker written from that description:
the byte count, a super-block whose parameters are exact (codes and weights come back
bit for bit), all-zero and all-positive sub-blocks, the nearest-code property of every
weight given its sub-block's parameters, the error bound, and the GEMV against numpy's
float64 product with the unpacked matrix.
"""
import numpy as np
import pytest

import oracle as O


def _unpack(blocks):
    """numpy: [rows, nsb, 144] -> (d, dm [rows, nsb], sc, m [rows, nsb, 8], q [rows, nsb, 256])."""
    b = blocks.astype(np.uint64)
    d = (b[..., 0] | (b[..., 1] << 8)).astype(np.uint16).view(np.float16).astype(np.float32)
    dm = (b[..., 2] | (b[..., 3] << 8)).astype(np.uint16).view(np.float16).astype(np.float32)

    def six(off):
        w = np.zeros(b.shape[:-1], np.uint64)
        for k in range(6):
            w |= b[..., off + k] << np.uint64(8 * k)
        return np.stack([((w >> np.uint64(6 * j)) & np.uint64(63)).astype(np.int64) for j in range(8)], -1)

    sc, m = six(4), six(10)
    codes = blocks[..., 16:].astype(np.int64)
    q = np.stack([codes & 15, codes >> 4], -1).reshape(*blocks.shape[:-1], 256)
    return d, dm, sc, m, q


def _dequant(blocks):
    d, dm, sc, m, q = _unpack(blocks)
    step = d[..., None] * sc.astype(np.float32)                 # [rows, nsb, 8]
    off = dm[..., None] * m.astype(np.float32)
    w = np.repeat(step, 32, -1) * q.astype(np.float32) - np.repeat(off, 32, -1)
    return w.reshape(blocks.shape[0], -1).astype(np.float32)


def test_layout_bytes():
    w = np.zeros((2, 1024), np.float32)
    assert O.quantize_q4k(w).shape == (2, 4, 144)
    assert 144 * 8 / 256 == 4.5


def test_exact_superblock_round_trip():
    rng = np.random.default_rng(0)
    d, dm = np.float32(2.0 ** -9), np.float32(2.0 ** -10)
    sc = rng.integers(1, 64, 8)
    m = rng.integers(0, 64, 8)
    sc[3], m[5] = 63, 63                          # the super-block maxima: d and dm come out exact
    q = rng.integers(0, 16, (8, 32))
    q[:, 0], q[:, 1] = 0, 15                      # every sub-block spans its whole range
    w = ((d * sc[:, None]).astype(np.float32) * q.astype(np.float32) - (dm * m[:, None]).astype(np.float32))
    w = w.astype(np.float32).reshape(1, 256)
    blocks = O.quantize_q4k(w)
    dd, ddm, ssc, mm, qq = _unpack(blocks)
    assert dd[0, 0] == d and ddm[0, 0] == dm
    assert np.array_equal(ssc[0, 0], sc) and np.array_equal(mm[0, 0], m)
    assert np.array_equal(qq[0, 0].reshape(8, 32), q)
    assert np.array_equal(_dequant(blocks), w)


def test_zero_and_positive_subblocks():
    w = np.zeros((1, 256), np.float32)
    w[0, 32:64] = np.linspace(0.1, 0.4, 32, dtype=np.float32)   # all positive: min 0
    blocks = O.quantize_q4k(w)
    d, dm, sc, m, q = _unpack(blocks)
    assert dm[0, 0] == 0 and np.all(m == 0)
    assert np.all(q[0, 0, :32] == 0) and np.all(q[0, 0, 64:] == 0) and sc[0, 0, 0] == 0
    deq = _dequant(blocks)
    assert np.all(deq[0, :32] == 0) and np.all(deq[0, 64:] == 0)
    assert np.max(np.abs(deq[0, 32:64] - w[0, 32:64])) <= 0.4 / 15 / 2 * 1.05


def test_nearest_code_and_error_bound():
    rng = np.random.default_rng(1)
    w = (rng.normal(0.0, 0.02, (37, 512)) * (1 + 3 * (rng.random((37, 512)) < 0.01))).astype(np.float32)
    blocks = O.quantize_q4k(w)
    d, dm, sc, m, q = _unpack(blocks)
    step = np.repeat((d[..., None] * sc).astype(np.float32), 32, -1).reshape(37, -1)
    off = np.repeat((dm[..., None] * m).astype(np.float32), 32, -1).reshape(37, -1)
    deq = _dequant(blocks)
    err = np.abs(deq.astype(np.float64) - w)
    # every code is the nearest of the 16 values its sub-block can represent
    cand = step[..., None].astype(np.float64) * np.arange(16) - off[..., None]
    best = np.min(np.abs(cand - w[..., None]), -1)
    assert np.all(err <= best + 1e-7 * (np.abs(w) + step))
    # and the sub-block's range covers its weights up to the 6-bit rounding of the scale
    # and the min: half a step plus the drift of 15 steps and of the offset
    assert np.sqrt(np.mean(err ** 2)) < 0.2 * np.sqrt(np.mean(w.astype(np.float64) ** 2))


def test_gemv_matches_unpacked_product():
    rng = np.random.default_rng(2)
    w = rng.normal(0.0, 0.02, (61, 768)).astype(np.float32)
    x = rng.normal(size=768).astype(np.float32)
    blocks = O.quantize_q4k(w)
    deq = _dequant(blocks).astype(np.float64)
    ref = deq @ x.astype(np.float64)
    mag = np.abs(deq) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(O.gemv_q4k(blocks, x) - ref) <= 2 * 768 * 2.0 ** -24 * mag + 1e-30)


def test_shape_errors():
    with pytest.raises(O.OracleError):
        O.quantize_q4k(np.zeros((2, 100), np.float32))

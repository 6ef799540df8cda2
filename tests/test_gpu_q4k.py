"""Q4_K super-block quantisation and its GEMV on the GPU against the oracle.

The codes, the 6-bit sub-block scales and mins and the two half super-block scales are
decisions taken in the same fp32 arithmetic on both sides (IEEE division, half-away
rounding), so the 144 bytes of every super-block must match bit for bit.  The GEMV is
an fp32 sum on the GPU (per lane d sc_j times its 8 code products, minus dm m_j times
its 8 inputs) against the oracle's fp64 sum of the dequantised products, compared within
the fp32 accumulation bound of the terms it adds.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _quantize_gpu(w_t):
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    rows, K = w_t.shape
    blocks = torch.zeros((rows, K // 256, 144), dtype=torch.uint8, device="cuda")
    qd.qd_quantize_q4k(w_t, blocks)
    return blocks


def _matrix(rows, K, seed):
    w = W.normal(f"q4k/{rows}x{K}/{seed}", (rows, K), seed, 0.0, 0.02)
    w[0, :32] = 0.0                                   # an all-zero sub-block
    w[0, 32:64] = np.abs(w[0, 32:64]) + 0.01          # an all-positive one
    w[min(1, rows - 1), :256] = 0.0                   # an all-zero super-block
    return w


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("rows,K", [(333, 512), (100, 1024), (77, 2048), (5, 256), (3, 768)])
def test_blocks_are_bit_exact(rows, K, bf16):
    import torch
    import oracle as O
    w = _matrix(rows, K, 0)
    wt = torch.from_numpy(w).cuda()
    if bf16:
        wt = wt.to(torch.bfloat16)
        w = wt.float().cpu().numpy()
    got = _quantize_gpu(wt).cpu().numpy()
    ref = O.quantize_q4k(w)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


def _terms_magnitude(blocks, x):
    """sum_k (d sc_j q + dm m_j) |x_k|: the magnitude of the terms the GPU adds."""
    b = blocks.astype(np.uint64)
    d = (b[..., 0] | (b[..., 1] << 8)).astype(np.uint16).view(np.float16).astype(np.float64)
    dm = (b[..., 2] | (b[..., 3] << 8)).astype(np.uint16).view(np.float16).astype(np.float64)

    def six(off):
        w = np.zeros(b.shape[:-1], np.uint64)
        for k in range(6):
            w |= b[..., off + k] << np.uint64(8 * k)
        return np.stack([((w >> np.uint64(6 * j)) & np.uint64(63)).astype(np.float64) for j in range(8)], -1)

    sc, m = six(4), six(10)
    codes = blocks[..., 16:].astype(np.int64)
    q = np.stack([codes & 15, codes >> 4], -1).reshape(*blocks.shape[:-1], 256).astype(np.float64)
    t = np.repeat(d[..., None] * sc, 32, -1) * q + np.repeat(dm[..., None] * m, 32, -1)
    return t.reshape(blocks.shape[0], -1) @ np.abs(x.astype(np.float64))


@pytest.mark.parametrize("rows,K", [(333, 512), (1000, 1024), (77, 2048), (4097, 512), (1, 1024)])
def test_gemv_matches_oracle(rows, K):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    w = _matrix(rows, K, 1)
    x = W.normal(f"q4k/x/{K}", (K,), 1, 0.0, 1.0)
    blocks = _quantize_gpu(torch.from_numpy(w).cuda())
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    qd.qd_gemv_q4k(blocks, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    b = blocks.cpu().numpy()
    ref = O.gemv_q4k(b, x)
    mag = _terms_magnitude(b, x)
    assert np.all(np.abs(y.cpu().numpy() - ref) <= 4 * K * 2.0 ** -24 * mag + 1e-30)


def test_full_size_lm_head_sampled_rows():
    """The ASR workload's 151936 x 512 LM head (bf16): every super-block quantised on the
    GPU, sampled rows' bytes and products against the oracle."""
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import to_device
    s = W.ASR
    wt = to_device(W.model_weights(W.scaled(s, n_layers=1, name="asr_q4k"))["lm_head.0"])
    blocks = _quantize_gpu(wt)
    x = W.normal("q4k/head_x", (s.hidden,), 2, 0.0, 1.0)
    y = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    qd.qd_gemv_q4k(blocks, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    rows = np.unique(np.random.default_rng(3).integers(0, s.vocab, 512))
    wr = wt[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref_b = O.quantize_q4k(wr)
    got_b = blocks.cpu().numpy()[rows]
    assert np.array_equal(got_b, ref_b)
    ref = O.gemv_q4k(ref_b, x)
    mag = _terms_magnitude(ref_b, x)
    assert np.all(np.abs(y.cpu().numpy()[rows] - ref) <= 4 * s.hidden * 2.0 ** -24 * mag + 1e-30)


def test_errors():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    w = torch.zeros((4, 300), dtype=torch.float32, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_quantize_q4k(w, torch.zeros((4, 1, 144), dtype=torch.uint8, device="cuda"))
    assert ei.value.status == qd.QD_EINVAL
    blocks = torch.zeros((4, 3, 144), dtype=torch.uint8, device="cuda")
    x = torch.zeros(768, dtype=torch.float32, device="cuda")
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_gemv_q4k(blocks, x, y)                  # K = 768: no instantiation
    assert ei.value.status == qd.QD_EUNSUPPORTED
    with pytest.raises(qd.QDError) as ei:
        qd.qd_gemv_q4k(blocks.cpu(), x, y)            # host blocks
    assert ei.value.status == qd.QD_EINVAL

"""Weight-only 8-bit block quantisation and its GEMV on the GPU against the oracle.

The codes and the half scales are integer decisions taken in the same fp32 arithmetic
on both sides, so they must match bit for bit; the GEMV is a K-term fp32 sum on the
GPU (per 16-code chunk, then scaled) against the oracle's fp64 sum of the same
dequantised products, compared within a bound derived from fp32 accumulation.
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
    codes = torch.empty((rows, K), dtype=torch.int8, device="cuda")
    scales = torch.empty((rows, K // 32), dtype=torch.int16, device="cuda")
    qd.qd_quantize_q8(w_t, codes, scales)
    return codes, scales


def _matrix(rows, K, seed, special=True):
    w = W.normal(f"q8/{rows}x{K}/{seed}", (rows, K), seed, 0.0, 0.02)
    if special:
        w[0, :32] = 0.0                                   # an all-zero block
        d = np.float32(0.01)
        w[1, :32] = 0.0
        w[1, 0] = 127 * d                                 # d = 0.01 exactly in fp32 arithmetic terms
        w[1, 1:5] = np.array([1.5, -1.5, 2.5, -0.5], np.float32) * d
    return w


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("rows,K", [(333, 512), (1000, 1024), (77, 2048), (5, 96)])
def test_codes_and_scales_are_bit_exact(rows, K, bf16):
    import torch
    import oracle as O
    w = _matrix(rows, K, 0)
    if bf16:
        wt = torch.from_numpy(w).cuda().to(torch.bfloat16)
        w_ref = wt.float().cpu().numpy()
    else:
        wt = torch.from_numpy(w).cuda()
        w_ref = w
    codes, scales = _quantize_gpu(wt)
    rc, rs = O.quantize_q8(w_ref)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs)


@pytest.mark.parametrize("rows,K", [(333, 512), (1000, 1024), (77, 2048), (4097, 512)])
def test_gemv_matches_oracle(rows, K):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    w = _matrix(rows, K, 1)
    x = W.normal(f"q8/x/{K}", (K,), 1, 0.0, 1.0)
    codes, scales = _quantize_gpu(torch.from_numpy(w).cuda())
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    qd.qd_gemv_q8(codes, scales, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    rc, rs = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    ref = O.gemv_q8(rc, rs, x)
    # bound: fp32 accumulation of K products of magnitude |code * d * x|
    deq = rc.astype(np.float64) * np.repeat(rs.view(np.float16).astype(np.float64), 32, axis=1)
    mag = np.abs(deq) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(y.cpu().numpy() - ref) <= 4 * K * 2.0 ** -24 * mag + 1e-30)


def test_full_size_lm_head():
    """The ASR LM head (151936 x 512, bf16): codes bit-exact, every logit within the
    accumulation bound."""
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import to_device
    s = W.ASR
    head = W.model_weights(s)["lm_head.0"]
    wt = to_device(head)
    codes, scales = _quantize_gpu(wt)
    w_ref = wt.float().cpu().numpy()
    rc, rs = O.quantize_q8(w_ref)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs)
    x = W.normal("q8/x/asr", (s.hidden,), 2, 0.0, 1.0)
    y = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    qd.qd_gemv_q8(codes, scales, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    ref = O.gemv_q8(rc, rs, x)
    deq = np.abs(rc.astype(np.float32)) * np.repeat(rs.view(np.float16).astype(np.float32), 32, axis=1)
    mag = (deq @ np.abs(x)).astype(np.float64)
    assert np.all(np.abs(y.cpu().numpy() - ref) <= 4 * s.hidden * 2.0 ** -24 * mag + 1e-30)


def test_errors():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    w = torch.zeros((4, 48), device="cuda")
    with pytest.raises(qd.QDError) as ei:
        _quantize_gpu(w)
    assert ei.value.status == qd.QD_EINVAL
    codes = torch.zeros((4, 96), dtype=torch.int8, device="cuda")
    scales = torch.zeros((4, 3), dtype=torch.int16, device="cuda")
    x = torch.zeros(96, device="cuda")
    y = torch.empty(4, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_gemv_q8(codes, scales, x, y)
    assert ei.value.status == qd.QD_EUNSUPPORTED
    codes = torch.zeros((4, 512), dtype=torch.int8, device="cuda")
    scales = torch.zeros((4, 16), dtype=torch.int16, device="cuda")
    xb = torch.zeros(513, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_gemv_q8(codes, scales, xb[1:], y)                 # x not 16-byte aligned
    assert ei.value.status == qd.QD_EINVAL

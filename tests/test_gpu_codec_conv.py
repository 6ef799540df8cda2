"""The codec decoder's convolution stages on the GPU against the oracle.

Both are fp32 sums (the GPU's in a fixed chunk order, the oracle's in fp64), compared
within the bound of fp32 accumulation over the terms of each output.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).normal(size=shape) * scale).astype(np.float32)


def _check(y, ref, mag, terms):
    assert np.all(np.abs(y - ref) <= 4 * terms * 2.0 ** -24 * mag + 1e-30)


@pytest.mark.parametrize("Cin,Cout,K,d,T", [(3, 4, 3, 1, 20), (16, 40, 7, 3, 300), (9, 33, 3, 9, 129),
                                           (256, 256, 7, 1, 1000), (1, 1, 1, 1, 5),
                                           # the largest staged layouts: 16 taps, and a
                                           # history span of 510 and of exactly 512 frames
                                           (12, 35, 16, 34, 700), (10, 33, 3, 256, 900)])
def test_causal_conv_matches_oracle(Cin, Cout, K, d, T):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    x, W, b = _rand((Cin, T), 1), _rand((Cout, Cin, K), 2, 0.05), _rand((Cout,), 3)
    y = qd.qd_conv1d_causal(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda(),
                            dilation=d).cpu().numpy()
    ref = O.conv1d_causal(x, W, b, dilation=d)
    mag = O.conv1d_causal(np.abs(x), np.abs(W), np.abs(b), dilation=d).astype(np.float64)
    _check(y, ref, mag, Cin * K + 1)


@pytest.mark.parametrize("Cin,Cout,s,T", [(3, 4, 2, 10), (256, 128, 4, 250), (64, 32, 8, 33), (1, 1, 1, 3)])
def test_transposed_conv_matches_oracle(Cin, Cout, s, T):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    x, W, b = _rand((Cin, T), 4), _rand((Cin, Cout, 2 * s), 5, 0.05), _rand((Cout,), 6)
    y = qd.qd_conv_transpose1d_causal(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(),
                                      torch.from_numpy(b).cuda(), stride=s).cpu().numpy()
    ref = O.conv_transpose1d_causal(x, W, b, stride=s)
    mag = O.conv_transpose1d_causal(np.abs(x), np.abs(W), np.abs(b), stride=s).astype(np.float64)
    _check(y, ref, mag, 2 * Cin + 1)


def test_without_bias_and_errors():
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    x, W = _rand((5, 40), 7), _rand((6, 5, 3), 8)
    y = qd.qd_conv1d_causal(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), None, dilation=2)
    ref = O.conv1d_causal(x, W, None, dilation=2)
    assert np.max(np.abs(y.cpu().numpy() - ref)) < 1e-4
    xc, Wc = torch.from_numpy(x).cuda(), torch.from_numpy(_rand((6, 5, 17), 9)).cuda()
    with pytest.raises(qd.QDError) as ei:
        qd.qd_conv1d_causal(xc, Wc)                         # K > 16
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_conv1d_causal(xc, torch.from_numpy(W).cuda(), dilation=300)   # history span > 512
    assert ei.value.status == qd.QD_EUNSUPPORTED


# ---- the tensor-core forms (qd_*_tc): weights rounded to bf16 by the library, the
# signal carried as bf16 hi + lo parts.  The weights here are bf16 values already (so
# the oracle sees exactly the weights the GPU uses); the signal split leaves at most
# 2^-18 |x| per element, so each output is within 2^-17 of the magnitude sum of its
# terms plus the fp32 accumulation bound.

def _bf16(a):
    import torch
    return torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()


def _check_tc(y, ref, mag, terms):
    tol = (2.0 ** -17 + 4 * terms * 2.0 ** -24) * mag + 1e-30
    bad = np.abs(y - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], np.abs(y - ref)[bad][:5], tol[bad][:5])


@pytest.mark.parametrize("Cin,Cout,K,d,T", [(3, 4, 3, 1, 20), (16, 40, 7, 3, 300), (9, 33, 3, 9, 129),
                                           (256, 256, 7, 1, 1000), (1, 1, 1, 1, 5),
                                           (12, 35, 16, 34, 700), (10, 33, 3, 256, 900),
                                           # ragged tiles in every dimension, and a long history
                                           (130, 200, 5, 2, 333), (64, 128, 33, 40, 2000),
                                           (512, 256, 3, 4, 2048)])
def test_causal_conv_tc_matches_oracle(Cin, Cout, K, d, T):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    x, W, b = _rand((Cin, T), 11), _bf16(_rand((Cout, Cin, K), 12, 0.05)), _rand((Cout,), 13)
    y = qd.qd_conv1d_causal_tc(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda(),
                               dilation=d).cpu().numpy()
    ref = O.conv1d_causal(x, W, b, dilation=d)
    mag = O.conv1d_causal(np.abs(x), np.abs(W), np.abs(b), dilation=d).astype(np.float64)
    _check_tc(y, ref, mag, Cin * K + 1)


@pytest.mark.parametrize("Cin,Cout,s,T", [(3, 4, 2, 10), (256, 128, 4, 250), (64, 32, 8, 33), (1, 1, 1, 3),
                                         (100, 130, 3, 77), (512, 256, 4, 1024)])
def test_transposed_conv_tc_matches_oracle(Cin, Cout, s, T):
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    x, W, b = _rand((Cin, T), 14), _bf16(_rand((Cin, Cout, 2 * s), 15, 0.05)), _rand((Cout,), 16)
    y = qd.qd_conv_transpose1d_causal_tc(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(),
                                         torch.from_numpy(b).cuda(), stride=s).cpu().numpy()
    ref = O.conv_transpose1d_causal(x, W, b, stride=s)
    mag = O.conv_transpose1d_causal(np.abs(x), np.abs(W), np.abs(b), stride=s).astype(np.float64)
    _check_tc(y, ref, mag, 2 * Cin + 1)


def test_tc_forms_round_the_weights_and_check_arguments():
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    # fp32 weights that are not bf16 values: the result is the oracle's on the rounded
    # weights, not on the given ones
    x, W = _rand((64, 300), 17), _rand((128, 64, 3), 18, 0.05)
    y = qd.qd_conv1d_causal_tc(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), None, dilation=2)
    y = y.cpu().numpy()
    Wr = _bf16(W)
    ref = O.conv1d_causal(x, Wr, None, dilation=2)
    mag = O.conv1d_causal(np.abs(x), np.abs(Wr), None, dilation=2).astype(np.float64)
    _check_tc(y, ref, mag, 64 * 3)
    assert np.max(np.abs(y - O.conv1d_causal(x, W, None, dilation=2))) > 1e-5
    xc = torch.from_numpy(x).cuda()
    with pytest.raises(qd.QDError) as ei:
        qd.qd_conv1d_causal_tc(xc, torch.from_numpy(_rand((4, 64, 65), 19)).cuda())   # K > 64
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_conv_transpose1d_causal_tc(xc.cpu(), torch.from_numpy(_rand((64, 4, 4), 20)).cuda(), stride=2)
    assert ei.value.status == qd.QD_EINVAL                                            # host signal

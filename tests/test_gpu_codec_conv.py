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

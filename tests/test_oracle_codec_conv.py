"""Pins of the oracle's codec-decoder convolution stages.

"qwen3-tts-hip OPTIMIZATION_LOG" (decoder transposed-convolution entries) profiles the
codec decoder as causal dilated convolutions and transposed convolutions, and rewrites
the transposed convolution per output phase.  In this repository's notation, with
kernel length 2 * stride and weights W[i][o][k], the output sample s = t * stride + p
(0 <= p < stride) only receives two taps: k = p from input frame t and k = p + stride
from frame t - 1, so y[o][s] = b[o] + sum_i (W[i][o][p] x[i][t] + W[i][o][p + stride]
x[i][t - 1]), one matrix product per tap and phase.  The oracle computes both stages
from their definitions (a tap sum and a scatter); the pins check them against other
formulations: numpy's full convolution with the reversed dilated kernel, the two
products per phase, torch's transposed convolution trimmed to the causal length,
impulse responses, causality and linearity.
"""
import numpy as np
import pytest

import oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).normal(size=shape).astype(np.float32)


@pytest.mark.parametrize("Cin,Cout,K,d,T", [(3, 4, 3, 1, 20), (2, 5, 7, 3, 40), (4, 2, 3, 9, 50), (1, 1, 1, 1, 5)])
def test_causal_conv_is_numpys_convolution_with_the_reversed_dilated_kernel(Cin, Cout, K, d, T):
    x, W, b = _rand((Cin, T), 1), _rand((Cout, Cin, K), 2), _rand((Cout,), 3)
    y = O.conv1d_causal(x, W, b, dilation=d)
    ref = np.zeros((Cout, T))
    for o in range(Cout):
        for i in range(Cin):
            v = np.zeros((K - 1) * d + 1)
            for k in range(K):
                v[(K - 1 - k) * d] = W[o, i, k]
            ref[o] += np.convolve(x[i].astype(np.float64), v)[:T]
        ref[o] += b[o]
    assert np.max(np.abs(y - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))


def test_causal_conv_impulse_response_and_causality():
    Cin, Cout, K, d, T = 2, 3, 3, 2, 16
    W = _rand((Cout, Cin, K), 4)
    x = np.zeros((Cin, T), np.float32)
    x[1, 5] = 1.0
    y = O.conv1d_causal(x, W, None, dilation=d)
    want = np.zeros((Cout, T), np.float32)
    for k in range(K):
        want[:, 5 + (K - 1 - k) * d] = W[:, 1, k]
    assert np.array_equal(y, want)
    # changing the future leaves the past alone
    x2 = _rand((Cin, T), 5)
    x3 = x2.copy()
    x3[:, 9:] = _rand((Cin, T - 9), 6)
    assert np.array_equal(O.conv1d_causal(x2, W, dilation=d)[:, :9], O.conv1d_causal(x3, W, dilation=d)[:, :9])


@pytest.mark.parametrize("Cin,Cout,s,T", [(3, 4, 2, 10), (5, 2, 4, 7), (2, 3, 8, 5), (1, 1, 1, 3)])
def test_transposed_conv_equals_the_pages_per_phase_gemms(Cin, Cout, s, T):
    x, W, b = _rand((Cin, T), 7), _rand((Cin, Cout, 2 * s), 8), _rand((Cout,), 9)
    y = O.conv_transpose1d_causal(x, W, b, stride=s)
    xt = x.T.astype(np.float64)                                 # time-major [T, Cin]
    prev = np.vstack([np.zeros((1, Cin)), xt[:-1]])             # the one-frame-shifted copy
    ref = np.zeros((Cout, T * s))
    for p in range(s):
        out_p = xt @ W[:, :, p].astype(np.float64) + prev @ W[:, :, p + s].astype(np.float64) + b
        ref[:, p::s] = out_p.T                                  # phase p of every frame
    assert np.max(np.abs(y - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))


def test_transposed_conv_matches_torch_trimmed_to_the_causal_length():
    import torch
    Cin, Cout, s, T = 4, 3, 3, 12
    x, W, b = _rand((Cin, T), 10), _rand((Cin, Cout, 2 * s), 11), _rand((Cout,), 12)
    ref = torch.nn.functional.conv_transpose1d(torch.from_numpy(x)[None].double(), torch.from_numpy(W).double(),
                                               torch.from_numpy(b).double(), stride=s)[0, :, :T * s].numpy()
    y = O.conv_transpose1d_causal(x, W, b, stride=s)
    assert np.max(np.abs(y - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))


def test_transposed_conv_impulse_and_linearity():
    Cin, Cout, s, T = 2, 2, 4, 6
    W = _rand((Cin, Cout, 2 * s), 13)
    x = np.zeros((Cin, T), np.float32)
    x[0, 2] = 1.0
    y = O.conv_transpose1d_causal(x, W, None, stride=s)
    want = np.zeros((Cout, T * s), np.float32)
    want[:, 2 * s:2 * s + 2 * s] = W[0]
    assert np.array_equal(y, want)
    x1, x2 = _rand((Cin, T), 14), _rand((Cin, T), 15)
    lhs = O.conv_transpose1d_causal(2 * x1 - 3 * x2, W, stride=s)
    rhs = 2 * O.conv_transpose1d_causal(x1, W, stride=s) - 3 * O.conv_transpose1d_causal(x2, W, stride=s)
    assert np.max(np.abs(lhs - rhs)) < 1e-4


def test_bad_arguments():
    with pytest.raises(O.OracleError):
        O.conv1d_causal(_rand((2, 4), 0), _rand((2, 2, 3), 0), dilation=0)
    with pytest.raises(ValueError):
        O.conv_transpose1d_causal(_rand((2, 4), 0), _rand((2, 2, 5), 0), stride=2)

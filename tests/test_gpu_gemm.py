"""Parity of the tensor-core GEMM (tcgen05 + TMA, bf16 weights, activations as bf16
hi + lo parts) with the oracle's batched linear.

Shapes cover the decode projections at 64 streams (split-K over CTAs, including
uneven splits), ragged token counts (a partial token tile), the prefill tile path
(several tiles per CTA, both accumulators) and the three epilogues.  The bar: the
hi/lo split carries ~16 bits of every activation, so the result must match the
oracle's fp32 product to within a small multiple of fp32 summation error.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _run(R, K, T, mode=0, seed=0, init=None):
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import to_device
    w = W.normal(f"gemm_w_{R}_{K}", (R, K), seed=seed, std=0.02, bf16=True)
    x = W.normal(f"gemm_x_{T}_{K}", (T, K), seed=seed)
    cols = R // 2 if mode == 2 else R
    out = torch.zeros((T, cols), dtype=torch.float32, device="cuda") if init is None else \
        torch.from_numpy(init.copy()).cuda()
    qd.qd_gemm_bf16(to_device(w), torch.from_numpy(x).cuda(), out, mode)
    return w, x, out.cpu().numpy()


def _close(got, ref):
    # Both sides sum in fp32 in different orders (the oracle in index order, the
    # tensor cores in their own tree), so they differ by fp32 summation noise, ~1e-6 of
    # the result's scale.  Dropping the activation's low part, a wrong tile or a wrong
    # row would show at ~1e-3 or more.
    d = got.astype(np.float64) - ref.astype(np.float64)
    scale = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
    assert np.sqrt(np.mean(d ** 2)) <= 5e-6 * max(scale, 1e-30), (np.sqrt(np.mean(d ** 2)), scale)
    bound = 2e-5 * (np.abs(ref.astype(np.float64)) + scale)
    assert np.all(np.abs(d) <= bound), (np.abs(d).max(), scale)


@pytest.mark.parametrize("R,K,T", [
    (256, 128, 64),      # 2 tiles x 2 splits
    (4096, 1024, 64),    # fused QKV of the Talker at 64 streams: 32 tiles x 4 splits
    (1024, 3072, 64),    # down projection: 8 tiles x 8 splits of 6 chunks
    (1024, 832, 64),     # 8 tiles x 8 uneven splits (13 chunks of 64)
    (1024, 2048, 5),     # 5 tokens: a partial token tile (zero-filled rows)
    (512, 1024, 300),    # 128-token tiles, ragged last tile
    (3072, 1024, 1024),  # prefill-like: 192 tiles, several per CTA, no split
])
def test_gemm_store_matches_oracle(R, K, T):
    w, x, got = _run(R, K, T)
    _close(got, O.linear(w, x))


def test_gemm_residual_adds_into_out():
    R, K, T = 1024, 2048, 64
    init = W.normal("gemm_res_init", (T, R), seed=1)
    w, x, got = _run(R, K, T, mode=1, init=init)
    _close(got - init, O.linear(w, x))
    assert np.allclose(got, init + O.linear(w, x), rtol=0, atol=1e-4)


@pytest.mark.parametrize("R,K,T", [(6144, 1024, 64), (768, 256, 200)])
def test_gemm_swiglu_pairs_rows(R, K, T):
    w, x, got = _run(R, K, T, mode=2)
    lin = O.linear(w, x).astype(np.float64)
    g, u = lin[:, 0::2], lin[:, 1::2]
    ref = g / (1.0 + np.exp(-g)) * u
    # the gate and up sums carry the summation noise of the store case; it reaches
    # the product through the partial derivatives of silu(g) * u
    scale = np.sqrt(np.mean(lin ** 2))
    eg, eu = 2e-5 * (np.abs(g) + scale), 2e-5 * (np.abs(u) + scale)
    sg = 1.0 / (1.0 + np.exp(-g))
    bound = np.abs(sg * (1 + g * (1 - sg)) * u) * eg + np.abs(g * sg) * eu + 1e-6 * np.abs(ref) + 1e-9
    d = np.abs(got.astype(np.float64) - ref)
    assert np.all(d <= bound), (d.max(), (d / bound).max())
    assert np.sqrt(np.mean(d ** 2)) <= 5e-6 * np.sqrt(np.mean(ref ** 2))


def test_gemm_is_deterministic():
    a = _run(1024, 3072, 64)[2]
    b = _run(1024, 3072, 64)[2]
    assert np.array_equal(a, b)

"""Pins of the oracle pieces the batched paths add (CPU only)."""
import numpy as np

import oracle as O
import workloads as W


def test_linear_equals_fp64_product_within_the_fp32_bound():
    w = W.normal("lin_w", (96, 320), seed=4, std=0.02, bf16=True)
    x = W.normal("lin_x", (7, 320), seed=4)
    wf = np.stack([O.table_row(w, r) for r in range(96)]).astype(np.float64)
    exact = x.astype(np.float64) @ wf.T
    bound = 320 * 2.0 ** -24 * (np.abs(x.astype(np.float64)) @ np.abs(wf).T)
    assert np.all(np.abs(O.linear(w, x) - exact) <= bound + 1e-30)


def test_linear_rows_are_the_decode_matvec():
    # a batch row is the same product one decode step computes: transposing the
    # operands or mixing rows changes the result
    w = W.normal("lin_w2", (64, 128), seed=5)
    x = W.normal("lin_x2", (3, 128), seed=5)
    out = O.linear(w, x)
    for t in range(3):
        assert np.array_equal(out[t], O.linear(w, x[t:t + 1])[0])
    assert not np.allclose(out[0], out[1])
    sq = W.normal("lin_sq", (128, 128), seed=5)
    assert not np.allclose(O.linear(sq, x), O.linear(np.ascontiguousarray(sq.T), x))


def test_linear_exact_on_small_integers():
    rng = np.random.default_rng(1)
    w = rng.integers(-4, 5, size=(32, 64)).astype(np.float32)
    x = rng.integers(-4, 5, size=(5, 64)).astype(np.float32)
    assert np.array_equal(O.linear(w, x), (x.astype(np.int64) @ w.astype(np.int64).T).astype(np.float32))


def _small_shape():
    return W.scaled(W.TALKER, name="talker_kv", hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32,
                    ffn=256, vocab=96, embed_rows=96, buckets=(32, 64), prefill=20)


def _cache_of(o, s):
    """The oracle's cache as [n_layers, 2, kvh, pos, hd] bf16 bits."""
    kv = np.stack([np.stack([o.kv(l, w) for w in range(2)]) for l in range(s.n_layers)])
    return (kv.view(np.uint32) >> 16).astype(np.uint16)


def test_set_kv_restores_a_stream_exactly():
    s = _small_shape()
    w = W.model_weights(s)
    a = O.Oracle(s, w)
    first, _, _ = a.prefill(embeds=W.prefill_embeds(s))
    kv = _cache_of(a, s)
    b = O.Oracle(s, w)
    b.set_kv(kv, s.prefill)
    assert b.pos == s.prefill and b.smax == 32
    tok = first
    for _ in range(15):                             # crosses the 32 -> 64 bucket on both
        ia, la, _, _ = a.step(token=tok)
        ib, lb, _, _ = b.step(token=tok)
        assert ia == ib and np.array_equal(la, lb)
        tok = ia
    assert np.array_equal(a.emitted(), b.emitted())


def test_set_kv_layout_is_layer_kv_head_position():
    # swapping K and V, or two kv heads, in the given cache changes the next step
    s = _small_shape()
    w = W.model_weights(s)
    a = O.Oracle(s, w)
    first, _, _ = a.prefill(embeds=W.prefill_embeds(s))
    kv = _cache_of(a, s)
    _, ref, _, _ = a.step(token=first)
    for bad in (kv[:, ::-1], kv[:, :, ::-1], kv[::-1]):
        b = O.Oracle(s, w)
        b.set_kv(np.ascontiguousarray(bad), s.prefill)
        _, lg, _, _ = b.step(token=first)
        assert not np.allclose(lg, ref)


def test_set_kv_picks_the_smallest_bucket_and_rejects_overflow():
    s = _small_shape()
    w = W.model_weights(s)
    o = O.Oracle(s, w)
    o.set_kv(W.batch_stream_kv(s, 0, 40), 40)
    assert (o.pos, o.smax) == (40, 64)
    o.set_kv(np.zeros(0, np.uint16), 0)
    assert (o.pos, o.smax) == (0, 32)
    try:
        o.set_kv(W.batch_stream_kv(s, 0, 65), 65)
        raise AssertionError("accepted a cache longer than the last bucket")
    except O.OracleError as e:
        assert e.status == O.EKVFULL

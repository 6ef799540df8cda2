"""Pins of the oracle's interleaved multimodal RoPE and of prefill with explicit
rotary positions.

The Talker section of "Qwen3-TTS ncnn port: pure C++/ncnn end-to-end reproduction"
fixes the layout: three position streams (t, h, w) with sections [24, 20, 20] over
the 64 rotation frequencies of head_dim 128, interleaved; channel c takes stream
``base % 3`` for ``base = c % 64 < 60`` and stream t otherwise; with equal streams it
is plain RoPE.  The pins probe the oracle's rotation from the outside (which
channels move when only one stream's position is non-zero) and check what RoPE must
satisfy in every stream: scores depend only on position differences.  Decode steps
after a positioned prompt continue at the prompt's largest position + 1 (the reading
this build takes; the pages do not spell it out), which the shift-invariance pin
checks end to end.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W

SEC128 = (24, 20, 20)
SEC64 = (12, 10, 10)


def _moved_channels(hd, section, stream):
    """Channels of a unit vector that the rotation moves when only `stream`'s
    position is non-zero."""
    pos3 = [0, 0, 0]
    pos3[stream] = 1
    moved = set()
    for c in range(hd):
        e = np.zeros(hd, np.float32)
        e[c] = 1.0
        if not np.array_equal(O.rope_mrope(e, pos3, section, 1e6), e):
            moved.add(c)
    return moved


def test_channels_follow_the_pages_interleave():
    hd = 128
    streams = [_moved_channels(hd, SEC128, s) for s in range(3)]
    for c in range(hd):
        base = c % (hd // 2)
        want = base % 3 if base < 60 else 0
        assert [c in streams[s] for s in range(3)] == [s == want for s in range(3)], c
    # 24 / 20 / 20 rotation pairs per stream
    assert [len(x) // 2 for x in streams] == [24, 20, 20]


def test_smaller_head_interleaves_its_own_sections():
    streams = [_moved_channels(64, SEC64, s) for s in range(3)]
    assert [len(x) // 2 for x in streams] == [12, 10, 10]
    assert all(c in streams[(c % 32) % 3] for c in range(60) if c % 32 < 30)


@pytest.mark.parametrize("hd,sec", [(128, SEC128), (64, SEC64)])
def test_equal_streams_are_plain_rope(hd, sec):
    rng = np.random.default_rng(3)
    for p in (0, 1, 17, 399, 1023):
        v = rng.normal(size=hd).astype(np.float32)
        assert np.array_equal(O.rope_mrope(v, (p, p, p), sec, 1e6), O.rope(v, p, 1e6))


def test_plain_rope_ignores_the_h_and_w_streams():
    v = np.random.default_rng(4).normal(size=128).astype(np.float32)
    assert np.array_equal(O.rope_mrope(v, (9, 100, 3), (0, 0, 0), 1e6), O.rope(v, 9, 1e6))


def test_scores_depend_only_on_per_stream_position_differences():
    rng = np.random.default_rng(5)
    hd = 128
    q = rng.normal(size=hd).astype(np.float32)
    k = rng.normal(size=hd).astype(np.float32)

    def score(a, b):
        return float(np.dot(O.rope_mrope(q, a, SEC128, 1e6).astype(np.float64),
                            O.rope_mrope(k, b, SEC128, 1e6).astype(np.float64)))

    a, b = (5, 9, 2), (3, 1, 7)
    s0 = score(a, b)
    for d in [(11, 4, 20), (0, 30, 0), (100, 0, 0), (7, 7, 7)]:
        sa = tuple(x + y for x, y in zip(a, d))
        sb = tuple(x + y for x, y in zip(b, d))
        assert abs(score(sa, sb) - s0) < 1e-4 * hd, d
    # every stream is live: changing one stream's relative position changes the score
    for s in range(3):
        b2 = list(b)
        b2[s] += 3
        assert abs(score(a, tuple(b2)) - s0) > 1e-2, s


def _tiny_mrope():
    return dataclasses.replace(W.TINY, name="tiny_mrope", mrope_section=SEC64)


def _run(shape, w, e, positions, n_steps):
    o = O.Oracle(shape, w)
    rid, rlog, _ = o.prefill(embeds=e, positions=positions)
    ids, logs = [rid], [rlog]
    for _ in range(n_steps):
        rid, rlog, _, _ = o.step(token=ids[-1])
        ids.append(rid)
        logs.append(rlog)
    o.close()
    return ids, np.array(logs)


def test_prompt_positions_equal_to_the_index_are_the_plain_prefill():
    s = _tiny_mrope()
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    n = len(e)
    a = _run(s, w, e, None, 6)
    b = _run(s, w, e, np.tile(np.arange(n, dtype=np.int32), (3, 1)), 6)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_shifted_positions_change_nothing_and_decode_continues_after_the_prompt():
    """Shifting every rotary position by the same amount leaves every score, hence
    every logit, unchanged up to the cos/sin rounding -- through the decode steps too,
    which must continue at the prompt's largest position + 1."""
    s = _tiny_mrope()
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    n = len(e)
    base = _run(s, w, e, None, 6)
    idx = np.tile(np.arange(n, dtype=np.int32), (3, 1))
    # the same shift in every stream: the prompt and six decode steps
    ids, lg = _run(s, w, e, idx + 7, 6)
    assert ids == base[0]
    assert np.max(np.abs(lg - base[1])) < 1e-3
    # a different shift per stream: the prompt (the decode rule then uses equal streams)
    _, lg = _run(s, w, e, idx + np.array([[5], [40], [12]], np.int32), 0)
    assert np.max(np.abs(lg[0] - base[1][0])) < 1e-3


def test_distinct_streams_reach_the_logits_only_with_sections():
    s = _tiny_mrope()
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    n = len(e)
    pos = np.tile(np.arange(n, dtype=np.int32), (3, 1))
    pos2 = pos.copy()
    pos2[1] = np.arange(n)[::-1]                  # the h stream runs backwards
    a = _run(s, w, e, pos, 0)[1][0]
    b = _run(s, w, e, pos2, 0)[1][0]
    assert np.max(np.abs(a - b)) > 1e-2
    plain = dataclasses.replace(W.TINY, name="tiny_plain")
    a = _run(plain, w, e, pos, 0)[1][0]
    b = _run(plain, w, e, pos2, 0)[1][0]
    assert np.array_equal(a, b)


def test_invalid_positions_and_sections():
    s = _tiny_mrope()
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    o = O.Oracle(s, w)
    pos = np.tile(np.arange(len(e), dtype=np.int32), (3, 1))
    pos[2, 3] = -1
    with pytest.raises(O.OracleError):
        o.prefill(embeds=e, positions=pos)
    o.close()
    with pytest.raises(O.OracleError):
        O.Oracle(dataclasses.replace(W.TINY, mrope_section=(12, 10, 9)), w)

"""Interleaved multimodal RoPE on the GPU against the oracle.

A prompt laid out as text, an image grid and text gets distinct t, h, w rotary
positions through ``qd_prefill_mrope``; the decode steps after it rotate at the
prompt's largest position + 1 in all three streams.  Covered paths: the batched
prefill kernels (bf16, no taps), the position-by-position prefill through the decode
step (debug taps on, or the fp32 model), the persistent step and the per-phase
kernels.  Tolerances are the decode path's (``_pair``).
"""
import dataclasses

import numpy as np
import pytest

import workloads as W
from _pair import Pair

pytestmark = pytest.mark.gpu

TALKER2 = dataclasses.replace(W.scaled(W.TALKER, n_layers=2, name="talker2_mrope"), mrope_section=(24, 20, 20))
TINY = dataclasses.replace(W.TINY, name="tiny_mrope", mrope_section=(12, 10, 10))


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _positions(s, n):
    gh, gw = (6, 8) if n >= 64 else (4, 5)
    return W.grid_prompt_positions(n, text_before=n // 6, grid_h=gh, grid_w=gw)


@pytest.mark.parametrize("shape,taps", [(TALKER2, False), (TALKER2, True), (TINY, True)])
@pytest.mark.parametrize("per_phase", [False, True])
def test_grid_prompt_then_decode_matches_oracle(shape, taps, per_phase, monkeypatch):
    if per_phase:
        monkeypatch.setenv("QD_PER_PHASE", "1")
    w = W.model_weights(shape)
    e = W.prefill_embeds(shape)
    n = len(e)
    pos = _positions(shape, n)
    p = Pair(shape, w, taps=taps)
    rid = p.prefill(embeds=e, positions=pos)
    for _ in range(12):
        rid = p.step(token=rid)
    p.trace.check()
    assert p.qd.qd_get_pos(p.h)[0] == n + 12
    p.close()


def test_positions_equal_to_the_index_are_the_plain_prefill():
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    import torch
    s = TALKER2
    w = W.model_weights(s)
    e = torch.from_numpy(W.prefill_embeds(s)).cuda()
    n = e.shape[0]
    y = torch.empty(s.hidden, dtype=torch.float32, device="cuda")

    def run(positions):
        h = qd.qd_create(upload(w), config_from_shape(s))
        if positions is None:
            ids = [qd.qd_prefill(h, embeds=e)]
        else:
            ids = [qd.qd_prefill_mrope(h, positions, embeds=e)]
        for _ in range(6):
            ids.append(qd.qd_decode_step(h, token=ids[-1]))
        qd.qd_get_hidden(h, y)
        out = (ids, y.cpu().numpy().copy())
        qd.qd_destroy(h)
        return out

    a = run(None)
    b = run(np.tile(np.arange(n, dtype=np.int32), (3, 1)))
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_position_errors_rotary_bound_and_reset():
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    import torch
    s = TALKER2
    w = W.model_weights(s)
    e = torch.from_numpy(W.prefill_embeds(s)).cuda()
    n = e.shape[0]
    last = s.buckets[-1]
    h = qd.qd_create(upload(w), config_from_shape(s))
    plain = [qd.qd_prefill(h, embeds=e)]
    plain.append(qd.qd_decode_step(h, token=plain[-1]))
    qd.qd_reset(h)
    # a position outside the table: rejected, the handle stays usable
    bad = np.tile(np.arange(n, dtype=np.int32), (3, 1))
    bad[1, 5] = last
    with pytest.raises(qd.QDError) as ei:
        qd.qd_prefill_mrope(h, bad, embeds=e)
    assert ei.value.status == qd.QD_EINVAL
    # the prompt ends at rotary position last - 3: two decode steps fit, the third does not
    hi = np.tile(np.arange(n, dtype=np.int32), (3, 1))
    hi[2, -1] = last - 3
    first = qd.qd_prefill_mrope(h, hi, embeds=e)
    t = qd.qd_decode_step(h, token=first)
    t = qd.qd_decode_step(h, token=t)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_decode_step(h, token=t)
    assert ei.value.status == qd.QD_EKVFULL
    # a reset returns to the plain positions
    qd.qd_reset(h)
    again = [qd.qd_prefill(h, embeds=e)]
    again.append(qd.qd_decode_step(h, token=again[-1]))
    assert again == plain
    qd.qd_destroy(h)


def test_bad_sections_are_rejected():
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    s = dataclasses.replace(TALKER2, mrope_section=(24, 20, 19))
    with pytest.raises(qd.QDError) as ei:
        qd.qd_create(upload(W.model_weights(TALKER2)), config_from_shape(s))
    assert ei.value.status == qd.QD_EINVAL

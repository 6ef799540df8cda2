"""The decode step with 8-bit weight rows (qd_config.weight_q8) against the oracle.

The GPU quantises the bf16 matrices and output heads at qd_create (codes and half
scales bit-exact with the oracle's quantiser, pinned in test_gpu_q8) and multiplies
each code by its block's scale in the persistent step; the oracle runs the same model
with those matrices dequantised to float32 and the cache in bf16.  The only
differences are the order of the fp32 sums and the cache rounding that both sides
share, so the decode path's acceptance bar applies unchanged: per-layer hidden state
and logits relative L2 <= 2e-3 and equal ids above the top-2 margin.
"""
import numpy as np
import pytest

import workloads as W
from _pair import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _tf(shape, n_steps, taps=True):
    w = W.model_weights(shape)
    p = Pair(shape, w, taps=taps, q8=True)
    tr = p.run_teacher_forced(W.prefill_embeds(shape), n_steps)
    return p, tr


def test_q8_asr_two_layers_crosses_both_migrations():
    s = W.scaled(W.ASR, n_layers=2, name="asr2")
    p, tr = _tf(s, 200)
    tr.check()
    assert p.qd.qd_get_pos(p.h) == (310, 512)
    p.close()


def test_q8_talker_four_layers_gqa_qknorm_penalty():
    s = W.scaled(W.TALKER, n_layers=4, name="talker4")
    p, tr = _tf(s, 100)
    tr.check()
    assert len(tr.hidden_rel) == 100
    p.close()


def test_q8_asr_full_size_graph_path():
    s = W.ASR
    p, tr = _tf(s, s.decode_steps, taps=False)
    tr.check()
    assert p.qd.qd_get_pos(p.h) == (400, 512)
    p.close()


def test_q8_talker_full_size():
    """28 layers at full size, with the taps (every layer's hidden state) for 24 steps,
    then the graph path the benchmark times for 40 more."""
    s = W.TALKER
    p, tr = _tf(s, 24, taps=True)
    tr.check()
    p.close()
    p, tr = _tf(s, 40, taps=False)
    tr.check()
    p.close()


def test_q8_differs_from_bf16_and_refusals():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    s = W.scaled(W.ASR, n_layers=1, name="asr1")
    dev_w = upload(W.model_weights(s))
    e = torch.from_numpy(W.prefill_embeds(s, 8)).cuda()
    hid = []
    for q8 in (False, True):
        h = qd.qd_create(dev_w, config_from_shape(s, weight_q8=q8))
        qd.qd_prefill(h, embeds=e)
        y = torch.empty(s.hidden, dtype=torch.float32, device="cuda")
        qd.qd_get_hidden(h, y)
        hid.append(y.cpu().numpy())
        if q8:
            assert qd.qd_time_kernel(h, 6, 3) > 0.0                      # the whole step
            for which in (0, 1, 2, 3, 5):                                 # per-phase GEMV kernels
                with pytest.raises(qd.QDError) as ei:
                    qd.qd_time_kernel(h, which, 3)
                assert ei.value.status == qd.QD_EUNSUPPORTED
            with pytest.raises(qd.QDError) as ei:
                qd.qd_batch_create(h, 4, 256)
            assert ei.value.status == qd.QD_EUNSUPPORTED
        qd.qd_destroy(h)
    # the 8-bit model is a different model: close to the bf16 one, not equal
    d = np.linalg.norm(hid[0] - hid[1]) / np.linalg.norm(hid[0])
    assert 0.0 < d < 0.1

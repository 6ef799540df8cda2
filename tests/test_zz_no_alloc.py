"""The allocation-free output head gives the same result as the decode step's head.

qd_head_argmax_noalloc serves callers that cannot allocate device memory (a host
application that owns every device buffer through its own pool, or a real-time
thread where an allocation's locking and synchronisation are not allowed): it takes
only the caller's buffers and keeps its scratch in a fixed device array.  For the
normalised hidden state of a decode step (qd_get_hidden) and the step's emitted set,
it must produce the step's logits and id, on two calls in a row (the second call
reuses the array the first one left behind), and the oracle's: W_head . y in the
oracle's own matvec, then its penalty, EOS mask and argmax over the same emitted set
(equal ids wherever the oracle's top-2 margin exceeds the acceptance margin).
Collected last so that a failure here comes after every other test has run.
"""
import numpy as np
import pytest

import workloads as W
from _pair import MARGIN, REL_TOL, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape_name", ["asr2", "talker2"])
def test_noalloc_head_matches_decode_step(shape_name, cuda_ok):
    import torch
    import __graft_entry__
    import oracle as O
    __graft_entry__.build_library()
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload

    s = {"asr2": W.scaled(W.ASR, n_layers=2, name="asr2"),
         "talker2": W.scaled(W.TALKER, n_layers=2, name="talker2")}[shape_name]
    w = W.model_weights(s)
    dev_w = upload(w)
    h = qd.qd_create(dev_w, config_from_shape(s))
    logits_tap = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    qd.qd_set_debug_taps(h, None, logits_tap)
    tok = qd.qd_prefill(h, embeds=torch.from_numpy(W.prefill_embeds(s, 50)).cuda())
    y = torch.empty(s.hidden, dtype=torch.float32, device="cuda")
    emitted = torch.empty((s.vocab + 31) // 32, dtype=torch.int32, device="cuda")
    out_id = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    for _ in range(2):                                   # two calls in a row
        tok = qd.qd_decode_step(h, token=tok)
        qd.qd_get_hidden(h, y)
        qd.qd_get_emitted(h, emitted)
        qd.qd_head_argmax_noalloc(y, dev_w["lm_head.0"], s.vocab, s.hidden, s.bf16, emitted, s.rep_penalty,
                                  s.eos_mask_id, out_id, logits)
        torch.cuda.synchronize()
        assert int(out_id.item()) == tok
        got = logits.cpu().numpy()
        assert rel_l2(got, logits_tap.cpu().numpy()) <= REL_TOL
        # against the oracle, from the same normalised hidden state and emitted set
        em = emitted.cpu().numpy().view(np.uint32)
        ids_em = [i for i in range(s.vocab) if (em[i >> 5] >> (i & 31)) & 1]
        ref = O.linear(w["lm_head.0"], y.cpu().numpy()[None])[0]
        ref_id, _, margin = O.penalty_argmax(ref, ids_em, s.rep_penalty, s.eos_mask_id)
        assert rel_l2(got, ref) <= REL_TOL
        if margin > MARGIN:
            assert int(out_id.item()) == ref_id
    # host buffers are refused before any work
    with pytest.raises(qd.QDError) as ei:
        qd.qd_head_argmax_noalloc(y.cpu(), dev_w["lm_head.0"], s.vocab, s.hidden, s.bf16, emitted, s.rep_penalty,
                                  s.eos_mask_id, out_id, logits)
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_head_argmax_noalloc(y, dev_w["lm_head.0"], s.vocab, s.hidden, s.bf16, emitted, s.rep_penalty,
                                  -2, out_id, logits)
    assert ei.value.status == qd.QD_EINVAL
    qd.qd_destroy(h)

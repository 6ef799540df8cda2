"""On-device sampling (top-k, temperature, top-p, SplitMix64 counter draws) against the
oracle's sampler.

Both sides draw u = draw n_gen of the seed's sequence, bit-identically (integer
arithmetic), and apply the same steps; only the logits differ, within the decode
tolerance.  Teacher-forced with the oracle's ids, the GPU's id must equal the oracle's
wherever the oracle's decision margin (see orc_sample: distances of the draw and of the
top-p cut from the cumulative boundaries, and of the picked logit from its neighbours)
exceeds ten times what the step's logit error can move it: the largest difference
between the GPU's raw logits (debug tap) and the oracle's, over the temperature.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": W.TINY,
    "asr2": W.scaled(W.ASR, n_layers=2, name="asr2"),
    "talker2": W.scaled(W.TALKER, n_layers=2, name="talker2"),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _model(s, w):
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    return qd, qd.qd_create(upload(w), config_from_shape(s))


def _free_run(s, w, e, n, sampling=None):
    import torch
    qd, h = _model(s, w)
    if sampling is not None:
        qd.qd_set_sampling(h, *sampling)
    ids = [qd.qd_prefill(h, embeds=torch.from_numpy(e).cuda())]
    for _ in range(n):
        ids.append(qd.qd_decode_step(h, token=ids[-1]))
    qd.qd_destroy(h)
    return ids


@pytest.mark.parametrize("shape_name,k,t", [("tiny", 50, 0.9), ("asr2", 50, 0.9), ("talker2", 8, 0.7)])
def test_sampled_ids_match_oracle(shape_name, k, t):
    """talker2's bf16 logits lie too close together among its top 50 for the error
    bound to decide most draws there; 8 candidates at temperature 0.7 are resolvable."""
    import torch
    import oracle as O
    s = SHAPES[shape_name]
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    p, seed = 0.95, 1234
    qd, h = _model(s, w)
    hid = torch.empty((s.n_layers + 1, s.hidden), dtype=torch.float32, device="cuda")
    lg = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    qd.qd_set_debug_taps(h, hid, lg)
    qd.qd_set_sampling(h, k, t, p, seed)
    o = O.Oracle(s, w)
    o.set_sampling(k, t, p, seed)
    gid = qd.qd_prefill(h, embeds=torch.from_numpy(e).cuda())
    rid, rlog, margin = o.prefill(embeds=e)
    checked = 0
    steps = 8 if shape_name == "tiny" else 30
    for i in range(steps + 1):
        err = float(np.abs(lg.cpu().numpy() - rlog).max())
        assert err < 1e-2, (i, err)
        if margin > 10 * err / min(t, 1.0):
            assert gid == rid, (i, gid, rid, margin, err)
            checked += 1
        if i == steps:
            break
        gid = qd.qd_decode_step(h, token=rid)
        rid, rlog, margin, _ = o.step(token=rid)
    assert checked >= (steps + 1) // 3, checked
    o.close()
    qd.qd_destroy(h)


@pytest.mark.parametrize("shape_name", ["tiny", "asr2"])
def test_top1_sampling_equals_greedy(shape_name):
    s = SHAPES[shape_name]
    w = W.model_weights(s)
    e = W.prefill_embeds(s, 40)
    n = 12
    assert _free_run(s, w, e, n, (1, 0.7, 1.0, 99)) == _free_run(s, w, e, n)


@pytest.mark.parametrize("shape_name", ["tiny", "asr2"])
def test_sampling_persistent_step_equals_per_phase_kernels(shape_name, monkeypatch):
    s = SHAPES[shape_name]
    w = W.model_weights(s)
    e = W.prefill_embeds(s, 40)
    a = _free_run(s, w, e, 16, (40, 1.1, 0.9, 7))
    monkeypatch.setenv("QD_PER_PHASE", "1")
    b = _free_run(s, w, e, 16, (40, 1.1, 0.9, 7))
    assert a == b


@pytest.mark.parametrize("shape_name", ["tiny", "asr2"])
@pytest.mark.parametrize("per_phase", [False, True])
@pytest.mark.parametrize("k,p", [(50, 1.0), (64, 0.93)])
def test_all_equal_logits(shape_name, per_phase, k, p, monkeypatch):
    """A zero LM head makes every logit exactly 0 on both sides (the EOS id -inf): the
    candidates are the k lowest ids, every per-CTA selection runs into ties and the merge
    keeps far more entries than it ranks directly.  With exact logits the draws agree
    without a margin (the cumulative weights are small integers)."""
    import torch
    import oracle as O
    s = SHAPES[shape_name]
    w = W.model_weights(s)
    for j in range(s.n_heads_out):
        w[f"lm_head.{j}"] = np.zeros_like(w[f"lm_head.{j}"])
    e = W.prefill_embeds(s, 20)
    if per_phase:
        monkeypatch.setenv("QD_PER_PHASE", "1")
    t, seed, n = 0.9, 21, 10
    got = _free_run(s, w, e, n, (k, t, p, seed))
    o = O.Oracle(s, w)
    o.set_sampling(k, t, p, seed)
    ref = [o.prefill(embeds=e)[0]]
    for _ in range(n):
        ref.append(o.step(token=ref[-1])[0])
    o.close()
    assert got == ref
    assert max(ref) < k + 1 and len(set(ref)) > 1


def test_sampling_settings_seed_reset_and_errors():
    import torch
    s = SHAPES["asr2"]
    w = W.model_weights(s)
    e = torch.from_numpy(W.prefill_embeds(s, 40)).cuda()
    qd, h = _model(s, w)

    def run(n=10):
        qd.qd_reset(h)
        ids = [qd.qd_prefill(h, embeds=e)]
        for _ in range(n):
            ids.append(qd.qd_decode_step(h, token=ids[-1]))
        return ids

    greedy = run()
    qd.qd_set_sampling(h, 50, 1.5, 1.0, 5)
    a, b = run(), run()                       # the settings survive a reset; the draws restart
    assert a == b and a != greedy
    qd.qd_set_sampling(h, 50, 1.5, 1.0, 6)
    assert run() != a
    qd.qd_set_sampling(h, 0, 1.0, 1.0, 0)
    assert run() == greedy
    for args in [(65, 1.0, 1.0, 0), (-1, 1.0, 1.0, 0), (10, 0.0, 1.0, 0), (10, 1.0, 0.0, 0), (10, 1.0, 1.5, 0)]:
        with pytest.raises(qd.QDError) as ei:
            qd.qd_set_sampling(h, *args)
        assert ei.value.status == qd.QD_EINVAL
    qd.qd_destroy(h)

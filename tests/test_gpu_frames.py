"""Parity of the device-resident two-level frame loop (qd_frame_generate) with the
oracle's frame loop.

The oracle runs free; the GPU is fed the oracle's ids (teacher forcing through the
call's force argument), so every argmax of every frame is comparable.  Bars: ids
equal wherever the oracle's top-2 margin exceeds 1e-2; summed embeddings and
hidden states within relative L2 2e-3; positions and emitted sets exact.
"""
import numpy as np
import pytest

import workloads as W
from _pair import MARGIN, REL_TOL, rel_l2

pytestmark = pytest.mark.gpu

# Reduced pair: the real dimensions (hidden 1024, 16/8 heads of 128, FFN 3072,
# vocabularies 3072 and 2048, 15 predictor heads) with 2 layers each.
TALKER2 = W.scaled(W.TALKER, n_layers=2, name="talker2")
CP2 = W.scaled(W.CODE_PREDICTOR, n_layers=2, name="cp2")


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


class FramePair:
    def __init__(self, ts, cs, talker_buckets=None, seed=0):
        import torch
        import oracle as O
        import transformer_autoregressive_decode_gb300 as qd
        from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, to_device, upload

        self.qd, self.torch, self.ts, self.cs = qd, torch, ts, cs
        tw = W.model_weights(ts, seed=seed)
        cw = W.model_weights(cs, seed=seed)
        tables = W.frame_tables(seed=seed, rows=cs.vocab, hidden=ts.hidden)
        code_tables = [tables[f"code_embed.{j}"] for j in range(1, 16)]
        self.T = qd.qd_create(upload(tw), config_from_shape(ts, talker_buckets))
        self.C = qd.qd_create(upload(cw), config_from_shape(cs))
        dev_tables = [to_device(t) for t in code_tables]
        self.F = qd.qd_frame_create(self.T, self.C, dev_tables, bf16=ts.bf16)
        del dev_tables                                   # the frame handle holds its own copy
        self.ot = O.Oracle(ts, tw, buckets=talker_buckets)
        self.oc = O.Oracle(cs, cw)
        self.loop = O.FrameLoop(self.ot, self.oc, tw["embed"], code_tables)
        self.prompt = W.prefill_embeds(ts)
        self.y = torch.empty(ts.hidden, dtype=torch.float32, device="cuda")

    def dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def prefill(self):
        g = self.qd.qd_prefill(self.T, embeds=self.dev(self.prompt))
        r, _, m = self.ot.prefill(embeds=self.prompt, want_logits=False)
        return g, r, m

    def oracle_frames(self, n, text, primary, margin):
        return self.loop.generate(n, text, primary, margin)

    def gpu_frames(self, n, text, force=None):
        torch = self.torch
        codes = torch.full((n, 16), -1, dtype=torch.int32, device="cuda")
        nxt = torch.empty(self.ts.hidden, dtype=torch.float32, device="cuda")
        self.qd.qd_frame_generate(self.F, n, self.dev(text), codes, None if force is None else self.dev(force), nxt)
        torch.cuda.synchronize()
        return codes.cpu().numpy(), nxt.cpu().numpy()

    def talker_hidden(self):
        self.qd.qd_get_hidden(self.T, self.y)
        return self.y.cpu().numpy()

    def talker_emitted(self):
        words = self.torch.zeros((self.ts.vocab + 31) // 32, dtype=self.torch.int32, device="cuda")
        self.qd.qd_get_emitted(self.T, words)
        return words.cpu().numpy().view(np.uint32)

    def close(self):
        self.qd.qd_frame_destroy(self.F)
        self.qd.qd_destroy(self.C)
        self.qd.qd_destroy(self.T)
        self.ot.close()
        self.oc.close()


def _assert_ids(got, ref, margins):
    sel = margins > MARGIN
    bad = np.argwhere(sel & (got != ref))
    assert len(bad) == 0, f"id mismatches above the margin at (frame, code) {bad[:10].tolist()}"


def _teacher_forced(ts, cs, n, talker_buckets=None):
    fp = FramePair(ts, cs, talker_buckets)
    text = W.frame_text_embeds(n, hidden=ts.hidden)
    g0, r0, m0 = fp.prefill()
    if m0 > MARGIN:
        assert g0 == r0
    codes_r, margins_r, next_r, _ = fp.oracle_frames(n, text, r0, m0)
    force = codes_r.copy()
    force[0, 0] = r0
    codes_g, next_g = fp.gpu_frames(n, text, force)
    _assert_ids(codes_g, codes_r, margins_r)
    assert rel_l2(next_g, next_r[-1]) <= REL_TOL
    assert rel_l2(fp.talker_hidden(), fp.ot.hidden()) <= REL_TOL
    assert fp.qd.qd_get_pos(fp.T)[0] == ts.prefill + n - 1
    assert fp.qd.qd_get_pos(fp.C) == (16, cs.buckets[0])
    assert np.array_equal(fp.talker_emitted(), fp.ot.emitted())
    return fp, codes_g, margins_r


def test_frames_reduced_teacher_forced():
    fp, codes, margins = _teacher_forced(TALKER2, CP2, 6)
    assert codes.min() >= 0
    assert (margins > MARGIN).mean() > 0.5        # the comparison is not vacuous
    fp.close()


def test_frames_one_call_per_frame_match_each_frame():
    """One frame per call, the Talker step issued by the caller in between: every
    frame's summed embedding and the Talker's hidden state match the oracle's."""
    n = 4
    fp = FramePair(TALKER2, CP2)
    text = W.frame_text_embeds(n, hidden=TALKER2.hidden)
    g0, r0, m0 = fp.prefill()
    codes_r, margins_r, next_r, h_t_r = fp.oracle_frames(n, text, r0, m0)
    force = codes_r.copy()
    force[0, 0] = r0
    nxt = fp.torch.empty(TALKER2.hidden, dtype=fp.torch.float32, device="cuda")
    codes = fp.torch.empty((1, 16), dtype=fp.torch.int32, device="cuda")
    for f in range(n):
        assert rel_l2(fp.talker_hidden(), h_t_r[f]) <= REL_TOL, f
        fp.qd.qd_frame_generate(fp.F, 1, fp.dev(text[f:f + 1]), codes, fp.dev(force[f:f + 1]), nxt)
        got = codes.cpu().numpy()[0]
        sel = margins_r[f, 1:] > MARGIN
        assert np.array_equal(got[1:][sel], codes_r[f, 1:][sel]), f
        assert rel_l2(nxt.cpu().numpy(), next_r[f]) <= REL_TOL, f
        if f < n - 1:
            pid = fp.qd.qd_decode_step(fp.T, embed=nxt, token=int(force[f, 0]))
            if margins_r[f + 1, 0] > MARGIN:
                assert pid == codes_r[f + 1, 0], f
    fp.close()


def test_free_run_equals_run_forced_with_its_own_ids():
    n = 5
    text = W.frame_text_embeds(n, hidden=TALKER2.hidden)
    a = FramePair(TALKER2, CP2)
    g0, _, _ = a.prefill()
    free_codes, free_next = a.gpu_frames(n, text)
    assert free_codes[0, 0] == g0
    free_hidden = a.talker_hidden()
    a.close()
    b = FramePair(TALKER2, CP2)
    b.prefill()
    forced_codes, forced_next = b.gpu_frames(n, text, free_codes)
    assert np.array_equal(forced_codes, free_codes)
    assert np.array_equal(forced_next, free_next)
    assert np.array_equal(b.talker_hidden(), free_hidden)
    b.close()


def test_frame_graphs_equal_eager_and_repeat():
    n = 3
    text = W.frame_text_embeds(n, hidden=TALKER2.hidden)
    out = []
    for graphs in (True, False, True):
        fp = FramePair(TALKER2, CP2)
        fp.qd.qd_frame_set_graphs(fp.F, graphs)
        fp.prefill()
        out.append(fp.gpu_frames(n, text))
        fp.close()
    for codes, nxt in out[1:]:
        assert np.array_equal(codes, out[0][0]) and np.array_equal(nxt, out[0][1])


def test_frames_cross_a_talker_bucket():
    # buckets 64 -> 128: prefill 64 fills the first, the first Talker step migrates
    fp, _, _ = _teacher_forced(TALKER2, CP2, 4, talker_buckets=(64, 128))
    assert fp.qd.qd_get_pos(fp.T) == (67, 128)
    fp.close()


def test_frame_errors():
    import torch
    fp = FramePair(TALKER2, CP2, talker_buckets=(64, 128))
    qd = fp.qd
    text = fp.dev(W.frame_text_embeds(70, hidden=TALKER2.hidden))
    codes = torch.empty((70, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(qd.QDError) as ei:          # the Talker has produced no id
        qd.qd_frame_generate(fp.F, 1, text, codes)
    assert ei.value.status == qd.QD_ESTATE
    fp.prefill()
    with pytest.raises(qd.QDError) as ei:          # 64 + 65 positions > 128
        qd.qd_frame_generate(fp.F, 66, text, codes)
    assert ei.value.status == qd.QD_EKVFULL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_frame_generate(fp.F, 1, text.cpu(), codes)
    assert ei.value.status == qd.QD_EINVAL
    assert qd.qd_get_pos(fp.T) == (64, 64)         # nothing ran
    # a forced id outside its table: the kernels' bounds checks flag it on the device
    force = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    force[0, 5] = CP2.vocab + 7
    qd.qd_frame_generate(fp.F, 1, text, codes, force)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_decode_step(fp.C, embed=text[0], head_idx=1)
    assert ei.value.status == qd.QD_EDEVICE
    qd.qd_reset(fp.C)                              # the status clears with a reset
    fp.close()
    # mismatched handles
    a = FramePair(TALKER2, CP2)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_frame_create(a.T, a.T, [torch.zeros((2048, 1024), dtype=torch.bfloat16, device="cuda")] * 15, True)
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_frame_create(a.T, a.C, [torch.zeros((16, 1024), dtype=torch.bfloat16, device="cuda")] * 15, True)
    assert ei.value.status == qd.QD_EINVAL        # fewer rows than the predictor's vocabulary
    a.close()


def test_destroying_a_model_first_detaches_the_frame_handle():
    import torch
    fp = FramePair(TALKER2, CP2)
    qd = fp.qd
    fp.prefill()
    codes, _ = fp.gpu_frames(2, W.frame_text_embeds(2, hidden=TALKER2.hidden))
    qd.qd_destroy(fp.C)                            # waits for the frame work, detaches
    text = fp.dev(W.frame_text_embeds(1, hidden=TALKER2.hidden))
    out = torch.empty((1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_frame_generate(fp.F, 1, text, out)
    assert ei.value.status == qd.QD_ESTATE
    qd.qd_frame_destroy(fp.F)
    assert qd.qd_decode_step(fp.T, embed=text[0], token=int(codes[1, 0])) >= 0   # the Talker is intact
    qd.qd_destroy(fp.T)
    fp.ot.close()
    fp.oc.close()


def test_frames_sampled_match_oracle():
    """Sampling in the frame loop on the Talker and the Code Predictor: each model draws
    u from its seed at its own counter (ids produced since its last reset; the predictor
    restarts every frame, as its id history does), on both sides.  Teacher-forced with
    the oracle's draws, every code whose draw the oracle's margin decides (beyond ten
    times a 2e-3 logit error over the temperature) equals the oracle's.  8 candidates at
    temperature 0.7: on these 2-layer shapes the 50 best logits of the pages' default
    lie too close together for most draws to be decidable (the batched test checks the
    sampler itself at the default settings)."""
    n, k, t, p = 6, 8, 0.7, 1.0
    fp = FramePair(TALKER2, CP2)
    for h, o, seed in ((fp.T, fp.ot, 11), (fp.C, fp.oc, 22)):
        fp.qd.qd_set_sampling(h, k, t, p, seed)
        o.set_sampling(k, t, p, seed)
    text = W.frame_text_embeds(n, hidden=TALKER2.hidden)
    g0, r0, m0 = fp.prefill()
    codes_r, margins_r, next_r, _ = fp.oracle_frames(n, text, r0, m0)
    force = codes_r.copy()
    force[0, 0] = r0
    codes_g, next_g = fp.gpu_frames(n, text, force)
    decided = margins_r > 10 * 2e-3 / t
    bad = np.argwhere(decided & (codes_g != codes_r))
    assert len(bad) == 0, f"sampled codes differ at (frame, code) {bad[:10].tolist()}"
    assert decided.mean() >= 0.1, decided.mean()           # the comparison is not vacuous
    assert rel_l2(next_g, next_r[-1]) <= REL_TOL
    # and the draws are not the argmax throughout: sampling took effect
    fg = FramePair(TALKER2, CP2)
    fg.prefill()
    greedy, _ = fg.gpu_frames(n, text, force)
    assert (greedy[:, 1:] != codes_g[:, 1:]).any()
    fg.close()
    fp.close()


@pytest.mark.slow
def test_frames_full_size():
    """The frame workload at full size: 28-layer Talker, 5-layer Code Predictor,
    150 frames (149 Talker steps, 2400 predictor positions), Talker cache 128 -> 256."""
    n = W.FRAME_COUNT
    fp, codes, margins = _teacher_forced(W.TALKER, W.CODE_PREDICTOR, n)
    assert fp.qd.qd_get_pos(fp.T) == (W.TALKER.prefill + n - 1, 256)
    fp.close()


@pytest.mark.slow
def test_frames_full_size_per_frame_logits():
    """The full-size frame workload one frame per call, with debug taps on both models:
    for every one of the 150 frames, the Code Predictor's last head (14) logits and
    final-norm state, and the Talker step's logits and per-layer hidden states, against
    the oracle's, within relative L2 2e-3; every code above the margin equal.  The
    oracle's predictor starts each frame from the GPU Talker's final-norm state (the
    predictor's first input), so its comparison measures the predictor alone; the
    Talker chains run side by side, fed the same ids."""
    import oracle as O
    ts, cs = W.TALKER, W.CODE_PREDICTOR
    n = W.FRAME_COUNT
    fp = FramePair(ts, cs)
    torch = fp.torch
    qd = fp.qd
    cw = W.model_weights(cs)
    head14 = cw["lm_head.14"]
    c_logits = torch.empty(cs.vocab, dtype=torch.float32, device="cuda")
    c_hidden = torch.empty((cs.n_layers + 1, cs.hidden), dtype=torch.float32, device="cuda")
    t_logits = torch.empty(ts.vocab, dtype=torch.float32, device="cuda")
    t_hidden = torch.empty((ts.n_layers + 1, ts.hidden), dtype=torch.float32, device="cuda")
    qd.qd_set_debug_taps(fp.C, c_hidden, c_logits)
    qd.qd_set_debug_taps(fp.T, t_hidden, t_logits)
    text = W.frame_text_embeds(n, hidden=ts.hidden)
    g0, r0, m0 = fp.prefill()
    if m0 > MARGIN:
        assert g0 == r0
    primary, pm = r0, m0
    nxt = torch.empty(ts.hidden, dtype=torch.float32, device="cuda")
    codes = torch.empty((1, 16), dtype=torch.int32, device="cuda")
    worst = {"cp_logits": 0.0, "cp_y": 0.0, "talker_logits": 0.0, "talker_hidden": 0.0}
    class _GpuTalkerState:
        """The Talker as the predictor's frame start sees it: the GPU's final-norm state."""
        def hidden(self):
            return _final_y(qd, fp.T, ts)
    loop = O.FrameLoop(_GpuTalkerState(), fp.oc, fp.loop.tables[0], fp.loop.tables[1:])
    for f in range(n):
        codes_r, margins_r, next_r, _ = loop.generate(1, text[f:f + 1], primary, pm)
        force = codes_r.copy()
        qd.qd_frame_generate(fp.F, 1, fp.dev(text[f:f + 1]), codes, fp.dev(force), nxt)
        got = codes.cpu().numpy()
        _assert_ids(got, codes_r, margins_r)
        y_ref = fp.oc.hidden()
        worst["cp_y"] = max(worst["cp_y"], rel_l2(_final_y(qd, fp.C, cs), y_ref))
        worst["cp_logits"] = max(worst["cp_logits"],
                                 rel_l2(c_logits.cpu().numpy(), O.linear(head14, y_ref[None])[0]))
        assert rel_l2(nxt.cpu().numpy(), next_r[0]) <= REL_TOL, f
        if f < n - 1:
            p = int(force[0, 0])
            pid = qd.qd_decode_step(fp.T, embed=nxt, token=p)
            primary, rlog, pm, rtaps = fp.ot.step(token=p, embed=next_r[0], head_idx=0, taps=True)
            if pm > MARGIN:
                assert pid == primary, f
            worst["talker_logits"] = max(worst["talker_logits"], rel_l2(t_logits.cpu().numpy(), rlog))
            g = t_hidden.cpu().numpy()
            worst["talker_hidden"] = max(worst["talker_hidden"],
                                         max(rel_l2(g[l], rtaps[l]) for l in range(len(rtaps))))
    assert max(worst.values()) <= REL_TOL, worst
    assert qd.qd_get_pos(fp.T) == (ts.prefill + n - 1, 256)
    fp.close()


def _final_y(qd, h, shape):
    import torch
    y = torch.empty(shape.hidden, dtype=torch.float32, device="cuda")
    qd.qd_get_hidden(h, y)
    return y.cpu().numpy()

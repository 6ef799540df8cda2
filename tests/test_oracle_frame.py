"""Pins of the oracle's two-level frame loop (CPU only).

The frame loop composes pieces that are pinned elsewhere (the decoder step, the
penalty and argmax); what it adds is the wiring: which vector enters which model
at which position, which table a code indexes, which head decodes it, and which
id joins which emitted set.  These tests rebuild each model's input sequence from
the definition ("Qwen3-TTS ncnn port", section "Talker: non-standard structure and
two-level generation") and recompute every argmax from scratch with the uncached
full-prefix route, so a wiring mistake (a table off by one, a head off by one, the
wrong hidden state as the predictor's first position, a code that skips the sum,
the primary missing from the Talker's emitted set) fails here.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

# Small Talker/Code-Predictor pair with the real structure (GQA, QK-norm, penalty
# 1.05 on the Talker, 15 predictor heads) and dimensions the oracle runs in
# milliseconds.
TALKER_S = W.scaled(W.TALKER, name="talker_s", hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32,
                    ffn=256, vocab=96, embed_rows=96, buckets=(32, 64), prefill=6)
CP_S = W.scaled(W.CODE_PREDICTOR, name="cp_s", hidden=128, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=32,
                ffn=256, vocab=48, buckets=(16,))
CODE_ROWS = 48


def _setup(n_frames, seed=0):
    tw = W.model_weights(TALKER_S, seed=seed)
    cw = W.model_weights(CP_S, seed=seed)
    tables = W.frame_tables(seed=seed, rows=CODE_ROWS, hidden=TALKER_S.hidden)
    code_tables = [tables[f"code_embed.{j}"] for j in range(1, 16)]
    text = W.frame_text_embeds(n_frames, seed=seed, hidden=TALKER_S.hidden)
    prompt = W.prefill_embeds(TALKER_S)
    return tw, cw, code_tables, text, prompt


def _run(n_frames, force=None, seed=0):
    tw, cw, code_tables, text, prompt = _setup(n_frames, seed)
    talker = O.Oracle(TALKER_S, tw)
    cp = O.Oracle(CP_S, cw)
    p0, _, m0 = talker.prefill(embeds=prompt)
    loop = O.FrameLoop(talker, cp, tw["embed"], code_tables)
    out = loop.generate(n_frames, text, p0, m0, force=force)
    return (tw, cw, code_tables, text, prompt, talker, cp) + out


# ----------------------------------------------------------------- embedding sum

def test_frame_sum_pairs_each_code_with_its_own_table():
    # table j is zero except column j of row r, which holds r + 1: the sum is then
    # exactly ids_j + 1 in column j, so any table/code mispairing shows
    hidden, rows = 16, 40
    tables = []
    for j in range(16):
        t = np.zeros((rows, hidden), np.float32)
        t[:, j] = np.arange(rows, dtype=np.float32) + 1
        tables.append(t)
    ids = [(7 * j + 3) % rows for j in range(16)]
    out = O.frame_sum(tables, ids, np.zeros(hidden, np.float32))
    assert np.array_equal(out, np.array(ids, np.float32) + 1)
    text = np.arange(hidden, dtype=np.float32) * 0.5
    assert np.array_equal(O.frame_sum(tables, ids, text), np.array(ids, np.float32) + 1 + text)


def test_frame_sum_exact_on_small_integers_bf16():
    rng = np.random.default_rng(5)
    vals = rng.integers(-100, 100, size=(16, 8, 32)).astype(np.float32)     # exact in bf16
    tables = [(v.view(np.uint32) >> 16).astype(np.uint16) for v in vals]
    ids = rng.integers(0, 8, size=16)
    text = rng.integers(-5, 5, size=32).astype(np.float32)
    ref = sum(vals[j, ids[j]] for j in range(16)) + text
    assert np.array_equal(O.frame_sum(tables, ids, text), ref.astype(np.float32))


def test_frame_sum_within_fp32_bound_of_fp64_sum():
    tables = [W.normal(f"fs{j}", (64, 256), seed=2, std=0.02, bf16=True) for j in range(16)]
    ids = W.uniform_int("fs_ids", 16, 0, 63, seed=2)
    text = W.normal("fs_text", (256,), seed=2)
    rows = [O.table_row(tables[j], ids[j]).astype(np.float64) for j in range(16)]
    exact = np.sum(rows, axis=0) + text.astype(np.float64)
    bound = 17 * 2.0 ** -24 * (np.sum(np.abs(rows), axis=0) + np.abs(text))
    err = np.abs(O.frame_sum(tables, ids, text).astype(np.float64) - exact)
    assert np.all(err <= bound)


def test_table_row_widens_bf16_bits():
    t = np.array([[0x3F80, 0xC000, 0x0000, 0x3E80]], np.uint16)     # 1, -2, 0, 0.25
    assert np.array_equal(O.table_row(t, 0), np.array([1.0, -2.0, 0.0, 0.25], np.float32))


# ----------------------------------------------------------------- loop wiring

def _wiring_errors(tw, cw, code_tables, text, prompt, codes, h_t, next_in):
    """Rebuild both models' inputs from the definition and recompute every argmax
    from scratch; returns the places where the loop's outputs disagree."""
    errors = []
    n = len(codes)
    tables = [tw["embed"]] + code_tables
    talker_inputs = [prompt]
    primaries = []
    head = (tw["lm_head.0"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for f in range(n):
        p = int(codes[f, 0])
        primaries.append(p)
        raw = O.recompute_logits(TALKER_S, tw, embeds=np.concatenate(talker_inputs))
        if f > 0:
            # the primary: Talker over the prompt and every earlier frame's sum, the
            # repetition penalty over the primaries fed back so far
            pid, _, _ = O.penalty_argmax(raw, primaries[:-1], TALKER_S.rep_penalty)
            if pid != p:
                errors.append(("primary", f))
        # h_T is the Talker's final-norm output at its last position: the head
        # applied to it gives that position's raw logits
        if not np.allclose(head @ h_t[f].astype(np.float64), raw, rtol=1e-4, atol=1e-5):
            errors.append(("h_T", f))
        # the predictor: [h_T, E_0[p], E_1[c_1], ..., E_j[c_j]] decoded by head j
        cp_seq = [h_t[f], O.table_row(tables[0], p)]
        for j in range(15):
            if j > 0:
                cp_seq.append(O.table_row(tables[j], codes[f, j]))
            raw_c = O.recompute_logits(CP_S, cw, embeds=np.stack(cp_seq), head_idx=j)
            cid, _, _ = O.penalty_argmax(raw_c, [], 1.0)
            if cid != codes[f, j + 1]:
                errors.append(("code", f, j + 1))
        # the sum uses every code of the frame, each in its own table, and the text
        rows = [O.table_row(tables[j], codes[f, j]).astype(np.float64) for j in range(16)]
        exact = np.sum(rows, axis=0) + text[f]
        if np.max(np.abs(next_in[f] - exact)) >= 1e-5:
            errors.append(("sum", f))
        talker_inputs.append(next_in[f][None, :])
    return errors


def test_frame_loop_matches_full_recompute_of_both_models():
    n = 3
    (tw, cw, code_tables, text, prompt, talker, cp, codes, margins, next_in, h_t) = _run(n)
    assert _wiring_errors(tw, cw, code_tables, text, prompt, codes, h_t, next_in) == []
    # n frames ran n - 1 Talker steps; the predictor holds 16 positions (context <= 17)
    assert talker.pos == TALKER_S.prefill + n - 1
    assert cp.pos == 16


class _HeadShift:
    """A predictor whose steps decode with the previous head (a planted mistake)."""

    def __init__(self, o):
        self.o = o

    def __getattr__(self, k):
        return getattr(self.o, k)

    def step(self, **kw):
        kw["head_idx"] = max(0, kw["head_idx"] - 1)
        return self.o.step(**kw)


class _FirstPositionIsInput:
    """A Talker whose reported hidden state is its last input, not its final-norm output."""

    def __init__(self, o, inputs):
        self.o, self.inputs = o, inputs

    def __getattr__(self, k):
        return getattr(self.o, k)

    def hidden(self):
        return self.inputs[-1]

    def step(self, **kw):
        self.inputs.append(kw["embed"])
        return self.o.step(**kw)


@pytest.mark.parametrize("mutant", ["tables_rotated", "text_dropped", "head_shift", "hidden_is_input"])
def test_planted_wiring_mistakes_are_caught(mutant):
    n = 2
    tw, cw, code_tables, text, prompt = _setup(n)
    talker = O.Oracle(TALKER_S, tw)
    cp = O.Oracle(CP_S, cw)
    p0, _, m0 = talker.prefill(embeds=prompt)
    tabs, txt = code_tables, text
    if mutant == "tables_rotated":
        tabs = code_tables[1:] + code_tables[:1]
    if mutant == "text_dropped":
        txt = np.zeros_like(text)
    if mutant == "head_shift":
        cp = _HeadShift(cp)
    if mutant == "hidden_is_input":
        talker = _FirstPositionIsInput(talker, [prompt[-1]])
    codes, _, next_in, h_t = O.FrameLoop(talker, cp, tw["embed"], tabs).generate(n, txt, p0, m0)
    assert _wiring_errors(tw, cw, code_tables, text, prompt, codes, h_t, next_in) != []


def test_primary_joins_the_talker_emitted_set():
    n = 3
    (_, _, _, _, _, talker, _, codes, _, _, _) = _run(n)
    words = talker.emitted()
    got = {i for i in range(TALKER_S.vocab) if words[i >> 5] >> (i & 31) & 1}
    assert got == {int(c) for c in codes[: n - 1, 0]}     # the last frame's primary is not fed back yet


def test_forcing_with_own_codes_reproduces_the_free_run():
    n = 3
    free = _run(n)
    codes, next_in = free[7], free[9]
    forced = _run(n, force=codes.copy())
    assert np.array_equal(forced[7], codes)
    assert np.array_equal(forced[9], next_in)


def test_forcing_changes_what_is_fed_back():
    n = 2
    free = _run(n)
    force = free[7].copy()
    force[0, 3] = (force[0, 3] + 1) % CODE_ROWS          # a different code_3 in frame 0
    forced = _run(n, force=force)
    # codes up to code_3 are unchanged, the sum differs, argmaxes are still reported
    assert np.array_equal(forced[7][0, :4], free[7][0, :4])
    assert not np.array_equal(forced[9][0], free[9][0])


def test_frame_loop_rejects_bad_ids():
    tw, cw, code_tables, text, prompt = _setup(1)
    with pytest.raises(O.OracleError):
        O.frame_sum([tw["embed"]] + code_tables, [TALKER_S.embed_rows] + [0] * 15, text[0])

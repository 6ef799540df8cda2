"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: closed forms,
invariants, special cases that reduce to a textbook or library routine, and the
one worked figure the pages print for this path (the talker's bytes per token).
The set is chosen so that a plausible mistake (a dropped term, a wrong sign or
index, a transposed operand, a wrong group mapping, a wrong cache index) fails
at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- generator

def test_splitmix64_matches_published_vectors():
    g = _golden("splitmix64_seed1234567.json")
    out = W.raw_u64(g["state"], len(g["outputs"]))
    assert [int(v) for v in out] == [int(v) for v in g["outputs"]]


def test_generator_is_counter_based_and_normal():
    a = W.normal("x", (1000,), seed=3)
    b = W.normal("x", (2000,), seed=3)
    assert np.array_equal(a, b[:1000])             # prefix-stable: element i depends only on i
    assert not np.array_equal(a, W.normal("y", (1000,), seed=3))
    big = W.normal("z", (200000,), seed=0)
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1.0) < 0.01
    bits = W.normal("z", (10,), seed=0, bf16=True)
    import torch
    ref = torch.from_numpy(big[:10].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)                # RNE to bf16 equals torch's conversion


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_rms_and_scale_invariance():
    x = W.normal("rms", (256,), seed=1)
    g = np.ones(256, np.float32)
    y = O.rmsnorm(x, g, 0.0)
    assert abs(math.sqrt(float(np.mean(y.astype(np.float64) ** 2))) - 1.0) < 1e-6
    assert np.allclose(O.rmsnorm(7.5 * x, g, 0.0), y, rtol=1e-6, atol=1e-7)
    gam = W.normal("rmsg", (256,), seed=1, mean=1.0, std=0.1)
    assert np.allclose(O.rmsnorm(x, gam, 0.0), y * gam, rtol=1e-6, atol=1e-7)


def test_rmsnorm_eps_inside_the_root():
    # n = 1, x = 1, eps = 3: 1 / sqrt(1 + 3) = 0.5 exactly
    assert O.rmsnorm(np.array([1.0]), np.array([1.0]), 3.0)[0] == 0.5
    # constant vector c: output sign(c) * gamma when eps = 0
    y = O.rmsnorm(np.full(64, -3.0), np.full(64, 2.0), 0.0)
    assert np.all(y == -2.0)
    assert np.all(O.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0.0)


# ----------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    v = W.normal("rope0", (128,), seed=2)
    assert np.array_equal(O.rope(v, 0, 1e6), v)


def test_rope_two_dims_is_plane_rotation():
    # head_dim 2: one pair, frequency theta^0 = 1, so position p rotates by p radians
    for p in (1, 2, 7, 100):
        r = O.rope([1.0, 0.0], p, 1e6)
        assert abs(r[0] - math.cos(p)) < 1e-6 and abs(r[1] - math.sin(p)) < 1e-6


def test_rope_pairs_m_with_m_plus_half_at_frequency():
    # head_dim 4, theta 1e4: pair (1, 3) turns at 1e4^(-2/4) = 0.01 rad per position
    e1 = np.array([0.0, 1.0, 0.0, 0.0])
    r = O.rope(e1, 50, 1e4)
    assert abs(r[1] - math.cos(0.5)) < 1e-6 and abs(r[3] - math.sin(0.5)) < 1e-6
    assert r[0] == 0.0 and r[2] == 0.0


def test_rope_preserves_norm_and_relative_position():
    rng_q = W.normal("rq", (128,), seed=4)
    rng_k = W.normal("rk", (128,), seed=4)
    for p in (1, 17, 300, 1023):
        r = O.rope(rng_q, p, 1e6)
        assert abs(np.linalg.norm(r.astype(np.float64)) / np.linalg.norm(rng_q.astype(np.float64)) - 1) < 1e-6
    for (m, n, s) in ((3, 10, 5), (0, 40, 100), (200, 7, 333)):
        a = float(np.dot(O.rope(rng_q, m, 1e6).astype(np.float64), O.rope(rng_k, n, 1e6)))
        b = float(np.dot(O.rope(rng_q, m + s, 1e6).astype(np.float64), O.rope(rng_k, n + s, 1e6)))
        assert abs(a - b) < 1e-4 * (1 + abs(a))


# ----------------------------------------------------------------- attention

def test_attention_single_position_returns_value():
    q = W.normal("aq", (64,), seed=5)
    K = W.normal("aK", (1, 64), seed=5)
    V = W.normal("aV", (1, 64), seed=5)
    assert np.array_equal(O.attend(q, K, V), V[0])


def test_attention_equal_scores_average_values():
    V = W.normal("aV2", (5, 8), seed=6)
    K = np.zeros((5, 8), np.float32)
    out = O.attend(np.ones(8), K, V)
    assert np.allclose(out, V.astype(np.float64).mean(0), atol=1e-6)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # hd = 4: q . k1 - q . k2 = sqrt(4) * ln 3 makes the weights exactly 3/4 and 1/4
    hd = 4
    q = np.array([1.0, 0.0, 0.0, 0.0])
    K = np.array([[2 * math.log(3.0), 0, 0, 0], [0, 0, 0, 0]])
    V = np.array([[4.0, 0, 0, 0], [0, 8.0, 0, 0]])
    out = O.attend(q, K, V)
    assert np.allclose(out, [3.0, 2.0, 0, 0], atol=1e-6)
    assert hd == 4


def test_attention_brute_force_tiny_and_permutation():
    # hd 4, L 5: a brute-force softmax over hand-enumerated scores
    q = W.normal("bq", (4,), seed=7)
    K = W.normal("bK", (5, 4), seed=7)
    V = W.normal("bV", (5, 4), seed=7)
    s = [float(np.dot(q.astype(np.float64), K[j])) / 2.0 for j in range(5)]
    w = [math.exp(v) for v in s]
    ref = sum(w[j] * V[j].astype(np.float64) for j in range(5)) / sum(w)
    out = O.attend(q, K, V)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)
    perm = [3, 0, 4, 1, 2]
    assert np.allclose(O.attend(q, K[perm], V[perm]), out, rtol=1e-6, atol=1e-7)


# ----------------------------------------------------------------- SwiGLU

def test_silu_closed_forms():
    assert O.silu_mul(0.0, 5.0) == 0.0
    # sigmoid(ln 3) = 3/4
    assert abs(O.silu_mul(math.log(3.0), 2.0) - 2.0 * 0.75 * math.log(3.0)) < 1e-6
    assert abs(O.silu_mul(30.0, 1.0) - 30.0) < 1e-6
    assert abs(O.silu_mul(-30.0, 1.0)) < 1e-10


# ----------------------------------------------------------------- penalty / argmax

def test_penalty_hand_example():
    # logits [2, -2, 1], emitted {0, 1}, r = 2 -> [1, -4, 1]; tie goes to index 0
    idx, lg, margin = O.penalty_argmax([2.0, -2.0, 1.0], [0, 1], 2.0)
    assert list(lg) == [1.0, -4.0, 1.0] and idx == 0 and margin == 0.0


def test_penalty_one_is_identity_and_eos_mask():
    lg = W.normal("pl", (100,), seed=8)
    idx, out, _ = O.penalty_argmax(lg, range(100), 1.0)
    assert np.array_equal(out, lg) and idx == int(np.argmax(lg))
    top = int(np.argmax(lg))
    idx2, out2, _ = O.penalty_argmax(lg, [], 1.0, eos_id=top)
    assert out2[top] == -np.inf and idx2 == int(np.argsort(-lg.astype(np.float64), kind="stable")[1])


def test_argmax_lowest_index_on_ties():
    assert O.penalty_argmax([0.0, 5.0, 1.0, 5.0, 5.0], [], 1.0)[0] == 1


# ----------------------------------------------------------------- bf16 storage

def test_bf16_round_to_nearest_even():
    import torch
    vals = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 3.14159, 1e-30, 65504.0, -0.0]
    for v in vals:
        ref = int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
        assert O.round_bf16(v) == ref, v
    assert O.round_bf16(1.0 + 2 ** -8) == 0x3F80          # tie -> even (1.0)
    assert O.round_bf16(1.0 + 3 * 2 ** -8) == 0x3F82      # tie -> even (1 + 2^-6)


# ----------------------------------------------------------------- model-level

def _tiny(**kw):
    return W.scaled(W.TINY, **kw)


def _run(shape, weights, embeds, steps, buckets=None, acc64=False, taps=False):
    o = O.Oracle(shape, weights, acc64=acc64, buckets=buckets)
    fid, lg, _ = o.prefill(embeds=embeds)
    ids, logits, tp = [fid], [lg], []
    for _ in range(steps):
        oid, lg, _, t = o.step(token=ids[-1], taps=taps)
        ids.append(oid)
        logits.append(lg)
        tp.append(t)
    return o, ids, logits, tp


def test_cached_decode_equals_full_recompute():
    s = W.TINY
    w = W.model_weights(s)
    e = W.prefill_embeds(s, 12)
    o = O.Oracle(s, w)
    for n in (1, 2, 5, 12):
        o.reset()
        _, lg, _ = o.prefill(embeds=e[:n])
        ref = O.recompute_logits(s, w, embeds=e[:n])
        assert np.array_equal(lg, ref), n
    # bf16 cache path too (rounding at the same point on both routes)
    sb = W.scaled(W.TINY, bf16=True, name="tiny_bf16")
    wb = W.model_weights(sb)
    ob = O.Oracle(sb, wb)
    _, lgb, _ = ob.prefill(embeds=e[:9])
    assert np.array_equal(lgb, O.recompute_logits(sb, wb, embeds=e[:9]))


def test_gqa_equals_mha_with_duplicated_kv_heads():
    s = W.TINY                      # 4 q heads, 2 kv heads
    w = W.model_weights(s)
    m = W.scaled(s, n_kv_heads=4, name="tiny_mha")
    wm = dict(w)
    hd = s.head_dim
    for l in range(s.n_layers):
        for key in ("wk", "wv"):
            a = w[f"layers.{l}.{key}"].reshape(s.n_kv_heads, hd, s.hidden)
            wm[f"layers.{l}.{key}"] = np.ascontiguousarray(np.repeat(a, 2, axis=0).reshape(4 * hd, s.hidden))
    e = W.prefill_embeds(s, 10)
    _, ids_g, lg_g, _ = _run(s, w, e, 4)
    _, ids_m, lg_m, _ = _run(m, wm, e, 4)
    assert ids_g == ids_m
    for a, b in zip(lg_g, lg_m):
        assert np.array_equal(a, b)
    # the other mapping (q head i -> kv head i % kvh) is a different model
    wx = dict(w)
    for l in range(s.n_layers):
        for key in ("wk", "wv"):
            a = w[f"layers.{l}.{key}"].reshape(s.n_kv_heads, hd, s.hidden)
            wx[f"layers.{l}.{key}"] = np.ascontiguousarray(np.tile(a, (2, 1, 1)).reshape(4 * hd, s.hidden))
    _, _, lg_x, _ = _run(m, wx, e, 0)
    assert not np.array_equal(lg_x[0], lg_g[0])


def test_bucket_migration_is_bit_identical():
    s = W.scaled(W.TINY, buckets=(32, 64, 128))
    w = W.model_weights(W.TINY)
    e = W.prefill_embeds(W.TINY, 20)
    o1, ids1, lg1, _ = _run(s, w, e, 60)                       # crosses 32 and 64
    o2, ids2, lg2, _ = _run(s, w, e, 60, buckets=(128,))
    assert o1.smax == 128 and o1.pos == 80
    assert ids1 == ids2
    for a, b in zip(lg1, lg2):
        assert np.array_equal(a, b)
    for l in range(s.n_layers):
        for which in (0, 1):
            assert np.array_equal(o1.kv(l, which), o2.kv(l, which))


def test_kv_full_after_last_bucket():
    s = W.scaled(W.TINY, buckets=(32,))
    w = W.model_weights(W.TINY)
    o = O.Oracle(s, w)
    o.prefill(embeds=W.prefill_embeds(W.TINY, 32))
    with pytest.raises(O.OracleError) as ei:
        o.step(token=3)
    assert ei.value.status == O.EKVFULL and o.pos == 32


def test_greedy_determinism_and_acc64_agreement():
    s = W.TINY
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    _, ids1, lg1, _ = _run(s, w, e, 8)
    _, ids2, lg2, _ = _run(s, w, e, 8)
    assert ids1 == ids2 and all(np.array_equal(a, b) for a, b in zip(lg1, lg2))
    _, ids3, lg3, _ = _run(s, w, e, 8, acc64=True)
    for a, b in zip(lg1, lg3):
        assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(b)


def test_zero_residual_branches_pass_input_through():
    s = W.scaled(W.TINY, n_layers=2, name="tiny2")
    w = W.model_weights(s)
    for l in range(2):
        w[f"layers.{l}.wo"] = np.zeros_like(w[f"layers.{l}.wo"])
        w[f"layers.{l}.wd"] = np.zeros_like(w[f"layers.{l}.wd"])
    e = W.prefill_embeds(s, 3)
    o = O.Oracle(s, w)
    o.prefill(embeds=e[:2], want_logits=False)
    _, lg, _, taps = o.step(embed=e[2], taps=True)
    for l in range(1, 3):
        assert np.array_equal(taps[l], e[2])
    y = O.rmsnorm(e[2], w["final_norm"], s.rms_eps)
    assert np.allclose(lg, w["lm_head.0"].astype(np.float64) @ y.astype(np.float64), rtol=1e-5, atol=1e-6)
    assert np.allclose(o.hidden(), y)


def test_zero_query_attends_uniformly_over_the_prefix():
    # wq = 0 -> every score is 0 -> the attention output is the mean of v over
    # positions 0..p; with wd = 0 the layer output is x + Wo . mean(v).
    s = W.scaled(W.TINY, qk_norm=False, name="tiny_noqk")
    w = W.model_weights(s)
    w["layers.0.wq"] = np.zeros_like(w["layers.0.wq"])
    w["layers.0.wd"] = np.zeros_like(w["layers.0.wd"])
    e = W.prefill_embeds(s, 6)
    o = O.Oracle(s, w)
    o.prefill(embeds=e[:5], want_logits=False)
    _, _, _, taps = o.step(embed=e[5], taps=True)
    V = []
    for t in range(6):
        xn = O.rmsnorm(e[t], w["layers.0.attn_norm"], s.rms_eps).astype(np.float64)
        V.append(w["layers.0.wv"].astype(np.float64) @ xn)
    vbar = np.mean(V, axis=0)                                   # [kvh * hd]
    hd, grp = s.head_dim, s.n_q_heads // s.n_kv_heads
    att = np.concatenate([vbar[(i // grp) * hd:(i // grp + 1) * hd] for i in range(s.n_q_heads)])
    ref = e[5].astype(np.float64) + w["layers.0.wo"].astype(np.float64) @ att
    assert np.allclose(taps[1], ref, rtol=1e-4, atol=1e-5)
    # and the cache holds exactly the rotated-free v rows of every position
    kvv = o.kv(0, 1)
    assert np.allclose(kvv.transpose(1, 0, 2).reshape(6, -1), np.array(V), rtol=1e-5, atol=1e-6)


def test_mlp_branch_is_down_of_silu_gate_times_up():
    # wq = 0 makes the attention branch x + Wo . mean(v) (pinned above); the layer's
    # output must then add Wd (silu(Wg x^) * (Wu x^)) with x^ = RMSNorm(x1; mlp gamma):
    # the gate, not the up projection, goes through silu, and Wd multiplies the
    # product.  Evaluated here in float64 from the definition.
    s = W.scaled(W.TINY, qk_norm=False, name="tiny_noqk")
    w = W.model_weights(s)
    w["layers.0.wq"] = np.zeros_like(w["layers.0.wq"])
    e = W.prefill_embeds(s, 6)
    o = O.Oracle(s, w)
    o.prefill(embeds=e[:5], want_logits=False)
    _, _, _, taps = o.step(embed=e[5], taps=True)
    f64 = lambda k: w[k].astype(np.float64)
    V = [f64("layers.0.wv") @ O.rmsnorm(e[t], w["layers.0.attn_norm"], s.rms_eps).astype(np.float64)
         for t in range(6)]
    vbar = np.mean(V, axis=0)
    hd, grp = s.head_dim, s.n_q_heads // s.n_kv_heads
    att = np.concatenate([vbar[(i // grp) * hd:(i // grp + 1) * hd] for i in range(s.n_q_heads)])
    x1 = e[5].astype(np.float64) + f64("layers.0.wo") @ att
    xn = x1 / np.sqrt(np.mean(x1 * x1) + s.rms_eps) * f64("layers.0.mlp_norm")
    g, u = f64("layers.0.wg") @ xn, f64("layers.0.wu") @ xn
    ref = x1 + f64("layers.0.wd") @ (g / (1.0 + np.exp(-g)) * u)
    assert np.allclose(taps[1], ref, rtol=1e-4, atol=1e-5)
    # the branch is not negligible here: dropping it or swapping gate and up is visible
    swapped = x1 + f64("layers.0.wd") @ (u / (1.0 + np.exp(-u)) * g)
    assert not np.allclose(taps[1], swapped, rtol=1e-4, atol=1e-5)
    assert not np.allclose(taps[1], x1, rtol=1e-4, atol=1e-5)


def test_emitted_set_follows_fed_tokens_not_prompt():
    s = W.TINY
    w = W.model_weights(s)
    o = O.Oracle(s, w)
    o.prefill(tokens=np.array([5, 6, 7], np.int32))
    assert not o.emitted().any()                     # prompt tokens do not join the set
    for t in (9, 40, 9, 1023):
        o.step(token=t)
    em = o.emitted()
    got = [i for i in range(s.vocab) if (em[i >> 5] >> (i & 31)) & 1]
    assert got == [9, 40, 1023]


def test_repetition_penalty_changes_the_trajectory_only_through_emitted_ids():
    s = W.TINY
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    o = O.Oracle(s, w)
    fid, _, _ = o.prefill(embeds=e)
    oid, raw, _, _ = o.step(token=fid)
    idx, pen, _ = O.penalty_argmax(raw, [fid], s.rep_penalty)
    assert oid == idx                                  # model applies exactly the pinned rule


def test_talker_shape_reproduces_page_bytes_per_token():
    g = _golden("talker_weight_bytes.json")
    s = W.TALKER
    assert s.n_layers * 7 == g["matmuls_per_token"]
    mb = s.matrix_params() * g["q8_0_bytes_per_32_weights"] / 32 / 1e6
    assert abs(mb - g["mb_per_token"]) <= g["mb_tolerance"]


def test_invalid_configs_and_inputs_are_rejected():
    s = W.TINY
    w = W.model_weights(s)
    with pytest.raises(O.OracleError):
        O.Oracle(W.scaled(s, n_q_heads=3), w)
    with pytest.raises(O.OracleError):
        O.Oracle(s, w, buckets=(128, 64))
    o = O.Oracle(s, w)
    with pytest.raises(O.OracleError):
        o.prefill(embeds=np.zeros((0, s.hidden), np.float32))
    with pytest.raises(O.OracleError):
        o.step(token=s.embed_rows)
    o.prefill(embeds=W.prefill_embeds(s, 4))
    with pytest.raises(O.OracleError):
        o.prefill(embeds=W.prefill_embeds(s, 4))        # prefill needs an empty cache
    assert o.pos == 4

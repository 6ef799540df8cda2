"""Parity of the CUDA decode path (through the C-ABI) with the CPU oracle.

Shapes: the five decode workloads and reduced versions of them that the oracle
finishes in seconds while still spanning several GEMV stages per CTA, several
attention splits, ragged tails (KV lengths that are not multiples of the split
size) and every bucket migration of the ladder.
"""
import numpy as np
import pytest

import workloads as W
from _pair import MARGIN, REL_TOL, Pair, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


def _tf(shape, n_steps, buckets=None, taps=True, graphs=True, prefill=None, seed=None):
    w = W.model_weights(shape, seed=seed)
    e = W.prefill_embeds(shape, prefill)
    p = Pair(shape, w, buckets=buckets, taps=taps, graphs=graphs)
    tr = p.run_teacher_forced(e, n_steps)
    return p, tr


# ------------------------------------------------------------------ workloads


def test_tiny_fp32_full_workload():
    s = W.TINY
    p, tr = _tf(s, s.decode_steps)
    tr.check()
    assert max(tr.logits_rel) < 1e-4          # fp32 weights and cache: only summation order differs
    assert tr.ids_gpu == tr.ids_ref           # every margin of this workload is above the bar
    p.close()


def test_asr_two_layers_crosses_both_migrations():
    s = W.scaled(W.ASR, n_layers=2, name="asr2")
    p, tr = _tf(s, 200)                        # prefill 110 -> KV length 310: 128 -> 256 -> 512
    tr.check()
    pos, smax = p.qd.qd_get_pos(p.h)
    assert pos == 310 and smax == 512
    assert all(i != s.eos_mask_id for i in tr.ids_gpu)
    p.close()


def test_talker_four_layers_gqa_qknorm_penalty():
    s = W.scaled(W.TALKER, n_layers=4, name="talker4")
    p, tr = _tf(s, 100)                        # 64 -> 165 positions: crosses 128
    tr.check()
    p.close()


def test_asr_full_size_graph_path():
    """The ASR workload at full size in the launch configuration the benchmark
    times (CUDA graphs, no taps): prefill 110, greedy to KV length 400."""
    s = W.ASR
    p, tr = _tf(s, s.decode_steps, taps=False)
    tr.check()
    pos, smax = p.qd.qd_get_pos(p.h)
    assert pos == 400 and smax == 512
    p.close()


def test_asr_full_size_logits_and_layers():
    s = W.ASR
    p, tr = _tf(s, 40, taps=True)
    tr.check()
    p.close()


@pytest.mark.slow
def test_talker_full_size_every_layer_every_step():
    """The full Talker workload (28 layers, prefill 64, 600 teacher-forced steps across
    the buckets 128 -> 256 -> 512 -> 1024) with the debug taps on: every step's logits
    and the hidden state after every layer against the oracle's, relative L2 <= 2e-3,
    and every id above the margin equal."""
    s = W.TALKER
    p, tr = _tf(s, s.decode_steps, taps=True)
    tr.check()
    assert len(tr.logits_rel) == s.decode_steps + 1 and len(tr.hidden_rel) == s.decode_steps
    assert len(tr.ids_ref) - len(tr.low_margin) > s.decode_steps // 2     # the id comparison is not vacuous
    pos, smax = p.qd.qd_get_pos(p.h)
    assert pos == 664 and smax == 1024
    p.close()


@pytest.mark.slow
def test_talker_full_size_graph_path():
    s = W.TALKER
    p, tr = _tf(s, s.decode_steps, taps=False)
    tr.check()
    pos, smax = p.qd.qd_get_pos(p.h)
    assert pos == 664 and smax == 1024
    p.close()


def test_code_predictor_heads_and_embedding_inputs():
    s = W.CODE_PREDICTOR
    w = W.model_weights(s)
    p = Pair(s, w)
    e = W.prefill_embeds(s, 2)
    steps = W.normal("cp/step_embeds", (14, s.hidden), 0, 0.0, 1.0)
    rid = p.prefill(embeds=e, head_idx=0)
    for j in range(1, 15):
        rid = p.step(token=rid, embed=steps[j - 1], head_idx=j)
    p.trace.check()
    pos, smax = p.qd.qd_get_pos(p.h)
    assert pos == 16 and smax == 32
    p.close()


# ------------------------------------------------------------------ invariants on the GPU


def _ids_logits(shape, w, e, n, buckets=None, graphs=True, grow_at=None):
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    h = qd.qd_create(upload(w), config_from_shape(shape, buckets))
    qd.qd_set_graphs(h, graphs)
    y = torch.empty(shape.hidden, dtype=torch.float32, device="cuda")
    ids = [qd.qd_prefill(h, embeds=torch.from_numpy(e).cuda())]
    hid = []
    for i in range(n):
        if grow_at is not None and i == grow_at[0]:
            qd.qd_grow_kv(h, grow_at[1])
        ids.append(qd.qd_decode_step(h, token=ids[-1]))
        qd.qd_get_hidden(h, y)
        hid.append(y.cpu().numpy().copy())
    n_bytes = qd.qd_copy_kv(h)
    kv = torch.empty(n_bytes, dtype=torch.uint8, device="cuda")
    qd.qd_copy_kv(h, kv)
    pos, smax = qd.qd_get_pos(h)
    qd.qd_destroy(h)
    return ids, np.array(hid), kv.cpu().numpy(), pos, smax


def _bf16_to_f32(b):
    u = np.ascontiguousarray(b).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def _valid_kv(kv_bytes, shape, smax, pos):
    es = 2 if shape.bf16 else 4
    a = kv_bytes.reshape(shape.n_layers, 2, shape.n_kv_heads, smax, shape.head_dim * es)
    return a[:, :, :, :pos, :]


def test_bucket_migration_is_bit_identical_on_gpu():
    s = W.scaled(W.ASR, n_layers=2, name="asr2")
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    a = _ids_logits(s, w, e, 180)                       # 128 -> 256 -> 512
    b = _ids_logits(s, w, e, 180, buckets=(512,))       # starts at 512
    assert a[0] == b[0]
    assert np.array_equal(a[1], b[1])
    assert a[3] == b[3] == 290
    assert np.array_equal(_valid_kv(a[2], s, a[4], a[3]), _valid_kv(b[2], s, b[4], b[3]))


def test_explicit_grow_is_bit_identical():
    s = W.scaled(W.TALKER, n_layers=2, name="talker2")
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    a = _ids_logits(s, w, e, 30)
    b = _ids_logits(s, w, e, 30, grow_at=(10, 1024))     # jump 128 -> 1024 mid-stream
    assert a[0] == b[0] and np.array_equal(a[1], b[1])
    assert b[4] == 1024
    assert np.array_equal(_valid_kv(a[2], s, a[4], a[3]), _valid_kv(b[2], s, b[4], b[3]))


def test_graph_replay_equals_eager_and_is_deterministic():
    s = W.scaled(W.TALKER, n_layers=3, name="talker3")
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    g1 = _ids_logits(s, w, e, 70)
    g2 = _ids_logits(s, w, e, 70)
    ea = _ids_logits(s, w, e, 70, graphs=False)
    assert g1[0] == g2[0] == ea[0]
    assert np.array_equal(g1[1], g2[1]) and np.array_equal(g1[1], ea[1])
    assert np.array_equal(g1[2], g2[2])


def test_kv_cache_and_emitted_set_match_oracle():
    s = W.scaled(W.TALKER, n_layers=2, name="talker2")
    w = W.model_weights(s)
    e = W.prefill_embeds(s, 40)
    p = Pair(s, w)
    p.run_teacher_forced(e, 100)                        # crosses 128
    kv, pos = p.kv()
    assert pos == p.ref.pos == 140
    for l in range(s.n_layers):
        for which in (0, 1):
            ref = p.ref.kv(l, which)                    # [kvh, pos, hd]
            got = kv[l, which, :, :pos, :]
            assert rel_l2(got, ref) <= REL_TOL
    import torch
    em = torch.empty((s.vocab + 31) // 32, dtype=torch.int32, device="cuda")
    p.qd.qd_get_emitted(p.h, em)
    assert np.array_equal(em.cpu().numpy().view(np.uint32), p.ref.emitted())   # integer work: bit-exact
    p.close()


def test_prefill_from_tokens():
    s = W.scaled(W.ASR, n_layers=2, name="asr2")
    w = W.model_weights(s)
    toks = W.uniform_int("asr2/prompt", 77, 0, s.vocab - 1)
    p = Pair(s, w)
    rid = p.prefill(tokens=toks)
    for _ in range(20):
        rid = p.step(token=rid)
    p.trace.check()
    p.close()


def test_device_greedy_loop_matches_stepwise():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    s = W.scaled(W.ASR, n_layers=2, name="asr2")
    w = W.model_weights(s)
    e = torch.from_numpy(W.prefill_embeds(s)).cuda()
    h = qd.qd_create(upload(w), config_from_shape(s))
    first = qd.qd_prefill(h, embeds=e)
    ids = torch.empty(150, dtype=torch.int32, device="cuda")
    qd.qd_decode_greedy(h, 150, first, ids)
    torch.cuda.synchronize()
    greedy = ids.cpu().tolist()
    qd.qd_reset(h)
    assert qd.qd_prefill(h, embeds=e) == first
    step = []
    tok = first
    for _ in range(150):
        tok = qd.qd_decode_step(h, token=tok)
        step.append(tok)
    assert greedy == step
    # async variant with device-resident token / id
    qd.qd_reset(h)
    qd.qd_prefill(h, embeds=e)
    t_dev = torch.tensor([first], dtype=torch.int32, device="cuda")
    for i in range(10):
        qd.qd_decode_step_async(h, None, t_dev, 0, t_dev)
    torch.cuda.synchronize()
    assert int(t_dev.item()) == step[9]
    qd.qd_destroy(h)


def test_errors_leave_the_handle_usable():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    s = W.scaled(W.TINY, buckets=(32, 64))
    w = W.model_weights(W.TINY)
    h = qd.qd_create(upload(w), config_from_shape(s))
    with pytest.raises(qd.QDError) as ei:
        qd.qd_decode_step(h, token=1)
    assert ei.value.status == qd.QD_ESTATE
    e = torch.from_numpy(W.prefill_embeds(W.TINY, 40)).cuda()
    with pytest.raises(qd.QDError) as ei:
        qd.qd_prefill(h, embeds=e[:0])
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_prefill(h, embeds=torch.zeros((65, s.hidden), device="cuda"))
    assert ei.value.status == qd.QD_EKVFULL
    first = qd.qd_prefill(h, embeds=e)                  # 40 positions -> bucket 64
    assert qd.qd_get_pos(h) == (40, 64)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_prefill(h, embeds=e)
    assert ei.value.status == qd.QD_ESTATE
    with pytest.raises(qd.QDError) as ei:
        qd.qd_decode_step(h, token=s.embed_rows)
    assert ei.value.status == qd.QD_EINVAL
    with pytest.raises(qd.QDError) as ei:
        qd.qd_grow_kv(h, 48)
    assert ei.value.status == qd.QD_EINVAL
    tok = first
    for _ in range(24):
        tok = qd.qd_decode_step(h, token=tok)
    assert qd.qd_get_pos(h) == (64, 64)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_decode_step(h, token=tok)
    assert ei.value.status == qd.QD_EKVFULL
    assert qd.qd_get_pos(h) == (64, 64)
    qd.qd_reset(h)
    assert qd.qd_prefill(h, embeds=e) == first          # usable after every error
    qd.qd_destroy(h)


def test_time_kernel_leaves_state_unchanged():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    s = W.scaled(W.TALKER, n_layers=2, name="talker2")
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    ref = _ids_logits(s, w, e, 12)
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    h = qd.qd_create(upload(w), config_from_shape(s))
    ids = [qd.qd_prefill(h, embeds=torch.from_numpy(e).cuda())]
    for i in range(12):
        if i == 5:
            for which in range(6):
                assert qd.qd_time_kernel(h, which, 3) > 0
        ids.append(qd.qd_decode_step(h, token=ids[-1]))
    assert ids == ref[0]
    qd.qd_destroy(h)


@pytest.mark.parametrize("shape_name", ["tiny", "asr2", "talker2"])
def test_persistent_step_equals_per_phase_kernels(shape_name, monkeypatch):
    """The persistent decode step and the per-phase kernels compute the same step with
    sums in different orders: the persistent step splits each GEMV's K over its warps,
    applies the RMSNorm scale after the dot products and, on bf16 weights, takes the
    dot products on the tensor cores with the fp32 input as two bf16 parts (16
    significant bits, fp32 accumulation in the tensor cores' order).  Equal ids, hidden
    states within 5e-4 relative L2 (a few ulp of bf16 input splitting and summation
    order, compounded over the layers and steps), caches equal up to the bf16 rounding
    flips those differences cause."""
    s = {"tiny": W.TINY, "asr2": W.scaled(W.ASR, n_layers=2, name="asr2"),
         "talker2": W.scaled(W.TALKER, n_layers=2, name="talker2")}[shape_name]
    w = W.model_weights(s)
    e = W.prefill_embeds(s, 40)
    n = 30 if shape_name != "tiny" else 8
    a = _ids_logits(s, w, e, n)
    monkeypatch.setenv("QD_PER_PHASE", "1")
    b = _ids_logits(s, w, e, n)
    assert a[0] == b[0]
    worst = max(rel_l2(ya, yb) for ya, yb in zip(a[1], b[1]))
    print(f"{shape_name}: hidden rel_l2 max {worst:.3g}")
    assert worst <= 5e-4, worst
    ka = _valid_kv(a[2], s, a[4], a[3])
    kb = _valid_kv(b[2], s, b[4], b[3])
    if s.bf16:
        ka, kb = _bf16_to_f32(ka), _bf16_to_f32(kb)
    else:
        ka, kb = ka.view(np.float32), kb.view(np.float32)
    kv = rel_l2(ka, kb)
    print(f"{shape_name}: kv rel_l2 {kv:.3g}")
    assert kv <= 1e-3, kv


@pytest.mark.parametrize("shape_name,prompt", [("asr2", "embeds"), ("talker2", "embeds"), ("asr2", "tokens")])
def test_prompt_prefill_through_batched_kernels_matches_oracle(shape_name, prompt):
    """qd_prefill from embeddings on a bf16 model runs every prompt position at once
    (tensor-core GEMMs, causal flash attention, then the cache rows are copied into the
    bucket): its cache, final-norm hidden state and first id against the oracle's
    position-by-position prefill, and the state it leaves (position, first id) for the
    decode steps after it; decoding on from it then tracks the oracle."""
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    s = {"asr2": W.scaled(W.ASR, n_layers=2, name="asr2"),
         "talker2": W.scaled(W.TALKER, n_layers=2, name="talker2")}[shape_name]
    w = W.model_weights(s)
    e = W.prefill_embeds(s)
    n = len(e)
    toks = W.uniform_int(f"{shape_name}/prompt_tokens", n, 0, s.embed_rows - 1).astype(np.int32)
    h = qd.qd_create(upload(w), config_from_shape(s))
    if prompt == "embeds":
        first = qd.qd_prefill(h, embeds=torch.from_numpy(e).cuda())
    else:
        first = qd.qd_prefill(h, tokens=toks)
    y = torch.empty(s.hidden, dtype=torch.float32, device="cuda")
    qd.qd_get_hidden(h, y)
    pos, smax = qd.qd_get_pos(h)
    assert pos == n
    nb = qd.qd_copy_kv(h)
    kv = torch.empty(nb, dtype=torch.uint8, device="cuda")
    qd.qd_copy_kv(h, kv)
    g = kv.cpu().numpy().view(np.uint16).reshape(s.n_layers, 2, s.n_kv_heads, smax, s.head_dim)
    o = O.Oracle(s, w)
    rid, rlog, margin = o.prefill(embeds=e) if prompt == "embeds" else o.prefill(tokens=toks)
    assert margin <= MARGIN or first == rid, (first, rid, margin)
    assert rel_l2(y.cpu().numpy(), o.hidden()) <= REL_TOL
    for l in range(s.n_layers):
        for which in range(2):
            got = (g[l, which, :, :n].astype(np.uint32) << 16).view(np.float32)
            assert rel_l2(got, o.kv(l, which)) <= REL_TOL, (l, which)
    # decode on, teacher-forced with the oracle's ids
    fed = rid
    for i in range(6):
        gid = qd.qd_decode_step(h, token=fed)
        oid, _, om, _ = o.step(token=fed)
        assert om <= MARGIN or gid == oid, (i, gid, oid, om)
        fed = oid
    assert qd.qd_get_pos(h)[0] == n + 6
    o.close()
    qd.qd_destroy(h)

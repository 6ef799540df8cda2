"""Parity of the batched multi-stream decode (tensor-core GEMMs, per-stream attention)
with the oracle, one oracle stream per GPU stream.

Each stream starts from its own seeded cache of its own length and a seeded input
token; the GPU is fed the oracle's ids (teacher forcing), so every step of every
checked stream is comparable.  Bars: raw logits relative L2 <= 2e-3 per stream and
step, equal ids wherever the oracle's top-2 margin exceeds 1e-2, the copied cache
region bit-exact and the appended rows within the same tolerance.
"""
import numpy as np
import pytest

import workloads as W
from _pair import MARGIN, REL_TOL, rel_l2

pytestmark = pytest.mark.gpu

TALKER2 = W.scaled(W.TALKER, n_layers=2, name="talker2")


@pytest.fixture(scope="module", autouse=True)
def _cuda(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    yield


class BatchPair:
    def __init__(self, shape, B, smax, lens, oracle_streams=None, seed=0):
        import torch
        import oracle as O
        import transformer_autoregressive_decode_gb300 as qd
        from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, to_device, upload

        self.qd, self.torch, self.shape, self.B, self.smax = qd, torch, shape, B, smax
        self.lens = [int(v) for v in lens]
        self.w = W.model_weights(shape, seed=seed)
        self.h = qd.qd_create(upload(self.w), config_from_shape(shape))
        self.bh = qd.qd_batch_create(self.h, B, smax)
        self.tokens = W.batch_first_tokens(B, shape.vocab, seed=seed)
        self.oracle_streams = list(range(B)) if oracle_streams is None else list(oracle_streams)
        self.kv0 = {}
        self.ref = {}
        for b in range(B):
            kv = W.batch_stream_kv(shape, b, self.lens[b], seed=seed)
            qd.qd_batch_set_stream(self.bh, b, to_device(kv), self.lens[b], int(self.tokens[b]))
            if b in self.oracle_streams:
                self.kv0[b] = kv
                o = O.Oracle(shape, self.w, buckets=(smax,))
                o.set_kv(kv, self.lens[b])
                self.ref[b] = o
        self.logits = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
        self.fed = {b: int(self.tokens[b]) for b in self.oracle_streams}

    def step(self):
        """One teacher-forced step; returns per checked stream (gpu id, oracle id,
        margin, logits rel L2)."""
        torch = self.torch
        out = {}
        force = np.zeros((1, self.B), np.int32)
        for b, o in self.ref.items():
            rid, rlog, margin, _ = o.step(token=self.fed[b])
            out[b] = [None, rid, margin, rlog]
            force[0, b] = rid
        ids = torch.empty((1, self.B), dtype=torch.int32, device="cuda")
        self.qd.qd_batch_decode(self.bh, 1, ids, torch.from_numpy(force).cuda())
        self.qd.qd_batch_sync(self.bh)
        self.qd.qd_batch_get_logits(self.bh, self.logits)
        g_ids = ids.cpu().numpy()[0]
        g_log = self.logits.cpu().numpy()
        for b in self.ref:
            out[b][0] = int(g_ids[b])
            out[b][3] = rel_l2(g_log[b], out[b][3])
            self.fed[b] = out[b][1]
        return out

    def gpu_cache(self, b):
        torch = self.torch
        n = self.qd.qd_batch_copy_kv(self.bh, b)
        buf = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.qd.qd_batch_copy_kv(self.bh, b, buf)
        s = self.shape
        return buf.view(torch.int16).cpu().numpy().view(np.uint16).reshape(
            s.n_layers, 2, s.n_kv_heads, self.smax, s.head_dim)

    def close(self):
        self.qd.qd_batch_destroy(self.bh)
        self.qd.qd_destroy(self.h)
        for o in self.ref.values():
            o.close()


def _check_steps(bp, n_steps):
    worst = 0.0
    checked = 0
    for i in range(n_steps):
        for b, (gid, rid, margin, lrel) in bp.step().items():
            worst = max(worst, lrel)
            if margin > MARGIN:
                checked += 1
                assert gid == rid, (i, b, gid, rid, margin)
    assert worst <= REL_TOL, worst
    return checked


def _bf16_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def test_batch_reduced_all_streams_match_oracle():
    B, smax, n = 8, 512, 12
    lens = W.batch_initial_lengths(n=B, lo=100, hi=400)
    bp = BatchPair(TALKER2, B, smax, lens)
    checked = _check_steps(bp, n)
    assert checked > B * n // 2
    s = bp.shape
    for b in range(B):
        assert bp.qd.qd_batch_get_pos(bp.bh, b) == bp.lens[b] + n
        g = bp.gpu_cache(b)
        L0 = bp.lens[b]
        assert np.array_equal(g[:, :, :, :L0], bp.kv0[b])            # copied region untouched
        for l in range(s.n_layers):
            for w in range(2):
                ref = bp.ref[b].kv(l, w)[:, L0:L0 + n]                 # appended rows
                got = _bf16_to_f32(g[l, w, :, L0:L0 + n])
                assert rel_l2(got, ref) <= REL_TOL
    bp.close()


def test_batch_multi_step_call_equals_single_steps_and_graphs_equal_eager():
    import torch
    B, smax, n = 4, 256, 6
    lens = W.batch_initial_lengths(n=B, lo=40, hi=200)
    force = W.uniform_int("batched/test_force", n * B, 0, TALKER2.vocab - 1).reshape(n, B)
    outs = []
    for mode in ("one_call", "per_step", "eager"):
        bp = BatchPair(TALKER2, B, smax, lens, oracle_streams=[])
        if mode == "eager":
            bp.qd.qd_batch_set_graphs(bp.bh, False)
        ids = torch.empty((n, B), dtype=torch.int32, device="cuda")
        f = torch.from_numpy(np.ascontiguousarray(force)).cuda()
        if mode == "per_step":
            for i in range(n):
                bp.qd.qd_batch_decode(bp.bh, 1, ids[i:i + 1], f[i:i + 1])
        else:
            bp.qd.qd_batch_decode(bp.bh, n, ids, f)
        bp.qd.qd_batch_sync(bp.bh)
        bp.qd.qd_batch_get_logits(bp.bh, bp.logits)
        outs.append((ids.cpu().numpy(), bp.logits.cpu().numpy(), bp.gpu_cache(B - 1)))
        bp.close()
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("k,t", [(50, 0.9), (8, 0.7)])
def test_batch_sampled_streams_match_oracle(k, t):
    """Sampling in the batched decode (the pages' generation defaults top-k 50,
    temperature 0.9, top-p 1.0; and 8 candidates at 0.7, where more draws are decidable
    on this 2-layer shape): stream b draws from seed + b at its own counter, as the
    oracle stream does with set_sampling(seed + b), teacher-forced with the oracle's
    draws.  The sampler exactly: every GPU id equals the oracle's sampler applied to the
    GPU's own final logits (the oracle's penalty and EOS mask over the same emitted set,
    the same u).  Against the oracle's whole step: the logits within 2e-3, and every id
    whose draw the oracle's margin decides (beyond ten times a 2e-3 logit error over the
    temperature) equal."""
    import torch
    import oracle as O
    B, smax, n = 6, 512, 10
    p, seed = 1.0, 77
    lens = W.batch_initial_lengths(n=B, lo=100, hi=400)
    bp = BatchPair(TALKER2, B, smax, lens)
    bp.qd.qd_batch_set_sampling(bp.bh, k, t, p, seed)
    for b, o in bp.ref.items():
        o.set_sampling(k, t, p, seed + b)
    s = bp.shape
    decided = 0
    for i in range(n):
        out = bp.step()
        g_log = bp.logits.cpu().numpy()
        for b, (gid, rid, margin, lrel) in out.items():
            assert lrel <= REL_TOL
            em = bp.ref[b].emitted()
            ids_em = [v for v in range(s.vocab) if (em[v >> 5] >> (v & 31)) & 1]
            _, final, _ = O.penalty_argmax(g_log[b], ids_em, s.rep_penalty, s.eos_mask_id)
            want, m_own = O.sample(final, k, t, p, O.uniform(seed + b, i))
            assert gid == want or m_own < 1e-6, (i, b, gid, want, m_own)
            if margin > 10 * 2e-3 / t:
                decided += 1
                assert gid == rid, (i, b, gid, rid, margin)
    if k == 8:
        assert decided >= B * n // 10, decided
    bp.close()
    # the draws are not the argmaxes, and top_k 0 is greedy again
    ids_g = torch.empty((n, B), dtype=torch.int32, device="cuda")
    g = BatchPair(TALKER2, B, smax, lens, oracle_streams=[])
    g.qd.qd_batch_decode(g.bh, n, ids_g)
    g.close()
    ids_s = torch.empty((n, B), dtype=torch.int32, device="cuda")
    sp = BatchPair(TALKER2, B, smax, lens, oracle_streams=[])
    sp.qd.qd_batch_set_sampling(sp.bh, k, t, p, seed)
    sp.qd.qd_batch_decode(sp.bh, n, ids_s)
    assert (ids_s.cpu().numpy() != ids_g.cpu().numpy()).any()
    sp.qd.qd_batch_set_sampling(sp.bh, 0, 1.0, 1.0, 0)
    for b in range(B):
        sp.qd.qd_batch_set_stream(sp.bh, b, torch.from_numpy(W.batch_stream_kv(TALKER2, b, sp.lens[b])).cuda(),
                                  sp.lens[b], int(sp.tokens[b]))
    ids_g2 = torch.empty((n, B), dtype=torch.int32, device="cuda")
    sp.qd.qd_batch_decode(sp.bh, n, ids_g2)
    assert np.array_equal(ids_g2.cpu().numpy(), ids_g.cpu().numpy())
    with pytest.raises(sp.qd.QDError) as ei:
        sp.qd.qd_batch_set_sampling(sp.bh, 65, t, p, seed)
    assert ei.value.status == sp.qd.QD_EINVAL
    sp.close()


def test_batch_greedy_feeds_back_its_own_ids():
    import torch
    B, smax, n = 4, 256, 5
    lens = W.batch_initial_lengths(n=B, lo=40, hi=200)
    bp = BatchPair(TALKER2, B, smax, lens, oracle_streams=[])
    ids = torch.empty((n, B), dtype=torch.int32, device="cuda")
    bp.qd.qd_batch_decode(bp.bh, n, ids)
    free = ids.cpu().numpy()
    bp.close()
    # the same run forced with its own ids
    bp = BatchPair(TALKER2, B, smax, lens, oracle_streams=[])
    bp.qd.qd_batch_decode(bp.bh, n, ids, torch.from_numpy(free).cuda())
    assert np.array_equal(ids.cpu().numpy(), free)
    bp.close()


def test_batch_errors():
    import torch
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    h = qd.qd_create(upload(W.model_weights(TALKER2)), config_from_shape(TALKER2))
    with pytest.raises(qd.QDError) as ei:
        qd.qd_batch_create(h, 4, 100)                 # not a multiple of 32
    assert ei.value.status == qd.QD_EINVAL
    bh = qd.qd_batch_create(h, 2, 64)
    ids = torch.empty((4, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_batch_decode(bh, 1, ids)                # streams never set
    assert ei.value.status == qd.QD_ESTATE
    qd.qd_batch_set_stream(bh, 0, None, 0, 5)
    qd.qd_batch_set_stream(bh, 1, None, 0, 6)
    with pytest.raises(qd.QDError) as ei:
        qd.qd_batch_set_stream(bh, 1, None, 0, TALKER2.embed_rows)
    assert ei.value.status == qd.QD_EINVAL
    qd.qd_batch_decode(bh, 4, ids)
    qd.qd_batch_sync(bh)
    assert qd.qd_batch_get_pos(bh, 0) == 4
    big = torch.empty((61, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(qd.QDError) as ei:
        qd.qd_batch_decode(bh, 61, big)               # 4 + 61 > 64
    assert ei.value.status == qd.QD_EKVFULL
    qd.qd_batch_destroy(bh)
    qd.qd_destroy(h)


@pytest.mark.slow
def test_batch_full_size_sampled_streams():
    """The batched workload's shapes: 28-layer Talker, 64 streams, smax 2048, lengths
    U{256..1792}.  The first step of all 64 streams, then all of the workload's 256
    teacher-forced steps of streams 0, 21, 42 and 63, against the oracle."""
    import oracle as O
    B, smax = W.BATCH_STREAMS, W.BATCH_SMAX
    lens = W.batch_initial_lengths()
    s = W.TALKER
    bp = BatchPair(s, B, smax, lens, oracle_streams=[0, 21, 42, 63])
    # first step: every stream (oracle streams created one at a time)
    first_ref = {}
    for b in range(B):
        if b in bp.ref:
            continue
        o = O.Oracle(s, bp.w, buckets=(smax,))
        o.set_kv(W.batch_stream_kv(s, b, bp.lens[b]), bp.lens[b])
        rid, rlog, margin, _ = o.step(token=int(bp.tokens[b]))
        first_ref[b] = (rid, rlog, margin)
        o.close()
    out = bp.step()
    g_log = bp.logits.cpu().numpy()
    import torch  # noqa: F401
    for b, (rid, rlog, margin) in first_ref.items():
        assert rel_l2(g_log[b], rlog) <= REL_TOL, b
    for b, (gid, rid, margin, lrel) in out.items():
        assert lrel <= REL_TOL and (margin <= MARGIN or gid == rid), b
    checked = _check_steps(bp, W.BATCH_STEPS - 1)
    assert checked > 4 * (W.BATCH_STEPS - 1) // 2          # the comparison is not vacuous
    for b in (0, 21, 42, 63):
        assert bp.qd.qd_batch_get_pos(bp.bh, b) == bp.lens[b] + W.BATCH_STEPS
    bp.close()


def _prefill_pair(shape, B, smax, streams, n, seed=0):
    """GPU batch prefill of `streams` with n N(0,1) positions each, and the oracle's
    prefill of the same prompts."""
    import torch
    import oracle as O
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    w = W.model_weights(shape, seed=seed)
    h = qd.qd_create(upload(w), config_from_shape(shape))
    bh = qd.qd_batch_create(h, B, smax)
    prompts = np.stack([W.normal(f"batched/prompt/{s}", (n, shape.hidden), seed) for s in streams])
    first = torch.empty(len(streams), dtype=torch.int32, device="cuda")
    qd.qd_batch_prefill(bh, streams, torch.from_numpy(prompts).cuda(), first)
    qd.qd_batch_sync(bh)
    logits = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
    qd.qd_batch_get_logits(bh, logits)
    refs = []
    for k, s in enumerate(streams):
        o = O.Oracle(shape, w, buckets=(smax,))
        rid, rlog, margin = o.prefill(embeds=prompts[k])
        refs.append((o, rid, rlog, margin))
    return qd, h, bh, first.cpu().numpy(), logits.cpu().numpy(), refs


def test_batch_prefill_matches_oracle_and_decodes_on():
    import torch
    B, smax, n = 4, 256, 100                      # 100 positions: ragged query and key tiles
    streams = [3, 1]
    qd, h, bh, first, logits, refs = _prefill_pair(TALKER2, B, smax, streams, n)
    s = TALKER2
    for k, st in enumerate(streams):
        o, rid, rlog, margin = refs[k]
        assert rel_l2(logits[st], rlog) <= REL_TOL
        if margin > MARGIN:
            assert first[k] == rid
        assert qd.qd_batch_get_pos(bh, st) == n
        # the cache the prefill wrote, every layer, K and V
        nb = qd.qd_batch_copy_kv(bh, st)
        buf = torch.empty(nb, dtype=torch.uint8, device="cuda")
        qd.qd_batch_copy_kv(bh, st, buf)
        g = buf.view(torch.int16).cpu().numpy().view(np.uint16).reshape(s.n_layers, 2, s.n_kv_heads, smax, s.head_dim)
        for l in range(s.n_layers):
            for w_ in range(2):
                assert rel_l2(_bf16_to_f32(g[l, w_, :, :n]), o.kv(l, w_)) <= REL_TOL, (st, l, w_)
    # decoding continues from the prefilled caches (the other streams start empty)
    for b in range(B):
        if b not in streams:
            qd.qd_batch_set_stream(bh, b, None, 0, 7)
    ids = torch.empty((3, B), dtype=torch.int32, device="cuda")
    force = np.zeros((3, B), np.int32)
    ref_steps = []
    for k, st in enumerate(streams):
        o, rid, _, _ = refs[k]
        fed = rid
        out = []
        for i in range(3):
            oid, olog, om, _ = o.step(token=fed)
            out.append((oid, olog, om))
            force[i, st] = oid
            fed = oid
        ref_steps.append(out)
    # first step's input is the prefill's own argmax (equal to the oracle's when the margin allows)
    qd.qd_batch_decode(bh, 3, ids, torch.from_numpy(force).cuda())
    qd.qd_batch_sync(bh)
    got = ids.cpu().numpy()
    for k, st in enumerate(streams):
        if refs[k][3] > MARGIN:                   # the fed first id agrees with the oracle's
            for i in range(3):
                oid, _, om = ref_steps[k][i]
                if om > MARGIN:
                    assert got[i, st] == oid, (st, i)
    qd.qd_batch_destroy(bh)
    qd.qd_destroy(h)
    for o, *_ in refs:
        o.close()


@pytest.mark.slow
def test_batch_prefill_full_size_two_streams():
    """The 28-layer Talker prefilling 512 positions on two of the eight prompt streams
    of the prefill workload (the oracle runs those two)."""
    B, smax, n = W.BATCH_PREFILL[0], W.BATCH_SMAX, W.BATCH_PREFILL[1]
    streams = [0, 5]
    qd, h, bh, first, logits, refs = _prefill_pair(W.TALKER, B, smax, streams, n)
    for k, st in enumerate(streams):
        o, rid, rlog, margin = refs[k]
        assert rel_l2(logits[st], rlog) <= REL_TOL
        if margin > MARGIN:
            assert first[k] == rid
    qd.qd_batch_destroy(bh)
    qd.qd_destroy(h)
    for o, *_ in refs:
        o.close()


@pytest.mark.parametrize("hd,qh,kvh,n,smax", [
    (128, 16, 8, 300, 320),   # three query blocks, the last ragged; the cache ends inside the last key chunk
    (128, 8, 1, 129, 256),    # a one-query last block; 8 q heads per kv head
    (64, 8, 8, 257, 512),     # head_dim 64, one query past two whole chunks
    (64, 8, 2, 384, 416),     # whole chunks only: no tail to zero
])
def test_batch_prefill_attention_variants(hd, qh, kvh, n, smax):
    """The tensor-core prefill attention's shapes on one-layer models: several 128-query
    blocks and 128-key chunks, ragged ends, GQA groups of 1, 2 and 8, both head sizes;
    the logits and the written cache against the oracle's prefill."""
    import torch
    hidden = qh * hd
    s = W.scaled(W.TALKER, name=f"pfa_{hd}_{qh}_{kvh}", n_layers=1, hidden=hidden, n_q_heads=qh,
                 n_kv_heads=kvh, head_dim=hd, ffn=2 * hidden, vocab=1024, embed_rows=1024)
    B, streams = 3, [2, 0]
    qd, h, bh, first, logits, refs = _prefill_pair(s, B, smax, streams, n)
    for k, st in enumerate(streams):
        o, rid, rlog, margin = refs[k]
        assert rel_l2(logits[st], rlog) <= REL_TOL, (st, rel_l2(logits[st], rlog))
        if margin > MARGIN:
            assert first[k] == rid
        nb = qd.qd_batch_copy_kv(bh, st)
        buf = torch.empty(nb, dtype=torch.uint8, device="cuda")
        qd.qd_batch_copy_kv(bh, st, buf)
        g = buf.view(torch.int16).cpu().numpy().view(np.uint16).reshape(1, 2, kvh, smax, hd)
        for w_ in range(2):
            assert rel_l2(_bf16_to_f32(g[0, w_, :, :n]), o.kv(0, w_)) <= REL_TOL, (st, w_)
    qd.qd_batch_destroy(bh)
    qd.qd_destroy(h)
    for o, *_ in refs:
        o.close()


@pytest.mark.parametrize("hd,qh,kvh", [(64, 8, 8), (64, 8, 2), (64, 8, 1), (128, 8, 1)])
def test_batch_attention_variants_match_oracle(hd, qh, kvh):
    """The attention's other instantiations (head_dim 64 or 128; 1, 4 or 8 q heads per
    kv head) on one-layer models, cached lengths from one to three 512-position attention
    chunks (the merge of several, and the single-chunk path)."""
    hidden = qh * hd
    s = W.scaled(W.TALKER, name=f"batt_{hd}_{qh}_{kvh}", n_layers=1, hidden=hidden, n_q_heads=qh,
                 n_kv_heads=kvh, head_dim=hd, ffn=2 * hidden, vocab=1024, embed_rows=1024)
    B, smax, n = 4, 1600, 3
    lens = W.batch_initial_lengths(n=B, lo=100, hi=1500)   # 1001, 445, 1412, 590: 1 to 3 chunks
    bp = BatchPair(s, B, smax, lens)
    _check_steps(bp, n)
    bp.close()

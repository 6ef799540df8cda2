// Persistent decode step: the whole per-token step of the decoder in one cooperative
// launch with one CTA per SM.
//
// Sources (page title, section):
//  - "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile and graph-replay entries:
//    the step is a chain of small dependent operations per layer whose launch and
//    synchronisation costs dominate at batch 1; replaying it as a graph helped only a
//    little.  Here the chain lives inside one kernel: each phase waits for the data it
//    gathers from the others (below), and each CTA's producer warp streams that CTA's
//    slice of every phase's weights (and its attention K/V tile) through one
//    shared-memory ring without waiting on them, so HBM keeps streaming while the
//    phases synchronise.
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation", and "Audio8-ASR: dynamic KV-cache buckets", section "Implemented
//    dynamic window mechanism": the arithmetic of each phase (shared with the
//    per-phase kernels through decode_common.cuh).
//
// Phases of layer l:
//   A  x^ = RMSNorm(x), qkv = [Wq;Wk;Wv] x^   (layer 0 also resolves the step input)
//   B  attention: CTA i < kv_heads * splits takes (group, split) i; QK-norm, RoPE, KV
//      append, scores/softmax/P.V of the split -> partials
//   C  output projection: merge the splits, x += Wo o
//   D  x^ = RMSNorm(x), act = silu(Wg x^) * (Wu x^)
//   E  x += Wd act
// then the head: y = RMSNorm(x), logits, penalty, EOS mask, argmax (last CTA reduces).
//
// Between phases.  The vectors every CTA gathers (qkv after A, x after C and E, act
// after D) are also written as 64-bit words {tag, value}, the tag naming the launch
// (a sequence number advanced once per launch) and the phase; a reader polls the words
// it needs until their tags match, so the data and its readiness travel in one access
// and these four boundaries need no barrier round trip.  A buffer is only rewritten
// after every CTA has read its previous contents: each rewrite depends, through the
// chain of gathers, on every CTA having finished the phase that read them.  Only the
// attention partials (B -> C) cross a grid barrier, which also orders the plain
// writes of the step input and the emitted set.
#include "decode_common.cuh"

namespace qd {

// Grid barrier over all CTAs (consumer threads of every CTA arrive).  Thread 0
// publishes the CTA's writes with a release reduction and polls with acquire loads,
// for at most kWaitLimitNs.  Returns false on timeout (uniform across the CTA).
__device__ __forceinline__ bool grid_sync(unsigned *counter, unsigned &epoch, int *flag) {
    named_sync(1, kConsumerWarps * 32);
    ++epoch;
    if (threadIdx.x == 0) {
        const unsigned target = epoch * gridDim.x;
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
        const unsigned long long t0 = global_timer_ns();
        int ok = 1;
        while (true) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= target) break;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                ok = 0;
                break;
            }
        }
        *flag = ok;
    }
    named_sync(1, kConsumerWarps * 32);
    return *flag != 0;
}

// Tagged words: the value's bits low, the tag high, in one 64-bit access.
__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
// The tag of phase k of layer l in the launch with sequence number seq (1 + 5l + k < 256).
// The tag keeps the low 24 bits of seq: consecutive launches always differ, and a word
// could only pass as fresh if no launch had rewritten it for 2^24 launches.  The phase
// field is never 0, so the zeroed words of a new handle never match.
__device__ __forceinline__ uint32_t phase_tag(uint32_t seq, int l, int k) { return (seq << 8) | (uint32_t)(1 + 5 * l + k); }

// Advance the launch sequence number from `seq` (the value this launch read) to seq + 1,
// modulo 2^32, exactly once however many threads of the launch call it.
__device__ __forceinline__ void advance_seq(unsigned *p, uint32_t seq) { (void)atomicCAS(p, seq, seq + 1u); }

struct TagSeg {                    // dst[i] = value of src[i], i < n
    const uint64_t *src;
    int n;
    float *dst;
};
// Consumer threads: the values of up to three tagged segments once their tags equal
// `tag`, into shared memory.  Each thread loads a batch of words at once and re-polls
// every still-stale word of the batch together (one round trip per poll, not one per
// word), for at most kWaitLimitNs.  False (uniform across the CTA) on timeout.  Ends
// with a consumer barrier.
__device__ __noinline__ bool gather_tagged(TagSeg s0, TagSeg s1, TagSeg s2, uint32_t tag) {
    constexpr int NC = kConsumerWarps * 32, B = 8;
    const int tid = threadIdx.x;
    const int n01 = s0.n + s1.n, n = n01 + s2.n;
    bool ok = true;
    unsigned long long t0 = 0;
    for (int base = tid; base < n; base += B * NC) {
        const uint64_t *src[B];
        uint64_t w[B];
        unsigned pending = 0;
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = base + k * NC;
            src[k] = i < s0.n ? s0.src + i : (i < n01 ? s1.src + (i - s0.n) : s2.src + (i - n01));
            w[k] = i < n ? ld_tagged(src[k]) : (uint64_t)tag << 32;
        }
#pragma unroll
        for (int k = 0; k < B; ++k)
            if ((uint32_t)(w[k] >> 32) != tag) pending |= 1u << k;
        while (pending && ok) {
            const unsigned long long t = global_timer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitLimitNs) ok = false;
#pragma unroll
            for (int k = 0; k < B; ++k)
                if ((pending >> k) & 1u) w[k] = ld_tagged(src[k]);
#pragma unroll
            for (int k = 0; k < B; ++k)
                if ((uint32_t)(w[k] >> 32) == tag) pending &= ~(1u << k);
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = base + k * NC;
            if (i >= n) continue;
            float *dst = i < s0.n ? s0.dst + i : (i < n01 ? s1.dst + (i - s0.n) : s2.dst + (i - n01));
            *dst = __uint_as_float((uint32_t)w[k]);
        }
    }
    return !named_sync_or(1, NC, !ok);
}
__device__ __forceinline__ bool gather_tagged(const uint64_t *src, int n, float *dst, uint32_t tag) {
    return gather_tagged(TagSeg{src, n, dst}, TagSeg{nullptr, 0, nullptr}, TagSeg{nullptr, 0, nullptr}, tag);
}

// Stage a vector of weights (gamma) into shared memory (consumer threads).
__device__ __forceinline__ void stage_vec(float *dst, const float *src, int n) {
    for (int i = threadIdx.x * 4; i < n; i += kConsumerWarps * 32 * 4)
        *reinterpret_cast<float4 *>(dst + i) = *reinterpret_cast<const float4 *>(src + i);
}

// Merge the attention splits into `dst` (shared memory, q_dim floats): thread t of
// the consumers merges 8 consecutive columns (one head), with every load it needs in
// flight at once (flash-decoding combine, splits in index order; the same operations
// in the same order as the cluster merge of the per-phase attention kernel).
template <int HD>
__device__ __forceinline__ void combine_to_smem(const float *part_o, const float *part_ml, int ns, int q_dim,
                                                float *dst) {
    constexpr int CPT = 8;   // columns per thread
    for (int c0 = threadIdx.x * CPT; c0 < q_dim; c0 += kConsumerWarps * 32 * CPT) {
        const int h = c0 / HD, d0 = c0 % HD;
        const float *ml = part_ml + (size_t)h * kAttnMaxSplits * 2;
        const float *po = part_o + (size_t)h * kAttnMaxSplits * HD + d0;
        float2 m_l[kAttnMaxSplits];
        float4 oa[kAttnMaxSplits], ob[kAttnMaxSplits];
#pragma unroll
        for (int t = 0; t < kAttnMaxSplits; ++t) {
            if (t < ns) {
                m_l[t] = __ldcg(reinterpret_cast<const float2 *>(ml + 2 * t));
                oa[t] = __ldcg(reinterpret_cast<const float4 *>(po + (size_t)t * HD));
                ob[t] = __ldcg(reinterpret_cast<const float4 *>(po + (size_t)t * HD + 4));
            } else {
                m_l[t] = make_float2(-INFINITY, 0.f);
                oa[t] = ob[t] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int t = 0; t < kAttnMaxSplits; ++t) M = fmaxf(M, m_l[t].x);
        float acc[CPT] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float den = 0.f;
#pragma unroll
        for (int t = 0; t < kAttnMaxSplits; ++t) {
            if (t < ns) {
                const float w = expf(m_l[t].x - M);
                acc[0] = fmaf(oa[t].x, w, acc[0]);
                acc[1] = fmaf(oa[t].y, w, acc[1]);
                acc[2] = fmaf(oa[t].z, w, acc[2]);
                acc[3] = fmaf(oa[t].w, w, acc[3]);
                acc[4] = fmaf(ob[t].x, w, acc[4]);
                acc[5] = fmaf(ob[t].y, w, acc[5]);
                acc[6] = fmaf(ob[t].z, w, acc[6]);
                acc[7] = fmaf(ob[t].w, w, acc[7]);
                den = fmaf(m_l[t].y, w, den);
            }
        }
        // two 16-byte stores (one per column would put every fourth lane on one bank)
        *reinterpret_cast<float4 *>(dst + c0) = make_float4(acc[0] / den, acc[1] / den, acc[2] / den, acc[3] / den);
        *reinterpret_cast<float4 *>(dst + c0 + 4) = make_float4(acc[4] / den, acc[5] / den, acc[6] / den, acc[7] / den);
    }
}

__device__ __forceinline__ void cta_rows(int rows, int unit, int &r0, int &nr) {
    const int units = rows / unit;
    const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
    r0 = u0 * unit;
    nr = (u1 - u0) * unit;
}

template <typename WT, int HD, int NS_H, int NS_Q, int NS_F>
__global__ void __launch_bounds__(kGemvThreads, 1) decode_step_kernel(const StepArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    typedef WT KT;
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    constexpr int NC = kConsumerWarps * 32;
    constexpr int HALF = HD / 2;
    constexpr size_t ES = sizeof(WT);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_full);
    uint64_t *empty = full + a.nst;
    float *gsm = reinterpret_cast<float *>(smem + a.off_gsm);
    float *misc = reinterpret_cast<float *>(smem + a.off_misc);   // 64 words
    int *misc_i = reinterpret_cast<int *>(misc + 32);
    volatile int *ctl = reinterpret_cast<volatile int *>(misc_i + 16);   // [0] stop [1] issued [2] producer done
    int *flag = misc_i + 20;
    float *res = reinterpret_cast<float *>(smem + a.off_res);
    uint32_t *emw = reinterpret_cast<uint32_t *>(smem + a.off_emw);
    float *xin = reinterpret_cast<float *>(smem + a.off_xin);   // phase input vector
    const Ring R{smem, full, empty, a.nst};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.qh / a.kvh;
    const int hidden = a.hidden, q_dim = a.qh * HD, kv_dim = a.kvh * HD;
    const int CM = a.chunk_max;

    // The step's position: the previous launch has completed, so it is final.
    const int p = a.st->pos;
    const int L = p + 1;
    const int C = attn_chunk(L);
    const int nsplit = attn_splits(L);
    const bool valid = p < a.S && C <= CM;
    const bool has_item = valid && (int)blockIdx.x < a.kvh * nsplit;
    const int ig = has_item ? (int)blockIdx.x / nsplit : 0;
    const int is = has_item ? (int)blockIdx.x % nsplit : 0;
    const int j0 = is * C;
    const int n_att = has_item ? (L - j0 < C ? L - j0 : C) : 0;
    const int n_old = has_item ? ((p - j0) < n_att ? (p - j0) : n_att) : 0;

    int r0_qkv, n_qkv, r0_o, n_o, r0_gu, n_gu, r0_d, n_d, r0_hd, n_hd;
    cta_rows(q_dim + 2 * kv_dim, 1, r0_qkv, n_qkv);
    cta_rows(hidden, 1, r0_o, n_o);
    cta_rows(2 * a.ffn, 2, r0_gu, n_gu);
    cta_rows(hidden, 1, r0_d, n_d);
    cta_rows(a.vocab, 1, r0_hd, n_hd);
    const uint32_t rb_h = (uint32_t)(hidden * ES), rb_q = (uint32_t)(q_dim * ES), rb_f = (uint32_t)(a.ffn * ES);
    const size_t layer_kv = (size_t)2 * kv_dim * a.S * ES;

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        ctl[0] = 0;
        ctl[1] = 0;
        ctl[2] = 0;
        if (!valid && blockIdx.x == 0) atomicOr(&a.st->status, DEV_ERR_BAD_POS);
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: every phase's weights, in consumption order
        if (lane == 0) {
            const uint64_t pw = a.evict_last ? policy_evict_last() : policy_evict_first();
            const uint64_t pf = policy_evict_first();
            uint32_t sidx = 0;
            bool ok = true;
            for (int l = 0; l < a.n_layers && ok && !ctl[0]; ++l) {
                const LayerDev &Ld = a.layers[l];
                ok = ok && produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(Ld.w_qkv) + (size_t)r0_qkv * rb_h,
                                        n_qkv, rb_h, a.rps_h, pw);
                if (has_item) {
                    // K and V rows [j0, j0 + n_old) of this CTA's group: written by earlier steps
                    const uint8_t *kb = reinterpret_cast<const uint8_t *>(a.kv) + (size_t)l * layer_kv +
                                        ((size_t)ig * a.S + j0) * HD * ES;
                    const uint32_t bytes = (uint32_t)(n_old * HD * ES);
                    ok = ok && produce_block(R, sidx, kb, bytes, pf);
                    ok = ok && produce_block(R, sidx, kb + layer_kv / 2, bytes, pf);
                }
                ok = ok && produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(Ld.w_o) + (size_t)r0_o * rb_q, n_o,
                                        rb_q, a.rps_q, pw);
                ok = ok && produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(Ld.w_gu) + (size_t)r0_gu * rb_h,
                                        n_gu, rb_h, a.rps_h, pw);
                ok = ok && produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(Ld.w_d) + (size_t)r0_d * rb_f, n_d,
                                        rb_f, a.rps_f, pw);
            }
            if (ok && a.with_head && !ctl[0]) {
                const uint8_t *Wh = reinterpret_cast<const uint8_t *>(a.heads[a.st->head_idx]);
                ok = produce_rows(R, sidx, Wh + (size_t)r0_hd * rb_h, n_hd, rb_h, a.rps_h, pf);
            }
            if (!ok) atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
            ctl[1] = (int)sidx;
            __threadfence_block();
            ctl[2] = 1;
        }
        return;
    }

    // ---------------- consumers
    // attention scratch: q heads, k, v, RoPE row of position p, QK-norm gammas, scores,
    // split output; the RoPE row is constant for the launch
    float *qs = reinterpret_cast<float *>(smem + a.off_att);
    float *kn = qs + G * HD, *vn = kn + HD, *rc = vn + HD, *qg = rc + HD, *kg = qg + HD, *sc = kg + HD;
    float *po = sc + G * CM, *pm = po + G * HD, *pl = pm + G;
    if (has_item) {
        // rotary position: the cache position + delta, or per stream from the staged prompt
        const int *stage = a.st->rope_staged ? a.rope_stage : nullptr;
        const int pr = p + a.st->rope_delta;
        for (int m = tid; m < HALF; m += NC) {
            const size_t r = (size_t)rope_row(m, a.mrope_h, stage, a.rope_stride, p, pr, a.rope_rows);
            rc[m] = a.rope_cos[r * HALF + m];
            rc[HALF + m] = a.rope_sin[r * HALF + m];
        }
    }
    const int rr_h = warp / a.rs_h, colb_h = (warp % a.rs_h) * (hidden / a.rs_h);
    const int colb_q = (warp % a.rs_q) * (q_dim / a.rs_q);
    const int colb_f = (warp % a.rs_f) * (a.ffn / a.rs_f);
    uint32_t sidx = 0;
    unsigned epoch = 0;
    bool ok = true;
    // this launch's sequence number (advanced once every CTA has read it: at the commit)
    const uint32_t seq = *reinterpret_cast<volatile const unsigned *>(a.seq);

    for (int l = 0; l < a.n_layers && ok; ++l) {
        const LayerDev &Ld = a.layers[l];
        // ---- A: qkv = [Wq; Wk; Wv] RMSNorm(x)
        stage_vec(gsm, Ld.attn_norm, hidden);
        {
            float xr[NS_H * EPL];
            if (l == 0) {
                step_input_slice<WT, NS_H>(a.in, a.st, hidden, a.rs_h, colb_h, xr, misc_i, a.x, a.tap_hidden);
            } else {
                ok = gather_tagged(a.x_t, hidden, xin, phase_tag(seq, l - 1, 4));
                if (!ok) break;
                smem_slice<WT, NS_H>(xin, colb_h, xr);
                if (a.tap_hidden && blockIdx.x == 0 && rr_h == 0) {
#pragma unroll
                    for (int sg = 0; sg < NS_H; ++sg)
#pragma unroll
                        for (int e = 0; e < EPL; ++e)
                            a.tap_hidden[(size_t)l * hidden + colb_h + sg * SEGW + lane * EPL + e] = xr[sg * EPL + e];
                }
            }
            rmsnorm_slice<WT, NS_H>(xr, gsm, hidden, a.rs_h, colb_h, a.eps, misc, nullptr);
            const bool got = gemv_consume<WT, NS_H>(R, sidx, n_qkv, a.rps_h, rb_h, a.rs_h, colb_h, xr, res);
            ok = !named_sync_or(1, NC, !got);
            if (!ok) break;
        }
        for (int r = tid; r < n_qkv; r += NC) {
            float v = 0.f;
            for (int j = 0; j < a.rs_h; ++j) v += res[r * a.rs_h + j];
            a.qkv[r0_qkv + r] = v;
            st_tagged(a.qkv_t + r0_qkv + r, v, phase_tag(seq, l, 0));
        }
        if (has_item && Ld.q_norm)
            for (int i = tid; i < HD; i += NC) {
                qg[i] = Ld.q_norm[i];
                kg[i] = Ld.k_norm[i];
            }

        // ---- B: attention of this CTA's (group, split)
        if (has_item) {
            // the group's q heads, k and v, as their writers tag them
            ok = gather_tagged(TagSeg{a.qkv_t + (size_t)ig * G * HD, G * HD, qs},
                               TagSeg{a.qkv_t + (size_t)q_dim + (size_t)ig * HD, HD, kn},
                               TagSeg{a.qkv_t + (size_t)(q_dim + kv_dim) + (size_t)ig * HD, HD, vn},
                               phase_tag(seq, l, 0));
            if (!ok) break;
            qk_norm_rope<HD, kConsumerWarps>(qs, kn, G, Ld.q_norm ? qg : nullptr, kg, a.eps, rc, 1);
            const uint8_t *kslot = slot_acquire(R, sidx);
            const uint8_t *vslot = kslot ? slot_acquire(R, sidx + 1) : nullptr;
            ok = !named_sync_or(1, NC, vslot == nullptr);
            if (!ok) break;
            KT *Ks = reinterpret_cast<KT *>(const_cast<uint8_t *>(kslot));
            KT *Vs = reinterpret_cast<KT *>(const_cast<uint8_t *>(vslot));
            if (n_old < n_att) {
                // this split holds position p: append the new row (cache type)
                KT *kw = reinterpret_cast<KT *>(reinterpret_cast<uint8_t *>(a.kv) + (size_t)l * layer_kv) +
                         ((size_t)ig * a.S + p) * HD;
                KT *vw = reinterpret_cast<KT *>(reinterpret_cast<uint8_t *>(a.kv) + (size_t)l * layer_kv +
                                                layer_kv / 2) +
                         ((size_t)ig * a.S + p) * HD;
                for (int i = tid; i < HD; i += NC) {
                    Elem<KT>::store(Ks + n_old * HD, i, kn[i]);
                    Elem<KT>::store(Vs + n_old * HD, i, vn[i]);
                    Elem<KT>::store(kw, i, kn[i]);
                    Elem<KT>::store(vw, i, vn[i]);
                }
                fence_proxy_async_global();
            }
            named_sync(1, NC);
            attn_split<KT, HD, kConsumerWarps>(Ks, Vs, qs, G, n_att, CM, a.scale, sc, po, pm, pl, 1);
            named_sync(1, NC);
            for (int i = tid; i < G * HD; i += NC) {
                const int hh = i / HD, d = i % HD;
                a.part_o[((size_t)(ig * G + hh) * kAttnMaxSplits + is) * HD + d] = po[i];
            }
            for (int hh = tid; hh < G; hh += NC) {
                float *ml = a.part_ml + ((size_t)(ig * G + hh) * kAttnMaxSplits + is) * 2;
                ml[0] = pm[hh];
                ml[1] = pl[hh];
            }
            fence_proxy_async_smem();   // generic writes into the slots precede their next bulk fill
            slot_release(R, sidx, lane);
            slot_release(R, sidx + 1, lane);
            sidx += 2;
        }
        ok = grid_sync(a.barrier, epoch, flag);
        if (!ok) break;

        // ---- C: x += Wo (merged attention output)
        {
            const float xold = tid < n_o ? __ldcg(a.x + r0_o + tid) : 0.f;
            float xr[NS_Q * EPL];
            combine_to_smem<HD>(a.part_o, a.part_ml, valid ? nsplit : 0, q_dim, xin);
            named_sync(1, NC);
            smem_slice<WT, NS_Q>(xin, colb_q, xr);
            const bool got = gemv_consume<WT, NS_Q>(R, sidx, n_o, a.rps_q, rb_q, a.rs_q, colb_q, xr, res);
            ok = !named_sync_or(1, NC, !got);
            if (!ok) break;
            if (tid < n_o) {
                float v = 0.f;
                for (int j = 0; j < a.rs_q; ++j) v += res[tid * a.rs_q + j];
                a.x[r0_o + tid] = xold + v;
                st_tagged(a.x_t + r0_o + tid, xold + v, phase_tag(seq, l, 2));
            }
        }
        stage_vec(gsm, Ld.mlp_norm, hidden);

        // ---- D: act = silu(Wg x^) * (Wu x^), x^ = RMSNorm(x)
        {
            float xr[NS_H * EPL];
            ok = gather_tagged(a.x_t, hidden, xin, phase_tag(seq, l, 2));
            if (!ok) break;
            smem_slice<WT, NS_H>(xin, colb_h, xr);
            rmsnorm_slice<WT, NS_H>(xr, gsm, hidden, a.rs_h, colb_h, a.eps, misc, nullptr);
            const bool got = gemv_consume<WT, NS_H>(R, sidx, n_gu, a.rps_h, rb_h, a.rs_h, colb_h, xr, res);
            ok = !named_sync_or(1, NC, !got);
            if (!ok) break;
        }
        for (int i = tid; i < n_gu / 2; i += NC) {
            float g = 0.f, u = 0.f;
            for (int j = 0; j < a.rs_h; ++j) {
                g += res[(2 * i) * a.rs_h + j];
                u += res[(2 * i + 1) * a.rs_h + j];
            }
            const float act = g / (1.0f + expf(-g)) * u;
            a.act[r0_gu / 2 + i] = act;
            st_tagged(a.act_t + r0_gu / 2 + i, act, phase_tag(seq, l, 3));
        }

        // ---- E: x += Wd act (x rows: this thread's own, written in C)
        {
            const float xold = tid < n_d ? __ldcg(a.x + r0_d + tid) : 0.f;
            float xr[NS_F * EPL];
            ok = gather_tagged(a.act_t, a.ffn, xin, phase_tag(seq, l, 3));
            if (!ok) break;
            smem_slice<WT, NS_F>(xin, colb_f, xr);
            const bool got = gemv_consume<WT, NS_F>(R, sidx, n_d, a.rps_f, rb_f, a.rs_f, colb_f, xr, res);
            ok = !named_sync_or(1, NC, !got);
            if (!ok) break;
            if (tid < n_d) {
                float v = 0.f;
                for (int j = 0; j < a.rs_f; ++j) v += res[tid * a.rs_f + j];
                a.x[r0_d + tid] = xold + v;
                st_tagged(a.x_t + r0_d + tid, xold + v, phase_tag(seq, l, 4));
            }
        }
    }

    if (ok && a.with_head) {
        // ---- head: y = RMSNorm(x); logits; penalty; EOS mask; argmax
        stage_vec(gsm, a.final_norm, hidden);
        const int w0 = r0_hd >> 5;
        const int nw = n_hd > 0 ? ((r0_hd + n_hd - 1) >> 5) - w0 + 1 : 0;
        if (a.penalty != 1.0f)
            for (int i = tid; i < nw; i += NC) emw[i] = __ldcg(a.in.emitted + w0 + i);
        ok = gather_tagged(a.x_t, hidden, xin, phase_tag(seq, a.n_layers - 1, 4));
        if (ok) {
            float xr[NS_H * EPL];
            smem_slice<WT, NS_H>(xin, colb_h, xr);
            if (a.tap_hidden && blockIdx.x == 0 && rr_h == 0) {
#pragma unroll
                for (int sg = 0; sg < NS_H; ++sg)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        a.tap_hidden[(size_t)a.n_layers * hidden + colb_h + sg * SEGW + lane * EPL + e] =
                            xr[sg * EPL + e];
            }
            rmsnorm_slice<WT, NS_H>(xr, gsm, hidden, a.rs_h, colb_h, a.eps, misc,
                                    blockIdx.x == 0 ? a.y_out : nullptr);
            const bool got = gemv_consume<WT, NS_H>(R, sidx, n_hd, a.rps_h, rb_h, a.rs_h, colb_h, xr, res);
            ok = !named_sync_or(1, NC, !got);
        }
        if (ok) {
            // greedy: per-thread, per-warp, per-CTA argmax.  Sampling (top-k > 0): the
            // CTA's final logits stay in res and the CTA's top-k candidates go out.
            const int sk = a.st->sample_k;
            float best_v = -INFINITY;
            int best_i = INT_MAX;
            for (int r = tid; r < n_hd; r += NC) {
                float v = 0.f;
                for (int j = 0; j < a.rs_h; ++j) v += res[r * a.rs_h + j];
                const int row = r0_hd + r;
                if (a.tap_logits) a.tap_logits[row] = v;
                if (a.penalty != 1.0f && ((emw[(row >> 5) - w0] >> (row & 31)) & 1u))
                    v = v > 0.f ? v / a.penalty : v * a.penalty;
                if (row == a.eos) v = -INFINITY;
                if (sk > 0) {
                    res[r * a.rs_h] = v;
                } else if (arg_better(v, row, best_v, best_i)) {
                    best_v = v;
                    best_i = row;
                }
            }
            // sampling scratch over the ring, idle now: the CTA's candidates, the
            // selection scratch, then (last CTA) every CTA's candidates
            float *cv = reinterpret_cast<float *>(smem);
            int *ci = reinterpret_cast<int *>(cv + kMaxTopK);
            int *scr = ci + kMaxTopK;
            uint64_t *all_k = reinterpret_cast<uint64_t *>(scr + kTopkScratchWords);   // 8-byte aligned
            if (sk > 0) {
                named_sync(1, NC);
                block_topk(res, a.rs_h, nullptr, r0_hd, n_hd, sk, cv, ci, scr);
                if (tid < sk) {
                    a.part_v[(size_t)blockIdx.x * sk + tid] = cv[tid];
                    a.part_i[(size_t)blockIdx.x * sk + tid] = ci[tid];
                }
            } else {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
                    if (arg_better(ov, oi, best_v, best_i)) {
                        best_v = ov;
                        best_i = oi;
                    }
                }
                if (lane == 0) {
                    misc[8 + warp] = best_v;
                    misc_i[8 + warp] = best_i;
                }
            }
            named_sync(1, NC);
            if (tid == 0) {
                if (sk == 0) {
                    float bv = misc[8];
                    int bi = misc_i[8];
                    for (int w = 1; w < kConsumerWarps; ++w)
                        if (arg_better(misc[8 + w], misc_i[8 + w], bv, bi)) {
                            bv = misc[8 + w];
                            bi = misc_i[8 + w];
                        }
                    a.part_v[blockIdx.x] = bv;
                    a.part_i[blockIdx.x] = bi;
                }
                __threadfence();
                const int prev = atomicAdd(a.head_counter, 1);
                misc_i[5] = (prev == (int)gridDim.x - 1);
            }
            named_sync(1, NC);
            // last CTA: the step's id, published; the position advanced
            auto commit = [&](int id) {
                *a.head_counter = 0;
                DevState *st = a.st;
                st->out_id = id;
                const int n = st->n_gen;
                if (n < a.ids_cap) a.ids[n] = id;
                else atomicOr(&st->status, DEV_ERR_IDS_FULL);
                st->n_gen = n + 1;
                st->pos = p + 1;
                advance_seq(a.seq, seq);
            };
            if (misc_i[5] && sk > 0) {
                // every CTA's sorted candidates -> merged -> the draw
                __threadfence();
                merge_candidate_lists(a.part_v, a.part_i, (int)gridDim.x, sk, all_k, cv, ci, scr);
                if (warp == 0) {
                    const DevState *st = a.st;
                    const uint64_t seed = ((uint64_t)st->seed_hi << 32) | st->seed_lo;
                    const int id = warp_sample(cv, ci, sk, st->sample_temp, st->sample_top_p,
                                               uniform53(seed, (uint64_t)st->n_gen));
                    if (lane == 0) commit(id);
                }
            } else if (misc_i[5] && warp == 0) {
                // reduce the per-CTA argmax candidates
                __threadfence();
                float bv = -INFINITY;
                int bi = INT_MAX;
                for (int c = lane; c < (int)gridDim.x; c += 32) {
                    const float v = __ldcg(a.part_v + c);
                    const int i = __ldcg(a.part_i + c);
                    if (arg_better(v, i, bv, bi)) {
                        bv = v;
                        bi = i;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (arg_better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if (lane == 0) commit(bi);
            }
        }
    } else if (ok) {
        // no head: after every CTA is done, CTA 0 records x and advances the position
        ok = grid_sync(a.barrier, epoch, flag);
        if (ok && blockIdx.x == 0) {
            if (a.tap_hidden)
                for (int i = tid; i < hidden; i += NC)
                    a.tap_hidden[(size_t)a.n_layers * hidden + i] = __ldcg(a.x + i);
            if (tid == 0) {
                a.st->pos = p + 1;
                advance_seq(a.seq, seq);
            }
        }
    }

    if (!ok) {
        // timeout: stop the producer, let copies already issued land, leave
        named_sync(1, NC);
        if (tid == 0) {
            atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
            advance_seq(a.seq, seq);   // no tag of this launch is ever taken as fresh
            ctl[0] = 1;
            const unsigned long long t0 = global_timer_ns();
            while (!ctl[2] && global_timer_ns() - t0 < 2 * kWaitLimitNs + 100000000ull) {
            }
            const uint32_t issued = (uint32_t)ctl[1];
            for (uint32_t s2 = sidx; s2 < issued; ++s2)
                (void)mbar_wait_bounded(&full[s2 % a.nst], (s2 / a.nst) & 1, 10000000ull);
        }
    }
}

// ---------------------------------------------------------------------------------
// Host side: instantiations and launch
// ---------------------------------------------------------------------------------

typedef void (*StepFn)(const StepArgs);

// Shapes with an instantiation: (dtype, head_dim, hidden, q_dim, ffn)
static StepFn step_fn(bool bf16, int hd, int hidden, int q_dim, int ffn) {
    if (!bf16 && hd == 64 && hidden == 256 && q_dim == 256 && ffn == 768)
        return decode_step_kernel<float, 64, 2, 2, 3>;          // one-layer fp32 decoder
    if (bf16 && hd == 64 && hidden == 512 && q_dim == 512 && ffn == 2048)
        return decode_step_kernel<__nv_bfloat16, 64, 2, 2, 4>;  // ASR decoder
    if (bf16 && hd == 128 && hidden == 1024 && q_dim == 2048 && ffn == 3072)
        return decode_step_kernel<__nv_bfloat16, 128, 4, 4, 3>; // talker / code predictor
    return nullptr;
}

bool persistent_supported(bool bf16, int hd, int hidden, int q_dim, int ffn) {
    return step_fn(bf16, hd, hidden, q_dim, ffn) != nullptr;
}

size_t persistent_att_bytes(int group, int hd, int chunk_max) {
    return ((size_t)group * hd + 5 * (size_t)hd + (size_t)group * chunk_max + (size_t)group * hd + 2 * (size_t)group) *
           4;
}

cudaError_t persistent_init(bool bf16, int hd, int hidden, int q_dim, int ffn) {
    StepFn f = step_fn(bf16, hd, hidden, q_dim, ffn);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kStepMaxSmem);
}

cudaError_t launch_persistent(bool bf16, int hd, int hidden, int q_dim, int ffn, const StepArgs &a, int grid,
                              size_t smem, cudaStream_t s) {
    StepFn f = step_fn(bf16, hd, hidden, q_dim, ffn);
    if (!f) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(a.barrier, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void *args[1] = {const_cast<StepArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(f), args);
}

}  // namespace qd

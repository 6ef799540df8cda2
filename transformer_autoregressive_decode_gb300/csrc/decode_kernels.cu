// Decode-step kernels for one stream (batch 1) on sm_103a.
//
// Sources (page title, section):
//  - "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile entry: the per-layer
//    sequence input_norm -> qkv_gemm -> qk_layout_cache -> attention ->
//    output_gemm_residual -> post_norm -> gate_up_gemm -> swiglu ->
//    down_gemm_residual.  Here norm+projection, gate/up+SwiGLU and
//    projection+residual are each one kernel, and the q/k layout step vanishes:
//    QK-norm, RoPE and the KV append run in the attention kernel's prologue,
//    writing the new row straight into the [kv_heads, Smax, head_dim] cache.
//    The same entry found a naive one-block-per-column GEMV slower than the
//    library GEMM; these GEMVs stream each CTA's contiguous row block through a
//    shared-memory ring with bulk async copies instead.
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and
//    two-level generation": QK-norm over head_dim, GQA 8 -> 16, plain RoPE,
//    repetition penalty on emitted ids, greedy argmax.
//  - "Audio8-ASR: dynamic KV-cache buckets", section "Implemented dynamic
//    window mechanism": [heads, Smax, head_dim] cache written in place; bucket
//    migration copies the valid region of every layer's K and V; the embedding
//    lookup of the fed-back token is part of the step.
#include "decode_common.cuh"

namespace qd {

// =====================================================================================
// GEMV: out[r] = W[r, :] . v  with v = RMSNorm(in) (QKV, GU, HEAD) or v = in (RES).
//
// Each CTA owns a contiguous block of rows.  A producer warp streams the block
// through a ring of `nst` stages (kSlotBytes each) with cp.async.bulk, gated by
// per-stage full/empty mbarriers; it never waits on the previous kernel, because
// weights never depend on it, so under programmatic dependent launch the weight
// stream starts while the previous kernel is still running.  Eight consumer warps
// reduce the rows: a row is split over `rs` warps, each lane keeps its slice of v
// in registers.  Partial sums go to shared memory and the epilogue runs once, over
// all rows in parallel, after the stage loop.  All sums have a fixed order, so the
// results are bitwise reproducible.
// =====================================================================================

template <typename WT, int NSEG, int MODE>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int EPL = Elem<WT>::kPer16B;   // elements per lane per 16 bytes
    constexpr int SEGW = 32 * EPL;           // elements per warp segment
    constexpr int NC = kConsumerWarps * 32;  // consumer threads
    const int K = a.K;
    const uint32_t row_bytes = (uint32_t)K * (uint32_t)sizeof(WT);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nst * kSlotBytes);
    uint64_t *empty = full + a.nst;
    float *gsm = reinterpret_cast<float *>(empty + a.nst);   // [K] RMSNorm gamma (16-byte aligned)
    float *misc = gsm + K;                                   // [64]
    int *misc_i = reinterpret_cast<int *>(misc + 32);
    float *xin = misc + 64;                                  // [K] input vector
    float *res = xin + K;                                    // [rows_max][rs]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = a.rows / a.unit;
    const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
    const int row0 = u0 * a.unit;
    const int nrows = (u1 - u0) * a.unit;
    const int rps = a.rps;
    const int nstages = (nrows + rps - 1) / rps;

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        misc_i[4] = 0;   // failure flag
        fence_barrier_init();
    }
    __syncthreads();

    const Ring R{ring, full, empty, a.nst};
    if (warp == kConsumerWarps) {
        // ---------------- producer: stream this CTA's rows through the ring
        if (lane == 0 && nstages > 0) {
            const WT *W = MODE == GEMV_HEAD ? reinterpret_cast<const WT *>(a.W_table[a.st->head_idx])
                                            : reinterpret_cast<const WT *>(a.W);
            const uint8_t *Wb = reinterpret_cast<const uint8_t *>(W) + (size_t)row0 * row_bytes;
            uint32_t sidx = 0;
            if (!produce_rows(R, sidx, Wb, nrows, row_bytes, rps,
                              a.evict_last ? policy_evict_last() : policy_evict_first()))
                atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers
    const int rs = a.rs;
    const int sub = warp % rs;
    const int rr = warp / rs;
    const int rpp = kConsumerWarps / rs;
    const int colbase = sub * (K / rs);
    float xr[NSEG * EPL];
    if (MODE != GEMV_RES) {
        // gamma is a weight: stage it in shared memory before waiting on the previous kernel
        for (int i = tid * 4; i < K; i += NC * 4)
            *reinterpret_cast<float4 *>(gsm + i) = *reinterpret_cast<const float4 *>(a.gamma + i);
    }
    uint32_t *emw = reinterpret_cast<uint32_t *>(res + a.rows_max * a.rs);   // HEAD: emitted words of the rows
    const int w0 = row0 >> 5;
    const int nw = nrows > 0 ? ((row0 + nrows - 1) >> 5) - w0 + 1 : 0;
    if (MODE == GEMV_HEAD && a.penalty != 1.0f) {
        // the emitted set was last written by the first kernel of this step, at least
        // two launches back, so it is complete before griddepcontrol.wait
        for (int i = tid; i < nw; i += NC) emw[i] = __ldcg(a.emitted + w0 + i);
    }
    pdl_wait();
    // RES: the residual rows this CTA updates, fetched now rather than in the epilogue
    float xold = 0.f;
    if (MODE == GEMV_RES && tid < nrows) xold = __ldcg(a.out + row0 + tid);

    if (a.input_mode) {
        // first kernel of the step: resolve the step's input vector
        const StepInput in{a.table, a.table_rows, a.vocab, a.S, a.embed_in, a.stage_tokens, a.stage_embeds,
                           a.emitted_w};
        step_input_slice<WT, NSEG>(in, a.st, K, rs, colbase, xr, misc_i, a.x_out, nullptr);
    } else {
        load_vec_smem(a.in, K, xin);
        named_sync(1, NC);
        smem_slice<WT, NSEG>(xin, colbase, xr);
    }

    if (MODE != GEMV_RES)
        rmsnorm_slice<WT, NSEG>(xr, gsm, K, rs, colbase, a.eps, misc,
                                (MODE == GEMV_HEAD && blockIdx.x == 0) ? a.y_out : nullptr);
    pdl_launch_dependents();

    // ---------------- stage loop
    uint32_t sidx = 0;
    const bool ok = gemv_consume<WT, NSEG>(R, sidx, nrows, rps, row_bytes, rs, colbase, xr, res);
    if (!ok && lane == 0) {
        atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
        misc_i[4] = 1;
    }
    named_sync(1, NC);
    if (misc_i[4]) {
        if (tid == 0) {
            // let copies still in flight land before the CTA's shared memory is released
            for (uint32_t s2 = sidx; s2 < (uint32_t)nstages && s2 < sidx + (uint32_t)a.nst; ++s2)
                (void)mbar_wait_bounded(&full[s2 % a.nst], (s2 / a.nst) & 1, 10000000ull);
        }
        if (MODE != GEMV_HEAD) return;
    }

    // ---------------- epilogue over all rows of the CTA
    if (MODE == GEMV_GU) {
        for (int i = tid; i < nrows / 2; i += NC) {
            float g = 0.f, u = 0.f;
            for (int j = 0; j < rs; ++j) {
                g += res[(2 * i) * rs + j];
                u += res[(2 * i + 1) * rs + j];
            }
            a.out[row0 / 2 + i] = g / (1.0f + expf(-g)) * u;
        }
    } else if (MODE == GEMV_QKV) {
        for (int r = tid; r < nrows; r += NC) {
            float v = 0.f;
            for (int j = 0; j < rs; ++j) v += res[r * rs + j];
            a.out[row0 + r] = v;
        }
    } else if (MODE == GEMV_RES) {
        if (tid < nrows) {
            float v = 0.f;
            for (int j = 0; j < rs; ++j) v += res[tid * rs + j];
            a.out[row0 + tid] = xold + v;
        }
    } else {  // GEMV_HEAD
        // greedy: per-thread, per-warp, per-CTA argmax.  Sampling (top-k > 0): the
        // CTA's final logits stay in res and the CTA's top-k candidates go out.
        const int sk = a.st->sample_k;
        float best_v = -INFINITY;
        int best_i = INT_MAX;
        for (int r = tid; r < nrows; r += NC) {
            float v = 0.f;
            for (int j = 0; j < rs; ++j) v += res[r * rs + j];
            const int row = row0 + r;
            if (a.out) a.out[row] = v;
            if (a.penalty != 1.0f && ((emw[(row >> 5) - w0] >> (row & 31)) & 1u))
                v = v > 0.f ? v / a.penalty : v * a.penalty;
            if (row == a.eos) v = -INFINITY;
            if (sk > 0) {
                res[r * rs] = v;
            } else if (arg_better(v, row, best_v, best_i)) {
                best_v = v;
                best_i = row;
            }
        }
        // sampling scratch over the ring, idle now: the CTA's candidates, the selection
        // scratch, then (last CTA) every CTA's candidates
        float *cv = reinterpret_cast<float *>(ring);
        int *ci = reinterpret_cast<int *>(cv + kMaxTopK);
        int *scr = ci + kMaxTopK;
        uint64_t *all_k = reinterpret_cast<uint64_t *>(scr + kTopkScratchWords);   // 8-byte aligned
        if (sk > 0) {
            named_sync(1, NC);
            block_topk(res, rs, nullptr, row0, nrows, sk, cv, ci, scr);
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
            const int prev = atomicAdd(a.counter, 1);
            misc_i[5] = (prev == (int)gridDim.x - 1);
        }
        named_sync(1, NC);
        // last CTA: publish the id, advance the position
        auto commit = [&](int id) {
            *a.counter = 0;
            if (a.commit) {
                DevState *st = a.st;
                st->out_id = id;
                const int n = st->n_gen;
                if (n < a.ids_cap) a.ids[n] = id;
                else atomicOr(&st->status, DEV_ERR_IDS_FULL);
                st->n_gen = n + 1;
                st->pos = st->pos + 1;
            }
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
    if (a.advance_pos && blockIdx.x == 0 && tid == 0) a.st->pos = a.st->pos + 1;
}

// =====================================================================================
// Attention over the cache.  Grid (kv group g, split s); the kAttnMaxSplits CTAs of a
// group form one thread-block cluster.  The split size is attn_chunk(L), a function
// of the attended length L only, so a bucket migration cannot change the partition.
// Prologue: QK-RMSNorm and RoPE of the group's q heads and of k, rounding of k and v
// to the cache type and, in the CTA whose split holds position p, the KV append.
// Body: scores, softmax and P.V of the split for every q head of the group (GQA: the
// group's K/V rows are read once for all of its q heads).  The splits are then merged
// through distributed shared memory (flash-decoding combine, splits in index order):
// CTA rank r of the cluster produces slice r of the group's outputs.
// =====================================================================================

template <typename KT, int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int HALF = HD / 2;
    const int G = a.qh / a.kvh;
    const int CM = a.chunk_max;
    KT *Ks = reinterpret_cast<KT *>(smem);
    KT *Vs = Ks + (size_t)CM * HD;
    float *qs = reinterpret_cast<float *>(Vs + (size_t)CM * HD);  // [G][HD]
    float *kn = qs + G * HD;                                       // [HD]
    float *vn = kn + HD;                                           // [HD]
    float *rc = vn + HD;                                           // [HALF] cos, [HALF] sin
    float *sc = rc + HD;                                           // [G][CM]
    float *po = sc + G * CM;                                       // [G][HD] split output (unnormalised)
    float *pm = po + G * HD;                                       // [G] split max
    float *pl = pm + G;                                            // [G] split exp-sum
    // mbarrier: 8-byte aligned, after the G split sums
    uint64_t *bar = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(pl + G) + 7) & ~uintptr_t(7));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x, s = blockIdx.y;
    // The position was advanced by the previous step's last kernel, at least two
    // launches back, so it is complete and visible before griddepcontrol.wait.
    const int p = a.st->pos;
    const int L = p + 1;
    const int C = attn_chunk(L);
    const int nsplit = attn_splits(L);
    const bool valid = p < a.S && C <= CM;
    const bool active = valid && s < nsplit;
    if (!valid && tid == 0 && s == 0 && g == 0) atomicOr(&a.st->status, DEV_ERR_BAD_POS);

    bool ok = true;
    if (active) {
        const int j0 = s * C;
        const int n = L - j0 < C ? L - j0 : C;
        const int n_old = (p - j0) < n ? (p - j0) : n;   // cached rows [j0, j0 + n_old)
        const size_t grp_off = (size_t)g * a.S * HD;
        const KT *kc = reinterpret_cast<const KT *>(a.kcache) + grp_off;
        const KT *vc = reinterpret_cast<const KT *>(a.vcache) + grp_off;
        if (tid == 0) {
            mbar_init(bar, 1);
            fence_barrier_init();
            const uint32_t bytes = (uint32_t)(n_old * HD * sizeof(KT));
            mbar_arrive_expect_tx(bar, 2 * bytes);
            if (bytes) {
                const uint64_t pol = policy_evict_first();
                bulk_copy_g2s(Ks, kc + (size_t)j0 * HD, bytes, bar, pol);
                bulk_copy_g2s(Vs, vc + (size_t)j0 * HD, bytes, bar, pol);
            }
        }
        // RoPE table rows of the rotary position (the cache position + delta, or per
        // stream from the staged prompt): constant data during the chain
        const int *stage = a.st->rope_staged ? a.rope_stage : nullptr;
        const int pr = p + a.st->rope_delta;
        for (int m = tid; m < HALF; m += kAttnThreads) {
            const size_t r = (size_t)rope_row(m, a.mrope_h, stage, a.rope_stride, p, pr, a.rope_rows);
            rc[m] = a.rope_cos[r * HALF + m];
            rc[HALF + m] = a.rope_sin[r * HALF + m];
        }
        pdl_wait();
        pdl_launch_dependents();
        const float *qsrc = a.qkv + (size_t)g * G * HD;
        const float *ksrc = a.qkv + (size_t)a.qh * HD + (size_t)g * HD;
        const float *vsrc = a.qkv + (size_t)(a.qh + a.kvh) * HD + (size_t)g * HD;
        for (int i = tid; i < G * HD; i += kAttnThreads) qs[i] = __ldcg(qsrc + i);
        for (int i = tid; i < HD; i += kAttnThreads) {
            kn[i] = __ldcg(ksrc + i);
            vn[i] = __ldcg(vsrc + i);
        }
        __syncthreads();
        qk_norm_rope<HD, kAttnThreads / 32>(qs, kn, G, a.q_gamma, a.k_gamma, a.eps, rc, 1);
        if (n_old < n) {
            // this split holds position p: append the new row (cache type) to the cache
            KT *kw = reinterpret_cast<KT *>(a.kcache) + grp_off + (size_t)p * HD;
            KT *vw = reinterpret_cast<KT *>(a.vcache) + grp_off + (size_t)p * HD;
            for (int i = tid; i < HD; i += kAttnThreads) {
                Elem<KT>::store(Ks + n_old * HD, i, kn[i]);
                Elem<KT>::store(Vs + n_old * HD, i, vn[i]);
                Elem<KT>::store(kw, i, kn[i]);
                Elem<KT>::store(vw, i, vn[i]);
            }
            fence_proxy_async_global();
        }
        const bool got = mbar_wait_bounded(bar, 0);
        if (__syncthreads_or(!got)) {
            if (tid == 0) {
                atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
                (void)mbar_wait_bounded(bar, 0, 10000000ull);
            }
            ok = false;
        }
        if (ok) attn_split<KT, HD, kAttnThreads / 32>(Ks, Vs, qs, G, n, CM, a.scale, sc, po, pm, pl, 1);
    } else {
        pdl_wait();
        pdl_launch_dependents();
    }
    if (!active || !ok) {
        for (int hh = tid; hh < G; hh += kAttnThreads) {
            pm[hh] = -INFINITY;
            pl[hh] = 0.f;
        }
    }

    // ---- merge the splits of group g across the cluster
    cluster_sync();
    if (valid) {
        const int per = G * HD / kAttnMaxSplits;
        for (int i = tid; i < per; i += kAttnThreads) {
            const int idx = s * per + i;
            const int hh = idx / HD;
            float m_t[kAttnMaxSplits], M = -INFINITY;
#pragma unroll
            for (int t = 0; t < kAttnMaxSplits; ++t) {
                m_t[t] = t < nsplit ? ld_cluster_f32(cluster_map(pm + hh, t)) : -INFINITY;
                M = fmaxf(M, m_t[t]);
            }
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int t = 0; t < kAttnMaxSplits; ++t) {
                if (t < nsplit) {
                    const float w = expf(m_t[t] - M);
                    num = fmaf(ld_cluster_f32(cluster_map(po + idx, t)), w, num);
                    den = fmaf(ld_cluster_f32(cluster_map(pl + hh, t)), w, den);
                }
            }
            a.out[(size_t)g * G * HD + idx] = num / den;
        }
    }
    cluster_sync();   // no CTA leaves while another may still read its shared memory
}

// =====================================================================================
// Bucket migration: copy rows [0, n_pos) of every [S, hd] segment (layer x K/V x group).
// =====================================================================================

__global__ void __launch_bounds__(256) kv_migrate_kernel(const uint8_t *src, int S_old, uint8_t *dst, int S_new,
                                                         size_t row_bytes, int n_pos) {
    const size_t seg = blockIdx.y;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + seg * (size_t)S_old * row_bytes);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst + seg * (size_t)S_new * row_bytes);
    const size_t n16 = (size_t)n_pos * row_bytes / 16;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        d4[i] = s4[i];
}

// cos/sin of p * theta^(-2m/hd), evaluated in fp64 and rounded to fp32.
__global__ void rope_table_kernel(float *cos_t, float *sin_t, int n_pos, int head_dim, double theta) {
    const int half = head_dim / 2;
    const int total = n_pos * half;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
        const int p = idx / half, m = idx % half;
        const double inv_freq = pow(theta, -2.0 * (double)m / (double)head_dim);
        const double ang = (double)p * inv_freq;
        cos_t[idx] = (float)cos(ang);
        sin_t[idx] = (float)sin(ang);
    }
}

__global__ void to_f32_kernel(const void *src, int bf16, float *dst, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        dst[i] = bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[i])
                      : reinterpret_cast<const float *>(src)[i];
}

// =====================================================================================
// Host launchers
// =====================================================================================

template <typename F>
static cudaError_t launch_ex(F kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             const void *argp) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? at : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[1] = {const_cast<void *>(argp)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args);
}

bool gemv_split(int K, bool bf16, int *nseg, int *rs) {
    const int segw = bf16 ? 256 : 128;
    if (K <= 0 || K % segw) return false;
    const int t = K / segw;
    for (int r = 1; r <= kConsumerWarps; r *= 2) {
        if (t % r == 0 && t / r <= 4) {
            *nseg = t / r;
            *rs = r;
            return true;
        }
    }
    return false;
}

size_t gemv_smem_bytes(int nst, int rows_max, int rs, int K) {
    return (size_t)nst * kSlotBytes + (size_t)nst * 16 + (size_t)rows_max * rs * 4 + 64 * 4 + 2 * (size_t)K * 4 +
           ((size_t)rows_max / 32 + 2) * 4;
}

typedef void (*GemvFn)(const GemvArgs);

template <typename WT, int MODE>
static GemvFn gemv_pick(int nseg) {
    switch (nseg) {
        case 1: return gemv_kernel<WT, 1, MODE>;
        case 2: return gemv_kernel<WT, 2, MODE>;
        case 3: return gemv_kernel<WT, 3, MODE>;
        case 4: return gemv_kernel<WT, 4, MODE>;
    }
    return nullptr;
}

template <typename WT>
static GemvFn gemv_pick_mode(int mode, int nseg) {
    switch (mode) {
        case GEMV_QKV: return gemv_pick<WT, GEMV_QKV>(nseg);
        case GEMV_RES: return gemv_pick<WT, GEMV_RES>(nseg);
        case GEMV_GU: return gemv_pick<WT, GEMV_GU>(nseg);
        case GEMV_HEAD: return gemv_pick<WT, GEMV_HEAD>(nseg);
    }
    return nullptr;
}

static GemvFn gemv_fn(int mode, bool bf16, int nseg) {
    return bf16 ? gemv_pick_mode<__nv_bfloat16>(mode, nseg) : gemv_pick_mode<float>(mode, nseg);
}

typedef void (*AttnFn)(const AttnArgs);
static AttnFn attn_fn(bool bf16, int hd) {
    if (bf16) return hd == 64 ? attn_decode_kernel<__nv_bfloat16, 64> : attn_decode_kernel<__nv_bfloat16, 128>;
    return hd == 64 ? attn_decode_kernel<float, 64> : attn_decode_kernel<float, 128>;
}

cudaError_t kernels_init() {
    const int max_smem = 220 * 1024;
    for (int bf = 0; bf < 2; ++bf)
        for (int mode = 0; mode < 4; ++mode)
            for (int ns = 1; ns <= 4; ++ns) {
                cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(gemv_fn(mode, bf, ns)),
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
                if (e != cudaSuccess) return e;
            }
    for (int bf = 0; bf < 2; ++bf)
        for (int hd = 64; hd <= 128; hd *= 2) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(attn_fn(bf, hd)),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_gemv(int mode, bool bf16, const GemvArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl) {
    int nseg = 0, rs = 0;
    if (!gemv_split(a.K, bf16, &nseg, &rs) || rs != a.rs) return cudaErrorInvalidValue;
    GemvFn f = gemv_fn(mode, bf16, nseg);
    if (!f) return cudaErrorInvalidValue;
    return launch_ex(f, dim3(grid), dim3(kGemvThreads), smem, s, pdl, &a);
}

size_t attention_smem_bytes(bool bf16, int hd, int group, int chunk_max) {
    const size_t es = bf16 ? 2 : 4;
    return 2 * (size_t)chunk_max * hd * es + (size_t)group * hd * 4 + 3 * (size_t)hd * 4 +
           (size_t)group * chunk_max * 4 + (size_t)group * hd * 4 + (2 * (size_t)group + 2) * 4 + 16;
}

cudaError_t launch_attention(bool bf16, int hd, const AttnArgs &a, cudaStream_t s, bool pdl) {
    AttnFn f = attn_fn(bf16, hd);
    const size_t smem = attention_smem_bytes(bf16, hd, a.qh / a.kvh, a.chunk_max);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.kvh, kAttnMaxSplits);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = kAttnMaxSplits;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    void *args[1] = {const_cast<AttnArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(f), args);
}

cudaError_t launch_kv_migrate(const void *src, int S_old, void *dst, int S_new, int n_segments, size_t row_bytes,
                              int n_pos, cudaStream_t s) {
    if (n_pos <= 0) return cudaSuccess;
    const size_t n16 = (size_t)n_pos * row_bytes / 16;
    int gx = (int)((n16 + 255) / 256);
    if (gx > 64) gx = 64;
    kv_migrate_kernel<<<dim3(gx, n_segments), 256, 0, s>>>(reinterpret_cast<const uint8_t *>(src), S_old,
                                                           reinterpret_cast<uint8_t *>(dst), S_new, row_bytes, n_pos);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(float *cos_t, float *sin_t, int n_pos, int head_dim, double theta, cudaStream_t s) {
    const int total = n_pos * (head_dim / 2);
    int blocks = (total + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    rope_table_kernel<<<blocks, 256, 0, s>>>(cos_t, sin_t, n_pos, head_dim, theta);
    return cudaGetLastError();
}

cudaError_t launch_to_f32(const void *src, bool bf16, float *dst, int n, cudaStream_t s) {
    int blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    to_f32_kernel<<<blocks, 256, 0, s>>>(src, bf16 ? 1 : 0, dst, n);
    return cudaGetLastError();
}

}  // namespace qd

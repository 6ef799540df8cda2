// Kernels of the batched multi-stream decode (B independent streams, one token each
// per step) other than the tensor-core GEMMs: attention over each stream's own cache
// and length, RMSNorm with the bf16 hi/lo split that feeds the GEMMs (and the embedding
// gather of the step's tokens), and the per-stream penalty + argmax.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation": QK-norm over head_dim, GQA, plain RoPE, repetition penalty, greedy
//    argmax, per stream.
//  - "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile: the stages of one step,
//    here run for every stream at once.
#include "decode_common.cuh"

namespace qd {

namespace {

// ---- attention: grid (kv group, split, stream); the splits of one (stream, group) are
// one 8-CTA cluster and merge through distributed shared memory.  Same prologue
// (QK-norm, RoPE, KV append), split body and merge as the single-stream kernel, with
// each stream's own position, cache and rows.
template <int HD>
__global__ void __launch_bounds__(kAttnThreads) batch_attn_kernel(const BatchAttnArgs a) {
    using KT = __nv_bfloat16;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int HALF = HD / 2;
    const int G = a.qh / a.kvh;
    const int CM = a.chunk_max;
    KT *Ks = reinterpret_cast<KT *>(smem);
    KT *Vs = Ks + (size_t)CM * HD;
    float *qs = reinterpret_cast<float *>(Vs + (size_t)CM * HD);  // [G][HD]
    float *kn = qs + G * HD;
    float *vn = kn + HD;
    float *rc = vn + HD;
    float *sc = rc + HD;                                           // [G][CM]
    float *po = sc + G * CM;
    float *pm = po + G * HD;
    float *pl = pm + G;
    uint64_t *bar = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(pl + G) + 7) & ~uintptr_t(7));

    const int tid = threadIdx.x;
    const int g = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int p = a.pos[b];
    const int L = p + 1;
    const int C = attn_chunk(L);
    const int nsplit = attn_splits(L);
    const bool valid = p >= 0 && p < a.S && C <= CM;
    const bool active = valid && s < nsplit;
    if (!valid && tid == 0 && s == 0 && g == 0) atomicOr(a.status, DEV_ERR_BAD_POS);

    KT *kbase = reinterpret_cast<KT *>(a.kv) + (size_t)b * a.stream_elems + a.layer_elems;
    KT *vbase = kbase + (size_t)a.kvh * a.S * HD;
    const float *row = a.qkv + (size_t)b * a.qkv_ld;

    bool ok = true;
    if (active) {
        const int j0 = s * C;
        const int n = L - j0 < C ? L - j0 : C;
        const int n_old = (p - j0) < n ? (p - j0) : n;
        const size_t grp_off = (size_t)g * a.S * HD;
        const KT *kc = kbase + grp_off;
        const KT *vc = vbase + grp_off;
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
        for (int m = tid; m < HALF; m += kAttnThreads) {
            rc[m] = a.rope_cos[(size_t)p * HALF + m];
            rc[HALF + m] = a.rope_sin[(size_t)p * HALF + m];
        }
        const float *qsrc = row + (size_t)g * G * HD;
        const float *ksrc = row + (size_t)a.qh * HD + (size_t)g * HD;
        const float *vsrc = row + (size_t)(a.qh + a.kvh) * HD + (size_t)g * HD;
        for (int i = tid; i < G * HD; i += kAttnThreads) qs[i] = __ldcg(qsrc + i);
        for (int i = tid; i < HD; i += kAttnThreads) {
            kn[i] = __ldcg(ksrc + i);
            vn[i] = __ldcg(vsrc + i);
        }
        __syncthreads();
        qk_norm_rope<HD, kAttnThreads / 32>(qs, kn, G, a.q_gamma, a.k_gamma, a.eps, rc, 1);
        if (n_old < n) {
            KT *kw = kbase + grp_off + (size_t)p * HD;
            KT *vw = vbase + grp_off + (size_t)p * HD;
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
                atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
                (void)mbar_wait_bounded(bar, 0, 10000000ull);
            }
            ok = false;
        }
        if (ok) attn_split<KT, HD, kAttnThreads / 32>(Ks, Vs, qs, G, n, CM, a.scale, sc, po, pm, pl, 1);
    }
    if (!active || !ok) {
        for (int hh = tid; hh < G; hh += kAttnThreads) {
            pm[hh] = -INFINITY;
            pl[hh] = 0.f;
        }
    }

    cluster_sync();
    if (valid) {
        const int per = G * HD / kAttnMaxSplits;
        const size_t obase = (size_t)b * a.qh * HD + (size_t)g * G * HD;
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
            const float o = num / den;
            const __nv_bfloat16 h = __float2bfloat16_rn(o);
            a.out_hi[obase + idx] = h;
            a.out_lo[obase + idx] = __float2bfloat16_rn(o - __bfloat162float(h));
        }
    }
    cluster_sync();
}

// ---- RMSNorm + hi/lo split, one CTA per row (optional embedding gather first)
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) norm_split_kernel(const NormSplitArgs a) {
    __shared__ float red[kRowThreads / 32];
    __shared__ int sh_tok;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *x = a.x + (size_t)b * a.K;
    if (a.table) {
        if (tid == 0) {
            int t = a.tokens[b];
            if (t < 0 || t >= a.table_rows) {
                atomicOr(a.status, DEV_ERR_BAD_TOKEN);
                t = -1;
            } else if (t < a.vocab) {
                a.emitted[(size_t)b * a.emitted_words + (t >> 5)] |= 1u << (t & 31);
            }
            sh_tok = t;
        }
        __syncthreads();
        const int t = sh_tok;
        const __nv_bfloat16 *row = reinterpret_cast<const __nv_bfloat16 *>(a.table) + (size_t)(t < 0 ? 0 : t) * a.K;
        for (int i = tid; i < a.K; i += kRowThreads) x[i] = t < 0 ? 0.f : __bfloat162float(row[i]);
        __syncthreads();
    }
    float ss = 0.f;
    for (int i = tid; i < a.K; i += kRowThreads) ss = fmaf(x[i], x[i], ss);
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kRowThreads / 32; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)a.K + a.eps);
    for (int i = tid; i < a.K; i += kRowThreads) {
        const float v = x[i] * inv * a.gamma[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        a.hi[(size_t)b * a.K + i] = h;
        a.lo[(size_t)b * a.K + i] = __float2bfloat16_rn(v - __bfloat162float(h));
        if (a.y) a.y[(size_t)b * a.K + i] = v;
    }
}

// ---- per-stream penalty + EOS mask + argmax; the last CTA of the step advances the
// control block's step index
__global__ void __launch_bounds__(kRowThreads) batch_argmax_kernel(const BatchArgmaxArgs a) {
    __shared__ float bv_s[kRowThreads / 32];
    __shared__ int bi_s[kRowThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *lg = a.logits + (size_t)b * a.V;
    const uint32_t *em = a.emitted + (size_t)b * a.words;
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    for (int i = tid; i < a.V; i += kRowThreads) {
        float v = lg[i];
        if (a.penalty != 1.0f && ((em[i >> 5] >> (i & 31)) & 1u)) v = v > 0.f ? v / a.penalty : v * a.penalty;
        if (i == a.eos) v = -INFINITY;
        if (arg_better(v, i, best_v, best_i)) {
            best_v = v;
            best_i = i;
        }
    }
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
        bv_s[warp] = best_v;
        bi_s[warp] = best_i;
    }
    __syncthreads();
    if (tid == 0) {
        float bv = bv_s[0];
        int bi = bi_s[0];
        for (int w = 1; w < kRowThreads / 32; ++w)
            if (arg_better(bv_s[w], bi_s[w], bv, bi)) {
                bv = bv_s[w];
                bi = bi_s[w];
            }
        BatchCtl *c = a.ctl;
        const int step = c->step;
        const int B = gridDim.x;
        if (step >= 0 && step < c->n_steps) {
            c->ids[(size_t)step * B + b] = bi;
            a.tokens[b] = c->force ? c->force[(size_t)step * B + b] : bi;
        } else {
            atomicOr(a.status, DEV_ERR_IDS_FULL);
        }
        a.pos[b] = a.pos[b] + 1;
        __threadfence();
        if (atomicAdd(&c->done, 1) == B - 1) {
            c->done = 0;
            c->step = step + 1;
        }
    }
}

}  // namespace

size_t batch_attention_smem_bytes(int hd, int group, int chunk_max) {
    return 2 * (size_t)chunk_max * hd * 2 + (size_t)group * hd * 4 + 3 * (size_t)hd * 4 +
           (size_t)group * chunk_max * 4 + (size_t)group * hd * 4 + (2 * (size_t)group + 2) * 4 + 16;
}

cudaError_t batch_kernels_init() {
    for (const void *fn : {reinterpret_cast<const void *>(batch_attn_kernel<128>),
                           reinterpret_cast<const void *>(batch_attn_kernel<64>)}) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_batch_attention(int hd, int B, const BatchAttnArgs &a, cudaStream_t s) {
    const size_t smem = batch_attention_smem_bytes(hd, a.qh / a.kvh, a.chunk_max);
    const void *fn = hd == 128 ? reinterpret_cast<const void *>(batch_attn_kernel<128>)
                               : reinterpret_cast<const void *>(batch_attn_kernel<64>);
    if (smem > 160 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.kvh, kAttnMaxSplits, B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = kAttnMaxSplits;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void *args[1] = {const_cast<BatchAttnArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_norm_split(const NormSplitArgs &a, int rows, cudaStream_t s) {
    norm_split_kernel<<<rows, kRowThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_batch_argmax(const BatchArgmaxArgs &a, int B, cudaStream_t s) {
    batch_argmax_kernel<<<B, kRowThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qd

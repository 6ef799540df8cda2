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
//    migration copies the valid region of every layer's K and V.
#include <float.h>
#include <limits.h>

#include "qd_device.cuh"
#include "qd_internal.h"

namespace qd {

// =====================================================================================
// GEMV: out[r] = W[r, :] . v  with v = RMSNorm(in) (QKV, GU, HEAD) or v = in (RES).
//
// Each CTA owns a contiguous block of rows.  Thread 0 streams that block through a
// ring of `nst` stages of kStageRows rows with cp.async.bulk; the copies for the
// first stages are issued before griddepcontrol.wait, since weights never depend on
// the previous kernel.  A row is reduced by `rs` warps; each lane keeps its slice of
// v in registers (NSEG segments of 16 bytes of weights per lane).  Row sums are
// combined in a fixed order, so results are bitwise reproducible.
// =====================================================================================

__device__ __forceinline__ bool arg_better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <typename WT, int NSEG, int MODE>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int EPL = Elem<WT>::kPer16B;   // elements per lane per 16 bytes
    constexpr int SEGW = 32 * EPL;           // elements per warp segment
    const int K = a.K;
    const uint32_t row_bytes = (uint32_t)K * (uint32_t)sizeof(WT);
    const uint32_t stage_bytes = kStageRows * row_bytes;
    uint8_t *ring = smem;
    float *xs = reinterpret_cast<float *>(smem + (size_t)a.nst * stage_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(xs + K);
    float *red = reinterpret_cast<float *>(bars + a.nst);   // [2][8 rows][8 parts]
    float *misc = red + 128;                                 // [32]
    int *misc_i = reinterpret_cast<int *>(misc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = a.rows / a.unit;
    const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
    const int row0 = u0 * a.unit;
    const int nrows = (u1 - u0) * a.unit;
    const int nstages = (nrows + kStageRows - 1) / kStageRows;
    const WT *W = MODE == GEMV_HEAD ? reinterpret_cast<const WT *>(a.W_table[a.st->head_idx])
                                    : reinterpret_cast<const WT *>(a.W);
    const uint8_t *Wb = reinterpret_cast<const uint8_t *>(W) + (size_t)row0 * row_bytes;

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        const uint64_t pol = a.evict_last ? policy_evict_last() : policy_evict_first();
        const int pre = nstages < a.nst ? nstages : a.nst;
        for (int s = 0; s < pre; ++s) {
            const int r = s * kStageRows;
            const int n = nrows - r < kStageRows ? nrows - r : kStageRows;
            mbar_arrive_expect_tx(&bars[s], n * row_bytes);
            bulk_copy_g2s(ring + (size_t)s * stage_bytes, Wb + (size_t)r * row_bytes, n * row_bytes, &bars[s], pol);
        }
    }

    // ---- activations: wait for the producer kernel
    pdl_wait();
    if (MODE == GEMV_RES) {
        for (int i = tid; i < K; i += kGemvThreads) xs[i] = a.in[i];
    } else {
        float ss = 0.f;
        for (int i = tid; i < K; i += kGemvThreads) {
            const float v = a.in[i];
            xs[i] = v;
            ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) misc[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kGemvThreads / 32; ++w) tot += misc[w];
        const float inv = 1.0f / sqrtf(tot / (float)K + a.eps);
        const bool wy = (MODE == GEMV_HEAD) && blockIdx.x == 0 && a.y_out != nullptr;
        for (int i = tid; i < K; i += kGemvThreads) {
            const float v = xs[i] * inv * a.gamma[i];
            xs[i] = v;
            if (wy) a.y_out[i] = v;
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    const int rs = a.rs;
    const int sub = warp % rs;
    const int rr = warp / rs;
    const int rows_per_pass = (kGemvThreads / 32) / rs;
    const int colbase = sub * (K / rs);
    float xr[NSEG * EPL];
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg) {
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(xs + colbase + sg * SEGW + lane * EPL + e);
            xr[sg * EPL + e + 0] = v4.x;
            xr[sg * EPL + e + 1] = v4.y;
            xr[sg * EPL + e + 2] = v4.z;
            xr[sg * EPL + e + 3] = v4.w;
        }
    }

    float best_v = -INFINITY;
    int best_i = INT_MAX;
    bool failed = false;
    int s = 0;
    for (; s < nstages; ++s) {
        const int slot = s % a.nst;
        const bool ok = mbar_wait_bounded(&bars[slot], (uint32_t)((s / a.nst) & 1));
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        const uint8_t *sbase = ring + (size_t)slot * stage_bytes;
        const int rbase = s * kStageRows;
        const int nr = nrows - rbase < kStageRows ? nrows - rbase : kStageRows;
        float *redb = red + (s & 1) * 64;
        for (int ps = 0; ps < rs; ++ps) {
            const int r = ps * rows_per_pass + rr;
            if (r < nr) {
                const WT *wrow = reinterpret_cast<const WT *>(sbase + (size_t)r * row_bytes) + colbase;
                float acc = 0.f;
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(wrow + sg * SEGW + lane * EPL);
                    float f[EPL];
                    Elem<WT>::unpack(u, f);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(f[e], xr[sg * EPL + e], acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) redb[r * 8 + sub] = acc;
            }
        }
        __syncthreads();  // slot consumed, partial sums complete
        if (tid == 0 && s + a.nst < nstages) {
            const int s2 = s + a.nst;
            const int r = s2 * kStageRows;
            const int n = nrows - r < kStageRows ? nrows - r : kStageRows;
            const uint64_t pol = a.evict_last ? policy_evict_last() : policy_evict_first();
            mbar_arrive_expect_tx(&bars[slot], n * row_bytes);
            bulk_copy_g2s(ring + (size_t)slot * stage_bytes, Wb + (size_t)r * row_bytes, n * row_bytes, &bars[slot],
                          pol);
        }
        if (MODE == GEMV_GU) {
            if (tid < nr / 2) {
                float g = 0.f, u = 0.f;
                for (int j = 0; j < rs; ++j) {
                    g += redb[(2 * tid) * 8 + j];
                    u += redb[(2 * tid + 1) * 8 + j];
                }
                const float sg = g / (1.0f + expf(-g));
                a.out[(row0 + rbase) / 2 + tid] = sg * u;
            }
        } else if (tid < nr) {
            float v = 0.f;
            for (int j = 0; j < rs; ++j) v += redb[tid * 8 + j];
            const int row = row0 + rbase + tid;
            if (MODE == GEMV_QKV) {
                a.out[row] = v;
            } else if (MODE == GEMV_RES) {
                a.out[row] += v;
            } else {  // GEMV_HEAD
                if (a.out) a.out[row] = v;
                if (a.penalty != 1.0f && ((a.emitted[row >> 5] >> (row & 31)) & 1u))
                    v = v > 0.f ? v / a.penalty : v * a.penalty;
                if (row == a.eos) v = -INFINITY;
                if (arg_better(v, row, best_v, best_i)) {
                    best_v = v;
                    best_i = row;
                }
            }
        }
    }

    if (failed) {
        if (tid == 0) {
            atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
            // let copies still in flight land before the CTA's shared memory is released
            for (int s2 = s; s2 < nstages && s2 < s + a.nst; ++s2)
                (void)mbar_wait_bounded(&bars[s2 % a.nst], (uint32_t)((s2 / a.nst) & 1));
        }
        __syncthreads();
        if (MODE != GEMV_HEAD) return;
    }

    if (MODE == GEMV_HEAD) {
        // CTA argmax over its rows (threads 0..7 hold the candidates)
        if (warp == 0) {
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
                a.part_v[blockIdx.x] = best_v;
                a.part_i[blockIdx.x] = best_i;
                __threadfence();
                const int prev = atomicAdd(a.counter, 1);
                misc_i[0] = (prev == (int)gridDim.x - 1);
            }
        }
        __syncthreads();
        if (misc_i[0] && warp == 0) {
            // last CTA: reduce the per-CTA candidates
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
            if (lane == 0) {
                *a.counter = 0;
                if (a.commit) {
                    DevState *st = a.st;
                    st->out_id = bi;
                    const int n = st->n_gen;
                    if (n < a.ids_cap) a.ids[n] = bi;
                    else atomicOr(&st->status, DEV_ERR_IDS_FULL);
                    st->n_gen = n + 1;
                }
            }
        }
    }
}

// =====================================================================================
// Attention over the cache, one CTA per (kv group g, split s of kAttnChunk positions).
// Prologue: QK-RMSNorm and RoPE of the group's q heads and of k, rounding of k and v
// to the cache type and, in the CTA whose split holds position p, the KV append.
// Body: scores, softmax and P.V of the split for every q head of the group (GQA: the
// group's K/V rows are read once for all of its q heads).  The last CTA of a group to
// finish merges the splits in split order (flash-decoding combine), so the result
// does not depend on which CTA finishes last, nor on Smax.
// =====================================================================================

template <typename KT, int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int C = kAttnChunk;
    constexpr int HALF = HD / 2;
    const int G = a.qh / a.kvh;
    KT *Ks = reinterpret_cast<KT *>(smem);
    KT *Vs = Ks + C * HD;
    float *qs = reinterpret_cast<float *>(Vs + C * HD);  // [G][HD]
    float *kn = qs + G * HD;                             // [HD]
    float *vn = kn + HD;                                 // [HD]
    float *sc = vn + HD;                                 // [G][C]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sc + G * C);
    int *flag = reinterpret_cast<int *>(bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x, s = blockIdx.y;
    // The step's position was claimed by the first kernel of the step, at least two
    // launches back, so it is complete and visible before griddepcontrol.wait.
    const int p = a.st->cur;
    const int L = p + 1;
    const int nsplit = (L + C - 1) / C;
    if (s >= nsplit) return;
    if (p >= a.S) {
        if (tid == 0 && s == 0 && g == 0) atomicOr(&a.st->status, DEV_ERR_BAD_POS);
        return;
    }
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

    pdl_wait();
    const float *qsrc = a.qkv + (size_t)g * G * HD;
    const float *ksrc = a.qkv + (size_t)a.qh * HD + (size_t)g * HD;
    const float *vsrc = a.qkv + (size_t)(a.qh + a.kvh) * HD + (size_t)g * HD;
    for (int i = tid; i < G * HD; i += kAttnThreads) qs[i] = qsrc[i];
    for (int i = tid; i < HD; i += kAttnThreads) {
        kn[i] = ksrc[i];
        vn[i] = vsrc[i];
    }
    __syncthreads();
    if (a.q_gamma) {
        // QK-norm: RMSNorm over head_dim of each q head and of k (one warp per vector)
        for (int hh = warp; hh <= G; hh += kAttnThreads / 32) {
            float *v = hh < G ? qs + hh * HD : kn;
            const float *gam = hh < G ? a.q_gamma : a.k_gamma;
            float ss = 0.f;
            for (int i = lane; i < HD; i += 32) ss = fmaf(v[i], v[i], ss);
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
            for (int i = lane; i < HD; i += 32) v[i] = v[i] * inv * gam[i];
        }
        __syncthreads();
    }
    // RoPE at position p: pairs (m, m + HD/2)
    {
        const float *cs = a.rope_cos + (size_t)p * HALF;
        const float *sn = a.rope_sin + (size_t)p * HALF;
        for (int idx = tid; idx < (G + 1) * HALF; idx += kAttnThreads) {
            const int hh = idx / HALF, m = idx % HALF;
            float *v = hh < G ? qs + hh * HD : kn;
            const float c = cs[m], si = sn[m];
            const float x0 = v[m], x1 = v[m + HALF];
            v[m] = x0 * c - x1 * si;
            v[m + HALF] = x1 * c + x0 * si;
        }
    }
    __syncthreads();
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
    pdl_launch_dependents();
    const bool ok = mbar_wait_bounded(bar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
            (void)mbar_wait_bounded(bar, 0);
        }
        return;
    }

    // scores: warp per position, lanes over head_dim
    constexpr int DPL = HD / 32;
    for (int j = warp; j < n; j += kAttnThreads / 32) {
        float kr[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) kr[e] = Elem<KT>::load(Ks + j * HD, lane * DPL + e);
        for (int hh = 0; hh < G; ++hh) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) d = fmaf(qs[hh * HD + lane * DPL + e], kr[e], d);
            d = warp_sum(d);
            if (lane == 0) sc[hh * C + j] = d * a.scale;
        }
    }
    __syncthreads();
    float *part_base = a.part;
    const int stride = HD + 2;
    for (int hh = warp; hh < G; hh += kAttnThreads / 32) {
        const float v = lane < n ? sc[hh * C + lane] : -INFINITY;
        const float mx = warp_max(v);
        const float e = lane < n ? expf(v - mx) : 0.f;
        const float l = warp_sum(e);
        if (lane < n) sc[hh * C + lane] = e;
        if (lane == 0) {
            float *pp = part_base + ((size_t)(g * G + hh) * a.max_splits + s) * stride;
            pp[HD] = mx;
            pp[HD + 1] = l;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * HD; idx += kAttnThreads) {
        const int hh = idx / HD, d = idx % HD;
        float o = 0.f;
        for (int j = 0; j < n; ++j) o = fmaf(sc[hh * C + j], Elem<KT>::load(Vs + j * HD, d), o);
        part_base[((size_t)(g * G + hh) * a.max_splits + s) * stride + d] = o;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&a.counter[g], 1);
        *flag = (prev == nsplit - 1);
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    for (int idx = tid; idx < G * HD; idx += kAttnThreads) {
        const int hh = idx / HD, d = idx % HD;
        const float *base = part_base + (size_t)(g * G + hh) * a.max_splits * stride;
        float M = -INFINITY;
        for (int t = 0; t < nsplit; ++t) M = fmaxf(M, __ldcg(base + (size_t)t * stride + HD));
        float num = 0.f, den = 0.f;
        for (int t = 0; t < nsplit; ++t) {
            const float w = expf(__ldcg(base + (size_t)t * stride + HD) - M);
            num = fmaf(__ldcg(base + (size_t)t * stride + d), w, num);
            den = fmaf(__ldcg(base + (size_t)t * stride + HD + 1), w, den);
        }
        a.out[(size_t)(g * G + hh) * HD + d] = num / den;
    }
    if (tid == 0) a.counter[g] = 0;
}

// =====================================================================================
// Step input: claim the position, pick the token or embedding, record the emitted id.
// =====================================================================================

__global__ void __launch_bounds__(256) embed_kernel(const EmbedArgs a) {
    __shared__ int s_tok, s_mode, s_cur, s_bad;
    pdl_wait();
    if (threadIdx.x == 0) {
        DevState *st = a.st;
        const int cur = st->pos;
        st->cur = cur;
        st->pos = cur + 1;
        const int mode = st->in_mode;
        int tok = st->token_in;
        if (mode == IN_FEEDBACK) tok = st->out_id;
        else if (mode == IN_STAGED_TOKENS) tok = cur < a.S ? a.stage_tokens[cur] : -1;
        else if (mode == IN_STAGED_EMBEDS) tok = -1;
        int bad = 0;
        if (cur >= a.S) {
            // never index the staged inputs outside the bucket
            bad = 1;
            atomicOr(&st->status, DEV_ERR_BAD_POS);
        }
        const bool needs_row = (mode == IN_TOKEN || mode == IN_FEEDBACK || mode == IN_STAGED_TOKENS);
        if (!bad && needs_row && (tok < 0 || tok >= a.rows || a.table == nullptr)) {
            bad = 1;
            atomicOr(&st->status, DEV_ERR_BAD_TOKEN);
        }
        if (st->add_emitted && tok >= 0 && tok < a.vocab) a.emitted[tok >> 5] |= 1u << (tok & 31);
        s_tok = tok;
        s_mode = mode;
        s_cur = cur;
        s_bad = bad;
    }
    __syncthreads();
    const int mode = s_mode, tok = s_tok;
    for (int i = threadIdx.x; i < a.hidden; i += blockDim.x) {
        float v;
        if (s_bad) v = 0.f;
        else if (mode == IN_EMBED) v = a.embed_in[i];
        else if (mode == IN_STAGED_EMBEDS) v = a.stage_embeds[(size_t)s_cur * a.hidden + i];
        else if (a.bf16) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.table)[(size_t)tok * a.hidden + i]);
        else v = reinterpret_cast<const float *>(a.table)[(size_t)tok * a.hidden + i];
        a.x[i] = v;
    }
    pdl_launch_dependents();
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
    for (int r = 1; r <= 8; r *= 2) {
        if (t % r == 0 && t / r <= 4) {
            *nseg = t / r;
            *rs = r;
            return true;
        }
    }
    return false;
}

size_t gemv_smem_bytes(int K, bool bf16, int nst) {
    const size_t row = (size_t)K * (bf16 ? 2 : 4);
    return (size_t)nst * kStageRows * row + (size_t)K * 4 + (size_t)nst * 8 + 128 * 4 + 32 * 4;
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
    const int max_smem = 200 * 1024;
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
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
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

size_t attention_smem_bytes(bool bf16, int hd, int group) {
    const size_t es = bf16 ? 2 : 4;
    return 2 * (size_t)kAttnChunk * hd * es + (size_t)group * hd * 4 + 2 * (size_t)hd * 4 +
           (size_t)group * kAttnChunk * 4 + 16 + 16;
}

cudaError_t launch_attention(bool bf16, int hd, const AttnArgs &a, int max_splits, cudaStream_t s, bool pdl) {
    AttnFn f = attn_fn(bf16, hd);
    const size_t smem = attention_smem_bytes(bf16, hd, a.qh / a.kvh);
    return launch_ex(f, dim3(a.kvh, max_splits), dim3(kAttnThreads), smem, s, pdl, &a);
}

cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t s, bool pdl) {
    return launch_ex(embed_kernel, dim3(1), dim3(256), 0, s, pdl, &a);
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

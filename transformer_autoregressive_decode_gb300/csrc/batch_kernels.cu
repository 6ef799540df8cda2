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

// ---- attention: one CTA per (stream, kv group, chunk of 256 cached positions), 8
// consumer warps and a producer warp.  The producer streams the chunk's K rows, then
// its V rows, in 32-position tiles through a 6-slot shared-memory ring (1-D bulk
// copies; full/empty mbarriers per slot).  Consumer warp w owns rows 4w..4w+3 of every
// tile, so 32 rows of the chunk, one per lane: pass 1 computes their scores (4 rows x
// G heads reduced with one butterfly, then each score moved to its row's lane), a
// softmax over the warp's rows runs lane-parallel, pass 2 accumulates P.V.  The
// warps' partials (and, in the chunk that holds it, the new position, whose k and v
// are QK-normed, rotated, rounded to the cache type and appended) are combined into
// the chunk's (max, sum, output); the last chunk CTA of a (stream, group) to finish
// merges the chunks in order (flash-decoding merge) and writes the output.  Equal
// chunks keep the work balanced whatever the lengths; no CTA waits for another.  As a
// programmatic dependent of the QKV GEMM, the producer starts on the cached rows
// (written by earlier steps) before the consumers wait for the GEMM's q, k and v.
constexpr int kBattConsumers = 8;
constexpr int kBattThreads = (kBattConsumers + 1) * 32;
constexpr int kBattTile = 32;        // positions per ring slot
constexpr int kBattSlots = 6;
constexpr int kBattMaxGroup = 8;     // q heads per kv head
constexpr int kBattRowsPerWarp = kBattTile / kBattConsumers;   // 4
static_assert(kBattChunk / kBattTile * kBattRowsPerWarp == 32, "one chunk row per lane of each warp");

// Sums N per-lane values over the lanes of a warp with one butterfly: each halving
// step trades half of the values with the partner lane, so N values cost about N
// shuffles instead of 5 N.  Afterwards v[0] of lane l holds the total of value idx,
// where idx collects the halves lane l kept; lanes with (l & (32 / N - 1)) == 0 own
// the N distinct indices.
template <int N, int MASK> struct ReduceScatter {
    __device__ __forceinline__ static void run(float *v, int lane, int &idx) {
        if constexpr (N > 1 && MASK > 0) {
            const bool up = (lane & MASK) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = up ? v[i] : v[i + N / 2];
                const float keep = up ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
            }
            if (up) idx += N / 2;
            ReduceScatter<N / 2, MASK / 2>::run(v, lane, idx);
        } else if constexpr (MASK > 0) {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
            ReduceScatter<1, MASK / 2>::run(v, lane, idx);
        }
    }
};

// Row jj of a tile of bf16 rows of HD elements: this lane's DPL consecutive elements
// (zeros when the row is past the tile's end).
template <int DPL, int HD>
__device__ __forceinline__ void tile_row(const __nv_bfloat16 *tile, int jj, int lane, bool in, float *f) {
    if (!in) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) f[e] = 0.f;
        return;
    }
    if constexpr (DPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(tile + (size_t)jj * HD + lane * 4);
        f[0] = bf16lo(u.x);
        f[1] = bf16hi(u.x);
        f[2] = bf16lo(u.y);
        f[3] = bf16hi(u.y);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(tile + (size_t)jj * HD + lane * 2);
        f[0] = bf16lo(u);
        f[1] = bf16hi(u);
    }
}

// Owner lane of value i after ReduceScatter<N, 16>: the lane bits set by the halving
// steps that kept the upper half.
template <int N> __device__ __forceinline__ int scatter_owner(int i) {
    int lane = 0, mask = 16;
#pragma unroll
    for (int half = N / 2; half >= 1; half >>= 1, mask >>= 1)
        if (i & half) lane |= mask;
    return lane;
}

template <int HD, int G>
__global__ void __launch_bounds__(kBattThreads, G <= 2 ? 4 : 2) batch_attn_kernel(const BatchAttnArgs a) {
    using KT = __nv_bfloat16;
    constexpr int HALF = HD / 2;
    constexpr int DPL = HD / 32;                       // dimensions per lane
    constexpr uint32_t kTileBytes = kBattTile * HD * 2;
    constexpr int NV = kBattRowsPerWarp * G;           // scores of one warp per tile
    constexpr int RS = HD + 2;                         // partial record: output, max, sum
    static_assert(G >= 1 && G <= kBattMaxGroup && NV <= 32, "group size");
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;                                                    // [slots][tile]
    float *red = reinterpret_cast<float *>(ring);                            // [warps + 1][G][RS], after the ring
    float *qs = reinterpret_cast<float *>(ring + kBattSlots * kTileBytes);  // [G][HD]
    float *kn = qs + G * HD;                                                 // [HD]
    float *vn = kn + HD;                                                     // [HD]
    float *rc = vn + HD;                                                     // [HALF] cos, [HALF] sin
    uint64_t *full = reinterpret_cast<uint64_t *>(rc + HD);                  // [slots]
    uint64_t *empty = full + kBattSlots;                                     // [slots]
    int *flag = reinterpret_cast<int *>(empty + kBattSlots);                 // [0] abort, [1] last chunk

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pairs = gridDim.x / batch_attn_max_chunks(a.S);
    const int c = blockIdx.x / pairs;                  // chunk
    const int pair = blockIdx.x - c * pairs;           // (stream, kv group)
    const int b = pair / a.kvh, g = pair - b * a.kvh;
    const int p = a.pos[b];
    const bool valid = p >= 0 && p < a.S && a.qh == G * a.kvh;
    if (!valid) {
        if (tid == 0 && g == 0 && c == 0) atomicOr(a.status, DEV_ERR_BAD_POS);
        return;
    }
    const int nC = p / kBattChunk + 1;                 // chunks of [0, p], the last holds p
    if (c >= nC) return;
    const bool holds_new = c == nC - 1;
    const int j0 = c * kBattChunk;
    const int rows_c = (holds_new ? p : j0 + kBattChunk) - j0;   // cached rows of the chunk
    const int nT = (rows_c + kBattTile - 1) / kBattTile;
    const int total = 2 * nT;                          // K tiles, then V tiles
    const size_t grp_off = (size_t)g * a.S * HD;
    KT *kbase = reinterpret_cast<KT *>(a.kv) + (size_t)b * a.stream_elems + a.layer_elems + grp_off;
    KT *vbase = kbase + (size_t)a.kvh * a.S * HD;

    if (tid == 0) {
        for (int i = 0; i < kBattSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kBattConsumers);
        }
        flag[0] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kBattConsumers) {
        // ---- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (; issued < total; ++issued) {
                const int slot = issued % kBattSlots;
                if (issued >= kBattSlots &&
                    !mbar_wait_bounded(&empty[slot], (uint32_t)(issued / kBattSlots - 1) & 1u)) {
                    atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
                    *reinterpret_cast<volatile int *>(flag) = 1;
                    break;
                }
                const int i = issued < nT ? issued : issued - nT;
                const int rows = rows_c - i * kBattTile < kBattTile ? rows_c - i * kBattTile : kBattTile;
                const uint32_t bytes = (uint32_t)rows * HD * 2;
                mbar_arrive_expect_tx(&full[slot], bytes);
                bulk_copy_g2s(ring + (size_t)slot * kTileBytes,
                              (issued < nT ? kbase : vbase) + (size_t)(j0 + i * kBattTile) * HD, bytes, &full[slot],
                              pol);
            }
            // copies in flight land before the CTA can leave
            for (int k = 0; k < kBattSlots; ++k) {
                int last = -1;
                for (int t = k; t < issued; t += kBattSlots) last = t;
                if (last >= 0) (void)mbar_wait_bounded(&full[k], (uint32_t)(last / kBattSlots) & 1u, 10000000ull);
            }
        }
        return;
    }

    // ---- consumers: q (and k, v) of the new position, QK-norm and RoPE
    constexpr int NC = kBattConsumers * 32;
    pdl_wait();
    pdl_launch_dependents();
    const float *row = a.qkv + (size_t)b * a.qkv_ld;
    for (int m = tid; m < HALF; m += NC) {
        rc[m] = a.rope_cos[(size_t)p * HALF + m];
        rc[HALF + m] = a.rope_sin[(size_t)p * HALF + m];
    }
    for (int i = tid; i < G * HD; i += NC) qs[i] = __ldcg(row + (size_t)g * G * HD + i);
    for (int i = tid; i < HD; i += NC) {
        kn[i] = __ldcg(row + (size_t)a.qh * HD + (size_t)g * HD + i);
        vn[i] = __ldcg(row + (size_t)(a.qh + a.kvh) * HD + (size_t)g * HD + i);
    }
    named_sync(1, NC);
    qk_norm_rope<HD, kBattConsumers>(qs, kn, G, a.q_gamma, a.k_gamma, a.eps, rc, 1);
    if (holds_new) {
        for (int i = tid; i < HD; i += NC) {
            const KT kb = __float2bfloat16_rn(kn[i]), vb = __float2bfloat16_rn(vn[i]);
            kbase[(size_t)p * HD + i] = kb;
            vbase[(size_t)p * HD + i] = vb;
            kn[i] = __bfloat162float(kb);
            vn[i] = __bfloat162float(vb);
        }
        named_sync(1, NC);
    }
    float qr[G][DPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < DPL; ++e) qr[hh][e] = qs[hh * HD + lane * DPL + e];

    // pass 1: scores; lane l ends with the score of this warp's row l (tile l / 4,
    // row 4 * warp + l % 4 of that tile), -inf past the chunk's rows
    bool ok = true;
    float smine[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) smine[hh] = -INFINITY;
    for (int t = 0; t < nT; ++t) {
        const int slot = t % kBattSlots;
        if (!mbar_wait_bounded(&full[slot], (uint32_t)(t / kBattSlots) & 1u)) {
            ok = false;
            break;
        }
        const KT *tile = reinterpret_cast<const KT *>(ring + (size_t)slot * kTileBytes);
        const int rows = rows_c - t * kBattTile < kBattTile ? rows_c - t * kBattTile : kBattTile;
        float v[NV];
#pragma unroll
        for (int r = 0; r < kBattRowsPerWarp; ++r) {
            const int jj = warp * kBattRowsPerWarp + r;
            float kf[DPL];
            tile_row<DPL, HD>(tile, jj, lane, jj < rows, kf);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) d = fmaf(qr[hh][e], kf[e], d);
                v[r * G + hh] = d;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        int idx = 0;
        ReduceScatter<NV, 16>::run(v, lane, idx);
#pragma unroll
        for (int r = 0; r < kBattRowsPerWarp; ++r)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float x = __shfl_sync(0xffffffffu, v[0], scatter_owner<NV>(r * G + hh));
                if (lane == t * kBattRowsPerWarp + r && warp * kBattRowsPerWarp + r < rows) smine[hh] = x * a.scale;
            }
    }
    // softmax over this warp's rows, one per lane
    float pm_[G], pl_[G], pr[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const float mx = warp_max(smine[hh]);
        pr[hh] = mx == -INFINITY ? 0.f : expf(smine[hh] - mx);
        pm_[hh] = mx;
        pl_[hh] = warp_sum(pr[hh]);
    }
    // pass 2: P.V
    float acc[G][DPL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[hh][e] = 0.f;
    for (int t = nT; t < total && ok; ++t) {
        const int slot = t % kBattSlots;
        if (!mbar_wait_bounded(&full[slot], (uint32_t)(t / kBattSlots) & 1u)) {
            ok = false;
            break;
        }
        const KT *tile = reinterpret_cast<const KT *>(ring + (size_t)slot * kTileBytes);
        const int i = t - nT;
        const int rows = rows_c - i * kBattTile < kBattTile ? rows_c - i * kBattTile : kBattTile;
#pragma unroll
        for (int r = 0; r < kBattRowsPerWarp; ++r) {
            const int jj = warp * kBattRowsPerWarp + r;
            if (jj < rows) {
                float vf[DPL];
                tile_row<DPL, HD>(tile, jj, lane, true, vf);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float pj = __shfl_sync(0xffffffffu, pr[hh], i * kBattRowsPerWarp + r);
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[hh][e] = fmaf(pj, vf[e], acc[hh][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!ok) {
        if (lane == 0) atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
        *reinterpret_cast<volatile int *>(flag) = 1;
    }
    // combine the warps and the new position into the chunk's record (the ring is
    // idle once every tile was consumed)
    named_sync(1, NC);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float *rw = red + ((size_t)warp * G + hh) * RS;
#pragma unroll
        for (int e = 0; e < DPL; ++e) rw[lane * DPL + e] = acc[hh][e];
        if (lane == 0) {
            rw[HD] = pm_[hh];
            rw[HD + 1] = pl_[hh];
        }
    }
    const int nrec = holds_new ? kBattConsumers + 1 : kBattConsumers;
    if (holds_new && warp == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) d = fmaf(qr[hh][e], kn[lane * DPL + e], d);
            d = warp_sum(d) * a.scale;
            float *rw = red + ((size_t)kBattConsumers * G + hh) * RS;
            for (int i = lane; i < HD; i += 32) rw[i] = vn[i];
            if (lane == 0) {
                rw[HD] = d;
                rw[HD + 1] = 1.f;
            }
        }
    }
    named_sync(1, NC);
    const int nchunks_max = batch_attn_max_chunks(a.S);
    float *prec = a.partial + ((size_t)pair * nchunks_max + c) * G * RS;   // this chunk's record
    const size_t obase = (size_t)b * a.qh * HD + (size_t)g * G * HD;
    for (int idx = tid; idx < G * RS; idx += NC) {
        const int hh = idx / RS, d = idx - hh * RS;
        float M = -INFINITY;
        for (int w = 0; w < nrec; ++w) M = fmaxf(M, red[((size_t)w * G + hh) * RS + HD]);
        float val;
        if (d == HD) {
            val = M;
        } else {
            float acc2 = 0.f;
            for (int w = 0; w < nrec; ++w) {
                const float *rw = red + ((size_t)w * G + hh) * RS;
                const float wt = rw[HD] == -INFINITY ? 0.f : expf(rw[HD] - M);
                acc2 = fmaf(rw[d], wt, acc2);   // d == HD + 1: the sums
            }
            val = acc2;
        }
        if (nC == 1) {
            red[(size_t)(kBattConsumers + 1) * G * RS + idx] = val;   // single chunk: finish below
        } else {
            __stcg(prec + idx, val);
        }
    }
    if (nC == 1) {
        named_sync(1, NC);
        const float *fin = red + (size_t)(kBattConsumers + 1) * G * RS;
        for (int idx = tid; idx < G * HD; idx += NC) {
            const int hh = idx / HD, d = idx - hh * HD;
            const float o = fin[hh * RS + d] / fin[hh * RS + HD + 1];
            const __nv_bfloat16 h = __float2bfloat16_rn(o);
            a.out_hi[obase + idx] = h;
            a.out_lo[obase + idx] = __float2bfloat16_rn(o - __bfloat162float(h));
        }
        return;
    }
    // the last chunk of the pair to finish merges every chunk's record, in order
    __threadfence();
    named_sync(1, NC);
    if (tid == 0) {
        const int done = atomicAdd(&a.counter[pair], 1);
        flag[1] = done == nC - 1;
        if (done == nC - 1) a.counter[pair] = 0;
    }
    named_sync(1, NC);
    if (!flag[1]) return;
    __threadfence();
    const float *p0 = a.partial + (size_t)pair * nchunks_max * G * RS;
    for (int idx = tid; idx < G * HD; idx += NC) {
        const int hh = idx / HD, d = idx - hh * HD;
        float M = -INFINITY;
        for (int k = 0; k < nC; ++k) M = fmaxf(M, __ldcg(p0 + ((size_t)k * G + hh) * RS + HD));
        float num = 0.f, den = 0.f;
        for (int k = 0; k < nC; ++k) {
            const float *rk = p0 + ((size_t)k * G + hh) * RS;
            const float mk = __ldcg(rk + HD);
            const float wt = mk == -INFINITY ? 0.f : expf(mk - M);
            num = fmaf(__ldcg(rk + d), wt, num);
            den = fmaf(__ldcg(rk + HD + 1), wt, den);
        }
        const float o = num / den;
        const __nv_bfloat16 h = __float2bfloat16_rn(o);
        a.out_hi[obase + idx] = h;
        a.out_lo[obase + idx] = __float2bfloat16_rn(o - __bfloat162float(h));
    }
}

// ---- RMSNorm + hi/lo split, one CTA per row (optional embedding gather first)
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) norm_split_kernel(const NormSplitArgs a) {
    __shared__ float red[kRowThreads / 32];
    __shared__ int sh_tok;
    pdl_wait();
    pdl_launch_dependents();
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
static_assert(kRowThreads == kConsumerWarps * 32, "the block top-k selection runs on every thread of the CTA");

__global__ void __launch_bounds__(kRowThreads) batch_argmax_kernel(const BatchArgmaxArgs a) {
    __shared__ float bv_s[kRowThreads / 32];
    __shared__ int bi_s[kRowThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *lg = a.logits + (size_t)b * a.V;
    const uint32_t *em = a.emitted + (size_t)b * a.words;
    const int sk = a.samp->top_k;
    if (sk > 0) {
        // sampling: the stream's final logits in shared memory, its top-k candidates, one
        // draw (the same selection and draw as the single-stream head)
        extern __shared__ __align__(16) float sm_v[];
        float *cv = sm_v + a.V;
        int *ci = reinterpret_cast<int *>(cv + kMaxTopK);
        int *scr = ci + kMaxTopK;                 // 8-byte aligned: V + 2 kMaxTopK words before it
        for (int i = tid; i < a.V; i += kRowThreads) {
            float v = lg[i];
            if (a.penalty != 1.0f && ((em[i >> 5] >> (i & 31)) & 1u)) v = v > 0.f ? v / a.penalty : v * a.penalty;
            if (i == a.eos) v = -INFINITY;
            sm_v[i] = v;
        }
        named_sync(1, kRowThreads);
        block_topk(sm_v, 1, nullptr, 0, a.V, sk, cv, ci, scr);
        if (warp == 0) {
            const BatchSampling sp = *a.samp;
            const uint64_t seed = (((uint64_t)sp.seed_hi << 32) | sp.seed_lo) + (uint64_t)b;
            const int id = warp_sample(cv, ci, sk, sp.temperature, sp.top_p, uniform53(seed, (uint64_t)a.drawn[b]));
            if (lane == 0) {
                bi_s[0] = id;
                a.drawn[b] = a.drawn[b] + 1;
            }
        }
        __syncthreads();
    }
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    for (int i = tid; i < a.V && sk == 0; i += kRowThreads) {
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
    if (lane == 0 && sk == 0) {
        bv_s[warp] = best_v;
        bi_s[warp] = best_i;
    }
    __syncthreads();
    if (tid == 0) {
        float bv = bv_s[0];
        int bi = bi_s[0];
        for (int w = 1; w < kRowThreads / 32 && sk == 0; ++w)
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

typedef void (*BattFn)(const BatchAttnArgs);

BattFn batt_fn(int hd, int group) {
#define QD_BATT(HDV, GV) \
    if (hd == HDV && group == GV) return batch_attn_kernel<HDV, GV>;
    QD_BATT(128, 1) QD_BATT(128, 2) QD_BATT(128, 4) QD_BATT(128, 8)
    QD_BATT(64, 1) QD_BATT(64, 2) QD_BATT(64, 4) QD_BATT(64, 8)
#undef QD_BATT
    return nullptr;
}

}  // namespace

size_t batch_attention_smem_bytes(int hd, int group) {
    // ring (holds the records of the warps, the new position and the chunk at the
    // end), q heads, k, v, cos/sin, barriers, flags
    const size_t ring = (size_t)kBattSlots * kBattTile * hd * 2;
    const size_t red = (size_t)(kBattConsumers + 2) * group * (hd + 2) * 4;
    return (ring > red ? ring : red) + (size_t)group * hd * 4 + 3 * (size_t)hd * 4 + 2 * kBattSlots * 8 + 16;
}

bool batch_attention_supported(int hd, int group) { return batt_fn(hd, group) != nullptr; }

cudaError_t batch_kernels_init() {
    cudaError_t ea = cudaFuncSetAttribute(reinterpret_cast<const void *>(batch_argmax_kernel),
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)((size_t)kBatchSampleVocabMax * 4 + (2 * kMaxTopK + kTopkScratchWords) * 4));
    if (ea != cudaSuccess) return ea;
    for (int hd : {64, 128})
        for (int g : {1, 2, 4, 8}) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(batt_fn(hd, g)),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

// Launch `fn` with `args` on `s`, as a programmatic dependent of the previous kernel
// in the stream when `pdl` is set.
cudaError_t launch_ex(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void **args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_batch_attention(int hd, int B, const BatchAttnArgs &a, cudaStream_t s, bool pdl) {
    const size_t smem = batch_attention_smem_bytes(hd, a.qh / a.kvh);
    const BattFn fn = a.qh % a.kvh ? nullptr : batt_fn(hd, a.qh / a.kvh);
    if (!fn || smem > 160 * 1024 || !a.partial || !a.counter) return cudaErrorInvalidValue;
    // chunk-major order: every pair's first chunk, then every pair's second, ...
    void *args[1] = {const_cast<BatchAttnArgs *>(&a)};
    return launch_ex(reinterpret_cast<const void *>(fn), dim3(batch_attn_max_chunks(a.S) * B * a.kvh),
                     dim3(kBattThreads), smem, s, pdl, args);
}

cudaError_t launch_norm_split(const NormSplitArgs &a, int rows, cudaStream_t s, bool pdl) {
    void *args[1] = {const_cast<NormSplitArgs *>(&a)};
    return launch_ex(reinterpret_cast<const void *>(norm_split_kernel), dim3(rows), dim3(kRowThreads), 0, s, pdl,
                     args);
}

cudaError_t launch_batch_argmax(const BatchArgmaxArgs &a, int B, cudaStream_t s, bool pdl) {
    void *args[1] = {const_cast<BatchArgmaxArgs *>(&a)};
    // shared memory for the sampling branch (the greedy branch uses none of it)
    const size_t smem =
        a.V <= kBatchSampleVocabMax ? (size_t)a.V * 4 + (size_t)(2 * kMaxTopK + kTopkScratchWords) * 4 : 0;
    return launch_ex(reinterpret_cast<const void *>(batch_argmax_kernel), dim3(B), dim3(kRowThreads), smem, s, pdl,
                     args);
}

}  // namespace qd

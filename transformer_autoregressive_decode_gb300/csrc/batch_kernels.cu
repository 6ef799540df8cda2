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

// ---- attention: grid (kv group, split, stream); the splits of one (stream, group)
// form an 8-CTA cluster and merge through distributed shared memory (flash-decoding
// combine, splits in index order); a split holds batch_attn_chunk(L) = ceil(L / 8)
// positions, so all 8 CTAs of a cluster have work.  Each CTA streams its split's cached K rows, then its V rows,
// in 32-position tiles through a 4-slot shared-memory ring (1-D bulk copies, one
// mbarrier per slot), so several CTAs share an SM and one CTA's copies overlap the
// others' arithmetic.  The new position's k and v (QK-norm and RoPE applied, rounded
// to the cache type) are appended to the cache and enter the sums from shared memory.
// Scores: warp w takes rows w, w+8, ... of a tile, each lane 4 (or 2) dimensions of
// the row; P.V the same rows, each lane accumulating its dimensions, then the warps'
// partial outputs are summed.
constexpr int kBattThreads = 256;
constexpr int kBattWarps = kBattThreads / 32;
constexpr int kBattTile = 32;        // positions per ring slot
constexpr int kBattSlots = 4;
constexpr int kBattMaxGroup = 8;     // q heads per kv head
constexpr int kBattRowsPerWarp = kBattTile / kBattWarps;   // 4

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

template <int HD, int G>
__global__ void __launch_bounds__(kBattThreads, 4) batch_attn_kernel(const BatchAttnArgs a) {
    using KT = __nv_bfloat16;
    constexpr int HALF = HD / 2;
    constexpr int DPL = HD / 32;                       // dimensions per lane
    constexpr uint32_t kTileBytes = kBattTile * HD * 2;
    static_assert(G >= 1 && G <= kBattMaxGroup, "group size");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int CM = a.chunk_max;
    uint8_t *ring = smem;                                                    // [slots][tile]
    float *red = reinterpret_cast<float *>(ring);                            // [warps][G][HD], after the ring
    float *qs = reinterpret_cast<float *>(ring + kBattSlots * kTileBytes);  // [G][HD]
    float *kn = qs + G * HD;                                                 // [HD]
    float *vn = kn + HD;                                                     // [HD]
    float *rc = vn + HD;                                                     // [HALF] cos, [HALF] sin
    float *sc = rc + HD;                                                     // [G][CM]
    float *po = sc + G * CM;                                                 // [G][HD]
    float *pm = po + G * HD;                                                 // [G]
    float *pl = pm + G;                                                      // [G]
    uint64_t *full = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(pl + G) + 7) & ~uintptr_t(7));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int p = a.pos[b];
    const int L = p + 1;
    const int C = batch_attn_chunk(L);
    const int nsplit = batch_attn_splits(L);
    const bool valid = p >= 0 && p < a.S && C <= CM && a.qh == G * a.kvh;
    const bool active = valid && s < nsplit;
    if (!valid && tid == 0 && s == 0 && g == 0) atomicOr(a.status, DEV_ERR_BAD_POS);

    KT *kbase = reinterpret_cast<KT *>(a.kv) + (size_t)b * a.stream_elems + a.layer_elems;
    KT *vbase = kbase + (size_t)a.kvh * a.S * HD;
    const float *row = a.qkv + (size_t)b * a.qkv_ld;

    bool ok = true;
    if (active) {
        const int j0 = s * C;
        const int n = L - j0 < C ? L - j0 : C;
        const int n_old = (p - j0) < n ? (p - j0) : n;   // cached rows [j0, j0 + n_old)
        const int nT = (n_old + kBattTile - 1) / kBattTile;
        const int total = 2 * nT;                         // K tiles, then V tiles
        const size_t grp_off = (size_t)g * a.S * HD;
        const KT *kc = kbase + grp_off;
        const KT *vc = vbase + grp_off;
        int issued = 0;                                   // thread 0: tiles issued so far
        uint64_t pol = 0;
        auto issue = [&](int t) {
            const int slot = t % kBattSlots;
            const int i = t < nT ? t : t - nT;
            const int rows = n_old - i * kBattTile < kBattTile ? n_old - i * kBattTile : kBattTile;
            const KT *src = (t < nT ? kc : vc) + (size_t)(j0 + i * kBattTile) * HD;
            const uint32_t bytes = (uint32_t)rows * HD * 2;
            mbar_arrive_expect_tx(&full[slot], bytes);
            bulk_copy_g2s(ring + (size_t)slot * kTileBytes, src, bytes, &full[slot], pol);
        };
        if (tid == 0) {
            for (int i = 0; i < kBattSlots; ++i) mbar_init(&full[i], 1);
            fence_barrier_init();
            pol = policy_evict_first();
            for (; issued < total && issued < kBattSlots; ++issued) issue(issued);
        }
        for (int m = tid; m < HALF; m += kBattThreads) {
            rc[m] = a.rope_cos[(size_t)p * HALF + m];
            rc[HALF + m] = a.rope_sin[(size_t)p * HALF + m];
        }
        const float *qsrc = row + (size_t)g * G * HD;
        const float *ksrc = row + (size_t)a.qh * HD + (size_t)g * HD;
        const float *vsrc = row + (size_t)(a.qh + a.kvh) * HD + (size_t)g * HD;
        for (int i = tid; i < G * HD; i += kBattThreads) qs[i] = __ldcg(qsrc + i);
        for (int i = tid; i < HD; i += kBattThreads) {
            kn[i] = __ldcg(ksrc + i);
            vn[i] = __ldcg(vsrc + i);
        }
        __syncthreads();
        qk_norm_rope<HD, kBattWarps>(qs, kn, G, a.q_gamma, a.k_gamma, a.eps, rc, 1);
        if (n_old < n) {
            // this split holds position p: append the new row and use its cache value
            KT *kw = kbase + grp_off + (size_t)p * HD;
            KT *vw = vbase + grp_off + (size_t)p * HD;
            for (int i = tid; i < HD; i += kBattThreads) {
                const KT kb = __float2bfloat16_rn(kn[i]), vb = __float2bfloat16_rn(vn[i]);
                kw[i] = kb;
                vw[i] = vb;
                kn[i] = __bfloat162float(kb);
                vn[i] = __bfloat162float(vb);
            }
            fence_proxy_async_global();
        }
        __syncthreads();
        float qr[G][DPL];
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < DPL; ++e) qr[hh][e] = qs[hh * HD + lane * DPL + e];

        // pass 1: scores of the cached rows
        for (int t = 0; t < nT; ++t) {
            const int slot = t % kBattSlots;
            const bool got = mbar_wait_bounded(&full[slot], (uint32_t)(t / kBattSlots) & 1u);
            if (got) {
                const KT *tile = reinterpret_cast<const KT *>(ring + (size_t)slot * kTileBytes);
                const int rows = n_old - t * kBattTile < kBattTile ? n_old - t * kBattTile : kBattTile;
                // this warp's 4 rows x G heads, reduced together
                constexpr int NV = kBattRowsPerWarp * G;
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
                int idx = 0;
                ReduceScatter<NV, 16>::run(v, lane, idx);
                if ((lane & (32 / NV - 1)) == 0) {
                    const int r = idx / G, hh = idx - r * G;
                    const int jj = warp * kBattRowsPerWarp + r;
                    if (jj < rows) sc[hh * CM + t * kBattTile + jj] = v[0] * a.scale;
                }
            }
            if (__syncthreads_or(!got)) {
                ok = false;
                break;
            }
            if (tid == 0 && issued < total) {
                fence_proxy_async_smem();
                issue(issued++);
            }
        }
        if (ok && n_old < n && warp == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) d = fmaf(qr[hh][e], kn[lane * DPL + e], d);
                d = warp_sum(d);
                if (lane == 0) sc[hh * CM + n_old] = d * a.scale;
            }
        }
        __syncthreads();
        if (ok) {
            for (int hh = warp; hh < G; hh += kBattWarps) {
                float mx = -INFINITY;
                for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sc[hh * CM + j]);
                mx = warp_max(mx);
                float l = 0.f;
                for (int j = lane; j < n; j += 32) {
                    const float e = expf(sc[hh * CM + j] - mx);
                    sc[hh * CM + j] = e;
                    l += e;
                }
                l = warp_sum(l);
                if (lane == 0) {
                    pm[hh] = mx;
                    pl[hh] = l;
                }
            }
        }
        __syncthreads();

        // pass 2: P.V over the cached rows, then the new row
        float acc[G][DPL];
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[hh][e] = 0.f;
        for (int t = nT; t < total && ok; ++t) {
            const int slot = t % kBattSlots;
            const bool got = mbar_wait_bounded(&full[slot], (uint32_t)(t / kBattSlots) & 1u);
            if (got) {
                const KT *tile = reinterpret_cast<const KT *>(ring + (size_t)slot * kTileBytes);
                const int i = t - nT;
                const int rows = n_old - i * kBattTile < kBattTile ? n_old - i * kBattTile : kBattTile;
#pragma unroll
                for (int r = 0; r < kBattRowsPerWarp; ++r) {
                    const int jj = warp * kBattRowsPerWarp + r;
                    if (jj < rows) {
                        float vf[DPL];
                        tile_row<DPL, HD>(tile, jj, lane, true, vf);
                        const int j = i * kBattTile + jj;
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) {
                            const float pj = sc[hh * CM + j];
#pragma unroll
                            for (int e = 0; e < DPL; ++e) acc[hh][e] = fmaf(pj, vf[e], acc[hh][e]);
                        }
                    }
                }
            }
            if (__syncthreads_or(!got)) {
                ok = false;
                break;
            }
            if (tid == 0 && issued < total) {
                fence_proxy_async_smem();
                issue(issued++);
            }
        }
        if (ok && n_old < n && warp == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float pj = sc[hh * CM + n_old];
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[hh][e] = fmaf(pj, vn[lane * DPL + e], acc[hh][e]);
            }
        }
        if (!ok) {
            // let every copy issued land before the ring is reused or the CTA leaves
            if (tid == 0) {
                atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
                for (int k = 0; k < kBattSlots; ++k) {
                    int last = -1;
                    for (int t = 0; t < issued; ++t)
                        if (t % kBattSlots == k) last = t;
                    if (last >= 0) (void)mbar_wait_bounded(&full[k], (uint32_t)(last / kBattSlots) & 1u, 10000000ull);
                }
            }
            __syncthreads();
        } else {
            // the warps' partial outputs, summed through the (now idle) ring
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < DPL; ++e) red[((size_t)warp * G + hh) * HD + lane * DPL + e] = acc[hh][e];
            __syncthreads();
            for (int idx = tid; idx < G * HD; idx += kBattThreads) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kBattWarps; ++w) v += red[(size_t)w * G * HD + idx];
                po[idx] = v;
            }
        }
    }
    if (!active || !ok) {
        for (int i = tid; i < G * HD; i += kBattThreads) po[i] = 0.f;
        for (int hh = tid; hh < G; hh += kBattThreads) {
            pm[hh] = -INFINITY;
            pl[hh] = 0.f;
        }
    }

    cluster_sync();
    if (valid) {
        const int per = G * HD / kAttnMaxSplits;
        const size_t obase = (size_t)b * a.qh * HD + (size_t)g * G * HD;
        for (int i = tid; i < per; i += kBattThreads) {
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

size_t batch_attention_smem_bytes(int hd, int group, int chunk_max) {
    // ring, q heads, k, v, cos/sin, scores, split output, split max/sum, barriers
    return (size_t)kBattSlots * kBattTile * hd * 2 + (size_t)group * hd * 4 + 3 * (size_t)hd * 4 +
           (size_t)group * chunk_max * 4 + (size_t)group * hd * 4 + 2 * (size_t)group * 4 + 8 + kBattSlots * 8;
}

bool batch_attention_supported(int hd, int group) { return batt_fn(hd, group) != nullptr; }

cudaError_t batch_kernels_init() {
    for (int hd : {64, 128})
        for (int g : {1, 2, 4, 8}) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(batt_fn(hd, g)),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_batch_attention(int hd, int B, const BatchAttnArgs &a, cudaStream_t s) {
    const size_t smem = batch_attention_smem_bytes(hd, a.qh / a.kvh, a.chunk_max);
    const BattFn fn = a.qh % a.kvh ? nullptr : batt_fn(hd, a.qh / a.kvh);
    if (!fn || smem > 160 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.kvh, kAttnMaxSplits, B);
    cfg.blockDim = dim3(kBattThreads);
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
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fn), args);
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

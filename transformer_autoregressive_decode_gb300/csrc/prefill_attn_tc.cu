// Causal prefill attention on the tcgen05 tensor cores.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation": GQA attention over the prompt with QK-norm and RoPE applied before it.
//  - "audio.cpp Rockchip NPU build notes", section "What this path is not for": the
//    prompt's products are real dense contractions, where matrix units pay.
//
// One CTA per (prompt stream i, q head h, block of 128 queries), the blocks with the
// most keys first.  Per chunk c of 128 keys up to the block's last query:
//   S_c = Q K_c^T            tensor memory, fp32; M = the 128 queries, N = the keys,
//                            K = head_dim; Q as bf16 hi + lo parts (two MMAs per k-step)
//   softmax (8 warps)        S_c rows read back with tcgen05.ld: thread = query row,
//                            two warps per tensor-memory lane quarter with 64 keys each;
//                            causal mask, running max m and sum l per row, the chunk's
//                            probabilities P_c = exp(S - m) as bf16 hi + lo parts into
//                            shared memory in the MMA's K-major layout (128-byte swizzle)
//   O_c = P_c V_c            tensor memory; V straight from the cache tile as the
//                            MN-major B operand (N = head_dim contiguous, K = keys)
//   softmax warps            O <- O * exp(m_old - m_new) + O_c in registers (the chunk's
//                            products are formed fresh, so no rescaling in tensor memory)
// S and O have two tensor-memory buffers each (4 x 128 columns), so the MMAs of S_{c+1}
// run while the softmax warps work on S_c.  K and V tiles arrive by 3-D TMA from the
// cache [planes][S][head_dim] (box 64 x 128 keys; keys past the cache load as zeros,
// and the prompt's tail up to the next 128 is zeroed by the q/k kernel, so every V row
// an MMA reads is finite).
//
// Roles (352 threads): warp 0 lane 0 loads Q and the K tiles, warp 10 lane 0 the V
// tiles (each waits only for its own tile's last reader, so the next K tile streams in
// while the softmax warps work), warp 1 owns the tensor memory and lane 0 issues the
// MMAs, warps 2-9 run the softmax and the epilogue.  Every
// wait is bounded (role_wait); on expiry the kernel records DEV_ERR_WAIT_TIMEOUT, the
// roles stop, the MMAs and copies in flight are drained and the tensor memory is freed.
#include <cuda.h>

#include "mma_sync.cuh"
#include "qd_device.cuh"
#include "qd_internal.h"
#include "tc_common.cuh"

namespace qd {

namespace {

constexpr int kAtThreads = 352;
constexpr int kAtSoftWarps = 8;
constexpr int kAtRows = 128;                   // queries per CTA (MMA M)
constexpr int kAtKeys = 128;                   // keys per chunk
constexpr uint32_t kAtBox = 128 * 128;         // one 128-row x 128-byte swizzled box (16 KB)
constexpr unsigned long long kAtDrainNs = 20000000ull;

template <int HD> struct AtCfg {
    static constexpr int KB = HD / 64;                      // 64-wide head_dim blocks
    static constexpr uint32_t kQ = 0;                       // Q [part][KB] boxes
    static constexpr uint32_t kK = kQ + 2 * KB * kAtBox;    // K [KB]
    static constexpr uint32_t kV = kK + KB * kAtBox;        // V [KB] (64 head dims x 128 keys each)
    static constexpr uint32_t kP = kV + KB * kAtBox;        // P [part][2 key blocks]
    static constexpr uint32_t kRed = kP + 4 * kAtBox;       // row max [2][2][128], row sums [2][128]
    static constexpr uint32_t kBar = kRed + (4 + 2) * kAtRows * 4;
    static constexpr size_t kSmem = 1024 + kBar + 32 * 8 + 16;
};

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle: rows of
// 128 bytes along MN (64 bf16), 8-row groups along K `sbo` bytes apart, 64-element MN
// blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// N consecutive fp32 columns of this thread's tensor-memory lane: N / 16 loads, one wait.
template <int N> __device__ __forceinline__ void ld_cols(uint32_t taddr, float *v) {
    uint32_t r[N];
#pragma unroll
    for (int j = 0; j < N / 16; ++j) tc_ld16_nowait(taddr + 16u * j, r + 16 * j);
    tc_wait_ld_u32<N>(r);
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = __uint_as_float(r[e]);
}

// Byte offset of 16-byte chunk `ch` of row r in a K-major 128-byte-swizzled box.
__device__ __forceinline__ uint32_t at_swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

template <int HD>
__global__ void __launch_bounds__(kAtThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                           const __grid_constant__ CUtensorMap map_kv, const PrefillAttnArgs a, int kv_plane0_mul) {
    static_assert(kAtThreads == (3 + kAtSoftWarps) * 32, "roles");
    using C = AtCfg<HD>;
    constexpr int KB = C::KB;
    constexpr int HH = HD / 2;                 // output columns per softmax warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float *red_max = reinterpret_cast<float *>(sm + C::kRed);          // [2 bufs][2 halves][128]
    float *red_sum = red_max + 4 * kAtRows;                            // [2 halves][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::kBar);
    uint64_t *q_full = bars + 0, *k_full = bars + 1, *k_empty = bars + 2, *v_full = bars + 3, *v_empty = bars + 4;
    uint64_t *p_full = bars + 5, *p_empty = bars + 6, *drain = bars + 7;
    uint64_t *s_full = bars + 8, *s_free = bars + 10, *o_full = bars + 12, *o_free = bars + 14;   // [2] each
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 17);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqb = (a.n + kAtRows - 1) / kAtRows;
    const int heads = gridDim.x / nqb;                                  // ns x qh
    const int qb = nqb - 1 - (int)(blockIdx.x / heads);                  // most keys first
    const int pair = (int)blockIdx.x - (nqb - 1 - qb) * heads;
    const int i = pair / a.qh, h = pair - i * a.qh;
    const int g = h / (a.qh / a.kvh);
    const int q0 = qb * kAtRows;
    const int nc = qb + 1;                                               // key chunks [0, q0 + 128)
    // cache planes [S][HD] of this stream's layer: K of group g, V kvh planes further
    const int plane_k = a.streams[i] * kv_plane0_mul + (int)(a.layer_elems / ((size_t)a.S * HD)) + g;
    const int plane_v = plane_k + a.kvh;

    if (threadIdx.x == 0) {
        // the softmax warps' barriers (s_free, o_free, p_full) take one arrival per warp
        for (int b = 0; b < 16; ++b)
            mbar_init(&bars[b], (b == 5 || b == 10 || b == 11 || b == 14 || b == 15) ? kAtSoftWarps : 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer: Q once, then per chunk its K tile and its V tile
            const int qrow = (i * a.qh + h) * a.n + q0;
            mbar_arrive_expect_tx(q_full, 2 * KB * kAtBox);
            for (int part = 0; part < 2; ++part)
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_2d(sm + C::kQ + (uint32_t)(part * KB + kb) * kAtBox, part ? &map_ql : &map_qh, kb * 64,
                                qrow, q_full);
            int kis = 0;
            for (int c = 0; c < nc; ++c) {
                if (c > 0 && !role_wait(k_empty, (uint32_t)(c - 1) & 1u, abort_flag, a.status)) break;
                mbar_arrive_expect_tx(k_full, KB * kAtBox);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d_plain(sm + C::kK + (uint32_t)kb * kAtBox, &map_kv, kb * 64, c * kAtKeys, plane_k, k_full);
                ++kis;
            }
            // copies in flight land before the CTA can leave
            (void)mbar_wait_bounded(q_full, 0u, kAtDrainNs);
            if (kis) (void)mbar_wait_bounded(k_full, (uint32_t)(kis - 1) & 1u, kAtDrainNs);
        }
    } else if (warp == 2 + kAtSoftWarps) {
        if (lane == 0) {
            // ---- TMA producer of the V tiles
            int vis = 0;
            for (int c = 0; c < nc; ++c) {
                if (c > 0 && !role_wait(v_empty, (uint32_t)(c - 1) & 1u, abort_flag, a.status)) break;
                mbar_arrive_expect_tx(v_full, KB * kAtBox);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d_plain(sm + C::kV + (uint32_t)kb * kAtBox, &map_kv, kb * 64, c * kAtKeys, plane_v, v_full);
                ++vis;
            }
            if (vis) (void)mbar_wait_bounded(v_full, (uint32_t)(vis - 1) & 1u, kAtDrainNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: S_c, then O_{c-1} (whose P the softmax warps wrote meanwhile)
            constexpr uint32_t idesc_s = tc_idesc_mn<kAtRows, kAtKeys>();
            constexpr uint32_t idesc_o = tc_idesc_mn<kAtRows, HD, true>();
            const uint32_t sQ = smem_addr(sm + C::kQ), sK = smem_addr(sm + C::kK), sV = smem_addr(sm + C::kV),
                           sP = smem_addr(sm + C::kP);
            bool ok = role_wait(q_full, 0u, abort_flag, a.status);
            for (int c = 0; c <= nc && ok; ++c) {
                if (c < nc) {
                    ok = role_wait(k_full, (uint32_t)c & 1u, abort_flag, a.status) &&
                         (c < 2 || role_wait(&s_free[c & 1], (uint32_t)((c >> 1) - 1) & 1u, abort_flag, a.status));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(c & 1) * kAtKeys;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t bd = sw128_desc(sK + (uint32_t)kb * kAtBox + 32u * k);
                            tc_mma(d, sw128_desc(sQ + (uint32_t)kb * kAtBox + 32u * k), bd, idesc_s, (kb | k) ? 1u : 0u);
                            tc_mma(d, sw128_desc(sQ + (uint32_t)(KB + kb) * kAtBox + 32u * k), bd, idesc_s, 1u);
                        }
                    tc_commit(&s_full[c & 1]);
                    tc_commit(k_empty);
                }
                if (c > 0) {
                    const int cc = c - 1;
                    ok = role_wait(p_full, (uint32_t)cc & 1u, abort_flag, a.status) &&
                         role_wait(v_full, (uint32_t)cc & 1u, abort_flag, a.status) &&
                         (cc < 2 || role_wait(&o_free[cc & 1], (uint32_t)((cc >> 1) - 1) & 1u, abort_flag, a.status));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + 2u * kAtKeys + (uint32_t)(cc & 1) * HD;
#pragma unroll
                    for (int ks = 0; ks < kAtKeys / 16; ++ks) {
                        // keys 16 ks .. + 15: P's key block ks / 4 at 32-byte steps; V's rows 16 ks ..
                        const uint32_t po = (uint32_t)(ks >> 2) * kAtBox + 32u * (ks & 3);
                        const uint64_t bd = sw128_desc_mn(sV + (uint32_t)ks * 2048u, kAtBox, 1024u);
                        tc_mma(d, sw128_desc(sP + po), bd, idesc_o, ks ? 1u : 0u);
                        tc_mma(d, sw128_desc(sP + 2 * kAtBox + po), bd, idesc_o, 1u);
                    }
                    tc_commit(&o_full[cc & 1]);
                    tc_commit(p_empty);
                    tc_commit(v_empty);
                }
            }
            // every MMA issued has completed before the tensor memory can be freed
            tc_commit(drain);
            (void)mbar_wait_bounded(drain, 0u, kAtDrainNs);
        }
    } else {
        // ---- softmax and epilogue: row r of the block, keys [64 hf, 64 hf + 64) of each chunk
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int r = q4 * 32 + lane;
        const int query = q0 + r;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        uint8_t *pbh = sm + C::kP + (uint32_t)hf * kAtBox, *pbl = pbh + 2 * kAtBox;
        float o[HH];
#pragma unroll
        for (int e = 0; e < HH; ++e) o[e] = 0.f;
        float m = -INFINITY, l = 0.f, alpha_prev = 0.f;   // m in log2 units
        const float scale2 = a.scale * 1.4426950408889634f;                 // log2(e) / sqrt(hd)
        bool ok = true;
        for (int c = 0; c < nc; ++c) {
            float s[64];
            ok = ok && role_wait(&s_full[c & 1], (uint32_t)(c >> 1) & 1u, abort_flag, a.status);
            if (ok) {
                tc_fence_after();
                ld_cols<64>(tmem + lane_base + (uint32_t)(c & 1) * kAtKeys + (uint32_t)(hf * 64), s);
                tc_fence_before();
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) s[e] = 0.f;
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&s_free[c & 1]);
            // the scale (with log2 e: the exponentials are powers of two) and the causal
            // mask, which only the diagonal chunk and a chunk past the prompt's end need;
            // the chunk's maximum over both halves of the row
            const int key0 = c * kAtKeys + hf * 64;
            float cmax = -INFINITY;
            if (c == qb || (c + 1) * kAtKeys > a.n) {
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const int key = key0 + e;
                    s[e] = (key <= query && key < a.n) ? s[e] * scale2 : -INFINITY;
                    cmax = fmaxf(cmax, s[e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    s[e] *= scale2;
                    cmax = fmaxf(cmax, s[e]);
                }
            }
            float *rm = red_max + (c & 1) * 2 * kAtRows;
            rm[hf * kAtRows + r] = cmax;
            named_sync(1, kAtSoftWarps * 32);
            ok = ok && !*abort_flag;
            const float m_new = fmaxf(m, fmaxf(cmax, rm[(hf ^ 1) * kAtRows + r]));
            const float alpha = m == -INFINITY ? 0.f : exp2f(m - m_new);
            float psum = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                s[e] = exp2f(s[e] - m_new);   // exactly 0 for a masked key (-inf)
                psum += s[e];
            }
            l = l * alpha + psum;
            m = m_new;
            // P_c (hi, lo) into this half's key block, once the MMAs of O_{c-1} have read P_{c-1}
            if (c > 0) ok = ok && role_wait(p_empty, (uint32_t)(c - 1) & 1u, abort_flag, a.status);
            if (ok) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 vh, vl;
                    split_pack(s[8 * ch], s[8 * ch + 1], vh.x, vl.x);
                    split_pack(s[8 * ch + 2], s[8 * ch + 3], vh.y, vl.y);
                    split_pack(s[8 * ch + 4], s[8 * ch + 5], vh.z, vl.z);
                    split_pack(s[8 * ch + 6], s[8 * ch + 7], vh.w, vl.w);
                    *reinterpret_cast<uint4 *>(pbh + at_swz(r, ch)) = vh;
                    *reinterpret_cast<uint4 *>(pbl + at_swz(r, ch)) = vl;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(p_full);
            // O_{c-1} into the running output
            if (c > 0) {
                const int cc = c - 1;
                ok = ok && role_wait(&o_full[cc & 1], (uint32_t)(cc >> 1) & 1u, abort_flag, a.status);
                if (ok) {
                    tc_fence_after();
                    float v[HH];
                    ld_cols<HH>(tmem + lane_base + 2u * kAtKeys + (uint32_t)(cc & 1) * HD + (uint32_t)(hf * HH), v);
#pragma unroll
                    for (int e = 0; e < HH; ++e) o[e] = fmaf(o[e], alpha_prev, v[e]);
                    tc_fence_before();
                }
                __syncwarp();
                if (ok && lane == 0) mbar_arrive(&o_free[cc & 1]);
            }
            alpha_prev = alpha;
        }
        {
            const int cc = nc - 1;
            ok = ok && role_wait(&o_full[cc & 1], (uint32_t)(cc >> 1) & 1u, abort_flag, a.status);
            if (ok) {
                tc_fence_after();
                float v[HH];
                ld_cols<HH>(tmem + lane_base + 2u * kAtKeys + (uint32_t)(cc & 1) * HD + (uint32_t)(hf * HH), v);
#pragma unroll
                for (int e = 0; e < HH; ++e) o[e] = fmaf(o[e], alpha_prev, v[e]);
                tc_fence_before();
            }
        }
        // the row's sum over both halves, then O / l as bf16 hi + lo parts
        red_sum[hf * kAtRows + r] = l;
        named_sync(1, kAtSoftWarps * 32);
        ok = ok && !*abort_flag;
        const float inv = 1.0f / (l + red_sum[(hf ^ 1) * kAtRows + r]);
        if (ok && query < a.n) {
            const size_t ob = ((size_t)i * a.n + query) * a.qh * HD + (size_t)h * HD + hf * HH;
#pragma unroll
            for (int e = 0; e < HH; e += 8) {
                uint4 vh, vl;
                split_pack(o[e] * inv, o[e + 1] * inv, vh.x, vl.x);
                split_pack(o[e + 2] * inv, o[e + 3] * inv, vh.y, vl.y);
                split_pack(o[e + 4] * inv, o[e + 5] * inv, vh.z, vl.z);
                split_pack(o[e + 6] * inv, o[e + 7] * inv, vh.w, vl.w);
                *reinterpret_cast<uint4 *>(a.out_hi + ob + e) = vh;
                *reinterpret_cast<uint4 *>(a.out_lo + ob + e) = vl;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

typedef void (*AtFn)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const PrefillAttnArgs, int);

template <int HD> cudaError_t at_attr() {
    static cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(prefill_attn_tc_kernel<HD>),
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AtCfg<HD>::kSmem);
    return e;
}

template <int HD> cudaError_t launch_hd(int ns, const PrefillAttnArgs &a, const PrefillAttnMaps &m, cudaStream_t s) {
    cudaError_t e = at_attr<HD>();
    if (e != cudaSuccess) return e;
    const size_t plane = (size_t)a.S * HD;
    if (a.layer_elems % plane) return cudaErrorInvalidValue;
    const int nqb = (a.n + kAtRows - 1) / kAtRows;
    prefill_attn_tc_kernel<HD><<<ns * a.qh * nqb, kAtThreads, AtCfg<HD>::kSmem, s>>>(
        m.qh, m.ql, m.kv, a, (int)(a.stream_elems / plane));
    return cudaGetLastError();
}

}  // namespace

bool make_prefill_attn_maps(int hd, int ns, const PrefillAttnArgs &a, PrefillAttnMaps *m) {
    if ((hd != 64 && hd != 128) || a.qh % a.kvh || a.n < 1 || a.S < 1) return false;
    // the cache's planes [S][hd]: each stream's caches are stream_elems apart, a whole
    // number of planes
    const size_t plane = (size_t)a.S * hd;
    if (a.stream_elems % plane) return false;
    const long long planes = (long long)((size_t)a.cache_streams * a.stream_elems / plane);
    const long long qrows = (long long)ns * a.qh * a.n;
    return qrows <= INT32_MAX && make_bf16_rows_map(&m->qh, a.q_hi, (int)qrows, hd, kAtRows) &&
           make_bf16_rows_map(&m->ql, a.q_lo, (int)qrows, hd, kAtRows) &&
           make_kv_tile_map(&m->kv, a.kv, hd, a.S, planes, kAtKeys);
}

cudaError_t launch_prefill_attention_tc(int hd, int ns, const PrefillAttnArgs &a, const PrefillAttnMaps &m,
                                        cudaStream_t s) {
    if (a.qh % a.kvh || a.n < 1) return cudaErrorInvalidValue;
    if (hd == 128) return launch_hd<128>(ns, a, m, s);
    if (hd == 64) return launch_hd<64>(ns, a, m, s);
    return cudaErrorInvalidValue;
}

}  // namespace qd

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
#include <cuda.h>

#include "decode_common.cuh"
#include "mma_sync.cuh"

namespace qd {

namespace {

// ---- attention: one CTA per (stream, kv group, chunk of kBattChunk = 512 cached
// positions), 4 consumer warps and a producer warp.  The producer streams the chunk's tiles of 32
// positions, each tile's K rows then its V rows, into 4 shared-memory slots (3-D tiled
// TMA loads of the cache's [S][head_dim] planes with the 128-byte swizzle; full/empty
// mbarriers per slot).  The consumer warps go in pairs: pair i takes tiles i, i + 2,
// i + 4, ... through its own two slots (K and V; so every waiter sees every phase of the
// barriers it waits on), warp 2i + j the tile's positions 16 j .. 16 j + 15.  They
// compute on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with the
// positions as the fragments' M: the scores (A = the 16 K rows, B = the G q heads of
// the group as bf16 hi and lo columns, so a score is column 2h + column 2h + 1), an
// online-softmax update per head (running max and sum; the output rescaled when the
// max grows), then P.V (A = the V rows transposed, 16 head dimensions at a time;
// B = the probabilities as bf16 hi and lo columns, moved from the score fragments'
// layout through a small per-warp buffer).  The tensor cores serve here to cut the
// instruction count per cached row (one product per 16 positions x 16 dimensions),
// not for their FLOP rate: the kernel is bound by the bytes of the cache.
// The warps' partials (and, in the chunk that holds it, the new position, whose k and
// v are QK-normed, rotated, rounded to the cache type and appended) are combined into
// the chunk's (max, sum, output); the last chunk CTA of a (stream, group) to finish
// merges the chunks in order (flash-decoding merge) and writes the output.  Equal
// chunks keep the work balanced whatever the lengths; no CTA waits for another.  As a
// programmatic dependent of the QKV GEMM, the producer starts on the cached rows
// (written by earlier steps) before the consumers wait for the GEMM's q, k and v.
constexpr int kBattConsumers = 4;
constexpr int kBattThreads = (kBattConsumers + 1) * 32;
constexpr int kBattTile = 32;        // positions per ring slot
constexpr int kBattSlots = 4;        // two per warp pair
constexpr int kBattMaxGroup = 8;     // q heads per kv head
constexpr int kBattPairs = kBattConsumers / 2;
constexpr int kBattTiles = kBattChunk / kBattTile;
constexpr int kBattUnits = kBattTiles / kBattPairs;   // tiles per pair
static_assert(kBattTiles % kBattPairs == 0 && kBattSlots == 2 * kBattPairs, "whole tiles per warp pair");

// Slots of tile i: pair (i mod pairs)'s two slots, K in the first and V in the second;
// the pair's u-th tile (i / pairs) is the slots' use u (barrier phase parity u & 1).
__host__ __device__ constexpr int batt_kslot(int i) { return 2 * (i % kBattPairs); }

// Byte offset of 16-byte chunk `ch` of row r in a tile written by TMA with the 128-byte
// swizzle: head_dim / 64 boxes of kBattTile rows x 128 bytes, the chunk index XOR
// (r mod 8) inside each (1024-byte aligned) box.
__device__ __forceinline__ uint32_t kv_swz(int r, int ch) {
    return (uint32_t)((ch >> 3) * (kBattTile * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

template <int HD, int G> struct BattShape {
    static constexpr int NT = (2 * G + 7) / 8;   // 8-column n-tiles holding the heads' hi/lo columns
    static constexpr uint32_t kTileBytes = kBattTile * HD * 2;
    static constexpr int RS = HD + 2;            // partial record: output, max, sum
    // after the 1024-byte alignment: ring (the warps' records once it is idle), q heads,
    // k, v, cos/sin, the warps' P^T buffers, barriers, flags
    static constexpr size_t kRing = (size_t)kBattSlots * kTileBytes;
    static constexpr size_t kRed = (size_t)(kBattConsumers + 2) * G * RS * 4;
    static constexpr size_t kPt = (size_t)kBattConsumers * NT * 8 * 16 * 2;
    static constexpr size_t kSmem = 1024 + (kRing > kRed ? kRing : kRed) + (size_t)G * HD * 4 + 3 * (size_t)HD * 4 +
                                    kPt + 2 * kBattSlots * 8 + 16;
};

template <int HD, int G>
__global__ void __launch_bounds__(kBattThreads, 4)
    batch_attn_kernel(const __grid_constant__ CUtensorMap kv_map, const BatchAttnArgs a) {
    using KT = __nv_bfloat16;
    using S_ = BattShape<HD, G>;
    constexpr int HALF = HD / 2;
    constexpr int NT = S_::NT;
    constexpr uint32_t kTileBytes = S_::kTileBytes;
    constexpr int RS = S_::RS;
    constexpr int KS = HD / 16;                        // k-steps of a score
    constexpr int MT = HD / 16;                        // 16-dimension m-tiles of the output
    static_assert(G >= 1 && G <= kBattMaxGroup && HD % 64 == 0, "group size / head_dim");
    extern __shared__ uint8_t smem_raw[];
    // the swizzle pattern is anchored at 1024-byte boundaries of the shared window
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = smem;                                                           // [slots][tile]
    float *red = reinterpret_cast<float *>(ring);                                   // [warps + 2][G][RS]
    float *qs = reinterpret_cast<float *>(ring + (S_::kRing > S_::kRed ? S_::kRing : S_::kRed));  // [G][HD]
    float *kn = qs + G * HD;                                                        // [HD]
    float *vn = kn + HD;                                                            // [HD]
    float *rc = vn + HD;                                                            // [HALF] cos, [HALF] sin
    KT *pt = reinterpret_cast<KT *>(rc + HD);                                       // [warps][NT * 8][16]
    uint64_t *full = reinterpret_cast<uint64_t *>(pt + (size_t)kBattConsumers * NT * 8 * 16);   // [slots]
    uint64_t *empty = full + kBattSlots;                                            // [slots]
    int *flag = reinterpret_cast<int *>(empty + kBattSlots);                        // [0] abort, [1] last chunk

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
    const int total = 2 * nT;                          // each tile K, then its V
    const size_t grp_off = (size_t)g * a.S * HD;
    KT *kbase = reinterpret_cast<KT *>(a.kv) + (size_t)b * a.stream_elems + a.layer_elems + grp_off;
    KT *vbase = kbase + (size_t)a.kvh * a.S * HD;
    // [S][HD] planes of the caches: this pair's K plane; its V plane kvh further
    const int plane_k = (int)(((size_t)b * a.stream_elems + a.layer_elems) / ((size_t)a.S * HD)) + g;

    if (tid == 0) {
        for (int i = 0; i < kBattSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);                   // the two warps of the pair that reads it
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
                // tile i's K then its V; the pair's second tile reuses its slots once both
                // of its warps have read the first
                const int i = issued >> 1, kv = issued & 1;
                const int slot = batt_kslot(i) + kv;
                if (i >= kBattPairs && !mbar_wait_bounded(&empty[slot], (uint32_t)(i / kBattPairs - 1) & 1u)) {
                    atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
                    *reinterpret_cast<volatile int *>(flag) = 1;
                    break;
                }
                const int z = plane_k + kv * a.kvh;
                // whole tiles: positions past the plane's S load as zeros; those past
                // the chunk's rows get probability 0
                mbar_arrive_expect_tx(&full[slot], kTileBytes);
#pragma unroll
                for (int h = 0; h < HD / 64; ++h)
                    tma_load_3d(ring + (size_t)slot * kTileBytes + h * (kBattTile * 128), &kv_map, h * 64,
                                j0 + i * kBattTile, z, &full[slot], pol);
            }
            // copies in flight land before the CTA can leave: each slot's last use
            for (int k = 0; k < issued; ++k) {
                const int i = k >> 1;
                if (k + 2 * kBattPairs >= issued)   // no later use of this slot was issued
                    (void)mbar_wait_bounded(&full[batt_kslot(i) + (k & 1)], (uint32_t)(i / kBattPairs) & 1u, 10000000ull);
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
    // the P^T columns past the heads' stay zero
    for (int i = tid; i < kBattConsumers * NT * 8 * 16; i += NC) pt[i] = __float2bfloat16_rn(0.f);
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

    // B fragments of the scores: column n of n-tile nt is q head (8 nt + n) / 2, its hi
    // part for even n, lo for odd (zero past the G heads); lane (gl, tl) holds rows
    // (k) 2 tl, 2 tl + 1 and 2 tl + 8, 2 tl + 9 of column gl
    const int gl = lane >> 2, tl = lane & 3;
    uint32_t qb[NT][KS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + gl, hq = n >> 1;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const float *qr = qs + (size_t)(hq < G ? hq : 0) * HD + ks * 16 + 2 * tl;
            const float x0 = hq < G ? qr[0] : 0.f, x1 = hq < G ? qr[1] : 0.f;
            const float x2 = hq < G ? qr[8] : 0.f, x3 = hq < G ? qr[9] : 0.f;
            uint32_t h01, l01, h89, l89;
            split_pack(x0, x1, h01, l01);
            split_pack(x2, x3, h89, l89);
            qb[nt][ks][0] = (n & 1) ? l01 : h01;
            qb[nt][ks][1] = (n & 1) ? l89 : h89;
        }
    }

    const int pr = warp >> 1, mb = warp & 1;           // warp pair, 16-position half of its tiles
    const int mi = lane >> 3, rr = lane & 7;           // ldmatrix: matrix and row this lane addresses
    bool ok = true;
    // One pass over the warp's units (tiles pr, pr + pairs, ...; its 16 positions of each): the
    // scores of the unit's K tile, an online-softmax update (running max and sum per
    // head, the output rescaled when the max grows), then P.V over the unit's V tile.
    // Lane (gl, tl) keeps head 4 nt + tl's running max / sum, and its output dimensions
    // 16 mt + gl (+ 8) as the hi + lo columns of the accumulators.
    float pm_[NT], pl_[NT];
    float o[NT][MT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        pm_[nt] = -INFINITY;
        pl_[nt] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    }
    KT *ptw = pt + (size_t)warp * NT * 8 * 16;         // [NT * 8 columns][16 positions]
#pragma unroll 1
    for (int u = 0; u < kBattUnits; ++u) {
        const int t = pr + u * kBattPairs;
        if (t >= nT || !ok) continue;
        const int ks_slot = batt_kslot(t), vs_slot = ks_slot + 1;
        if (!mbar_wait_bounded(&full[ks_slot], (uint32_t)u & 1u)) {
            ok = false;
            continue;
        }
        uint32_t tile = smem_addr(ring + (size_t)ks_slot * kTileBytes);
        float d[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t af[4];
            ldsm_x4(tile + kv_swz(16 * mb + rr + 8 * (mi & 1), 2 * ks + (mi >> 1)), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(d[nt], af, qb[nt][ks][0], qb[nt][ks][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ks_slot]);
        const int pos = t * kBattTile + 16 * mb + gl;
        float pv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float s0 = pos < rows_c ? (d[nt][0] + d[nt][1]) * a.scale : -INFINITY;
            const float s1 = pos + 8 < rows_c ? (d[nt][2] + d[nt][3]) * a.scale : -INFINITY;
            float mx = fmaxf(s0, s1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(pm_[nt], mx);
            // rescale what came before (nothing to rescale while the max is -inf)
            const float f = pm_[nt] == -INFINITY ? 0.f : expf(pm_[nt] - mn);
            pv[nt][0] = mn == -INFINITY || s0 == -INFINITY ? 0.f : expf(s0 - mn);
            pv[nt][1] = mn == -INFINITY || s1 == -INFINITY ? 0.f : expf(s1 - mn);
            float sum = pv[nt][0] + pv[nt][1];
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            pl_[nt] = pl_[nt] * f + sum;
            pm_[nt] = mn;
            // lane (gl, tl)'s accumulators hold head 4 nt + tl: the same head as its
            // scores, so the factor needs no exchange
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[nt][mt][0] *= f;
                o[nt][mt][1] *= f;
                o[nt][mt][2] *= f;
                o[nt][mt][3] *= f;
            }
        }
        // this unit's probabilities, hi/lo columns 2h, 2h + 1 of head h = 4 nt + tl
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hq = nt * 4 + tl;
            if (hq < G) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const KT hi = __float2bfloat16_rn(pv[nt][e]);
                    ptw[(2 * hq) * 16 + gl + 8 * e] = hi;
                    ptw[(2 * hq + 1) * 16 + gl + 8 * e] = __float2bfloat16_rn(pv[nt][e] - __bfloat162float(hi));
                }
            }
        }
        __syncwarp();
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const KT *col = ptw + (size_t)(nt * 8 + gl) * 16;
            pb[nt][0] = *reinterpret_cast<const uint32_t *>(col + 2 * tl);
            pb[nt][1] = *reinterpret_cast<const uint32_t *>(col + 2 * tl + 8);
        }
        __syncwarp();
        if (!mbar_wait_bounded(&full[vs_slot], (uint32_t)u & 1u)) {
            ok = false;
            continue;
        }
        tile = smem_addr(ring + (size_t)vs_slot * kTileBytes);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            // A = V^T: head dimensions 16 mt .. + 15 x the unit's 16 positions
            uint32_t af[4];
            ldsm_x4_t(tile + kv_swz(16 * mb + rr + 8 * (mi >> 1), 2 * mt + (mi & 1)), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(o[nt][mt], af, pb[nt][0], pb[nt][1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[vs_slot]);
    }
    if (!ok) {
        if (lane == 0) atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
        *reinterpret_cast<volatile int *>(flag) = 1;
    }
    // combine the warps and the new position into the chunk's record (the ring is
    // idle once every tile was consumed): lane (gl, tl) holds head 4 nt + tl's output
    // dimensions 16 mt + gl and 16 mt + gl + 8 as its hi + lo columns
    named_sync(1, NC);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hq = nt * 4 + tl;
        if (hq < G) {
            float *rw = red + ((size_t)warp * G + hq) * RS;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                rw[16 * mt + gl] = o[nt][mt][0] + o[nt][mt][1];
                rw[16 * mt + gl + 8] = o[nt][mt][2] + o[nt][mt][3];
            }
            if (gl == 0) {
                rw[HD] = pm_[nt];
                rw[HD + 1] = pl_[nt];
            }
        }
    }
    const int nrec = holds_new ? kBattConsumers + 1 : kBattConsumers;
    if (holds_new && warp == 0) {
        constexpr int DPL = HD / 32;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) d = fmaf(qs[hh * HD + lane * DPL + e], kn[lane * DPL + e], d);
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

typedef void (*BattFn)(const CUtensorMap, const BatchAttnArgs);

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
#define QD_BATT(HDV, GV) \
    if (hd == HDV && group == GV) return BattShape<HDV, GV>::kSmem;
    QD_BATT(128, 1) QD_BATT(128, 2) QD_BATT(128, 4) QD_BATT(128, 8)
    QD_BATT(64, 1) QD_BATT(64, 2) QD_BATT(64, 4) QD_BATT(64, 8)
#undef QD_BATT
    return 0;
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

cudaError_t launch_batch_attention(int hd, int B, const BatchAttnArgs &a, const CUtensorMap &kv_map, cudaStream_t s,
                                   bool pdl) {
    const BattFn fn = a.qh % a.kvh ? nullptr : batt_fn(hd, a.qh / a.kvh);
    const size_t smem = fn ? batch_attention_smem_bytes(hd, a.qh / a.kvh) : 0;
    if (!fn || smem > 160 * 1024 || !a.partial || !a.counter) return cudaErrorInvalidValue;
    // chunk-major order: every pair's first chunk, then every pair's second, ...
    void *args[2] = {const_cast<CUtensorMap *>(&kv_map), const_cast<BatchAttnArgs *>(&a)};
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

// Device building blocks shared by the per-phase kernels (decode_kernels.cu) and
// the persistent decode-step kernel (decode_persistent.cu).  Both paths call the
// same functions with the same work partition, so they produce bitwise identical
// results.
//
// Weight stream: a ring of `nst` shared-memory slots of kSlotBytes.  The producer
// (one thread) issues cp.async.bulk copies of whole rows into the slots in a fixed
// order; consumers walk the same order.  Slot i of stage index `sidx` is
// sidx % nst and its phase parity is (sidx / nst) & 1; `full[i]` completes when the
// bytes have landed, `empty[i]` when all kConsumerWarps consumer warps are done.
#pragma once

#include <float.h>
#include <limits.h>

#include "qd_device.cuh"
#include "qd_internal.h"

namespace qd {

struct Ring {
    uint8_t *base;
    uint64_t *full;
    uint64_t *empty;
    int nst;
};

// Producer: stream `nrows` rows of `row_bytes` from `src` in stages of `rps` rows.
// Returns false if a wait on a free slot expired.
__device__ __forceinline__ bool produce_rows(const Ring &R, uint32_t &sidx, const uint8_t *src, int nrows,
                                             uint32_t row_bytes, int rps, uint64_t pol) {
    for (int r = 0; r < nrows; r += rps) {
        const int slot = (int)(sidx % (uint32_t)R.nst);
        const uint32_t use = sidx / (uint32_t)R.nst;
        if (use > 0 && !mbar_wait_bounded(&R.empty[slot], (use - 1) & 1)) return false;
        const int n = nrows - r < rps ? nrows - r : rps;
        mbar_arrive_expect_tx(&R.full[slot], n * row_bytes);
        bulk_copy_g2s(R.base + (size_t)slot * kSlotBytes, src + (size_t)r * row_bytes, n * row_bytes, &R.full[slot],
                      pol);
        ++sidx;
    }
    return true;
}

// Producer: one slot holding `bytes` (may be 0) from `src`.
__device__ __forceinline__ bool produce_block(const Ring &R, uint32_t &sidx, const void *src, uint32_t bytes,
                                              uint64_t pol) {
    const int slot = (int)(sidx % (uint32_t)R.nst);
    const uint32_t use = sidx / (uint32_t)R.nst;
    if (use > 0 && !mbar_wait_bounded(&R.empty[slot], (use - 1) & 1)) return false;
    mbar_arrive_expect_tx(&R.full[slot], bytes);
    if (bytes) bulk_copy_g2s(R.base + (size_t)slot * kSlotBytes, src, bytes, &R.full[slot], pol);
    ++sidx;
    return true;
}

// Consumer side of one slot: wait until it is full; returns its address or null on timeout.
__device__ __forceinline__ const uint8_t *slot_acquire(const Ring &R, uint32_t sidx) {
    const int slot = (int)(sidx % (uint32_t)R.nst);
    if (!mbar_wait_bounded(&R.full[slot], (sidx / (uint32_t)R.nst) & 1)) return nullptr;
    return R.base + (size_t)slot * kSlotBytes;
}
// Each consumer warp releases the slot once (lane 0 after __syncwarp).
__device__ __forceinline__ void slot_release(const Ring &R, uint32_t sidx, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[sidx % (uint32_t)R.nst]);
}

// Consumers: reduce `nrows` rows (in stages of `rps`) against the register slice xr
// of the input vector.  A row is split over `rs` warps (warp = rr * rs + sub); the
// partial sum of each part goes to res[row * rs + sub].  R rows per warp at a time:
// independent accumulators, then one butterfly that reduces all R rows together.
template <typename WT, int NSEG>
__device__ __forceinline__ bool gemv_consume(const Ring &R, uint32_t &sidx, int nrows, int rps, uint32_t row_bytes,
                                             int rs, int colbase, const float *xr, float *res) {
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    constexpr int RR = NSEG <= 2 ? 4 : 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % rs, rr = warp / rs, rpp = kConsumerWarps / rs;
    for (int rbase = 0; rbase < nrows; rbase += rps) {
        const uint8_t *sbase = slot_acquire(R, sidx);
        if (!sbase) return false;
        const int n = nrows - rbase < rps ? nrows - rbase : rps;
        for (int r = rr; r < n; r += RR * rpp) {
            uint4 w[RR][NSEG];
#pragma unroll
            for (int q = 0; q < RR; ++q) {
                const int rq = r + q * rpp;
                const WT *wrow = reinterpret_cast<const WT *>(sbase + (size_t)(rq < n ? rq : r) * row_bytes) + colbase;
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg)
                    w[q][sg] = rq < n ? *reinterpret_cast<const uint4 *>(wrow + sg * SEGW + lane * EPL)
                                      : make_uint4(0u, 0u, 0u, 0u);
            }
            float acc[RR];
#pragma unroll
            for (int q = 0; q < RR; ++q) {
                acc[q] = 0.f;
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg) {
                    float f[EPL];
                    Elem<WT>::unpack(w[q][sg], f);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[q] = fmaf(f[e], xr[sg * EPL + e], acc[q]);
                }
            }
            const bool b4 = (lane & 16) != 0;
            float v;
            int q;
            if (RR == 4) {
                const bool b3 = (lane & 8) != 0;
                float k0 = b4 ? acc[2 % RR] : acc[0], s0 = b4 ? acc[0] : acc[2 % RR];
                float k1 = b4 ? acc[3 % RR] : acc[1], s1 = b4 ? acc[1] : acc[3 % RR];
                k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
                k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
                v = b3 ? k1 : k0;
                const float sx = b3 ? k0 : k1;
                v += __shfl_xor_sync(0xffffffffu, sx, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                q = (b4 ? 2 : 0) + (b3 ? 1 : 0);   // lanes 0, 8, 16, 24 hold rows 0..3
            } else {
                v = b4 ? acc[1] : acc[0];
                const float sx = b4 ? acc[0] : acc[1];
                v += __shfl_xor_sync(0xffffffffu, sx, 16);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                q = b4 ? 1 : 0;                     // lanes 0, 16 hold rows 0, 1
            }
            const int rq = r + q * rpp;
            if ((lane & (RR == 4 ? 7 : 15)) == 0 && rq < n) res[(rbase + rq) * rs + sub] = v;
        }
        slot_release(R, sidx, lane);
        ++sidx;
    }
    return true;
}

// Register slice of a vector for the consumer thread: columns colbase + sg*SEGW + lane*EPL + e.
template <typename WT, int NSEG>
__device__ __forceinline__ void load_slice(const float *v, int colbase, float *xr) {
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
            const float4 v4 = __ldcg(reinterpret_cast<const float4 *>(v + colbase + sg * SEGW + lane * EPL + e));
            xr[sg * EPL + e] = v4.x;
            xr[sg * EPL + e + 1] = v4.y;
            xr[sg * EPL + e + 2] = v4.z;
            xr[sg * EPL + e + 3] = v4.w;
        }
}

// Whole vector (n floats, n a multiple of 4) into shared memory, loaded once per CTA
// by the consumer threads: every SM reads a freshly written activation vector right
// after a dependency, so per-warp loads of the same lines would queue at the few L2
// slices that hold them.  The caller synchronises the consumers before use.
__device__ __forceinline__ void load_vec_smem(const float *src, int n, float *dst) {
    for (int i = threadIdx.x * 4; i < n; i += kConsumerWarps * 32 * 4)
        *reinterpret_cast<float4 *>(dst + i) = __ldcg(reinterpret_cast<const float4 *>(src + i));
}

// Register slice of a shared-memory vector for the consumer thread.
template <typename WT, int NSEG>
__device__ __forceinline__ void smem_slice(const float *v, int colbase, float *xr) {
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(v + colbase + sg * SEGW + lane * EPL + e);
            xr[sg * EPL + e] = v4.x;
            xr[sg * EPL + e + 1] = v4.y;
            xr[sg * EPL + e + 2] = v4.z;
            xr[sg * EPL + e + 3] = v4.w;
        }
}

// RMSNorm of the register slices across the consumer warps (warps rr == 0 hold each
// column once): xr <- xr * rsqrt(mean(x^2) + eps) * gamma.  `misc` holds >= 8 floats;
// `gsm` is gamma staged in shared memory.  Named barrier 1 over the consumers.
template <typename WT, int NSEG>
__device__ __forceinline__ void rmsnorm_slice(float *xr, const float *gsm, int K, int rs, int colbase, float eps,
                                              float *misc, float *y_out) {
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % rs, rr = warp / rs;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NSEG * EPL; ++i) ss = fmaf(xr[i], xr[i], ss);
    ss = warp_sum(ss);
    if (lane == 0 && rr == 0) misc[sub] = ss;
    named_sync(1, kConsumerWarps * 32);
    float tot = 0.f;
    for (int j = 0; j < rs; ++j) tot += misc[j];
    const float inv = 1.0f / sqrtf(tot / (float)K + eps);
    const bool wy = y_out != nullptr && rr == 0;
    // the gammas (and y) four at a time: a lane's EPL columns are contiguous, so one
    // scalar access per column would put every fourth (fp32: eighth) lane on one bank
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
        for (int e = 0; e < EPL; e += 4) {
            const int i = sg * EPL + e;
            const int col = colbase + sg * SEGW + lane * EPL + e;
            const float4 g = *reinterpret_cast<const float4 *>(gsm + col);
            xr[i] = xr[i] * inv * g.x;
            xr[i + 1] = xr[i + 1] * inv * g.y;
            xr[i + 2] = xr[i + 2] * inv * g.z;
            xr[i + 3] = xr[i + 3] * inv * g.w;
            if (wy) *reinterpret_cast<float4 *>(y_out + col) = make_float4(xr[i], xr[i + 1], xr[i + 2], xr[i + 3]);
        }
    named_sync(1, kConsumerWarps * 32);   // misc is reused by the caller
}

// The step's input vector (first phase of a step): the token row of the embedding
// table, the caller's embedding, or the staged prompt input at position `pos`.
// Thread 0 resolves the step description from the device state; CTA 0 records the
// token in the emitted set.  Fills the register slice xr; warps rr == 0 of CTA
// `writer_cta` also store the vector to x_out (and to tap when given).
typedef StepInputArgs StepInput;

template <typename WT, int NSEG>
__device__ __forceinline__ void step_input_slice(const StepInput &in, DevState *st, int K, int rs, int colbase,
                                                 float *xr, int *misc_i, float *x_out, float *tap) {
    constexpr int EPL = Elem<WT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        const int pos = st->pos;
        const int mode = st->in_mode;
        int tok = st->token_in;
        if (mode == IN_FEEDBACK) tok = st->out_id;
        else if (mode == IN_STAGED_TOKENS) tok = pos < in.S ? in.stage_tokens[pos] : -1;
        else if (mode == IN_STAGED_EMBEDS) tok = -1;
        int bad = 0;
        if (pos >= in.S) {
            bad = 1;
            if (blockIdx.x == 0) atomicOr(&st->status, DEV_ERR_BAD_POS);
        }
        const bool needs_row = (mode == IN_TOKEN || mode == IN_FEEDBACK || mode == IN_STAGED_TOKENS);
        if (!bad && needs_row && (tok < 0 || tok >= in.table_rows || in.table == nullptr)) {
            bad = 1;
            if (blockIdx.x == 0) atomicOr(&st->status, DEV_ERR_BAD_TOKEN);
        }
        if (blockIdx.x == 0 && st->add_emitted && tok >= 0 && tok < in.vocab)
            in.emitted[tok >> 5] |= 1u << (tok & 31);
        misc_i[0] = mode;
        misc_i[1] = tok;
        misc_i[2] = bad;
        misc_i[3] = pos;
    }
    named_sync(1, kConsumerWarps * 32);
    const int mode = misc_i[0], tok = misc_i[1], bad = misc_i[2], pos = misc_i[3];
    const bool writer = blockIdx.x == 0 && (warp / rs) == 0;
#pragma unroll
    for (int sg = 0; sg < NSEG; ++sg) {
        const int col = colbase + sg * SEGW + lane * EPL;
        float v[EPL];
        if (bad) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) v[e] = 0.f;
        } else if (mode == IN_EMBED || mode == IN_STAGED_EMBEDS) {
            const float *src = mode == IN_EMBED ? in.embed_in + col : in.stage_embeds + (size_t)pos * K + col;
#pragma unroll
            for (int e = 0; e < EPL; e += 4) {
                const float4 f4 = __ldcg(reinterpret_cast<const float4 *>(src + e));
                v[e] = f4.x; v[e + 1] = f4.y; v[e + 2] = f4.z; v[e + 3] = f4.w;
            }
        } else {
            const uint4 u = *reinterpret_cast<const uint4 *>(reinterpret_cast<const WT *>(in.table) +
                                                             (size_t)tok * K + col);
            Elem<WT>::unpack(u, v);
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) xr[sg * EPL + e] = v[e];
        if (writer) {
#pragma unroll
            for (int e = 0; e < EPL; e += 4) {
                const float4 f4 = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                *reinterpret_cast<float4 *>(x_out + col + e) = f4;
                if (tap) *reinterpret_cast<float4 *>(tap + col + e) = f4;
            }
        }
    }
}

__device__ __forceinline__ bool arg_better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// ---------------------------------------------------------------------------------
// Sampling: the top-k candidates of a set of logits, the counter-based draw, and the
// pick (the same steps, in the same order, as the oracle's sampler).
// ---------------------------------------------------------------------------------

// Order-preserving unsigned key of a float: a larger float has a larger key; -0 counts
// as +0 (they compare equal).
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One 64-bit key per candidate (value, index >= 0): a larger key is the better
// candidate (the larger value, then the lower index).  The value and the index come
// back out of it (a -0 as +0).
__device__ __forceinline__ uint64_t cand_key(float v, int i) {
    return ((uint64_t)order_key(v) << 32) | (uint32_t)(0x7fffffff - i);
}
__device__ __forceinline__ float cand_value(uint64_t c) {
    const uint32_t k = (uint32_t)(c >> 32);
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ int cand_index(uint64_t c) { return 0x7fffffff - (int)(uint32_t)c; }

// Consumer threads (named barrier 1; ck written and synchronised by the caller): the
// m <= NC keys ck ranked by counting, for each, the keys above it (equal keys -- only
// identical padding -- by position); the best Ke go to out_v / out_i[0..Ke) and slots
// Ke..K get -inf / INT_MAX.
static __device__ __noinline__ void rank_keys(const uint64_t *ck, int m, int Ke, int K, float *out_v, int *out_i) {
    constexpr int NC = kConsumerWarps * 32;
    const int tid = threadIdx.x;
    if (tid < m) {
        const uint64_t c = ck[tid];
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < m; ++j) {
            const uint64_t cj = ck[j];
            r += (int)(cj > c) | ((int)(cj == c) & (int)(j < tid));
        }
        if (r < Ke) {
            out_v[r] = cand_value(c);
            out_i[r] = cand_index(c);
        }
    }
    if (tid >= Ke && tid < K) {
        out_v[tid] = -INFINITY;
        out_i[tid] = INT_MAX;
    }
    named_sync(1, NC);
}

// Consumer threads (named barrier 1): the K (<= kMaxTopK) largest of n values -- value
// i at vals[i * stride], its index idx[i] (or base + i when idx is null) -- with ties
// to the lower index, into out_v / out_i[0..K) sorted by value descending, then index
// ascending; entries past n are -inf / INT_MAX.  Among equal values the indices must
// ascend with i.  Radix select of the K-th largest key (8-bit passes over shared
// histograms): as soon as the keys in or above the K-th key's bin fit one per thread
// they are gathered and ranked; otherwise, after four passes, every larger key and, in
// index order, as many equal keys as are needed are ranked.  out_* must not overlap
// the scratch (8-byte aligned, kTopkScratchWords words).
static_assert(kConsumerWarps * 32 <= 256, "block_topk gathers at most one key per histogram bin");
static __device__ __noinline__ void block_topk(const float *vals, int stride, const int *idx, int base, int n, int K,
                                               float *out_v, int *out_i, int *scratch) {
    constexpr int NC = kConsumerWarps * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // ctl[0]: the bin of the pass, ctl[2]: slot counter, ctl[4 + p]: keys still needed
    // entering pass p (ctl[8]: equal keys to take after the last pass), ctl[9]: keys in
    // or above the bin of the pass.  The gathered keys reuse hist and cnt.
    int *hist = scratch, *cnt = scratch + 256, *ctl = cnt + NC;
    uint64_t *gk = reinterpret_cast<uint64_t *>(scratch);
    float *tv = reinterpret_cast<float *>(ctl + 16);
    int *ti = reinterpret_cast<int *>(tv + kMaxTopK);
    const int Ke = K < n ? K : n;
    if (tid == 0) {
        ctl[4] = Ke;
        ctl[2] = 0;
    }
    if (Ke == 0) {
        named_sync(1, NC);
        rank_keys(gk, 0, 0, K, out_v, out_i);
        return;
    }
    uint32_t prefix = 0, mask = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int b = tid; b < 256; b += NC) hist[b] = 0;
        named_sync(1, NC);
        for (int i = tid; i < n; i += NC) {
            const uint32_t k = order_key(vals[(size_t)i * stride]);
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
        }
        named_sync(1, NC);
        if (warp == 0) {
            // the bin holding the need-th largest key: lane l sums bins 255-8l .. 248-8l,
            // a prefix sum from the top finds the lane, the lane finds the bin
            const int need = ctl[4 + pass];
            int hb[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                hb[j] = hist[255 - 8 * lane - j];
                sum += hb[j];
            }
            int x = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int before = x - sum;
            if (before < need && need <= x) {
                int cum = before;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + hb[j] >= need) {
                        ctl[0] = 255 - 8 * lane - j;
                        ctl[5 + pass] = need - cum;
                        ctl[9] = ctl[4] - need + cum + hb[j];
                        break;
                    }
                    cum += hb[j];
                }
            }
        }
        named_sync(1, NC);
        prefix |= (uint32_t)ctl[0] << shift;
        mask |= 255u << shift;
        if (ctl[9] <= NC) {
            // every key >= the bin's lower bound, one per thread
            for (int i = tid; i < n; i += NC) {
                const float v = vals[(size_t)i * stride];
                if (order_key(v) >= prefix) gk[atomicAdd(&ctl[2], 1)] = cand_key(v, idx ? idx[i] : base + i);
            }
            named_sync(1, NC);
            rank_keys(gk, ctl[2], Ke, K, out_v, out_i);
            return;
        }
    }
    // after four passes prefix is the K-th largest key: every larger key (in any order),
    // then the equal keys with the lowest indices, from contiguous per-thread segments
    // placed by an exclusive prefix sum of their counts
    const uint32_t kth = prefix;
    const int take_eq = ctl[8];
    const int n_gt = Ke - take_eq;
    for (int i = tid; i < n; i += NC) {
        const float v = vals[(size_t)i * stride];
        if (order_key(v) > kth) gk[atomicAdd(&ctl[2], 1)] = cand_key(v, idx ? idx[i] : base + i);
    }
    const int seg = (n + NC - 1) / NC, lo = tid * seg, hi = lo + seg < n ? lo + seg : n;
    int c = 0;
    for (int i = lo; i < hi; ++i) c += order_key(vals[(size_t)i * stride]) == kth;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) cnt[warp] = x;
    named_sync(1, NC);
    int off = x - c;
    for (int w = 0; w < warp; ++w) off += cnt[w];
    for (int i = lo; i < hi && off < take_eq; ++i) {
        const float v = vals[(size_t)i * stride];
        if (order_key(v) == kth) gk[n_gt + off++] = cand_key(v, idx ? idx[i] : base + i);
    }
    named_sync(1, NC);
    rank_keys(gk, Ke, Ke, K, out_v, out_i);
}

// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014) as a counter-based generator: draw `counter` of `seed` is the output for
// state seed + (counter + 1) * gamma; its top 53 bits as a double in [0, 1).
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t counter) {
    uint64_t z = seed + (counter + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
__device__ __forceinline__ double uniform53(uint64_t seed, uint64_t counter) {
    return (double)(splitmix64(seed, counter) >> 11) * (1.0 / 9007199254740992.0);
}

// Consumer threads (named barrier 1): the K best entries, sorted, of L lists of K
// entries each in global memory (list c at part_v / part_i [c * K ..]), every list
// sorted by value descending then index ascending, the lists' index ranges disjoint.
// No entry worse than the K-th best list head can be among the K best, so only each
// list's prefix down to that head is kept and selected from (by rank counting when
// the kept entries fit one per thread, else by block_topk).  sm: 2 * L * K words of
// scratch (8-byte aligned); scratch: as for block_topk.
static __device__ __noinline__ void merge_candidate_lists(const float *part_v, const int *part_i, int L, int K,
                                                          uint64_t *sm, float *out_v, int *out_i, int *scratch) {
    constexpr int NC = kConsumerWarps * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the K-th best list head (every list when there are fewer than K)
    uint64_t tkey = 0;
    if (L >= K && L <= NC) {
        if (tid < L) sm[tid] = cand_key(__ldcg(part_v + (size_t)tid * K), __ldcg(part_i + (size_t)tid * K));
        named_sync(1, NC);
        rank_keys(sm, L, K, K, out_v, out_i);
        tkey = cand_key(out_v[K - 1], out_i[K - 1]);
    } else if (L > NC) {
        float *hv = reinterpret_cast<float *>(sm);
        int *hx = reinterpret_cast<int *>(hv + L);
        for (int c = tid; c < L; c += NC) {
            hv[c] = __ldcg(part_v + (size_t)c * K);
            hx[c] = __ldcg(part_i + (size_t)c * K);
        }
        named_sync(1, NC);
        block_topk(hv, 1, hx, 0, L, K, out_v, out_i, scratch);
        tkey = cand_key(out_v[K - 1], out_i[K - 1]);
    }
    // the kept prefixes of this thread's contiguous lists (their first 8 entries loaded
    // at once: the prefixes are short), then a block prefix sum of their lengths
    const int seg = (L + NC - 1) / NC, lo = tid * seg, hi = lo + seg < L ? lo + seg : L;
    int cnt = 0;
    for (int c = lo; c < hi; ++c) {
        int m = 0;
        bool more = true;
        while (more && m < K) {
            uint64_t b[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                b[j] = m + j < K ? cand_key(__ldcg(part_v + (size_t)c * K + m + j), __ldcg(part_i + (size_t)c * K + m + j)) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                more = more && m < K && b[j] >= tkey;
                m += more;
            }
        }
        cnt += m;
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    int *wsum = scratch + 256;   // free between the selections
    named_sync(1, NC);
    if (lane == 31) wsum[warp] = x;
    named_sync(1, NC);
    int off = x - cnt, total = 0;
    for (int w = 0; w < kConsumerWarps; ++w) {
        if (w < warp) off += wsum[w];
        total += wsum[w];
    }
    // kept entries as keys to rank, or (more than one per thread) as values and indices
    // in list order for the radix select
    float *kv = reinterpret_cast<float *>(sm);
    int *ki = reinterpret_cast<int *>(kv + total);
    for (int c = lo; c < hi; ++c)
        for (int m = 0; m < K; ++m) {
            const float v = __ldcg(part_v + (size_t)c * K + m);
            const int i = __ldcg(part_i + (size_t)c * K + m);
            const uint64_t k = cand_key(v, i);
            if (k < tkey) break;
            if (total <= NC) {
                sm[off] = k;
            } else {
                kv[off] = v;
                ki[off] = i;
            }
            ++off;
        }
    named_sync(1, NC);
    if (total <= NC)
        rank_keys(sm, total, total < K ? total : K, K, out_v, out_i);
    else
        block_topk(kv, 1, ki, 0, total, K, out_v, out_i, scratch);
}

// One warp: the id drawn from K (<= 64) candidates sorted by value: weights
// exp((v - v_max) / temperature), the smallest prefix reaching top_p of their sum,
// the first whose running sum exceeds u times the kept sum.  Lane l holds candidates
// l and l + 32; the running sums are a warp prefix sum.
static __device__ __noinline__ int warp_sample(const float *cv, const int *ci, int K, float temperature,
                                               float top_p, double u) {
    const int lane = threadIdx.x & 31;
    const float v0 = cv[0];
    auto weight = [&](int j) {
        return (j < K && cv[j] != -INFINITY) ? expf((cv[j] - v0) / temperature) : 0.f;
    };
    float c0 = weight(lane), c1 = weight(lane + 32);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, c0, o), y1 = __shfl_up_sync(0xffffffffu, c1, o);
        if (lane >= o) {
            c0 += y0;
            c1 += y1;
        }
    }
    c1 += __shfl_sync(0xffffffffu, c0, 31);
    const float total = __shfl_sync(0xffffffffu, K > 32 ? c1 : c0, (K > 32 ? K - 33 : K - 1) & 31);
    // the top-p prefix: the first running sum reaching top_p of the total
    const unsigned r0 = __ballot_sync(0xffffffffu, lane < K && c0 >= top_p * total);
    const unsigned r1 = __ballot_sync(0xffffffffu, lane + 32 < K && c1 >= top_p * total);
    const int m = r0 ? __ffs(r0) : (r1 ? 32 + __ffs(r1) : K);
    const float z = __shfl_sync(0xffffffffu, m > 32 ? c1 : c0, (m - 1) & 31);
    const float t = (float)(u * (double)z);
    const unsigned p0 = __ballot_sync(0xffffffffu, lane < m && c0 > t);
    const unsigned p1 = __ballot_sync(0xffffffffu, lane + 32 < m && c1 > t);
    const int pick = p0 ? __ffs(p0) - 1 : (p1 ? 32 + __ffs(p1) - 1 : m - 1);
    return ci[pick];
}

// ---------------------------------------------------------------------------------
// Attention of one (kv group, split) on shared-memory tiles.
// Ks/Vs: n cached rows in the cache type (row n_old already holds position p when the
// split owns it); qs: the G query heads (normalised, rotated), fp32; sc: [G][CM]
// scratch.  Outputs the split's unnormalised output po[G][HD], max pm[G], sum pl[G].
// Threads: kAttnWarps warps (the caller's first kAttnWarps * 32 threads).
// ---------------------------------------------------------------------------------
template <typename KT, int HD, int NW>
__device__ __forceinline__ void attn_split(const KT *Ks, const KT *Vs, const float *qs, int G, int n, int CM,
                                           float scale, float *sc, float *po, float *pm, float *pl, int bar_id) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NT = NW * 32;
    // scores: a group of LPP lanes per position, 16 bytes of the key row per lane
    constexpr int EPL = 16 / (int)sizeof(KT);     // key elements per lane
    constexpr int LPP = HD / EPL;                 // lanes per position (8 or 16 for bf16)
    constexpr int PPW = 32 / LPP;                 // positions per warp per pass
    const int sub = lane / LPP, l8 = lane % LPP;
    for (int j0 = warp * PPW; j0 < n; j0 += NW * PPW) {
        const int j = j0 + sub;
        const int jj = j < n ? j : n - 1;
        float kf[EPL];
        Elem<KT>::unpack(*reinterpret_cast<const uint4 *>(Ks + (size_t)jj * HD + l8 * EPL), kf);
        for (int hh = 0; hh < G; ++hh) {
            // this lane's EPL query values as float4 loads (scalar loads: 2-way bank conflicts)
            float q[EPL];
#pragma unroll
            for (int e = 0; e < EPL; e += 4) {
                const float4 q4 = *reinterpret_cast<const float4 *>(qs + hh * HD + l8 * EPL + e);
                q[e] = q4.x;
                q[e + 1] = q4.y;
                q[e + 2] = q4.z;
                q[e + 3] = q4.w;
            }
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) d = fmaf(q[e], kf[e], d);
#pragma unroll
            for (int o = LPP / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (l8 == 0 && j < n) sc[hh * CM + j] = d * scale;
        }
    }
    named_sync(bar_id, NT);
    for (int hh = warp; hh < G; hh += NW) {
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
    named_sync(bar_id, NT);
    // P.V: thread per (head, pair of dims); positions in order, 4 independent partial sums
    for (int idx = tid; idx < G * HD / 2; idx += NT) {
        const int hh = idx / (HD / 2), d = (idx % (HD / 2)) * 2;
        const float *p = sc + hh * CM;
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f, e0 = 0.f, e1 = 0.f;
        int j = 0;
        for (; j + 4 <= n; j += 4) {
            const float2 v0 = Elem<KT>::load2(Vs + (size_t)j * HD, d);
            const float2 v1 = Elem<KT>::load2(Vs + (size_t)(j + 1) * HD, d);
            const float2 v2 = Elem<KT>::load2(Vs + (size_t)(j + 2) * HD, d);
            const float2 v3 = Elem<KT>::load2(Vs + (size_t)(j + 3) * HD, d);
            a0 = fmaf(p[j], v0.x, a0);
            a1 = fmaf(p[j], v0.y, a1);
            b0 = fmaf(p[j + 1], v1.x, b0);
            b1 = fmaf(p[j + 1], v1.y, b1);
            c0 = fmaf(p[j + 2], v2.x, c0);
            c1 = fmaf(p[j + 2], v2.y, c1);
            e0 = fmaf(p[j + 3], v3.x, e0);
            e1 = fmaf(p[j + 3], v3.y, e1);
        }
        for (; j < n; ++j) {
            const float2 v0 = Elem<KT>::load2(Vs + (size_t)j * HD, d);
            a0 = fmaf(p[j], v0.x, a0);
            a1 = fmaf(p[j], v0.y, a1);
        }
        po[hh * HD + d] = (a0 + b0) + (c0 + e0);
        po[hh * HD + d + 1] = (a1 + b1) + (c1 + e1);
    }
}

// Row of the RoPE tables for frequency m.  Interleaved multimodal RoPE deals the
// frequencies to the position streams t, h, w in turn while the h and w sections (mh
// frequencies each) have room, the rest to t: frequency m < 3 mh takes stream m % 3.
// stage: [3][stride] per-stream positions of the staged prompt (position index p), or
// null for the single position r.  Clamped into the table (the host validates).
__device__ __forceinline__ int rope_row(int m, int mh, const int *stage, int stride, int p, int r, int rows) {
    if (stage) r = stage[(m < 3 * mh ? m % 3 : 0) * stride + p];
    return r < 0 ? 0 : (r >= rows ? rows - 1 : r);
}

// QK-RMSNorm (if gammas are given) and RoPE at position p of the G query heads in
// qs and of the key in kn; cos/sin row in rc ([HD/2] cos then [HD/2] sin).
template <int HD, int NW>
__device__ __forceinline__ void qk_norm_rope(float *qs, float *kn, int G, const float *q_gamma, const float *k_gamma,
                                             float eps, const float *rc, int bar_id) {
    constexpr int HALF = HD / 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (q_gamma) {
        for (int hh = warp; hh <= G; hh += NW) {
            float *v = hh < G ? qs + hh * HD : kn;
            const float *gam = hh < G ? q_gamma : k_gamma;
            float ss = 0.f;
            for (int i = lane; i < HD; i += 32) ss = fmaf(v[i], v[i], ss);
            ss = warp_sum(ss);
            const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
            for (int i = lane; i < HD; i += 32) v[i] = v[i] * inv * gam[i];
        }
        named_sync(bar_id, NW * 32);
    }
    for (int idx = tid; idx < (G + 1) * HALF; idx += NW * 32) {
        const int hh = idx / HALF, m = idx % HALF;
        float *v = hh < G ? qs + hh * HD : kn;
        const float c = rc[m], si = rc[HALF + m];
        const float x0 = v[m], x1 = v[m + HALF];
        v[m] = x0 * c - x1 * si;
        v[m + HALF] = x1 * c + x0 * si;
    }
    named_sync(bar_id, NW * 32);
}

}  // namespace qd

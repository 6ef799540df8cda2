// Persistent decode step: the whole per-token step of the decoder in one cooperative
// launch with one CTA per SM.
//
// Sources (page title, section):
//  - "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile and graph-replay entries:
//    the step is a chain of small dependent operations per layer whose launch and
//    synchronisation costs dominate at batch 1; replaying it as a graph helped only a
//    little.  Here the chain lives inside one kernel: each phase waits only for the
//    words it reads, and each CTA's producer warp streams that CTA's slice of every
//    phase's weights (and its attention K/V tile) through one shared-memory ring
//    without waiting on them, so HBM keeps streaming while the phases synchronise.
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation", and "Audio8-ASR: dynamic KV-cache buckets", section "Implemented
//    dynamic window mechanism": the arithmetic of each phase.
//
// Phases of layer l:
//   A  qkv = [Wq;Wk;Wv] RMSNorm(x)   (layer 0 also resolves the step input)
//   B  attention: CTA i < kv_heads * splits takes (group, split) i; QK-norm, RoPE, KV
//      append, scores/softmax/P.V of the split -> the split's partial; then the
//      split CTAs of a group merge the partials, each a slice of the group's columns
//   C  x += Wo o
//   D  act = silu(Wg x^) * (Wu x^), x^ = RMSNorm(x)
//   E  x += Wd act
// then the head: y = RMSNorm(x), logits, penalty, EOS mask, argmax (last CTA reduces).
//
// Between phases.  Every vector a phase hands to other CTAs (qkv, the attention
// partials and merged output, x after C and after E, act) is written once per launch
// into its own buffer of 64-bit words {launch sequence number, value}, one buffer per
// layer and phase, with one relaxed 64-bit store per value.  A reader polls the words
// it needs until their sequence number is the launch's: the data and its readiness
// travel in one access, no barrier round trip is needed, and a word is never rewritten
// within a launch.
//
// The GEMV phases split K over the consumer warps: warp w owns a contiguous chunk of
// the input vector's columns and polls exactly those words, straight into registers,
// so it can start on its rows as soon as its own chunk has arrived.  The chunk's dot
// products with the rows of each ring stage run on the tensor cores (mma.sync
// m16n8k16: 16 rows x 16 columns per instruction, the input as two bf16 parts, or, for
// 8-bit rows, as two f16 parts against the exactly converted codes, one block scale
// per lane and 32 columns) on bf16 and 8-bit weights, and as per-lane FMAs with one
// transposing butterfly per stage on fp32 weights; after the last stage one CTA
// barrier lets a thread per row add the warps' chunk sums in warp order.  RMSNorm is a
// scalar per vector, so W (g * x * r) is computed as r * W (g * x): the chunk sums of
// squares travel beside the row partials and r is applied by the row's thread.
#include <cuda_fp16.h>

#include <type_traits>

#include "decode_common.cuh"

namespace qd {

// Phase timeline (built only with -DQD_STEP_TRACE, by step_timeline.py): thread 0 of
// every CTA records %globaltimer at the phase boundaries of one layer.  Slots: 4 ph + 0
// phase start, + 1 input gathered, + 2 GEMV done, + 3 rows published (ph 0 = QKV,
// 1 = O-projection, 2 = gate/up, 3 = down); 16 q/k/v polled, 17 attention done,
// 18 split partial published, 19 merged output published; 22 next layer's input
// gathered.  The product build compiles none of it.
#ifdef QD_STEP_TRACE
__device__ unsigned long long g_step_trace[kStepTraceCtas][kStepTraceSlots];
__device__ int g_step_trace_layer = 3;
#define QD_TS(l, k)                                                                                     \
    do {                                                                                                \
        if ((l) == g_step_trace_layer && threadIdx.x == 0 && blockIdx.x < kStepTraceCtas) {             \
            unsigned long long t_;                                                                      \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                      \
            g_step_trace[blockIdx.x][(k)] = t_;                                                         \
        }                                                                                               \
    } while (0)
#else
#define QD_TS(l, k) do { } while (0)
#endif

constexpr int kNW = kConsumerWarps;          // consumer warps
constexpr int kNC = kNW * 32;                // consumer threads
constexpr int kGMax = kStepGroupMax;         // q heads per kv head handled by the step kernel

__host__ __device__ constexpr int pow2_ceil(int v) { return v <= 1 ? 1 : 2 * pow2_ceil((v + 1) / 2); }

// Grid barrier over all CTAs (consumer threads of every CTA arrive).  Thread 0
// publishes the CTA's writes with a release reduction and polls with acquire loads,
// for at most kWaitLimitNs.  Returns false on timeout (uniform across the CTA).
__device__ __forceinline__ bool grid_sync(unsigned *counter, unsigned &epoch, int *flag) {
    named_sync(1, kNC);
    ++epoch;
    if (threadIdx.x == 0) {
        const unsigned target = epoch * gridDim.x;
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
        const unsigned long long t0 = cycles_now();
        int ok = 1;
        while (true) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= target) break;
            if (cycles_now() - t0 > wait_cycles(kWaitLimitNs)) {
                ok = 0;
                break;
            }
        }
        *flag = ok;
    }
    named_sync(1, kNC);
    return *flag != 0;
}

// ---------------------------------------------------------------- tagged words
// {seq, value}: the value's bits low, the launch's sequence number high.  A new
// handle's words are all zero and no launch has sequence number 0.
__device__ __forceinline__ void st_tag(uint64_t *p, float v, uint32_t seq) {
    const uint64_t w = ((uint64_t)seq << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ void ld_tagged2(const uint64_t *p, uint64_t &a, uint64_t &b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Advance the launch sequence number from `seq` (the value this launch read) to the
// next non-zero value, exactly once however many threads of the launch call it.
__device__ __forceinline__ void advance_seq(unsigned *p, uint32_t seq) {
    (void)atomicCAS(p, seq, seq + 1u == 0u ? 1u : seq + 1u);
}

// One thread: the N consecutive words at p (16-byte aligned when N is even) once all
// carry `seq`; every still-stale word is re-polled together (one round trip per poll),
// for at most kWaitLimitNs.  False on timeout.
template <int N>
__device__ __forceinline__ bool poll_tagged(const uint64_t *p, uint32_t seq, float *v) {
    uint64_t w[N];
    if constexpr (N % 2 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 2) ld_tagged2(p + e, w[e], w[e + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) w[e] = ld_tagged(p + e);
    }
    unsigned pending = 0;
#pragma unroll
    for (int e = 0; e < N; ++e)
        if ((uint32_t)(w[e] >> 32) != seq) pending |= 1u << e;
    unsigned long long t0 = 0;
    while (pending) {
        const unsigned long long t = cycles_now();
        if (t0 == 0) t0 = t;
        else if (t - t0 > wait_cycles(kWaitLimitNs)) return false;
#pragma unroll
        for (int e = 0; e < N; ++e)
            if ((pending >> e) & 1u) w[e] = ld_tagged(p + e);
#pragma unroll
        for (int e = 0; e < N; ++e)
            if ((uint32_t)(w[e] >> 32) == seq) pending &= ~(1u << e);
    }
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = __uint_as_float((uint32_t)w[e]);
    return true;
}

// One thread: n <= N scattered words, addr(i) the address of word i, all loaded at
// once and every still-stale word re-polled together until each carries `seq`, for
// at most kWaitLimitNs.  False on timeout.
template <int N, typename Addr>
__device__ __forceinline__ bool poll_batch(int n, uint32_t seq, Addr addr, float *v) {
    static_assert(N <= 32, "pending mask");
    uint64_t w[N];
    uint32_t pending = 0;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n) w[i] = ld_tagged(addr(i));
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n && (uint32_t)(w[i] >> 32) != seq) pending |= 1u << i;
    unsigned long long t0 = 0;
    while (pending) {
        const unsigned long long t = cycles_now();
        if (t0 == 0) t0 = t;
        else if (t - t0 > wait_cycles(kWaitLimitNs)) return false;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((pending >> i) & 1u) w[i] = ld_tagged(addr(i));
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (((pending >> i) & 1u) && (uint32_t)(w[i] >> 32) == seq) pending &= ~(1u << i);
    }
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (i < n) v[i] = __uint_as_float((uint32_t)w[i]);
    return true;
}

struct TagSeg {                    // dst[i] = value of src[i], i < n
    const uint64_t *src;
    int n;
    float *dst;
};
// Consumer threads: the values of a tagged vector once its words carry `seq`, into
// shared memory (each thread a batch of words in flight, stale words re-polled
// together), for at most kWaitLimitNs.  False (uniform across the CTA) on timeout.
// Ends with a consumer barrier.
__device__ __noinline__ bool gather_tagged(const uint64_t *src, int n, float *dst, uint32_t seq) {
    constexpr int B = 8;
    const int tid = threadIdx.x;
    bool ok = true;
    unsigned long long t0 = 0;
    for (int base = tid; base < n; base += B * kNC) {
        uint64_t w[B];
        unsigned pending = 0;
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = base + k * kNC;
            w[k] = i < n ? ld_tagged(src + i) : (uint64_t)seq << 32;
            if ((uint32_t)(w[k] >> 32) != seq) pending |= 1u << k;
        }
        while (pending && ok) {
            const unsigned long long t = cycles_now();
            if (t0 == 0) t0 = t;
            else if (t - t0 > wait_cycles(kWaitLimitNs)) ok = false;
#pragma unroll
            for (int k = 0; k < B; ++k)
                if ((pending >> k) & 1u) w[k] = ld_tagged(src + base + k * kNC);
#pragma unroll
            for (int k = 0; k < B; ++k)
                if ((uint32_t)(w[k] >> 32) == seq) pending &= ~(1u << k);
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int i = base + k * kNC;
            if (i < n) dst[i] = __uint_as_float((uint32_t)w[k]);
        }
    }
    return !named_sync_or(1, kNC, !ok);
}

// Stage a vector of weights (gamma) into shared memory (consumer threads).
__device__ __forceinline__ void stage_vec(float *dst, const float *src, int n) {
    for (int i = threadIdx.x * 4; i < n; i += kNC * 4)
        *reinterpret_cast<float4 *>(dst + i) = *reinterpret_cast<const float4 *>(src + i);
}

__device__ __forceinline__ void cta_rows(int rows, int unit, int &r0, int &nr) {
    const int units = rows / unit;
    const int u0 = (int)((long long)units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)units * (blockIdx.x + 1) / gridDim.x);
    r0 = u0 * unit;
    nr = (u1 - u0) * unit;
}

// ---------------------------------------------------------------- K-chunk GEMV
// E consecutive elements at p as floats, in 16-, 8- or 4-byte pieces (p aligned to
// the piece).
template <typename WT, int E>
__device__ __forceinline__ void load_elems(const WT *p, float *f) {
    constexpr int B = E * (int)sizeof(WT);
    constexpr int PER4 = 4 / (int)sizeof(WT);
    if constexpr (B % 16 == 0) {
#pragma unroll
        for (int i = 0; i < B / 16; ++i)
            Elem<WT>::unpack(reinterpret_cast<const uint4 *>(p)[i], f + i * 4 * PER4);
    } else if constexpr (B % 8 == 0) {
#pragma unroll
        for (int i = 0; i < B / 8; ++i) {
            const uint2 u = reinterpret_cast<const uint2 *>(p)[i];
            if constexpr (sizeof(WT) == 2) {
                f[4 * i] = bf16lo(u.x); f[4 * i + 1] = bf16hi(u.x);
                f[4 * i + 2] = bf16lo(u.y); f[4 * i + 3] = bf16hi(u.y);
            } else {
                f[2 * i] = __uint_as_float(u.x); f[2 * i + 1] = __uint_as_float(u.y);
            }
        }
    } else if constexpr (B % 4 != 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = Elem<WT>::load(p, e);
    } else {
#pragma unroll
        for (int i = 0; i < B / 4; ++i) {
            const uint32_t u = reinterpret_cast<const uint32_t *>(p)[i];
            if constexpr (sizeof(WT) == 2) {
                f[2 * i] = bf16lo(u); f[2 * i + 1] = bf16hi(u);
            } else {
                f[i] = __uint_as_float(u);
            }
        }
    }
}

// Transposing butterfly over a warp: lane l holds RP values (RP a power of two <= 32);
// afterwards lane l holds the sum over the 32 lanes of value l / (32 / RP).  Each
// level keeps half of the values and receives the partner's other half.
template <int RP, int O = 16>
__device__ __forceinline__ float treduce(float *v, int lane) {
    if constexpr (RP == 1) {
        float s = v[0];
#pragma unroll
        for (int o = O; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        return s;
    } else {
        constexpr int H = RP / 2;
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const float send = up ? v[i] : v[i + H];
            const float keep = up ? v[i + H] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        return treduce<H, O / 2>(v, lane);
    }
}

// Ring stages of the persistent step: a compile-time count, so a stage's slot and
// phase parity are cheap to compute (the host checks that the layout has exactly it).
constexpr int kStepStages = kStepRingStages;

// Consumer side of stage sidx: a non-blocking test first (the weights are normally
// there long before), then the bounded wait.  Null on timeout.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ const uint8_t *stage_get(const Ring &R, uint32_t sidx) {
    const uint32_t slot = sidx % kStepStages, par = (sidx / kStepStages) & 1u;
    if (!mbar_test_wait(&R.full[slot], par) && !mbar_wait_bounded(&R.full[slot], par)) return nullptr;
    return R.base + (size_t)slot * kSlotBytes;
}
__device__ __forceinline__ void stage_put(const Ring &R, uint32_t sidx, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[sidx % kStepStages]);
}

__host__ __device__ constexpr int min_c(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int max_c(int a, int b) { return a > b ? a : b; }

// Consumer warp: the CTA's `nrows` rows of W, arriving in ring stages of `rps` rows,
// against this warp's K-chunk: nc column chunks of 32 x EL, whose values (already
// scaled by the RMSNorm gamma) the warp keeps in shared memory at xw, chunk c at
// xw[c * 32 EL ..], lane l's columns at l EL.  Rows go in groups of 8 (all loads of a
// group in flight at once), the chunks of a group in a rolled loop, then one
// transposing butterfly; part[r] (this warp's row of the partial-sum table) gets the
// chunk's sum of row r.  One body serves every phase: it runs for every phase of
// every layer, and what the instruction cache holds, not trip counts, sets its speed.
// False if a stage never arrived.
template <typename WT, int EL>
__device__ __forceinline__ bool kc_gemv(const Ring &R, uint32_t &sidx, int nrows, int rps, uint32_t row_bytes,
                                        int colw, int nc, const float *xw, float *part) {
    const int lane = threadIdx.x & 31;
    const int nst = (nrows + rps - 1) / rps;
#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
        const uint8_t *sb = stage_get(R, sidx + st);
        if (!sb) return false;
        const int n = min_c(rps, nrows - st * rps);
#pragma unroll 1
        for (int g0 = 0; g0 < n; g0 += 8) {
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.f;
#pragma unroll 1
            for (int c = 0; c < nc; ++c) {
                float xv[EL];
                load_elems<float, EL>(xw + c * 32 * EL + lane * EL, xv);
                // every load unconditional (rows past n re-read row n - 1, counted zero below)
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = g0 + r < n ? g0 + r : n - 1;
                    float f[EL];
                    load_elems<WT, EL>(reinterpret_cast<const WT *>(sb + (size_t)row * row_bytes) + colw + c * 32 * EL +
                                           lane * EL,
                                       f);
#pragma unroll
                    for (int e = 0; e < EL; ++e) acc[r] = fmaf(f[e], xv[e], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = g0 + r < n ? acc[r] : 0.f;
            const float v = treduce<8>(acc, lane);
            const int row = g0 + lane / 4;
            if ((lane & 3) == 0 && row < n) part[st * rps + row] = v;
        }
        stage_put(R, sidx + st, lane);
    }
    sidx += nst;
    return true;
}

// Row pitch in the ring of the bf16 layer phases: each row 16 bytes past a multiple of
// 128, so the 8 rows a tensor-core fragment reads at one column fall in 8 different
// 16-byte bank groups (conflict-free), and the rows of a stage that fit in a slot.
__host__ __device__ constexpr uint32_t mma_pitch(int K) { return (uint32_t)(K * 2 + 16); }
__host__ __device__ constexpr int mma_rps(int K) { return kSlotBytes / (int)mma_pitch(K); }

// Producer: rows [0, nrows) of a row-major matrix into ring stages of `rps` rows, row
// i of a stage at i * pitch (one bulk copy per row).
__device__ __forceinline__ bool produce_rows_pitched(const Ring &R, uint32_t &sidx, const uint8_t *src, int nrows,
                                                     uint32_t row_bytes, uint32_t pitch, int rps, uint64_t pol) {
    for (int r = 0; r < nrows; r += rps) {
        const int slot = (int)(sidx % (uint32_t)kStepStages);
        const uint32_t use = sidx / (uint32_t)kStepStages;
        if (use > 0 && !mbar_wait_bounded(&R.empty[slot], (use - 1) & 1)) return false;
        const int n = nrows - r < rps ? nrows - r : rps;
        mbar_arrive_expect_tx(&R.full[slot], n * row_bytes);
        uint8_t *dst = R.base + (size_t)slot * kSlotBytes;
        for (int i = 0; i < n; ++i)
            bulk_copy_g2s(dst + (size_t)i * pitch, src + (size_t)(r + i) * row_bytes, row_bytes, &R.full[slot], pol);
        ++sidx;
    }
    return true;
}

// d += a b for one m16n8k16 tile (bf16 operands, fp32 accumulation)
__device__ __forceinline__ void mma_bf16(float &d0, float &d1, float &d2, float &d3, uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The bf16 form of kc_gemv: the same partial sums (rows of the CTA's stages against
// this warp's K-chunk [colw, colw + 16 nks)) from one m16n8k16 tensor-core product per
// 16 rows x 16 columns.  The rows are the tile's M; its N holds the fp32 input as two
// bf16 columns, x0 = bf16(x) and x1 = bf16(x - x0) (16 significant bits: |x - x0 - x1|
// <= 2^-17 |x|), the other six columns zero, so row r's sum is D[r][0] + D[r][1]
// (fp32 accumulation of exact bf16 x bf16 products).  xp: the warp's chunk as the two
// bf16 parts in shared memory, k-step by k-step: 8 words of x0's 16 columns, then 8 of
// x1's (the two parts' loads fall in different banks).  At batch 1 this is not
// about tensor throughput: one instruction replaces the conversions, FMAs and shuffle
// reduction of 16 rows x 16 columns, whose issue and latency bound this phase on the
// CUDA cores.  (A third part, x - x0 - x1, makes the split exact; it measured 3 %
// slower per step and left the difference to the CUDA-core step at the same ~1e-4,
// which the tensor cores' accumulation sets.)
__device__ __forceinline__ bool kc_gemv_mma(const Ring &R, uint32_t &sidx, int nrows, int rps, uint32_t pitch,
                                            int colw, int nks, const uint32_t *xp, float *part) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int nst = (nrows + rps - 1) / rps;
    const uint32_t *xb = xp + (g < 2 ? g : 0) * 8;   // N column g < 2: part g of each k-step
    const bool live = g < 2;
#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
        const uint8_t *sb = stage_get(R, sidx + st);
        if (!sb) return false;
        const int n = min_c(rps, nrows - st * rps);
#pragma unroll 1
        for (int r0 = 0; r0 < n; r0 += 16) {
            // rows past n re-read row n - 1 (results dropped below)
            const int ra = min_c(r0 + g, n - 1), rb = min_c(r0 + g + 8, n - 1);
            const uint8_t *pa = sb + (size_t)ra * pitch + (size_t)colw * 2 + t * 4;
            const uint8_t *pb = sb + (size_t)rb * pitch + (size_t)colw * 2 + t * 4;
            float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f, e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
#pragma unroll 4
            for (int ks = 0; ks < nks; ks += 2) {
                // two independent accumulators: k-steps ks (c) and ks + 1 (e)
                const uint32_t b0 = live ? xb[ks * 16 + t] : 0u, b1 = live ? xb[ks * 16 + t + 4] : 0u;
                const uint32_t b2 = live ? xb[ks * 16 + 16 + t] : 0u, b3 = live ? xb[ks * 16 + 20 + t] : 0u;
                const uint32_t *qa = reinterpret_cast<const uint32_t *>(pa + ks * 32);
                const uint32_t *qb = reinterpret_cast<const uint32_t *>(pb + ks * 32);
                mma_bf16(c0, c1, c2, c3, qa[0], qb[0], qa[4], qb[4], b0, b1);
                mma_bf16(e0, e1, e2, e3, qa[8], qb[8], qa[12], qb[12], b2, b3);
            }
            // columns 0 and 1 sit in lane t = 0
            if (t == 0) {
                if (r0 + g < n) part[st * rps + r0 + g] = (c0 + c1) + (e0 + e1);
                if (r0 + g + 8 < n) part[st * rps + r0 + g + 8] = (c2 + c3) + (e2 + e3);
            }
        }
        stage_put(R, sidx + st, lane);
    }
    sidx += nst;
    return true;
}

// ---- weight-only 8-bit rows (q8_row_bytes: K int8 codes, then K / 32 half scales)

// Marker of the 8-bit head's register slices: a lane holds 16 consecutive columns of
// each 512-column segment (the 16 codes of one 16-byte load).
struct Q8Code {};
template <> struct Elem<Q8Code> {
    static constexpr int kPer16B = 16;
};

// The four int8 codes of a 32-bit word as floats, lowest byte first.
__device__ __forceinline__ void q8_word(int u, float *f) {
    f[0] = (float)((u << 24) >> 24);
    f[1] = (float)((u << 16) >> 24);
    f[2] = (float)((u << 8) >> 24);
    f[3] = (float)(u >> 24);
}
__device__ __forceinline__ float q8_scale(const uint8_t *row, int K, int col) {
    return __half2float(*reinterpret_cast<const __half *>(row + K + (col >> 5) * 2));
}

// Row pitch in the ring of 8-bit layer rows (codes then scales), 16 bytes past a
// multiple of 32 words for every supported K (as mma_pitch: the 8 rows a fragment
// reads at one column fall in different bank groups), and the rows of a stage.
__host__ __device__ constexpr uint32_t q8_pitch(int K) { return q8_row_bytes(K) + 16; }
__host__ __device__ constexpr int q8_prs(int K) { return kSlotBytes / (int)q8_pitch(K); }

// d += a b for one m16n8k16 tile (f16 operands, fp32 accumulation)
__device__ __forceinline__ void mma_f16(float &d0, float &d1, float &d2, float &d3, uint32_t a0, uint32_t a1,
                                        uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The four int8 codes of a word (lowest byte first) as two f16x2 registers, (c0, c1)
// and (c2, c3), exactly: the code's sign bit flipped gives c + 128 in [0, 255]; placed
// under the exponent byte 0x64 it is the half 1024 + c + 128, and subtracting 1152
// leaves c.
__device__ __forceinline__ void q8_f16x4(uint32_t w, uint32_t &c01, uint32_t &c23) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c01) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c23) : "r"(b), "r"(0x64806480u));
}

// kc_gemv on 8-bit rows on the tensor cores: the same partial sums, per 16 rows and
// per group of KG k-steps (KG / 2 blocks of 32 columns) one m16n8k16 f16 product per
// k-step.  The codes are the tile's M x K, exact in f16; within a k-step lane t takes
// columns 4t .. 4t + 3 of its rows (one word) as the k slots 2t, 2t + 1, 2t + 8, 2t + 9,
// and the input goes through the same permutation.  N column 2j + p carries part p
// (x = x0 + x1, two f16 parts of the input times 2^e, e from the warp's largest
// magnitude so that neither part overflows nor loses its low bits) on block j of the
// group and zero elsewhere, so D[r][2j + p] is block j's sum of part p for row r and
// lane t holds block t's two sums: it scales them by row r's half scale of that block
// and accumulates; a 4-lane butterfly adds the blocks, and `post` = 2^-e undoes the
// input scaling.  xh, xl: the warp's K / 8 columns of x0 and x1 as f16, column order.
template <int KG>
__device__ __forceinline__ bool kc_gemv_q8_mma(const Ring &R, uint32_t &sidx, int nrows, int rps, int K, int colw,
                                               const __half *xh, const __half *xl, float post, float *part) {
    static_assert(KG == 4 || KG == 8, "k-steps per group");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int nst = (nrows + rps - 1) / rps;
    const uint32_t pitch = q8_pitch(K);
    const int ngroups = K / (kNW * 16 * KG);
    const int jb = g >> 1;                                   // the block this lane's N column carries
    const bool live = jb < KG / 2;
    const __half *xs = ((g & 1) ? xl : xh) + jb * 32 + 4 * t;
#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
        const uint8_t *sb = stage_get(R, sidx + st);
        if (!sb) return false;
        const int n = min_c(rps, nrows - st * rps);
#pragma unroll 1
        for (int r0 = 0; r0 < n; r0 += 16) {
            // rows past n re-read row n - 1 (results dropped below)
            const int ra = min_c(r0 + g, n - 1), rb = min_c(r0 + g + 8, n - 1);
            const uint8_t *pa = sb + (size_t)ra * pitch + colw + t * 4;
            const uint8_t *pb = sb + (size_t)rb * pitch + colw + t * 4;
            const __half *sca = reinterpret_cast<const __half *>(sb + (size_t)ra * pitch + K) + (colw >> 5) + t;
            const __half *scb = reinterpret_cast<const __half *>(sb + (size_t)rb * pitch + K) + (colw >> 5) + t;
            float acc_a = 0.f, acc_b = 0.f;
#pragma unroll 1
            for (int gq = 0; gq < ngroups; ++gq) {
                uint2 u0 = make_uint2(0u, 0u), u1 = make_uint2(0u, 0u);
                if (live) {
                    u0 = *reinterpret_cast<const uint2 *>(xs + gq * KG * 16);
                    u1 = *reinterpret_cast<const uint2 *>(xs + gq * KG * 16 + 16);
                }
                // two independent accumulators: even (c) and odd (e) k-steps
                float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f, e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
#pragma unroll
                for (int ks = 0; ks < KG; ++ks) {
                    const int kb = (gq * KG + ks) * 16;
                    uint32_t a0, a1, a2, a3;
                    q8_f16x4(*reinterpret_cast<const uint32_t *>(pa + kb), a0, a2);
                    q8_f16x4(*reinterpret_cast<const uint32_t *>(pb + kb), a1, a3);
                    const bool mine = (ks >> 1) == jb;
                    const uint32_t b0 = mine ? ((ks & 1) ? u1.x : u0.x) : 0u;
                    const uint32_t b1 = mine ? ((ks & 1) ? u1.y : u0.y) : 0u;
                    if (ks & 1)
                        mma_f16(e0, e1, e2, e3, a0, a1, a2, a3, b0, b1);
                    else
                        mma_f16(c0, c1, c2, c3, a0, a1, a2, a3, b0, b1);
                }
                if (t < KG / 2) {
                    const int blk = gq * (KG / 2);
                    acc_a = fmaf(__half2float(sca[blk]), (c0 + c1) + (e0 + e1), acc_a);
                    acc_b = fmaf(__half2float(scb[blk]), (c2 + c3) + (e2 + e3), acc_b);
                }
            }
            acc_a += __shfl_xor_sync(0xffffffffu, acc_a, 1);
            acc_b += __shfl_xor_sync(0xffffffffu, acc_b, 1);
            acc_a += __shfl_xor_sync(0xffffffffu, acc_a, 2);
            acc_b += __shfl_xor_sync(0xffffffffu, acc_b, 2);
            if (t == 0) {
                if (r0 + g < n) part[st * rps + r0 + g] = acc_a * post;
                if (r0 + g + 8 < n) part[st * rps + r0 + g + 8] = acc_b * post;
            }
        }
        stage_put(R, sidx + st, lane);
    }
    sidx += nst;
    return true;
}

// The head on 8-bit rows: each consumer warp takes whole rows (two at a time), a lane
// 16 codes of each 512-column segment against xr (Elem<Q8Code> slices), scaled per
// half block; one butterfly leaves row q's sum in lane 16 q; res[row] gets it.
template <int NSEG>
__device__ __forceinline__ bool gemv_consume_q8(const Ring &R, uint32_t &sidx, int nrows, int rps, int K,
                                                const float *xr, float *res) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rb = q8_row_bytes(K);
    for (int rbase = 0; rbase < nrows; rbase += rps) {
        const uint8_t *sbase = stage_get(R, sidx);
        if (!sbase) return false;
        const int n = nrows - rbase < rps ? nrows - rbase : rps;
        for (int r = warp; r < n; r += 2 * kNW) {
            float acc[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int rq = r + q * kNW;
                const uint8_t *rp = sbase + (size_t)(rq < n ? rq : r) * rb;
                float a2 = 0.f;
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(rp + sg * 512 + lane * 16);
                    float f[16];
                    q8_word((int)w.x, f);
                    q8_word((int)w.y, f + 4);
                    q8_word((int)w.z, f + 8);
                    q8_word((int)w.w, f + 12);
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) d = fmaf(f[e], xr[sg * 16 + e], d);
                    a2 = fmaf(q8_scale(rp, K, sg * 512 + lane * 16), d, a2);
                }
                acc[q] = rq < n ? a2 : 0.f;
            }
            const bool b4 = (lane & 16) != 0;
            float v = b4 ? acc[1] : acc[0];
            const float sx = b4 ? acc[0] : acc[1];
            v += __shfl_xor_sync(0xffffffffu, sx, 16);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            const int rq = r + (b4 ? kNW : 0);
            if ((lane & 15) == 0 && rq < n) res[rbase + rq] = v;
        }
        stage_put(R, sidx, lane);
        ++sidx;
    }
    return true;
}

// Sum over the consumer warps, in warp order, of entry i of a [kNW][ps] table.
__device__ __forceinline__ float warp_parts(const float *tab, int ps, int i) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kNW; ++w) v += tab[w * ps + i];
    return v;
}
// RMSNorm scale from the warps' chunk sums of squares.
__device__ __forceinline__ float rms_scale(const float *ss, int K, float eps) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kNW; ++w) t += ss[w];
    return rsqrtf(t / (float)K + eps);
}

// This lane's E columns of the step's input vector (token row of the embedding
// table, caller embedding, or staged prompt row), resolved from the description
// that thread 0 staged in misc_i.
template <typename WT, int E>
__device__ __forceinline__ void input_cols(const StepInputArgs &in, int K, int mode, int tok, int pos, bool bad, int col,
                                           float *v) {
    if (bad) {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = 0.f;
    } else if (mode == IN_EMBED || mode == IN_STAGED_EMBEDS) {
        const float *src = mode == IN_EMBED ? in.embed_in + col : in.stage_embeds + (size_t)pos * K + col;
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __ldcg(src + e);
    } else {
        load_elems<WT, E>(reinterpret_cast<const WT *>(in.table) + (size_t)tok * K + col, v);
    }
}

// Rotate-half RoPE of one head held across a warp: lane l holds elements
// [l E, l E + E); the partner element of the first half sits E * 16 further, in lane
// l ^ 16.  cs / sn: this lane's frequencies ((l & 15) E + e).
template <int E>
__device__ __forceinline__ void rope_lane(float *v, const float *cs, const float *sn, int lane) {
    const bool second = (lane & 16) != 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], 16);
        v[e] = second ? v[e] * cs[e] + o * sn[e] : v[e] * cs[e] - o * sn[e];
    }
}

// Per-head RMSNorm of one head held across a warp (E elements per lane).
template <int E>
__device__ __forceinline__ void head_norm(float *v, const float *gam, int hd, float eps) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)hd + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = v[e] * inv * gam[e];
}

template <typename T> __device__ __forceinline__ float round_to(float v);
template <> __device__ __forceinline__ float round_to<float>(float v) { return v; }
template <> __device__ __forceinline__ float round_to<__nv_bfloat16>(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// E values of one cache row in the cache type (one 16-, 8- or 4-byte store).
template <typename KT, int E>
__device__ __forceinline__ void store_row_elems(KT *dst, const float *v) {
#pragma unroll
    for (int e = 0; e < E; ++e) Elem<KT>::store(dst, e, v[e]);
}

// Scores, softmax and P.V of one warp's positions [jw0, jw0 + nwp) of the split, for
// the G query heads q (lane: E elements of each), in blocks of 8 positions with a
// running max and sum (the blocks in order).  Row jp (the new position) comes from kr /
// vr, the others from the shared-memory tiles.  Outputs the warp's unnormalised o, and
// per head its max and sum of exponentials (-inf and 0 for a warp without positions).
template <typename KT, int HD, int G>
__device__ __forceinline__ void warp_attention(const KT *Ks, const KT *Vs, const float (*q)[HD / 32], int jw0, int nwp,
                                               int jp, const float *kr, const float *vr, float scale,
                                               float (*o)[HD / 32], float *mh, float *lh) {
    constexpr int E = HD / 32;
    constexpr int RA = 8, LPV = 32 / RA;   // positions per block, lanes holding each score
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        mh[h] = -INFINITY;
        lh[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[h][e] = 0.f;
    }
#pragma unroll 1
    for (int b0 = 0; b0 < nwp; b0 += RA) {
        const int nb = nwp - b0 < RA ? nwp - b0 : RA;
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            // unconditional loads of a clamped row, the new position's row from the
            // register copy; dead positions count zero
            float acc[RA];
#pragma unroll
            for (int jj = 0; jj < RA; ++jj) {
                const int j = jw0 + b0 + (jj < nb ? jj : nb - 1);
                float kf[E];
                load_elems<KT, E>(Ks + (size_t)j * HD + lane * E, kf);
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) d = fmaf(q[h][e], j == jp ? kr[e] : kf[e], d);
                acc[jj] = jj < nb ? d : 0.f;
            }
            float sc = treduce<RA>(acc, lane);
            const bool live = lane / LPV < nb;
            sc = live ? sc * scale : -INFINITY;
            const float mn = fmaxf(mh[h], warp_max(sc));
            const float corr = __expf(mh[h] - mn);   // 0 for the first block
            const float ex = live ? __expf(sc - mn) : 0.f;
            lh[h] = lh[h] * corr + warp_sum(lane % LPV == 0 ? ex : 0.f);
#pragma unroll
            for (int e = 0; e < E; ++e) o[h][e] *= corr;
            mh[h] = mn;
            pr[h] = ex;
        }
#pragma unroll
        for (int jj = 0; jj < RA; ++jj) {
            // dead positions carry weight 0 and re-read a live row
            const int j = jw0 + b0 + (jj < nb ? jj : nb - 1);
            float vf[E];
            load_elems<KT, E>(Vs + (size_t)j * HD + lane * E, vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ph = __shfl_sync(0xffffffffu, pr[h], jj * LPV);
#pragma unroll
                for (int e = 0; e < E; ++e) o[h][e] = fmaf(ph, j == jp ? vr[e] : vf[e], o[h][e]);
            }
        }
    }
}

// Threads: kNW consumer warps and one producer warpgroup, whose first lane issues the
// weight stream.  Launched with 168 registers a thread (12 warps on one SM); the
// producer warpgroup gives back all but 40 of its registers and the consumers take
// them, 232 each: 128 x 40 + 256 x 232 = 384 x 168, the launch's whole register file.
constexpr int kStepThreads = (kNW + 4) * 32;
constexpr int kProducerRegs = 40, kConsumerRegs = 232;
static_assert(4 * 32 * kProducerRegs + kNW * 32 * kConsumerRegs == kStepThreads * 168, "register split");

template <typename WT, int HD, int KH, int KQ, int KF, int KVH, bool Q8 = false>
__global__ void __launch_bounds__(kStepThreads, 1) decode_step_kernel(const StepArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    typedef WT KT;
    // Q8: the layer matrices and heads as 8-bit rows (q8_row_bytes); the embedding table
    // and the cache stay WT
    using HT = typename std::conditional<Q8, Q8Code, WT>::type;   // the head's slices
    constexpr int EPL = Elem<HT>::kPer16B;
    constexpr int SEGW = 32 * EPL;
    constexpr int NS_H = KH / SEGW;                       // the head's segments per warp
    constexpr int ES = (int)sizeof(WT);
    constexpr int KV = KVH * HD;                                  // k (and v) rows
    constexpr int GQ = KQ / KV;                                   // q heads per kv head
    // stage shapes of the GEMV phases (rows per stage padded, stages per butterfly)
    // GEMV K-chunks: a warp holds K / 8 columns as chunks of 32 lanes x EL (EL from the
    // hidden size); the phases need NC0 <= NC1 <= NC2 chunks (one GEMV body each)
    constexpr int EL = KH / kNC;
    constexpr int NCA = KH / (256 * EL), NCQ = KQ / (256 * EL), NCF = KF / (256 * EL);
    constexpr int NCMAX = NCF;
    constexpr int XSW = NCMAX * 32 * EL;                         // floats of a warp's input slice
    static_assert(NCA == 1 && NCQ >= 1 && NCF >= NCQ && KQ == NCQ * 256 * EL && KF == NCF * 256 * EL, "chunks");
    static_assert(!Q8 || (KH % 512 == 0 && KQ % 512 == 0 && KF % 512 == 0), "8-bit rows: groups of 4 or 8 k-steps");
    constexpr int EH = HD / 32;
    constexpr int HALF = HD / 2;
    constexpr int PS = kStepRowsMax;
    static_assert(KH % kNC == 0 && KQ % kNC == 0 && KF % kNC == 0, "K-chunks of whole lanes");
    static_assert(GQ >= 1 && GQ <= kGMax && KQ == GQ * KV, "q heads per kv head");
    static_assert(NS_H >= 1 && NS_H <= 4 && KH == NS_H * SEGW, "head segments");
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_full);
    uint64_t *empty = full + a.nst;
    float *gsm = reinterpret_cast<float *>(smem + a.off_gsm);
    float *misc = reinterpret_cast<float *>(smem + a.off_misc);   // 64 words
    int *misc_i = reinterpret_cast<int *>(misc + 32);
    volatile int *ctl = reinterpret_cast<volatile int *>(misc_i + 16);   // [0] stop [1] issued [2] producer done
    int *flag = misc_i + 20;
    float *res = reinterpret_cast<float *>(smem + a.off_res);
    uint32_t *emw = reinterpret_cast<uint32_t *>(smem + a.off_emw);
    float *xin = reinterpret_cast<float *>(smem + a.off_xin);   // the head's gathered input
    float *kc_part = reinterpret_cast<float *>(smem + a.off_kc);  // [2][kNW][PS] row partials
    float *kc_ss = kc_part + 2 * kNW * PS;                          // [2][kNW] sums of squares
    float *xres = reinterpret_cast<float *>(smem + a.off_xres);    // residual rows of this CTA
    float *xs = reinterpret_cast<float *>(smem + a.off_xs);        // [kNW][ffn / kNW] input slices
    const Ring R{smem, full, empty, a.nst};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int G = GQ;
    const int hidden = KH, q_dim = KQ, kv_dim = KV;
    const int CM = a.chunk_max;

    // The step's position: the previous launch has completed, so it is final.
    const int p = a.st->pos;
    const int L = p + 1;
    const int C = attn_chunk(L);
    const int nsplit = attn_splits(L);
    if (!(p < a.S && C <= CM)) {
        // outside the bucket: the host never launches this; report it and leave
        if (blockIdx.x == 0 && tid == 0) atomicOr(&a.st->status, DEV_ERR_BAD_POS);
        return;
    }
    const bool has_item = (int)blockIdx.x < a.kvh * nsplit;
    const int ig = has_item ? (int)blockIdx.x / nsplit : 0;
    const int is = has_item ? (int)blockIdx.x % nsplit : 0;
    const int j0 = is * C;
    const int n_att = has_item ? (L - j0 < C ? L - j0 : C) : 0;
    const int n_old = has_item ? ((p - j0) < n_att ? (p - j0) : n_att) : 0;

    int r0_qkv, n_qkv, r0_x, n_x, r0_gu, n_gu, r0_hd, n_hd;
    cta_rows(q_dim + 2 * kv_dim, 1, r0_qkv, n_qkv);
    cta_rows(hidden, 1, r0_x, n_x);                  // rows of Wo and Wd: the residual rows this CTA owns
    cta_rows(2 * a.ffn, 2, r0_gu, n_gu);
    cta_rows(a.vocab, 1, r0_hd, n_hd);
    const uint32_t rb_h = (uint32_t)(hidden * ES), rb_q = (uint32_t)(q_dim * ES), rb_f = (uint32_t)(a.ffn * ES);
    const size_t layer_kv = (size_t)2 * kv_dim * a.S * ES;

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kNW);
        }
        ctl[0] = 0;
        ctl[1] = 0;
        ctl[2] = 0;
        misc_i[6] = 0;   // the head's wait for the emitted-set flag timed out
        fence_barrier_init();
    }
    __syncthreads();

    if (warp >= kNW) {
        // ---------------- producer: every phase's weights, in consumption order
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kProducerRegs) : "memory");
        if (warp == kNW && lane == 0) {
            const uint64_t pw = a.evict_last ? policy_evict_last() : policy_evict_first();
            const uint64_t pf = policy_evict_first();
            uint32_t sidx = 0;
            bool ok = true;
            for (int l = 0; l < a.n_layers && ok && !ctl[0]; ++l) {
                const LayerDev &Ld = a.layers[l];
                // bf16 layer rows at the tensor-core pitch; 8-bit and fp32 rows packed
                auto rows = [&](const void *w, int r0, int n, uint32_t rb, int K, int rps) {
                    if constexpr (Q8) {
                        const uint32_t qb = q8_row_bytes(K);
                        return produce_rows_pitched(R, sidx, reinterpret_cast<const uint8_t *>(w) + (size_t)r0 * qb,
                                                    n, qb, q8_pitch(K), q8_prs(K), pw);
                    } else if constexpr (sizeof(WT) == 2) {
                        return produce_rows_pitched(R, sidx, reinterpret_cast<const uint8_t *>(w) + (size_t)r0 * rb,
                                                    n, rb, mma_pitch(K), mma_rps(K), pw);
                    } else {
                        return produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(w) + (size_t)r0 * rb, n, rb,
                                            rps, pw);
                    }
                };
                ok = ok && rows(Ld.w_qkv, r0_qkv, n_qkv, rb_h, KH, a.rps_h);
                if (has_item) {
                    // K and V rows [j0, j0 + n_old) of this CTA's group: written by earlier steps
                    const uint8_t *kb = reinterpret_cast<const uint8_t *>(a.kv) + (size_t)l * layer_kv +
                                        ((size_t)ig * a.S + j0) * HD * ES;
                    const uint32_t bytes = (uint32_t)(n_old * HD * ES);
                    ok = ok && produce_block(R, sidx, kb, bytes, pf);
                    ok = ok && produce_block(R, sidx, kb + layer_kv / 2, bytes, pf);
                }
                ok = ok && rows(Ld.w_o, r0_x, n_x, rb_q, KQ, a.rps_q);
                ok = ok && rows(Ld.w_gu, r0_gu, n_gu, rb_h, KH, a.rps_h);
                ok = ok && rows(Ld.w_d, r0_x, n_x, rb_f, KF, a.rps_f);
            }
            if (ok && a.with_head && !ctl[0]) {
                const uint8_t *Wh = reinterpret_cast<const uint8_t *>(a.heads[a.st->head_idx]);
                if constexpr (Q8)
                    ok = produce_rows(R, sidx, Wh + (size_t)r0_hd * q8_row_bytes(KH), n_hd, q8_row_bytes(KH),
                                      q8_rps(KH), pf);
                else
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsumerRegs) : "memory");
    float *wo = reinterpret_cast<float *>(smem + a.off_att);   // [kNW][HD] warp partials of the split
    float *wml = wo + (size_t)kNW * HD;                        // [kNW][2]
    float *rc = wml + (size_t)kNW * 2;                         // [HD]: cos then sin of each frequency
    if (has_item) {
        // rotary cos / sin at the step's rotary position (per stream from the staged
        // prompt positions for a multimodal prompt row); constant for the launch
        const int *stage = a.st->rope_staged ? a.rope_stage : nullptr;
        const int pr = p + a.st->rope_delta;
        for (int m = tid; m < HALF; m += kNC) {
            const size_t r = (size_t)rope_row(m, a.mrope_h, stage, a.rope_stride, p, pr, a.rope_rows);
            rc[m] = a.rope_cos[r * HALF + m];
            rc[HALF + m] = a.rope_sin[r * HALF + m];
        }
    }
    const int rr_h = warp / a.rs_h, colb_h = (warp % a.rs_h) * (hidden / a.rs_h);
    uint32_t sidx = 0;
    unsigned epoch = 0;
    bool ok = true;
    int buf = 0;   // partial-sum table of the phase (alternates: a phase's row threads read
                   // one table while warps already on the next phase fill the other)
    // this launch's sequence number (advanced once every CTA has read it: at the commit)
    const uint32_t seq = *reinterpret_cast<volatile const unsigned *>(a.seq);

    // the layer table in shared memory: each layer's gamma pointers are one
    // shared-memory load away, not a global round trip
    LayerDev *ldev = reinterpret_cast<LayerDev *>(smem + a.off_ldev);
    for (int i = tid; i < a.n_layers * (int)(sizeof(LayerDev) / 8); i += kNC)
        reinterpret_cast<uint64_t *>(ldev)[i] = reinterpret_cast<const uint64_t *>(a.layers)[i];
    named_sync(1, kNC);

    for (int l = 0; l < a.n_layers && ok; ++l) {
        const LayerDev &Ld = ldev[l];
        uint64_t *T = a.tg + (size_t)l * a.tg_stride;
        float gq[EH], gk[EH];
        if (has_item && Ld.q_norm) {
            load_elems<float, EH>(Ld.q_norm + lane * EH, gq);
            load_elems<float, EH>(Ld.k_norm + lane * EH, gk);
        }
        // The four GEMV phases share one body (rolled, so its code is fetched once per
        // layer): A qkv = [Wq; Wk; Wv] RMSNorm(x); then the attention; C x += Wo o;
        // D act = silu(Wg x^) * (Wu x^), x^ = RMSNorm(x); E x += Wd act.
#pragma unroll 1
        for (int ph = 0; ph < 4 && ok; ++ph) {
            QD_TS(l, ph * 4);
            if (ph == 1) {
                // ---- B: attention of this CTA's (group, split), then its share of the merge
                bool okb = true;
                do {
            // kNW / G warps per q head of the group, each over a slice of the split's
            // positions; the warps of a head are merged, then the splits.
            if (has_item) {
                constexpr int WPH = kNW / G;
                const int hq = warp / WPH, ws = warp % WPH;
                const int pw = (n_att + WPH - 1) / WPH;     // positions per warp
                const int jw0 = ws * pw;
                const int nwp = n_att - jw0 < pw ? (n_att - jw0 > 0 ? n_att - jw0 : 0) : pw;
                const int jp = p - j0;                      // the new position within the split
                const bool owner = n_old < n_att && jp >= jw0 && jp < jw0 + nwp;
                // this lane's columns of q head hq, and (owner) of k and v, in one batch
                const uint64_t *qb = T + a.tg_qkv + (size_t)(ig * G + hq) * HD + lane * EH;
                const uint64_t *kb = T + a.tg_qkv + q_dim + (size_t)ig * HD + lane * EH;
                float wv[3 * EH];
                bool okw = poll_batch<3 * EH>(owner ? 3 * EH : EH, seq,
                                              [&](int i) {
                                                  return i < EH ? qb + i
                                                                : kb + (size_t)((i - EH) / EH) * kv_dim + (i - EH) % EH;
                                              },
                                              wv);
                okw = __all_sync(0xffffffffu, okw);
                QD_TS(l, 16);
                float q[1][EH], kr[EH], vr[EH];
#pragma unroll
                for (int e = 0; e < EH; ++e) {
                    q[0][e] = wv[e];
                    kr[e] = wv[EH + e];
                    vr[e] = wv[2 * EH + e];
                }
                if (Ld.q_norm) {
                    head_norm<EH>(q[0], gq, HD, a.eps);
                    if (owner) head_norm<EH>(kr, gk, HD, a.eps);
                }
                float rcs[EH], rsn[EH];
#pragma unroll
                for (int e = 0; e < EH; ++e) {
                    rcs[e] = rc[(lane & 15) * EH + e];
                    rsn[e] = rc[HALF + (lane & 15) * EH + e];
                }
                rope_lane<EH>(q[0], rcs, rsn, lane);
                if (owner) {
                    // the new row in the cache type; head 0's owner appends it to the cache
                    rope_lane<EH>(kr, rcs, rsn, lane);
#pragma unroll
                    for (int e = 0; e < EH; ++e) {
                        kr[e] = round_to<KT>(kr[e]);
                        vr[e] = round_to<KT>(vr[e]);
                    }
                    if (hq == 0) {
                        const size_t row = ((size_t)ig * a.S + p) * HD + lane * EH;
                        KT *kw = reinterpret_cast<KT *>(reinterpret_cast<uint8_t *>(a.kv) + (size_t)l * layer_kv) + row;
                        KT *vw = reinterpret_cast<KT *>(reinterpret_cast<uint8_t *>(a.kv) + (size_t)l * layer_kv +
                                                        layer_kv / 2) + row;
                        store_row_elems<KT, EH>(kw, kr);
                        store_row_elems<KT, EH>(vw, vr);
                    }
                }
                const uint8_t *kslot = okw ? stage_get(R, sidx) : nullptr;
                const uint8_t *vslot = kslot ? stage_get(R, sidx + 1) : nullptr;
                okw = __all_sync(0xffffffffu, vslot != nullptr);
                if (okw) {
                    float o[1][EH], mh[1], lh[1];
                    warp_attention<KT, HD, 1>(reinterpret_cast<const KT *>(kslot), reinterpret_cast<const KT *>(vslot), q,
                                              jw0, nwp, jp, kr, vr, a.scale, o, mh, lh);
                    float *dst = wo + (size_t)warp * HD + lane * EH;
#pragma unroll
                    for (int e = 0; e < EH; ++e) dst[e] = o[0][e];
                    if (lane == 0) {
                        wml[warp * 2] = mh[0];
                        wml[warp * 2 + 1] = lh[0];
                    }
                    stage_put(R, sidx, lane);
                    stage_put(R, sidx + 1, lane);
                }
                sidx += 2;
                ok = !named_sync_or(1, kNC, !okw);
                if (!ok) { okb = false; break; }
                QD_TS(l, 17);
                // the split's partial, the warps of each head merged in order: its
                // normalised output o / l and, per head, its log-sum-exp m + log(l)
                const int GD = G * HD;
                uint64_t *Tpo = T + a.tg_po + ((size_t)ig * kAttnMaxSplits + is) * GD;
                uint64_t *Tml = T + a.tg_ml + ((size_t)ig * kAttnMaxSplits + is) * G * 2;
                for (int t = tid; t < GD; t += kNC) {
                    const int h = t / HD, d = t % HD;
                    float M = -INFINITY;
#pragma unroll 1
                    for (int w = h * WPH; w < (h + 1) * WPH; ++w) M = fmaxf(M, wml[w * 2]);
                    float den = 0.f, num = 0.f;
#pragma unroll 1
                    for (int w = h * WPH; w < (h + 1) * WPH; ++w) {
                        const float mw = wml[w * 2];
                        if (mw != -INFINITY) {
                            const float f = __expf(mw - M);
                            den = fmaf(f, wml[w * 2 + 1], den);
                            num = fmaf(f, wo[(size_t)w * HD + d], num);
                        }
                    }
                    st_tag(Tpo + t, __fdividef(num, den), seq);
                    if (d == 0) st_tag(Tml + 2 * h, M + __logf(den), seq);
                }
                // this CTA's slice [d0, d1) of the group's merged output: every split's output
                // weighted by exp(lse_s - max) over their sum.  A group of LP lanes (LP >=
                // splits, a power of two) takes one column, lane s its split s; each thread
                // takes two (column, split) pairs, polled in one batch, and the group reduces
                // them with shuffles.
                QD_TS(l, 18);
                const int d0 = is * GD / nsplit, d1 = (is + 1) * GD / nsplit;
                const int LP = nsplit <= 1 ? 1 : (nsplit <= 2 ? 2 : (nsplit <= 4 ? 4 : 8));
                const uint64_t *Gpo = T + a.tg_po + (size_t)ig * kAttnMaxSplits * GD;
                const uint64_t *Gml = T + a.tg_ml + (size_t)ig * kAttnMaxSplits * G * 2;
                bool okm = true;
                for (int c0 = 0; c0 < (d1 - d0) * LP; c0 += 2 * kNC) {
                    // pairs c and c + kNC: the same split (LP divides kNC), so the second is
                    // live only when the first is
                    const int ca = c0 + tid, cb = ca + kNC;
                    const int sp = ca % LP, cola = d0 + ca / LP, colb = d0 + cb / LP;
                    const bool la = cola < d1 && sp < nsplit, lb = colb < d1 && sp < nsplit;
                    float wv[4];
                    const bool got = poll_batch<4>(la ? (lb ? 4 : 2) : 0, seq,
                                                   [&](int i) {
                                                       const int cl = i < 2 ? cola : colb;
                                                       return (i & 1) ? Gpo + (size_t)sp * GD + cl
                                                                      : Gml + ((size_t)sp * G + cl / HD) * 2;
                                                   },
                                                   wv);
                    okm = okm && got;
    #pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const bool lv = k == 0 ? la : lb;
                        const float lse = lv ? wv[2 * k] : -INFINITY;
                        const float ov = lv ? wv[2 * k + 1] : 0.f;
                        float M = lse;
                        for (int o = 1; o < LP; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                        float f = lv ? __expf(lse - M) : 0.f;
                        float num = f * ov;
                        for (int o = 1; o < LP; o <<= 1) {
                            f += __shfl_xor_sync(0xffffffffu, f, o);
                            num += __shfl_xor_sync(0xffffffffu, num, o);
                        }
                        if (lv && sp == 0) st_tag(T + a.tg_att + (size_t)ig * GD + (k == 0 ? cola : colb), __fdividef(num, f), seq);
                    }
                }
                if (!okm) ok = false;
                QD_TS(l, 19);
            }

                } while (false);
                if (!okb) break;
            }
            // this phase: input words, RMSNorm gamma (A, D), K, rows of W
            const uint64_t *src;
            const float *gam;
            int K, nrows, rps;
            uint32_t rbytes;
            constexpr bool kMma = sizeof(WT) == 2 && !Q8;
            // rows of a ring stage of each phase's K
            constexpr int rpsH = Q8 ? q8_prs(KH) : mma_rps(KH), rpsQ = Q8 ? q8_prs(KQ) : mma_rps(KQ),
                          rpsF = Q8 ? q8_prs(KF) : mma_rps(KF);
            constexpr bool kPacked = Q8 || kMma;   // rows per stage from the layout, not the host
            if (ph == 0) {
                src = l ? a.tg + (size_t)(l - 1) * a.tg_stride + a.tg_xe : nullptr;
                gam = Ld.attn_norm; K = KH; nrows = n_qkv; rps = kPacked ? rpsH : a.rps_h; rbytes = rb_h;
            } else if (ph == 1) {
                src = T + a.tg_att; gam = nullptr; K = KQ; nrows = n_x; rps = kPacked ? rpsQ : a.rps_q; rbytes = rb_q;
            } else if (ph == 2) {
                src = T + a.tg_xc; gam = Ld.mlp_norm; K = KH; nrows = n_gu; rps = kPacked ? rpsH : a.rps_h; rbytes = rb_h;
            } else {
                src = T + a.tg_act; gam = nullptr; K = KF; nrows = n_x; rps = kPacked ? rpsF : a.rps_f; rbytes = rb_f;
            }
            const int nc = K / (256 * EL);          // column chunks of 32 x EL per warp
            const int colw = warp * (K / kNW);       // this warp's first column
            float x[NCMAX][EL], gv[NCMAX][EL];
#pragma unroll
            for (int cc = 0; cc < NCMAX; ++cc)
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    x[cc][e] = 0.f;
                    gv[cc][e] = 1.f;
                }
            // lane-contiguous order: element (cc, e) of this lane is column
            // colw + cc * 32 EL + e * 32 + lane, so each load instruction of the warp
            // reads 32 consecutive words (every L2 sector once per poll)
            if (gam)
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
#pragma unroll
                    for (int e = 0; e < EL; ++e)
                        if (cc < nc) gv[cc][e] = gam[colw + cc * 32 * EL + e * 32 + lane];
            bool okw = true;
            if (src) {
                // this lane's words of every chunk, in one batch of polls
                float wv[NCMAX * EL];
                okw = poll_batch<NCMAX * EL>(nc * EL, seq,
                                             [&](int i) { return src + colw + i * 32 + lane; },
                                             wv);
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
#pragma unroll
                    for (int e = 0; e < EL; ++e) x[cc][e] = cc < nc ? wv[cc * EL + e] : 0.f;
                if (ph == 0 && a.tap_hidden && blockIdx.x == 0)
#pragma unroll
                    for (int cc = 0; cc < NCMAX; ++cc)
#pragma unroll
                        for (int e = 0; e < EL; ++e)
                            if (cc < nc) a.tap_hidden[(size_t)l * hidden + colw + cc * 32 * EL + e * 32 + lane] = x[cc][e];
            } else {
                // the step input: thread 0 resolves the step description; CTA 0 records
                // the token in the emitted set and publishes that with a release flag
                if (tid == 0) {
                    DevState *st = a.st;
                    const int mode = st->in_mode;
                    int tok = st->token_in;
                    if (mode == IN_FEEDBACK) tok = st->out_id;
                    else if (mode == IN_STAGED_TOKENS) tok = p < a.in.S ? a.in.stage_tokens[p] : -1;
                    else if (mode == IN_STAGED_EMBEDS) tok = -1;
                    const bool needs_row = (mode == IN_TOKEN || mode == IN_FEEDBACK || mode == IN_STAGED_TOKENS);
                    int bad = 0;
                    if (needs_row && (tok < 0 || tok >= a.in.table_rows || a.in.table == nullptr)) {
                        bad = 1;
                        if (blockIdx.x == 0) atomicOr(&st->status, DEV_ERR_BAD_TOKEN);
                    }
                    if (blockIdx.x == 0) {
                        if (st->add_emitted && tok >= 0 && tok < a.in.vocab)
                            a.in.emitted[tok >> 5] |= 1u << (tok & 31);
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.emit_flag), "r"(seq) : "memory");
                    }
                    misc_i[0] = mode;
                    misc_i[1] = tok;
                    misc_i[2] = bad;
                }
                named_sync(1, kNC);
                const int mode = misc_i[0], tok = misc_i[1];
                const bool bad = misc_i[2] != 0;
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
                    if (cc < nc)
#pragma unroll
                        for (int e = 0; e < EL; ++e) {
                            const int col = colw + cc * 32 * EL + e * 32 + lane;
                            input_cols<WT, 1>(a.in, hidden, mode, tok, p, bad, col, &x[cc][e]);
                            if (blockIdx.x == 0) {
                                a.x[col] = x[cc][e];
                                if (a.tap_hidden) a.tap_hidden[col] = x[cc][e];
                            }
                        }
                if (tid < n_x) {
                    float xo;
                    input_cols<WT, 1>(a.in, hidden, mode, tok, p, bad, r0_x + tid, &xo);
                    xres[tid] = xo;
                }
            }
            okw = __all_sync(0xffffffffu, okw);
            QD_TS(l, ph * 4 + 1);
            if (ph == 0) QD_TS(l - 1, 22);
            float ss = 0.f;
            float *xw = xs + (size_t)warp * XSW;      // this warp's slice of the input, times gamma
            float *part = kc_part + buf * kNW * PS;
            if constexpr (Q8) {
                // the slice as two f16 parts of x * 2^e (e: the largest magnitude lands
                // in [2^13, 2^14)); x0 at xw, x1 XSW halves further
                float vmax = 0.f;
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
                    if (cc < nc)
#pragma unroll
                        for (int e = 0; e < EL; ++e) {
                            ss = fmaf(x[cc][e], x[cc][e], ss);
                            vmax = fmaxf(vmax, fabsf(x[cc][e] * gv[cc][e]));
                        }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
                const int ex = min_c(120, max_c(-120, 140 - ((__float_as_int(vmax) >> 23) & 0xff)));
                const float up = __int_as_float((127 + ex) << 23), down = __int_as_float((127 - ex) << 23);
                __half *xh = reinterpret_cast<__half *>(xw), *xl = xh + XSW;
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
                    if (cc < nc)
#pragma unroll
                        for (int e = 0; e < EL; ++e) {
                            const float v = x[cc][e] * gv[cc][e] * up;
                            const __half h = __float2half_rn(v);
                            const int i = cc * 32 * EL + e * 32 + lane;
                            xh[i] = h;
                            xl[i] = __float2half_rn(v - __half2float(h));
                        }
                __syncwarp();
                if (okw) {
                    if constexpr (KH % 1024 == 0 && KQ % 1024 == 0 && KF % 1024 == 0)
                        okw = kc_gemv_q8_mma<8>(R, sidx, nrows, rps, K, colw, xh, xl, down, part + warp * PS);
                    else if (K % 1024 == 0)
                        okw = kc_gemv_q8_mma<8>(R, sidx, nrows, rps, K, colw, xh, xl, down, part + warp * PS);
                    else
                        okw = kc_gemv_q8_mma<4>(R, sidx, nrows, rps, K, colw, xh, xl, down, part + warp * PS);
                }
            } else if constexpr (kMma) {
                // as two bf16 parts (the slice's K / 8 values twice: the same bytes as fp32)
                __nv_bfloat16 *x0 = reinterpret_cast<__nv_bfloat16 *>(xw), *x1 = x0 + 16;
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
                    if (cc < nc) {
#pragma unroll
                        for (int e = 0; e < EL; ++e) {
                            ss = fmaf(x[cc][e], x[cc][e], ss);
                            const float v = x[cc][e] * gv[cc][e];
                            const __nv_bfloat16 h = __float2bfloat16_rn(v);
                            const int i = cc * 32 * EL + e * 32 + lane;
                            const int j = (i >> 4) * 32 + (i & 15);   // k-step i / 16: x0's 16, then x1's
                            x0[j] = h;
                            x1[j] = __float2bfloat16_rn(v - __bfloat162float(h));
                        }
                    }
                __syncwarp();
                if (okw)
                    okw = kc_gemv_mma(R, sidx, nrows, rps, rbytes + 16, colw, K / (kNW * 16),
                                      reinterpret_cast<const uint32_t *>(x0), part + warp * PS);
            } else {
#pragma unroll
                for (int cc = 0; cc < NCMAX; ++cc)
                    if (cc < nc) {
#pragma unroll
                        for (int e = 0; e < EL; ++e) {
                            ss = fmaf(x[cc][e], x[cc][e], ss);
                            xw[cc * 32 * EL + e * 32 + lane] = x[cc][e] * gv[cc][e];
                        }
                    }
                __syncwarp();
                if (okw) okw = kc_gemv<WT, EL>(R, sidx, nrows, rps, rbytes, colw, nc, xw, part + warp * PS);
            }
            if (gam) {
                ss = warp_sum(ss);
                if (lane == 0) kc_ss[buf * kNW + warp] = ss;
            }
            ok = !named_sync_or(1, kNC, !okw);
            QD_TS(l, ph * 4 + 2);
            if (!ok) break;
            // the phase's rows: thread i sums row i over the warps, in warp order
            if (ph == 0) {
                if (tid < n_qkv)
                    st_tag(T + a.tg_qkv + r0_qkv + tid,
                           rms_scale(kc_ss + buf * kNW, hidden, a.eps) * warp_parts(part, PS, tid), seq);
            } else if (ph == 2) {
                if (tid < n_gu / 2) {
                    const float r = rms_scale(kc_ss + buf * kNW, hidden, a.eps);
                    const float gt = r * warp_parts(part, PS, 2 * tid);
                    const float up = r * warp_parts(part, PS, 2 * tid + 1);
                    st_tag(T + a.tg_act + r0_gu / 2 + tid, __fdividef(gt, 1.0f + __expf(-gt)) * up, seq);
                }
            } else if (tid < n_x) {
                const float xn = xres[tid] + warp_parts(part, PS, tid);
                xres[tid] = xn;
                a.x[r0_x + tid] = xn;
                st_tag(T + (ph == 1 ? a.tg_xc : a.tg_xe) + r0_x + tid, xn, seq);
            }
            QD_TS(l, ph * 4 + 3);
            buf ^= 1;
        }
    }

    if (ok && a.with_head) {
        // ---- head: y = RMSNorm(x); logits; penalty; EOS mask; argmax
        stage_vec(gsm, a.final_norm, hidden);
        const int w0 = r0_hd >> 5;
        const int nw = n_hd > 0 ? ((r0_hd + n_hd - 1) >> 5) - w0 + 1 : 0;
        if (tid == 0 && a.penalty != 1.0f) {
            // the emitted set as CTA 0 left it at this step's start (its release flag)
            const unsigned long long t0 = cycles_now();
            while (true) {
                unsigned v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.emit_flag) : "memory");
                if (v == seq) break;
                if (cycles_now() - t0 > wait_cycles(kWaitLimitNs)) {
                    misc_i[6] = 1;
                    break;
                }
            }
        }
        ok = gather_tagged(a.tg + (size_t)(a.n_layers - 1) * a.tg_stride + a.tg_xe, hidden, xin, seq);
        if (ok && a.penalty != 1.0f)
            for (int i = tid; i < nw; i += kNC) emw[i] = __ldcg(a.in.emitted + w0 + i);
        if (ok) {
            float xr[NS_H * EPL];
            smem_slice<HT, NS_H>(xin, colb_h, xr);
            if (a.tap_hidden && blockIdx.x == 0 && rr_h == 0) {
#pragma unroll
                for (int sg = 0; sg < NS_H; ++sg)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        a.tap_hidden[(size_t)a.n_layers * hidden + colb_h + sg * SEGW + lane * EPL + e] =
                            xr[sg * EPL + e];
            }
            rmsnorm_slice<HT, NS_H>(xr, gsm, hidden, a.rs_h, colb_h, a.eps, misc,
                                    blockIdx.x == 0 ? a.y_out : nullptr);
            bool got;
            if constexpr (Q8)
                got = gemv_consume_q8<NS_H>(R, sidx, n_hd, q8_rps(KH), KH, xr, res);
            else
                got = gemv_consume<WT, NS_H>(R, sidx, n_hd, a.rps_h, rb_h, a.rs_h, colb_h, xr, res);
            ok = !named_sync_or(1, kNC, !got || (tid == 0 && misc_i[6] != 0));
        }
        if (ok) {
            // greedy: per-thread, per-warp, per-CTA argmax.  Sampling (top-k > 0): the
            // CTA's final logits stay in res and the CTA's top-k candidates go out.
            const int sk = a.st->sample_k;
            float best_v = -INFINITY;
            int best_i = INT_MAX;
            for (int r = tid; r < n_hd; r += kNC) {
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
                named_sync(1, kNC);
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
            named_sync(1, kNC);
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
            named_sync(1, kNC);
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
                for (int i = tid; i < hidden; i += kNC)
                    a.tap_hidden[(size_t)a.n_layers * hidden + i] = __ldcg(a.x + i);
            if (tid == 0) {
                a.st->pos = p + 1;
                advance_seq(a.seq, seq);
            }
        }
    }

    if (!ok) {
        // timeout: stop the producer, let copies already issued land, leave
        named_sync(1, kNC);
        if (tid == 0) {
            atomicOr(&a.st->status, DEV_ERR_WAIT_TIMEOUT);
            advance_seq(a.seq, seq);   // no tag of this launch is ever taken as fresh
            ctl[0] = 1;
            const unsigned long long t0 = cycles_now();
            while (!ctl[2] && cycles_now() - t0 < wait_cycles(2 * kWaitLimitNs + 100000000ull)) {
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
static StepFn step_fn(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, bool q8) {
    if (!q8 && !bf16 && hd == 64 && hidden == 256 && q_dim == 256 && ffn == 768 && kvh == 2)
        return decode_step_kernel<float, 64, 256, 256, 768, 2>;             // one-layer fp32 decoder
    if (bf16 && hd == 64 && hidden == 512 && q_dim == 512 && ffn == 2048 && kvh == 8)   // ASR decoder
        return q8 ? decode_step_kernel<__nv_bfloat16, 64, 512, 512, 2048, 8, true>
                  : decode_step_kernel<__nv_bfloat16, 64, 512, 512, 2048, 8>;
    if (bf16 && hd == 128 && hidden == 1024 && q_dim == 2048 && ffn == 3072 && kvh == 8)   // talker / code predictor
        return q8 ? decode_step_kernel<__nv_bfloat16, 128, 1024, 2048, 3072, 8, true>
                  : decode_step_kernel<__nv_bfloat16, 128, 1024, 2048, 3072, 8>;
    return nullptr;
}

bool persistent_supported(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, bool q8) {
    return step_fn(bf16, hd, hidden, q_dim, ffn, kvh, q8) != nullptr;
}

size_t persistent_att_bytes(int group, int hd, int chunk_max) {
    (void)chunk_max;
    (void)group;
    // warp partials of a split, their (max, sum), the RoPE row
    return ((size_t)kNW * hd + (size_t)kNW * 2 + (size_t)hd) * 4;
}

cudaError_t persistent_init(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, bool q8) {
    StepFn f = step_fn(bf16, hd, hidden, q_dim, ffn, kvh, q8);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kStepMaxSmem);
}

cudaError_t launch_persistent(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, const StepArgs &a, int grid,
                              size_t smem, cudaStream_t s, bool q8) {
    StepFn f = step_fn(bf16, hd, hidden, q_dim, ffn, kvh, q8);
    if (!f) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(a.barrier, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStepThreads);
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

#ifdef QD_STEP_TRACE
// Timeline readers of the traced build (not declared in include/qd.h: the product
// library has no such symbols).
extern "C" int qd_step_trace_read(unsigned long long *host, int slots) {
    if (slots != qd::kStepTraceCtas * qd::kStepTraceSlots) return -1;
    return (int)cudaMemcpyFromSymbol(host, qd::g_step_trace, sizeof(unsigned long long) * slots);
}
extern "C" int qd_step_trace_reset(int layer) {
    static unsigned long long zero[qd::kStepTraceCtas * qd::kStepTraceSlots];
    cudaError_t e = cudaMemcpyToSymbol(qd::g_step_trace, zero, sizeof(zero));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(qd::g_step_trace_layer, &layer, sizeof(int));
    return (int)e;
}
#endif

// Tensor-core GEMM for the batched paths: prefill (thousands of tokens) and the
// multi-stream decode (one token per stream), where the projections and the MLP are
// real dense contractions.
//
//   out[t][r] = sum_k W[r][k] * x[t][k],   W [R, K] bf16,   x = x_hi + x_lo (bf16 parts)
//
// Blackwell path (sm_103a): TMA tiled loads with the 128-byte swizzle into a ring of
// shared-memory stages, tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulation) issued
// by one thread with the accumulator in tensor memory, tcgen05.ld for the epilogue.
// The weight tile is the MMA's A operand (M = 128 weight rows), the token tile the B
// operand (N = 64 or 128 tokens); both are K-major, as the row-major matrices are.
// Every k-step issues two MMAs on the same weight tile, one per activation part, so the
// products keep ~16 bits of the fp32 activation (x_lo holds the rounding residue of
// x_hi) while the weights stay bf16.
//
// Roles (576 threads): warp 0 lane 0 issues the TMA loads, warp 1 owns the tensor
// memory and lane 0 issues the MMAs, warps 2-17 read the accumulator and run the
// epilogue: each warp may only touch its quarter of the 128 lanes (warp w reads lanes
// 32*(w%4)..+31), so four warps share a quarter, each with a quarter of the columns.
// The epilogue is a chain of dependent instructions per element (SwiGLU: exp, divide,
// bf16 split); four warps per scheduler hide its latency.  Two accumulators alternate
// so a tile's epilogue overlaps the next tile's MMAs.  When the tiles alone cannot fill the GPU (decode: 64 tokens) the K
// range is split over several CTAs (launched cooperatively, one unit each, so all are
// resident); each writes its partial tile to scratch, the split CTAs of a tile meet on
// a counter, and each then sums its share of the tile's columns over all splits in
// split order and runs the epilogue on it, so the result does not depend on timing.
//
// Launched as a programmatic dependent of the kernel before it, the producer loads the
// weight tiles of its first stages (weights are never written) before waiting for that
// kernel, then the activation tiles; the epilogue waits before it reads or writes.
//
// Every wait is bounded (1 s on %globaltimer); on expiry the kernel records
// DEV_ERR_WAIT_TIMEOUT, every role stops, copies and MMAs in flight are drained, the
// tensor memory is freed and the kernel returns.
#include <cuda.h>

#include <mutex>

#include "qd_device.cuh"
#include "qd_internal.h"
#include "tc_common.cuh"

namespace qd {

namespace {

constexpr int kEpiWarps = 16;                  // epilogue warps: 4 per tensor-memory lane quarter
constexpr int kEpiGroups = kEpiWarps / 4;      // column groups of a quarter
constexpr int kTcThreads = (2 + kEpiWarps) * 32;
constexpr int kBM = 128;                       // weight rows per tile (MMA M)
constexpr int kBK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kTileA = kBM * kBK * 2;     // 16 KB
constexpr unsigned long long kDrainNs = 20000000ull;   // 20 ms for clean-up waits

template <int BN> struct TcCfg {
    static constexpr uint32_t kTileB = BN * kBK * 2;
    static constexpr uint32_t kStage = kTileA + 2 * kTileB;
    static constexpr int kStages = BN == 64 ? 6 : 4;
    static constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators of BN fp32 columns
    // stages, barriers (256 bytes), the folded RMSNorm's scales of a token tile (<= 1 KB)
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + 256 + 1024;
};

// Instruction descriptor of this GEMM: M = kBM weight rows, N = BN tokens, both K-major.
template <int BN> __device__ __forceinline__ constexpr uint32_t tc_idesc() { return tc_idesc_mn<kBM, BN>(); }

__device__ __forceinline__ int ld_acquire_s32(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

struct Unit {
    int tile, rt, nt, k0, k1;
};
__device__ __forceinline__ Unit unit_of(int u, int splits, int tok_tiles, int KC) {
    Unit x;
    x.tile = u / splits;
    const int s = u - x.tile * splits;
    x.rt = x.tile / tok_tiles;
    x.nt = x.tile - x.rt * tok_tiles;
    x.k0 = (int)((long long)s * KC / splits);
    x.k1 = (int)((long long)(s + 1) * KC / splits);
    return x;
}

// Epilogue of one output element: token t, weight row r (rows of a warp are
// consecutive lanes; the SwiGLU pairing uses the neighbouring lane, so every lane of
// the warp must call this together).
__device__ __forceinline__ void epi_apply(const TcGemmArgs &a, int t, int r, float v, int lane) {
    if (a.mode == TC_STORE) {
        a.out[(size_t)t * a.ldo + r] = v;
    } else if (a.mode == TC_STORE_RT) {
        if (r < a.r_valid) a.out[(size_t)r * a.ldo + (size_t)t * a.ldt] = v + (a.bias ? a.bias[r] : 0.f);
    } else if (a.mode == TC_RESIDUAL) {
        float *p = a.out + (size_t)t * a.ldo + r;
        *p = *p + v;
    } else {
        const float u = __shfl_down_sync(0xffffffffu, v, 1);
        if ((lane & 1) == 0) {
            const float act = v / (1.0f + expf(-v)) * u;
            const __nv_bfloat16 hi = __float2bfloat16_rn(act);
            const __nv_bfloat16 lo = __float2bfloat16_rn(act - __bfloat162float(hi));
            const size_t o = (size_t)t * (a.R / 2) + (r >> 1);
            a.act_hi[o] = hi;
            a.act_lo[o] = lo;
            if (a.out) a.out[(size_t)t * a.ldo + (r >> 1)] = act;
        }
    }
}

// The folded RMSNorm's scale of token t: the producing GEMM's partial sums of squares
// (one per 32-row quarter of each row tile), summed in order.
__device__ __forceinline__ float rms_scale_of(const TcGemmArgs &a, int t) {
    float s = 0.f;
    for (int i = 0; i < a.rs_tiles; ++i) s += __ldcg(a.rs_part + (size_t)i * a.T + t);
    return 1.0f / sqrtf(s / (float)a.rs_K + a.rs_eps);
}

// Epilogue of tokens t0..t0+n-1 (n <= N) of weight row r (row q * 32 + lane of row tile
// rt).  The residual reads are all issued before any write: a read after a write to the
// same array cannot be moved ahead of it, so element-by-element read-add-write would
// queue N round trips.  rsc: the folded norm's scales of tokens t0.. (null: none).
template <int N>
__device__ __forceinline__ void epi_apply_n(const TcGemmArgs &a, int t0, int r, float *v, int n, int lane, int q,
                                            int rt, const float *rsc) {
    if (rsc) {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] *= rsc[j];
    }
    if (a.mode == TC_RESIDUAL || a.mode == TC_RESIDUAL_NORM) {
        float old[N];
#pragma unroll
        for (int j = 0; j < N; ++j) old[j] = j < n ? a.out[(size_t)(t0 + j) * a.ldo + r] : 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            old[j] += v[j];
            if (j < n) a.out[(size_t)(t0 + j) * a.ldo + r] = old[j];
        }
        if (a.mode == TC_RESIDUAL_NORM) {
            // the next norm's input parts, and this warp's 32 rows' sum of squares per
            // token (a shuffle tree; one partial per row-tile quarter)
            const float g = a.norm_gamma[r];
#pragma unroll
            for (int j = 0; j < N; ++j) {
                if (j < n) {
                    const float y = g * old[j];
                    const __nv_bfloat16 h = __float2bfloat16_rn(y);
                    a.nh[(size_t)(t0 + j) * a.R + r] = h;
                    a.nl[(size_t)(t0 + j) * a.R + r] = __float2bfloat16_rn(y - __bfloat162float(h));
                }
                float sq = j < n ? old[j] * old[j] : 0.f;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
                if (lane == 0 && j < n) a.ss_out[(size_t)(rt * 4 + q) * a.T + t0 + j] = sq;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j)
            if (j < n) epi_apply(a, t0 + j, r, v[j], lane);
    }
}

// TMA coordinates of reduction chunk kc (tap kc / KCt, columns of chunk kc % KCt) for
// the unit's row tile rt and token tile nt: the weight tile (wx, wy) and the token
// tile (xx, xy); xy may be negative or past T (those rows load as zero).
__device__ __forceinline__ void chunk_xy(const TcGemmArgs &a, int KCt, int kc, int rt, int nt, int bn, int &wx,
                                         int &wy, int &xy) {
    const int tap = kc / KCt, kk = kc - tap * KCt;
    wx = kk * kBK;
    wy = (a.w_slab0 + tap * a.w_slab_step) * a.R + rt * kBM;
    xy = nt * bn - (a.x_shift0 + tap * a.x_shift_step);
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                   const __grid_constant__ CUtensorMap tm_xl, const TcGemmArgs a, const int tok_tiles,
                   const int splits, const int units) {
    using C = TcCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)C::kStages * C::kStage);
    uint64_t *empty = full + C::kStages;
    uint64_t *acc_full = empty + C::kStages;   // [2]
    uint64_t *acc_empty = acc_full + 2;        // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *is_last = reinterpret_cast<int *>(tmem_slot + 2);
    float *rsm = reinterpret_cast<float *>(sm + (size_t)C::kStages * C::kStage + 256);   // [BN] folded-norm scales

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KCt = a.K / kBK;          // chunks of one tap
    const int KC = KCt * a.taps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;   // per-stage bits: armed at least once / parity of last arming
            // the weight tiles of the first unit's first stages go out before the wait for
            // the previous kernel, its activation tiles after it
            int pre = 0;
            if ((int)blockIdx.x < units) {
                const Unit x0 = unit_of(blockIdx.x, splits, tok_tiles, KC);
                pre = x0.k1 - x0.k0 < C::kStages ? x0.k1 - x0.k0 : C::kStages;
                for (int i = 0; i < pre; ++i) {
                    int wx, wy, xy;
                    chunk_xy(a, KCt, x0.k0 + i, x0.rt, x0.nt, BN, wx, wy, xy);
                    mbar_arrive_expect_tx(&full[i], C::kStage);
                    tma_load_2d(sm + (size_t)i * C::kStage, &tm_w, wx, wy, &full[i]);
                }
                pdl_wait();
                pdl_launch_dependents();
                for (int i = 0; i < pre; ++i) {
                    int wx, wy, xy;
                    chunk_xy(a, KCt, x0.k0 + i, x0.rt, x0.nt, BN, wx, wy, xy);
                    uint8_t *st = sm + (size_t)i * C::kStage;
                    tma_load_2d(st + kTileA, &tm_xh, wx, xy, &full[i]);
                    tma_load_2d(st + kTileA + C::kTileB, &tm_xl, wx, xy, &full[i]);
                }
                armed = (1u << pre) - 1u;
                stage = pre % C::kStages;
                phase = pre == C::kStages ? 1u : 0u;
            } else {
                pdl_wait();
                pdl_launch_dependents();
            }
            for (int u = blockIdx.x; u < units && !*abort_flag; u += gridDim.x) {
                const Unit x = unit_of(u, splits, tok_tiles, KC);
                bool ok = true;
                for (int kc = x.k0 + (u == (int)blockIdx.x ? pre : 0); kc < x.k1; ++kc) {
                    if (!role_wait(&empty[stage], phase ^ 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    int wx, wy, xy;
                    chunk_xy(a, KCt, kc, x.rt, x.nt, BN, wx, wy, xy);
                    mbar_arrive_expect_tx(&full[stage], C::kStage);
                    uint8_t *st = sm + (size_t)stage * C::kStage;
                    tma_load_2d(st, &tm_w, wx, wy, &full[stage]);
                    tma_load_2d(st + kTileA, &tm_xh, wx, xy, &full[stage]);
                    tma_load_2d(st + kTileA + C::kTileB, &tm_xl, wx, xy, &full[stage]);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                // let every copy this thread issued land before the CTA exits
                for (int s = 0; s < C::kStages; ++s)
                    if (armed >> s & 1) mbar_wait_bounded(&full[s], armed_parity >> s & 1, kDrainNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t idesc = tc_idesc<BN>();
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            for (int u = blockIdx.x; u < units && !*abort_flag; u += gridDim.x, ++local) {
                const Unit x = unit_of(u, splits, tok_tiles, KC);
                const int acc = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!role_wait(&acc_empty[acc], (use & 1) ^ 1, abort_flag, a.status)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kc = x.k0; kc < x.k1; ++kc) {
                    if (!role_wait(&full[stage], phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(sm + (size_t)stage * C::kStage);
                    const uint32_t sh = sa + kTileA, sl = sh + C::kTileB;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = sw128_desc(sa + 32u * k);
                        tc_mma(d, ad, sw128_desc(sh + 32u * k), idesc, (kc > x.k0 || k > 0) ? 1u : 0u);
                        tc_mma(d, ad, sw128_desc(sl + 32u * k), idesc, 1u);
                    }
                    tc_commit(&empty[stage]);   // the stage is free once these MMAs have read it
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(&acc_full[acc]);
            }
            // every MMA issued has completed before the tensor memory is released
            tc_commit(drain);
            mbar_wait_bounded(drain, 0, kDrainNs);
        }
    } else {
        // ---- epilogue warps 2..17
        const int q = warp & 3;                 // tensor-memory lane quarter of this warp
        const int cg = (warp - 2) >> 2;         // its column group within the quarter
        const int row_in_tile = q * 32 + lane;
        constexpr int kEpiT = kEpiWarps * 32;
        pdl_wait();   // outputs, residuals, scratch and counters may belong to the previous kernel
        int local = 0, rs_tile = -1;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
            const Unit x = unit_of(u, splits, tok_tiles, KC);
            const int acc = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (a.rs_part && x.nt != rs_tile) {
                // the folded norm's scales of this token tile, while the products run
                named_sync(1, kEpiT);   // the previous tile's scales are no longer read
                const int et = (warp - 2) * 32 + lane;
                for (int t = et; t < BN; t += kEpiT) {
                    const int tt = x.nt * BN + t;
                    rsm[t] = tt < a.T ? rms_scale_of(a, tt) : 0.f;
                }
                named_sync(1, kEpiT);
                rs_tile = x.nt;
            }
            bool ok = true;
            if (lane == 0) ok = role_wait(&acc_full[acc], use & 1, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            // all epilogue warps agree before any of them goes on
            if (named_sync_or(1, kEpiT, !ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const int r = x.rt * kBM + row_in_tile;
            if (splits == 1) {
#pragma unroll 1
                for (int c0 = cg * 16; c0 < BN; c0 += 16 * kEpiGroups) {
                    float v[16];
                    tc_ld16(tbase + (uint32_t)c0, v);
                    const int t0 = x.nt * BN + c0;
                    epi_apply_n<16>(a, t0, r, v, a.T - t0 < 16 ? a.T - t0 : 16, lane, q, x.rt,
                                    a.rs_part ? rsm + (t0 - x.nt * BN) : nullptr);
                }
            } else {
                float *part = a.partial + (size_t)u * BN * kBM;
#pragma unroll 1
                for (int c0 = cg * 16; c0 < BN; c0 += 16 * kEpiGroups) {
                    float v[16];
                    tc_ld16(tbase + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) __stcg(part + (size_t)(c0 + j) * kBM + row_in_tile, v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            if (splits > 1) {
                // The split CTAs of a tile meet (the launch is cooperative, so all of them
                // are resident), then each sums its share of the tile's columns over every
                // split, in split order, and runs the epilogue on it.
                __threadfence();
                named_sync(1, kEpiT);
                int *arrive = a.tile_counter + 2 * x.tile;
                int *depart = arrive + 1;
                if (warp == 2 && lane == 0) {
                    atomicAdd(arrive, 1);
                    int met = 1;
                    const unsigned long long t0 = global_timer_ns();
                    while (ld_acquire_s32(arrive) < splits) {
                        if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
                            if (!*abort_flag) atomicOr(a.status, DEV_ERR_WAIT_TIMEOUT);
                            *abort_flag = 1;
                            met = 0;
                            break;
                        }
                    }
                    *is_last = met;
                }
                named_sync(1, kEpiT);
                const bool met = *is_last != 0;
                if (met) {
                    __threadfence();
                    const int s_idx = u - x.tile * splits;
                    const int c_lo = s_idx * BN / splits, c_hi = (s_idx + 1) * BN / splits;
                    const float *p0 = a.partial + (size_t)x.tile * splits * BN * kBM + row_in_tile;
#pragma unroll 1
                    for (int c = c_lo + 4 * cg; c < c_hi; c += 4 * kEpiGroups) {
                        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                        for (int s2 = 0; s2 < splits; ++s2) {
                            const float *ps = p0 + (size_t)s2 * BN * kBM;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (c + j < c_hi) v[j] += __ldcg(ps + (size_t)(c + j) * kBM);
                        }
                        const int t0 = x.nt * BN + c;
                        int n = c_hi - c < 4 ? c_hi - c : 4;
                        if (a.T - t0 < n) n = a.T - t0;
                        epi_apply_n<4>(a, t0, r, v, n, lane, q, x.rt, a.rs_part ? rsm + (t0 - x.nt * BN) : nullptr);
                    }
                }
                named_sync(1, kEpiT);
                if (warp == 2 && lane == 0 && met) {
                    // the last CTA to leave puts the tile's counters back at rest
                    if (atomicAdd(depart, 1) == splits - 1) {
                        *arrive = 0;
                        *depart = 0;
                        __threadfence();
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

__global__ void split_bf16_kernel(const float *x, __nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = x[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        hi[i] = h;
        lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

// ---- host side: tensor maps through the driver entry point (no libcuda link)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 [rows, K] row-major, box of 64 elements (128 bytes, the swizzle span) x box_rows.
bool make_map(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN> cudaError_t set_attr() {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(reinterpret_cast<const void *>(tc_gemm_kernel<BN>),
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<BN>::kSmem);
    });
    return attr;
}

template <int BN> cudaError_t launch_bn(const TcGemmPlan &p, const void *w, const void *xh, const void *xl,
                                        const TcGemmArgs &a, cudaStream_t s, bool pdl) {
    cudaError_t attr = set_attr<BN>();
    if (attr != cudaSuccess) return attr;
    CUtensorMap mw, mh, ml;
    if (!make_map(&mw, w, a.w_rows, a.K, kBM) || !make_map(&mh, xh, a.T, a.K, BN) ||
        !make_map(&ml, xl, a.T, a.K, BN))
        return cudaErrorInvalidValue;
    if (p.splits == 1 && !pdl) {
        tc_gemm_kernel<BN><<<p.grid, kTcThreads, TcCfg<BN>::kSmem, s>>>(mw, mh, ml, a, p.tok_tiles, p.splits,
                                                                          p.units);
        return cudaGetLastError();
    }
    // split-K: the split CTAs of a tile wait for one another, so they must all be
    // resident.  A cooperative launch guarantees it; as a programmatic dependent (one
    // unit per CTA, grid <= SMs, one CTA per SM) every CTA has started before any
    // kernel after it may (each signals only once running), and the kernel before it
    // only ends, so all of them become resident.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcCfg<BN>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    if (pdl) {
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
    } else {
        at[0].id = cudaLaunchAttributeCooperative;
        at[0].val.cooperative = 1;
    }
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int tok_tiles = p.tok_tiles, splits = p.splits, units = p.units;
    void *args[7] = {&mw, &mh, &ml, const_cast<TcGemmArgs *>(&a), &tok_tiles, &splits, &units};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(tc_gemm_kernel<BN>), args);
}

}  // namespace

cudaError_t tc_gemm_init() {
    if (!encode_fn()) return cudaErrorNotSupported;
    cudaError_t e = set_attr<64>();
    return e != cudaSuccess ? e : set_attr<128>();
}

bool make_bf16_rows_map(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows) {
    if (rows < 1 || K % 64 || box_rows < 1 || box_rows > 256) return false;
    return make_map(m, ptr, rows, K, box_rows);
}

bool make_kv_tile_map(CUtensorMap *m, const void *kv, int hd, int S, long long planes, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(kv) & 15) || hd % 64 || S % 32 || planes < 1 || planes > INT32_MAX ||
        box_rows < 1 || box_rows > 256)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)S, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)hd * 2 * S};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(kv), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxSplits = 8;

bool tc_gemm_plan(int R, int K, int T, int num_sms, TcGemmPlan *p) {
    if (R <= 0 || K <= 0 || T <= 0 || R % kBM || K % kBK || num_sms <= 0) return false;
    TcGemmPlan q = {};
    q.bn = T <= 64 ? 64 : 128;
    q.row_tiles = R / kBM;
    q.tok_tiles = (T + q.bn - 1) / q.bn;
    const int tiles = q.row_tiles * q.tok_tiles;
    const int KC = K / kBK;
    q.splits = 1;
    // split K to fill the SMs, at most kMaxSplits ways: the split CTAs of a tile meet
    // and each reads every split's partial of its columns, which at 19 splits (a
    // 1024-row product over K = 2048 or 3072 at 64 tokens) cost more than the
    // streaming the extra splits spread out
    if (tiles < num_sms) q.splits = std::max(1, std::min(std::min(KC, num_sms / tiles), kMaxSplits));
    q.units = tiles * q.splits;
    q.grid = std::min(q.units, num_sms);
    q.smem = q.bn == 64 ? TcCfg<64>::kSmem : TcCfg<128>::kSmem;
    q.partial_floats = q.splits > 1 ? (size_t)q.units * q.bn * kBM : 0;
    *p = q;
    return true;
}

cudaError_t launch_tc_gemm(const TcGemmPlan &p, const void *w, const void *x_hi, const void *x_lo,
                           const TcGemmArgs &a_in, cudaStream_t s, bool pdl) {
    TcGemmArgs a = a_in;
    if (a.taps < 1) {
        // the plain product: one tap, the first slab, no shift
        a.taps = 1;
        a.w_slab0 = a.w_slab_step = a.x_shift0 = a.x_shift_step = 0;
    }
    if (a.w_rows <= 0) a.w_rows = a.R;
    if (p.splits > 1 && (!a.partial || !a.tile_counter || p.units > p.grid)) return cudaErrorInvalidValue;
    if (a.mode == TC_SWIGLU && (!a.act_hi || !a.act_lo)) return cudaErrorInvalidValue;
    if (a.mode == TC_STORE_RT && a.ldt <= 0) return cudaErrorInvalidValue;
    if (a.mode == TC_RESIDUAL_NORM && (!a.norm_gamma || !a.nh || !a.nl || !a.ss_out)) return cudaErrorInvalidValue;
    if (a.rs_part && (a.rs_tiles < 1 || a.rs_K < 1)) return cudaErrorInvalidValue;
    // every tap's weight slab inside W
    for (int j = 0; j < a.taps; j += a.taps - 1 > 0 ? a.taps - 1 : 1) {
        const int slab = a.w_slab0 + j * a.w_slab_step;
        if (slab < 0 || (long long)(slab + 1) * a.R > a.w_rows) return cudaErrorInvalidValue;
    }
    return p.bn == 64 ? launch_bn<64>(p, w, x_hi, x_lo, a, s, pdl) : launch_bn<128>(p, w, x_hi, x_lo, a, s, pdl);
}

cudaError_t launch_split_bf16(const float *x, __nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t n, cudaStream_t s) {
    const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
    split_bf16_kernel<<<grid, 256, 0, s>>>(x, hi, lo, n);
    return cudaGetLastError();
}

}  // namespace qd

// Kernels of the batched prefill (ns prompt streams x n positions) other than the
// tensor-core GEMMs: QK-norm + RoPE + cache append of every prompt position, causal
// flash attention on the tensor cores, and the first-id argmax.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation" (QK-norm over head_dim, GQA, plain RoPE) and section "Integration and
//    performance optimisation" (the prompt is prefilled once; decoding continues from
//    its cache).
//  - "Audio8-ASR: dynamic KV-cache buckets", section "Implemented dynamic window
//    mechanism": a fixed-length prefill produces the first token.
//
// The attention is a dense contraction here (n queries x n keys per stream), so it
// runs on the tensor cores: mma.sync m16n8k16 (bf16 inputs, fp32 accumulation) with
// the queries and the probabilities entering as bf16 hi + lo parts (two MMAs each), K
// and V from the bf16 cache; tiles are staged with cp.async into XOR-swizzled shared
// memory and read with ldmatrix, conflict-free.
#include "decode_common.cuh"
#include "mma_sync.cuh"

namespace qd {

namespace {

// ---- QK-norm + RoPE + append, one CTA (8 warps) per prompt token
constexpr int kPqThreads = 256;

template <int HD>
__global__ void __launch_bounds__(kPqThreads) prefill_qk_kernel(const PrefillQkArgs a) {
    constexpr int DPL = HD / 32;
    constexpr int HALF = HD / 2;
    if ((int)blockIdx.x >= gridDim.x - a.ns_tail) {
        // one CTA per (prompt stream, K or V plane of a kv head): rows [n, next multiple
        // of 128) of the layer are zeroed (below the cache's end), so the attention's last
        // 128-key chunk reads finite values past the prompt; 16-byte stores (a row is
        // HD * 2 bytes, a multiple of 16)
        const int t = (int)blockIdx.x - (gridDim.x - a.ns_tail);
        const int i = t / (2 * a.kvh), plane = t - i * 2 * a.kvh;
        const int end = min((a.n + 127) / 128 * 128, a.S);
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.kv) +
                                               (size_t)a.streams[i] * a.stream_elems + a.layer_elems +
                                               ((size_t)plane * a.S + a.n) * HD);
        const int n16 = (end - a.n) * HD / 8;
        for (int k = threadIdx.x; k < n16; k += kPqThreads) dst[k] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const int tok = blockIdx.x;
    const int i = tok / a.n, j = tok - i * a.n;        // prompt stream, position
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *row = a.qkv + (size_t)tok * a.qkv_ld;
    const int stream = a.streams[i];
    __nv_bfloat16 *kc = reinterpret_cast<__nv_bfloat16 *>(a.kv) + (size_t)stream * a.stream_elems + a.layer_elems;
    __nv_bfloat16 *vc = kc + (size_t)a.kvh * a.S * HD;
    // vectors: q heads 0..qh-1, k heads qh..qh+kvh-1 (normed, rotated), v heads (copied)
    for (int vec = warp; vec < a.qh + 2 * a.kvh; vec += kPqThreads / 32) {
        float v[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[e] = __ldcg(row + (size_t)vec * HD + lane * DPL + e);
        if (vec < a.qh + a.kvh) {
            const float *gam = vec < a.qh ? a.q_gamma : a.k_gamma;
            if (gam) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) ss = fmaf(v[e], v[e], ss);
                ss = warp_sum(ss);
                const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
#pragma unroll
                for (int e = 0; e < DPL; ++e) v[e] = v[e] * inv * gam[lane * DPL + e];
            }
            // rotate-half RoPE at position j (or the prompt's rotary positions): dims d
            // and d + HD/2 sit 16 lanes apart
            float w[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) w[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
            const bool low = lane < 16;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const int m = (lane & 15) * DPL + e;
                const size_t r = (size_t)rope_row(m, a.mrope_h, a.rope_pos, a.rope_stride, j, j, a.rope_rows);
                const float c = a.rope_cos[r * HALF + m], sn = a.rope_sin[r * HALF + m];
                v[e] = low ? v[e] * c - w[e] * sn : v[e] * c + w[e] * sn;
            }
        }
        if (vec < a.qh) {
            const size_t o = (((size_t)i * a.qh + vec) * a.n + j) * HD + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const __nv_bfloat16 h = __float2bfloat16_rn(v[e]);
                a.q_hi[o + e] = h;
                a.q_lo[o + e] = __float2bfloat16_rn(v[e] - __bfloat162float(h));
            }
        } else {
            const bool isk = vec < a.qh + a.kvh;
            const int g = isk ? vec - a.qh : vec - a.qh - a.kvh;
            __nv_bfloat16 *dst = (isk ? kc : vc) + ((size_t)g * a.S + j) * HD + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) dst[e] = __float2bfloat16_rn(v[e]);
        }
    }
}

__global__ void gather_last_kernel(const float *x, int n, int K, float *out) {
    const int i = blockIdx.x;
    const float *src = x + ((size_t)i * n + n - 1) * K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) out[(size_t)i * K + k] = src[k];
}

// First id of each prompt stream: EOS mask and argmax (lowest index on ties); the
// emitted set is empty after a prefill, so the repetition penalty has nothing to do.
__global__ void __launch_bounds__(256) prefill_finish_kernel(const PrefillFinishArgs a) {
    __shared__ float bv_s[8];
    __shared__ int bi_s[8];
    const int i = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *lg = a.logits + (size_t)i * a.V;
    float *lo = a.logits_out + (size_t)a.streams[i] * a.V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int k = tid; k < a.V; k += 256) {
        lo[k] = lg[k];
        const float v = k == a.eos ? -INFINITY : lg[k];
        if (arg_better(v, k, bv, bi)) {
            bv = v;
            bi = k;
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
        bv_s[warp] = bv;
        bi_s[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < 8; ++w)
            if (arg_better(bv_s[w], bi_s[w], bv_s[0], bi_s[0])) {
                bv_s[0] = bv_s[w];
                bi_s[0] = bi_s[w];
            }
        const int s = a.streams[i];
        a.first_ids[i] = bi_s[0];
        a.tokens[s] = bi_s[0];
        a.pos[s] = a.n;
    }
}

}  // namespace

cudaError_t launch_prefill_qk(int hd, int ns, const PrefillQkArgs &a_in, cudaStream_t s) {
    PrefillQkArgs a = a_in;
    a.ns_tail = a.n % 128 && a.n < a.S ? ns * 2 * a.kvh : 0;   // the streams' tail-zeroing CTAs
    const int grid = ns * a.n + a.ns_tail;
    if (hd == 128) prefill_qk_kernel<128><<<grid, kPqThreads, 0, s>>>(a);
    else if (hd == 64) prefill_qk_kernel<64><<<grid, kPqThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_gather_last(const float *x, int n, int K, int ns, float *out, cudaStream_t s) {
    gather_last_kernel<<<ns, 256, 0, s>>>(x, n, K, out);
    return cudaGetLastError();
}

__global__ void prefill_commit_kernel(DevState *st, int pos, const int *batch_status) {
    st->pos = pos;
    st->status |= *batch_status;
}

cudaError_t launch_prefill_commit(DevState *st, int pos, const int *batch_status, cudaStream_t s) {
    prefill_commit_kernel<<<1, 1, 0, s>>>(st, pos, batch_status);
    return cudaGetLastError();
}

__global__ void embed_rows_kernel(const __nv_bfloat16 *table, const int32_t *tokens, int hidden, float *x) {
    const __nv_bfloat16 *row = table + (size_t)tokens[blockIdx.x] * hidden;
    float *o = x + (size_t)blockIdx.x * hidden;
    for (int j = threadIdx.x; j < hidden; j += blockDim.x) o[j] = __bfloat162float(row[j]);
}

cudaError_t launch_embed_rows(const void *table, const int32_t *tokens, int n, int hidden, float *x, cudaStream_t s) {
    embed_rows_kernel<<<n, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(table), tokens, hidden, x);
    return cudaGetLastError();
}

cudaError_t launch_prefill_finish(const PrefillFinishArgs &a, int ns, cudaStream_t s) {
    prefill_finish_kernel<<<ns, 256, 0, s>>>(a);
    return cudaGetLastError();
}

namespace {

// ---- causal flash attention on the tensor cores (mma.sync m16n8k16, bf16 -> fp32)
//
// One CTA (8 warps) per (prompt stream, kv group, block of QB = 128 / G queries): the
// block's G x QB query rows (head-major) are the MMAs' M dimension, 16 rows per warp.
// Keys go in tiles of 64 through a 2-stage cp.async pipeline.  Per tile: S = Q K^T
// (Q as hi + lo parts: 2 MMAs per fragment), causal mask, online softmax per row
// (running max and sum, output rescaled), O += P V (P as hi + lo parts).
constexpr int kFaThreads = 256;
constexpr int kFaKeys = 64;

// 16-byte asynchronous copy; bytes < 16 zero-fills the rest (0: all zeros)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a swizzled tile with rows of HD bf16.
template <int HD> __device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * HD * 2 + ((c ^ (r & 7)) << 4));
}

template <int HD, int G>
__global__ void __launch_bounds__(kFaThreads, 1) prefill_attn_kernel(const PrefillAttnArgs a) {
    constexpr int QB = 128 / G;                 // queries per CTA
    constexpr int CH = HD / 8;                  // 16-byte chunks per row
    constexpr uint32_t kQTile = 128 * HD * 2;   // one query part (hi or lo)
    constexpr uint32_t kKVTile = kFaKeys * HD * 2;
    constexpr int NT = kFaKeys / 8;             // score n-tiles per warp
    constexpr int OT = HD / 8;                  // output n-tiles per warp
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t s_qh = smem_addr(smem), s_ql = s_qh + kQTile;
    const uint32_t s_kv = s_ql + kQTile;        // [stage][K, V]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t4 = lane & 3;
    const int nqb = (a.n + QB - 1) / QB;
    const int pairs = gridDim.x / nqb;
    // blocks with the most keys first
    const int qb = nqb - 1 - (int)(blockIdx.x / pairs);
    const int pair = blockIdx.x - (nqb - 1 - qb) * pairs;
    const int i = pair / a.kvh, g = pair - i * a.kvh;
    const int q0 = qb * QB;
    const int stream = a.streams[i];
    const __nv_bfloat16 *kc = reinterpret_cast<const __nv_bfloat16 *>(a.kv) + (size_t)stream * a.stream_elems +
                              a.layer_elems + (size_t)g * a.S * HD;
    const __nv_bfloat16 *vc = kc + (size_t)a.kvh * a.S * HD;

    // queries: row r = head (g * G + r / QB), query q0 + r % QB; zeros past n
    for (int idx = tid; idx < 2 * 128 * CH; idx += kFaThreads) {
        const int part = idx / (128 * CH), rem = idx - part * 128 * CH;
        const int r = rem / CH, c = rem - r * CH;
        const int h = g * G + r / QB, q = q0 + r % QB;
        const __nv_bfloat16 *src = (part ? a.q_lo : a.q_hi) + (((size_t)i * a.qh + h) * a.n + (q < a.n ? q : 0)) * HD + c * 8;
        cp_async16((part ? s_ql : s_qh) + swz<HD>(r, c), src, q < a.n ? 16u : 0u);
    }
    const int last_q = q0 + QB - 1 < a.n - 1 ? q0 + QB - 1 : a.n - 1;
    const int nkt = last_q / kFaKeys + 1;       // key tiles up to the block's last query
    auto load_kv = [&](int kt, int stage) {
        const uint32_t base = s_kv + (uint32_t)stage * 2 * kKVTile;
        for (int idx = tid; idx < 2 * kFaKeys * CH; idx += kFaThreads) {
            const int part = idx / (kFaKeys * CH), rem = idx - part * kFaKeys * CH;
            const int r = rem / CH, c = rem - r * CH;
            const int key = kt * kFaKeys + r;
            const __nv_bfloat16 *src = (part ? vc : kc) + (size_t)(key < a.n ? key : 0) * HD + c * 8;
            cp_async16(base + part * kKVTile + swz<HD>(r, c), src, key < a.n ? 16u : 0u);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const int row0 = warp * 16;                 // this warp's rows
    const int qw = q0 + row0 % QB;              // query of row0
    float o[OT][4];
#pragma unroll
    for (int t = 0; t < OT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[t][e] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int kt = 0; kt < nkt; ++kt) {
        if (kt + 1 < nkt) {
            load_kv(kt + 1, (kt + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t s_k = s_kv + (uint32_t)(kt & 1) * 2 * kKVTile, s_v = s_k + kKVTile;
        // S = Q K^T for this warp's 16 rows x 64 keys
        float sacc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[t][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
            uint32_t ah[4], al[4];
            {
                const int mat = lane >> 3, r8 = lane & 7;
                const int r = row0 + r8 + ((mat & 1) ? 8 : 0), c = 2 * ks + (mat >> 1);
                ldsm_x4(s_qh + swz<HD>(r, c), ah[0], ah[1], ah[2], ah[3]);
                ldsm_x4(s_ql + swz<HD>(r, c), al[0], al[1], al[2], al[3]);
            }
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int mat = lane >> 3, r8 = lane & 7;
                const int key = np * 16 + r8 + ((mat >> 1) ? 8 : 0), c = 2 * ks + (mat & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(s_k + swz<HD>(key, c), b0, b1, b2, b3);
                mma16816(sacc[2 * np], ah, b0, b1);
                mma16816(sacc[2 * np], al, b0, b1);
                mma16816(sacc[2 * np + 1], ah, b2, b3);
                mma16816(sacc[2 * np + 1], al, b2, b3);
            }
        }
        // scale, causal mask, online softmax (rows gid and gid + 8 of the warp)
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kt * kFaKeys + t * 8 + t4 * 2 + (e & 1);
                const int q = qw + gid + ((e >> 1) ? 8 : 0);
                const float v = (key > q || key >= a.n) ? -INFINITY : sacc[t][e] * a.scale;
                sacc[t][e] = v;
                tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
            }
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
            tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
            const float mnew = fmaxf(mrow[h], tmax[h]);
            corr[h] = mnew == -INFINITY ? 1.f : expf(mrow[h] - mnew);
            mrow[h] = mnew;
            lrow[h] *= corr[h];
        }
#pragma unroll
        for (int t = 0; t < OT; ++t) {
            o[t][0] *= corr[0];
            o[t][1] *= corr[0];
            o[t][2] *= corr[1];
            o[t][3] *= corr[1];
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float m = mrow[e >> 1];
                const float pv = sacc[t][e] == -INFINITY ? 0.f : expf(sacc[t][e] - m);
                sacc[t][e] = pv;
                lrow[e >> 1] += pv;
            }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < kFaKeys / 16; ++kk) {
            uint32_t ph[4], pl[4];
            split_pack(sacc[2 * kk][0], sacc[2 * kk][1], ph[0], pl[0]);
            split_pack(sacc[2 * kk][2], sacc[2 * kk][3], ph[1], pl[1]);
            split_pack(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1], ph[2], pl[2]);
            split_pack(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
            for (int dn = 0; dn < OT / 2; ++dn) {
                const int mat = lane >> 3, r8 = lane & 7;
                const int key = kk * 16 + r8 + ((mat & 1) ? 8 : 0), c = 2 * dn + (mat >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(s_v + swz<HD>(key, c), b0, b1, b2, b3);
                mma16816(o[2 * dn], ph, b0, b1);
                mma16816(o[2 * dn], pl, b0, b1);
                mma16816(o[2 * dn + 1], ph, b2, b3);
                mma16816(o[2 * dn + 1], pl, b2, b3);
            }
        }
        __syncthreads();   // the stage is reloaded two tiles later
    }
    // normalise and store: row -> (head, query), columns head * HD + dim
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
    }
    const int head = g * G + row0 / QB;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = qw + gid + 8 * h;
        if (q >= a.n) continue;
        const float inv = 1.0f / lrow[h];
        const size_t ob = ((size_t)i * a.n + q) * a.qh * HD + (size_t)head * HD;
#pragma unroll
        for (int t = 0; t < OT; ++t) {
            const int d = t * 8 + t4 * 2;
            uint32_t hi, lo;
            split_pack(o[t][2 * h] * inv, o[t][2 * h + 1] * inv, hi, lo);
            *reinterpret_cast<uint32_t *>(a.out_hi + ob + d) = hi;
            *reinterpret_cast<uint32_t *>(a.out_lo + ob + d) = lo;
        }
    }
}

typedef void (*FaFn)(const PrefillAttnArgs);
FaFn fa_fn(int hd, int group) {
#define QD_FA(HDV, GV) \
    if (hd == HDV && group == GV) return prefill_attn_kernel<HDV, GV>;
    QD_FA(128, 1) QD_FA(128, 2) QD_FA(128, 4) QD_FA(128, 8)
    QD_FA(64, 1) QD_FA(64, 2) QD_FA(64, 4) QD_FA(64, 8)
#undef QD_FA
    return nullptr;
}
size_t fa_smem(int hd) { return 2 * (size_t)128 * hd * 2 + 2 * 2 * (size_t)kFaKeys * hd * 2; }

}  // namespace

bool prefill_attention_supported(int hd, int group) { return fa_fn(hd, group) != nullptr; }

cudaError_t prefill_kernels_init() {
    for (int hd : {64, 128})
        for (int g : {1, 2, 4, 8}) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fa_fn(hd, g)),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fa_smem(hd));
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_prefill_attention(int hd, int ns, const PrefillAttnArgs &a, cudaStream_t s) {
    const int G = a.qh / a.kvh;
    const FaFn fn = a.qh % a.kvh ? nullptr : fa_fn(hd, G);
    if (!fn) return cudaErrorInvalidValue;
    const int QB = 128 / G;
    const int nqb = (a.n + QB - 1) / QB;
    fn<<<ns * a.kvh * nqb, kFaThreads, fa_smem(hd), s>>>(a);
    return cudaGetLastError();
}
}  // namespace qd

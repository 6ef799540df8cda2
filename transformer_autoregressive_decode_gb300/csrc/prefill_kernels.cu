// Kernels of the batched prefill (ns prompt streams x n positions) other than the
// tensor-core GEMMs and the attention (prefill_attn_tc.cu): QK-norm + RoPE + cache
// append of every prompt position, and the first-id argmax.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation" (QK-norm over head_dim, GQA, plain RoPE) and section "Integration and
//    performance optimisation" (the prompt is prefilled once; decoding continues from
//    its cache).
//  - "Audio8-ASR: dynamic KV-cache buckets", section "Implemented dynamic window
//    mechanism": a fixed-length prefill produces the first token.
//
#include "decode_common.cuh"

namespace qd {

namespace {

// ---- QK-norm + RoPE + append, one CTA (8 warps) per prompt token
constexpr int kPqThreads = 256;

// N consecutive floats (16- or 8-byte aligned for N = 4 or 2) in one load, through L2.
template <int N> __device__ __forceinline__ void load_f32(const float *p, float *v) {
    if constexpr (N == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(p));
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    } else {
        static_assert(N == 2, "elements per lane");
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(p));
        v[0] = t.x, v[1] = t.y;
    }
}
// N consecutive bf16 (8- or 4-byte aligned for N = 4 or 2) in one store.
template <int N> __device__ __forceinline__ void store_bf16(__nv_bfloat16 *p, const __nv_bfloat16 *h) {
    if constexpr (N == 4) {
        __nv_bfloat162 a2 = __halves2bfloat162(h[0], h[1]), b2 = __halves2bfloat162(h[2], h[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a2);
        u.y = *reinterpret_cast<uint32_t *>(&b2);
        *reinterpret_cast<uint2 *>(p) = u;
    } else {
        static_assert(N == 2, "elements per lane");
        *reinterpret_cast<__nv_bfloat162 *>(p) = __halves2bfloat162(h[0], h[1]);
    }
}

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
    // the lane's rotary cos / sin (dims lane * DPL .. of the rotate-half pairs, at position
    // j or the prompt's rotary positions) and gammas: the same for every head of the token
    float rcos[DPL], rsin[DPL], gq[DPL], gk[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        const int m = (lane & 15) * DPL + e;
        const size_t r = (size_t)rope_row(m, a.mrope_h, a.rope_pos, a.rope_stride, j, j, a.rope_rows);
        rcos[e] = a.rope_cos[r * HALF + m];
        rsin[e] = a.rope_sin[r * HALF + m];
        gq[e] = a.q_gamma ? a.q_gamma[lane * DPL + e] : 1.f;
        gk[e] = a.k_gamma ? a.k_gamma[lane * DPL + e] : 1.f;
    }
    // vectors: q heads 0..qh-1, k heads qh..qh+kvh-1 (normed, rotated), v heads (copied)
    for (int vec = warp; vec < a.qh + 2 * a.kvh; vec += kPqThreads / 32) {
        float v[DPL];
        load_f32<DPL>(row + (size_t)vec * HD + lane * DPL, v);
        if (vec < a.qh + a.kvh) {
            const bool isq = vec < a.qh;
            if (isq ? a.q_gamma != nullptr : a.k_gamma != nullptr) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) ss = fmaf(v[e], v[e], ss);
                ss = warp_sum(ss);
                const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
#pragma unroll
                for (int e = 0; e < DPL; ++e) v[e] = v[e] * inv * (isq ? gq[e] : gk[e]);
            }
            // rotate-half RoPE: dims d and d + HD/2 sit 16 lanes apart
            float w[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) w[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
            const bool low = lane < 16;
#pragma unroll
            for (int e = 0; e < DPL; ++e) v[e] = low ? v[e] * rcos[e] - w[e] * rsin[e] : v[e] * rcos[e] + w[e] * rsin[e];
        }
        if (vec < a.qh) {
            const size_t o = (((size_t)i * a.qh + vec) * a.n + j) * HD + lane * DPL;
            __nv_bfloat16 h[DPL], l[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                h[e] = __float2bfloat16_rn(v[e]);
                l[e] = __float2bfloat16_rn(v[e] - __bfloat162float(h[e]));
            }
            store_bf16<DPL>(a.q_hi + o, h);
            store_bf16<DPL>(a.q_lo + o, l);
        } else {
            const bool isk = vec < a.qh + a.kvh;
            const int g = isk ? vec - a.qh : vec - a.qh - a.kvh;
            __nv_bfloat16 *dst = (isk ? kc : vc) + ((size_t)g * a.S + j) * HD + lane * DPL;
            __nv_bfloat16 h[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) h[e] = __float2bfloat16_rn(v[e]);
            store_bf16<DPL>(dst, h);
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


}  // namespace qd

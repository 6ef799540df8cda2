// C-ABI entry points of the batched paths: the tensor-core contraction tap and the
// multi-stream decode.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "qd_model.h"

using namespace qd;

namespace {

struct DevBuf {
    void *p = nullptr;
    ~DevBuf() {
        if (p) cudaFree(p);
    }
    cudaError_t alloc(size_t bytes) { return cudaMalloc(&p, std::max<size_t>(bytes, 16)); }
};

}  // namespace

extern "C" {

qd_status qd_gemm_bf16(const void *w_dev, const float *x_dev, float *out_dev, int R, int K, int T, int mode,
                       void *cuda_stream, int reps, float *avg_ms) {
    if (!is_device_ptr(w_dev) || !is_device_ptr(x_dev) || !is_device_ptr(out_dev)) return QD_EINVAL;
    if (mode < TC_STORE || mode > TC_SWIGLU) return QD_EINVAL;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return QD_ECUDA;
    TcGemmPlan plan;
    if (!tc_gemm_plan(R, K, T, sms, &plan)) return QD_EUNSUPPORTED;
    if (tc_gemm_init() != cudaSuccess) return QD_ECUDA;
    if (reinterpret_cast<uintptr_t>(w_dev) & 15) return QD_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const size_t nx = (size_t)T * K;
    DevBuf xh, xl, part, cnt, st, ah, al;
    if (xh.alloc(nx * 2) || xl.alloc(nx * 2) || part.alloc(plan.partial_floats * 4) ||
        cnt.alloc((size_t)plan.row_tiles * plan.tok_tiles * 8) || st.alloc(4) ||
        ah.alloc((size_t)T * (R / 2) * 2) || al.alloc((size_t)T * (R / 2) * 2))
        return QD_ENOMEM;
    if (cudaMemsetAsync(cnt.p, 0, (size_t)plan.row_tiles * plan.tok_tiles * 8, s) ||
        cudaMemsetAsync(st.p, 0, 4, s))
        return QD_ECUDA;
    if (launch_split_bf16(x_dev, static_cast<__nv_bfloat16 *>(xh.p), static_cast<__nv_bfloat16 *>(xl.p), nx, s))
        return QD_ECUDA;
    TcGemmArgs a = {};
    a.R = R;
    a.K = K;
    a.T = T;
    a.mode = mode;
    a.out = out_dev;
    a.ldo = mode == TC_SWIGLU ? R / 2 : R;
    a.act_hi = static_cast<__nv_bfloat16 *>(ah.p);
    a.act_lo = static_cast<__nv_bfloat16 *>(al.p);
    a.partial = plan.splits > 1 ? static_cast<float *>(part.p) : nullptr;
    a.tile_counter = static_cast<int *>(cnt.p);
    a.status = static_cast<int *>(st.p);
    if (launch_tc_gemm(plan, w_dev, xh.p, xl.p, a, s)) return QD_ECUDA;
    if (avg_ms) {
        if (reps < 1) return QD_EINVAL;
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) || cudaEventCreate(&e1)) return QD_ECUDA;
        cudaEventRecord(e0, s);
        for (int i = 0; i < reps; ++i)
            if (launch_tc_gemm(plan, w_dev, xh.p, xl.p, a, s)) return QD_ECUDA;
        cudaEventRecord(e1, s);
        cudaEventSynchronize(e1);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        *avg_ms = ms / reps;
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
    }
    int status = 0;
    if (cudaMemcpyAsync(&status, st.p, 4, cudaMemcpyDeviceToHost, s) || cudaStreamSynchronize(s)) return QD_ECUDA;
    return status ? QD_EDEVICE : QD_OK;
}

}  // extern "C"

// ====================================================================================
// Batched multi-stream decode: B independent streams over one model's weights.
//
// Per step, for every stream at once: embedding gather of each stream's input token
// (it joins that stream's emitted set) fused with the first RMSNorm; per layer the
// fused QKV projection as a tensor-core GEMM (M = 128 weight rows, N = the streams),
// attention of every stream over its own cache and length (QK-norm, RoPE and the KV
// append in its prologue), the output projection GEMM with the residual add, RMSNorm,
// the gate/up GEMM with SwiGLU in its epilogue, the down GEMM with the residual add;
// then the final RMSNorm, the head GEMM and the per-stream penalty + argmax, which
// feeds each stream's id (or the caller's forced id) back as its next input.  One
// CUDA graph holds a whole step; the step index and the output pointers live in a
// device control block.
// ====================================================================================

struct qd_batch {
    qd_model *m = nullptr;
    int B = 0, S = 0;
    cudaStream_t ls = nullptr;
    void *arena = nullptr;
    void *kv = nullptr;
    size_t stream_elems = 0;
    CUtensorMap kv_map;           // the caches as [S][hd] planes, for the attention's TMA loads
    float *x = nullptr, *qkv = nullptr, *logits = nullptr, *rope_cos = nullptr, *rope_sin = nullptr;
    __nv_bfloat16 *xh = nullptr, *xl = nullptr, *ah = nullptr, *al = nullptr;
    // the next RMSNorm's input: bf16 hi/lo parts of gamma * x [B][hidden] and the sums of
    // squares of x per 32 rows [hidden / 32][B] (written by the residual GEMMs'
    // epilogue; the GEMM that consumes them applies the norm's scale)
    __nv_bfloat16 *nh = nullptr, *nl = nullptr;
    float *ssp = nullptr;
    float *partial = nullptr;
    float *att_part = nullptr;   // attention chunk records [B * kvh][chunks][G][hd + 2]
    int *att_count = nullptr;    // [B * kvh]
    int *counters = nullptr, *pos = nullptr, *status = nullptr;
    int32_t *tokens = nullptr;
    uint32_t *emitted = nullptr;
    int words = 0;
    BatchCtl *ctl = nullptr;
    BatchSampling *samp = nullptr;   // device; top_k 0 = greedy
    int *drawn = nullptr;            // [B] draws of each stream since it was set
    TcGemmPlan p_qkv{}, p_o{}, p_gu{}, p_d{}, p_head{};
    std::vector<int> h_pos;     // host view of each stream's position
    std::vector<char> h_ready;  // stream has a cache and an input token
    cudaGraphExec_t graph = nullptr;
    bool use_graphs = true;
    long long launches = 0;
    int kernels_per_step = 0;
    // prefill scratch, sized for the largest prefill so far (tokens)
    void *pf_arena = nullptr;
    size_t pf_tokens = 0, pf_ns = 0, pf_part_cap = 0, pf_tiles_cap = 0;
    float *pf_partial = nullptr;   // split-K partials of the prefill GEMMs
    int *pf_counters = nullptr;    // their tile counters, zero at rest
    float *pf_x = nullptr, *pf_qkv = nullptr, *pf_last = nullptr, *pf_logits = nullptr;
    __nv_bfloat16 *pf_xh = nullptr, *pf_xl = nullptr, *pf_ah = nullptr, *pf_al = nullptr, *pf_qh = nullptr,
                  *pf_ql = nullptr;
    int *pf_streams = nullptr;
};

namespace {

constexpr size_t kAlign = 256;

qd_status batch_fail(qd_batch *b, qd_status st, const char *what) { return fail(b->m, st, "%s", what); }

// The RMSNorms between the step's GEMMs: `next_gamma` makes a residual GEMM also write
// the next norm's input parts and sums of squares (TC_RESIDUAL_NORM); `scaled` makes a
// GEMM apply the norm's scale from those sums to its products.
struct NormFold {
    const float *next_gamma = nullptr;
    bool scaled = false;
};

// One tensor-core GEMM of the step over the B streams.
cudaError_t batch_gemm(qd_batch *b, const TcGemmPlan &p, const void *w, const __nv_bfloat16 *xh,
                       const __nv_bfloat16 *xl, int R, int K, int mode, float *out, int ldo, cudaStream_t s,
                       bool pdl = false, NormFold nf = NormFold()) {
    TcGemmArgs a = {};
    const qd_config &c = b->m->cfg;
    if (nf.next_gamma) {
        mode = TC_RESIDUAL_NORM;
        a.norm_gamma = nf.next_gamma;
        a.nh = b->nh;
        a.nl = b->nl;
        a.ss_out = b->ssp;
    }
    if (nf.scaled) {
        a.rs_part = b->ssp;
        a.rs_tiles = c.hidden / 32;
        a.rs_K = c.hidden;
        a.rs_eps = (float)c.rms_eps;
    }
    a.R = R;
    a.K = K;
    a.T = b->B;
    a.mode = mode;
    a.out = out;
    a.ldo = ldo;
    a.act_hi = b->ah;
    a.act_lo = b->al;
    a.partial = p.splits > 1 ? b->partial : nullptr;
    a.tile_counter = b->counters;
    a.status = b->status;
    return launch_tc_gemm(p, w, xh, xl, a, s, pdl);
}

// Attention arguments of layer l (output: the bf16 parts feeding the O GEMM).
BatchAttnArgs batch_attn_args(qd_batch *b, int l) {
    const qd_model *m = b->m;
    const qd_config &c = m->cfg;
    const Layer &L = m->layers[l];
    BatchAttnArgs at = {};
    at.qkv = b->qkv;
    at.qkv_ld = m->q_dim() + 2 * m->kv_dim();
    at.q_gamma = c.qk_norm ? L.q_norm : nullptr;
    at.k_gamma = c.qk_norm ? L.k_norm : nullptr;
    at.eps = (float)c.rms_eps;
    at.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
    at.rope_cos = b->rope_cos;
    at.rope_sin = b->rope_sin;
    at.kv = b->kv;
    at.stream_elems = b->stream_elems;
    at.layer_elems = (size_t)l * 2 * c.n_kv_heads * b->S * c.head_dim;
    at.S = b->S;
    at.qh = c.n_q_heads;
    at.kvh = c.n_kv_heads;
    at.partial = b->att_part;
    at.counter = b->att_count;
    at.pos = b->pos;
    at.out_hi = b->xh;
    at.out_lo = b->xl;
    at.status = b->status;
    return at;
}

// Every launch of one step, on stream s.
qd_status enqueue_batch_step(qd_batch *b, cudaStream_t s) {
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    const int B = b->B, h = c.hidden, qd_ = m->q_dim(), rows_qkv = qd_ + 2 * m->kv_dim();
    int n = 0;
    auto norm = [&](const float *gamma, bool gather) -> cudaError_t {
        NormSplitArgs a = {};
        a.x = b->x;
        a.K = h;
        a.gamma = gamma;
        a.eps = (float)c.rms_eps;
        a.hi = b->nh;
        a.lo = b->nl;
        if (gather) {
            a.table = m->embed;
            a.table_rows = c.embed_rows;
            a.tokens = b->tokens;
            a.emitted = b->emitted;
            a.emitted_words = b->words;
            a.vocab = c.vocab;
        }
        a.status = b->status;
        ++n;
        return launch_norm_split(a, B, s, true);
    };
    auto gemm = [&](const TcGemmPlan &p, const void *w, const __nv_bfloat16 *xh, const __nv_bfloat16 *xl, int R,
                    int K, int mode, float *out, int ldo, NormFold nf = NormFold()) -> cudaError_t {
        ++n;
        return batch_gemm(b, p, w, xh, xl, R, K, mode, out, ldo, s, true, nf);
    };
    // Only the step's first RMSNorm (with the embedding gather) is a kernel of its own;
    // each later one is folded into the GEMMs around it: the residual GEMM before it
    // writes gamma * x as bf16 parts and the per-tile sums of squares, the GEMM after it
    // scales its products by 1 / sqrt(mean(x^2) + eps).
    if (norm(m->layers[0].attn_norm, true)) return batch_fail(b, QD_ECUDA, "norm/embedding launch failed");
    for (int l = 0; l < c.n_layers; ++l) {
        const Layer &L = m->layers[l];
        NormFold in_qkv;
        in_qkv.scaled = l > 0;
        if (gemm(b->p_qkv, L.w_qkv, b->nh, b->nl, rows_qkv, h, TC_STORE, b->qkv, rows_qkv, in_qkv))
            return batch_fail(b, QD_ECUDA, "QKV GEMM launch failed");
        ++n;
        if (launch_batch_attention(c.head_dim, B, batch_attn_args(b, l), b->kv_map, s, true))
            return batch_fail(b, QD_ECUDA, "attention launch failed");
        NormFold o_out;
        o_out.next_gamma = L.mlp_norm;
        if (gemm(b->p_o, L.w_o, b->xh, b->xl, h, qd_, TC_RESIDUAL, b->x, h, o_out))
            return batch_fail(b, QD_ECUDA, "O GEMM launch failed");
        NormFold gu_in;
        gu_in.scaled = true;
        if (gemm(b->p_gu, L.w_gu, b->nh, b->nl, 2 * c.ffn, h, TC_SWIGLU, nullptr, c.ffn, gu_in))
            return batch_fail(b, QD_ECUDA, "gate/up GEMM launch failed");
        NormFold d_out;
        d_out.next_gamma = l + 1 < c.n_layers ? m->layers[l + 1].attn_norm : m->final_norm;
        if (gemm(b->p_d, L.w_d, b->ah, b->al, h, c.ffn, TC_RESIDUAL, b->x, h, d_out))
            return batch_fail(b, QD_ECUDA, "down GEMM launch failed");
    }
    NormFold head_in;
    head_in.scaled = true;
    if (gemm(b->p_head, m->heads[0], b->nh, b->nl, c.vocab, h, TC_STORE, b->logits, c.vocab, head_in))
        return batch_fail(b, QD_ECUDA, "head GEMM launch failed");
    BatchArgmaxArgs am = {};
    am.logits = b->logits;
    am.V = c.vocab;
    am.emitted = b->emitted;
    am.words = b->words;
    am.penalty = (float)c.rep_penalty;
    am.eos = c.eos_mask_id;
    am.ctl = b->ctl;
    am.tokens = b->tokens;
    am.pos = b->pos;
    am.status = b->status;
    am.samp = b->samp;
    am.drawn = b->drawn;
    ++n;
    if (launch_batch_argmax(am, B, s, true)) return batch_fail(b, QD_ECUDA, "argmax launch failed");
    b->kernels_per_step = n;
    return QD_OK;
}

// One kernel of the step with the step's arguments, for timing: 1 = attention of the
// last layer at the current positions (it rewrites the row each stream would write
// next, which the next step overwrites), 2..6 = the QKV, O, gate/up, down GEMMs of layer
// 0 and the head GEMM (they overwrite step scratch only).
qd_status enqueue_batch_kernel(qd_batch *b, int which, cudaStream_t s) {
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    const int h = c.hidden, qd_ = m->q_dim(), rows_qkv = qd_ + 2 * m->kv_dim();
    const Layer &L0 = m->layers[0];
    cudaError_t e = cudaSuccess;
    switch (which) {
        case 1: e = launch_batch_attention(c.head_dim, b->B, batch_attn_args(b, c.n_layers - 1), b->kv_map, s); break;
        case 2: e = batch_gemm(b, b->p_qkv, L0.w_qkv, b->nh, b->nl, rows_qkv, h, TC_STORE, b->qkv, rows_qkv, s); break;
        case 3: {
            NormFold nf;
            nf.next_gamma = L0.mlp_norm;
            e = batch_gemm(b, b->p_o, L0.w_o, b->xh, b->xl, h, qd_, TC_RESIDUAL, b->x, h, s, false, nf);
            break;
        }
        case 4: {
            NormFold nf;
            nf.scaled = true;
            e = batch_gemm(b, b->p_gu, L0.w_gu, b->nh, b->nl, 2 * c.ffn, h, TC_SWIGLU, nullptr, c.ffn, s, false, nf);
            break;
        }
        case 5: {
            NormFold nf;
            nf.next_gamma = c.n_layers > 1 ? m->layers[1].attn_norm : m->final_norm;
            e = batch_gemm(b, b->p_d, L0.w_d, b->ah, b->al, h, c.ffn, TC_RESIDUAL, b->x, h, s, false, nf);
            break;
        }
        case 6: {
            NormFold nf;
            nf.scaled = true;
            e = batch_gemm(b, b->p_head, m->heads[0], b->nh, b->nl, c.vocab, h, TC_STORE, b->logits, c.vocab, s, false, nf);
            break;
        }
        default: return fail(m, QD_EINVAL, "kernel %d: use 1..6", which);
    }
    CU(e);
    return QD_OK;
}

// The five contractions of a prefill of ns streams x n positions.
bool prefill_plans(const qd_model *m, int ns, int n, TcGemmPlan *p) {
    const qd_config &c = m->cfg;
    const int h = c.hidden, T = ns * n;
    return tc_gemm_plan(m->q_dim() + 2 * m->kv_dim(), h, T, m->num_sms, &p[0]) &&
           tc_gemm_plan(h, m->q_dim(), T, m->num_sms, &p[1]) && tc_gemm_plan(2 * c.ffn, h, T, m->num_sms, &p[2]) &&
           tc_gemm_plan(h, c.ffn, T, m->num_sms, &p[3]) && tc_gemm_plan(c.vocab, h, ns, m->num_sms, &p[4]);
}

// Prefill scratch for ns streams of n positions (grown, never shrunk).
qd_status ensure_prefill_scratch(qd_batch *b, int ns, int n) {
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    const size_t T = (size_t)ns * n;
    TcGemmPlan plans[5];
    if (!prefill_plans(m, ns, n, plans)) return fail(m, QD_EUNSUPPORTED, "prefill GEMM shapes");
    size_t part = 1, tiles = 1;
    for (const TcGemmPlan &p : plans) {
        part = std::max(part, p.partial_floats);
        tiles = std::max(tiles, (size_t)p.row_tiles * p.tok_tiles);
    }
    if (b->pf_arena && T <= b->pf_tokens && (size_t)ns <= b->pf_ns && part <= b->pf_part_cap &&
        tiles <= b->pf_tiles_cap)
        return QD_OK;
    if (b->pf_arena) {
        CU(cudaStreamSynchronize(b->ls));
        cudaFree(b->pf_arena);
        b->pf_arena = nullptr;
    }
    const int h = c.hidden, rows_qkv = m->q_dim() + 2 * m->kv_dim();
    const size_t kmax = std::max({(size_t)h, (size_t)m->q_dim(), (size_t)c.ffn});
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = (off + bytes + kAlign - 1) / kAlign * kAlign;
        return o;
    };
    const size_t o_x = take(T * h * 4), o_qkv = take(T * rows_qkv * 4), o_xh = take(T * kmax * 2),
                 o_xl = take(T * kmax * 2), o_ah = take(T * c.ffn * 2), o_al = take(T * c.ffn * 2),
                 o_qh = take(T * m->q_dim() * 2), o_ql = take(T * m->q_dim() * 2), o_last = take((size_t)ns * h * 4),
                 o_lg = take((size_t)ns * c.vocab * 4), o_st = take((size_t)ns * 4), o_part = take(part * 4),
                 o_cnt = take(tiles * 8);
    void *p = nullptr;
    CU(cudaMalloc(&p, off));
    uint8_t *A = static_cast<uint8_t *>(p);
    b->pf_arena = p;
    b->pf_tokens = T;
    b->pf_ns = ns;
    b->pf_part_cap = part;
    b->pf_tiles_cap = tiles;
    b->pf_partial = reinterpret_cast<float *>(A + o_part);
    b->pf_counters = reinterpret_cast<int *>(A + o_cnt);
    CU(cudaMemsetAsync(b->pf_counters, 0, tiles * 8, b->ls));
    b->pf_x = reinterpret_cast<float *>(A + o_x);
    b->pf_qkv = reinterpret_cast<float *>(A + o_qkv);
    b->pf_xh = reinterpret_cast<__nv_bfloat16 *>(A + o_xh);
    b->pf_xl = reinterpret_cast<__nv_bfloat16 *>(A + o_xl);
    b->pf_ah = reinterpret_cast<__nv_bfloat16 *>(A + o_ah);
    b->pf_al = reinterpret_cast<__nv_bfloat16 *>(A + o_al);
    b->pf_qh = reinterpret_cast<__nv_bfloat16 *>(A + o_qh);
    b->pf_ql = reinterpret_cast<__nv_bfloat16 *>(A + o_ql);
    b->pf_last = reinterpret_cast<float *>(A + o_last);
    b->pf_logits = reinterpret_cast<float *>(A + o_lg);
    b->pf_streams = reinterpret_cast<int *>(A + o_st);
    return QD_OK;
}

// Every launch of a prefill of ns streams x n positions, on the batch's stream.  With
// with_head false it stops after gathering each stream's last hidden state into
// pf_last (the caller runs a head on it).
qd_status enqueue_prefill(qd_batch *b, int ns, int n, int32_t *first_ids, bool with_head = true,
                          const int *rope_pos = nullptr, int rope_stride = 0) {
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    const int h = c.hidden, qd_ = m->q_dim(), rows_qkv = qd_ + 2 * m->kv_dim();
    const int T = ns * n;
    cudaStream_t s = b->ls;
    TcGemmPlan plans[5];
    if (!prefill_plans(m, ns, n, plans)) return fail(m, QD_EUNSUPPORTED, "prefill GEMM shapes");
    const TcGemmPlan &p_qkv = plans[0], &p_o = plans[1], &p_gu = plans[2], &p_d = plans[3], &p_head = plans[4];
    auto gemm = [&](const TcGemmPlan &p, const void *w, const __nv_bfloat16 *xh, const __nv_bfloat16 *xl, int R,
                    int K, int rows, int mode, float *out, int ldo) -> cudaError_t {
        TcGemmArgs a = {};
        a.R = R;
        a.K = K;
        a.T = rows;
        a.mode = mode;
        a.out = out;
        a.ldo = ldo;
        a.act_hi = b->pf_ah;
        a.act_lo = b->pf_al;
        a.partial = p.splits > 1 ? b->pf_partial : nullptr;
        a.tile_counter = b->pf_counters;
        a.status = b->status;
        b->launches++;
        return launch_tc_gemm(p, w, xh, xl, a, s);
    };
    auto norm = [&](float *x, int rows, const float *gamma) -> cudaError_t {
        NormSplitArgs a = {};
        a.x = x;
        a.K = h;
        a.gamma = gamma;
        a.eps = (float)c.rms_eps;
        a.hi = b->pf_xh;
        a.lo = b->pf_xl;
        a.status = b->status;
        b->launches++;
        return launch_norm_split(a, rows, s);
    };
    PrefillAttnMaps fmaps;
    for (int l = 0; l < c.n_layers; ++l) {
        const Layer &L = m->layers[l];
        if (norm(b->pf_x, T, L.attn_norm)) return batch_fail(b, QD_ECUDA, "prefill norm launch failed");
        if (gemm(p_qkv, L.w_qkv, b->pf_xh, b->pf_xl, rows_qkv, h, T, TC_STORE, b->pf_qkv, rows_qkv))
            return batch_fail(b, QD_ECUDA, "prefill QKV GEMM launch failed");
        PrefillQkArgs qa = {};
        qa.qkv = b->pf_qkv;
        qa.qkv_ld = rows_qkv;
        qa.n = n;
        qa.qh = c.n_q_heads;
        qa.kvh = c.n_kv_heads;
        qa.q_gamma = c.qk_norm ? L.q_norm : nullptr;
        qa.k_gamma = c.qk_norm ? L.k_norm : nullptr;
        qa.eps = (float)c.rms_eps;
        qa.rope_cos = b->rope_cos;
        qa.rope_sin = b->rope_sin;
        qa.rope_rows = b->S;
        qa.mrope_h = c.mrope_section[1];
        qa.rope_pos = rope_pos;
        qa.rope_stride = rope_stride;
        qa.kv = b->kv;
        qa.stream_elems = b->stream_elems;
        qa.layer_elems = (size_t)l * 2 * c.n_kv_heads * b->S * c.head_dim;
        qa.S = b->S;
        qa.streams = b->pf_streams;
        qa.q_hi = b->pf_qh;
        qa.q_lo = b->pf_ql;
        b->launches++;
        if (launch_prefill_qk(c.head_dim, ns, qa, s)) return batch_fail(b, QD_ECUDA, "prefill q/k launch failed");
        PrefillAttnArgs fa = {};
        fa.q_hi = b->pf_qh;
        fa.q_lo = b->pf_ql;
        fa.kv = b->kv;
        fa.stream_elems = b->stream_elems;
        fa.layer_elems = qa.layer_elems;
        fa.S = b->S;
        fa.n = n;
        fa.qh = c.n_q_heads;
        fa.kvh = c.n_kv_heads;
        fa.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
        fa.streams = b->pf_streams;
        fa.out_hi = b->pf_xh;
        fa.out_lo = b->pf_xl;
        fa.status = b->status;
        fa.cache_streams = b->B;
        if (l == 0 && !make_prefill_attn_maps(c.head_dim, ns, fa, &fmaps))
            return batch_fail(b, QD_ECUDA, "prefill attention tensor maps refused");
        b->launches++;
        if (launch_prefill_attention_tc(c.head_dim, ns, fa, fmaps, s))
            return batch_fail(b, QD_ECUDA, "prefill attention launch failed");
        if (gemm(p_o, L.w_o, b->pf_xh, b->pf_xl, h, qd_, T, TC_RESIDUAL, b->pf_x, h))
            return batch_fail(b, QD_ECUDA, "prefill O GEMM launch failed");
        if (norm(b->pf_x, T, L.mlp_norm)) return batch_fail(b, QD_ECUDA, "prefill norm launch failed");
        if (gemm(p_gu, L.w_gu, b->pf_xh, b->pf_xl, 2 * c.ffn, h, T, TC_SWIGLU, nullptr, c.ffn))
            return batch_fail(b, QD_ECUDA, "prefill gate/up GEMM launch failed");
        if (gemm(p_d, L.w_d, b->pf_ah, b->pf_al, h, c.ffn, T, TC_RESIDUAL, b->pf_x, h))
            return batch_fail(b, QD_ECUDA, "prefill down GEMM launch failed");
    }
    // the head on each stream's last position
    b->launches++;
    if (launch_gather_last(b->pf_x, n, h, ns, b->pf_last, s)) return batch_fail(b, QD_ECUDA, "gather launch failed");
    if (!with_head) return QD_OK;
    if (norm(b->pf_last, ns, m->final_norm)) return batch_fail(b, QD_ECUDA, "prefill norm launch failed");
    if (gemm(p_head, m->heads[0], b->pf_xh, b->pf_xl, c.vocab, h, ns, TC_STORE, b->pf_logits, c.vocab))
        return batch_fail(b, QD_ECUDA, "prefill head GEMM launch failed");
    PrefillFinishArgs fin = {};
    fin.logits = b->pf_logits;
    fin.V = c.vocab;
    fin.eos = c.eos_mask_id;
    fin.streams = b->pf_streams;
    fin.n = n;
    fin.first_ids = first_ids;
    fin.logits_out = b->logits;
    fin.tokens = b->tokens;
    fin.pos = b->pos;
    fin.status = b->status;
    b->launches++;
    if (launch_prefill_finish(fin, ns, s)) return batch_fail(b, QD_ECUDA, "prefill finish launch failed");
    return QD_OK;
}

qd_status run_batch_step(qd_batch *b) {
    qd_model *m = b->m;
    if (!b->use_graphs) return enqueue_batch_step(b, b->ls);
    if (!b->graph) {
        cudaGraph_t g = nullptr;
        CU(cudaStreamBeginCapture(b->ls, cudaStreamCaptureModeThreadLocal));
        qd_status st = enqueue_batch_step(b, b->ls);
        cudaError_t ce = cudaStreamEndCapture(b->ls, &g);
        if (st) {
            if (g) cudaGraphDestroy(g);
            return st;
        }
        CU(ce);
        cudaError_t ie = cudaGraphInstantiate(&b->graph, g, 0);
        cudaGraphDestroy(g);
        CU(ie);
    }
    CU(cudaGraphLaunch(b->graph, b->ls));
    return QD_OK;
}

void destroy_batch(qd_batch *b) {
    if (!b) return;
    if (b->ls) cudaStreamSynchronize(b->ls);
    if (b->graph) cudaGraphExecDestroy(b->graph);
    if (b->pf_arena) cudaFree(b->pf_arena);
    if (b->arena) cudaFree(b->arena);
    if (b->kv) cudaFree(b->kv);
    if (b->ls) cudaStreamDestroy(b->ls);
    delete b;
}

// Order the batch's stream after the model's caller stream and back.
void batch_enter(qd_batch *b) {
    cudaEventRecord(b->m->ev_in, b->m->user);
    cudaStreamWaitEvent(b->ls, b->m->ev_in, 0);
}
void batch_leave(qd_batch *b) {
    cudaEventRecord(b->m->ev_out, b->ls);
    cudaStreamWaitEvent(b->m->user, b->m->ev_out, 0);
}

}  // namespace

// qd_prefill through the batched prefill kernels: an internal one-stream batch over the
// model's weights runs the prompt's layers (device embeddings, or device token ids
// whose embedding rows are gathered first); its K/V rows [0, n) are copied into the
// model's bucket buffer and the last position's hidden state into the model's x, and
// the model's position becomes n - 1.  The model's stream waits for it; the caller then
// runs the model's head step, which gives the first id (greedy or sampled, like every
// later step) and advances the position to n.  QD_EUNSUPPORTED, with nothing enqueued,
// when the model or the shapes do not allow it.
qd_status model_prefill_batched(qd_model *m, const float *embeds_dev, const int32_t *tokens_dev, int n, int bucket,
                                const int *rope_pos, int rope_stride) {
    const qd_config &c = m->cfg;
    TcGemmPlan plans[5];
    if (!m->bf16 || m->q8 || c.n_heads_out != 1 || !m->embed || !prefill_plans(m, 1, n, plans)) return QD_EUNSUPPORTED;
    if (!m->pf_batch) {
        qd_batch_handle nb = nullptr;
        const std::string err = m->err;
        if (qd_batch_create(m, 1, m->max_pos, &nb) != QD_OK) {
            m->err = err;   // not an error of the caller's: the per-step prefill runs instead
            return QD_EUNSUPPORTED;
        }
        m->pf_batch = nb;
        CU(cudaEventCreateWithFlags(&m->pf_ev[0], cudaEventDisableTiming));
        CU(cudaEventCreateWithFlags(&m->pf_ev[1], cudaEventDisableTiming));
    }
    qd_batch *b = m->pf_batch;
    CU(cudaEventRecord(m->pf_ev[0], m->ls));
    CU(cudaStreamWaitEvent(b->ls, m->pf_ev[0], 0));
    qd_status st = ensure_prefill_scratch(b, 1, n);
    if (st) return st;
    const long long l0 = b->launches;
    CU(cudaMemsetAsync(b->pf_streams, 0, sizeof(int), b->ls));   // stream 0
    CU(cudaMemsetAsync(b->status, 0, sizeof(int), b->ls));
    if (tokens_dev) {
        CU(launch_embed_rows(m->embed, tokens_dev, n, c.hidden, b->pf_x, b->ls));
        ++m->launches;
    } else {
        CU(cudaMemcpyAsync(b->pf_x, embeds_dev, (size_t)n * c.hidden * 4, cudaMemcpyDeviceToDevice, b->ls));
    }
    st = enqueue_prefill(b, 1, n, nullptr, false, rope_pos, rope_stride);
    if (st) return st;
    // K/V rows [0, n) of every (layer, K/V, kv head) segment into the model's bucket
    const size_t row = (size_t)c.head_dim * m->esize;
    CU(cudaMemcpy2DAsync(m->kv[bucket], (size_t)c.buckets[bucket] * row, b->kv, (size_t)b->S * row, (size_t)n * row,
                         (size_t)c.n_layers * 2 * c.n_kv_heads, cudaMemcpyDeviceToDevice, b->ls));
    CU(cudaMemcpyAsync(m->x, b->pf_last, (size_t)c.hidden * 4, cudaMemcpyDeviceToDevice, b->ls));
    CU(launch_prefill_commit(m->st, n - 1, b->status, b->ls));
    m->launches += b->launches - l0 + 1;
    CU(cudaEventRecord(m->pf_ev[1], b->ls));
    CU(cudaStreamWaitEvent(m->ls, m->pf_ev[1], 0));
    return QD_OK;
}

extern "C" {

qd_status qd_batch_create(qd_handle model, int n_streams, int smax, qd_batch_handle *out) {
    if (!out) return QD_EINVAL;
    *out = nullptr;
    if (!model) return QD_EINVAL;
    qd_model *m = model;
    const qd_config &c = m->cfg;
    if (n_streams < 1 || n_streams > 1024) return fail(m, QD_EINVAL, "n_streams %d out of range", n_streams);
    if (smax < 32 || smax % 32) return fail(m, QD_EINVAL, "smax must be a positive multiple of 32");
    if (!m->bf16 || m->q8) return fail(m, QD_EUNSUPPORTED, "the batched path needs bf16 weights");
    if (c.n_heads_out != 1 || !m->embed) return fail(m, QD_EUNSUPPORTED, "the batched path needs one head and an embedding table");
    const int rows_qkv = m->q_dim() + 2 * m->kv_dim();
    int sms = m->num_sms;
    qd_batch *b = new qd_batch();
    b->m = m;
    b->B = n_streams;
    b->S = smax;
    if (!tc_gemm_plan(rows_qkv, c.hidden, n_streams, sms, &b->p_qkv) ||
        !tc_gemm_plan(c.hidden, m->q_dim(), n_streams, sms, &b->p_o) ||
        !tc_gemm_plan(2 * c.ffn, c.hidden, n_streams, sms, &b->p_gu) ||
        !tc_gemm_plan(c.hidden, c.ffn, n_streams, sms, &b->p_d) ||
        !tc_gemm_plan(c.vocab, c.hidden, n_streams, sms, &b->p_head)) {
        delete b;
        return fail(m, QD_EUNSUPPORTED, "GEMM shapes: rows must be multiples of 128, K of 64");
    }
    if (!batch_attention_supported(c.head_dim, c.n_q_heads / c.n_kv_heads)) {
        delete b;
        return fail(m, QD_EUNSUPPORTED, "the batched attention takes 1, 2, 4 or 8 q heads per kv head");
    }
    if (batch_attention_smem_bytes(c.head_dim, c.n_q_heads / c.n_kv_heads) > 160 * 1024) {
        delete b;
        return fail(m, QD_EUNSUPPORTED, "smax %d too long for the attention tile", smax);
    }
    if (tc_gemm_init() != cudaSuccess || batch_kernels_init() != cudaSuccess) {
        delete b;
        return fail(m, QD_ECUDA, "tensor-core GEMM or attention kernel setup failed");
    }
    const int B = n_streams, h = c.hidden;
    const int kmax = std::max({h, m->q_dim(), c.ffn});
    b->words = (c.vocab + 31) / 32;
    size_t part = 0;
    int tiles = 0;
    for (const TcGemmPlan *p : {&b->p_qkv, &b->p_o, &b->p_gu, &b->p_d, &b->p_head}) {
        part = std::max(part, p->partial_floats);
        tiles = std::max(tiles, p->row_tiles * p->tok_tiles);
    }
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = (off + bytes + kAlign - 1) / kAlign * kAlign;
        return o;
    };
    const size_t o_x = take((size_t)B * h * 4), o_qkv = take((size_t)B * rows_qkv * 4),
                 o_lg = take((size_t)B * c.vocab * 4), o_xh = take((size_t)B * kmax * 2),
                 o_xl = take((size_t)B * kmax * 2), o_ah = take((size_t)B * c.ffn * 2),
                 o_al = take((size_t)B * c.ffn * 2), o_part = take(std::max<size_t>(part, 1) * 4),
                 o_cnt = take((size_t)tiles * 8), o_pos = take((size_t)B * 4), o_st = take(16),
                 o_tok = take((size_t)B * 4), o_em = take((size_t)B * b->words * 4), o_ctl = take(sizeof(BatchCtl)),
                 o_cos = take((size_t)smax * (c.head_dim / 2) * 4), o_sin = take((size_t)smax * (c.head_dim / 2) * 4),
                 o_ap = take((size_t)B * c.n_kv_heads * batch_attn_max_chunks(smax) *
                             (c.n_q_heads / c.n_kv_heads) * (c.head_dim + 2) * 4),
                 o_ac = take((size_t)B * c.n_kv_heads * 4), o_smp = take(sizeof(BatchSampling)),
                 o_drn = take((size_t)B * 4), o_nh = take((size_t)B * h * 2), o_nl = take((size_t)B * h * 2),
                 o_ssp = take((size_t)(h / 32) * B * 4);
    b->stream_elems = (size_t)c.n_layers * 2 * c.n_kv_heads * smax * c.head_dim;
    qd_status st = QD_OK;
    auto check = [&](cudaError_t e, const char *what) {
        if (e != cudaSuccess && !st)
            st = fail(m, e == cudaErrorMemoryAllocation ? QD_ENOMEM : QD_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    };
    check(cudaStreamCreateWithFlags(&b->ls, cudaStreamNonBlocking), "cudaStreamCreate");
    check(cudaMalloc(&b->arena, off), "cudaMalloc(batch scratch)");
    check(cudaMalloc(&b->kv, b->stream_elems * 2 * B), "cudaMalloc(batch KV caches)");
    if (!st) {
        uint8_t *A = static_cast<uint8_t *>(b->arena);
        b->x = reinterpret_cast<float *>(A + o_x);
        b->qkv = reinterpret_cast<float *>(A + o_qkv);
        b->logits = reinterpret_cast<float *>(A + o_lg);
        b->xh = reinterpret_cast<__nv_bfloat16 *>(A + o_xh);
        b->xl = reinterpret_cast<__nv_bfloat16 *>(A + o_xl);
        b->ah = reinterpret_cast<__nv_bfloat16 *>(A + o_ah);
        b->al = reinterpret_cast<__nv_bfloat16 *>(A + o_al);
        b->partial = reinterpret_cast<float *>(A + o_part);
        b->counters = reinterpret_cast<int *>(A + o_cnt);
        b->pos = reinterpret_cast<int *>(A + o_pos);
        b->status = reinterpret_cast<int *>(A + o_st);
        b->tokens = reinterpret_cast<int32_t *>(A + o_tok);
        b->emitted = reinterpret_cast<uint32_t *>(A + o_em);
        b->ctl = reinterpret_cast<BatchCtl *>(A + o_ctl);
        b->rope_cos = reinterpret_cast<float *>(A + o_cos);
        b->rope_sin = reinterpret_cast<float *>(A + o_sin);
        b->att_part = reinterpret_cast<float *>(A + o_ap);
        b->att_count = reinterpret_cast<int *>(A + o_ac);
        b->samp = reinterpret_cast<BatchSampling *>(A + o_smp);
        b->drawn = reinterpret_cast<int *>(A + o_drn);
        b->nh = reinterpret_cast<__nv_bfloat16 *>(A + o_nh);
        b->nl = reinterpret_cast<__nv_bfloat16 *>(A + o_nl);
        b->ssp = reinterpret_cast<float *>(A + o_ssp);
        check(cudaMemsetAsync(b->arena, 0, off, b->ls), "cudaMemsetAsync");
        // positions past a stream's length hold zeros or values this library wrote (the
        // attention loads whole 32-position tiles and gives the rows past a chunk
        // probability 0, which needs them finite)
        check(cudaMemsetAsync(b->kv, 0, b->stream_elems * 2 * B, b->ls), "cudaMemsetAsync(batch KV caches)");
        if (!st && !make_kv_tile_map(&b->kv_map, b->kv, c.head_dim, smax,
                                     (long long)B * c.n_layers * 2 * c.n_kv_heads))
            st = fail(m, QD_EUNSUPPORTED, "TMA map of the batch KV caches refused");
        check(launch_rope_table(b->rope_cos, b->rope_sin, smax, c.head_dim, c.rope_theta, b->ls), "RoPE table");
        check(cudaStreamSynchronize(b->ls), "cudaStreamSynchronize");
    }
    if (st) {
        destroy_batch(b);
        return st;
    }
    b->h_pos.assign(B, 0);
    b->h_ready.assign(B, 0);
    *out = b;
    return QD_OK;
}

qd_status qd_batch_destroy(qd_batch_handle b) {
    destroy_batch(b);
    return QD_OK;
}

qd_status qd_batch_set_graphs(qd_batch_handle b, int enable) {
    if (!b) return QD_EINVAL;
    b->use_graphs = enable != 0;
    return QD_OK;
}

qd_status qd_batch_set_stream(qd_batch_handle b, int stream, const void *kv_dev, int length, int32_t token) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    if (stream < 0 || stream >= b->B) return fail(m, QD_EINVAL, "stream %d out of range", stream);
    if (length < 0 || length >= b->S) return fail(m, QD_EINVAL, "length %d must be in [0, smax)", length);
    if (length > 0 && !is_device_ptr(kv_dev)) return fail(m, QD_EINVAL, "kv_dev is not a device pointer");
    if (token < 0 || token >= c.embed_rows) return fail(m, QD_EINVAL, "token %d outside the embedding table", token);
    batch_enter(b);
    const size_t row = (size_t)c.head_dim * 2;   // bytes of one position of one kv head
    const int segs = c.n_layers * 2 * c.n_kv_heads;
    uint8_t *dst = static_cast<uint8_t *>(b->kv) + (size_t)stream * b->stream_elems * 2;
    if (length > 0)
        CU(cudaMemcpy2DAsync(dst, (size_t)b->S * row, kv_dev, (size_t)length * row, (size_t)length * row, segs,
                             cudaMemcpyDeviceToDevice, b->ls));
    CU(cudaMemcpyAsync(b->pos + stream, &length, 4, cudaMemcpyHostToDevice, b->ls));
    CU(cudaMemcpyAsync(b->tokens + stream, &token, 4, cudaMemcpyHostToDevice, b->ls));
    CU(cudaMemsetAsync(b->emitted + (size_t)stream * b->words, 0, (size_t)b->words * 4, b->ls));
    CU(cudaMemsetAsync(b->drawn + stream, 0, 4, b->ls));
    CU(cudaStreamSynchronize(b->ls));
    batch_leave(b);
    b->h_pos[stream] = length;
    b->h_ready[stream] = 1;
    return QD_OK;
}

qd_status qd_batch_set_sampling(qd_batch_handle b, int top_k, float temperature, float top_p, uint64_t seed) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    if (top_k < 0 || top_k > kMaxTopK) return fail(m, QD_EINVAL, "top_k %d outside [0, %d]", top_k, kMaxTopK);
    if (!(temperature > 0.f) || !(top_p > 0.f) || top_p > 1.f)
        return fail(m, QD_EINVAL, "temperature must be > 0 and top_p in (0, 1]");
    if (top_k > 0 && m->cfg.vocab > kBatchSampleVocabMax)
        return fail(m, QD_EUNSUPPORTED, "batched sampling keeps at most %d logits per stream", kBatchSampleVocabMax);
    BatchSampling h = {};
    h.top_k = top_k;
    h.temperature = temperature;
    h.top_p = top_p;
    h.seed_lo = (uint32_t)seed;
    h.seed_hi = (uint32_t)(seed >> 32);
    batch_enter(b);
    CU(cudaMemcpyAsync(b->samp, &h, sizeof(h), cudaMemcpyHostToDevice, b->ls));
    CU(cudaStreamSynchronize(b->ls));
    batch_leave(b);
    return QD_OK;
}

qd_status qd_batch_decode(qd_batch_handle b, int n_steps, const int32_t *force_dev, int32_t *ids_dev) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    if (n_steps < 0) return fail(m, QD_EINVAL, "n_steps < 0");
    if (n_steps == 0) return QD_OK;
    if (!is_device_ptr(ids_dev)) return fail(m, QD_EINVAL, "ids_dev is not a device pointer");
    if (force_dev && !is_device_ptr(force_dev)) return fail(m, QD_EINVAL, "force_dev is not a device pointer");
    for (int i = 0; i < b->B; ++i) {
        if (!b->h_ready[i]) return fail(m, QD_ESTATE, "stream %d has no cache and input token", i);
        if (b->h_pos[i] + n_steps > b->S)
            return fail(m, QD_EKVFULL, "stream %d: position %d + %d steps exceeds smax %d", i, b->h_pos[i], n_steps,
                        b->S);
    }
    batch_enter(b);
    BatchCtl h = {};
    h.step = 0;
    h.n_steps = n_steps;
    h.force = force_dev;
    h.ids = ids_dev;
    h.done = 0;
    CU(cudaMemcpyAsync(b->ctl, &h, sizeof(h), cudaMemcpyHostToDevice, b->ls));
    for (int i = 0; i < n_steps; ++i) {
        qd_status st = run_batch_step(b);
        if (st) return st;
        b->launches += b->kernels_per_step;
    }
    for (int i = 0; i < b->B; ++i) b->h_pos[i] += n_steps;
    batch_leave(b);
    return QD_OK;
}

qd_status qd_batch_prefill(qd_batch_handle b, const int *streams, int ns, const float *embeds_dev, int n,
                           int32_t *first_ids_dev) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    const qd_config &c = m->cfg;
    if (ns < 1 || ns > b->B || !streams) return fail(m, QD_EINVAL, "ns %d out of range", ns);
    if (n < 1 || n >= b->S) return fail(m, QD_EINVAL, "n %d must be in [1, smax)", n);
    std::vector<char> seen(b->B, 0);
    for (int i = 0; i < ns; ++i) {
        if (streams[i] < 0 || streams[i] >= b->B || seen[streams[i]])
            return fail(m, QD_EINVAL, "stream list: index %d invalid or repeated", streams[i]);
        seen[streams[i]] = 1;
    }
    if (!is_device_ptr(embeds_dev) || !is_device_ptr(first_ids_dev))
        return fail(m, QD_EINVAL, "embeds_dev and first_ids_dev must be device pointers");
    if ((size_t)ns * n * std::max(m->q_dim(), c.ffn) > ((size_t)1 << 31))
        return fail(m, QD_EUNSUPPORTED, "prefill too large");
    batch_enter(b);
    qd_status st = ensure_prefill_scratch(b, ns, n);
    if (st) return st;
    // pageable source: staged by the runtime before the call returns
    CU(cudaMemcpyAsync(b->pf_streams, streams, (size_t)ns * 4, cudaMemcpyHostToDevice, b->ls));
    CU(cudaMemcpyAsync(b->pf_x, embeds_dev, (size_t)ns * n * c.hidden * 4, cudaMemcpyDeviceToDevice, b->ls));
    for (int i = 0; i < ns; ++i)
        CU(cudaMemsetAsync(b->emitted + (size_t)streams[i] * b->words, 0, (size_t)b->words * 4, b->ls));
    st = enqueue_prefill(b, ns, n, first_ids_dev);
    if (st) return st;
    for (int i = 0; i < ns; ++i) {
        b->h_pos[streams[i]] = n;
        b->h_ready[streams[i]] = 1;
    }
    batch_leave(b);
    return QD_OK;
}

// Synchronise and report device-side errors of the batch.
qd_status qd_batch_sync(qd_batch_handle b) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    int status = 0;
    CU(cudaMemcpyAsync(&status, b->status, 4, cudaMemcpyDeviceToHost, b->ls));
    CU(cudaStreamSynchronize(b->ls));
    if (status) return fail(m, QD_EDEVICE, "device error bits 0x%x", status);
    return QD_OK;
}

qd_status qd_batch_get_logits(qd_batch_handle b, float *dst_dev) {
    if (!b) return QD_EINVAL;
    qd_model *m = b->m;
    if (!is_device_ptr(dst_dev)) return fail(m, QD_EINVAL, "dst_dev is not a device pointer");
    CU(cudaMemcpyAsync(dst_dev, b->logits, (size_t)b->B * m->cfg.vocab * 4, cudaMemcpyDeviceToDevice, b->ls));
    CU(cudaStreamSynchronize(b->ls));
    return QD_OK;
}

qd_status qd_batch_copy_kv(qd_batch_handle b, int stream, void *dst_dev, size_t *bytes) {
    if (!b || !bytes) return QD_EINVAL;
    qd_model *m = b->m;
    if (stream < 0 || stream >= b->B) return fail(m, QD_EINVAL, "stream %d out of range", stream);
    const size_t n = b->stream_elems * 2;
    if (!dst_dev) {
        *bytes = n;
        return QD_OK;
    }
    if (*bytes < n || !is_device_ptr(dst_dev)) return fail(m, QD_EINVAL, "destination too small or not on the device");
    CU(cudaMemcpyAsync(dst_dev, static_cast<uint8_t *>(b->kv) + (size_t)stream * n, n, cudaMemcpyDeviceToDevice,
                       b->ls));
    CU(cudaStreamSynchronize(b->ls));
    *bytes = n;
    return QD_OK;
}

qd_status qd_batch_time_kernel(qd_batch_handle b, int which, int reps, float *avg_ms) {
    if (!b || !avg_ms || reps < 1) return QD_EINVAL;
    qd_model *m = b->m;
    for (int i = 0; i < b->B; ++i) {
        if (!b->h_ready[i]) return fail(m, QD_ESTATE, "stream %d has no cache and input token", i);
        if (b->h_pos[i] >= b->S) return fail(m, QD_EKVFULL, "stream %d is full", i);
    }
    // the launches are captured into a graph so that host work does not pace them
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ex = nullptr;
    CU(cudaStreamBeginCapture(b->ls, cudaStreamCaptureModeThreadLocal));
    qd_status st = QD_OK;
    for (int i = 0; i < reps && !st; ++i) st = enqueue_batch_kernel(b, which, b->ls);
    cudaError_t ce = cudaStreamEndCapture(b->ls, &g);
    if (st) {
        if (g) cudaGraphDestroy(g);
        return st;
    }
    CU(ce);
    cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    CU(ie);
    cudaEvent_t e0, e1;
    CU(cudaEventCreate(&e0));
    CU(cudaEventCreate(&e1));
    CU(cudaGraphLaunch(ex, b->ls));   // warm-up
    CU(cudaEventRecord(e0, b->ls));
    CU(cudaGraphLaunch(ex, b->ls));
    CU(cudaEventRecord(e1, b->ls));
    CU(cudaEventSynchronize(e1));
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaGraphExecDestroy(ex);
    *avg_ms = ms / reps;
    b->launches += 2LL * reps;
    return QD_OK;
}

qd_status qd_batch_get_pos(qd_batch_handle b, int stream, int *pos) {
    if (!b || !pos || stream < 0 || stream >= b->B) return QD_EINVAL;
    *pos = b->h_pos[stream];
    return QD_OK;
}

qd_status qd_batch_get_launch_count(qd_batch_handle b, long long *kernels, int *kernels_per_step) {
    if (!b) return QD_EINVAL;
    if (kernels) *kernels = b->launches;
    if (kernels_per_step) *kernels_per_step = b->kernels_per_step;
    return QD_OK;
}

}  // extern "C"

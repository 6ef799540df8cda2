// Decode engine behind the C-ABI in include/qd.h: weight repacking, the KV bucket
// ladder, per-bucket CUDA graphs of the step, and the entry points.
//
// Sources (page title, section):
//  - "Audio8-ASR: dynamic KV-cache buckets", section "Implemented dynamic window
//    mechanism": start from the smallest usable Smax; when the write position
//    reaches Smax copy the valid K/V region into a larger buffer and switch to
//    that bucket's compiled graph (one graph per bucket); continue from the same
//    token and RoPE position.  The cache is owned outside the compute graphs.
//  - "NEON Library", sections "Contracts" and "Validation": validation happens
//    before any work and a failed call leaves the plan reusable; outputs belong
//    to the plan until the next run; invalid-input recovery is tested.
//  - "qwen3-tts-hip OPTIMIZATION_LOG": graph replay of the decode-step stack.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "qd_model.h"

using namespace qd;

// ------------------------------------------------------------------ errors

qd_status fail(qd_model *m, qd_status st, const char *fmt, ...) {
    if (m) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof(buf), fmt, ap);
        va_end(ap);
        int rt = 0, drv = 0;
        cudaRuntimeGetVersion(&rt);
        cudaDriverGetVersion(&drv);
        char ver[96];
        snprintf(ver, sizeof(ver), " [qd 0.1, CUDA runtime %d, driver %d]", rt, drv);
        m->err = std::string(buf) + ver;
    }
    return st;
}

// ------------------------------------------------------------------ helpers

bool is_device_ptr(const void *p) {
    if (!p) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static qd_status validate_config(qd_model *m, const qd_config *c) {
    if (!c) return fail(m, QD_EINVAL, "config is NULL");
    if (c->hidden <= 0 || c->n_layers <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->ffn <= 0 || c->vocab <= 0 || c->embed_rows < 0)
        return fail(m, QD_EINVAL, "non-positive dimension in config");
    if (c->dtype != QD_F32 && c->dtype != QD_BF16) return fail(m, QD_EINVAL, "dtype must be QD_F32 or QD_BF16");
    if (c->n_q_heads % c->n_kv_heads) return fail(m, QD_EINVAL, "n_q_heads must be a multiple of n_kv_heads");
    if (c->n_q_heads / c->n_kv_heads > 8) return fail(m, QD_EUNSUPPORTED, "more than 8 q heads per kv head");
    if (c->head_dim != 64 && c->head_dim != 128) return fail(m, QD_EUNSUPPORTED, "head_dim must be 64 or 128");
    if (c->n_heads_out < 1 || c->n_heads_out > QD_MAX_HEADS) return fail(m, QD_EINVAL, "n_heads_out out of range");
    if (c->eos_mask_id >= c->vocab) return fail(m, QD_EINVAL, "eos_mask_id >= vocab");
    if (c->n_buckets < 1 || c->n_buckets > QD_MAX_BUCKETS) return fail(m, QD_EINVAL, "n_buckets out of range");
    for (int i = 0; i < c->n_buckets; ++i) {
        if (c->buckets[i] <= 0 || c->buckets[i] % 32)
            return fail(m, QD_EINVAL, "bucket %d (%d) must be a positive multiple of 32", i, c->buckets[i]);
        if (i && c->buckets[i] <= c->buckets[i - 1]) return fail(m, QD_EINVAL, "buckets must ascend");
    }
    if (!(c->rms_eps >= 0.0) || !(c->rope_theta > 0.0) || !(c->rep_penalty > 0.0))
        return fail(m, QD_EINVAL, "rms_eps, rope_theta, rep_penalty out of range");
    {
        const int *sec = c->mrope_section;
        const bool plain = sec[0] == 0 && sec[1] == 0 && sec[2] == 0;
        if (!plain && !(sec[1] > 0 && sec[1] == sec[2] && sec[0] >= sec[1] && sec[0] + sec[1] + sec[2] == c->head_dim / 2))
            return fail(m, QD_EINVAL, "mrope_section (%d, %d, %d): need t >= h == w > 0 and t + h + w == head_dim/2",
                        sec[0], sec[1], sec[2]);
    }
    const bool bf = c->dtype == QD_BF16;
    if (c->weight_q8 != 0 && c->weight_q8 != 1) return fail(m, QD_EINVAL, "weight_q8 must be 0 or 1");
    if (c->weight_q8 && !bf) return fail(m, QD_EUNSUPPORTED, "8-bit weights need dtype QD_BF16");
    const int max_pos = c->buckets[c->n_buckets - 1];
    if (c->hidden > 16 * 1024)
        return fail(m, QD_EUNSUPPORTED, "hidden %d too large", c->hidden);
    if (attention_smem_bytes(bf, c->head_dim, c->n_q_heads / c->n_kv_heads, attn_chunk(max_pos)) > 160 * 1024)
        return fail(m, QD_EUNSUPPORTED, "largest bucket %d too long for the attention tile", max_pos);
    int ns, rs;
    const int Ks[3] = {c->hidden, c->n_q_heads * c->head_dim, c->ffn};
    for (int K : Ks)
        if (K % 256 || K > 8192 || !gemv_split(K, bf, &ns, &rs))
            return fail(m, QD_EUNSUPPORTED, "dimension %d must be a multiple of 256 and <= 8192", K);
    return QD_OK;
}

void enter(qd_model *m) {
    cudaEventRecord(m->ev_in, m->user);
    cudaStreamWaitEvent(m->ls, m->ev_in, 0);
}
void leave(qd_model *m) {
    cudaEventRecord(m->ev_out, m->ls);
    cudaStreamWaitEvent(m->user, m->ev_out, 0);
}

// Step parameters: in_mode, token_in, add_emitted, head_idx (contiguous in DevState).
static qd_status set_params(qd_model *m, int mode, int token, int add_emitted, int head_idx) {
    int p[4] = {mode, token, add_emitted, head_idx};
    // pageable source: staged by the runtime before the call returns
    CU(cudaMemcpyAsync(&m->st->in_mode, p, sizeof(p), cudaMemcpyHostToDevice, m->ls));
    return QD_OK;
}

static qd_status ensure_bucket(qd_model *m, int b) {
    if (m->kv[b]) return QD_OK;
    void *p = nullptr;
    CU(cudaMalloc(&p, m->kv_bytes(b)));
    m->kv[b] = p;
    return QD_OK;
}

static qd_status migrate(qd_model *m, int to) {
    qd_status st = ensure_bucket(m, to);
    if (st) return st;
    const int from = m->cur_bucket;
    const size_t row_bytes = (size_t)m->cfg.head_dim * m->esize;
    const int nseg = m->cfg.n_layers * 2 * m->cfg.n_kv_heads;
    CU(launch_kv_migrate(m->kv[from], m->cfg.buckets[from], m->kv[to], m->cfg.buckets[to], nseg, row_bytes, m->h_pos,
                         m->ls));
    if (m->h_pos > 0) m->launches += 1;
    m->cur_bucket = to;
    return QD_OK;
}

// Kernel arguments of the step's launches (shared by the step and by qd_time_kernel).
static GemvArgs qkv_args(qd_model *m, int l, bool input) {
    const qd_config &c = m->cfg;
    GemvArgs g = {};
    g.rows = m->q_dim() + 2 * m->kv_dim();
    g.K = c.hidden;
    g.rs = m->rs_h;
    g.unit = 1;
    g.nst = m->nst_qkv;
    g.rps = m->rps_h;
    g.rows_max = m->rmax_qkv;
    g.evict_last = m->evict_last_layers;
    g.W = m->layers[l].w_qkv;
    g.in = m->x;
    g.gamma = m->layers[l].attn_norm;
    g.eps = (float)c.rms_eps;
    g.out = m->qkv;
    g.st = m->st;
    if (input) {
        g.input_mode = 1;
        g.table = m->embed;
        g.table_rows = c.embed_rows;
        g.table_bf16 = m->bf16;
        g.vocab = c.vocab;
        g.S = m->S();
        g.embed_in = m->embed_in;
        g.stage_tokens = m->stage_tokens;
        g.stage_embeds = m->stage_embeds;
        g.emitted_w = m->emitted;
        g.x_out = m->x;
    }
    return g;
}

static AttnArgs attn_args(qd_model *m, int l) {
    const qd_config &c = m->cfg;
    const int S = m->S();
    const size_t layer_kv = (size_t)2 * m->kv_dim() * S * m->esize;
    AttnArgs a = {};
    a.qkv = m->qkv;
    a.q_gamma = c.qk_norm ? m->layers[l].q_norm : nullptr;
    a.k_gamma = c.qk_norm ? m->layers[l].k_norm : nullptr;
    a.eps = (float)c.rms_eps;
    a.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
    a.rope_cos = m->rope_cos;
    a.rope_sin = m->rope_sin;
    a.rope_rows = m->max_pos;
    a.mrope_h = c.mrope_section[1];
    a.rope_stage = m->stage_rpos;
    a.rope_stride = m->max_pos;
    uint8_t *kvl = reinterpret_cast<uint8_t *>(m->kv[m->cur_bucket]) + (size_t)l * layer_kv;
    a.kcache = kvl;
    a.vcache = kvl + layer_kv / 2;
    a.S = S;
    a.qh = c.n_q_heads;
    a.kvh = c.n_kv_heads;
    a.chunk_max = m->chunk_max;
    a.out = m->att;
    a.st = m->st;
    return a;
}

static GemvArgs o_args(qd_model *m, int l) {
    const qd_config &c = m->cfg;
    GemvArgs g = {};
    g.rows = c.hidden;
    g.K = m->q_dim();
    g.rs = m->rs_q;
    g.unit = 1;
    g.nst = m->nst_o;
    g.rps = m->rps_q;
    g.rows_max = m->rmax_o;
    g.evict_last = m->evict_last_layers;
    g.W = m->layers[l].w_o;
    g.in = m->att;
    g.out = m->x;
    g.st = m->st;
    return g;
}

static GemvArgs gu_args(qd_model *m, int l) {
    const qd_config &c = m->cfg;
    GemvArgs g = {};
    g.rows = 2 * c.ffn;
    g.K = c.hidden;
    g.rs = m->rs_h;
    g.unit = 2;
    g.nst = m->nst_gu;
    g.rps = m->rps_h;
    g.rows_max = m->rmax_gu;
    g.evict_last = m->evict_last_layers;
    g.W = m->layers[l].w_gu;
    g.in = m->x;
    g.gamma = m->layers[l].mlp_norm;
    g.eps = (float)c.rms_eps;
    g.out = m->act;
    g.st = m->st;
    return g;
}

static GemvArgs d_args(qd_model *m, int l) {
    const qd_config &c = m->cfg;
    GemvArgs g = {};
    g.rows = c.hidden;
    g.K = c.ffn;
    g.rs = m->rs_f;
    g.unit = 1;
    g.nst = m->nst_d;
    g.rps = m->rps_f;
    g.rows_max = m->rmax_d;
    g.evict_last = m->evict_last_layers;
    g.W = m->layers[l].w_d;
    g.in = m->act;
    g.out = m->x;
    g.st = m->st;
    return g;
}

static GemvArgs head_args(qd_model *m, float *logits_tap, int commit) {
    const qd_config &c = m->cfg;
    GemvArgs g = {};
    g.rows = c.vocab;
    g.K = c.hidden;
    g.rs = m->rs_h;
    g.unit = 1;
    g.nst = m->nst_head;
    g.rps = m->rps_h;
    g.rows_max = m->rmax_head;
    g.evict_last = 0;
    g.W_table = m->d_heads;
    g.in = m->x;
    g.gamma = m->final_norm;
    g.eps = (float)c.rms_eps;
    g.out = logits_tap;
    g.emitted = m->emitted;
    g.penalty = (float)c.rep_penalty;
    g.eos = c.eos_mask_id;
    g.y_out = commit ? m->y : nullptr;
    g.part_v = m->head_pv;
    g.part_i = m->head_pi;
    g.counter = m->head_cnt;
    g.ids = m->ids;
    g.ids_cap = kIdsCap;
    g.commit = commit;
    g.st = m->st;
    return g;
}

static StepArgs step_args(qd_model *m, bool with_head, bool taps) {
    const qd_config &c = m->cfg;
    StepArgs a = {};
    a.layers = m->d_layers;
    a.n_layers = c.n_layers;
    a.hidden = c.hidden;
    a.qh = c.n_q_heads;
    a.kvh = c.n_kv_heads;
    a.ffn = c.ffn;
    a.vocab = c.vocab;
    a.rs_h = m->rs_h;
    a.rs_q = m->rs_q;
    a.rs_f = m->rs_f;
    a.rps_h = m->rps_h;
    a.rps_q = m->rps_q;
    a.rps_f = m->rps_f;
    a.nst = m->nst_step;
    a.evict_last = m->evict_last_layers;
    a.eps = (float)c.rms_eps;
    a.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
    a.off_full = m->off_full;
    a.off_gsm = m->off_gsm;
    a.off_misc = m->off_misc;
    a.off_res = m->off_res;
    a.off_att = m->off_att;
    a.off_emw = m->off_emw;
    a.off_xin = m->off_xin;
    a.kv = m->kv[m->cur_bucket];
    a.S = m->S();
    a.chunk_max = m->chunk_max;
    a.rope_cos = m->rope_cos;
    a.rope_sin = m->rope_sin;
    a.rope_rows = m->max_pos;
    a.mrope_h = c.mrope_section[1];
    a.rope_stage = m->stage_rpos;
    a.rope_stride = m->max_pos;
    a.x = m->x;
    a.in = StepInputArgs{m->embed, c.embed_rows, c.vocab, m->S(), m->embed_in, m->stage_tokens, m->stage_embeds,
                         m->emitted};
    a.with_head = with_head ? 1 : 0;
    a.heads = m->d_heads;
    a.final_norm = m->final_norm;
    a.penalty = (float)c.rep_penalty;
    a.eos = c.eos_mask_id;
    a.y_out = m->y;
    a.part_v = m->head_pv;
    a.part_i = m->head_pi;
    a.head_counter = m->head_cnt;
    a.ids = m->ids;
    a.ids_cap = kIdsCap;
    a.tap_hidden = taps ? m->tap_hidden : nullptr;
    a.tap_logits = taps ? m->tap_logits : nullptr;
    a.barrier = m->barrier;
    a.st = m->st;
    if (m->tag_buf) {
        a.tg = m->tag_buf;
        a.tg_stride = m->tg_stride;
        a.tg_qkv = m->tg_qkv;
        a.tg_po = m->tg_po;
        a.tg_ml = m->tg_ml;
        a.tg_att = m->tg_att;
        a.tg_xc = m->tg_xc;
        a.tg_xe = m->tg_xe;
        a.tg_act = m->tg_act;
        a.seq = reinterpret_cast<unsigned *>(m->tag_buf + m->tg_words);
        a.emit_flag = a.seq + 1;
    }
    a.off_kc = m->off_kc;
    a.off_xres = m->off_xres;
    a.off_ldev = m->off_ldev;
    a.off_xs = m->off_xs;
    return a;
}

// Enqueue one step's kernels on stream s.
qd_status enqueue_step(qd_model *m, cudaStream_t s, bool with_head, bool taps) {
    const qd_config &c = m->cfg;
    const bool bf = m->bf16, pdl = m->use_pdl;
    const int h = c.hidden;
    if (m->persistent) {
        CU(launch_persistent(bf, c.head_dim, h, m->q_dim(), c.ffn, c.n_kv_heads, step_args(m, with_head, taps), m->num_sms,
                             m->smem_step, s, m->q8));
        return QD_OK;
    }
    for (int l = 0; l < c.n_layers; ++l) {
        CU(launch_gemv(GEMV_QKV, bf, qkv_args(m, l, l == 0), m->grid_qkv, m->smem_qkv, s, pdl));
        if (l == 0 && taps && m->tap_hidden)
            CU(cudaMemcpyAsync(m->tap_hidden, m->x, h * 4, cudaMemcpyDeviceToDevice, s));
        CU(launch_attention(bf, c.head_dim, attn_args(m, l), s, pdl));
        CU(launch_gemv(GEMV_RES, bf, o_args(m, l), m->grid_o, m->smem_o, s, pdl));
        CU(launch_gemv(GEMV_GU, bf, gu_args(m, l), m->grid_gu, m->smem_gu, s, pdl));
        GemvArgs d = d_args(m, l);
        d.advance_pos = (!with_head && l == c.n_layers - 1) ? 1 : 0;
        CU(launch_gemv(GEMV_RES, bf, d, m->grid_d, m->smem_d, s, pdl));
        if (taps && m->tap_hidden)
            CU(cudaMemcpyAsync(m->tap_hidden + (size_t)(l + 1) * h, m->x, h * 4, cudaMemcpyDeviceToDevice, s));
    }
    if (with_head)
        CU(launch_gemv(GEMV_HEAD, bf, head_args(m, taps ? m->tap_logits : nullptr, 1), m->grid_head, m->smem_head, s,
                       pdl));
    return QD_OK;
}

// One step on the library stream: graph replay of the current bucket, or eager.
static qd_status run_step(qd_model *m, bool with_head) {
    const bool taps = m->tap_hidden || m->tap_logits;
    if (taps || !m->use_graphs) {
        qd_status st = enqueue_step(m, m->ls, with_head, taps);
        if (st) return st;
    } else {
        cudaGraphExec_t &ex = m->graphs[with_head ? 1 : 0][m->cur_bucket];
        if (!ex) {
            cudaGraph_t g = nullptr;
            CU(cudaStreamBeginCapture(m->ls, cudaStreamCaptureModeThreadLocal));
            qd_status st = enqueue_step(m, m->ls, with_head, false);
            cudaError_t ce = cudaStreamEndCapture(m->ls, &g);
            if (st) {
                if (g) cudaGraphDestroy(g);
                return st;
            }
            CU(ce);
            cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
            cudaGraphDestroy(g);
            CU(ie);
        }
        CU(cudaGraphLaunch(ex, m->ls));
    }
    m->launches += m->kernels_per_step(with_head);
    return QD_OK;
}

// Grow along the ladder when the next write position has reached Smax.
qd_status grow_if_needed(qd_model *m) {
    if (m->h_pos < m->S()) return QD_OK;
    if (m->cur_bucket + 1 >= m->cfg.n_buckets)
        return fail(m, QD_EKVFULL, "position %d reaches the last bucket (%d)", m->h_pos, m->S());
    return migrate(m, m->cur_bucket + 1);
}

qd_status sync_and_check(qd_model *m, int *out_id) {
    CU(cudaMemcpyAsync(m->pin, &m->st->out_id, 3 * sizeof(int), cudaMemcpyDeviceToHost, m->ls));
    CU(cudaStreamSynchronize(m->ls));
    if (m->pin[2]) return fail(m, QD_EDEVICE, "device error bits 0x%x", m->pin[2]);
    if (out_id) *out_id = m->pin[0];
    return QD_OK;
}

// ------------------------------------------------------------------ weights

static qd_status load_weights(qd_model *m, const qd_weights *w) {
    const qd_config &c = m->cfg;
    const int h = c.hidden, qd_ = m->q_dim(), kd = m->kv_dim(), F = c.ffn, hd = c.head_dim;
    const size_t es = m->esize;
    if (!w || !w->layers) return fail(m, QD_EINVAL, "weights or weights->layers is NULL");
    if (!is_device_ptr(w->final_norm)) return fail(m, QD_EINVAL, "final_norm is not a device pointer");
    if (c.embed_rows && !is_device_ptr(w->embed)) return fail(m, QD_EINVAL, "embed is not a device pointer");
    for (int j = 0; j < c.n_heads_out; ++j)
        if (!is_device_ptr(w->lm_head[j])) return fail(m, QD_EINVAL, "lm_head[%d] is not a device pointer", j);
    for (int l = 0; l < c.n_layers; ++l) {
        const qd_layer_weights &L = w->layers[l];
        const void *req[] = {L.attn_norm, L.wq, L.wk, L.wv, L.wo, L.mlp_norm, L.wg, L.wu, L.wd};
        for (const void *p : req)
            if (!is_device_ptr(p)) return fail(m, QD_EINVAL, "layer %d: a weight is not a device pointer", l);
        if (c.qk_norm && (!is_device_ptr(L.q_norm) || !is_device_ptr(L.k_norm)))
            return fail(m, QD_EINVAL, "layer %d: q_norm/k_norm missing", l);
    }

    // arena layout
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    std::vector<size_t> o_qkv(c.n_layers), o_o(c.n_layers), o_gu(c.n_layers), o_d(c.n_layers), o_an(c.n_layers),
        o_mn(c.n_layers), o_qn(c.n_layers), o_kn(c.n_layers);
    // bytes of a row of K weights: es per weight, or an 8-bit row (codes + half scales)
    auto rowb = [&](int K) { return m->q8 ? (size_t)q8_row_bytes(K) : (size_t)K * es; };
    for (int l = 0; l < c.n_layers; ++l) {
        o_qkv[l] = take((size_t)(qd_ + 2 * kd) * rowb(h));
        o_o[l] = take((size_t)h * rowb(qd_));
        o_gu[l] = take((size_t)2 * F * rowb(h));
        o_d[l] = take((size_t)h * rowb(F));
    }
    size_t o_heads[QD_MAX_HEADS];
    for (int j = 0; j < c.n_heads_out; ++j) o_heads[j] = take((size_t)c.vocab * rowb(h));
    const size_t o_embed = c.embed_rows ? take((size_t)c.embed_rows * h * es) : 0;
    for (int l = 0; l < c.n_layers; ++l) {
        o_an[l] = take((size_t)h * 4);
        o_mn[l] = take((size_t)h * 4);
        o_qn[l] = take((size_t)hd * 4);
        o_kn[l] = take((size_t)hd * 4);
    }
    const size_t o_fn = take((size_t)h * 4);
    const size_t o_tab = take(sizeof(void *) * QD_MAX_HEADS);
    CU(cudaMalloc(&m->arena, off));
    uint8_t *A = reinterpret_cast<uint8_t *>(m->arena);
    cudaStream_t s = m->ls;

    m->layers.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const qd_layer_weights &W = w->layers[l];
        Layer &L = m->layers[l];
        L.w_qkv = A + o_qkv[l];
        L.w_o = A + o_o[l];
        L.w_gu = A + o_gu[l];
        L.w_d = A + o_d[l];
        L.attn_norm = reinterpret_cast<float *>(A + o_an[l]);
        L.mlp_norm = reinterpret_cast<float *>(A + o_mn[l]);
        L.q_norm = reinterpret_cast<float *>(A + o_qn[l]);
        L.k_norm = reinterpret_cast<float *>(A + o_kn[l]);
        uint8_t *q = reinterpret_cast<uint8_t *>(L.w_qkv);
        if (m->q8) {
            // the same fused layouts, quantised row by row: [wq; wk; wv], gate/up interleaved
            CU(launch_quantize_rows_q8(W.wq, m->bf16, qd_, h, q, 0, 1, s));
            CU(launch_quantize_rows_q8(W.wk, m->bf16, kd, h, q, qd_, 1, s));
            CU(launch_quantize_rows_q8(W.wv, m->bf16, kd, h, q, qd_ + kd, 1, s));
            CU(launch_quantize_rows_q8(W.wo, m->bf16, h, qd_, L.w_o, 0, 1, s));
            CU(launch_quantize_rows_q8(W.wg, m->bf16, F, h, L.w_gu, 0, 2, s));
            CU(launch_quantize_rows_q8(W.wu, m->bf16, F, h, L.w_gu, 1, 2, s));
            CU(launch_quantize_rows_q8(W.wd, m->bf16, h, F, L.w_d, 0, 1, s));
        } else {
            CU(cudaMemcpyAsync(q, W.wq, (size_t)qd_ * h * es, cudaMemcpyDeviceToDevice, s));
            CU(cudaMemcpyAsync(q + (size_t)qd_ * h * es, W.wk, (size_t)kd * h * es, cudaMemcpyDeviceToDevice, s));
            CU(cudaMemcpyAsync(q + (size_t)(qd_ + kd) * h * es, W.wv, (size_t)kd * h * es, cudaMemcpyDeviceToDevice,
                               s));
            CU(cudaMemcpyAsync(L.w_o, W.wo, (size_t)h * qd_ * es, cudaMemcpyDeviceToDevice, s));
            // gate/up rows interleaved: row 2i = wg[i], row 2i+1 = wu[i]
            const size_t rb = (size_t)h * es;
            CU(cudaMemcpy2DAsync(L.w_gu, 2 * rb, W.wg, rb, rb, F, cudaMemcpyDeviceToDevice, s));
            CU(cudaMemcpy2DAsync(reinterpret_cast<uint8_t *>(L.w_gu) + rb, 2 * rb, W.wu, rb, rb, F,
                                 cudaMemcpyDeviceToDevice, s));
            CU(cudaMemcpyAsync(L.w_d, W.wd, (size_t)h * F * es, cudaMemcpyDeviceToDevice, s));
        }
        CU(launch_to_f32(W.attn_norm, m->bf16, L.attn_norm, h, s));
        CU(launch_to_f32(W.mlp_norm, m->bf16, L.mlp_norm, h, s));
        if (c.qk_norm) {
            CU(launch_to_f32(W.q_norm, m->bf16, L.q_norm, hd, s));
            CU(launch_to_f32(W.k_norm, m->bf16, L.k_norm, hd, s));
        }
    }
    for (int j = 0; j < c.n_heads_out; ++j) {
        m->heads[j] = A + o_heads[j];
        if (m->q8)
            CU(launch_quantize_rows_q8(w->lm_head[j], m->bf16, c.vocab, h, m->heads[j], 0, 1, s));
        else
            CU(cudaMemcpyAsync(m->heads[j], w->lm_head[j], (size_t)c.vocab * h * es, cudaMemcpyDeviceToDevice, s));
    }
    if (c.embed_rows) {
        m->embed = A + o_embed;
        CU(cudaMemcpyAsync(m->embed, w->embed, (size_t)c.embed_rows * h * es, cudaMemcpyDeviceToDevice, s));
    }
    m->final_norm = reinterpret_cast<float *>(A + o_fn);
    CU(launch_to_f32(w->final_norm, m->bf16, m->final_norm, h, s));
    m->d_heads = reinterpret_cast<const void **>(A + o_tab);
    CU(cudaMemcpyAsync(m->d_heads, m->heads, sizeof(void *) * QD_MAX_HEADS, cudaMemcpyHostToDevice, s));
    CU(cudaStreamSynchronize(s));
    return QD_OK;
}

static qd_status alloc_scratch(qd_model *m) {
    const qd_config &c = m->cfg;
    const int h = c.hidden;
    m->max_pos = c.buckets[c.n_buckets - 1];
    m->chunk_max = attn_chunk(m->max_pos);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_x = take(h * 4), o_qkv = take((size_t)(m->q_dim() + 2 * m->kv_dim()) * 4),
                 o_act = take((size_t)c.ffn * 4),
                 o_att = take((size_t)m->q_dim() * 4), o_y = take(h * 4),
                 o_bar = take(128),
                 o_ein = take(h * 4), o_se = take((size_t)m->max_pos * h * 4), o_pv = take((size_t)kHeadCandidates * 4),
                 o_pi = take((size_t)kHeadCandidates * 4), o_hc = take(64 * 4), o_stok = take((size_t)m->max_pos * 4),
                 o_ids = take((size_t)kIdsCap * 4), o_em = take((size_t)((c.vocab + 31) / 32) * 4),
                 o_st = take(sizeof(DevState)), o_cos = take((size_t)m->max_pos * (c.head_dim / 2) * 4),
                 o_sin = take((size_t)m->max_pos * (c.head_dim / 2) * 4), o_rpos = take((size_t)3 * m->max_pos * 4);
    CU(cudaMalloc(&m->scratch, off));
    CU(cudaMemsetAsync(m->scratch, 0, off, m->ls));
    uint8_t *B = reinterpret_cast<uint8_t *>(m->scratch);
    m->x = reinterpret_cast<float *>(B + o_x);
    m->qkv = reinterpret_cast<float *>(B + o_qkv);
    m->act = reinterpret_cast<float *>(B + o_act);
    m->att = reinterpret_cast<float *>(B + o_att);
    m->barrier = reinterpret_cast<unsigned *>(B + o_bar);
    m->y = reinterpret_cast<float *>(B + o_y);
    m->embed_in = reinterpret_cast<float *>(B + o_ein);
    m->stage_embeds = reinterpret_cast<float *>(B + o_se);
    m->head_pv = reinterpret_cast<float *>(B + o_pv);
    m->head_pi = reinterpret_cast<int *>(B + o_pi);
    m->head_cnt = reinterpret_cast<int *>(B + o_hc);
    m->stage_tokens = reinterpret_cast<int *>(B + o_stok);
    m->ids = reinterpret_cast<int32_t *>(B + o_ids);
    m->emitted = reinterpret_cast<uint32_t *>(B + o_em);
    m->st = reinterpret_cast<DevState *>(B + o_st);
    m->rope_cos = reinterpret_cast<float *>(B + o_cos);
    m->rope_sin = reinterpret_cast<float *>(B + o_sin);
    m->stage_rpos = reinterpret_cast<int *>(B + o_rpos);
    CU(launch_rope_table(m->rope_cos, m->rope_sin, m->max_pos, c.head_dim, c.rope_theta, m->ls));
    CU(cudaMallocHost(&m->pin, 16 * sizeof(int)));
    return QD_OK;
}

static bool plan_launches(qd_model *m) {
    const qd_config &c = m->cfg;
    const bool bf = m->bf16;
    int ns;
    gemv_split(c.hidden, bf, &ns, &m->rs_h);
    gemv_split(m->q_dim(), bf, &ns, &m->rs_q);
    gemv_split(c.ffn, bf, &ns, &m->rs_f);
    m->rps_h = kSlotBytes / (int)(c.hidden * m->esize);
    m->rps_q = kSlotBytes / (int)(m->q_dim() * m->esize);
    m->rps_f = kSlotBytes / (int)(c.ffn * m->esize);
    const int sms = m->num_sms;
    auto plan = [&](int rows, int unit, int K, int rps, int rs, int max_nst, int *grid, int *nst, int *rmax,
                    size_t *smem, int min_nst = 1) {
        const int units = rows / unit;
        *grid = std::min(sms, units);
        *rmax = (units + *grid - 1) / *grid * unit;
        const int need = (*rmax + rps - 1) / rps;
        *nst = std::max(min_nst, std::min(need, max_nst));
        *smem = gemv_smem_bytes(*nst, *rmax, rs, K);
    };
    // Step kernels keep their ring at 4 stages (96 KB) so that the next kernel of the
    // step fits beside them on the SM under programmatic dependent launch; the head is
    // the last kernel of the step and takes a deeper ring.
    const int ring = kRingBytes / kSlotBytes;
    plan(m->q_dim() + 2 * m->kv_dim(), 1, c.hidden, m->rps_h, m->rs_h, ring, &m->grid_qkv, &m->nst_qkv,
         &m->rmax_qkv, &m->smem_qkv);
    plan(c.hidden, 1, m->q_dim(), m->rps_q, m->rs_q, ring, &m->grid_o, &m->nst_o, &m->rmax_o, &m->smem_o);
    plan(2 * c.ffn, 2, c.hidden, m->rps_h, m->rs_h, ring, &m->grid_gu, &m->nst_gu, &m->rmax_gu, &m->smem_gu);
    plan(c.hidden, 1, c.ffn, m->rps_f, m->rs_f, ring, &m->grid_d, &m->nst_d, &m->rmax_d, &m->smem_d);
    // the head's ring also holds, once its rows are consumed, the sampling merge of
    // every CTA's candidates (up to kMaxTopK each): at least three stages
    plan(c.vocab, 1, c.hidden, m->rps_h, m->rs_h, 2 * ring, &m->grid_head, &m->nst_head, &m->rmax_head,
         &m->smem_head, 3);
    // Layer weights that fit in 60% of L2 stay resident across steps (evict_last);
    // the output head always streams (evict_first).
    size_t layer_bytes = 0;
    auto mat = [&](int rows, int K) { return (size_t)rows * (m->q8 ? q8_row_bytes(K) : (size_t)K * m->esize); };
    for (int l = 0; l < c.n_layers; ++l)
        layer_bytes += mat(m->q_dim() + 2 * m->kv_dim() + 2 * c.ffn, c.hidden) + mat(c.hidden, m->q_dim()) +
                       mat(c.hidden, c.ffn);
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, m->device);
    m->evict_last_layers = layer_bytes * 10 <= (size_t)l2 * 6 ? 1 : 0;
    // residual kernels keep one row per consumer thread
    return m->rmax_o <= kConsumerWarps * 32 && m->rmax_d <= kConsumerWarps * 32;
}

// Set up the persistent decode step when the shape has an instantiation: the device
// layer table and the shared-memory layout (ring of up to 6 slots next to the
// phase scratch), and check that one CTA fits on every SM.
static qd_status setup_persistent(qd_model *m) {
    const qd_config &c = m->cfg;
    m->persistent = false;
    // 8-bit rows exist only in the persistent step: no per-phase fallback
    if (std::getenv("QD_PER_PHASE")) return m->q8 ? QD_EUNSUPPORTED : QD_OK;   // debug and profiling only
    // the 8-bit head takes whole rows per warp
    if (m->q8) m->rs_h = 1;
    if (!persistent_supported(m->bf16, c.head_dim, c.hidden, m->q_dim(), c.ffn, c.n_kv_heads, m->q8)) return QD_OK;
    if (m->num_sms < kStepMinSms) return QD_OK;
    const int G = c.n_q_heads / c.n_kv_heads;
    if (c.n_kv_heads * kAttnMaxSplits > m->num_sms) return QD_OK;
    if (G > kStepGroupMax) return QD_OK;
    if (m->chunk_max * c.head_dim * (int)m->esize > kSlotBytes) return QD_OK;
    // rows of any phase held by one CTA, times the warps per row
    auto rmax = [&](int rows, int unit) { return (rows / unit + m->num_sms - 1) / m->num_sms * unit; };
    if (rmax(m->q_dim() + 2 * m->kv_dim(), 1) > kStepRowsMax || rmax(c.hidden, 1) > kStepRowsMax ||
        rmax(2 * c.ffn, 2) > kStepRowsMax)
        return QD_OK;
    // a ring stage holds at most 32 rows of every phase (one transposing butterfly)
    if (kSlotBytes / (c.hidden * (int)m->esize) > 32 || kSlotBytes / (m->q_dim() * (int)m->esize) > 32 ||
        kSlotBytes / (c.ffn * (int)m->esize) > 32)
        return QD_OK;
    const int res_words = std::max({rmax(m->q_dim() + 2 * m->kv_dim(), 1) * m->rs_h, rmax(c.hidden, 1) * m->rs_q,
                                    rmax(2 * c.ffn, 2) * m->rs_h, rmax(c.hidden, 1) * m->rs_f,
                                    rmax(c.vocab, 1) * m->rs_h});
    const int head_rows = rmax(c.vocab, 1);
    size_t off = 0;
    auto take = [&](size_t bytes, size_t al) {
        off = align_up(off, al);
        const size_t o = off;
        off += bytes;
        return (int)o;
    };
    size_t tail = 0;
    {
        // everything but the ring
        tail += 2 * 8 * 8 + 16;                                        // barriers (<= 8 slots)
        tail += (size_t)c.hidden * 4 + 16;                             // gamma
        tail += 64 * 4;                                                // misc
        tail += (size_t)res_words * 4 + 16;                            // row partial sums
        tail += persistent_att_bytes(G, c.head_dim, m->chunk_max) + 16;
        tail += ((size_t)head_rows / 32 + 2) * 4 + 16;                 // emitted words of the head rows
        tail += (size_t)c.hidden * 4 + 16;                             // the head's input vector
        tail += ((size_t)2 * kConsumerWarps * kStepRowsMax + 2 * kConsumerWarps) * 4 + 16;   // row partials
        tail += (size_t)kStepRowsMax * 4 + 16;                         // residual rows
        tail += sizeof(LayerDev) * (size_t)c.n_layers + 16;            // layer table
        tail += (size_t)c.ffn * 4 + 16;                                // the warps' input slices
    }
    const size_t max_smem = kStepMaxSmem;
    const int nst = kStepRingStages;
    if (tail + (size_t)nst * kSlotBytes > max_smem) return QD_OK;
    off = 0;
    take((size_t)nst * kSlotBytes, 1024);
    m->off_full = take((size_t)2 * nst * 8, 16);
    m->off_gsm = take((size_t)c.hidden * 4, 16);
    m->off_misc = take(64 * 4, 16);
    m->off_res = take((size_t)res_words * 4, 16);
    m->off_att = take(persistent_att_bytes(G, c.head_dim, m->chunk_max), 16);
    m->off_emw = take(((size_t)head_rows / 32 + 2) * 4, 16);
    m->off_xin = take((size_t)c.hidden * 4, 16);
    m->off_kc = take(((size_t)2 * kConsumerWarps * kStepRowsMax + 2 * kConsumerWarps) * 4, 16);
    m->off_xres = take((size_t)kStepRowsMax * 4, 16);
    m->off_ldev = take(sizeof(LayerDev) * (size_t)c.n_layers, 16);
    m->off_xs = take((size_t)c.ffn * 4, 16);
    m->smem_step = align_up(off, 16);
    m->nst_step = nst;
    if (m->smem_step > max_smem) return QD_OK;
    CU(persistent_init(m->bf16, c.head_dim, c.hidden, m->q_dim(), c.ffn, c.n_kv_heads, m->q8));
    // layer table
    std::vector<LayerDev> host(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const Layer &L = m->layers[l];
        host[l] = LayerDev{L.w_qkv, L.w_o, L.w_gu, L.w_d, L.attn_norm, L.mlp_norm, c.qk_norm ? L.q_norm : nullptr,
                           c.qk_norm ? L.k_norm : nullptr};
    }
    CU(cudaMalloc(&m->d_layers, sizeof(LayerDev) * c.n_layers));
    CU(cudaMemcpy(m->d_layers, host.data(), sizeof(LayerDev) * c.n_layers, cudaMemcpyHostToDevice));
    // tagged words of every layer (all zero: no launch has sequence number 0), then the
    // sequence number (from 1) and the emitted-set flag; pieces start on 256-byte lines
    auto words32 = [](size_t n) { return (int)((n + 31) / 32 * 32); };
    int o = 0;
    m->tg_qkv = o; o += words32((size_t)m->q_dim() + 2 * m->kv_dim());
    m->tg_po = o;  o += words32((size_t)c.n_kv_heads * kAttnMaxSplits * G * c.head_dim);
    m->tg_ml = o;  o += words32((size_t)c.n_kv_heads * kAttnMaxSplits * G * 2);
    m->tg_att = o; o += words32((size_t)m->q_dim());
    m->tg_xc = o;  o += words32((size_t)c.hidden);
    m->tg_xe = o;  o += words32((size_t)c.hidden);
    m->tg_act = o; o += words32((size_t)c.ffn);
    m->tg_stride = o;
    m->tg_words = (size_t)o * c.n_layers;
    const size_t bytes = (m->tg_words + 32) * 8;
    CU(cudaMalloc(&m->tag_buf, bytes));
    CU(cudaMemset(m->tag_buf, 0, bytes));
    const unsigned one = 1;
    CU(cudaMemcpy(m->tag_buf + m->tg_words, &one, sizeof(one), cudaMemcpyHostToDevice));
    m->persistent = true;
    return QD_OK;
}

// ------------------------------------------------------------------ C-ABI

extern "C" {

const char *qd_status_string(int status) {
    switch (status) {
        case QD_OK: return "QD_OK";
        case QD_EINVAL: return "QD_EINVAL: invalid argument";
        case QD_ESTATE: return "QD_ESTATE: invalid in the current state";
        case QD_EKVFULL: return "QD_EKVFULL: beyond the last KV bucket";
        case QD_ENOMEM: return "QD_ENOMEM: device allocation failed";
        case QD_ECUDA: return "QD_ECUDA: CUDA runtime error";
        case QD_EUNSUPPORTED: return "QD_EUNSUPPORTED: shape not supported";
        case QD_EDEVICE: return "QD_EDEVICE: kernel reported an error";
    }
    return "unknown status";
}

const char *qd_last_error(qd_handle h) { return h ? h->err.c_str() : "null handle"; }

static void destroy_model(qd_model *m) {
    if (!m) return;
    while (!m->frames.empty()) frame_detach(m->frames.back());
    if (m->ls) cudaStreamSynchronize(m->ls);
    if (m->pf_batch) qd_batch_destroy(m->pf_batch);
    for (cudaEvent_t e : m->pf_ev)
        if (e) cudaEventDestroy(e);
    for (int v = 0; v < 2; ++v)
        for (auto &g : m->graphs[v])
            if (g) cudaGraphExecDestroy(g);
    for (void *p : m->kv)
        if (p) cudaFree(p);
    if (m->arena) cudaFree(m->arena);
    if (m->d_layers) cudaFree(m->d_layers);
    if (m->tag_buf) cudaFree(m->tag_buf);
    if (m->scratch) cudaFree(m->scratch);
    if (m->pin) cudaFreeHost(m->pin);
    if (m->ev_in) cudaEventDestroy(m->ev_in);
    if (m->ev_out) cudaEventDestroy(m->ev_out);
    if (m->ev_t0) cudaEventDestroy(m->ev_t0);
    if (m->ev_t1) cudaEventDestroy(m->ev_t1);
    if (m->ls) cudaStreamDestroy(m->ls);
    delete m;
}

qd_status qd_create(const qd_weights *weights, const qd_config *cfg, void *cuda_stream, qd_handle *out) {
    if (!out) return QD_EINVAL;
    *out = nullptr;
    qd_model tmp;
    qd_status vs = validate_config(&tmp, cfg);
    if (vs) return vs;
    qd_model *m = new qd_model();
    m->cfg = *cfg;
    m->bf16 = cfg->dtype == QD_BF16;
    m->q8 = cfg->weight_q8 != 0;
    m->esize = m->bf16 ? 2 : 4;
    m->user = reinterpret_cast<cudaStream_t>(cuda_stream);
    // debug and profiling only: launch every kernel without programmatic dependent
    // launch (results are identical; only the overlap between kernels changes)
    m->use_pdl = std::getenv("QD_NO_PDL") == nullptr;
    auto bail = [&](qd_status st) {
        destroy_model(m);
        return st;
    };
    if (cudaGetDevice(&m->device) != cudaSuccess) return bail(QD_ECUDA);
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, m->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, m->device);
    if (major != 10 || minor != 3) return bail(QD_EUNSUPPORTED);
    if (cudaStreamCreateWithFlags(&m->ls, cudaStreamNonBlocking) != cudaSuccess) return bail(QD_ECUDA);
    if (cudaEventCreateWithFlags(&m->ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->ev_out, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreate(&m->ev_t0) != cudaSuccess || cudaEventCreate(&m->ev_t1) != cudaSuccess)
        return bail(QD_ECUDA);
    if (kernels_init() != cudaSuccess) return bail(QD_ECUDA);
    enter(m);
    qd_status st = load_weights(m, weights);
    if (st) return bail(st);
    st = alloc_scratch(m);
    if (st) return bail(st);
    if (!plan_launches(m)) {
        destroy_model(m);
        return QD_EUNSUPPORTED;
    }
    st = setup_persistent(m);
    if (st) return bail(st);
    if (m->q8 && !m->persistent) return bail(QD_EUNSUPPORTED);
    m->kv.assign(cfg->n_buckets, nullptr);
    m->graphs[0].assign(cfg->n_buckets, nullptr);
    m->graphs[1].assign(cfg->n_buckets, nullptr);
    st = ensure_bucket(m, 0);
    if (st) return bail(st);
    if (cudaStreamSynchronize(m->ls) != cudaSuccess) return bail(QD_ECUDA);
    leave(m);
    *out = m;
    return QD_OK;
}

qd_status qd_destroy(qd_handle h) {
    destroy_model(h);
    return QD_OK;
}

qd_status qd_reset(qd_handle h) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    enter(m);
    CU(cudaMemsetAsync(m->st, 0, QD_DEVSTATE_RESET_BYTES, m->ls));
    CU(cudaMemsetAsync(m->emitted, 0, (size_t)((m->cfg.vocab + 31) / 32) * 4, m->ls));
    m->h_pos = 0;
    m->h_ngen = 0;
    m->h_rope_delta = 0;
    m->cur_bucket = 0;
    m->have_hidden = false;
    leave(m);
    return QD_OK;
}

}  // extern "C"

// The rotary-position fields of the device state: the decode steps' delta and whether
// the steps read the staged prompt positions.
static qd_status set_rope(qd_model *m, int delta, int staged) {
    const int v[2] = {delta, staged};
    // pageable source: staged by the runtime before the call returns
    CU(cudaMemcpyAsync(&m->st->rope_delta, v, sizeof(v), cudaMemcpyHostToDevice, m->ls));
    return QD_OK;
}

static qd_status prefill_impl(qd_handle h, const int32_t *tokens, const void *embeds, int n, int head_idx,
                              const int32_t *positions, int32_t *first_id) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    const qd_config &c = m->cfg;
    if (n < 1) return fail(m, QD_EINVAL, "prefill needs n >= 1 (got %d)", n);
    if ((tokens == nullptr) == (embeds == nullptr)) return fail(m, QD_EINVAL, "give exactly one of tokens/embeds");
    if (!first_id) return fail(m, QD_EINVAL, "first_id is NULL");
    if (head_idx < 0 || head_idx >= c.n_heads_out) return fail(m, QD_EINVAL, "head_idx %d out of range", head_idx);
    if (m->h_pos != 0) return fail(m, QD_ESTATE, "prefill at position %d: reset first", m->h_pos);
    if (n > m->max_pos) return fail(m, QD_EKVFULL, "prefill of %d exceeds the last bucket (%d)", n, m->max_pos);
    if (tokens) {
        if (!c.embed_rows) return fail(m, QD_EINVAL, "model has no embedding table");
        for (int i = 0; i < n; ++i)
            if (tokens[i] < 0 || tokens[i] >= c.embed_rows)
                return fail(m, QD_EINVAL, "token %d at %d outside the embedding table", tokens[i], i);
    } else if (!is_device_ptr(embeds)) {
        return fail(m, QD_EINVAL, "embeds is not a device pointer");
    }
    // the decode steps after the prompt rotate at its largest position + 1
    int top = n - 1;
    if (positions)
        for (int i = 0; i < 3 * n; ++i) {
            if (positions[i] < 0 || positions[i] >= m->max_pos)
                return fail(m, QD_EINVAL, "rotary position %d (stream %d, prompt position %d) outside [0, %d)",
                            positions[i], i / n, i % n, m->max_pos);
            top = positions[i] > top ? positions[i] : top;
        }
    const int delta = top + 1 - n;
    int b = 0;
    while (c.buckets[b] < n) ++b;
    enter(m);
    qd_status st = ensure_bucket(m, b);
    if (st) return st;
    m->cur_bucket = b;
    if (positions)
        for (int s = 0; s < 3; ++s)
            CU(cudaMemcpyAsync(m->stage_rpos + (size_t)s * m->max_pos, positions + (size_t)s * n, (size_t)n * 4,
                               cudaMemcpyHostToDevice, m->ls));
    if (!m->tap_hidden && !m->tap_logits) {
        // all positions at once through the batched prefill kernels, where they apply
        if (tokens) CU(cudaMemcpyAsync(m->stage_tokens, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, m->ls));
        st = model_prefill_batched(m, static_cast<const float *>(embeds), tokens ? m->stage_tokens : nullptr, n, b,
                                   positions ? m->stage_rpos : nullptr, m->max_pos);
        if (st == QD_OK) {
            // the head on the last position: the model's own head kernel, as in every step
            st = set_params(m, IN_EMBED, -1, 0, head_idx);
            if (st) return st;
            CU(launch_gemv(GEMV_HEAD, m->bf16, head_args(m, nullptr, 1), m->grid_head, m->smem_head, m->ls, false));
            m->launches += 1;
            st = set_rope(m, delta, 0);
            if (st) return st;
            m->h_pos = n;
            m->h_ngen++;
            m->h_rope_delta = delta;
            m->have_hidden = true;
            st = sync_and_check(m, first_id);
            leave(m);
            return st;
        }
        if (st != QD_EUNSUPPORTED) return st;
    }
    if (tokens) CU(cudaMemcpyAsync(m->stage_tokens, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, m->ls));
    else CU(cudaMemcpyAsync(m->stage_embeds, embeds, (size_t)n * c.hidden * 4, cudaMemcpyDeviceToDevice, m->ls));
    st = set_params(m, tokens ? IN_STAGED_TOKENS : IN_STAGED_EMBEDS, -1, 0, head_idx);
    if (st) return st;
    st = set_rope(m, 0, positions ? 1 : 0);
    if (st) return st;
    for (int i = 0; i < n; ++i) {
        st = run_step(m, i == n - 1);
        if (st) return st;
        m->h_pos++;
    }
    st = set_rope(m, delta, 0);
    if (st) return st;
    m->h_ngen++;
    m->h_rope_delta = delta;
    m->have_hidden = true;
    st = sync_and_check(m, first_id);
    leave(m);
    return st;
}

extern "C" {

qd_status qd_prefill(qd_handle h, const int32_t *tokens, const void *embeds, int n, int head_idx, int32_t *first_id) {
    return prefill_impl(h, tokens, embeds, n, head_idx, nullptr, first_id);
}

qd_status qd_prefill_mrope(qd_handle h, const int32_t *tokens, const void *embeds, int n, int head_idx,
                           const int32_t *positions, int32_t *first_id) {
    if (h && !positions) return fail(h, QD_EINVAL, "positions is NULL");
    return prefill_impl(h, tokens, embeds, n, head_idx, positions, first_id);
}

static qd_status check_decode(qd_model *m, int head_idx, int n_steps) {
    if (m->h_pos == 0) return fail(m, QD_ESTATE, "decode before prefill");
    if (head_idx < 0 || head_idx >= m->cfg.n_heads_out) return fail(m, QD_EINVAL, "head_idx %d out of range", head_idx);
    if (m->h_pos + n_steps > m->max_pos)
        return fail(m, QD_EKVFULL, "position %d + %d steps exceeds the last bucket (%d)", m->h_pos, n_steps, m->max_pos);
    if (m->h_pos + m->h_rope_delta + n_steps > m->max_pos)
        return fail(m, QD_EKVFULL, "rotary position %d + %d steps exceeds the RoPE table (%d rows)",
                    m->h_pos + m->h_rope_delta, n_steps, m->max_pos);
    return QD_OK;
}

qd_status qd_decode_step(qd_handle h, const void *embed, int32_t token, int head_idx, int32_t *out_id) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    const qd_config &c = m->cfg;
    if (!out_id) return fail(m, QD_EINVAL, "out_id is NULL");
    qd_status st = check_decode(m, head_idx, 1);
    if (st) return st;
    if (!embed) {
        if (token < 0 || token >= c.embed_rows) return fail(m, QD_EINVAL, "token %d outside the embedding table", token);
    } else if (!is_device_ptr(embed)) {
        return fail(m, QD_EINVAL, "embed is not a device pointer");
    }
    if (token >= c.vocab) return fail(m, QD_EINVAL, "token %d >= vocab", token);
    enter(m);
    st = grow_if_needed(m);
    if (st) return st;
    if (embed) CU(cudaMemcpyAsync(m->embed_in, embed, (size_t)c.hidden * 4, cudaMemcpyDeviceToDevice, m->ls));
    st = set_params(m, embed ? IN_EMBED : IN_TOKEN, token, token >= 0, head_idx);
    if (st) return st;
    st = run_step(m, true);
    if (st) return st;
    m->h_pos++;
    m->h_ngen++;
    m->have_hidden = true;
    st = sync_and_check(m, out_id);
    leave(m);
    return st;
}

qd_status qd_decode_step_async(qd_handle h, const void *embed, const int32_t *token_dev, int head_idx,
                               int32_t *out_id_dev) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    const qd_config &c = m->cfg;
    qd_status st = check_decode(m, head_idx, 1);
    if (st) return st;
    if (!embed && !token_dev) return fail(m, QD_EINVAL, "need an embedding or a token");
    if (embed && !is_device_ptr(embed)) return fail(m, QD_EINVAL, "embed is not a device pointer");
    if (token_dev && !is_device_ptr(token_dev)) return fail(m, QD_EINVAL, "token_dev is not a device pointer");
    if (out_id_dev && !is_device_ptr(out_id_dev)) return fail(m, QD_EINVAL, "out_id_dev is not a device pointer");
    enter(m);
    st = grow_if_needed(m);
    if (st) return st;
    if (embed) CU(cudaMemcpyAsync(m->embed_in, embed, (size_t)c.hidden * 4, cudaMemcpyDeviceToDevice, m->ls));
    st = set_params(m, embed ? IN_EMBED : IN_TOKEN, -1, 1, head_idx);
    if (st) return st;
    if (token_dev) CU(cudaMemcpyAsync(&m->st->token_in, token_dev, 4, cudaMemcpyDeviceToDevice, m->ls));
    st = run_step(m, true);
    if (st) return st;
    m->h_pos++;
    m->h_ngen++;
    m->have_hidden = true;
    if (out_id_dev) CU(cudaMemcpyAsync(out_id_dev, &m->st->out_id, 4, cudaMemcpyDeviceToDevice, m->ls));
    leave(m);
    return QD_OK;
}

qd_status qd_decode_greedy(qd_handle h, int n_steps, int32_t first_token, int32_t *ids_dev) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    const qd_config &c = m->cfg;
    if (n_steps < 0) return fail(m, QD_EINVAL, "n_steps < 0");
    if (n_steps == 0) return QD_OK;
    qd_status st = check_decode(m, 0, n_steps);
    if (st) return st;
    if (!ids_dev || !is_device_ptr(ids_dev)) return fail(m, QD_EINVAL, "ids_dev is not a device pointer");
    if (first_token >= 0 && (first_token >= c.embed_rows || first_token >= c.vocab))
        return fail(m, QD_EINVAL, "first_token %d out of range", first_token);
    if (first_token < 0 && m->h_ngen == 0) return fail(m, QD_ESTATE, "no previous id to feed back");
    if (!c.embed_rows) return fail(m, QD_EINVAL, "greedy feedback needs an embedding table");
    if (m->h_ngen + n_steps > kIdsCap) return fail(m, QD_EINVAL, "id history full: reset");
    enter(m);
    const int n0 = m->h_ngen;
    for (int i = 0; i < n_steps; ++i) {
        st = grow_if_needed(m);
        if (st) return st;
        if (i == 0) st = set_params(m, first_token >= 0 ? IN_TOKEN : IN_FEEDBACK, first_token, 1, 0);
        else if (i == 1) st = set_params(m, IN_FEEDBACK, -1, 1, 0);
        if (st) return st;
        st = run_step(m, true);
        if (st) return st;
        m->h_pos++;
        m->h_ngen++;
    }
    m->have_hidden = true;
    CU(cudaMemcpyAsync(ids_dev, m->ids + n0, (size_t)n_steps * 4, cudaMemcpyDeviceToDevice, m->ls));
    leave(m);
    return QD_OK;
}

qd_status qd_grow_kv(qd_handle h, int new_smax) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    int b = -1;
    for (int i = 0; i < m->cfg.n_buckets; ++i)
        if (m->cfg.buckets[i] == new_smax) b = i;
    if (b < 0) return fail(m, QD_EINVAL, "Smax %d is not in the bucket ladder", new_smax);
    if (b <= m->cur_bucket) return fail(m, QD_EINVAL, "Smax %d is not larger than the current %d", new_smax, m->S());
    enter(m);
    qd_status st = migrate(m, b);
    leave(m);
    return st;
}

qd_status qd_get_hidden(qd_handle h, float *out_dev) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    if (!m->have_hidden) return fail(m, QD_ESTATE, "no step with a head has run since reset");
    if (!is_device_ptr(out_dev)) return fail(m, QD_EINVAL, "out_dev is not a device pointer");
    enter(m);
    CU(cudaMemcpyAsync(out_dev, m->y, (size_t)m->cfg.hidden * 4, cudaMemcpyDeviceToDevice, m->ls));
    leave(m);
    return QD_OK;
}

qd_status qd_set_sampling(qd_handle h, int top_k, float temperature, float top_p, uint64_t seed) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    if (top_k < 0 || top_k > kMaxTopK) return fail(m, QD_EINVAL, "top_k %d outside [0, %d]", top_k, kMaxTopK);
    if (!(temperature > 0.f) || !std::isfinite(temperature))
        return fail(m, QD_EINVAL, "temperature must be > 0 (got %g)", (double)temperature);
    if (!(top_p > 0.f) || top_p > 1.f) return fail(m, QD_EINVAL, "top_p must be in (0, 1] (got %g)", (double)top_p);
    if (top_k > 0) {
        // every head CTA's candidates in the global scratch; the last CTA's selection
        // scratch and all candidates in its idle ring
        auto fits = [&](int grid, int nst) {
            const size_t words = 2 * (size_t)kMaxTopK + kTopkScratchWords + 2 * (size_t)grid * top_k;
            return (size_t)grid * top_k <= (size_t)kHeadCandidates && words * 4 <= (size_t)nst * kSlotBytes;
        };
        if (!fits(m->grid_head, m->nst_head) || (m->persistent && !fits(m->num_sms, m->nst_step)))
            return fail(m, QD_EUNSUPPORTED, "top_k %d too large for this model's head layout", top_k);
    }
    struct {
        int k;
        float t, p;
        uint32_t lo, hi;
    } v = {top_k, temperature, top_p, (uint32_t)seed, (uint32_t)(seed >> 32)};
    static_assert(sizeof(v) == 5 * 4, "sampling fields");
    enter(m);
    // pageable source: staged by the runtime before the call returns
    CU(cudaMemcpyAsync(&m->st->sample_k, &v, sizeof(v), cudaMemcpyHostToDevice, m->ls));
    leave(m);
    return QD_OK;
}

qd_status qd_set_debug_taps(qd_handle h, float *hidden_taps_dev, float *logits_dev) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    if (hidden_taps_dev && !is_device_ptr(hidden_taps_dev)) return fail(m, QD_EINVAL, "hidden taps not on device");
    if (logits_dev && !is_device_ptr(logits_dev)) return fail(m, QD_EINVAL, "logits tap not on device");
    m->tap_hidden = hidden_taps_dev;
    m->tap_logits = logits_dev;
    return QD_OK;
}

qd_status qd_set_graphs(qd_handle h, int enable) {
    if (!h) return QD_EINVAL;
    h->use_graphs = enable != 0;
    return QD_OK;
}

qd_status qd_copy_kv(qd_handle h, void *dst_dev, size_t *bytes) {
    if (!h || !bytes) return QD_EINVAL;
    qd_model *m = h;
    const size_t need = m->kv_bytes(m->cur_bucket);
    if (!dst_dev) {
        *bytes = need;
        return QD_OK;
    }
    if (*bytes < need) return fail(m, QD_EINVAL, "destination holds %zu bytes, need %zu", *bytes, need);
    if (!is_device_ptr(dst_dev)) return fail(m, QD_EINVAL, "dst_dev is not a device pointer");
    enter(m);
    CU(cudaMemcpyAsync(dst_dev, m->kv[m->cur_bucket], need, cudaMemcpyDeviceToDevice, m->ls));
    CU(cudaStreamSynchronize(m->ls));
    leave(m);
    *bytes = need;
    return QD_OK;
}

qd_status qd_get_emitted(qd_handle h, uint32_t *dst_dev) {
    if (!h) return QD_EINVAL;
    qd_model *m = h;
    if (!is_device_ptr(dst_dev)) return fail(m, QD_EINVAL, "dst_dev is not a device pointer");
    enter(m);
    CU(cudaMemcpyAsync(dst_dev, m->emitted, (size_t)((m->cfg.vocab + 31) / 32) * 4, cudaMemcpyDeviceToDevice, m->ls));
    leave(m);
    return QD_OK;
}

qd_status qd_get_pos(qd_handle h, int *pos, int *smax) {
    if (!h) return QD_EINVAL;
    if (pos) *pos = h->h_pos;
    if (smax) *smax = h->S();
    return QD_OK;
}

qd_status qd_get_launch_count(qd_handle h, long long *kernels, int *kernels_per_step) {
    if (!h) return QD_EINVAL;
    if (kernels) *kernels = h->launches;
    if (kernels_per_step) *kernels_per_step = h->kernels_per_step(true);
    return QD_OK;
}

// Time `reps` whole decode steps (the persistent step kernel, or the per-phase kernel
// sequence) as issued by the decode loop, between CUDA events on the library
// stream; then put back the position, the device state, the residual and the
// emitted set.  Rows written past the restored position are never read before
// being rewritten.
static qd_status time_step(qd_model *m, int reps, float *avg_ms) {
    const qd_config &c = m->cfg;
    if (m->h_pos + reps + 3 > m->S())
        return fail(m, QD_EINVAL, "%d timed steps do not fit in the current bucket from position %d", reps, m->h_pos);
    enter(m);
    CU(cudaStreamSynchronize(m->ls));
    const size_t emw = (size_t)((c.vocab + 31) / 32) * 4;
    std::vector<uint8_t> save_x(c.hidden * 4), save_st(sizeof(DevState)), save_em(emw);
    CU(cudaMemcpy(save_x.data(), m->x, save_x.size(), cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(save_st.data(), m->st, save_st.size(), cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(save_em.data(), m->emitted, emw, cudaMemcpyDeviceToHost));
    const int pos0 = m->h_pos;
    const long long launches0 = m->launches;
    qd_status st = QD_OK;
    for (int i = 0; i < 3 && !st; ++i, ++m->h_pos) st = run_step(m, true);
    if (!st) {
        CU(cudaEventRecord(m->ev_t0, m->ls));
        for (int i = 0; i < reps && !st; ++i, ++m->h_pos) st = run_step(m, true);
        CU(cudaEventRecord(m->ev_t1, m->ls));
        CU(cudaEventSynchronize(m->ev_t1));
    }
    m->h_pos = pos0;
    m->launches = launches0;
    if (st) return st;
    float ms = 0.f;
    CU(cudaEventElapsedTime(&ms, m->ev_t0, m->ev_t1));
    *avg_ms = ms / reps;
    CU(cudaMemcpy(m->x, save_x.data(), save_x.size(), cudaMemcpyHostToDevice));
    CU(cudaMemcpy(m->st, save_st.data(), save_st.size(), cudaMemcpyHostToDevice));
    CU(cudaMemcpy(m->emitted, save_em.data(), emw, cudaMemcpyHostToDevice));
    leave(m);
    return QD_OK;
}

qd_status qd_time_kernel(qd_handle h, int which, int reps, float *avg_ms) {
    if (!h || !avg_ms) return QD_EINVAL;
    qd_model *m = h;
    const qd_config &c = m->cfg;
    if (reps < 1 || which < 0 || which > 6) return fail(m, QD_EINVAL, "bad which/reps");
    if (m->h_pos == 0) return fail(m, QD_ESTATE, "time_kernel needs a prefilled handle");
    if (which == 6) return time_step(m, reps, avg_ms);
    if (m->q8 && which != 4)
        return fail(m, QD_EUNSUPPORTED, "8-bit weights: only the whole step and the attention kernel are timed");
    enter(m);
    CU(cudaStreamSynchronize(m->ls));
    // Save what the timed kernel overwrites (x, the device state and, for attention,
    // the cache rows of the last position of layer 0), then point the state at the
    // last position so that the kernels see the arguments of the step that wrote it.
    std::vector<uint8_t> save_x(c.hidden * 4), save_st(sizeof(DevState));
    CU(cudaMemcpy(save_x.data(), m->x, save_x.size(), cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(save_st.data(), m->st, save_st.size(), cudaMemcpyDeviceToHost));
    const int S = m->S();
    const size_t rowb = (size_t)c.head_dim * m->esize;
    std::vector<uint8_t> save_kv(2 * (size_t)c.n_kv_heads * rowb);
    uint8_t *kv0 = reinterpret_cast<uint8_t *>(m->kv[m->cur_bucket]);
    const int last = m->h_pos - 1;
    CU(cudaMemcpy2D(save_kv.data(), rowb, kv0 + (size_t)last * rowb, (size_t)S * rowb, rowb, 2 * c.n_kv_heads,
                    cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(&m->st->pos, &last, sizeof(int), cudaMemcpyHostToDevice));
    auto one = [&]() -> qd_status {
        switch (which) {
            case 0: CU(launch_gemv(GEMV_HEAD, m->bf16, head_args(m, nullptr, 0), m->grid_head, m->smem_head, m->ls, false)); break;
            case 1: CU(launch_gemv(GEMV_QKV, m->bf16, qkv_args(m, 0, false), m->grid_qkv, m->smem_qkv, m->ls, false)); break;
            case 2: CU(launch_gemv(GEMV_GU, m->bf16, gu_args(m, 0), m->grid_gu, m->smem_gu, m->ls, false)); break;
            case 3: CU(launch_gemv(GEMV_RES, m->bf16, d_args(m, 0), m->grid_d, m->smem_d, m->ls, false)); break;
            case 4: CU(launch_attention(m->bf16, c.head_dim, attn_args(m, 0), m->ls, false)); break;
            case 5: CU(launch_gemv(GEMV_RES, m->bf16, o_args(m, 0), m->grid_o, m->smem_o, m->ls, false)); break;
        }
        return QD_OK;
    };
    qd_status st = QD_OK;
    for (int i = 0; i < 3 && !st; ++i) st = one();
    if (st) return st;
    CU(cudaEventRecord(m->ev_t0, m->ls));
    for (int i = 0; i < reps && !st; ++i) st = one();
    if (st) return st;
    CU(cudaEventRecord(m->ev_t1, m->ls));
    CU(cudaEventSynchronize(m->ev_t1));
    float ms = 0.f;
    CU(cudaEventElapsedTime(&ms, m->ev_t0, m->ev_t1));
    *avg_ms = ms / reps;
    m->launches += 3 + reps;
    CU(cudaMemcpy(m->x, save_x.data(), save_x.size(), cudaMemcpyHostToDevice));
    CU(cudaMemcpy(m->st, save_st.data(), save_st.size(), cudaMemcpyHostToDevice));
    CU(cudaMemcpy2D(kv0 + (size_t)last * rowb, (size_t)S * rowb, save_kv.data(), rowb, rowb, 2 * c.n_kv_heads,
                    cudaMemcpyHostToDevice));
    leave(m);
    return QD_OK;
}

}  // extern "C"

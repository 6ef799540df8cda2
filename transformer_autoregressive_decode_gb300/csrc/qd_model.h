// Host-side state of one decode handle and the engine helpers shared by the
// entry points (qd_engine.cu) and the two-level frame loop (frame_engine.cu).
#pragma once

#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "../../include/qd.h"
#include "qd_device.cuh"
#include "qd_internal.h"

namespace qd {

struct Layer {
    void *w_qkv, *w_o, *w_gu, *w_d;
    float *attn_norm, *mlp_norm, *q_norm, *k_norm;
};

constexpr int kIdsCap = 1 << 20;

}  // namespace qd

struct qd_frame;

struct qd_model {
    qd_config cfg{};
    bool bf16 = false;
    bool q8 = false;    // layer matrices and heads as 8-bit rows (qd_config.weight_q8)
    size_t esize = 4;
    int device = 0, num_sms = 0;
    cudaStream_t user = nullptr, ls = nullptr;
    cudaEvent_t ev_in = nullptr, ev_out = nullptr, ev_t0 = nullptr, ev_t1 = nullptr;

    // library-owned weights
    void *arena = nullptr;
    std::vector<qd::Layer> layers;
    void *embed = nullptr;
    void *heads[QD_MAX_HEADS] = {};
    const void **d_heads = nullptr;
    float *final_norm = nullptr;
    float *rope_cos = nullptr, *rope_sin = nullptr;
    int max_pos = 0;

    // step scratch
    void *scratch = nullptr;
    float *x = nullptr, *qkv = nullptr, *att = nullptr, *act = nullptr, *y = nullptr;
    float *embed_in = nullptr, *stage_embeds = nullptr, *head_pv = nullptr;
    int *head_cnt = nullptr, *head_pi = nullptr, *stage_tokens = nullptr;
    int32_t *ids = nullptr;
    uint32_t *emitted = nullptr;
    qd::DevState *st = nullptr;
    int *pin = nullptr;  // pinned host words: out_id, n_gen, status
    int chunk_max = 0;

    // buckets
    std::vector<void *> kv;                   // per bucket, allocated on first use
    std::vector<cudaGraphExec_t> graphs[2];   // [with_head][bucket]
    int cur_bucket = 0;
    int h_pos = 0;
    int h_ngen = 0;
    int h_rope_delta = 0;          // rotary position of a decode step - its cache position
    int *stage_rpos = nullptr;     // [3][max_pos] staged prompt rotary positions (t, h, w)
    bool have_hidden = false;

    // launch geometry
    int grid_qkv = 0, grid_o = 0, grid_gu = 0, grid_d = 0, grid_head = 0;
    int rs_h = 0, rs_q = 0, rs_f = 0;
    int nst_qkv = 0, nst_o = 0, nst_gu = 0, nst_d = 0, nst_head = 0;
    int rps_h = 0, rps_q = 0, rps_f = 0;
    int rmax_qkv = 0, rmax_o = 0, rmax_gu = 0, rmax_d = 0, rmax_head = 0;
    size_t smem_qkv = 0, smem_o = 0, smem_gu = 0, smem_d = 0, smem_head = 0;
    int evict_last_layers = 0;

    // persistent decode step (one cooperative launch per step)
    bool persistent = false;
    // prompt prefill through the batched kernels: an internal one-stream batch
    qd_batch *pf_batch = nullptr;
    cudaEvent_t pf_ev[2] = {nullptr, nullptr};
    qd::LayerDev *d_layers = nullptr;
    // persistent step: the tagged words of every layer, then the launch sequence number
    // and the emitted-set flag
    uint64_t *tag_buf = nullptr;
    int tg_stride = 0, tg_qkv = 0, tg_po = 0, tg_ml = 0, tg_att = 0, tg_xc = 0, tg_xe = 0, tg_act = 0;
    size_t tg_words = 0;
    unsigned *barrier = nullptr;
    size_t smem_step = 0;
    int nst_step = 0, off_full = 0, off_gsm = 0, off_misc = 0, off_res = 0, off_att = 0, off_emw = 0, off_xin = 0;
    int off_kc = 0, off_xres = 0, off_ldev = 0, off_xs = 0;

    std::vector<qd_frame *> frames;          // frame generators bound to this handle
    bool use_graphs = true;
    bool use_pdl = true;
    float *tap_hidden = nullptr, *tap_logits = nullptr;
    long long launches = 0;
    std::string err;

    int q_dim() const { return cfg.n_q_heads * cfg.head_dim; }
    int kv_dim() const { return cfg.n_kv_heads * cfg.head_dim; }
    int S() const { return cfg.buckets[cur_bucket]; }
    int kernels_per_step(bool with_head) const {
        return persistent ? 1 : 5 * cfg.n_layers + (with_head ? 1 : 0);
    }
    size_t kv_bytes(int bucket) const {
        return (size_t)cfg.n_layers * 2 * kv_dim() * (size_t)cfg.buckets[bucket] * esize;
    }
};

// Engine helpers (qd_engine.cu).
qd_status fail(qd_model *m, qd_status st, const char *fmt, ...);
bool is_device_ptr(const void *p);
void enter(qd_model *m);
void leave(qd_model *m);
qd_status enqueue_step(qd_model *m, cudaStream_t s, bool with_head, bool taps);
qd_status grow_if_needed(qd_model *m);
qd_status sync_and_check(qd_model *m, int *out_id);
// Unbind a frame generator from both of its models (frame_engine.cu); called when
// either model is destroyed first.
void frame_detach(qd_frame *fr);
// The layers of a prefill of n positions from device embeddings (or device token ids of
// the embedding table) through the batched prefill kernels into KV bucket `bucket`; the
// last position's hidden state lands in x, the position at n - 1, for the head step
// (batch_engine.cu).  QD_EUNSUPPORTED, with nothing enqueued, where the model or the
// shapes do not allow it.
qd_status model_prefill_batched(qd_model *m, const float *embeds_dev, const int32_t *tokens_dev, int n, int bucket,
                                const int *rope_pos = nullptr, int rope_stride = 0);

#define CU(call)                                                                                   \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess)                                                                     \
            return fail(m, e_ == cudaErrorMemoryAllocation ? QD_ENOMEM : QD_ECUDA, "%s: %s (%s:%d)", #call, \
                        cudaGetErrorString(e_), __FILE__, __LINE__);                               \
    } while (0)

// Two-level frame loop behind qd_frame_create / qd_frame_generate: a Talker handle
// and a Code Predictor handle driven frame by frame on the device.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation": one primary code per Talker step, 15 residual codes from the Code
//    Predictor, the 16 code embeddings plus the text/pad embedding as the next Talker
//    input, and a predictor that keeps no cache across frames.
//  - "qwen3-tts-hip OPTIMIZATION_LOG": the predictor's sub-stages (prefix, two-position
//    stack prefill, first logits and token, then the remaining steps) and graph replay
//    of the repeated predictor steps.
//
// A frame is enqueued as: predictor prefill input, two predictor positions, 14 x
// (predictor input, predictor step), the embedding sum, and (all but the last frame
// of a call) the Talker step.  It is captured once per Talker bucket as a CUDA graph;
// the per-call pointers (text, forced ids, outputs) and the frame index live in a
// device control block, so the same graphs serve every call.
#include <cuda_runtime.h>

#include <vector>

#include "qd_model.h"

using namespace qd;

struct qd_frame {
    qd_model *T = nullptr, *C = nullptr;
    void *tables = nullptr;                  // E_1..E_15, library-owned copy
    FrameCtl *ctl = nullptr;                 // device control block
    FrameArgs args{};
    std::vector<cudaGraphExec_t> graphs[2];  // [frame ends with a Talker step][Talker bucket]
    bool use_graphs = true;
    int code_rows = 0;
};

namespace {

constexpr int kCodePredictorHeads = QD_FRAME_CODES - 1;
constexpr int kPredictorPositions = QD_FRAME_CODES;   // 2 prefill positions + 14 steps

int kernels_per_frame_predictor(const qd_model *C) {
    // prefill input + 2 positions + 14 x (input + step) + sum
    return 1 + C->kernels_per_step(false) + C->kernels_per_step(true) +
           (kCodePredictorHeads - 1) * (1 + C->kernels_per_step(true)) + 1;
}

// Enqueue one frame on stream s (captured into a graph, or run eagerly).
qd_status enqueue_frame(qd_frame *fr, cudaStream_t s, bool talker_step) {
    qd_model *m = fr->T;
    qd_model *C = fr->C;
    // debug taps (eager frames only: a frame with taps set is never captured) record
    // each model's last step of the frame
    const bool tc = C->tap_hidden || C->tap_logits, tt = m->tap_hidden || m->tap_logits;
    CU(launch_frame_cp_prefill(fr->args, s));
    qd_status st = enqueue_step(C, s, false, tc);      // position 0: the Talker's hidden state
    if (!st) st = enqueue_step(C, s, true, tc);        // position 1: E_0[primary], head 0
    for (int j = 1; j < kCodePredictorHeads && !st; ++j) {
        CU(launch_frame_cp_input(fr->args, j, s));
        st = enqueue_step(C, s, true, tc);
    }
    if (st) return fail(m, st, "code predictor step: %s", C->err.c_str());
    CU(launch_frame_sum(fr->args, s));
    if (talker_step) return enqueue_step(m, s, true, tt);
    return QD_OK;
}

qd_status run_frame(qd_frame *fr, bool talker_step) {
    qd_model *m = fr->T;
    const bool taps = m->tap_hidden || m->tap_logits || fr->C->tap_hidden || fr->C->tap_logits;
    if (taps || !fr->use_graphs) return enqueue_frame(fr, m->ls, talker_step);
    // a frame without the Talker step does not depend on the Talker's bucket
    cudaGraphExec_t &ex = fr->graphs[talker_step ? 1 : 0][talker_step ? m->cur_bucket : 0];
    if (!ex) {
        cudaGraph_t g = nullptr;
        CU(cudaStreamBeginCapture(m->ls, cudaStreamCaptureModeThreadLocal));
        qd_status st = enqueue_frame(fr, m->ls, talker_step);
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
    return QD_OK;
}

void unlink(qd_model *m, qd_frame *fr) {
    if (!m) return;
    auto &v = m->frames;
    for (size_t i = 0; i < v.size(); ++i)
        if (v[i] == fr) {
            v.erase(v.begin() + i);
            return;
        }
}

void destroy_frame(qd_frame *fr) {
    if (!fr) return;
    frame_detach(fr);
    if (fr->tables) cudaFree(fr->tables);
    if (fr->ctl) cudaFree(fr->ctl);
    delete fr;
}

}  // namespace

// Wait for the frame work in flight, drop the graphs (they capture the models'
// buffers) and forget both models; a detached generator only accepts destroy.
void frame_detach(qd_frame *fr) {
    if (fr->T && fr->T->ls) cudaStreamSynchronize(fr->T->ls);
    for (auto &v : fr->graphs)
        for (cudaGraphExec_t &g : v)
            if (g) {
                cudaGraphExecDestroy(g);
                g = nullptr;
            }
    unlink(fr->T, fr);
    unlink(fr->C, fr);
    fr->T = fr->C = nullptr;
}

extern "C" {

qd_status qd_frame_create(qd_handle talker, qd_handle predictor, const void *const *code_tables, int code_rows,
                          int dtype, qd_frame_handle *out) {
    if (!out) return QD_EINVAL;
    *out = nullptr;
    if (!talker || !predictor || talker == predictor) return QD_EINVAL;
    qd_model *m = talker;
    qd_model *C = predictor;
    const qd_config &tc = m->cfg, &cc = C->cfg;
    if (!code_tables) return fail(m, QD_EINVAL, "code_tables is NULL");
    if (tc.embed_rows < 1 || !m->embed) return fail(m, QD_EINVAL, "the Talker needs an embedding table");
    if (cc.hidden != tc.hidden) return fail(m, QD_EINVAL, "hidden sizes differ (%d vs %d)", cc.hidden, tc.hidden);
    if (cc.dtype != tc.dtype || dtype != tc.dtype) return fail(m, QD_EINVAL, "dtypes of models and tables differ");
    if (cc.n_heads_out != kCodePredictorHeads)
        return fail(m, QD_EINVAL, "the predictor needs %d output heads (has %d)", kCodePredictorHeads, cc.n_heads_out);
    if (cc.buckets[0] < kPredictorPositions)
        return fail(m, QD_EINVAL, "the predictor's first bucket must hold %d positions", kPredictorPositions);
    if (code_rows < cc.vocab) return fail(m, QD_EINVAL, "code_rows %d < predictor vocab %d", code_rows, cc.vocab);
    if (m->device != C->device) return fail(m, QD_EINVAL, "the handles are on different devices");
    for (int j = 0; j < kCodePredictorHeads; ++j)
        if (!is_device_ptr(code_tables[j])) return fail(m, QD_EINVAL, "code_tables[%d] is not a device pointer", j);

    qd_frame *fr = new qd_frame();
    fr->T = m;
    fr->C = C;
    fr->code_rows = code_rows;
    const size_t table_bytes = (size_t)code_rows * tc.hidden * m->esize;
    qd_status st = QD_OK;
    auto check = [&](cudaError_t e, const char *what) {
        if (e != cudaSuccess && !st)
            st = fail(m, e == cudaErrorMemoryAllocation ? QD_ENOMEM : QD_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    };
    check(cudaMalloc(&fr->tables, table_bytes * kCodePredictorHeads), "cudaMalloc(code tables)");
    check(cudaMalloc(&fr->ctl, sizeof(FrameCtl)), "cudaMalloc(frame control)");
    enter(m);
    for (int j = 0; j < kCodePredictorHeads && !st; ++j)
        check(cudaMemcpyAsync(static_cast<uint8_t *>(fr->tables) + j * table_bytes, code_tables[j], table_bytes,
                              cudaMemcpyDeviceToDevice, m->ls),
              "copy of a code table");
    if (!st) check(cudaMemsetAsync(fr->ctl, 0, sizeof(FrameCtl), m->ls), "cudaMemsetAsync");
    if (!st) check(cudaStreamSynchronize(m->ls), "cudaStreamSynchronize");
    leave(m);
    if (st) {
        destroy_frame(fr);
        return st;
    }
    FrameArgs &a = fr->args;
    a.table[0] = m->embed;
    for (int j = 1; j < QD_FRAME_CODES; ++j) a.table[j] = static_cast<uint8_t *>(fr->tables) + (j - 1) * table_bytes;
    a.rows0 = tc.embed_rows;
    a.rows = code_rows;
    a.bf16 = m->bf16 ? 1 : 0;
    a.hidden = tc.hidden;
    a.ctl = fr->ctl;
    a.t_st = m->st;
    a.t_y = m->y;
    a.t_embed_in = m->embed_in;
    a.c_st = C->st;
    a.c_ids = C->ids;
    a.c_embed_in = C->embed_in;
    a.c_stage = C->stage_embeds;
    a.c_emitted = C->emitted;
    a.c_emitted_words = (cc.vocab + 31) / 32;
    fr->graphs[0].assign(1, nullptr);
    fr->graphs[1].assign(tc.n_buckets, nullptr);
    m->frames.push_back(fr);
    C->frames.push_back(fr);
    *out = fr;
    return QD_OK;
}

qd_status qd_frame_destroy(qd_frame_handle f) {
    destroy_frame(f);
    return QD_OK;
}

qd_status qd_frame_set_graphs(qd_frame_handle f, int enable) {
    if (!f || !f->T) return QD_EINVAL;
    f->use_graphs = enable != 0;
    return QD_OK;
}

qd_status qd_frame_generate(qd_frame_handle fr, int n_frames, const float *text_dev, const int32_t *force_dev,
                            int32_t *codes_dev, float *next_in_dev) {
    if (!fr) return QD_EINVAL;
    if (!fr->T) return QD_ESTATE;      // a model was destroyed: only qd_frame_destroy is valid
    qd_model *m = fr->T;
    qd_model *C = fr->C;
    if (n_frames < 0) return fail(m, QD_EINVAL, "n_frames < 0");
    if (n_frames == 0) return QD_OK;
    if (!is_device_ptr(text_dev)) return fail(m, QD_EINVAL, "text_dev is not a device pointer");
    if (!is_device_ptr(codes_dev)) return fail(m, QD_EINVAL, "codes_dev is not a device pointer");
    if (force_dev && !is_device_ptr(force_dev)) return fail(m, QD_EINVAL, "force_dev is not a device pointer");
    if (next_in_dev && !is_device_ptr(next_in_dev)) return fail(m, QD_EINVAL, "next_in_dev is not a device pointer");
    if (m->h_ngen < 1 || !m->have_hidden) return fail(m, QD_ESTATE, "the Talker has produced no id yet");
    const int talker_steps = n_frames - 1;
    if (m->h_pos + talker_steps > m->max_pos)
        return fail(m, QD_EKVFULL, "position %d + %d Talker steps exceeds the last bucket (%d)", m->h_pos,
                    talker_steps, m->max_pos);
    if (m->h_ngen + talker_steps > kIdsCap) return fail(m, QD_EINVAL, "Talker id history full: reset");

    enter(m);
    // order after the predictor's prior work
    CU(cudaEventRecord(C->ev_in, C->user));
    CU(cudaStreamWaitEvent(m->ls, C->ev_in, 0));
    FrameCtl h = {};
    h.f = 0;
    h.n_frames = n_frames;
    h.text = text_dev;
    h.force = force_dev;
    h.codes = codes_dev;
    h.next_in = next_in_dev;
    // pageable source: staged by the runtime before the call returns
    CU(cudaMemcpyAsync(fr->ctl, &h, sizeof(h), cudaMemcpyHostToDevice, m->ls));
    C->cur_bucket = 0;   // every frame restarts the predictor in its first bucket
    const int per_frame = kernels_per_frame_predictor(C);
    qd_status st = QD_OK;
    int ran = 0;
    for (int f = 0; f < n_frames; ++f) {
        const bool talker_step = f < talker_steps;
        if (talker_step) st = grow_if_needed(m);
        if (!st) st = run_frame(fr, talker_step);
        if (st) break;
        ++ran;
        C->launches += per_frame;
        if (talker_step) {
            m->launches += m->kernels_per_step(true);
            m->h_pos++;
            m->h_ngen++;
        }
    }
    if (ran) {
        C->h_pos = kPredictorPositions;
        C->h_ngen = kCodePredictorHeads;
        C->have_hidden = true;
    }
    leave(m);
    CU(cudaStreamWaitEvent(C->user, m->ev_out, 0));
    CU(cudaStreamWaitEvent(C->ls, m->ev_out, 0));
    return st;
}

}  // extern "C"

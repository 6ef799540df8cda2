// Kernels of the two-level frame loop.
//
// Sources (page title, section):
//  - "Qwen3-TTS ncnn port", section "Talker: non-standard structure and two-level
//    generation": per frame the Talker emits one primary code; a 5-layer Code
//    Predictor then emits 15 residual codes one at a time, each from its own output
//    head; the 16 code embeddings are summed with the text (or pad) embedding to form
//    the Talker's next input; the Code Predictor starts afresh every frame.
//  - "qwen3-tts-hip OPTIMIZATION_LOG", Code Predictor sub-stages: the predictor is
//    prefilled with two positions (the Talker's hidden state and the primary code's
//    embedding), then every further code is one decode step.
//
// The ids never leave the device: each kernel reads the id it needs from the
// producing handle's device state (or from the caller's forced ids) and writes the
// next step's input and step description directly, so a whole frame is one
// stream-ordered (and graph-capturable) sequence with no host round trip.
// One CTA each: the work is a few rows of `hidden` elements.
#include "qd_device.cuh"
#include "qd_internal.h"

namespace qd {

namespace {

constexpr int kFrameThreads = 256;

__device__ __forceinline__ float table_elem(const void *t, int bf16, size_t off) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(t)[off])
                : reinterpret_cast<const float *>(t)[off];
}

// Frame index of the call in flight; false (and an error bit) if the host launched
// more frames than it announced.
__device__ __forceinline__ bool frame_index(const FrameArgs &a, int *f) {
    *f = a.ctl->f;
    return *f >= 0 && *f < a.ctl->n_frames;
}

// The id fed back for code j of frame f: the caller's forced id, else the argmax.
__device__ __forceinline__ int fed_id(const FrameArgs &a, int f, int j, int argmax) {
    return a.ctl->force ? a.ctl->force[(size_t)f * kFrameCodes + j] : argmax;
}

// Start of a frame: the Code Predictor starts from position 0 with an empty emitted
// set; its two prompt positions are the Talker's final-norm output and the primary
// code's row of the Talker's embedding table.  Records the primary argmax.
__global__ void __launch_bounds__(kFrameThreads) frame_cp_prefill_kernel(const FrameArgs a) {
    __shared__ int sh[2];
    if (threadIdx.x == 0) {
        int f = 0;
        const bool fok = frame_index(a, &f);
        const int primary = a.t_st->out_id;
        const int p = fok ? fed_id(a, f, 0, primary) : -1;
        const bool ok = fok && p >= 0 && p < a.rows0;
        if (!ok) atomicOr(&a.c_st->status, DEV_ERR_BAD_TOKEN);
        if (fok) a.ctl->codes[(size_t)f * kFrameCodes] = primary;
        DevState *c = a.c_st;
        c->pos = 0;
        c->in_mode = IN_STAGED_EMBEDS;
        c->token_in = -1;
        c->add_emitted = 0;
        c->head_idx = 0;
        c->n_gen = 0;
        sh[0] = ok ? p : -1;
    }
    __syncthreads();
    const int p = sh[0];
    const int h = a.hidden;
    for (int i = threadIdx.x; i < h; i += blockDim.x) {
        a.c_stage[i] = a.t_y[i];
        a.c_stage[h + i] = p >= 0 ? table_elem(a.table[0], a.bf16, (size_t)p * h + i) : 0.f;
    }
    for (int i = threadIdx.x; i < a.c_emitted_words; i += blockDim.x) a.c_emitted[i] = 0u;
}

// Input of Code Predictor step j (1..14): row code_j of table j, where code_j is the
// id the predictor produced at its previous step; head j decodes it.  The code
// joins the predictor's emitted set (the token rule of every decode step).
__global__ void __launch_bounds__(kFrameThreads) frame_cp_input_kernel(const FrameArgs a, int j) {
    __shared__ int sh[1];
    if (threadIdx.x == 0) {
        int f = 0;
        const bool fok = frame_index(a, &f);
        const int c = fok ? fed_id(a, f, j, a.c_ids[j - 1]) : -1;
        const bool ok = fok && c >= 0 && c < a.rows;
        if (!ok) atomicOr(&a.c_st->status, DEV_ERR_BAD_TOKEN);
        DevState *s = a.c_st;
        s->in_mode = IN_EMBED;
        s->token_in = ok ? c : -1;
        s->add_emitted = 1;
        s->head_idx = j;
        sh[0] = ok ? c : -1;
    }
    __syncthreads();
    const int c = sh[0];
    const int h = a.hidden;
    for (int i = threadIdx.x; i < h; i += blockDim.x)
        a.c_embed_in[i] = c >= 0 ? table_elem(a.table[j], a.bf16, (size_t)c * h + i) : 0.f;
}

// End of a frame: x = ((E_0[p] + E_1[c_1]) + ... + E_15[c_15]) + text[f], summed in
// fp32 in this order, becomes the Talker's next input, with the primary p as the
// step's token (it joins the Talker's emitted set).  Records the 15 residual
// argmaxes and advances the frame index.
__global__ void __launch_bounds__(kFrameThreads) frame_sum_kernel(const FrameArgs a) {
    __shared__ int ids[kFrameCodes];
    __shared__ int sh_f, sh_fok, sh_ok;
    if (threadIdx.x == 0) {
        int f = 0;
        sh_fok = sh_ok = frame_index(a, &f) ? 1 : 0;
        sh_f = f;
    }
    __syncthreads();
    const int f = sh_f;
    if (threadIdx.x < kFrameCodes && sh_fok) {
        const int j = threadIdx.x;
        const int argmax = j == 0 ? a.t_st->out_id : a.c_ids[j - 1];
        const int id = fed_id(a, f, j, argmax);
        const int rows = j == 0 ? a.rows0 : a.rows;
        if (id < 0 || id >= rows) atomicAnd(&sh_ok, 0);
        ids[j] = id;
        if (j > 0) a.ctl->codes[(size_t)f * kFrameCodes + j] = argmax;
    }
    __syncthreads();
    const bool ok = sh_ok != 0;
    const int h = a.hidden;
    const float *text = a.ctl->text + (size_t)f * h;
    for (int i = threadIdx.x; i < h; i += blockDim.x) {
        float v = 0.f;
        if (ok) {
            v = table_elem(a.table[0], a.bf16, (size_t)ids[0] * h + i);
            for (int j = 1; j < kFrameCodes; ++j) v += table_elem(a.table[j], a.bf16, (size_t)ids[j] * h + i);
            v += text[i];
        }
        a.t_embed_in[i] = v;
        if (a.ctl->next_in) a.ctl->next_in[i] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        DevState *t = a.t_st;
        if (!ok) atomicOr(&t->status, DEV_ERR_BAD_TOKEN);
        t->in_mode = IN_EMBED;
        t->token_in = ok ? ids[0] : -1;
        t->add_emitted = 1;
        t->head_idx = 0;
        a.ctl->f = f + 1;
    }
}

}  // namespace

cudaError_t launch_frame_cp_prefill(const FrameArgs &a, cudaStream_t s) {
    frame_cp_prefill_kernel<<<1, kFrameThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_frame_cp_input(const FrameArgs &a, int j, cudaStream_t s) {
    frame_cp_input_kernel<<<1, kFrameThreads, 0, s>>>(a, j);
    return cudaGetLastError();
}

cudaError_t launch_frame_sum(const FrameArgs &a, cudaStream_t s) {
    frame_sum_kernel<<<1, kFrameThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qd

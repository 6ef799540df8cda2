// Internal interface between the decode-step kernels and the engine (host C++).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qd {

struct DevState;

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;   // 8 consumer warps + 1 producer warp
constexpr int kAttnThreads = 128;
constexpr int kAttnMaxSplits = 8;       // splits of a kv group = CTAs of one cluster
constexpr int kSlotBytes = 32 * 1024;   // one ring stage: 32/16/8/5 rows of K = 512/1024/2048/3072 (bf16),
                                        // or one 128-position K or V tile at head_dim 128
constexpr int kRingBytes = 96 * 1024;   // ring of a per-phase kernel (3 stages)

// Positions per attention split for an attended length L: a function of L only
// (never of Smax), so a bucket migration cannot change the partition.  It keeps
// the number of splits at or below kAttnMaxSplits.
__host__ __device__ inline int attn_chunk(int L) {
    return 32 * ((L + 32 * kAttnMaxSplits - 1) / (32 * kAttnMaxSplits));
}
__host__ __device__ inline int attn_splits(int L) {
    const int c = attn_chunk(L);
    return (L + c - 1) / c;
}

enum GemvMode : int { GEMV_QKV = 0, GEMV_RES = 1, GEMV_GU = 2, GEMV_HEAD = 3 };

struct GemvArgs {
    const void *W;                 // [rows, K] row-major (not GEMV_HEAD)
    const void *const *W_table;    // GEMV_HEAD: device table of head matrices, index st->head_idx
    int rows, K;
    int rs;                        // warps per row (row split factor): 1, 2, 4 or 8
    int unit;                      // CTAs take rows in multiples of `unit` (2 for gate/up pairs)
    int nst;                       // ring stages
    int rps;                       // rows per stage
    int rows_max;                  // max rows of any CTA (sizes the result buffer)
    int evict_last;                // keep weights in L2 (evict_last) instead of evict_first
    const float *in;               // input vector [K]
    const float *gamma;            // RMSNorm gamma [K] (QKV, GU, HEAD)
    float eps;
    float *out;                    // QKV [rows]; RES [rows] (+=); GU [rows/2]; HEAD raw-logit tap or null
    // first kernel of a step: the input vector comes from the step description
    int input_mode;
    const void *table;             // embedding table [table_rows, K]
    int table_rows, table_bf16, vocab, S;
    const float *embed_in;
    const int32_t *stage_tokens;
    const float *stage_embeds;
    uint32_t *emitted_w;           // emitted bitmask (written by CTA 0)
    float *x_out;                  // x written by CTA 0 (the residual stream)
    // GEMV_HEAD
    const uint32_t *emitted;
    float penalty;
    int eos;
    float *y_out;                  // normalised input (CTA 0), or null
    float *part_v;                 // [gridDim.x]
    int *part_i;
    int *counter;                  // one int, zero at rest
    int32_t *ids;                  // id history
    int ids_cap;
    int commit;                    // 1: publish the id and advance the position (0 when timing)
    int advance_pos;               // last kernel of a step without a head: CTA 0 advances the position
    DevState *st;
};

struct AttnArgs {
    const float *qkv;              // [qh*hd | kvh*hd | kvh*hd] raw projections (fp32)
    const float *q_gamma, *k_gamma;// [hd] or null
    float eps;
    float scale;                   // 1/sqrt(hd), rounded to fp32 on the host
    const float *rope_cos, *rope_sin;  // [max_pos][hd/2]
    void *kcache, *vcache;         // this layer's [kvh][S][hd]
    int S;
    int qh, kvh;
    int chunk_max;                 // attn_chunk(max position): sizes the shared K/V tiles
    float *out;                    // [qh*hd] attention output
    DevState *st;
};

// ---------------------------------------------------------------------------------
// Persistent decode step: one cooperative launch per step, one CTA per SM.
// ---------------------------------------------------------------------------------
struct LayerDev {                  // device table, one entry per layer
    const void *w_qkv, *w_o, *w_gu, *w_d;
    const float *attn_norm, *mlp_norm, *q_norm, *k_norm;
};

struct StepInputArgs {             // where the step's input vector comes from
    const void *table;
    int table_rows, vocab, S;
    const float *embed_in;
    const int32_t *stage_tokens;
    const float *stage_embeds;
    uint32_t *emitted;
};

struct StepArgs {
    const LayerDev *layers;
    int n_layers, hidden, qh, kvh, ffn, vocab;
    int rs_h, rs_q, rs_f;          // warps per row for K = hidden, qh*hd, ffn
    int rps_h, rps_q, rps_f;       // rows per ring stage for the same
    int nst;                       // ring stages
    int evict_last;                // layer weights stay in L2
    float eps, scale;
    int off_full, off_gsm, off_misc, off_res, off_att, off_emw, off_xin;   // shared-memory layout (bytes)
    void *kv;                      // bucket buffer [n_layers][2][kvh][S][hd]
    int S, chunk_max;
    const float *rope_cos, *rope_sin;
    float *x, *qkv, *act;
    float *part_o;                 // [qh][kAttnMaxSplits][hd]
    float *part_ml;                // [qh][kAttnMaxSplits][2]
    StepInputArgs in;
    int with_head;
    const void *const *heads;
    const float *final_norm;
    float penalty;
    int eos;
    float *y_out, *part_v;
    int *part_i, *head_counter;
    int32_t *ids;
    int ids_cap;
    float *tap_hidden, *tap_logits;
    unsigned *barrier;             // zeroed before every launch
    DevState *st;
};

// Dynamic shared memory ceiling of the persistent step kernel.  The kernel's
// max-dynamic-smem attribute is set to this once for every instantiation, so
// handles of the same shape with different layouts can coexist.
constexpr int kStepMaxSmem = 227 * 1024;

// Persistent kernel for (dtype, head_dim, hidden, q_dim, ffn): false if there is no
// instantiation for the shape (the per-phase kernels are used then).
bool persistent_supported(bool bf16, int hd, int hidden, int q_dim, int ffn);
cudaError_t persistent_init(bool bf16, int hd, int hidden, int q_dim, int ffn);
cudaError_t launch_persistent(bool bf16, int hd, int hidden, int q_dim, int ffn, const StepArgs &a, int grid,
                              size_t smem, cudaStream_t s);
size_t persistent_att_bytes(int group, int hd, int chunk_max);

// Picks (nseg, rs) for K; false if K is not supported.
bool gemv_split(int K, bool bf16, int *nseg, int *rs);
// Dynamic shared memory of a GEMV launch.
size_t gemv_smem_bytes(int nst, int rows_max, int rs, int K);
// Set the max-dynamic-smem attribute on every GEMV / attention instantiation.
cudaError_t kernels_init();

cudaError_t launch_gemv(int mode, bool bf16, const GemvArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_attention(bool bf16, int hd, const AttnArgs &a, cudaStream_t s, bool pdl);
size_t attention_smem_bytes(bool bf16, int hd, int group, int chunk_max);
cudaError_t launch_kv_migrate(const void *src, int S_old, void *dst, int S_new, int n_segments, size_t row_bytes,
                              int n_pos, cudaStream_t s);
cudaError_t launch_rope_table(float *cos_t, float *sin_t, int n_pos, int head_dim, double theta, cudaStream_t s);
cudaError_t launch_to_f32(const void *src, bool bf16, float *dst, int n, cudaStream_t s);

// ---------------------------------------------------------------------------------
// Two-level frame loop: kernels that build the Code Predictor's and the Talker's
// inputs from device-resident ids.
// ---------------------------------------------------------------------------------
constexpr int kFrameCodes = 16;    // primary code + 15 residual codes per frame

struct FrameCtl {                  // device; written by the host once per call
    int f;                         // frame index within the call, advanced by the sum kernel
    int n_frames;
    const float *text;             // [n_frames][hidden] text/pad embedding of each frame
    const int32_t *force;          // [n_frames][16] ids fed back instead of the argmax, or null
    int32_t *codes;                // [n_frames][16] argmax ids: primary, then the 15 residual codes
    float *next_in;                // [hidden] the last frame's summed embedding, or null
};

struct FrameArgs {                 // fixed for a frame generator (graphs capture it)
    const void *table[kFrameCodes];// [0] the Talker's embedding table, [1..15] code tables
    int rows0, rows;               // rows of table 0 and of tables 1..15
    int bf16, hidden;
    FrameCtl *ctl;
    DevState *t_st;                // Talker
    const float *t_y;              // Talker final-norm output of its last position
    float *t_embed_in;
    DevState *c_st;                // Code Predictor
    const int32_t *c_ids;          // its id history (codes of the frame in flight)
    float *c_embed_in, *c_stage;
    uint32_t *c_emitted;
    int c_emitted_words;
};

cudaError_t launch_frame_cp_prefill(const FrameArgs &a, cudaStream_t s);
cudaError_t launch_frame_cp_input(const FrameArgs &a, int j, cudaStream_t s);
cudaError_t launch_frame_sum(const FrameArgs &a, cudaStream_t s);

}  // namespace qd

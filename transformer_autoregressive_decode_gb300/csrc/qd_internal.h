// Internal interface between the decode-step kernels and the engine (host C++).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qd {

struct DevState;

constexpr int kConsumerWarps = 8;
constexpr int kMaxTopK = 64;             // most sampling candidates (qd_set_sampling)
constexpr int kHeadCandidates = 16384;   // per-CTA head candidates in global scratch (CTAs x top-k)
// Shared-memory scratch of the block top-k selection, in 32-bit words.
constexpr int kTopkScratchWords = 256 + kConsumerWarps * 32 + 16 + 2 * kMaxTopK;
// the candidate keys after the per-CTA candidates and this scratch are 64-bit
static_assert((2 * kMaxTopK + kTopkScratchWords) % 2 == 0, "sampling scratch alignment");
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
    int rope_rows;                 // rows of the tables
    int mrope_h;                   // interleaved multimodal RoPE: the h (= w) section size, 0: plain
    const int *rope_stage;         // [3][rope_stride] staged prompt positions (t, h, w)
    int rope_stride;
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
    int rope_rows;                 // rows of the tables
    int mrope_h;                   // interleaved multimodal RoPE: the h (= w) section size, 0: plain
    const int *rope_stage;         // [3][rope_stride] staged prompt positions (t, h, w)
    int rope_stride;
    float *x;                      // the residual stream (plain copy, written by its row owners)
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
    // Tagged words {launch sequence number, value}, one block of tg_stride words per
    // layer; word offsets within a block: qkv [q + 2 kv], attention partials
    // [kvh][kAttnMaxSplits][G * hd] and their (max, sum) [kvh][kAttnMaxSplits][G][2],
    // merged attention output [q], x after the output projection [hidden], x after the
    // down projection [hidden], act [ffn]
    uint64_t *tg;
    int tg_stride, tg_qkv, tg_po, tg_ml, tg_att, tg_xc, tg_xe, tg_act;
    unsigned *seq;                 // launch sequence number (starts at 1, never 0)
    unsigned *emit_flag;           // CTA 0 stores the launch's seq (release) once the step's
                                   // token is in the emitted set
    int off_kc, off_xres, off_ldev, off_xs;   // shared memory: row-partial tables, residual rows,
                                              // layer table, the warps' input slices
    DevState *st;
};

// Rows of one GEMV phase a CTA of the persistent step may hold (its partial-sum
// tables and residual rows are sized by it), the largest q-heads-per-kv-head ratio it
// handles, its ring stages and the fewest SMs it runs on; other shapes and GPUs use
// the per-phase kernels.
constexpr int kStepRowsMax = 64;
constexpr int kStepRingStages = 6;
constexpr int kStepMinSms = 148;
constexpr int kStepGroupMax = 2;

// Weight-only 8-bit rows of the persistent step ("audio.cpp Rockchip NPU build notes",
// the talker's Q8_0 weights): a row of K weights is its K int8 codes, then its K / 32
// block scales as IEEE halves (d = max |w| / 127 per 32 weights, w ~ code * d); rows
// contiguous.  Bytes of a row, and the rows of a ring slot.
__host__ __device__ constexpr uint32_t q8_row_bytes(int K) { return (uint32_t)(K + K / 16); }
__host__ __device__ constexpr int q8_rps(int K) { return kSlotBytes / (int)q8_row_bytes(K); }
// W [rows, K] (bf16 or fp32) as 8-bit rows at dst: row r to row row0 + r * rstep.
cudaError_t launch_quantize_rows_q8(const void *w, bool bf16, int rows, int K, void *dst, int row0, int rstep,
                                    cudaStream_t s);
// Phase timeline of the traced build: CTAs and stamp slots recorded.
constexpr int kStepTraceCtas = 160;
constexpr int kStepTraceSlots = 24;

// Dynamic shared memory ceiling of the persistent step kernel.  The kernel's
// max-dynamic-smem attribute is set to this once for every instantiation, so
// handles of the same shape with different layouts can coexist.
constexpr int kStepMaxSmem = 227 * 1024;

// Persistent kernel for (dtype, head_dim, hidden, q_dim, ffn): false if there is no
// instantiation for the shape (the per-phase kernels are used then).
bool persistent_supported(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, bool q8 = false);
cudaError_t persistent_init(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, bool q8 = false);
cudaError_t launch_persistent(bool bf16, int hd, int hidden, int q_dim, int ffn, int kvh, const StepArgs &a, int grid,
                              size_t smem, cudaStream_t s, bool q8 = false);
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

// ---------------------------------------------------------------------------------
// Tensor-core GEMM (tcgen05 + TMA): out[t][r] = sum_k W[r][k] * x[t][k] for the
// batched paths (prefill, multi-stream decode).  W [R, K] bf16 row-major; x is given
// as two bf16 parts x = x_hi + x_lo ([T, K] row-major each), so the products carry
// ~16 bits of the fp32 activation; accumulation is fp32 in tensor memory.
// ---------------------------------------------------------------------------------
enum TcEpilogue : int {
    TC_STORE = 0,      // out[t][r] = acc
    TC_RESIDUAL = 1,   // out[t][r] += acc
    TC_SWIGLU = 2,     // rows (2i, 2i+1) = (gate_i, up_i): act[t][i] = silu(gate) * up,
                       // written as bf16 hi/lo parts (and fp32 when out != null)
    TC_STORE_RT = 3,   // out[r * ldo + t * ldt] = acc + bias[r] for rows r < r_valid
                       // (channel-major outputs of the codec convolutions)
    TC_RESIDUAL_NORM = 4,  // out[t][r] += acc, then the next RMSNorm's input parts:
                           // nh/nl[t][r] = bf16 hi/lo of norm_gamma[r] * out[t][r], and
                           // ss_out[r / 32][t] = sum over those 32 rows of out^2
};

struct TcGemmArgs {
    int R, K, T;                   // weight rows (multiple of 128), reduction (multiple of 64), tokens
    int mode;                      // TcEpilogue
    float *out;                    // [T][ldo] fp32 (TC_SWIGLU: optional fp32 act)
    int ldo;
    __nv_bfloat16 *act_hi, *act_lo;// TC_SWIGLU: [T][R/2]
    float *partial;                // split-K partial sums [units][BN][128], or null when splits == 1
    int *tile_counter;             // [row tiles x token tiles][2] (arrive, depart), zero at rest
    int *status;                   // DEV_ERR_* bits
    // Shifted taps (the codec convolutions; taps <= 1 is the plain product):
    // out[t][r] = sum_j sum_k W[slab(j)][r][k] * x[t - shift(j)][k], j < taps, with
    // slab(j) = w_slab0 + j w_slab_step, shift(j) = x_shift0 + j x_shift_step, rows of x
    // outside [0, T) read as zero; W then has w_rows = slabs x R rows.
    int taps, w_slab0, w_slab_step, x_shift0, x_shift_step, w_rows;
    int ldt;                       // TC_STORE_RT: token stride of out
    int r_valid;                   // TC_STORE_RT: rows written
    const float *bias;             // TC_STORE_RT: [r_valid] or null
    // TC_RESIDUAL_NORM outputs
    const float *norm_gamma;       // [R]
    __nv_bfloat16 *nh, *nl;        // [T][R]
    float *ss_out;                 // [R / 32][T]: one partial per 32-row quarter of a row tile
    // RMSNorm folded into this GEMM (its input parts were gamma * x, not yet scaled):
    // acc *= 1 / sqrt(sum_i rs_part[i][t] / rs_K + rs_eps) before the epilogue, i < rs_tiles
    const float *rs_part;
    int rs_tiles, rs_K;
    float rs_eps;
};

struct TcGemmPlan {
    int bn;                        // token tile: 64 or 128
    int row_tiles, tok_tiles, splits, units, grid;
    size_t smem;
    size_t partial_floats;         // scratch needed for split-K partials (floats)
};

// Resolve the tensor-map encoder and configure the kernels; call before any capture.
cudaError_t tc_gemm_init();
// Plan a GEMM of R x K over T tokens on `num_sms` SMs (split-K when the tiles alone
// cannot fill the GPU).  False if the shape is not supported.
bool tc_gemm_plan(int R, int K, int T, int num_sms, TcGemmPlan *p);
// Launch; w, x_hi, x_lo are device pointers (16-byte aligned, row strides K*2 bytes).
// pdl: launch as a programmatic dependent of the previous kernel in the stream (the
// chains of the batched decode step; every kernel of such a chain waits before it
// reads what its predecessor writes).
cudaError_t launch_tc_gemm(const TcGemmPlan &p, const void *w, const void *x_hi, const void *x_lo,
                           const TcGemmArgs &a, cudaStream_t s, bool pdl = false);
// x fp32 [n] -> hi = bf16(x), lo = bf16(x - hi)
cudaError_t launch_split_bf16(const float *x, __nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t n, cudaStream_t s);

// ---------------------------------------------------------------------------------
// Batched decode: B independent streams, one token each per step.
// ---------------------------------------------------------------------------------
struct BatchCtl {                  // device; written by the host once per call
    int step;                      // step index within the call, advanced by the argmax kernel
    int n_steps;
    const int32_t *force;          // [n_steps][B] ids fed back instead of the argmax, or null
    int32_t *ids;                  // [n_steps][B] argmax ids
    int done;                      // CTAs of the argmax kernel finished in this step
};

struct BatchAttnArgs {
    const float *qkv;              // [B][qkv_ld]: q heads, then k, then v of each stream
    int qkv_ld;
    const float *q_gamma, *k_gamma;// [hd] or null
    float eps, scale;
    const float *rope_cos, *rope_sin;
    void *kv;                      // [B][n_layers][2][kvh][S][hd] bf16
    size_t stream_elems;           // elements of one stream's cache
    size_t layer_elems;            // offset of this layer within a stream (elements)
    int S, qh, kvh;
    const int *pos;                // [B] position written by this step (attended length pos + 1)
    __nv_bfloat16 *out_hi, *out_lo;// [B][qh * hd] attention output as bf16 parts
    float *partial;                // [B * kvh][S / kBattChunk][G][hd + 2] chunk results
    int *counter;                  // [B * kvh] chunks done, zero at rest
    int *status;
};

// The batched attention works in chunks of kBattChunk cached positions: one CTA per
// (stream, kv group, chunk); the chunks of a pair are merged by the last of them.
constexpr int kBattChunk = 512;
__host__ __device__ inline int batch_attn_max_chunks(int S) { return (S + kBattChunk - 1) / kBattChunk; }

size_t batch_attention_smem_bytes(int hd, int group);
bool batch_attention_supported(int hd, int group);   // head_dim 64/128, 1, 2, 4 or 8 q heads per kv head
cudaError_t batch_kernels_init();   // call before any capture
// kv_map: make_kv_tile_map over the caches the arguments point into.
cudaError_t launch_batch_attention(int hd, int B, const BatchAttnArgs &a, const CUtensorMap &kv_map, cudaStream_t s,
                                   bool pdl = false);
// TMA map of bf16 caches seen as `planes` planes of [S][hd] (rows of hd elements), box
// of 64 elements x box_rows rows with the 128-byte swizzle (the batched attention's
// 32-position tiles, the prefill attention's 128-key chunks); false if the driver
// refuses it.
bool make_kv_tile_map(CUtensorMap *m, const void *kv, int hd, int S, long long planes, int box_rows = 32);
// TMA map of a row-major bf16 matrix [rows, K], box of 64 elements x box_rows rows with
// the 128-byte swizzle; false if the driver refuses it.
bool make_bf16_rows_map(CUtensorMap *m, const void *ptr, int rows, int K, int box_rows);

// Per row b < rows: optionally x[b] = E[tokens[b]] (the token joins stream b's emitted
// set), then hi/lo bf16 parts of gamma * x[b] / sqrt(mean(x[b]^2) + eps).
struct NormSplitArgs {
    float *x;                      // [rows][K]
    int K;
    const float *gamma;
    float eps;
    __nv_bfloat16 *hi, *lo;        // [rows][K]
    const void *table;             // embedding table (bf16) or null: no gather
    int table_rows;
    const int32_t *tokens;         // [rows]
    uint32_t *emitted;             // [rows][emitted_words]
    int emitted_words, vocab;
    float *y;                      // optional fp32 copy of the normalised rows
    int *status;
};
cudaError_t launch_norm_split(const NormSplitArgs &a, int rows, cudaStream_t s, bool pdl = false);

// Sampling settings of a batch, in device memory (read by the step at run time, so a
// captured step graph serves every setting): top_k 0 = greedy argmax.
struct BatchSampling {
    int top_k;
    float temperature, top_p;
    uint32_t seed_lo, seed_hi;
    int pad[3];
};
constexpr int kBatchSampleVocabMax = 32768;   // logits a stream's selection keeps in shared memory

// Per stream b: penalty over its emitted set, EOS mask, then the argmax (lowest index on
// ties) of logits[b], or (sampling on) a draw among its top-k (stream b draws u at its
// own counter from seed + b); ids and the next input token go through the control
// block; the stream's position advances.
struct BatchArgmaxArgs {
    const float *logits;           // [B][V]
    int V;
    const uint32_t *emitted;       // [B][words]
    int words;
    float penalty;
    int eos;
    BatchCtl *ctl;
    int32_t *tokens;               // [B] next input tokens
    int *pos;                      // [B]
    int *status;
    const BatchSampling *samp;
    int *drawn;                    // [B] ids each stream has drawn since it was set
};
cudaError_t launch_batch_argmax(const BatchArgmaxArgs &a, int B, cudaStream_t s, bool pdl = false);

// ---------------------------------------------------------------------------------
// Batched prefill: ns streams x n prompt positions, T = ns * n tokens per contraction.
// ---------------------------------------------------------------------------------
struct PrefillQkArgs {
    const float *qkv;              // [T][qkv_ld] raw projections, token t = stream i * n + position j
    int qkv_ld, n, qh, kvh;
    const float *q_gamma, *k_gamma;// [hd] or null
    float eps;
    const float *rope_cos, *rope_sin;
    int rope_rows;                 // rows of the tables
    int mrope_h;                   // interleaved multimodal RoPE: the h (= w) section size, 0: plain
    const int *rope_pos;           // [3][rope_stride] rotary positions of the prompt (t, h, w), null: position j
    int rope_stride;
    void *kv;                      // batch caches [B][n_layers][2][kvh][S][hd] bf16
    size_t stream_elems, layer_elems;
    int S;
    const int *streams;            // [ns] cache index of each prompt stream
    __nv_bfloat16 *q_hi, *q_lo;    // [ns][qh][n][hd]: normalised, rotated q as bf16 parts
    int ns_tail;                   // set by launch_prefill_qk: CTAs that zero the prompt's K/V tail
};
cudaError_t launch_prefill_qk(int hd, int ns, const PrefillQkArgs &a, cudaStream_t s);

struct PrefillAttnArgs {
    const __nv_bfloat16 *q_hi, *q_lo;  // [ns][qh][n][hd]
    const void *kv;
    size_t stream_elems, layer_elems;
    int S, n, qh, kvh;
    float scale;
    const int *streams;
    __nv_bfloat16 *out_hi, *out_lo;    // [ns * n][qh * hd]
    int *status;
    int cache_streams;                 // streams of the cache buffer kv (its planes: cache_streams x stream_elems)
};
// The same attention on the tcgen05 tensor cores (head_dim 64 or 128, any group size),
// with the TMA maps of one prefill call (q parts and the caches: the same for every
// layer) made once by make_prefill_attn_maps.
struct PrefillAttnMaps {
    CUtensorMap qh, ql, kv;
};
bool make_prefill_attn_maps(int hd, int ns, const PrefillAttnArgs &a, PrefillAttnMaps *m);
cudaError_t launch_prefill_attention_tc(int hd, int ns, const PrefillAttnArgs &a, const PrefillAttnMaps &m,
                                        cudaStream_t s);

// ns rows of x [T][K] at rows (i * n + n - 1): the last position of each prompt stream.
cudaError_t launch_gather_last(const float *x, int n, int K, int ns, float *out, cudaStream_t s);

struct PrefillFinishArgs {
    const float *logits;           // [ns][V]
    int V, eos;
    const int *streams;            // [ns]
    int n;
    int32_t *first_ids;            // [ns]
    float *logits_out;             // [B][V]: each prompt stream's raw logits, in its row
    int32_t *tokens;               // [B] next input token of each stream
    int *pos;                      // [B]
    int *status;
};
cudaError_t launch_prefill_finish(const PrefillFinishArgs &a, int ns, cudaStream_t s);
// After a single-stream prefill's layers ran through the batched kernels: the model's
// position becomes `pos` and the batch's error bits join the model's.
cudaError_t launch_prefill_commit(DevState *st, int pos, const int *batch_status, cudaStream_t s);
// x[i] = E[tokens[i]] (bf16 table [rows, hidden] -> fp32 [n, hidden]); ids were checked
// against the table on the host.
cudaError_t launch_embed_rows(const void *table, const int32_t *tokens, int n, int hidden, float *x, cudaStream_t s);

}  // namespace qd

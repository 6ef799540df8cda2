/*
 * CPU oracle for the per-token autoregressive decode step of a Qwen3-style
 * decoder over a static-shape, bucket-grown KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the GPU path; the two meet only in the seeded
 * inputs drawn by the `workloads` module.
 *
 * Precision: fp32 storage and arithmetic; every RMSNorm mean-square and every
 * softmax (max, exp-sum, weighted V sum) accumulates in fp64.  Dot products
 * accumulate in fp32 in index order (or fp64 when `acc64` is set, a check on
 * the oracle itself).  The KV cache stores entries in the path's KV type:
 * bfloat16 (round-to-nearest-even) on the bf16 path, fp32 otherwise.
 *
 * Parity pins: see the tests; functions without a pin say so in oracle.c.
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ESTATE (-2)
#define ORC_EKVFULL (-3)
#define ORC_ENOMEM (-4)

#define ORC_MAX_BUCKETS 8
#define ORC_MAX_HEADS 16

typedef struct {
    int hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab, embed_rows;
    int w_bf16;      /* weights are bfloat16 bit patterns (uint16), else float32 */
    int kv_bf16;     /* KV cache entries are rounded to bfloat16 */
    int qk_norm;     /* per-head RMSNorm of q and k over head_dim */
    int n_heads_out; /* number of output heads (1, or 15 for the Code Predictor) */
    int eos_mask_id; /* logit forced to -inf before the argmax; -1: none */
    int n_buckets;
    int buckets[ORC_MAX_BUCKETS]; /* ascending Smax ladder */
    int acc64;       /* accumulate dot products in fp64 */
    int mrope_section[3]; /* frequencies per position stream (t, h, w), interleaved;
                             all 0: plain RoPE (one stream) */
    double rms_eps, rope_theta, rep_penalty;
} orc_config;

/* Weight pointer table, host memory, in this order:
 *   [0] embed [embed_rows, hidden] (may be NULL when embed_rows == 0)
 *   [1] final_norm [hidden]
 *   [2 .. 2+n_heads_out) lm_head[j] [vocab, hidden]
 *   then per layer l, 11 entries: attn_norm, wq, wk, wv, q_norm, k_norm, wo,
 *   mlp_norm, wg, wu, wd (q_norm/k_norm may be NULL when qk_norm == 0).
 * Matrices are row-major [out, in].  The oracle borrows them. */
#define ORC_LAYER_SLOTS 11

typedef struct orc_model orc_model;

orc_model *orc_create(const orc_config *cfg, const void *const *weights, int *status);
void orc_destroy(orc_model *m);
int orc_reset(orc_model *m);
int orc_pos(const orc_model *m);
int orc_smax(const orc_model *m);

/* One decoder position.  Input: embed (fp32 [hidden]) or, when embed is NULL,
 * row `token` of the embedding table.  token >= 0 with add_emitted != 0 adds the
 * id to the emitted set first.  want_head != 0 runs the final norm, head
 * `head_idx`, the repetition penalty, the EOS mask and the argmax. */
int orc_forward(orc_model *m, const float *embed, int token, int add_emitted, int want_head,
                int head_idx, int *out_id, float *logits_raw, float *hidden_taps, double *margin);

/* Prefill n positions from pos 0 (tokens or embeds [n, hidden]); head on the last. */
int orc_prefill(orc_model *m, const int32_t *tokens, const float *embeds, int n, int head_idx,
                int *first_id, float *logits_raw, double *margin);

/* The same prefill with explicit rotary positions: positions[s * n + i] is the
 * position of prompt position i in stream s (t, h, w).  The decode steps after it
 * continue at the largest of them + 1, equal in the three streams. */
int orc_prefill_positions(orc_model *m, const int32_t *tokens, const float *embeds, int n, int head_idx,
                          const int32_t *positions, int *first_id, float *logits_raw, double *margin);

int orc_get_hidden(const orc_model *m, float *out);        /* final-norm output, last position */
int orc_get_kv(const orc_model *m, int layer, int which, float *out); /* [kvh, pos, hd] */
int orc_emitted_words(const orc_model *m, uint32_t *out);  /* bitmask copy */

/* Logits at the last of n positions by full causal recompute (no cache). */
int orc_recompute_logits(const orc_config *cfg, const void *const *weights, const int32_t *tokens,
                         const float *embeds, int n, int head_idx, float *logits_raw);

/* Two-level frame generation: the next Talker input of a frame,
 * out = ((E_0[ids_0] + E_1[ids_1]) + ... + E_{n-1}[ids_{n-1}]) + text in fp32.
 * tables[j] [rows[j], hidden] (bfloat16 bits when bf16, else float32). */
int orc_frame_sum(const void *const *tables, const int *rows, const int32_t *ids, int n_tables, int hidden,
                  int bf16, const float *text, float *out);

/* Start from a given cache: kv [n_layers][2][n_kv_heads][L][head_dim] in the cache
 * type (bf16 bits when kv_bf16), position L, empty emitted set. */
int orc_set_kv(orc_model *m, const void *kv, int L);

/* Batched linear: out[t][r] = sum_k W[r][k] x[t][k], x [T, K], out [T, R]. */
int orc_linear(const void *W, int w_bf16, int R, int K, const float *x, int T, float *out);

/* Primitives the model is built from, exposed for the pins. */
void orc_rmsnorm(const float *x, const float *gamma, int n, double eps, float *out);
void orc_rope(float *v, int head_dim, int pos, double theta);
void orc_rope_mrope(float *v, int head_dim, const int pos3[3], const int section[3], double theta);
int orc_mrope_stream(int m, const int section[3]);
void orc_attend(const float *q, const float *K, const float *V, int L, int head_dim, float *out);
int orc_penalty_argmax(float *logits, int n, const uint32_t *emitted, float penalty, int eos_id,
                       double *margin);
float orc_silu_mul(float g, float u);

/* Sampling instead of the greedy argmax (after the penalty and the EOS mask):
 * top_k candidates (largest logits, ties to the lower index; 1 = greedy), weights
 * exp((l - l_max) / temperature), the smallest prefix of them whose sum reaches
 * top_p of the total, and a draw u in [0, 1) of the counter-based generator
 * orc_uniform(seed, counter) where counter = ids generated so far.  top_k 0 turns
 * sampling off.  Errors: ORC_EINVAL (top_k > ORC_MAX_TOPK, temperature <= 0,
 * top_p outside (0, 1]). */
#define ORC_MAX_TOPK 64
int orc_set_sampling(orc_model *m, int top_k, double temperature, double top_p, uint64_t seed);
/* SplitMix64 output for state seed + (counter + 1) * 0x9E3779B97F4A7C15, and its top
 * 53 bits as a double in [0, 1). */
uint64_t orc_splitmix64(uint64_t seed, uint64_t counter);
double orc_uniform(uint64_t seed, uint64_t counter);
/* The sampler on final logits (penalty and mask applied): the chosen index and, in
 * *margin, how far the decision is from changing: the smallest of the distance of
 * u * (kept sum) from the cumulative-weight boundaries (relative to the kept sum), of
 * the top-p cut from its neighbouring prefix sums (relative to the total, when top_p
 * < 1), of the picked logit from its neighbours in the order, and, when the pick is
 * the last of the top_k, of that logit from the best excluded one. */
int orc_sample(const float *logits, int n, int top_k, double temperature, double top_p, double u,
               double *margin);
uint16_t orc_round_bf16(float f);

/* Weight-only 8-bit block quantisation (the talker's Q8_0 weights, "audio.cpp Rockchip
 * NPU build notes"): each row of W [rows, K] in blocks of 32 along K; per block the
 * scale d = max|w| / 127 (fp32), the codes round(w / d) (half away from zero, fp32
 * division; 0 for an all-zero block), d stored as IEEE half.  K % 32 == 0. */
uint16_t orc_f32_to_f16(float f);   /* round to nearest even */
float orc_f16_to_f32(uint16_t h);
int orc_quantize_q8(const float *w, int rows, int K, int8_t *codes, uint16_t *scales);
/* y[r] = sum_k (codes[r][k] * half(scales[r][k / 32])) * x[k], fp32 products summed in
 * fp64 in index order, rounded to fp32. */
int orc_gemv_q8(const int8_t *codes, const uint16_t *scales, int rows, int K, const float *x, float *y);
/* Q4_K super-blocks of 256 weights (144 bytes each, [rows][K/256]): see oracle.c. */
int orc_quantize_q4k(const float *w, int rows, int K, uint8_t *blocks);
int orc_gemv_q4k(const uint8_t *blocks, int rows, int K, const float *x, float *y);

/* Codec decoder convolution stages ("qwen3-tts-hip OPTIMIZATION_LOG", codec-profile and
 * transposed-convolution entries; the codec's SEANet upsampler in "Qwen3-TTS ncnn
 * port").  Channel-major signals x [Cin][T], y [Cout][...]; fp32 products summed in
 * fp64, rounded to fp32; bias may be NULL.
 *
 * Causal dilated convolution: y[o][t] = b[o] + sum_i sum_k W[o][i][k] x[i][t - (K-1-k) d],
 * x = 0 before t = 0; W [Cout][Cin][K]; y [Cout][T]. */
int orc_conv1d_causal(const float *x, int Cin, int T, const float *W, const float *bias, int Cout, int K, int dil,
                      float *y);
/* Causal transposed convolution with kernel 2 * stride: every input frame t spreads
 * into outputs t*stride + k, k < 2*stride, through W [Cin][Cout][2*stride]; the first
 * T*stride outputs are kept (y [Cout][T*stride]). */
int orc_conv_transpose1d_causal(const float *x, int Cin, int T, const float *W, const float *bias, int Cout,
                                int stride, float *y);
int orc_num_threads(void);
void orc_set_threads(int n);

#endif

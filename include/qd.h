/*
 * qd -- per-token autoregressive decode step of a Qwen3-style decoder over a
 * static-shape, bucket-grown KV cache, on one GB300 (sm_103a).
 *
 * The operation (sources by page title and section):
 *  - "Qwen3-TTS ncnn port: pure C++/ncnn end-to-end reproduction", section
 *    "Talker: non-standard structure and two-level generation": a 28-layer
 *    Qwen3-style stack with RMSNorm over head_dim on q and k after their
 *    projections (QK-norm), 8 kv heads broadcast to 16 q heads (GQA), rotary
 *    embedding that reduces to plain RoPE, a repetition penalty of 1.05 on ids
 *    already emitted, greedy decoding; section "Integration and performance
 *    optimisation": a KV cache computes only the new token's q/k/v and attends
 *    over the cache.
 *  - "Audio8-ASR: dynamic KV-cache buckets and multi-length end-to-end
 *    acceptance", section "Implemented dynamic window mechanism": the cache is
 *    a rank-3 [kv_heads, Smax, head_dim] buffer per layer written in place;
 *    a sequence starts at the smallest usable Smax; when the write position
 *    reaches Smax the valid K/V region of every layer is copied into a larger
 *    buffer and decoding continues from the same token and RoPE position; the
 *    host keeps the cache, the embedding lookup and the argmax.
 *  - "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile entry: the step is
 *    input_norm, qkv_gemm, qk_layout_cache, attention, output_gemm_residual,
 *    post_norm, gate_up_gemm, swiglu, down_gemm_residual, then the logits and
 *    the token.
 *
 * Per position p (0-based) and layer: x^ = RMSNorm(x); q,k,v = W x^; per-head
 * RMSNorm of q and k (if qk_norm); RoPE at p; K/V row p appended to the cache;
 * GQA attention of every q head over positions [0, p]; x += Wo o;
 * x^ = RMSNorm(x); x += Wd (silu(Wg x^) * (Wu x^)).  After the last layer:
 * y = RMSNorm(x); logits = Whead y; repetition penalty over the emitted ids;
 * EOS mask; argmax (lowest index on ties).
 *
 * Conventions for every entry point:
 *  - Every call validates its arguments before touching the device and returns
 *    a qd_status.  On any error the handle's state is unchanged and it stays
 *    usable; qd_last_error() gives the reason (with the CUDA runtime/driver
 *    versions).  No call falls back to the CPU.
 *  - "device" pointers are CUDA device memory of the handle's device; "host"
 *    pointers are ordinary host memory.  Floating-point activations and
 *    embeddings are fp32; weights are fp32 or bf16 as the config says.
 *  - Work is ordered after prior work on the caller's stream (given at
 *    qd_create) and later work on that stream is ordered after it.  Calls that
 *    return a host value synchronise; *_async calls do not.
 *  - A handle is used by one host thread at a time.
 */
#ifndef QD_H
#define QD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qd_model *qd_handle;

typedef enum {
    QD_OK = 0,
    QD_EINVAL = -1,        /* bad argument or configuration */
    QD_ESTATE = -2,        /* call not valid in the current state (e.g. decode before prefill) */
    QD_EKVFULL = -3,       /* the position would exceed the last bucket of the ladder */
    QD_ENOMEM = -4,        /* device allocation failed */
    QD_ECUDA = -5,         /* a CUDA runtime call failed */
    QD_EUNSUPPORTED = -6,  /* shape outside what the kernels implement */
    QD_EDEVICE = -7        /* a kernel reported an error (bounded wait expired, bad index) */
} qd_status;

enum { QD_F32 = 0, QD_BF16 = 1 };
#define QD_MAX_BUCKETS 8
#define QD_MAX_HEADS 16

/* Model configuration (plain data).  hidden, n_q_heads*head_dim and ffn must be
 * multiples of 256 and at most 8192; head_dim is 64 or 128; n_q_heads is a
 * multiple of n_kv_heads; bucket sizes ascend and are multiples of 32. */
typedef struct {
    int hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn;
    int vocab;       /* rows of every output head */
    int embed_rows;  /* rows of the input embedding table (0: inputs are embeddings only) */
    int dtype;       /* QD_F32 or QD_BF16: weights and KV cache entries */
    int qk_norm;     /* 1: per-head RMSNorm of q and k over head_dim */
    int n_heads_out; /* output heads (1, or 15 for a code predictor) */
    int eos_mask_id; /* logit forced to -inf before the argmax; -1: none */
    int n_buckets;
    int buckets[QD_MAX_BUCKETS]; /* ascending Smax ladder, e.g. 128, 256, 512 */
    double rms_eps;     /* e.g. 1e-6 */
    double rope_theta;  /* e.g. 1e6 */
    double rep_penalty; /* 1.0 = off */
    /* Interleaved multimodal RoPE ("Qwen3-TTS ncnn port", Talker section): the
     * head_dim/2 rotation frequencies are dealt to three position streams t, h, w
     * in turn, each while its section has room, the rest to t ([24, 20, 20] for
     * head_dim 128: frequency m < 60 takes stream m % 3, the last four take t).
     * All 0: plain RoPE.  Otherwise t >= h == w > 0 and t + h + w == head_dim/2.
     * The streams differ only for prompt positions given to qd_prefill_mrope. */
    int mrope_section[3];
    /* Weight-only 8-bit matrices ("audio.cpp Rockchip NPU build notes": the talker's
     * Q8_0 weights): 1 quantises every layer matrix and output head at qd_create into
     * rows of K int8 codes and K/32 IEEE-half block scales (d = max|w| / 127 per 32
     * weights along K, code = round(w / d) half away from zero, d rounded to a half;
     * qd_quantize_q8's arithmetic); the step multiplies each code by its block's
     * stored scale.  The embedding table, norms and KV cache keep dtype.  Only the
     * persistent decode step runs such a model (bf16 ASR and Talker shapes):
     * QD_EUNSUPPORTED otherwise, for the batched API, and for qd_time_kernel's GEMV
     * kernels (which 0-3, 5).  Prompts run one step per position.  0: off. */
    int weight_q8;
} qd_config;

/* Per-layer weights: device pointers, row-major [out, in], in the config's
 * dtype.  attn_norm/mlp_norm [hidden]; q_norm/k_norm [head_dim] (NULL when
 * qk_norm == 0); wq [n_q_heads*head_dim, hidden]; wk, wv [n_kv_heads*head_dim,
 * hidden]; wo [hidden, n_q_heads*head_dim]; wg, wu [ffn, hidden]; wd [hidden, ffn]. */
typedef struct {
    const void *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo, *mlp_norm, *wg, *wu, *wd;
} qd_layer_weights;

typedef struct {
    const void *embed;                  /* device [embed_rows, hidden] or NULL */
    const void *final_norm;             /* device [hidden] */
    const void *lm_head[QD_MAX_HEADS];  /* device [vocab, hidden], n_heads_out of them */
    const qd_layer_weights *layers;     /* HOST array of n_layers entries */
} qd_weights;

/* qd_create -- validate cfg, copy the weights into a library-owned layout
 * (fused [wq;wk;wv], row-interleaved [wg,wu], fp32 norm gammas), allocate the
 * first KV bucket, the step scratch and the emitted-id bitmask, and build the
 * RoPE table.  The caller's weight buffers are only read during this call and
 * may be freed after it returns.  cuda_stream: the caller's cudaStream_t (may
 * be the default stream).  Errors: QD_EINVAL (bad cfg or non-device pointer),
 * QD_EUNSUPPORTED, QD_ENOMEM, QD_ECUDA; *out is NULL then. */
qd_status qd_create(const qd_weights *weights, const qd_config *cfg, void *cuda_stream, qd_handle *out);

/* qd_destroy -- synchronise, free every device resource. NULL is a no-op. */
qd_status qd_destroy(qd_handle h);

/* qd_reset -- position 0, emitted set cleared, back to the smallest bucket
 * (the larger buckets' buffers are kept for reuse). Asynchronous. */
qd_status qd_reset(qd_handle h);

/* qd_prefill -- feed n prompt positions from position 0 and return the first
 * generated id (head 0 for a single-head model, head `head_idx` otherwise).
 * Exactly one of tokens (HOST int32 [n], ids < embed_rows) or embeds (DEVICE
 * fp32 [n, hidden], row-major) is non-NULL.  Prompt ids do not join the emitted
 * set.  The first bucket is the smallest Smax >= n.  On a bf16 model with one head
 * and an embedding table the prompt runs all positions at once through the batched
 * prefill kernels (tensor-core GEMMs, causal flash attention; an internal one-stream
 * qd_batch holds the scratch and is freed with the model), unless debug taps are set;
 * the other models run it position by position through the decode step.  Synchronises; first_id is a HOST pointer.  Errors: QD_EINVAL
 * (n < 1, both/neither inputs, bad id), QD_ESTATE (position != 0: call qd_reset
 * first), QD_EKVFULL (n > last bucket), QD_ECUDA, QD_EDEVICE. */
qd_status qd_prefill(qd_handle h, const int32_t *tokens, const void *embeds, int n, int head_idx,
                     int32_t *first_id);

/* qd_prefill_mrope -- qd_prefill with explicit rotary positions: positions is a
 * HOST int32 array [3][n], positions[s * n + i] the position of prompt position i
 * in stream s (t, h, w; see qd_config.mrope_section -- a plain-RoPE model reads
 * stream t only).  Every position lies in [0, last bucket).  The cache rows are
 * still 0..n-1; the decode steps that follow rotate at the prompt's largest
 * position + 1 (then + 2, ...) in all three streams, and qd_reset returns to the
 * plain positions.  Errors: as qd_prefill, and QD_EINVAL for a NULL positions
 * array or a position outside [0, last bucket); a decode step whose rotary
 * position would reach the last bucket returns QD_EKVFULL. */
qd_status qd_prefill_mrope(qd_handle h, const int32_t *tokens, const void *embeds, int n, int head_idx,
                           const int32_t *positions, int32_t *first_id);

/* qd_decode_step -- one position.  Input: embed (DEVICE fp32 [hidden]) if non-NULL,
 * else row `token` of the embedding table.  token >= 0 marks the id that entered
 * the sequence: it joins the emitted set (the repetition penalty's memory) in
 * both cases.  Grows the cache to the next bucket first when the position has
 * reached Smax.  Writes the argmax of head `head_idx` to *out_id (HOST) and
 * synchronises.  Errors: QD_ESTATE (before prefill), QD_EKVFULL, QD_EINVAL. */
qd_status qd_decode_step(qd_handle h, const void *embed, int32_t token, int head_idx, int32_t *out_id);

/* qd_decode_step_async -- as qd_decode_step but token_dev (DEVICE int32, may be
 * NULL for "no token") is read on the device and the id is written to out_id_dev
 * (DEVICE int32, may be NULL); no host synchronisation.  Device-side errors are
 * reported by the next synchronising call. */
qd_status qd_decode_step_async(qd_handle h, const void *embed, const int32_t *token_dev, int head_idx,
                               int32_t *out_id_dev);

/* qd_decode_greedy -- n_steps positions of the greedy loop kept on the device:
 * each step's input is the previous step's argmax (embedded and added to the
 * emitted set), as in a decoder that feeds its own argmax back.  The first
 * step's token is first_token if >= 0, else the last id produced.  Bucket
 * growth happens between steps as needed.  ids_dev: DEVICE int32 [n_steps]
 * receives the ids in order.  Asynchronous.  Errors: QD_ESTATE, QD_EKVFULL
 * (pos + n_steps beyond the last bucket, checked before any work). */
qd_status qd_decode_greedy(qd_handle h, int n_steps, int32_t first_token, int32_t *ids_dev);

/* qd_grow_kv -- migrate now to bucket new_smax (a ladder entry larger than the
 * current Smax): copy the valid [0, pos) region of every layer's K and V into
 * that bucket's buffer.  Decoding also grows on its own when it needs to. */
qd_status qd_grow_kv(qd_handle h, int new_smax);

/* ---- inspection and test taps (not on the hot path) ---- */

/* Final-norm output y [hidden] (fp32) of the last position that ran a head. */
qd_status qd_get_hidden(qd_handle h, float *out_dev);

/* When either pointer is non-NULL, following steps run without CUDA graphs and
 * write x after the embedding and after every layer (fp32 [n_layers+1, hidden])
 * and the raw logits before penalty/mask (fp32 [vocab]).  NULL, NULL restores
 * the graph path.  Both are DEVICE pointers owned by the caller. */
qd_status qd_set_debug_taps(qd_handle h, float *hidden_taps_dev, float *logits_dev);

/* Turn CUDA-graph replay on (default) or off; results are identical. */
qd_status qd_set_graphs(qd_handle h, int enable);

/* qd_set_sampling -- draw the heads' ids instead of taking the greedy argmax, after the
 * repetition penalty and the EOS mask (the pages' sampling settings: "qwen3-tts-hip
 * OPTIMIZATION_LOG", sampling entries -- top_k 50, top_p 1.0, temperature 0.9,
 * seeded): the top_k largest logits (ties to the lower id), weights
 * exp((l - l_max) / temperature), the smallest prefix of them whose weight reaches
 * top_p of their sum, then the first candidate whose running weight exceeds u times
 * the kept weight, u in [0, 1) being draw n of the counter-based SplitMix64 sequence
 * of `seed` (n = ids produced since the last reset).  top_k 0 restores the greedy
 * argmax (top_k 1 gives the same ids).  The settings hold for every later step and
 * survive qd_reset; the batched qd_batch_* path stays greedy.  Asynchronous, ordered
 * with the model's steps; no graph is recaptured.  Errors: QD_EINVAL (top_k outside
 * [0, 64], temperature not > 0, top_p outside (0, 1]), QD_EUNSUPPORTED (top_k too
 * large for this model's head layout). */
qd_status qd_set_sampling(qd_handle h, int top_k, float temperature, float top_p, uint64_t seed);

/* qd_quantize_q8 -- weight-only 8-bit block quantisation of W (DEVICE [rows, K],
 * row-major, fp32 or bf16 per dtype): per row, blocks of 32 weights along K, each with
 * the scale d = max|w| / 127 (fp32 division) stored as an IEEE half in scales (DEVICE
 * uint16 [rows, K/32]) and the codes round(w / d) (fp32 division, half away from
 * zero; 0 for an all-zero block) in codes (DEVICE int8 [rows, K]) -- the talker's
 * Q8_0 weights of "audio.cpp Rockchip NPU build notes" ("The talker is the only
 * DRAM-bound candidate, and it is not at the ceiling").  K a multiple of 32.  Runs on
 * cuda_stream and synchronises it.  Errors: QD_EINVAL (shape, dtype, a non-device
 * pointer), QD_ECUDA. */
qd_status qd_quantize_q8(const void *w_dev, int dtype, int rows, int K, int8_t *codes_dev, uint16_t *scales_dev,
                         void *cuda_stream);

/* qd_gemv_q8 -- y[r] = sum_k codes[r][k] * d[r][k/32] * x[k] for the layout of
 * qd_quantize_q8 (codes DEVICE int8 [rows, K], 16-byte aligned; scales DEVICE half
 * bits [rows, K/32]; x DEVICE fp32 [K], 16-byte aligned; y DEVICE fp32 [rows]): 1 +
 * 1/16 bytes per weight streamed once.  K is 512, 1024 or 2048.  Asynchronous: the kernel
 * is enqueued on cuda_stream; when avg_ms (HOST) is non-NULL it is then launched
 * `reps` more times between CUDA events, synchronised, and the mean duration of those
 * launches is written there.
 * Errors: QD_EINVAL (arguments, alignment), QD_EUNSUPPORTED (K), QD_ECUDA. */
qd_status qd_gemv_q8(const int8_t *codes_dev, const uint16_t *scales_dev, const float *x_dev, float *y_dev, int rows,
                     int K, void *cuda_stream, int reps, float *avg_ms);

/* qd_quantize_q4k -- Q4_K super-block quantisation of W (DEVICE [rows, K], row-major,
 * fp32 or bf16 per dtype; K a multiple of 256), the talker's 4.5-bit format of "audio.cpp
 * Rockchip NPU build notes" ("The talker is the only DRAM-bound candidate, and it is not
 * at the ceiling": 251 MB per token against 471 MB as Q8_0).  Per row, super-blocks of
 * 256 weights along K, 144 bytes each in blocks_dev (DEVICE uint8 [rows][K/256][144],
 * 16-byte aligned): bytes 0-1 the half scale d, 2-3 the half min dm, 4-9 the 8
 * sub-blocks' 6-bit scales sc_j and 10-15 their 6-bit mins m_j (each a 48-bit
 * little-endian word, field j at bit 6 j), 16-143 the 4-bit codes q (byte i: weight 2i in
 * the low nibble, 2i + 1 in the high one); weight = d sc_j q - dm m_j.  Quantiser, in fp32
 * with IEEE division and half-away rounding: per 32-weight sub-block mn_j = -min(0, min
 * w), s_j = (max w + mn_j) / 15; d = half(max s_j / 63), dm = half(max mn_j / 63); sc_j =
 * clamp(round(s_j / d), 0, 63), m_j = clamp(round(mn_j / dm), 0, 63), q = clamp(round((w +
 * dm m_j) / (d sc_j)), 0, 15) (0 where a divisor is 0).  Runs on cuda_stream and
 * synchronises it.  Errors: QD_EINVAL (shape, dtype, alignment, a non-device pointer),
 * QD_ECUDA. */
qd_status qd_quantize_q4k(const void *w_dev, int dtype, int rows, int K, uint8_t *blocks_dev, void *cuda_stream);

/* qd_gemv_q4k -- y[r] = sum_k (d sc_j q - dm m_j)[r][k] * x[k] for the layout of
 * qd_quantize_q4k (blocks DEVICE, 16-byte aligned; x DEVICE fp32 [K], 16-byte aligned;
 * y DEVICE fp32 [rows]): 0.5625 bytes per weight streamed once.  K is 512, 1024 or
 * 2048.  Asynchronous on cuda_stream; with avg_ms (HOST) non-NULL the kernel is then
 * launched `reps` more times between CUDA events, synchronised, and their mean
 * duration written there.  Errors: QD_EINVAL (arguments, alignment), QD_EUNSUPPORTED
 * (K), QD_ECUDA. */
qd_status qd_gemv_q4k(const uint8_t *blocks_dev, const float *x_dev, float *y_dev, int rows, int K, void *cuda_stream,
                      int reps, float *avg_ms);

/* qd_conv1d_causal -- the codec decoder's causal dilated convolution ("qwen3-tts-hip
 * OPTIMIZATION_LOG", codec entries): y[o][t] = bias[o] + sum_i sum_k W[o][i][k] *
 * x[i][t - (K-1-k) * dilation], zero history.  x DEVICE fp32 [Cin][T], W DEVICE fp32
 * [Cout][Cin][K], bias DEVICE fp32 [Cout] or NULL, y DEVICE fp32 [Cout][T].  K <= 16,
 * (K-1) * dilation <= 512.  Asynchronous on cuda_stream.  Errors: QD_EINVAL,
 * QD_EUNSUPPORTED (history span), QD_ECUDA. */
qd_status qd_conv1d_causal(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev, int Cout,
                           int K, int dilation, float *y_dev, void *cuda_stream);

/* qd_conv_transpose1d_causal -- the codec decoder's transposed convolution with kernel
 * length 2 * stride ("qwen3-tts-hip OPTIMIZATION_LOG", transposed-convolution
 * entries), evaluated per output phase: sample t * stride + p (t < T, p < stride) of
 * output channel o is bias[o] plus, over input channels i, tap p of W[i][o] times
 * x[i][t] and tap p + stride of W[i][o] times x[i][t - 1] (x[i][-1] = 0).
 * x DEVICE fp32 [Cin][T], W DEVICE fp32 [Cin][Cout][2 * stride], bias DEVICE fp32 [Cout]
 * or NULL, y DEVICE fp32 [Cout][T * stride].  stride <= 64.  Asynchronous on
 * cuda_stream.  Errors: QD_EINVAL, QD_ECUDA. */
qd_status qd_conv_transpose1d_causal(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev,
                                     int Cout, int stride, float *y_dev, void *cuda_stream);

/* qd_conv1d_causal_tc -- qd_conv1d_causal's convolution on the tensor cores: the GEMM
 * of qd_gemm_bf16 over the time-major signal with one weight slab per tap, tap k
 * reading the frames shifted by (K-1-k) * dilation ("qwen3-tts-hip OPTIMIZATION_LOG",
 * codec entries).  Same arguments and layouts as qd_conv1d_causal (x DEVICE fp32
 * [Cin][T], W DEVICE fp32 [Cout][Cin][K], bias DEVICE fp32 [Cout] or NULL, y DEVICE
 * fp32 [Cout][T]); the weights are rounded to bf16 (round to nearest even) and x is
 * carried as bf16 hi + lo parts (16 significant bits), fp32 accumulation.  Any Cin,
 * Cout (padded internally to 64 / 128), K <= 64.  Allocates its scratch (about
 * 2 K Cout Cin + 4 T Cin bytes), runs on cuda_stream and synchronises it.  When avg_ms
 * (HOST) is non-NULL the whole convolution (weight packing, signal transpose, GEMM) is
 * then run `reps` more times between CUDA events and its mean duration written there.
 * Errors: QD_EINVAL, QD_EUNSUPPORTED, QD_ENOMEM, QD_ECUDA, QD_EDEVICE (a bounded wait
 * expired). */
qd_status qd_conv1d_causal_tc(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev, int Cout,
                              int K, int dilation, float *y_dev, void *cuda_stream, int reps, float *avg_ms);

/* qd_conv_transpose1d_causal_tc -- qd_conv_transpose1d_causal's convolution on the
 * tensor cores in the page's per-phase form ("qwen3-tts-hip OPTIMIZATION_LOG",
 * transposed-convolution entry): for each phase p < stride one GEMM with two taps,
 * slab p of the weights on frame t and slab p + stride on frame t - 1, written to
 * samples t * stride + p.  Same arguments and layouts as qd_conv_transpose1d_causal
 * (W DEVICE fp32 [Cin][Cout][2 * stride]); precision, scratch, synchronisation, timing
 * and errors as qd_conv1d_causal_tc.  stride <= 64. */
qd_status qd_conv_transpose1d_causal_tc(const float *x_dev, int Cin, int T, const float *w_dev,
                                        const float *bias_dev, int Cout, int stride, float *y_dev, void *cuda_stream,
                                        int reps, float *avg_ms);

/* qd_gemm_bf16 -- the batched paths' tensor-core contraction on its own (a check
 * and measurement tap): out[t][r] = sum_k W[r][k] * x[t][k] for W (DEVICE bf16
 * [R, K] row-major, 16-byte aligned) and x (DEVICE fp32 [T, K] row-major), with x
 * split into bf16 hi + lo parts (x_lo = bf16(x - bf16(x))) so the products carry
 * ~16 bits of x; fp32 accumulation.  mode 0: out = the product (fp32 [T, R]);
 * 1: out += the product; 2: rows (2i, 2i+1) are (gate_i, up_i) and out (fp32
 * [T, R/2]) = silu(gate) * up.  R a multiple of 128, K of 64.  Allocates its
 * scratch, runs on cuda_stream and synchronises it.  When avg_ms (HOST) is non-NULL
 * the contraction kernel is then launched `reps` more times between CUDA events and
 * its mean duration is written there (mode 1 accumulates into out each time).
 * Errors: QD_EINVAL, QD_EUNSUPPORTED (shape), QD_ENOMEM, QD_ECUDA, QD_EDEVICE (a
 * bounded wait expired). */
qd_status qd_gemm_bf16(const void *w_dev, const float *x_dev, float *out_dev, int R, int K, int T, int mode,
                       void *cuda_stream, int reps, float *avg_ms);

/* Copy the current cache buffer, layout [n_layers][2 (K,V)][n_kv_heads][Smax][head_dim]
 * in the KV dtype, into dst_dev (DEVICE, at least *bytes). Query the size by
 * passing dst_dev = NULL. Synchronises. */
qd_status qd_copy_kv(qd_handle h, void *dst_dev, size_t *bytes);

/* Copy the emitted-id bitmask (uint32 [ceil(vocab/32)], bit i of word i/32) to dst_dev. */
qd_status qd_get_emitted(qd_handle h, uint32_t *dst_dev);

/* Host-side view of the position (positions held) and the current Smax. */
qd_status qd_get_pos(qd_handle h, int *pos, int *smax);

/* Number of this library's kernels launched so far by the handle (graph
 * replays count each kernel node), and kernels per decode step. */
qd_status qd_get_launch_count(qd_handle h, long long *kernels, int *kernels_per_step);

/* Time `reps` back-to-back launches of one kernel of the decode step with the
 * arguments the step uses, between CUDA events on the library's stream;
 * which: 0 = output head (norm + GEMV + penalty + argmax), 1 = fused QKV GEMV
 * of layer 0, 2 = gate/up GEMV of layer 0, 3 = down GEMV of layer 0,
 * 4 = attention of layer 0, 5 = output projection of layer 0, 6 = one whole decode
 * step as the decode loop issues it (the persistent step kernel where the shape has
 * one), repeated `reps` times at the following positions (they must fit in the
 * current bucket).  The position, state, residual and emitted set are restored
 * afterwards.  Needs a prefilled handle. */
qd_status qd_time_kernel(qd_handle h, int which, int reps, float *avg_ms);

const char *qd_last_error(qd_handle h);
const char *qd_status_string(int status);

/* ---- two-level frame generation ----
 *
 * Sources: "Qwen3-TTS ncnn port", section "Talker: non-standard structure and
 * two-level generation" (per frame the Talker emits one primary code, a Code
 * Predictor emits 15 residual codes autoregressively from 15 output heads, and the
 * 16 code embeddings plus the text/pad embedding form the Talker's next input; the
 * predictor starts afresh every frame); "qwen3-tts-hip OPTIMIZATION_LOG", Code
 * Predictor sub-stages (a two-position predictor prefill, then one decode step per
 * further code).
 *
 * One frame, given the Talker's last id `p` and final-norm output h_T:
 *   1. reset the predictor; prefill it with [h_T, E_0[p]] and decode code_1 with
 *      head 0 (E_0 is the Talker's own embedding table);
 *   2. for j = 1..14: decode step with input E_j[code_j] and head j -> code_{j+1}
 *      (code_j joins the predictor's emitted set);
 *   3. next_in = E_0[p] + E_1[code_1] + ... + E_15[code_15] + text[f], in fp32 in
 *      that order;
 *   4. unless this is the call's last frame: a Talker decode step with input next_in
 *      and token p (p joins the Talker's emitted set) -> the next frame's primary.
 * Everything stays on the device; one CUDA graph per frame and Talker bucket. */
#define QD_FRAME_CODES 16

typedef struct qd_frame *qd_frame_handle;

/* qd_frame_create -- bind a Talker handle and a Code Predictor handle.  Talker: a
 * single-head model with an embedding table (E_0).  Predictor: same hidden size and
 * dtype, n_heads_out = 15, vocab <= code_rows, first bucket >= 16 positions.
 * code_tables: HOST array of 15 DEVICE pointers E_1..E_15, each [code_rows, hidden]
 * in `dtype` (which must be the models' dtype); they are copied into library-owned
 * memory, so the caller may free them after the call.  Both handles stay owned by
 * the caller; while the frame handle exists, use the three on one host thread.
 * Destroying either model first detaches the frame handle (it waits for the frame
 * work in flight); a detached frame handle accepts only qd_frame_destroy, and
 * qd_frame_generate returns QD_ESTATE.  Errors (described by qd_last_error of the
 * Talker): QD_EINVAL, QD_ENOMEM, QD_ECUDA. */
qd_status qd_frame_create(qd_handle talker, qd_handle predictor, const void *const *code_tables, int code_rows,
                          int dtype, qd_frame_handle *out);

/* qd_frame_destroy -- synchronise and free the frame handle (not the models). */
qd_status qd_frame_destroy(qd_frame_handle f);

/* qd_frame_generate -- run n_frames frames.  The first frame starts from the
 * Talker as it stands (after qd_prefill or any decode step that ran its head);
 * each later frame starts with the Talker step of the previous one, so the call
 * runs n_frames - 1 Talker steps and n_frames predictor loops (16 predictor
 * positions each).
 *   text_dev    DEVICE fp32 [n_frames, hidden]: text/pad embedding of each frame.
 *   force_dev   DEVICE int32 [n_frames, 16] or NULL: when given, these ids are fed
 *               back (embedded, summed, added to the emitted sets) instead of the
 *               argmaxes, which are still reported; for teacher-forced comparison.
 *   codes_dev   DEVICE int32 [n_frames, 16]: per frame the primary argmax, then the
 *               15 residual argmaxes.
 *   next_in_dev DEVICE fp32 [hidden] or NULL: the last frame's summed embedding
 *               (the input of the Talker step that would start the next frame).
 * Queued on the Talker's stream (ordered after both handles' prior work) without a
 * host synchronisation; device-side errors (an id outside its table) are reported
 * by the next synchronising call of either handle.  The Talker's cache grows along
 * its ladder between frames.  Errors: QD_EINVAL, QD_ESTATE (the Talker has produced
 * no id yet), QD_EKVFULL (the Talker steps would pass its last bucket; checked
 * before any work). */
qd_status qd_frame_generate(qd_frame_handle f, int n_frames, const float *text_dev, const int32_t *force_dev,
                            int32_t *codes_dev, float *next_in_dev);

/* Turn the per-frame CUDA graphs on (default) or off; results are identical. */
qd_status qd_frame_set_graphs(qd_frame_handle f, int enable);

/* ---- output head without allocation ----
 *
 * The pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory: a host application that owns all device memory through
 * its own pool and forbids other allocators (an audio engine or plugin host, for
 * example), or code on a real-time thread where an allocation's locking and implicit
 * synchronisation are not allowed.  Such a caller passes its own buffers for every
 * input and output, and the call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * qd_head_argmax_noalloc -- logits = W y (W [vocab, hidden] row-major in `dtype`,
 * y fp32 [hidden] already RMS-normalised), then the repetition penalty over the ids
 * set in emitted_dev (uint32 bitmask, may be NULL), the EOS mask (eos_mask_id, -1:
 * none) and the argmax (lowest index on ties), written to *out_id_dev (DEVICE
 * int32).  logits_dev (DEVICE fp32 [vocab], may be NULL) receives the raw logits.
 * All pointers are DEVICE pointers (a host pointer returns QD_EINVAL before any
 * work); work is queued on cuda_stream and the call returns without synchronising.
 * It gives the same logits and id as the output head of qd_decode_step for the same
 * y.  *out_id_dev == -1 after the work completes means the kernel gave up: a stage
 * of the weight stream did not arrive within its one-second bound, and no id was
 * produced.  Errors: QD_EINVAL (null or non-device pointer, vocab or hidden < 1,
 * eos_mask_id outside [-1, vocab), rep_penalty <= 0, unknown dtype).
 *
 * Its scratch (one argmax candidate per CTA and a completion counter, about 8 KB)
 * is a fixed array in the library's device memory, held by every device that loads
 * the library until the process exits.  Limits: hidden a multiple of 256 and at most
 * 8192, at most 1024 CTAs (one per SM is used); larger requests return
 * QD_EUNSUPPORTED.  The first call on a device looks up that array's device
 * address and configures the kernels; make that first call before any stream
 * capture.  Every call shares the array: calls whose work overlaps on the GPU (on
 * different streams, or from different host threads) race and must not be issued. */
qd_status qd_head_argmax_noalloc(const float *y_dev, const void *w_dev, int vocab, int hidden, int dtype,
                                 const uint32_t *emitted_dev, double rep_penalty, int eos_mask_id,
                                 int32_t *out_id_dev, float *logits_dev, void *cuda_stream);

/* ---- batched multi-stream decode ----
 *
 * B independent streams decoded together over one model's weights, one token per
 * stream per step, so the projections and the MLP become dense contractions with the
 * streams as one dimension; they run on the tensor cores (bf16 weights, activations
 * as bf16 hi + lo parts, fp32 accumulation).  Each stream has its own cache
 * [n_layers][K, V][n_kv_heads][smax][head_dim] (bf16), position, input token and
 * emitted set; the step does for every stream what qd_decode_step does for one
 * (embedding row of the input token, which joins the stream's emitted set; every
 * layer; final norm, head, repetition penalty, EOS mask, argmax) and feeds each
 * stream's argmax back as its next input token.  Sources: "Qwen3-TTS ncnn port",
 * section "Talker: non-standard structure and two-level generation" (the per-stream
 * step); "qwen3-tts-hip OPTIMIZATION_LOG", decode-step profile (its stages). */
typedef struct qd_batch *qd_batch_handle;

/* qd_batch_create -- n_streams streams of at most smax positions (a multiple of 32)
 * over `model`'s weights (bf16, one output head, an embedding table; the model must
 * outlive the batch).  Allocates n_streams caches, filled with zeros.  Errors: QD_EINVAL,
 * QD_EUNSUPPORTED (shape), QD_ENOMEM, QD_ECUDA; described by qd_last_error(model). */
qd_status qd_batch_create(qd_handle model, int n_streams, int smax, qd_batch_handle *out);
qd_status qd_batch_destroy(qd_batch_handle b);

/* qd_batch_set_stream -- (re)start stream `stream` with `length` cached positions
 * copied from kv_dev (DEVICE bf16 [n_layers][2][n_kv_heads][length][head_dim], may be
 * NULL when length is 0) and input token `token` (< embed_rows) for its next step; its
 * emitted set is cleared.  Synchronises. */
qd_status qd_batch_set_stream(qd_batch_handle b, int stream, const void *kv_dev, int length, int32_t token);

/* qd_batch_set_sampling -- draw every stream's ids instead of taking the greedy argmax,
 * after the repetition penalty and the EOS mask, with the settings of qd_set_sampling
 * (top_k <= 64 candidates, temperature, top_p; "qwen3-tts-hip OPTIMIZATION_LOG",
 * sampling entries): stream b draws u from SplitMix64 of seed + b at its own counter
 * (ids it has drawn since its last qd_batch_set_stream).  top_k 0 restores the argmax.
 * The settings live in device memory, so captured step graphs keep serving.
 * Synchronises.  Errors: QD_EINVAL, QD_EUNSUPPORTED (vocabulary above 32768). */
qd_status qd_batch_set_sampling(qd_batch_handle b, int top_k, float temperature, float top_p, uint64_t seed);

/* qd_batch_decode -- n_steps steps of every stream (greedy unless qd_batch_set_sampling
 * turned sampling on).  ids_dev: DEVICE int32 [n_steps][B] receives each stream's id
 * per step.  force_dev: DEVICE int32
 * [n_steps][B] or NULL: when given, these ids are fed back as the next input tokens
 * instead of the argmaxes (teacher forcing).  Asynchronous; device-side errors are
 * reported by qd_batch_sync.  Errors: QD_EINVAL, QD_ESTATE (a stream never set),
 * QD_EKVFULL (a stream would pass smax; checked before any work). */
qd_status qd_batch_decode(qd_batch_handle b, int n_steps, const int32_t *force_dev, int32_t *ids_dev);

/* qd_batch_prefill -- (re)start ns streams (indices in HOST int[ns], distinct) from a
 * prompt of n positions each: embeds_dev (DEVICE fp32 [ns][n][hidden]).  All ns x n
 * positions go through each layer together: the projections and the MLP as tensor-core
 * GEMMs over ns x n tokens, causal attention on the tensor cores; every position's K
 * and V are written to its stream's cache.  The head runs on each stream's last
 * position; its argmax (EOS mask, the emitted set is empty) goes to first_ids_dev
 * (DEVICE int32 [ns]) and becomes the stream's next input token, at position n; its
 * raw logits go to the stream's row of the qd_batch_get_logits tap.
 * Queued on the batch's stream; returns after the launches are queued.  Errors:
 * QD_EINVAL (streams, n not in [1, smax)), QD_ENOMEM, QD_ECUDA. */
qd_status qd_batch_prefill(qd_batch_handle b, const int *streams, int ns, const float *embeds_dev, int n,
                           int32_t *first_ids_dev);

/* Synchronise; QD_EDEVICE if a kernel reported an error (bounded wait, bad id). */
qd_status qd_batch_sync(qd_batch_handle b);

/* Taps: raw logits of the last step (DEVICE fp32 [B][vocab]); one stream's cache
 * (query the size with dst_dev = NULL); host view of a stream's position; launches. */
qd_status qd_batch_get_logits(qd_batch_handle b, float *dst_dev);
qd_status qd_batch_copy_kv(qd_batch_handle b, int stream, void *dst_dev, size_t *bytes);
qd_status qd_batch_get_pos(qd_batch_handle b, int stream, int *pos);
qd_status qd_batch_get_launch_count(qd_batch_handle b, long long *kernels, int *kernels_per_step);

/* Turn the per-step CUDA graph on (default) or off; results are identical. */
qd_status qd_batch_set_graphs(qd_batch_handle b, int enable);

/* Time `reps` back-to-back launches of one kernel of the step with the step's
 * arguments (captured in a graph; CUDA events on the batch's stream): 1 = attention
 * of the last layer at the streams' current positions (it rewrites the rows the next
 * step writes again), 2 = QKV GEMM, 3 = output-projection GEMM, 4 = gate/up GEMM,
 * 5 = down GEMM of layer 0, 6 = head GEMM.  Between steps only; they change only
 * step scratch.  Synchronises. */
qd_status qd_batch_time_kernel(qd_batch_handle b, int which, int reps, float *avg_ms);

#ifdef __cplusplus
}
#endif
#endif /* QD_H */

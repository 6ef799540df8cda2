/*
 * CPU oracle: the textbook Qwen3-style decoder with a KV cache, computed
 * straightforwardly.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Sources, by page title and section:
 *  [ncnn]   "Qwen3-TTS ncnn port: pure C++/ncnn end-to-end reproduction"
 *           (Tencent/ncnn discussion 6799) -- section "Talker: non-standard
 *           structure and two-level generation" (28-layer Qwen3-style stack,
 *           QK-norm over head_dim after the q/k projections, 8 kv heads
 *           broadcast to 16 q heads, mRoPE that reduces to plain RoPE,
 *           repetition penalty 1.05 on already-emitted ids); section
 *           "Integration and performance optimisation" (a KV cache computes
 *           only the new token's Q/K/V and attends over the cache, equal to
 *           recomputing the whole prefix).
 *  [asr]    "Audio8-ASR: dynamic KV-cache buckets and multi-length end-to-end
 *           acceptance" -- section "Implemented dynamic window mechanism"
 *           (rank-3 cache [heads, Smax, head_dim] written in place; start at
 *           the smallest Smax, and when the write position reaches Smax copy
 *           each layer's valid K/V region into a larger buffer and continue
 *           from the same token and RoPE position; greedy argmax on the host).
 *  [hip]    "qwen3-tts-hip OPTIMIZATION_LOG" -- the decode-step profile entry
 *           (input_norm, qkv_gemm, qk_layout_cache, attention,
 *           output_gemm_residual, post_norm, gate_up_gemm, swiglu,
 *           down_gemm_residual) and the repetition-penalty parity entry.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 * RMSNorm is gamma * x / sqrt(mean(x^2) + eps); RoPE rotates pairs
 * (m, m + head_dim/2) by angle pos * theta^(-2m/head_dim); the attention scale
 * is 1/sqrt(head_dim); kv group of q head i is i / (n_q_heads / n_kv_heads);
 * the repetition penalty divides positive logits by r and multiplies negative
 * ones by r, once per distinct emitted id; argmax ties go to the lowest index.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

struct orc_model {
    orc_config c;
    const void **w; /* owned copy of the pointer table */
    int n_w;
    int pos;        /* positions held in the cache */
    int bucket;     /* index of the current Smax in the ladder */
    int S;          /* current Smax */
    void *kv;       /* [n_layers][2][n_kv_heads][S][head_dim], float or uint16 */
    uint32_t *emitted;
    int emitted_words;
    int have_hidden;
    float *y;       /* final-norm output of the last position with a head */
    int n_gen;      /* ids produced by heads since reset: the sampler's counter */
    int top_k;      /* sampling: 0 = greedy */
    double temperature, top_p;
    uint64_t seed;
    int rope_delta; /* rotary position of a decode step = cache position + rope_delta */
};

/* ---------------------------------------------------------------- helpers */

static inline float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE half from float, round to nearest even (subnormals and overflow to infinity
 * included): the storage of the 8-bit blocks' scales. */
uint16_t orc_f32_to_f16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t absu = u & 0x7fffffffu;
    if (absu > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);          /* NaN */
    if (absu >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);         /* rounds past 65504 */
    const int e = (int)(absu >> 23) - 127;
    if (e >= -14) {                                                     /* normal half */
        uint32_t mant = absu & 0x7fffffu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | (mant >> 13);
        const uint32_t rest = mant & 0x1fffu;
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) ++h;       /* carries into the exponent */
        return (uint16_t)(sign | h);
    }
    if (e < -25) return (uint16_t)sign;                                 /* below half the least subnormal */
    /* subnormal: the value in units of 2^-24, rounded to nearest even */
    const uint32_t mant = (absu & 0x7fffffu) | 0x800000u;
    const int shift = -e - 1;                                           /* 14 .. 24 */
    uint32_t h = mant >> shift;
    const uint32_t rest = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rest > half || (rest == half && (h & 1u))) ++h;
    return (uint16_t)(sign | h);
}

float orc_f16_to_f32(uint16_t h) {
    const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    const int e = (h >> 10) & 0x1f;
    const uint32_t m = h & 0x3ffu;
    float f;
    if (e == 0x1f) {
        uint32_t u = sign | 0x7f800000u | (m << 13);
        memcpy(&f, &u, 4);
        return f;
    }
    if (e == 0) {
        f = (float)m * 5.9604644775390625e-8f;                         /* m * 2^-24, exact */
        return sign ? -f : f;
    }
    uint32_t u = sign | ((uint32_t)(e - 15 + 127) << 23) | (m << 13);
    memcpy(&f, &u, 4);
    return f;
}

int orc_quantize_q8(const float *w, int rows, int K, int8_t *codes, uint16_t *scales) {
    if (rows < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < K / 32; ++b) {
            const float *blk = w + (size_t)r * K + (size_t)b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float a = fabsf(blk[i]);
                if (a > amax) amax = a;
            }
            const float d = amax / 127.0f;
            for (int i = 0; i < 32; ++i) {
                const float q = d > 0.0f ? roundf(blk[i] / d) : 0.0f;
                codes[(size_t)r * K + (size_t)b * 32 + i] = (int8_t)q;
            }
            scales[(size_t)r * (K / 32) + b] = orc_f32_to_f16(d);
        }
    return ORC_OK;
}

int orc_gemv_q8(const int8_t *codes, const uint16_t *scales, int rows, int K, const float *x, float *y) {
    if (rows < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
            const float wq = (float)codes[(size_t)r * K + k] * orc_f16_to_f32(scales[(size_t)r * (K / 32) + k / 32]);
            acc += (double)(wq * x[k]);
        }
        y[r] = (float)acc;
    }
    return ORC_OK;
}

/* Q4_K super-blocks ("audio.cpp Rockchip NPU build notes", "The talker is the only
 * DRAM-bound candidate, and it is not at the ceiling": the talker's matrices as Q4_K,
 * 251 MB per token against 471 MB as Q8_0).  The format, read as the k-quant layout:
 * 256 weights along K in 8 sub-blocks of 32; the super-block holds a half scale d and a
 * half min dm, each sub-block j a 6-bit scale sc_j and a 6-bit min m_j, each weight a
 * 4-bit code q; the weight it stands for is d sc_j q - dm m_j.  144 bytes per
 * super-block (4.5 bits per weight): d, dm (half bits, little-endian), the 8 scales then
 * the 8 mins as 6-bit fields of two 48-bit little-endian words, then 128 bytes of codes
 * (byte i: code 2i in the low nibble, code 2i + 1 in the high one).
 * The pages do not print the quantiser; the plain reading taken here, in fp32 with
 * IEEE division and half-away rounding: per sub-block mn_j = -min(0, min w) and
 * s_j = (max w + mn_j) / 15; d = half(max_j s_j / 63), dm = half(max_j mn_j / 63);
 * sc_j = clamp(round(s_j / d), 0, 63) (0 when d is 0), m_j = clamp(round(mn_j / dm),
 * 0, 63) (0 when dm is 0); q = clamp(round((w + dm m_j) / (d sc_j)), 0, 15) (0 when
 * d sc_j is 0).  d sc_j and dm m_j are exact in fp32 (11-bit by 6-bit significands). */
static void q4k_put6(uint8_t *p, const int *v) {
    uint64_t w = 0;
    for (int j = 0; j < 8; ++j) w |= (uint64_t)(v[j] & 63) << (6 * j);
    for (int b = 0; b < 6; ++b) p[b] = (uint8_t)(w >> (8 * b));
}
static void q4k_get6(const uint8_t *p, int *v) {
    uint64_t w = 0;
    for (int b = 0; b < 6; ++b) w |= (uint64_t)p[b] << (8 * b);
    for (int j = 0; j < 8; ++j) v[j] = (int)((w >> (6 * j)) & 63);
}
static float q4k_round_clamp(float v, float hi) {
    const float r = roundf(v);
    return r < 0.0f ? 0.0f : (r > hi ? hi : r);
}

int orc_quantize_q4k(const float *w, int rows, int K, uint8_t *blocks) {
    if (rows < 0 || K <= 0 || K % 256) return ORC_EINVAL;
    const int nsb = K / 256;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nsb; ++b) {
            const float *x = w + (size_t)r * K + (size_t)b * 256;
            uint8_t *o = blocks + ((size_t)r * nsb + b) * 144;
            float s[8], mn[8], smax = 0.0f, mnmax = 0.0f;
            for (int j = 0; j < 8; ++j) {
                float lo = x[32 * j], hi = x[32 * j];
                for (int i = 1; i < 32; ++i) {
                    if (x[32 * j + i] < lo) lo = x[32 * j + i];
                    if (x[32 * j + i] > hi) hi = x[32 * j + i];
                }
                mn[j] = lo < 0.0f ? -lo : 0.0f;
                s[j] = (hi + mn[j]) / 15.0f;
                if (s[j] > smax) smax = s[j];
                if (mn[j] > mnmax) mnmax = mn[j];
            }
            const uint16_t dh = orc_f32_to_f16(smax / 63.0f), dmh = orc_f32_to_f16(mnmax / 63.0f);
            const float d = orc_f16_to_f32(dh), dm = orc_f16_to_f32(dmh);
            int sc[8], m[8];
            for (int j = 0; j < 8; ++j) {
                sc[j] = d > 0.0f ? (int)q4k_round_clamp(s[j] / d, 63.0f) : 0;
                m[j] = dm > 0.0f ? (int)q4k_round_clamp(mn[j] / dm, 63.0f) : 0;
            }
            o[0] = (uint8_t)(dh & 0xff);
            o[1] = (uint8_t)(dh >> 8);
            o[2] = (uint8_t)(dmh & 0xff);
            o[3] = (uint8_t)(dmh >> 8);
            q4k_put6(o + 4, sc);
            q4k_put6(o + 10, m);
            for (int j = 0; j < 8; ++j) {
                const float step = d * (float)sc[j], off = dm * (float)m[j];
                for (int i = 0; i < 32; ++i) {
                    const int k = 32 * j + i;
                    const float t = x[k] + off;
                    const int q = step > 0.0f ? (int)q4k_round_clamp(t / step, 15.0f) : 0;
                    if (k & 1) o[16 + k / 2] |= (uint8_t)(q << 4);
                    else o[16 + k / 2] = (uint8_t)q;
                }
            }
        }
    return ORC_OK;
}

/* y[r] = sum_k w'[r][k] x[k] with w' = d sc_j q - dm m_j of the super-block layout
 * above: each weight formed in fp32, each product in fp32, summed in fp64. */
int orc_gemv_q4k(const uint8_t *blocks, int rows, int K, const float *x, float *y) {
    if (rows < 0 || K <= 0 || K % 256) return ORC_EINVAL;
    const int nsb = K / 256;
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int b = 0; b < nsb; ++b) {
            const uint8_t *o = blocks + ((size_t)r * nsb + b) * 144;
            const float d = orc_f16_to_f32((uint16_t)(o[0] | (o[1] << 8)));
            const float dm = orc_f16_to_f32((uint16_t)(o[2] | (o[3] << 8)));
            int sc[8], m[8];
            q4k_get6(o + 4, sc);
            q4k_get6(o + 10, m);
            for (int k = 0; k < 256; ++k) {
                const int q = (k & 1) ? (o[16 + k / 2] >> 4) : (o[16 + k / 2] & 15);
                const float wq = d * (float)sc[k / 32] * (float)q - dm * (float)m[k / 32];
                acc += (double)(wq * x[(size_t)b * 256 + k]);
            }
        }
        y[r] = (float)acc;
    }
    return ORC_OK;
}

/* Causal dilated 1-D convolution, written out from its definition: each output is the
 * bias plus the K taps of every input channel at t, t - d, ..., t - (K-1) d. */
int orc_conv1d_causal(const float *x, int Cin, int T, const float *W, const float *bias, int Cout, int K, int dil,
                      float *y) {
    if (Cin <= 0 || T < 0 || Cout <= 0 || K <= 0 || dil <= 0) return ORC_EINVAL;
    for (int o = 0; o < Cout; ++o)
        for (int t = 0; t < T; ++t) {
            double acc = bias ? (double)bias[o] : 0.0;
            for (int i = 0; i < Cin; ++i)
                for (int k = 0; k < K; ++k) {
                    const int ts = t - (K - 1 - k) * dil;
                    if (ts < 0) continue;
                    acc += (double)(W[((size_t)o * Cin + i) * K + k] * x[(size_t)i * T + ts]);
                }
            y[(size_t)o * T + t] = (float)acc;
        }
    return ORC_OK;
}

/* Causal transposed 1-D convolution, kernel 2 * stride, as the scatter that defines it:
 * input frame t adds W[i][o][k] x[i][t] to output t*stride + k; outputs at or past
 * T*stride are dropped. */
int orc_conv_transpose1d_causal(const float *x, int Cin, int T, const float *W, const float *bias, int Cout,
                                int stride, float *y) {
    if (Cin <= 0 || T < 0 || Cout <= 0 || stride <= 0) return ORC_EINVAL;
    const int K = 2 * stride, n = T * stride;
    double *acc = (double *)calloc((size_t)Cout * (n > 0 ? n : 1), sizeof(double));
    if (!acc) return ORC_ENOMEM;
    for (int i = 0; i < Cin; ++i)
        for (int t = 0; t < T; ++t)
            for (int o = 0; o < Cout; ++o)
                for (int k = 0; k < K; ++k) {
                    const int u = t * stride + k;
                    if (u < n) acc[(size_t)o * n + u] += (double)(W[((size_t)i * Cout + o) * K + k] * x[(size_t)i * T + t]);
                }
    for (int o = 0; o < Cout; ++o)
        for (int u = 0; u < n; ++u) y[(size_t)o * n + u] = (float)(acc[(size_t)o * n + u] + (bias ? (double)bias[o] : 0.0));
    free(acc);
    return ORC_OK;
}

/* Round-to-nearest-even float -> bfloat16 (the KV-cache storage rounding). */
uint16_t orc_round_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static inline float wval(const orc_model *m, const void *p, size_t i) {
    return m->c.w_bf16 ? bf16_to_f32(((const uint16_t *)p)[i]) : ((const float *)p)[i];
}

static void widen(const orc_config *c, const void *p, size_t n, float *out) {
    for (size_t i = 0; i < n; ++i)
        out[i] = c->w_bf16 ? bf16_to_f32(((const uint16_t *)p)[i]) : ((const float *)p)[i];
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* out[r] = W[r, :] . x for r in [0, rows); W row-major [rows, K].  Each dot
 * product runs in index order in fp32 (fp64 when acc64). */
static inline float wat(int bf, const void *W, size_t i) {
    return bf ? bf16_to_f32(((const uint16_t *)W)[i]) : ((const float *)W)[i];
}

static void matvec(const orc_config *c, const void *W, int rows, int K, const float *x, float *out) {
    const int bf = c->w_bf16, a64 = c->acc64;
    const int nblk = (rows + 3) / 4;
    /* Rows go in blocks of four only so that four independent sums advance
     * together; each row is still summed alone, in index order. */
#pragma omp parallel for schedule(static)
    for (int blk = 0; blk < nblk; ++blk) {
        int r0 = blk * 4, nr = rows - r0 < 4 ? rows - r0 : 4;
        size_t b[4];
        for (int i = 0; i < 4; ++i) b[i] = (size_t)(r0 + (i < nr ? i : 0)) * (size_t)K;
        if (a64) {
            double a[4] = {0.0, 0.0, 0.0, 0.0};
            for (int k = 0; k < K; ++k) {
                double xk = (double)x[k];
                for (int i = 0; i < 4; ++i) a[i] += (double)wat(bf, W, b[i] + k) * xk;
            }
            for (int i = 0; i < nr; ++i) out[r0 + i] = (float)a[i];
        } else {
            float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int k = 0; k < K; ++k) {
                float xk = x[k];
                for (int i = 0; i < 4; ++i) a[i] += wat(bf, W, b[i] + k) * xk;
            }
            for (int i = 0; i < nr; ++i) out[r0 + i] = a[i];
        }
    }
}

static float dotf(const float *a, const float *b, int n, int a64) {
    if (a64) {
        double acc = 0.0;
        for (int i = 0; i < n; ++i) acc += (double)a[i] * (double)b[i];
        return (float)acc;
    }
    float acc = 0.0f;
    for (int i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* ---------------------------------------------------------------- primitives */

/* RMSNorm as used by the Qwen3-style stack ([ncnn] Talker section; [hip]
 * input_norm / post_norm): out_i = gamma_i * x_i / sqrt(mean(x^2) + eps).
 * The mean-square and the scaling run in fp64. */
void orc_rmsnorm(const float *x, const float *gamma, int n, double eps, float *out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) out[i] = (float)((double)x[i] * inv * (double)gamma[i]);
}

/* Rotary position embedding at absolute position `pos` ([ncnn] Talker section:
 * the interleaved mRoPE with equal position streams is plain RoPE; [asr]: the
 * position continues unchanged across a bucket migration).  Pair m with
 * m + head_dim/2, angle pos * theta^(-2m/head_dim); cos/sin are evaluated in
 * fp64 and rounded to fp32, the rotation itself runs in fp32. */
void orc_rope(float *v, int head_dim, int pos, double theta) {
    const int pos3[3] = {pos, pos, pos}, plain[3] = {0, 0, 0};
    orc_rope_mrope(v, head_dim, pos3, plain, theta);
}

/* Interleaved multimodal RoPE ([ncnn] Talker section: the position encoding comes
 * in three sections, [24, 20, 20] for head_dim 128, interleaved over the channel
 * dimension, one position stream each).  Frequency m takes its position from the
 * stream the interleave deals it: the streams t, h, w in turn, each while it has
 * frequencies left in its section (once the shorter sections run out, the rest go
 * to t).  The two channels of a rotation pair (m, m + head_dim/2) share m.  With
 * every section 0 all frequencies take stream t: plain RoPE. */
int orc_mrope_stream(int m, const int section[3]) {
    if (section[0] + section[1] + section[2] == 0) return 0;
    int left[3] = {section[0], section[1], section[2]};
    int s = 0;
    for (int j = 0; j <= m; ++j) {
        /* deal frequency j to the next stream in turn that still has room */
        int tries = 0;
        while (left[s] == 0 && tries < 3) {
            s = (s + 1) % 3;
            ++tries;
        }
        if (j == m) return s;
        --left[s];
        s = (s + 1) % 3;
    }
    return 0;
}

/* Rotary embedding with a position per stream: pair (m, m + head_dim/2) rotates by
 * pos3[stream(m)] * theta^(-2m/head_dim); cos/sin are evaluated in fp64 and rounded
 * to fp32, the rotation itself runs in fp32. */
void orc_rope_mrope(float *v, int head_dim, const int pos3[3], const int section[3], double theta) {
    int half = head_dim / 2;
    for (int m = 0; m < half; ++m) {
        double inv_freq = pow(theta, -2.0 * (double)m / (double)head_dim);
        double ang = (double)pos3[orc_mrope_stream(m, section)] * inv_freq;
        float cs = (float)cos(ang), sn = (float)sin(ang);
        float a = v[m], b = v[m + half];
        v[m] = a * cs - b * sn;
        v[m + half] = b * cs + a * sn;
    }
}

/* Single-head scaled dot-product attention of one query over L cached
 * positions ([hip] attention bucket; [ncnn] KV-cache section): scores in fp32
 * index-order dot products times 1/sqrt(head_dim); softmax max, exp-sum and the
 * weighted V sum in fp64. */
void orc_attend(const float *q, const float *K, const float *V, int L, int head_dim, float *out) {
    const float scale = (float)(1.0 / sqrt((double)head_dim));
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    double mx = -INFINITY;
    for (int j = 0; j < L; ++j) {
        float d = dotf(q, K + (size_t)j * head_dim, head_dim, 0) * scale;
        s[j] = (double)d;
        if (s[j] > mx) mx = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < L; ++j) {
        s[j] = exp(s[j] - mx);
        l += s[j];
    }
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int j = 0; j < L; ++j) acc += s[j] * (double)V[(size_t)j * head_dim + d];
        out[d] = (float)(acc / l);
    }
    free(s);
}

/* SwiGLU gate ([hip] gate_up_gemm + swiglu): silu(g) * u with
 * silu(z) = z / (1 + exp(-z)), evaluated in fp64 and rounded to fp32. */
float orc_silu_mul(float g, float u) {
    double gd = (double)g;
    return (float)(gd / (1.0 + exp(-gd)) * (double)u);
}

/* Repetition penalty over the emitted ids ([ncnn] Talker section: ids that
 * already appeared are penalised with r = 1.05; [hip] repetition-penalty
 * entry: r = 1.0 leaves the greedy path unchanged), then the EOS mask, then the
 * greedy argmax with the lowest index winning exact ties.  Modifies `logits`
 * in place; returns the id and the top-2 margin of the final logits. */
int orc_penalty_argmax(float *logits, int n, const uint32_t *emitted, float penalty, int eos_id,
                       double *margin) {
    if (emitted && penalty != 1.0f) {
        for (int i = 0; i < n; ++i) {
            if ((emitted[i >> 5] >> (i & 31)) & 1u) {
                float l = logits[i];
                logits[i] = l > 0.0f ? l / penalty : l * penalty;
            }
        }
    }
    if (eos_id >= 0 && eos_id < n) logits[eos_id] = -INFINITY;
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (logits[i] > logits[best]) best = i;
    if (margin) {
        double second = -INFINITY;
        for (int i = 0; i < n; ++i)
            if (i != best && (double)logits[i] > second) second = (double)logits[i];
        *margin = (double)logits[best] - second;
    }
    return best;
}

/* ---------------------------------------------------------------- sampling */

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the state advances by the odd constant gamma and the
 * output is the state passed through the mixing function of that paper (two
 * xor-shift-multiply rounds and a final xor-shift).  Counter-based here: the state
 * of draw `counter` is seed + (counter + 1) * gamma, so any draw is computed
 * directly. */
uint64_t orc_splitmix64(uint64_t seed, uint64_t counter) {
    uint64_t z = seed + (counter + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

double orc_uniform(uint64_t seed, uint64_t counter) {
    return (double)(orc_splitmix64(seed, counter) >> 11) * (1.0 / 9007199254740992.0);   /* 2^-53 */
}

/* The sampling entry of the pages' generation settings ([hip] top_k 50, top_p 1.0,
 * temperature 0.9, seeded): candidates by value then index, weights in fp64,
 * top-p prefix, inverse-CDF draw. */
int orc_sample(const float *logits, int n, int top_k, double temperature, double top_p, double u,
               double *margin) {
    int K = top_k < n ? top_k : n;
    int idx[ORC_MAX_TOPK];
    int taken = 0;
    /* selection: K rounds of "largest not yet taken, lowest index on ties" */
    for (int r = 0; r < K; ++r) {
        int best = -1;
        for (int i = 0; i < n; ++i) {
            int used = 0;
            for (int j = 0; j < taken; ++j) used |= idx[j] == i;
            if (used) continue;
            if (best < 0 || logits[i] > logits[best]) best = i;
        }
        idx[taken++] = best;
    }
    double w[ORC_MAX_TOPK], cum[ORC_MAX_TOPK];
    const double top = (double)logits[idx[0]];
    double total = 0.0;
    for (int i = 0; i < K; ++i) {
        w[i] = (double)logits[idx[i]] == -INFINITY ? 0.0 : exp(((double)logits[idx[i]] - top) / temperature);
        total += w[i];
        cum[i] = total;
    }
    int m = K;   /* smallest prefix reaching top_p of the total */
    for (int i = 0; i < K; ++i)
        if (cum[i] >= top_p * total) {
            m = i + 1;
            break;
        }
    const double z = cum[m - 1], t = u * z;
    int pick = m - 1;
    for (int i = 0; i < m; ++i)
        if (cum[i] > t) {
            pick = i;
            break;
        }
    if (margin) {
        /* how far the decision is from changing: the draw from the cumulative
         * boundaries and the top-p cut from its prefix sums (fractions of the kept or
         * the total weight); the picked logit from its neighbours in the order (logit
         * units); when the pick is the last candidate, the k-th logit from the best
         * excluded one */
        double d = INFINITY;
        for (int i = 0; i < m; ++i) {
            const double e = fabs(cum[i] - t) / z;
            if (e < d) d = e;
        }
        if (top_p < 1.0)
            for (int i = m - 2; i < m; ++i)
                if (i >= 0) {
                    const double e = fabs(cum[i] - top_p * total) / total;
                    if (e < d) d = e;
                }
        const double lp = (double)logits[idx[pick]];
        if (pick > 0 && lp - (double)logits[idx[pick - 1]] > -d) d = (double)logits[idx[pick - 1]] - lp;
        if (pick + 1 < K && lp - (double)logits[idx[pick + 1]] < d) d = lp - (double)logits[idx[pick + 1]];
        if (pick == K - 1 && K < n) {
            double next = -INFINITY;
            for (int i = 0; i < n; ++i) {
                int used = 0;
                for (int j = 0; j < K; ++j) used |= idx[j] == i;
                if (!used && (double)logits[i] > next) next = (double)logits[i];
            }
            if (lp - next < d) d = lp - next;
        }
        *margin = d;
    }
    return idx[pick];
}

int orc_set_sampling(orc_model *m, int top_k, double temperature, double top_p, uint64_t seed) {
    if (top_k < 0 || top_k > ORC_MAX_TOPK || !(temperature > 0.0) || !(top_p > 0.0) || top_p > 1.0)
        return ORC_EINVAL;
    m->top_k = top_k;
    m->temperature = temperature;
    m->top_p = top_p;
    m->seed = seed;
    return ORC_OK;
}

/* ---------------------------------------------------------------- model *//* ---------------------------------------------------------------- model */

static const void *W_(const orc_model *m, int layer, int slot) {
    return m->w[2 + m->c.n_heads_out + layer * ORC_LAYER_SLOTS + slot];
}
enum { S_ATTN_NORM, S_WQ, S_WK, S_WV, S_QNORM, S_KNORM, S_WO, S_MLP_NORM, S_WG, S_WU, S_WD };

static size_t kv_elems(const orc_config *c, int S) {
    return (size_t)c->n_layers * 2 * c->n_kv_heads * (size_t)S * c->head_dim;
}
static size_t kv_esize(const orc_config *c) { return c->kv_bf16 ? 2 : 4; }

/* Address of cache entry [layer][which][g][p][0] in a buffer of Smax S. */
static size_t kv_index(const orc_config *c, int S, int layer, int which, int g, int p) {
    return ((((size_t)layer * 2 + which) * c->n_kv_heads + g) * (size_t)S + p) * c->head_dim;
}

static int validate(const orc_config *c) {
    if (c->hidden <= 0 || c->n_layers <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 ||
        c->head_dim <= 0 || c->ffn <= 0 || c->vocab <= 0)
        return ORC_EINVAL;
    if (c->n_q_heads % c->n_kv_heads) return ORC_EINVAL;
    if (c->head_dim % 2) return ORC_EINVAL;
    if (c->n_heads_out < 1 || c->n_heads_out > ORC_MAX_HEADS) return ORC_EINVAL;
    if (c->n_buckets < 1 || c->n_buckets > ORC_MAX_BUCKETS) return ORC_EINVAL;
    {
        const int *sec = c->mrope_section;
        int sum = sec[0] + sec[1] + sec[2];
        if (sec[0] < 0 || sec[1] < 0 || sec[2] < 0 || (sum != 0 && sum != c->head_dim / 2)) return ORC_EINVAL;
    }
    for (int i = 0; i < c->n_buckets; ++i) {
        if (c->buckets[i] <= 0) return ORC_EINVAL;
        if (i && c->buckets[i] <= c->buckets[i - 1]) return ORC_EINVAL;
    }
    return ORC_OK;
}

orc_model *orc_create(const orc_config *cfg, const void *const *weights, int *status) {
    int st = validate(cfg);
    if (st) {
        if (status) *status = st;
        return NULL;
    }
    orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
    m->c = *cfg;
    m->n_w = 2 + cfg->n_heads_out + cfg->n_layers * ORC_LAYER_SLOTS;
    m->w = (const void **)malloc(sizeof(void *) * (size_t)m->n_w);
    memcpy(m->w, weights, sizeof(void *) * (size_t)m->n_w);
    m->emitted_words = (cfg->vocab + 31) / 32;
    m->emitted = (uint32_t *)calloc((size_t)m->emitted_words, 4);
    m->y = (float *)calloc((size_t)cfg->hidden, 4);
    m->bucket = 0;
    m->S = cfg->buckets[0];
    m->kv = calloc(kv_elems(cfg, m->S), kv_esize(cfg));
    if (!m->kv) {
        orc_destroy(m);
        if (status) *status = ORC_ENOMEM;
        return NULL;
    }
    if (status) *status = ORC_OK;
    return m;
}

void orc_destroy(orc_model *m) {
    if (!m) return;
    free(m->kv);
    free(m->emitted);
    free(m->y);
    free(m->w);
    free(m);
}

/* Reset: empty cache, empty emitted set, back to the smallest bucket ([asr]:
 * each sequence starts from the smallest usable Smax). */
int orc_reset(orc_model *m) {
    m->pos = 0;
    memset(m->emitted, 0, (size_t)m->emitted_words * 4);
    m->have_hidden = 0;
    m->n_gen = 0;
    m->rope_delta = 0;
    if (m->bucket != 0) {
        free(m->kv);
        m->bucket = 0;
        m->S = m->c.buckets[0];
        m->kv = calloc(kv_elems(&m->c, m->S), kv_esize(&m->c));
        if (!m->kv) return ORC_ENOMEM;
    }
    return ORC_OK;
}

int orc_pos(const orc_model *m) { return m->pos; }
int orc_smax(const orc_model *m) { return m->S; }

/* Bucket migration ([asr] dynamic window mechanism; stress section 256->512):
 * allocate the next Smax and copy the valid region [0, pos) of every layer's K
 * and V, entry by entry, into it. */
static int grow_to(orc_model *m, int bucket) {
    const orc_config *c = &m->c;
    int S2 = c->buckets[bucket];
    size_t es = kv_esize(c);
    char *nkv = (char *)calloc(kv_elems(c, S2), es);
    if (!nkv) return ORC_ENOMEM;
    for (int l = 0; l < c->n_layers; ++l)
        for (int w = 0; w < 2; ++w)
            for (int g = 0; g < c->n_kv_heads; ++g)
                for (int p = 0; p < m->pos; ++p)
                    memcpy(nkv + kv_index(c, S2, l, w, g, p) * es,
                           (char *)m->kv + kv_index(c, m->S, l, w, g, p) * es, (size_t)c->head_dim * es);
    free(m->kv);
    m->kv = nkv;
    m->S = S2;
    m->bucket = bucket;
    return ORC_OK;
}

static void kv_store(orc_model *m, int layer, int which, int g, int p, const float *src) {
    const orc_config *c = &m->c;
    size_t idx = kv_index(c, m->S, layer, which, g, p);
    if (c->kv_bf16) {
        uint16_t *d = (uint16_t *)m->kv + idx;
        for (int i = 0; i < c->head_dim; ++i) d[i] = orc_round_bf16(src[i]);
    } else {
        memcpy((float *)m->kv + idx, src, sizeof(float) * (size_t)c->head_dim);
    }
}

static void kv_load_rows(const orc_model *m, int layer, int which, int g, int L, float *out) {
    const orc_config *c = &m->c;
    size_t idx = kv_index(c, m->S, layer, which, g, 0);
    size_t n = (size_t)L * c->head_dim;
    if (c->kv_bf16) {
        const uint16_t *s = (const uint16_t *)m->kv + idx;
        for (size_t i = 0; i < n; ++i) out[i] = bf16_to_f32(s[i]);
    } else {
        memcpy(out, (const float *)m->kv + idx, n * sizeof(float));
    }
}

/* The KV type's value of x: what a reader of the cache sees after a store. */
static void round_kv(const orc_config *c, float *v, int n) {
    if (!c->kv_bf16) return;
    for (int i = 0; i < n; ++i) v[i] = bf16_to_f32(orc_round_bf16(v[i]));
}

/* Final RMSNorm + output head: raw logits ([asr] final RMSNorm / LM-head shard). */
static void head_logits(const orc_config *c, const void *const *w, const float *x, int head_idx,
                        float *y, float *logits) {
    float *gam = (float *)malloc(sizeof(float) * (size_t)c->hidden);
    widen(c, w[1], (size_t)c->hidden, gam);
    orc_rmsnorm(x, gam, c->hidden, c->rms_eps, y);
    matvec(c, w[2 + head_idx], c->vocab, c->hidden, y, logits);
    free(gam);
}

/* One position through the layer stack with the cache: q/k/v of the new token
 * only, attention over positions [0, pos] ([ncnn] integration section). */
/* One position; pos3: its rotary positions (t, h, w), or NULL for the decode
 * rule: cache position + rope_delta in every stream. */
static int forward_at(orc_model *m, const float *embed, int token, int add_emitted, int want_head,
                      int head_idx, int *out_id, float *logits_raw, float *hidden_taps, double *margin,
                      const int *pos3) {
    const orc_config *c = &m->c;
    if (!embed && (token < 0 || token >= c->embed_rows || !m->w[0])) return ORC_EINVAL;
    if (token >= c->vocab && add_emitted) return ORC_EINVAL;
    if (want_head && (head_idx < 0 || head_idx >= c->n_heads_out)) return ORC_EINVAL;
    int p = m->pos;
    if (p == m->S) {
        if (m->bucket + 1 >= c->n_buckets) return ORC_EKVFULL;
        int st = grow_to(m, m->bucket + 1);
        if (st) return st;
    }
    const int h = c->hidden, hd = c->head_dim, qh = c->n_q_heads, kvh = c->n_kv_heads;
    const int qd = qh * hd, kd = kvh * hd, F = c->ffn, grp = qh / kvh;
    const int L = p + 1;
    int r3[3] = {p + m->rope_delta, p + m->rope_delta, p + m->rope_delta};
    if (pos3) memcpy(r3, pos3, sizeof(r3));
    float *x = (float *)malloc(sizeof(float) * (size_t)h);
    float *xn = (float *)malloc(sizeof(float) * (size_t)h);
    float *gam = (float *)malloc(sizeof(float) * (size_t)(h > hd ? h : hd));
    float *q = (float *)malloc(sizeof(float) * (size_t)qd);
    float *k = (float *)malloc(sizeof(float) * (size_t)kd);
    float *v = (float *)malloc(sizeof(float) * (size_t)kd);
    float *att = (float *)malloc(sizeof(float) * (size_t)qd);
    float *tmp = (float *)malloc(sizeof(float) * (size_t)(h > F ? h : F));
    float *g = (float *)malloc(sizeof(float) * (size_t)F);
    float *u = (float *)malloc(sizeof(float) * (size_t)F);
    float *Kr = (float *)malloc(sizeof(float) * (size_t)L * hd * kvh);
    float *Vr = (float *)malloc(sizeof(float) * (size_t)L * hd * kvh);

    /* input: embedding row or caller embedding; the token joins the emitted set */
    if (embed) memcpy(x, embed, sizeof(float) * (size_t)h);
    else for (int i = 0; i < h; ++i) x[i] = wval(m, m->w[0], (size_t)token * h + i);
    if (token >= 0 && add_emitted && token < c->vocab) m->emitted[token >> 5] |= 1u << (token & 31);
    if (hidden_taps) memcpy(hidden_taps, x, sizeof(float) * (size_t)h);

    for (int l = 0; l < c->n_layers; ++l) {
        /* input_norm -> q/k/v projections */
        widen(c, W_(m, l, S_ATTN_NORM), (size_t)h, gam);
        orc_rmsnorm(x, gam, h, c->rms_eps, xn);
        matvec(c, W_(m, l, S_WQ), qd, h, xn, q);
        matvec(c, W_(m, l, S_WK), kd, h, xn, k);
        matvec(c, W_(m, l, S_WV), kd, h, xn, v);
        /* QK-norm over head_dim, one gamma shared by all heads */
        if (c->qk_norm) {
            widen(c, W_(m, l, S_QNORM), (size_t)hd, gam);
            for (int i = 0; i < qh; ++i) {
                memcpy(tmp, q + i * hd, sizeof(float) * (size_t)hd);
                orc_rmsnorm(tmp, gam, hd, c->rms_eps, q + i * hd);
            }
            widen(c, W_(m, l, S_KNORM), (size_t)hd, gam);
            for (int i = 0; i < kvh; ++i) {
                memcpy(tmp, k + i * hd, sizeof(float) * (size_t)hd);
                orc_rmsnorm(tmp, gam, hd, c->rms_eps, k + i * hd);
            }
        }
        /* RoPE at the rotary positions (the absolute position unless the prompt gave others) */
        for (int i = 0; i < qh; ++i) orc_rope_mrope(q + i * hd, hd, r3, c->mrope_section, c->rope_theta);
        for (int i = 0; i < kvh; ++i) orc_rope_mrope(k + i * hd, hd, r3, c->mrope_section, c->rope_theta);
        /* KV append in the cache's type, then attention reads the cache */
        for (int i = 0; i < kvh; ++i) {
            kv_store(m, l, 0, i, p, k + i * hd);
            kv_store(m, l, 1, i, p, v + i * hd);
        }
        for (int i = 0; i < kvh; ++i) {
            kv_load_rows(m, l, 0, i, L, Kr + (size_t)i * L * hd);
            kv_load_rows(m, l, 1, i, L, Vr + (size_t)i * L * hd);
        }
        /* GQA: q head i reads kv group i / (qh / kvh) */
#pragma omp parallel for schedule(static)
        for (int i = 0; i < qh; ++i) {
            int gi = i / grp;
            orc_attend(q + i * hd, Kr + (size_t)gi * L * hd, Vr + (size_t)gi * L * hd, L, hd, att + i * hd);
        }
        /* output projection + residual */
        matvec(c, W_(m, l, S_WO), h, qd, att, tmp);
        for (int i = 0; i < h; ++i) x[i] = x[i] + tmp[i];
        /* post_norm -> gate/up -> SwiGLU -> down + residual */
        widen(c, W_(m, l, S_MLP_NORM), (size_t)h, gam);
        orc_rmsnorm(x, gam, h, c->rms_eps, xn);
        matvec(c, W_(m, l, S_WG), F, h, xn, g);
        matvec(c, W_(m, l, S_WU), F, h, xn, u);
        for (int i = 0; i < F; ++i) g[i] = orc_silu_mul(g[i], u[i]);
        matvec(c, W_(m, l, S_WD), h, F, g, tmp);
        for (int i = 0; i < h; ++i) x[i] = x[i] + tmp[i];
        if (hidden_taps) memcpy(hidden_taps + (size_t)(l + 1) * h, x, sizeof(float) * (size_t)h);
    }
    m->pos = p + 1;

    int st = ORC_OK;
    if (want_head) {
        float *logits = (float *)malloc(sizeof(float) * (size_t)c->vocab);
        head_logits(c, (const void *const *)m->w, x, head_idx, m->y, logits);
        m->have_hidden = 1;
        if (logits_raw) memcpy(logits_raw, logits, sizeof(float) * (size_t)c->vocab);
        int id;
        if (m->top_k > 0) {
            /* penalty and mask as for the argmax, then the sampler */
            (void)orc_penalty_argmax(logits, c->vocab, m->emitted, (float)c->rep_penalty, c->eos_mask_id, NULL);
            id = orc_sample(logits, c->vocab, m->top_k, m->temperature, m->top_p,
                            orc_uniform(m->seed, (uint64_t)m->n_gen), margin);
        } else {
            id = orc_penalty_argmax(logits, c->vocab, m->emitted, (float)c->rep_penalty, c->eos_mask_id, margin);
        }
        m->n_gen++;
        if (out_id) *out_id = id;
        free(logits);
    }
    free(x); free(xn); free(gam); free(q); free(k); free(v); free(att); free(tmp);
    free(g); free(u); free(Kr); free(Vr);
    return st;
}

int orc_forward(orc_model *m, const float *embed, int token, int add_emitted, int want_head,
                int head_idx, int *out_id, float *logits_raw, float *hidden_taps, double *margin) {
    return forward_at(m, embed, token, add_emitted, want_head, head_idx, out_id, logits_raw, hidden_taps,
                      margin, NULL);
}

/* Prefill: positions 0..n-1 in order, head on the last one ([asr]: prefill of
 * the prompt produces the first token; the first bucket is the smallest Smax
 * that holds the prompt).  Prompt tokens do not join the emitted set. */
static int prefill_impl(orc_model *m, const int32_t *tokens, const float *embeds, int n, int head_idx,
                        const int32_t *positions, int *first_id, float *logits_raw, double *margin) {
    const orc_config *c = &m->c;
    if (n <= 0 || (!tokens && !embeds)) return ORC_EINVAL;
    if (positions)
        for (int i = 0; i < 3 * n; ++i)
            if (positions[i] < 0) return ORC_EINVAL;
    if (m->pos != 0) return ORC_ESTATE;
    if (n > c->buckets[c->n_buckets - 1]) return ORC_EKVFULL;
    int b = 0;
    while (c->buckets[b] < n) ++b;
    if (b != m->bucket) {
        free(m->kv);
        m->bucket = b;
        m->S = c->buckets[b];
        m->kv = calloc(kv_elems(c, m->S), kv_esize(c));
        if (!m->kv) return ORC_ENOMEM;
    }
    int top = n - 1;
    for (int i = 0; i < n; ++i) {
        int last = (i == n - 1);
        int p3[3];
        if (positions) {
            for (int s = 0; s < 3; ++s) {
                p3[s] = positions[(size_t)s * n + i];
                if (p3[s] > top) top = p3[s];
            }
        }
        int st = forward_at(m, embeds ? embeds + (size_t)i * c->hidden : NULL, tokens ? tokens[i] : -1, 0,
                            last, head_idx, last ? first_id : NULL, last ? logits_raw : NULL, NULL,
                            last ? margin : NULL, positions ? p3 : NULL);
        if (st) return st;
    }
    /* decode steps continue after the largest rotary position of the prompt */
    m->rope_delta = top + 1 - n;
    return ORC_OK;
}

int orc_prefill(orc_model *m, const int32_t *tokens, const float *embeds, int n, int head_idx,
                int *first_id, float *logits_raw, double *margin) {
    return prefill_impl(m, tokens, embeds, n, head_idx, NULL, first_id, logits_raw, margin);
}

int orc_prefill_positions(orc_model *m, const int32_t *tokens, const float *embeds, int n, int head_idx,
                          const int32_t *positions, int *first_id, float *logits_raw, double *margin) {
    if (!positions) return ORC_EINVAL;
    return prefill_impl(m, tokens, embeds, n, head_idx, positions, first_id, logits_raw, margin);
}

int orc_get_hidden(const orc_model *m, float *out) {
    if (!m->have_hidden) return ORC_ESTATE;
    memcpy(out, m->y, sizeof(float) * (size_t)m->c.hidden);
    return ORC_OK;
}

int orc_get_kv(const orc_model *m, int layer, int which, float *out) {
    const orc_config *c = &m->c;
    if (layer < 0 || layer >= c->n_layers || which < 0 || which > 1) return ORC_EINVAL;
    for (int g = 0; g < c->n_kv_heads; ++g) kv_load_rows(m, layer, which, g, m->pos, out + (size_t)g * m->pos * c->head_dim);
    return ORC_OK;
}

int orc_emitted_words(const orc_model *m, uint32_t *out) {
    memcpy(out, m->emitted, (size_t)m->emitted_words * 4);
    return m->emitted_words;
}

/* Full causal recompute of the whole prefix, layer by layer over all positions,
 * with no cache ([ncnn] integration section: the first version recomputed the
 * whole sequence at every step).  K/V values are rounded to the cache type at
 * the same point as the cached path, so the two agree exactly. */
int orc_recompute_logits(const orc_config *c, const void *const *w, const int32_t *tokens,
                         const float *embeds, int n, int head_idx, float *logits_raw) {
    int st = validate(c);
    if (st) return st;
    if (n <= 0 || (!tokens && !embeds)) return ORC_EINVAL;
    const int h = c->hidden, hd = c->head_dim, qh = c->n_q_heads, kvh = c->n_kv_heads;
    const int qd = qh * hd, kd = kvh * hd, F = c->ffn, grp = qh / kvh;
    const int base = 2 + c->n_heads_out;
    float *X = (float *)malloc(sizeof(float) * (size_t)n * h);
    float *xn = (float *)malloc(sizeof(float) * (size_t)h);
    float *gam = (float *)malloc(sizeof(float) * (size_t)(h > hd ? h : hd));
    float *Q = (float *)malloc(sizeof(float) * (size_t)n * qd);
    float *Kx = (float *)malloc(sizeof(float) * (size_t)n * kd);
    float *Vx = (float *)malloc(sizeof(float) * (size_t)n * kd);
    float *Kh = (float *)malloc(sizeof(float) * (size_t)n * hd);
    float *Vh = (float *)malloc(sizeof(float) * (size_t)n * hd);
    float *att = (float *)malloc(sizeof(float) * (size_t)qd);
    float *tmp = (float *)malloc(sizeof(float) * (size_t)(h > F ? h : F));
    float *g = (float *)malloc(sizeof(float) * (size_t)F);
    float *u = (float *)malloc(sizeof(float) * (size_t)F);
    for (int t = 0; t < n; ++t) {
        if (embeds) memcpy(X + (size_t)t * h, embeds + (size_t)t * h, sizeof(float) * (size_t)h);
        else widen(c, (const char *)w[0] + (size_t)tokens[t] * h * (c->w_bf16 ? 2 : 4), (size_t)h, X + (size_t)t * h);
    }
    for (int l = 0; l < c->n_layers; ++l) {
        const void *const *lw = w + base + l * ORC_LAYER_SLOTS;
        for (int t = 0; t < n; ++t) {
            float *x = X + (size_t)t * h;
            widen(c, lw[S_ATTN_NORM], (size_t)h, gam);
            orc_rmsnorm(x, gam, h, c->rms_eps, xn);
            matvec(c, lw[S_WQ], qd, h, xn, Q + (size_t)t * qd);
            matvec(c, lw[S_WK], kd, h, xn, Kx + (size_t)t * kd);
            matvec(c, lw[S_WV], kd, h, xn, Vx + (size_t)t * kd);
            if (c->qk_norm) {
                widen(c, lw[S_QNORM], (size_t)hd, gam);
                for (int i = 0; i < qh; ++i) {
                    memcpy(tmp, Q + (size_t)t * qd + i * hd, sizeof(float) * (size_t)hd);
                    orc_rmsnorm(tmp, gam, hd, c->rms_eps, Q + (size_t)t * qd + i * hd);
                }
                widen(c, lw[S_KNORM], (size_t)hd, gam);
                for (int i = 0; i < kvh; ++i) {
                    memcpy(tmp, Kx + (size_t)t * kd + i * hd, sizeof(float) * (size_t)hd);
                    orc_rmsnorm(tmp, gam, hd, c->rms_eps, Kx + (size_t)t * kd + i * hd);
                }
            }
            for (int i = 0; i < qh; ++i) orc_rope(Q + (size_t)t * qd + i * hd, hd, t, c->rope_theta);
            for (int i = 0; i < kvh; ++i) orc_rope(Kx + (size_t)t * kd + i * hd, hd, t, c->rope_theta);
            round_kv(c, Kx + (size_t)t * kd, kd);
            round_kv(c, Vx + (size_t)t * kd, kd);
        }
        for (int t = 0; t < n; ++t) {
            float *x = X + (size_t)t * h;
            for (int i = 0; i < qh; ++i) {
                int gi = i / grp;
                for (int j = 0; j <= t; ++j) {
                    memcpy(Kh + (size_t)j * hd, Kx + (size_t)j * kd + gi * hd, sizeof(float) * (size_t)hd);
                    memcpy(Vh + (size_t)j * hd, Vx + (size_t)j * kd + gi * hd, sizeof(float) * (size_t)hd);
                }
                orc_attend(Q + (size_t)t * qd + i * hd, Kh, Vh, t + 1, hd, att + i * hd);
            }
            matvec(c, lw[S_WO], h, qd, att, tmp);
            for (int i = 0; i < h; ++i) x[i] = x[i] + tmp[i];
            widen(c, lw[S_MLP_NORM], (size_t)h, gam);
            orc_rmsnorm(x, gam, h, c->rms_eps, xn);
            matvec(c, lw[S_WG], F, h, xn, g);
            matvec(c, lw[S_WU], F, h, xn, u);
            for (int i = 0; i < F; ++i) g[i] = orc_silu_mul(g[i], u[i]);
            matvec(c, lw[S_WD], h, F, g, tmp);
            for (int i = 0; i < h; ++i) x[i] = x[i] + tmp[i];
        }
    }
    head_logits(c, w, X + (size_t)(n - 1) * h, head_idx, xn, logits_raw);
    free(X); free(xn); free(gam); free(Q); free(Kx); free(Vx); free(Kh); free(Vh);
    free(att); free(tmp); free(g); free(u);
    return ORC_OK;
}

/* ---------------------------------------------------------------- frame input */

/* Next Talker input of a frame, "Qwen3-TTS ncnn port", section "Talker:
 * non-standard structure and two-level generation": the embeddings of the frame's
 * 16 codes (primary code in the Talker's table, residual code j in table j) plus
 * the text/pad embedding, added in fp32 from table 0 to table n-1, text last.
 * Pinned by the tests against an fp64 sum (closed form) and exact small-integer
 * tables. */
int orc_frame_sum(const void *const *tables, const int *rows, const int32_t *ids, int n_tables, int hidden,
                  int bf16, const float *text, float *out) {
    if (n_tables < 1 || hidden < 1) return ORC_EINVAL;
    for (int j = 0; j < n_tables; ++j)
        if (!tables[j] || ids[j] < 0 || ids[j] >= rows[j]) return ORC_EINVAL;
    for (int i = 0; i < hidden; ++i) {
        float v = wat(bf16, tables[0], (size_t)ids[0] * hidden + i);
        for (int j = 1; j < n_tables; ++j) v += wat(bf16, tables[j], (size_t)ids[j] * hidden + i);
        out[i] = v + text[i];
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------- batched linear */

/* out[t][r] = sum_k W[r][k] x[t][k] for T input rows: the projection of every
 * token of a batch is the same matrix-vector product as one decode step's, row by
 * row in index order ([hip] "qkv_gemm" / "gate_up_gemm" stages; a batch of tokens
 * changes only how many vectors meet the same weights).  Pinned by the tests against
 * an fp64 product within the fp32 summation bound. */
int orc_linear(const void *W, int w_bf16, int R, int K, const float *x, int T, float *out) {
    if (!W || !x || !out || R < 1 || K < 1 || T < 0) return ORC_EINVAL;
    orc_config c;
    memset(&c, 0, sizeof(c));
    c.w_bf16 = w_bf16;
    for (int t = 0; t < T; ++t) matvec(&c, W, R, K, x + (size_t)t * K, out + (size_t)t * R);
    return ORC_OK;
}

/* Start a stream from a given cache (the multi-stream workload begins each stream
 * with a cache of its own length instead of a prefill): positions [0, L) of every
 * layer's K and V from `kv` ([n_layers][2][n_kv_heads][L][head_dim] in the cache
 * type: bfloat16 bits when kv_bf16, else float32), position L, empty emitted set, in
 * the smallest bucket that holds L positions.  The stored entries are taken as they
 * are (they are already values of the cache type). */
int orc_set_kv(orc_model *m, const void *kv, int L) {
    const orc_config *c = &m->c;
    if (L < 0 || (L > 0 && !kv)) return ORC_EINVAL;
    int b = 0;
    while (b < c->n_buckets && c->buckets[b] < L) ++b;
    if (b == c->n_buckets) return ORC_EKVFULL;
    int st = orc_reset(m);
    if (st) return st;
    if (b != 0) {
        free(m->kv);
        m->bucket = b;
        m->S = c->buckets[b];
        m->kv = calloc(kv_elems(c, m->S), kv_esize(c));
        if (!m->kv) return ORC_ENOMEM;
    }
    const size_t es = kv_esize(c), row = (size_t)c->head_dim * es;
    for (int l = 0; l < c->n_layers; ++l)
        for (int w = 0; w < 2; ++w)
            for (int g = 0; g < c->n_kv_heads; ++g) {
                const char *src = (const char *)kv + (((size_t)l * 2 + w) * c->n_kv_heads + g) * (size_t)L * row;
                memcpy((char *)m->kv + kv_index(c, m->S, l, w, g, 0) * es, src, (size_t)L * row);
            }
    m->pos = L;
    return ORC_OK;
}

// Internal interface between the decode-step kernels and the engine (host C++).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qd {

struct DevState;

constexpr int kGemvThreads = 256;   // 8 warps
constexpr int kStageRows = 8;       // rows per shared-memory stage
constexpr int kAttnThreads = 128;
constexpr int kAttnChunk = 32;      // positions per split; the split depends on L only
constexpr int kRingBytes = 96 * 1024;

enum GemvMode : int { GEMV_QKV = 0, GEMV_RES = 1, GEMV_GU = 2, GEMV_HEAD = 3 };

struct GemvArgs {
    const void *W;                 // [rows, K] row-major (not GEMV_HEAD)
    const void *const *W_table;    // GEMV_HEAD: device table of head matrices, index st->head_idx
    int rows, K;
    int rs;                        // warps per row (row split factor): 1, 2, 4 or 8
    int unit;                      // CTAs take rows in multiples of `unit` (2 for gate/up pairs)
    int nst;                       // ring stages
    int evict_last;                // keep weights in L2 (evict_last) instead of evict_first
    const float *in;               // input vector [K]
    const float *gamma;            // RMSNorm gamma [K] (QKV, GU, HEAD)
    float eps;
    float *out;                    // QKV [rows]; RES [rows] (+=); GU [rows/2]; HEAD raw-logit tap or null
    // GEMV_HEAD only
    const uint32_t *emitted;
    float penalty;
    int eos;
    float *y_out;                  // normalised input (CTA 0), or null
    float *part_v;                 // [gridDim.x]
    int *part_i;
    int *counter;                  // one int, zero at rest
    int32_t *ids;                  // id history
    int ids_cap;
    int commit;                    // 1: publish the id to the state (0 when timing)
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
    float *part;                   // [qh][max_splits][hd+2]
    int max_splits;
    int *counter;                  // [kvh], zero at rest
    float *out;                    // [qh*hd]
    DevState *st;
};

struct EmbedArgs {
    const void *table;             // [rows, hidden] or null
    int rows, hidden, bf16, vocab, S;
    const float *embed_in;         // [hidden]
    const int32_t *stage_tokens;   // [max_pos]
    const float *stage_embeds;     // [max_pos, hidden]
    uint32_t *emitted;
    float *x;
    DevState *st;
};

// Picks (nseg, rs) for K; false if K is not supported.
bool gemv_split(int K, bool bf16, int *nseg, int *rs);
// Dynamic shared memory of a GEMV launch.
size_t gemv_smem_bytes(int K, bool bf16, int nst);
// Set the max-dynamic-smem attribute on every GEMV / attention instantiation.
cudaError_t kernels_init();

cudaError_t launch_gemv(int mode, bool bf16, const GemvArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_attention(bool bf16, int hd, const AttnArgs &a, int max_splits, cudaStream_t s, bool pdl);
size_t attention_smem_bytes(bool bf16, int hd, int group);
cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t s, bool pdl);
cudaError_t launch_kv_migrate(const void *src, int S_old, void *dst, int S_new, int n_segments, size_t row_bytes,
                              int n_pos, cudaStream_t s);
cudaError_t launch_rope_table(float *cos_t, float *sin_t, int n_pos, int head_dim, double theta, cudaStream_t s);
cudaError_t launch_to_f32(const void *src, bool bf16, float *dst, int n, cudaStream_t s);

}  // namespace qd

// Weight-only 8-bit block quantisation and its GEMV.
//
// Sources (page title, section):
//  - "audio.cpp Rockchip NPU build notes", "The talker is the only DRAM-bound candidate,
//    and it is not at the ceiling": the talker's matrices stream as Q8_0 weights every
//    token, and the bytes of the weight stream are what a decode step pays for.  The
//    layout read here: each row in blocks of 32 weights along K, one half-precision
//    scale d = max|w| / 127 per block, codes round(w / d) (half away from zero; an
//    all-zero block has d = 0 and codes 0).  The product y = W x then reads 1 + 1/16
//    bytes per weight instead of 2 (bf16).
//
// qd_quantize_q8: one warp per block (lane = weight); the maximum by a warp reduction,
// then the same fp32 division and rounding as the definition, so the codes are exact.
// qd_gemv_q8: HBM-bound streaming.  A lane owns 16 consecutive codes of every row
// (one 16-byte load per 512 columns; K = 512, 1024 or 2048), their x values sit in
// registers, and a warp keeps 4 loads per lane in flight (4, 2 or 1 rows; two CTAs of
// 16 warps per SM for K = 512: occupancy beat double-buffering the loads); int8 ->
// fp32 goes through the exponent of 2^23 (exact for |code| <= 128) instead of a
// conversion instruction; each 16-code chunk's partial sum is scaled by its block's
// scale.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "qd.h"
#include "qd_device.cuh"
#include "qd_internal.h"
#include "qd_model.h"

namespace qd {
namespace {

constexpr int kQBlock = 32;
constexpr int kGemvQWarps = 16;

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// One 32-weight block, a warp (lane = weight): the block's code of this lane and the
// half bits of its scale.
__device__ __forceinline__ void q8_block(float v, int8_t &code, uint16_t &scale) {
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float q = d > 0.0f ? roundf(__fdiv_rn(v, d)) : 0.0f;
    code = (int8_t)q;
    scale = __half_as_ushort(__float2half_rn(d));
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_q8_kernel(const T *w, long long n_blocks, int8_t *codes,
                                                          uint16_t *scales) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks; b += warps) {
        int8_t c;
        uint16_t d;
        q8_block(to_f32(w[b * kQBlock + lane]), c, d);
        codes[b * kQBlock + lane] = c;
        if (lane == 0) scales[b] = d;
    }
}

// Rows of W [rows, K] as 8-bit rows (q8_row_bytes: codes, then half scales): row r goes
// to row row0 + r * rstep of dst.
template <typename T>
__global__ void __launch_bounds__(256) quantize_rows_q8_kernel(const T *w, int rows, int K, uint8_t *dst, int row0,
                                                               int rstep) {
    const int lane = threadIdx.x & 31, nb = K / kQBlock;
    const long long n_blocks = (long long)rows * nb, warps = (long long)gridDim.x * (blockDim.x >> 5);
    const size_t rb = q8_row_bytes(K);
    for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks; b += warps) {
        const int r = (int)(b / nb), j = (int)(b - (long long)r * nb);
        int8_t c;
        uint16_t d;
        q8_block(to_f32(w[(size_t)r * K + (size_t)j * kQBlock + lane]), c, d);
        uint8_t *row = dst + (size_t)(row0 + (size_t)r * rstep) * rb;
        row[(size_t)j * kQBlock + lane] = (uint8_t)c;
        if (lane == 0) *reinterpret_cast<uint16_t *>(row + K + (size_t)j * 2) = d;
    }
}

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Dot product of the 16 codes of `u` with x[0..16): each code c becomes the float
// 2^23 + (c + 128) through its biased byte, minus 2^23 + 128, exactly.
__device__ __forceinline__ float dot16(const uint4 &u, const float *x) {
    const uint32_t w[4] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u, u.z ^ 0x80808080u, u.w ^ 0x80808080u};
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float c = __uint_as_float(__byte_perm(w[j], 0x4B000000u, 0x7540u + b)) - 8388736.0f;
            acc = fmaf(c, x[4 * j + b], acc);
        }
    }
    return acc;
}

template <int NCH, int MINB>
__global__ void __launch_bounds__(kGemvQWarps * 32, MINB)
    gemv_q8_kernel(const int8_t *codes, const uint16_t *scales, const float *x, float *y, int rows) {
    constexpr int K = NCH * 512;
    constexpr int RU = 4 / NCH;   // rows per warp in flight
    const int lane = threadIdx.x & 31;
    float xr[NCH * 16];
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(x + c * 512 + lane * 16 + e);
            xr[c * 16 + e] = f.x;
            xr[c * 16 + e + 1] = f.y;
            xr[c * 16 + e + 2] = f.z;
            xr[c * 16 + e + 3] = f.w;
        }
    const int warps = gridDim.x * kGemvQWarps;
    for (int r0 = (blockIdx.x * kGemvQWarps + (threadIdx.x >> 5)) * RU; r0 < rows; r0 += warps * RU) {
        uint4 u[RU][NCH];
        float s[RU][NCH];
#pragma unroll
        for (int q = 0; q < RU; ++q) {
            const int r = r0 + q < rows ? r0 + q : rows - 1;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                u[q][c] = ld_stream16(codes + (size_t)r * K + c * 512 + lane * 16);
                s[q][c] = __half2float(__ushort_as_half(__ldg(scales + (size_t)r * (K / kQBlock) + c * 16 + lane / 2)));
            }
        }
        float acc[RU];
#pragma unroll
        for (int q = 0; q < RU; ++q) {
            acc[q] = 0.f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) acc[q] = fmaf(dot16(u[q][c], xr + c * 16), s[q][c], acc[q]);
        }
#pragma unroll
        for (int q = 0; q < RU; ++q)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        if (lane < RU && r0 + lane < rows) {
            float v = acc[0];
#pragma unroll
            for (int q = 1; q < RU; ++q) v = lane == q ? acc[q] : v;
            y[r0 + lane] = v;
        }
    }
}

typedef void (*GemvQFn)(const int8_t *, const uint16_t *, const float *, float *, int);

GemvQFn gemv_q8_fn(int nch) {
    switch (nch) {
        case 1: return gemv_q8_kernel<1, 2>;
        case 2: return gemv_q8_kernel<2, 1>;
        case 4: return gemv_q8_kernel<4, 1>;
        default: return nullptr;
    }
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- Q4_K super-blocks: 256 weights along K in 8 sub-blocks of 32, 144 bytes each
// (half d, half dm, the 8 six-bit scales and the 8 six-bit mins as two 48-bit
// little-endian words, then 128 bytes of 4-bit codes, low nibble first); weight =
// d sc_j q - dm m_j.  The quantiser takes the same fp32 steps as its definition
// (IEEE division, half-away rounding, round-to-nearest-even halves), so the bytes are
// exact.
constexpr int kQ4Bytes = 144;
constexpr int kGemvQ4Warps = 16;

__device__ __forceinline__ float q4k_rc(float v, float hi) {
    const float r = roundf(v);
    return r < 0.f ? 0.f : (r > hi ? hi : r);
}

// One warp per super-block: lane l holds weights 8 l .. 8 l + 7 (sub-block l / 4).
template <typename T>
__global__ void __launch_bounds__(256) quantize_q4k_kernel(const T *w, long long n_sb, int nsb_row, int K,
                                                           uint8_t *out) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_sb; b += warps) {
        const long long r = b / nsb_row;
        const int sb = (int)(b - r * nsb_row);
        const T *x = w + (size_t)r * K + (size_t)sb * 256 + lane * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = to_f32(x[e]);
        float lo = v[0], hi = v[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) {
            lo = v[e] < lo ? v[e] : lo;
            hi = v[e] > hi ? v[e] : hi;
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {   // the sub-block's four lanes
            const float l2 = __shfl_xor_sync(0xffffffffu, lo, o), h2 = __shfl_xor_sync(0xffffffffu, hi, o);
            lo = l2 < lo ? l2 : lo;
            hi = h2 > hi ? h2 : hi;
        }
        const float mn = lo < 0.f ? -lo : 0.f;
        const float sj = __fdiv_rn(__fadd_rn(hi, mn), 15.f);
        float smax = sj, mnmax = mn;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            mnmax = fmaxf(mnmax, __shfl_xor_sync(0xffffffffu, mnmax, o));
        }
        const __half dh = __float2half_rn(__fdiv_rn(smax, 63.f)), dmh = __float2half_rn(__fdiv_rn(mnmax, 63.f));
        const float d = __half2float(dh), dm = __half2float(dmh);
        const int sc = d > 0.f ? (int)q4k_rc(__fdiv_rn(sj, d), 63.f) : 0;
        const int m = dm > 0.f ? (int)q4k_rc(__fdiv_rn(mn, dm), 63.f) : 0;
        const float step = __fmul_rn(d, (float)sc), off = __fmul_rn(dm, (float)m);
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int q = step > 0.f ? (int)q4k_rc(__fdiv_rn(__fadd_rn(v[e], off), step), 15.f) : 0;
            packed |= (uint32_t)q << (4 * e);
        }
        uint8_t *o = out + (size_t)b * kQ4Bytes;
        *reinterpret_cast<uint32_t *>(o + 16 + lane * 4) = packed;
        // the header: sub-block j's scale and min from lane 4 j
        unsigned long long ws = 0, wm = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            ws |= (unsigned long long)__shfl_sync(0xffffffffu, sc, 4 * j) << (6 * j);
            wm |= (unsigned long long)__shfl_sync(0xffffffffu, m, 4 * j) << (6 * j);
        }
        if (lane == 0) {
            uint4 h;
            h.x = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(dmh) << 16);
            h.y = (uint32_t)ws;                                             // scale bytes 0-3
            h.z = (uint32_t)(ws >> 32) | ((uint32_t)(wm & 0xffffu) << 16);  // scale bytes 4-5, min bytes 0-1
            h.w = (uint32_t)(wm >> 16);                                     // min bytes 2-5
            *reinterpret_cast<uint4 *>(o) = h;
        }
    }
}

// y[r] = sum over sub-blocks of d sc_j (sum_i q_i x_i) - dm m_j (sum_i x_i).  A lane owns
// whole 32-weight sub-blocks of a row (one 16-byte code load each: LPR lanes per row,
// SPL sub-blocks per lane), their 32 x values and their sum in registers; RU rows per
// lane in flight; the row's lanes add their partials with a butterfly.
template <int NSB, int RU>
__global__ void __launch_bounds__(kGemvQ4Warps * 32)
    gemv_q4k_kernel(const uint8_t *blocks, const float *x, float *y, int rows) {
    constexpr int LPR = NSB * 8 < 32 ? NSB * 8 : 32;   // lanes per row
    constexpr int SPL = NSB * 8 / LPR;                  // sub-blocks per lane
    constexpr int RPW = 32 / LPR;                       // rows per warp
    const int lane = threadIdx.x & 31, rl = lane / LPR, li = lane % LPR;
    float xr[SPL][32], xsum[SPL];
#pragma unroll
    for (int k = 0; k < SPL; ++k) {
        const float *xp = x + (li + k * LPR) * 32;      // sub-block g covers columns 32 g ..
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(xp + e);
            xr[k][e] = f.x, xr[k][e + 1] = f.y, xr[k][e + 2] = f.z, xr[k][e + 3] = f.w;
            t += (f.x + f.y) + (f.z + f.w);
        }
        xsum[k] = t;
    }
    const int warps = gridDim.x * kGemvQ4Warps;
    const int w = blockIdx.x * kGemvQ4Warps + (threadIdx.x >> 5);
    for (int r0 = w * RPW * RU; r0 < rows; r0 += warps * RPW * RU) {
        uint4 cw[RU][SPL], hd[RU][SPL];
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            const int r = r0 + u * RPW + rl;
            const int rc = r < rows ? r : rows - 1;
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                const int g = li + k * LPR;
                const uint8_t *o = blocks + ((size_t)rc * NSB + (g >> 3)) * kQ4Bytes;
                cw[u][k] = ld_stream16(o + 16 + 16 * (g & 7));
                hd[u][k] = __ldg(reinterpret_cast<const uint4 *>(o));
            }
        }
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                const int j = (li + k * LPR) & 7;
                const uint4 h = hd[u][k];
                const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffffu)));
                const float dm = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                const unsigned long long ws = (unsigned long long)h.y | ((unsigned long long)(h.z & 0xffffu) << 32);
                const unsigned long long wm = (unsigned long long)(h.z >> 16) | ((unsigned long long)h.w << 16);
                const int sc = (int)((ws >> (6 * j)) & 63), m = (int)((wm >> (6 * j)) & 63);
                const uint32_t cws[4] = {cw[u][k].x, cw[u][k].y, cw[u][k].z, cw[u][k].w};
                float sq = 0.f;
#pragma unroll
                for (int wd = 0; wd < 4; ++wd)
#pragma unroll
                    for (int e = 0; e < 8; ++e) sq = fmaf((float)((cws[wd] >> (4 * e)) & 15u), xr[k][8 * wd + e], sq);
                acc = fmaf(d * (float)sc, sq, acc);
                acc = fmaf(-(dm * (float)m), xsum[k], acc);
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            const int r = r0 + u * RPW + rl;
            if (li == 0 && r < rows) y[r] = acc;
        }
    }
}

typedef void (*GemvQ4Fn)(const uint8_t *, const float *, float *, int);
constexpr int kQ4Ru = 2;   // rows per lane in flight
GemvQ4Fn gemv_q4k_fn(int nsb) {
    switch (nsb) {
        case 2: return gemv_q4k_kernel<2, kQ4Ru>;
        case 4: return gemv_q4k_kernel<4, kQ4Ru>;
        case 8: return gemv_q4k_kernel<8, kQ4Ru>;
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_quantize_rows_q8(const void *w, bool bf16, int rows, int K, void *dst, int row0, int rstep,
                                    cudaStream_t s) {
    if (rows <= 0 || K <= 0 || K % kQBlock) return cudaErrorInvalidValue;
    const long long n_blocks = (long long)rows * (K / kQBlock);
    const int grid = (int)std::min<long long>((n_blocks + 7) / 8, (long long)sm_count() * 16);
    uint8_t *d = static_cast<uint8_t *>(dst);
    if (bf16)
        quantize_rows_q8_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w), rows, K, d,
                                                                    row0, rstep);
    else
        quantize_rows_q8_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(w), rows, K, d, row0, rstep);
    return cudaGetLastError();
}

}  // namespace qd

using namespace qd;

extern "C" {

qd_status qd_quantize_q8(const void *w_dev, int dtype, int rows, int K, int8_t *codes_dev, uint16_t *scales_dev,
                         void *cuda_stream) {
    if (rows <= 0 || K <= 0 || K % kQBlock || (dtype != QD_F32 && dtype != QD_BF16)) return QD_EINVAL;
    if (!is_device_ptr(w_dev) || !is_device_ptr(codes_dev) || !is_device_ptr(scales_dev)) return QD_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const long long n_blocks = (long long)rows * (K / kQBlock);
    const int grid = (int)std::min<long long>((n_blocks + 7) / 8, (long long)sm_count() * 16);
    if (dtype == QD_BF16)
        quantize_q8_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w_dev), n_blocks,
                                                               codes_dev, scales_dev);
    else
        quantize_q8_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(w_dev), n_blocks, codes_dev,
                                                       scales_dev);
    if (cudaGetLastError() != cudaSuccess) return QD_ECUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QD_OK : QD_ECUDA;
}

qd_status qd_gemv_q8(const int8_t *codes_dev, const uint16_t *scales_dev, const float *x_dev, float *y_dev, int rows,
                     int K, void *cuda_stream, int reps, float *avg_ms) {
    if (rows <= 0 || K <= 0 || reps < 0) return QD_EINVAL;
    if (!is_device_ptr(codes_dev) || !is_device_ptr(scales_dev) || !is_device_ptr(x_dev) || !is_device_ptr(y_dev))
        return QD_EINVAL;
    if (!aligned(codes_dev, 16) || !aligned(x_dev, 16) || !aligned(scales_dev, 2)) return QD_EINVAL;
    const GemvQFn fn = K % 512 == 0 ? gemv_q8_fn(K / 512) : nullptr;
    if (!fn) return QD_EUNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int nch = K / 512, per_cta = kGemvQWarps * (4 / nch);
    const int grid = std::max(1, std::min((rows + per_cta - 1) / per_cta, (nch == 1 ? 2 : 1) * sm_count()));
    fn<<<grid, kGemvQWarps * 32, 0, s>>>(codes_dev, scales_dev, x_dev, y_dev, rows);
    if (cudaGetLastError() != cudaSuccess) return QD_ECUDA;
    if (reps > 0 && avg_ms) {
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) != cudaSuccess) return QD_ECUDA;
        if (cudaEventCreate(&e1) != cudaSuccess) {
            cudaEventDestroy(e0);
            return QD_ECUDA;
        }
        cudaEventRecord(e0, s);
        for (int i = 0; i < reps; ++i) fn<<<grid, kGemvQWarps * 32, 0, s>>>(codes_dev, scales_dev, x_dev, y_dev, rows);
        cudaEventRecord(e1, s);
        const bool ok = cudaEventSynchronize(e1) == cudaSuccess && cudaGetLastError() == cudaSuccess;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        *avg_ms = ms / (float)reps;
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        if (!ok) return QD_ECUDA;
    }
    return QD_OK;
}

qd_status qd_quantize_q4k(const void *w_dev, int dtype, int rows, int K, uint8_t *blocks_dev, void *cuda_stream) {
    if (rows <= 0 || K <= 0 || K % 256 || (dtype != QD_F32 && dtype != QD_BF16)) return QD_EINVAL;
    if (!is_device_ptr(w_dev) || !is_device_ptr(blocks_dev) || !aligned(blocks_dev, 16)) return QD_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const long long n_sb = (long long)rows * (K / 256);
    const int grid = (int)std::min<long long>((n_sb + 7) / 8, (long long)sm_count() * 16);
    if (dtype == QD_BF16)
        quantize_q4k_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w_dev), n_sb,
                                                                K / 256, K, blocks_dev);
    else
        quantize_q4k_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(w_dev), n_sb, K / 256, K,
                                                        blocks_dev);
    if (cudaGetLastError() != cudaSuccess) return QD_ECUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QD_OK : QD_ECUDA;
}

qd_status qd_gemv_q4k(const uint8_t *blocks_dev, const float *x_dev, float *y_dev, int rows, int K, void *cuda_stream,
                      int reps, float *avg_ms) {
    if (rows <= 0 || K <= 0 || reps < 0) return QD_EINVAL;
    if (!is_device_ptr(blocks_dev) || !is_device_ptr(x_dev) || !is_device_ptr(y_dev)) return QD_EINVAL;
    if (!aligned(blocks_dev, 16) || !aligned(x_dev, 16)) return QD_EINVAL;
    const GemvQ4Fn fn = K % 256 == 0 ? gemv_q4k_fn(K / 256) : nullptr;
    if (!fn) return QD_EUNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const int nsb = K / 256, lpr = nsb * 8 < 32 ? nsb * 8 : 32;
    const int per_cta = kGemvQ4Warps * (32 / lpr) * kQ4Ru;   // rows a CTA takes per pass
    const int grid = std::max(1, std::min((rows + per_cta - 1) / per_cta, 2 * sm_count()));
    fn<<<grid, kGemvQ4Warps * 32, 0, s>>>(blocks_dev, x_dev, y_dev, rows);
    if (cudaGetLastError() != cudaSuccess) return QD_ECUDA;
    if (reps > 0 && avg_ms) {
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) != cudaSuccess) return QD_ECUDA;
        if (cudaEventCreate(&e1) != cudaSuccess) {
            cudaEventDestroy(e0);
            return QD_ECUDA;
        }
        cudaEventRecord(e0, s);
        for (int i = 0; i < reps; ++i) fn<<<grid, kGemvQ4Warps * 32, 0, s>>>(blocks_dev, x_dev, y_dev, rows);
        cudaEventRecord(e1, s);
        const bool ok = cudaEventSynchronize(e1) == cudaSuccess && cudaGetLastError() == cudaSuccess;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        *avg_ms = ms / (float)reps;
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        if (!ok) return QD_ECUDA;
    }
    return QD_OK;
}

}  // extern "C"

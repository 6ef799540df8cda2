// Codec decoder convolution stages.
//
// Sources (page title, section):
//  - "qwen3-tts-hip OPTIMIZATION_LOG", codec-profile and transposed-convolution
//    entries: the codec decoder's time goes to causal dilated convolutions and to
//    transposed convolutions.  With kernel length 2 * stride, output sample
//    s = t * stride + p (p < stride) of a transposed convolution takes tap p of input
//    frame t and tap p + stride of frame t - 1, nothing else (the per-phase form).
//  - "Qwen3-TTS ncnn port", pipeline overview: the codec's SEANet upsampler.
//
// qd_conv1d_causal: y[o][t] = b[o] + sum_i sum_k W[o][i][k] x[i][t - (K-1-k) d], zero
// history.  A CTA computes 32 output channels x 128 frames (16 per thread); per chunk of
// 8 input channels it stages the 128 frames plus the (K-1) d frames of history and the
// chunk's taps in shared memory.
// qd_conv_transpose1d_causal: the per-phase form above, one thread per output sample,
// the two contributing input frames read directly.
// fp32 throughout.  Channel-major signals, row-major weights as the C-ABI states.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "qd.h"
#include "qd_model.h"

namespace qd {
namespace {

constexpr int kConvTO = 32;    // output channels per CTA
constexpr int kConvTT = 128;   // frames per CTA
constexpr int kConvCI = 8;     // input channels per chunk
constexpr int kConvMaxK = 16;
constexpr int kConvMaxHalo = 512;

__global__ void __launch_bounds__(256) conv1d_causal_kernel(const float *x, int Cin, int T, const float *W,
                                                            const float *bias, int Cout, int K, int dil, float *y) {
    extern __shared__ float cs[];
    const int halo = (K - 1) * dil, span = kConvTT + halo;
    float *xs = cs;                          // [CI][span]
    float *ws = xs + kConvCI * span;         // [TO][CI][K]
    const int t0 = blockIdx.x * kConvTT, o0 = blockIdx.y * kConvTO;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;   // frames tx + 32 m, channels 4 ty + a
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[a][m] = 0.f;
    for (int i0 = 0; i0 < Cin; i0 += kConvCI) {
        for (int e = tid; e < kConvCI * span; e += 256) {
            const int c = e / span, j = e % span, i = i0 + c, t = t0 - halo + j;
            xs[e] = (i < Cin && t >= 0 && t < T) ? x[(size_t)i * T + t] : 0.f;
        }
        for (int e = tid; e < kConvTO * kConvCI * K; e += 256) {
            const int o = e / (kConvCI * K), r = e % (kConvCI * K), c = r / K, k = r % K;
            const int oo = o0 + o, i = i0 + c;
            ws[e] = (oo < Cout && i < Cin) ? W[((size_t)oo * Cin + i) * K + k] : 0.f;
        }
        __syncthreads();
        for (int c = 0; c < kConvCI; ++c)
            for (int k = 0; k < K; ++k) {
                float xv[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) xv[m] = xs[c * span + tx + 32 * m + k * dil];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float w = ws[((4 * ty + a) * kConvCI + c) * K + k];
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc[a][m] = fmaf(w, xv[m], acc[a][m]);
                }
            }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int o = o0 + 4 * ty + a;
        if (o >= Cout) continue;
        const float b = bias ? bias[o] : 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int t = t0 + tx + 32 * m;
            if (t < T) y[(size_t)o * T + t] = acc[a][m] + b;
        }
    }
}

__global__ void __launch_bounds__(256) conv_transpose1d_causal_kernel(const float *x, int Cin, int T, const float *W,
                                                                      const float *bias, int Cout, int s, float *y) {
    const long long n = (long long)T * s, total = (long long)Cout * n;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int o = (int)(idx / n);
        const long long u = idx % n;
        const int t = (int)(u / s), p = (int)(u % s);
        float acc = 0.f;
        for (int i = 0; i < Cin; ++i) {
            const float *wr = W + ((size_t)i * Cout + o) * 2 * s;
            acc = fmaf(wr[p], x[(size_t)i * T + t], acc);
            if (t > 0) acc = fmaf(wr[p + s], x[(size_t)i * T + t - 1], acc);
        }
        y[idx] = acc + (bias ? bias[o] : 0.f);
    }
}

int sm_count_codec() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace
}  // namespace qd

using namespace qd;

extern "C" {

qd_status qd_conv1d_causal(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev, int Cout,
                           int K, int dilation, float *y_dev, void *cuda_stream) {
    if (Cin <= 0 || T <= 0 || Cout <= 0 || K <= 0 || K > kConvMaxK || dilation <= 0) return QD_EINVAL;
    if ((long long)(K - 1) * dilation > kConvMaxHalo) return QD_EUNSUPPORTED;
    if (!is_device_ptr(x_dev) || !is_device_ptr(w_dev) || !is_device_ptr(y_dev) || (bias_dev && !is_device_ptr(bias_dev)))
        return QD_EINVAL;
    const int span = kConvTT + (K - 1) * dilation;
    const size_t smem = ((size_t)kConvCI * span + (size_t)kConvTO * kConvCI * K) * sizeof(float);
    const dim3 grid((T + kConvTT - 1) / kConvTT, (Cout + kConvTO - 1) / kConvTO);
    conv1d_causal_kernel<<<grid, 256, smem, static_cast<cudaStream_t>(cuda_stream)>>>(x_dev, Cin, T, w_dev, bias_dev,
                                                                                      Cout, K, dilation, y_dev);
    return cudaGetLastError() == cudaSuccess ? QD_OK : QD_ECUDA;
}

qd_status qd_conv_transpose1d_causal(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev,
                                     int Cout, int stride, float *y_dev, void *cuda_stream) {
    if (Cin <= 0 || T <= 0 || Cout <= 0 || stride <= 0 || stride > 64) return QD_EINVAL;
    if (!is_device_ptr(x_dev) || !is_device_ptr(w_dev) || !is_device_ptr(y_dev) || (bias_dev && !is_device_ptr(bias_dev)))
        return QD_EINVAL;
    const long long total = (long long)Cout * T * stride;
    const int grid = (int)std::min<long long>((total + 255) / 256, (long long)sm_count_codec() * 8);
    conv_transpose1d_causal_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        x_dev, Cin, T, w_dev, bias_dev, Cout, stride, y_dev);
    return cudaGetLastError() == cudaSuccess ? QD_OK : QD_ECUDA;
}

}  // extern "C"

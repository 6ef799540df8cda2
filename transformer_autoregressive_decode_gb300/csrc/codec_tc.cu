// Codec decoder convolutions on the tensor cores (tcgen05, through the batched paths'
// GEMM with shifted taps).
//
// Sources (page title, section):
//  - "qwen3-tts-hip OPTIMIZATION_LOG", transposed-convolution entry: a transposed
//    convolution with kernel length 2 * stride is, per output phase p, two GEMMs, one
//    over the input frames and one over the frames shifted by one (tap p on frame t,
//    tap p + stride on frame t - 1); the causal dilated convolutions are the other
//    codec stage it profiles.
//
// Both become out[t][o] = sum_j sum_i Wj[o][i] x[t - shift_j][i] with the signal
// time-major (frames as the GEMM's tokens, channels as its reduction) and one weight
// slab per tap:
//  - causal convolution: taps k = 0..K-1, slab k = W[:, :, k], shift (K-1-k) d (zero
//    history: frames before 0 load as zeros);
//  - transposed convolution, phase p: taps 0, 1 with slabs p and p + stride of
//    W[i][o][.], shifts 0 and 1; the phase's outputs go to samples t * stride + p.
// The weights are rounded to bf16 (round to nearest even) and packed tap-major, zero
// padded to 128 output x 64 input channels; the signal enters as bf16 hi + lo parts
// (x_lo = bf16(x - bf16(x)): 16 significant bits); accumulation is fp32 in tensor
// memory; the epilogue adds the bias and writes the channel-major output directly.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "qd.h"
#include "qd_internal.h"
#include "qd_model.h"

namespace qd {
namespace {

constexpr int kPadO = 128;   // output channels: the GEMM's 128-row weight tiles
constexpr int kPadI = 64;    // input channels: its 64-wide reduction chunks

struct CodecBuf {
    void *p = nullptr;
    ~CodecBuf() {
        if (p) cudaFree(p);
    }
    cudaError_t alloc(size_t bytes) { return cudaMalloc(&p, std::max<size_t>(bytes, 16)); }
};

// Wp[j][o][i] = bf16(W at tap j, output o, input i) for o < Cout, i < Cin, else 0.
// layout 0: W[o][i][j] (convolution), layout 1: W[i][o][j] (transposed convolution).
__global__ void pack_taps_kernel(const float *W, int Cout, int Cin, int taps, int layout, __nv_bfloat16 *Wp,
                                 int Coutp, int Cinp) {
    const size_t total = (size_t)taps * Coutp * Cinp;
    for (size_t n = (size_t)blockIdx.x * blockDim.x + threadIdx.x; n < total; n += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(n % Cinp);
        const int o = (int)((n / Cinp) % Coutp);
        const int j = (int)(n / ((size_t)Cinp * Coutp));
        float v = 0.f;
        if (o < Cout && i < Cin)
            v = layout == 0 ? W[((size_t)o * Cin + i) * taps + j] : W[((size_t)i * Cout + o) * taps + j];
        Wp[n] = __float2bfloat16_rn(v);
    }
}

// Channel-major x [Cin][T] -> time-major hi / lo parts [T][Cinp] (channels past Cin
// zero), through 32 x 32 shared-memory tiles so both sides move whole rows.
__global__ void __launch_bounds__(256) time_major_kernel(const float *x, int Cin, int T, int Cinp,
                                                         __nv_bfloat16 *xh, __nv_bfloat16 *xl) {
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (int r = ty; r < 32; r += 8) {
        const int c = c0 + r, t = t0 + tx;
        tile[r][tx] = (c < Cin && t < T) ? x[(size_t)c * T + t] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int t = t0 + r, c = c0 + tx;
        if (t < T) {
            const float v = tile[tx][r];
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            xh[(size_t)t * Cinp + c] = h;
            xl[(size_t)t * Cinp + c] = __float2bfloat16_rn(v - __bfloat162float(h));
        }
    }
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// One convolution: pack the weights (slabs tap-major), the signal time-major, then
// `phases` GEMMs (1 for the causal convolution, stride for the transposed one).
qd_status conv_tc(const float *x, int Cin, int T, const float *w, int layout, int slabs, const float *bias, int Cout,
                  int taps, int phases, int x_shift0, int x_shift_step, int slab_step, float *y, int ldo, int ldt,
                  cudaStream_t s, int reps, float *avg_ms) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QD_ECUDA;
    const int Coutp = round_up(Cout, kPadO), Cinp = round_up(Cin, kPadI);
    TcGemmPlan plan;
    if (!tc_gemm_plan(Coutp, taps * Cinp, T, sms, &plan)) return QD_EUNSUPPORTED;
    if (tc_gemm_init() != cudaSuccess) return QD_ECUDA;
    const size_t nw = (size_t)slabs * Coutp * Cinp, nx = (size_t)T * Cinp;
    const size_t ncnt = (size_t)plan.row_tiles * plan.tok_tiles * 2;
    CodecBuf wp, xh, xl, part, cnt, st;
    if (wp.alloc(nw * 2) || xh.alloc(nx * 2) || xl.alloc(nx * 2) || part.alloc(plan.partial_floats * 4) ||
        cnt.alloc(ncnt * 4) || st.alloc(4))
        return QD_ENOMEM;
    if (cudaMemsetAsync(cnt.p, 0, ncnt * 4, s) || cudaMemsetAsync(st.p, 0, 4, s)) return QD_ECUDA;
    auto run = [&]() -> bool {
        const int gw = (int)std::min<size_t>((nw + 255) / 256, (size_t)sms * 16);
        pack_taps_kernel<<<gw, 256, 0, s>>>(w, Cout, Cin, slabs, layout, static_cast<__nv_bfloat16 *>(wp.p), Coutp,
                                            Cinp);
        time_major_kernel<<<dim3((T + 31) / 32, Cinp / 32), 256, 0, s>>>(
            x, Cin, T, Cinp, static_cast<__nv_bfloat16 *>(xh.p), static_cast<__nv_bfloat16 *>(xl.p));
        if (cudaGetLastError() != cudaSuccess) return false;
        for (int p = 0; p < phases; ++p) {
            TcGemmArgs a = {};
            a.R = Coutp;
            a.K = Cinp;
            a.T = T;
            a.mode = TC_STORE_RT;
            a.out = y + p;
            a.ldo = ldo;
            a.ldt = ldt;
            a.r_valid = Cout;
            a.bias = bias;
            a.taps = taps;
            a.w_slab0 = p;
            a.w_slab_step = slab_step;
            a.x_shift0 = x_shift0;
            a.x_shift_step = x_shift_step;
            a.w_rows = slabs * Coutp;
            a.partial = plan.splits > 1 ? static_cast<float *>(part.p) : nullptr;
            a.tile_counter = static_cast<int *>(cnt.p);
            a.status = static_cast<int *>(st.p);
            if (launch_tc_gemm(plan, wp.p, xh.p, xl.p, a, s) != cudaSuccess) return false;
        }
        return true;
    };
    if (!run()) return QD_ECUDA;
    if (avg_ms) {
        if (reps < 1) return QD_EINVAL;
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) || cudaEventCreate(&e1)) return QD_ECUDA;
        cudaEventRecord(e0, s);
        bool ok = true;
        for (int i = 0; i < reps && ok; ++i) ok = run();
        cudaEventRecord(e1, s);
        cudaEventSynchronize(e1);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        *avg_ms = ms / reps;
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        if (!ok) return QD_ECUDA;
    }
    int status = 0;
    if (cudaMemcpyAsync(&status, st.p, 4, cudaMemcpyDeviceToHost, s) || cudaStreamSynchronize(s)) return QD_ECUDA;
    return status ? QD_EDEVICE : QD_OK;
}

}  // namespace
}  // namespace qd

using namespace qd;

extern "C" {

qd_status qd_conv1d_causal_tc(const float *x_dev, int Cin, int T, const float *w_dev, const float *bias_dev, int Cout,
                              int K, int dilation, float *y_dev, void *cuda_stream, int reps, float *avg_ms) {
    if (Cin <= 0 || T <= 0 || Cout <= 0 || K <= 0 || K > 64 || dilation <= 0) return QD_EINVAL;
    if ((long long)(K - 1) * dilation > (1 << 20)) return QD_EUNSUPPORTED;
    if (!is_device_ptr(x_dev) || !is_device_ptr(w_dev) || !is_device_ptr(y_dev) || (bias_dev && !is_device_ptr(bias_dev)))
        return QD_EINVAL;
    // tap k reads frame t - (K-1-k) d: shifts (K-1) d, (K-2) d, ..., 0
    return conv_tc(x_dev, Cin, T, w_dev, 0, K, bias_dev, Cout, K, 1, (K - 1) * dilation, -dilation, 1, y_dev, T, 1,
                   static_cast<cudaStream_t>(cuda_stream), reps, avg_ms);
}

qd_status qd_conv_transpose1d_causal_tc(const float *x_dev, int Cin, int T, const float *w_dev,
                                        const float *bias_dev, int Cout, int stride, float *y_dev, void *cuda_stream,
                                        int reps, float *avg_ms) {
    if (Cin <= 0 || T <= 0 || Cout <= 0 || stride <= 0 || stride > 64) return QD_EINVAL;
    if (!is_device_ptr(x_dev) || !is_device_ptr(w_dev) || !is_device_ptr(y_dev) || (bias_dev && !is_device_ptr(bias_dev)))
        return QD_EINVAL;
    // phase p: slab p on frame t, slab p + stride on frame t - 1; samples t * stride + p
    return conv_tc(x_dev, Cin, T, w_dev, 1, 2 * stride, bias_dev, Cout, 2, stride, 0, 1, stride, y_dev, T * stride,
                   stride, static_cast<cudaStream_t>(cuda_stream), reps, avg_ms);
}

}  // extern "C"

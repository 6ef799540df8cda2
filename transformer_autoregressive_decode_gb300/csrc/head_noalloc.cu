// Output head (logits, repetition penalty, EOS mask, greedy argmax) for callers that
// cannot allocate device memory: all scratch the kernel needs lives in one
// fixed-size file-scope device array, so a call performs no allocation of any kind.
//
// The kernel streams the head matrix with the same producer/consumer ring and GEMV
// reduction as the decode step's head, so for the same normalised hidden state it
// produces the same logits and the same id.  The per-CTA argmax candidates and the
// completion counter that the decode step keeps in library-allocated scratch are
// kept here in `g_head_scratch`.
#include <cmath>
#include <mutex>

#include "../../include/qd.h"
#include "decode_common.cuh"
#include "qd_model.h"

namespace qd {

// Upper bound of CTAs one call may use (one per SM is used).  The array holds one
// argmax candidate per CTA and the completion counter: about 8 KB per device.
constexpr int kNoAllocMaxCtas = 1024;
constexpr int kNoAllocMaxHidden = 8192;

struct NoAllocScratch {
    float cand_v[kNoAllocMaxCtas];
    int cand_i[kNoAllocMaxCtas];
    unsigned counter;   // must be zero when a launch starts
    unsigned pad[63];
};

// Shared by every call on a device, for the life of the process.  Host code must not
// pass `g_head_scratch` itself to a kernel (on the host it names a host-side stand-in);
// it passes the device address obtained with cudaGetSymbolAddress.
static __device__ __align__(256) NoAllocScratch g_head_scratch;

struct HeadArgs {
    const void *W;            // [vocab, hidden]
    const float *y;           // [hidden], normalised
    const uint32_t *emitted;  // bitmask or null
    float penalty;
    int eos, vocab, hidden;
    int rs, rps, nst, rows_max;
    int32_t *out_id;
    float *logits;            // raw logits or null
    NoAllocScratch *scr;      // device address of g_head_scratch
};

template <typename WT, int NSEG>
__global__ void __launch_bounds__(kGemvThreads, 1) head_argmax_noalloc_kernel(const HeadArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int NC = kConsumerWarps * 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t row_bytes = (uint32_t)(a.hidden * sizeof(WT));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nst * kSlotBytes);
    uint64_t *empty = full + a.nst;
    float *yin = reinterpret_cast<float *>(empty + a.nst);   // [hidden]
    float *misc = yin + a.hidden;                              // [64]
    int *misc_i = reinterpret_cast<int *>(misc + 32);
    float *res = misc + 64;                                    // [rows_max][rs]
    uint32_t *emw = reinterpret_cast<uint32_t *>(res + a.rows_max * a.rs);
    const Ring R{smem, full, empty, a.nst};

    const int units = a.vocab;
    const int row0 = (int)((long long)units * blockIdx.x / gridDim.x);
    const int nrows = (int)((long long)units * (blockIdx.x + 1) / gridDim.x) - row0;

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        misc_i[4] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == kConsumerWarps) {
        if (lane == 0 && nrows > 0) {
            uint32_t sidx = 0;
            (void)produce_rows(R, sidx, reinterpret_cast<const uint8_t *>(a.W) + (size_t)row0 * row_bytes, nrows,
                               row_bytes, a.rps, policy_evict_first());
        }
        return;
    }

    const int w0 = row0 >> 5;
    const int nw = nrows > 0 ? ((row0 + nrows - 1) >> 5) - w0 + 1 : 0;
    if (a.emitted && a.penalty != 1.0f)
        for (int i = tid; i < nw; i += NC) emw[i] = __ldcg(a.emitted + w0 + i);
    load_vec_smem(a.y, a.hidden, yin);
    named_sync(1, NC);
    const int colbase = (warp % a.rs) * (a.hidden / a.rs);
    float xr[NSEG * Elem<WT>::kPer16B];
    smem_slice<WT, NSEG>(yin, colbase, xr);
    uint32_t sidx = 0;
    const bool got = gemv_consume<WT, NSEG>(R, sidx, nrows, a.rps, row_bytes, a.rs, colbase, xr, res);
    if (named_sync_or(1, NC, !got)) {
        // a stage never arrived: let copies still in flight land, report no id
        if (tid == 0) {
            for (uint32_t s2 = sidx; s2 < sidx + (uint32_t)a.nst; ++s2)
                (void)mbar_wait_bounded(&full[s2 % a.nst], (s2 / a.nst) & 1, 10000000ull);
            *a.out_id = -1;
        }
        return;
    }

    float best_v = -INFINITY;
    int best_i = INT_MAX;
    for (int r = tid; r < nrows; r += NC) {
        float v = 0.f;
        for (int j = 0; j < a.rs; ++j) v += res[r * a.rs + j];
        const int row = row0 + r;
        if (a.logits) a.logits[row] = v;
        if (a.emitted && a.penalty != 1.0f && ((emw[(row >> 5) - w0] >> (row & 31)) & 1u))
            v = v > 0.f ? v / a.penalty : v * a.penalty;
        if (row == a.eos) v = -INFINITY;
        if (arg_better(v, row, best_v, best_i)) {
            best_v = v;
            best_i = row;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (arg_better(ov, oi, best_v, best_i)) {
            best_v = ov;
            best_i = oi;
        }
    }
    if (lane == 0) {
        misc[8 + warp] = best_v;
        misc_i[8 + warp] = best_i;
    }
    named_sync(1, NC);
    if (tid == 0) {
        float bv = misc[8];
        int bi = misc_i[8];
        for (int w = 1; w < kConsumerWarps; ++w)
            if (arg_better(misc[8 + w], misc_i[8 + w], bv, bi)) {
                bv = misc[8 + w];
                bi = misc_i[8 + w];
            }
        a.scr->cand_v[blockIdx.x] = bv;
        a.scr->cand_i[blockIdx.x] = bi;
        __threadfence();
        const unsigned prev = atomicAdd(&a.scr->counter, 1u);
        misc_i[5] = (prev == gridDim.x - 1);
    }
    named_sync(1, NC);
    if (misc_i[5] && warp == 0) {
        // last CTA: reduce the candidates of every CTA (lowest index on ties)
        __threadfence();
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = lane; c < (int)gridDim.x; c += 32) {
            const float v = __ldcg(a.scr->cand_v + c);
            const int i = __ldcg(a.scr->cand_i + c);
            if (arg_better(v, i, bv, bi)) {
                bv = v;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (arg_better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            *a.out_id = bi;
            a.scr->counter = 0;
        }
    }
}

typedef void (*HeadFn)(const HeadArgs);

static HeadFn head_fn(bool bf16, int nseg) {
    if (bf16) {
        switch (nseg) {
            case 1: return head_argmax_noalloc_kernel<__nv_bfloat16, 1>;
            case 2: return head_argmax_noalloc_kernel<__nv_bfloat16, 2>;
            case 3: return head_argmax_noalloc_kernel<__nv_bfloat16, 3>;
            case 4: return head_argmax_noalloc_kernel<__nv_bfloat16, 4>;
        }
    } else {
        switch (nseg) {
            case 1: return head_argmax_noalloc_kernel<float, 1>;
            case 2: return head_argmax_noalloc_kernel<float, 2>;
            case 3: return head_argmax_noalloc_kernel<float, 3>;
            case 4: return head_argmax_noalloc_kernel<float, 4>;
        }
    }
    return nullptr;
}

// Per-device set-up, done by the first call on each device with that device current:
// the device address of g_head_scratch, the SM count and the kernels' shared-memory
// limit.  No allocation is involved.
struct NoAllocDevice {
    bool ready = false;
    NoAllocScratch *scr = nullptr;
    int sms = 0;
};
static std::mutex g_noalloc_mu;
static NoAllocDevice g_noalloc_dev[64];

static constexpr size_t kNoAllocSmemMax = 220 * 1024;

static qd_status noalloc_setup(int dev, NoAllocDevice **out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (dev < 0 || dev >= 64) return QD_EUNSUPPORTED;
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess) return QD_ECUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return QD_ECUDA;
        for (int bf = 0; bf < 2; ++bf)
            for (int ns = 1; ns <= 4; ++ns)
                if (cudaFuncSetAttribute(reinterpret_cast<const void *>(head_fn(bf != 0, ns)),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNoAllocSmemMax) !=
                    cudaSuccess)
                    return QD_ECUDA;
        d.scr = reinterpret_cast<NoAllocScratch *>(p);
        d.sms = sms;
        d.ready = true;
    }
    *out = &d;
    return QD_OK;
}

}  // namespace qd

using namespace qd;

extern "C" qd_status qd_head_argmax_noalloc(const float *y_dev, const void *w_dev, int vocab, int hidden, int dtype,
                                            const uint32_t *emitted_dev, double rep_penalty, int eos_mask_id,
                                            int32_t *out_id_dev, float *logits_dev, void *cuda_stream) {
    if (!y_dev || !w_dev || !out_id_dev) return QD_EINVAL;
    // every buffer must be device memory: a host pointer is refused here rather than
    // faulting inside the kernel (the pointer queries allocate nothing)
    if (!is_device_ptr(y_dev) || !is_device_ptr(w_dev) || !is_device_ptr(out_id_dev)) return QD_EINVAL;
    if ((emitted_dev && !is_device_ptr(emitted_dev)) || (logits_dev && !is_device_ptr(logits_dev))) return QD_EINVAL;
    if (dtype != QD_F32 && dtype != QD_BF16) return QD_EINVAL;
    if (vocab < 1 || hidden < 1 || eos_mask_id < -1 || eos_mask_id >= vocab || !(rep_penalty > 0.0)) return QD_EINVAL;
    const bool bf16 = dtype == QD_BF16;
    int nseg = 0, rs = 0;
    if (hidden > kNoAllocMaxHidden || hidden % 256 || !gemv_split(hidden, bf16, &nseg, &rs)) return QD_EUNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QD_ECUDA;
    NoAllocDevice *d = nullptr;
    qd_status st = noalloc_setup(dev, &d);
    if (st) return st;
    const int grid = d->sms < vocab ? d->sms : vocab;
    if (grid > kNoAllocMaxCtas) return QD_EUNSUPPORTED;

    HeadArgs a = {};
    a.W = w_dev;
    a.y = y_dev;
    a.emitted = emitted_dev;
    a.penalty = (float)rep_penalty;
    a.eos = eos_mask_id;
    a.vocab = vocab;
    a.hidden = hidden;
    a.rs = rs;
    a.rps = kSlotBytes / (int)(hidden * (bf16 ? 2 : 4));
    a.rows_max = (vocab + grid - 1) / grid;
    a.out_id = out_id_dev;
    a.logits = logits_dev;
    a.scr = d->scr;
    const size_t fixed = (size_t)hidden * 4 + 64 * 4 + (size_t)a.rows_max * rs * 4 + ((size_t)a.rows_max / 32 + 2) * 4;
    int nst = (int)((kNoAllocSmemMax - fixed - 256) / (kSlotBytes + 16));
    const int need = (a.rows_max + a.rps - 1) / a.rps;
    nst = nst < 8 ? nst : 8;
    nst = nst < need ? nst : need;
    if (nst < 1) return QD_EUNSUPPORTED;
    a.nst = nst;
    const size_t smem = (size_t)nst * kSlotBytes + (size_t)nst * 16 + fixed;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(cuda_stream);
    // the counter must start at zero (an earlier call that stopped early may have
    // left it otherwise); the candidates are all rewritten by this launch
    if (cudaMemsetAsync(&d->scr->counter, 0, sizeof(unsigned), s) != cudaSuccess) return QD_ECUDA;
    head_fn(bf16, nseg)<<<grid, kGemvThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? QD_OK : QD_ECUDA;
}

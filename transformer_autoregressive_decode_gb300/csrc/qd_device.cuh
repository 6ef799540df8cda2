// Device-side building blocks for the decode-step kernels (sm_103a).
//
// Weights stream from HBM into a shared-memory ring with 1-D bulk async copies
// (cp.async.bulk, completion counted on an mbarrier).  Kernels are launched with
// programmatic dependent launch: each one issues its weight copies, which do not
// depend on the previous kernel, before griddepcontrol.wait, so the HBM stream
// keeps running across kernel boundaries.  Every wait on an mbarrier is bounded
// in time; on expiry the kernel records an error bit in the device state and
// stops consuming, so no kernel can hang.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qd {

// ------------------------------------------------------------------ device state
// Lives in device memory, one per handle.  Every kernel of a step works on
// position `pos`; the last kernel of the step advances it.  The host writes the
// input description (in_mode .. head_idx) before a step; the head kernel
// publishes the id (out_id, n_gen) and any error bits (status).
struct DevState {
    int pos;          // positions held in the cache = position written by the step in flight
    int in_mode;      // IN_* below
    int token_in;     // token of the step (IN_TOKEN), -1: none
    int add_emitted;  // the step's token joins the emitted set
    int head_idx;     // output head of the step
    int out_id;       // id produced by the last step that ran a head
    int n_gen;        // ids produced since reset (index into the id history)
    int status;       // DEV_ERR_* bits, sticky until reset
    int rope_delta;   // rotary position of a step = its cache position + rope_delta
    int rope_staged;  // 1: the rotary positions come per stream from the staged prompt positions
    // sampling (kept by a reset): sample_k 0 = greedy argmax, else top-k candidates,
    // temperature, top-p, and the seed of the counter-based draws (draw n_gen)
    int sample_k;
    float sample_temp, sample_top_p;
    uint32_t seed_lo, seed_hi;
    int pad[1];
};
// bytes of DevState that a reset zeroes (the sampling settings follow them)
#define QD_DEVSTATE_RESET_BYTES (10 * sizeof(int))

enum : int {
    IN_TOKEN = 0,          // x = E[token_in]
    IN_EMBED = 1,          // x = embed_in (fp32 [hidden])
    IN_STAGED_TOKENS = 2,  // x = E[stage_tokens[cur]]
    IN_STAGED_EMBEDS = 3,  // x = stage_embeds[cur]
    IN_FEEDBACK = 4,       // x = E[out_id], the previous argmax
};

enum : int {
    DEV_ERR_WAIT_TIMEOUT = 1,  // an mbarrier wait expired
    DEV_ERR_BAD_TOKEN = 2,     // token outside the embedding table
    DEV_ERR_BAD_POS = 4,       // position outside the bucket
    DEV_ERR_IDS_FULL = 8,      // id history full
};

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on the barrier and add `bytes` to the transaction count it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded spins count SM cycles (clock64: cheap to read, unlike the global timer,
// whose reads in a spinning warp held back the other warps of its scheduler).  A
// limit of n ns is taken as 4n cycles: at least n ns at any SM clock up to 4 GHz.
__device__ __forceinline__ unsigned long long cycles_now() { return (unsigned long long)clock64(); }
__host__ __device__ constexpr unsigned long long wait_cycles(unsigned long long ns) { return 4ull * ns; }

// Wait for phase `parity` of the barrier to complete; false after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = cycles_now();
    while (!mbar_try_wait(bar, parity)) {
        if (cycles_now() - t0 > wait_cycles(limit_ns)) return false;
    }
    return true;
}

// L2 eviction policies for the bulk copies.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared; completion is counted on `bar` (bytes).
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Plain arrive (count 1) on a barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier among the first `nthreads` threads of the CTA (named barrier `id`).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- thread-block clusters: distributed shared memory and the cluster barrier
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of `p` (a shared-memory variable of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes before it
// are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Named barrier `id` over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes into the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------------ numerics
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Element loads/stores for the two storage types.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPer16B = 4;
    __device__ static float load(const float *p, int i) { return p[i]; }
    // elements i, i + 1 (i even) in one 8-byte access
    __device__ static float2 load2(const float *p, int i) { return *reinterpret_cast<const float2 *>(p + i); }
    __device__ static void store(float *p, int i, float v) { p[i] = v; }
    // 16 bytes -> 4 floats
    __device__ static void unpack(const uint4 &u, float *f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPer16B = 8;
    __device__ static float load(const __nv_bfloat16 *p, int i) { return __bfloat162float(p[i]); }
    // elements i, i + 1 (i even) in one 4-byte access
    __device__ static float2 load2(const __nv_bfloat16 *p, int i) {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p + i);
        return make_float2(bf16lo(u), bf16hi(u));
    }
    __device__ static void store(__nv_bfloat16 *p, int i, float v) { p[i] = __float2bfloat16_rn(v); }
    __device__ static void unpack(const uint4 &u, float *f) {
        f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
        f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
    }
};

}  // namespace qd

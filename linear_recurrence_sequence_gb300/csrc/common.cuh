// Device helpers shared by the SAMU and RG-LRU scan kernels (sm_103a).
//
// Nothing here is shared with the FP64 oracle: this is the CUDA side only.
#pragma once

#include <cstdint>
#include <cuda.h>            // CUtensorMap (type only)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/samu.h"

namespace lrs {

// ---------------------------------------------------------------------------
// Tiling.  A chain is one (batch row, group of 64 modes or channels); each
// lane of a warp owns two adjacent modes, so a warp covers a group and reads
// 128 contiguous bytes of each BF16 half per token.  A tile is a run of
// 16-token sub-chunks of one chain, one sub-chunk per worker warp.  Entry
// states are kept per sub-chunk, in slot t / 16 of the sequence.
// ---------------------------------------------------------------------------
constexpr int kGroup = 64;           // modes (SAMU) or channels (RG-LRU) per chain
constexpr int kSub = 16;             // tokens per warp sub-chunk
constexpr int kRowBytes = kGroup * 2;   // one BF16 row of a box (128 bytes)

// Look-back status values stored per (chain, chunk).
constexpr uint32_t kFlagEmpty = 0u;
constexpr uint32_t kFlagAgg = 1u;    // the tile's own affine map is published
constexpr uint32_t kFlagIncl = 2u;   // the state after the tile is published
constexpr uint32_t kFlagErr = 3u;    // the tile gave up; waiters abort

// Bounded waits.  Every wait on another warp, CTA or copy gives up after
// kWaitLimitNs of %globaltimer time (far above any legitimate wait: a whole
// scan takes well under a millisecond per 10^8 elements), records
// LRS_ERR_TIMEOUT in the status word and lets the kernel return.
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;

// Device status word bits (OR-ed together by failing CTAs).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusUpstream = 2u;
constexpr uint32_t kStatusLayout = 4u;    // a shared-memory buffer missed its required alignment (nothing copied)

// ---------------------------------------------------------------------------
// Memory-model primitives (PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// L2-only loads (never served from a possibly stale L1 line).
__device__ __forceinline__ float4 ldcg4(const float4* p) { return __ldcg(p); }
__device__ __forceinline__ float2 ldcg2(const float2* p) { return __ldcg(p); }

// Nanosecond global timer (PTX %globaltimer).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Deadline of one bounded wait: expired() is cheap (the timer is read every
// 32nd poll) and turns true once kWaitLimitNs have passed since the first read.
struct WaitClock {
    uint64_t t0 = 0;
    uint32_t n = 0;
    __device__ __forceinline__ bool expired() {
        if ((++n & 31u) != 0u) return false;
        const uint64_t t = global_ns();
        if (t0 == 0) {
            t0 = t;
            return false;
        }
        return t - t0 > kWaitLimitNs;
    }
};

// ---------------------------------------------------------------------------
// Shared-memory barriers and TMA (cp.async.bulk.tensor) loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait for the barrier phase of the given parity (try_wait lets the
// hardware park the warp between polls); false once the deadline passes.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    WaitClock clk;
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clk.expired()) return false;
    }
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 3-D tiled tensor load of one box into shared memory, completing on `bar`.
// The innermost coordinate x must be a multiple of 8 elements (16 bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled tensor store of one box from shared memory (bulk-group
// completion; rows outside the tensor are not written).  The innermost
// coordinate x must be a multiple of 8 elements (16 bytes) and no coordinate
// may be negative.  The writing threads order their shared-memory writes
// before it with fence_proxy_async() and a barrier.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, const void* src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
                 : "memory");
}
// 2-D tiled tensor store of one box from shared memory, the same rules.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global into shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Decoupled look-back, chain search, executed by one full warp.  For tile c
// of one chain, finds the nearest predecessor (walking in direction dir: -1
// towards tile 0, +1 towards tile C-1) whose state after the tile (kFlagIncl)
// is published while every closer predecessor has at least published its map
// (kFlagAgg).  Each poll inspects 32 predecessors (one per lane, acquire
// loads).  Returns the same value in every lane; -1 if a predecessor failed or
// the deadline passed.
//
// Publishing side: the warp's lanes store the map or state, __syncwarp()
// orders those stores before lane 0's, and lane 0's release store of the flag
// (cumulative at gpu scope) makes them visible to any warp that acquires the
// flag.  No separate fence per lane is needed.
__device__ __forceinline__ int lookback_find_warp(const uint32_t* flags, int c, int C, int dir) {
    const int lane = threadIdx.x & 31;
    int base = c + dir;
    uint32_t polls = 0;
    WaitClock clk;
    for (;;) {
        const int idx = base + dir * lane;
        const bool valid = idx >= 0 && idx < C;
        const uint32_t f = valid ? ld_acquire_gpu(flags + idx) : kFlagAgg;
        const unsigned incl = __ballot_sync(0xffffffffu, f == kFlagIncl);
        const unsigned empty = __ballot_sync(0xffffffffu, f == kFlagEmpty);
        const unsigned bad = __ballot_sync(0xffffffffu, f == kFlagErr);
        const int first = incl ? (__ffs(incl) - 1) : 32;
        const unsigned upto = first >= 31 ? 0xffffffffu : ((2u << first) - 1u);
        const unsigned before = first >= 32 ? 0xffffffffu : ((1u << first) - 1u);
        if (bad & upto) return -1;
        if (empty & before) {
            if (clk.expired()) return -1;
            if (++polls > 8) __nanosleep(64);
            continue;
        }
        if (first < 32) return base + dir * first;
        base += 32 * dir;
    }
}

// Programmatic dependent launch.  A kernel launched with
// launch_ex(..., pdl = true) may start while the previous kernel on the
// stream is still running; it must call pdl_wait() before it touches global
// memory that earlier kernels write or read.  pdl_trigger() lets the next
// kernel start once every CTA of this one has issued it.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// 2^x on the SFU (PTX ex2.approx, documented relative error ~2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 1/x, sqrt(x), 1/sqrt(x) on the SFU (PTX rcp/sqrt/rsqrt.approx; documented
// errors of about one ulp, 2^-23 and 2^-22.9 relative).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rsqrt_approx(float x) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// BF16 pairs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(h);
}

__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Complex affine maps T(h) = lam h + beta, stored as float4 {lam.re, lam.im,
// beta.re, beta.im}.  apply() is the single place where a map meets a state,
// so a state rebuilt during look-back is bitwise the state the owning tile
// published (explicit fmaf: no contraction choices left to the compiler).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 capply(float4 T, float2 h) {
    float re = __fmaf_rn(T.x, h.x, __fmaf_rn(-T.y, h.y, T.z));
    float im = __fmaf_rn(T.x, h.y, __fmaf_rn(T.y, h.x, T.w));
    return make_float2(re, im);
}

// lam * z (complex)
__device__ __forceinline__ float2 cmul(float2 a, float2 z) {
    return make_float2(__fmaf_rn(a.x, z.x, -__fmul_rn(a.y, z.y)),
                       __fmaf_rn(a.x, z.y, __fmul_rn(a.y, z.x)));
}

// conj(a) * z
__device__ __forceinline__ float2 cmulc(float2 a, float2 z) {
    return make_float2(__fmaf_rn(a.x, z.x, __fmul_rn(a.y, z.y)),
                       __fmaf_rn(a.x, z.y, -__fmul_rn(a.y, z.x)));
}

// T2 o T1 (T1 first): (l2 l1, l2 b1 + b2).
__device__ __forceinline__ float4 compose_maps(float4 T2, float4 T1) {
    const float2 L = cmul(make_float2(T2.x, T2.y), make_float2(T1.x, T1.y));
    const float2 Bv = capply(T2, make_float2(T1.z, T1.w));
    return make_float4(L.x, L.y, Bv.x, Bv.y);
}

// Real affine maps {a, b} for the RG-LRU chain.
__device__ __forceinline__ float rapply(float2 T, float h) { return __fmaf_rn(T.x, h, T.y); }

// T2 o T1 for real maps.
__device__ __forceinline__ float2 rcompose(float2 T2, float2 T1) {
    return make_float2(__fmul_rn(T2.x, T1.x), __fmaf_rn(T2.x, T1.y, T2.y));
}

}  // namespace lrs

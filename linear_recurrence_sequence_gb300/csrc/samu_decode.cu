// SAMU single-token decode step on sm_103a: one token of each of B
// sequences, controller projection + transition + FP32 state update + BF16
// output in one launch.
//
// Equations: SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比"), section 05
// (controller, transition, recurrence), applied to one token with the carried
// state as z_{t-1}: the forward over a sequence equals the decode step applied
// token after token.  The per-parameter work that does not depend on the token
// (unit directions, amplitude factors, lbar_m = e^{-nu_m} e^{i theta_m} as a
// double-float formed in FP64) is done once by samu_decode_prepare into a
// caller-owned parameter block, so that the step itself is one launch.
//
// GB300 organisation: one CTA of T threads per sequence (T = 128 for
// D <= 1024, else 256, so that every thread owns one to four mode pairs; at
// most 64 registers, so that 32 warps of it are resident per SM).  When the
// batch alone would leave most SMs idle, P CTAs per sequence (a separate
// instantiation): each forms the token's dot products and scalars in full
// (the same operations, so the same bits) and updates every P-th group of T
// mode pairs.
// Thread t owns the 8-channel chunks t, t+T, ... of the token's x_sel row for
// the two dot products (16-byte loads, paired FP32 arithmetic), reduced over
// the CTA in a fixed order behind a CTA barrier; lane 0 of every warp then
// forms the token's scalars from the warp sums (the same operations in every
// warp, so the same bits) and broadcasts them by shuffle (T = 256: thread 0
// forms them behind a second barrier).  Thread t owns
// the mode pairs (2t, 2t+1), (2t+2T, 2t+2T+1), ...: state, w and the outputs
// move as 16-byte (state) and 4-byte (BF16 pairs) accesses, coalesced across
// the CTA.  Bandwidth-bound: per sequence 2D (x_sel) + 2D (w) + 2D (y) + 8D
// (state read and written) bytes.
#include <algorithm>
#include <atomic>

#include "kernels.cuh"

namespace lrs {

constexpr int kDecThreads = 256;              // the prepare kernel, and the step for D > 1024
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecPairs = 4;   // mode pairs per thread: M <= 2 * 256 * kDecPairs = 2048 (D <= 4096)

// Parameter block (floats from the start of the caller's buffer):
//   w_hat_phi [D+1], w_hat_r [D+1], each starting on a 16-byte boundary
//   misc[8]        k_phi, k_r, (unused)
//   nu  [M]
//   modes [M] float4 lbar hi/lo (16-byte aligned)
__host__ __device__ inline size_t dec_row(int D) { return (size_t)(D + 1 + 3) & ~size_t(3); }
__host__ __device__ inline size_t dec_off_misc(int D) { return 2 * dec_row(D); }
__host__ __device__ inline size_t dec_off_nu(int D) { return dec_off_misc(D) + 8; }
__host__ __device__ inline size_t dec_off_modes(int D) { return (dec_off_nu(D) + D / 2 + 3) & ~size_t(3); }
size_t samu_decode_params_floats(int D) { return dec_off_modes(D) + (size_t)4 * (D / 2); }

// Block 0: the norms ||w_phi||, ||w_r|| over all D+1 entries (FP32, fixed
// order: per-thread strided sums, warp xor tree, warp-order sum), the unit
// directions and the amplitude factors.  Blocks 1..: the per-mode constants
// (FP64) and nu.
__global__ void __launch_bounds__(kDecThreads) samu_decode_prepare_kernel(SamuDecodePrepArgs a) {
    __shared__ float s_red[2][kDecWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = a.D, M = D / 2, n = D + 1;
    float* wh = a.params;
    float* misc = a.params + dec_off_misc(D);
    float* nu_out = a.params + dec_off_nu(D);
    float4* modes = reinterpret_cast<float4*>(a.params + dec_off_modes(D));
    if (blockIdx.x > 0) {
        const int m = (blockIdx.x - 1) * kDecThreads + tid;
        mode_constants(a.nu, a.theta, M, modes, m);
        if (m < M) nu_out[m] = a.nu[m];
        return;
    }
    float sp = 0.f, sr = 0.f;
    for (int j = tid; j < n; j += kDecThreads) {
        const float x = a.w_phi[j], y = a.w_r[j];
        sp = fmaf(x, x, sp);
        sr = fmaf(y, y, sr);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sr += __shfl_xor_sync(0xffffffffu, sr, o);
    }
    if (lane == 0) {
        s_red[0][warp] = sp;
        s_red[1][warp] = sr;
    }
    __syncthreads();
    float tp = 0.f, tr = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
        tp += s_red[0][w];
        tr += s_red[1][w];
    }
    const float inv_phi = 1.0f / sqrtf(tp), inv_r = 1.0f / sqrtf(tr);
    for (int j = tid; j < n; j += kDecThreads) {
        wh[j] = a.w_phi[j] * inv_phi;
        wh[dec_row(D) + j] = a.w_r[j] * inv_r;
    }
    if (tid == 0) {
        const float ism = 1.0f / sqrtf((float)M);
        misc[0] = tanhf(a.a_phi[0]) * ism;
        misc[1] = tanhf(a.a_r[0]) * ism;
    }
}

// One token of sequence blockIdx.x, T threads (SPLIT: of sequence
// blockIdx.x / P, part blockIdx.x % P of its modes).
template <int T, bool SPLIT>
__global__ void __launch_bounds__(T, 1024 / T) samu_decode_step_kernel(SamuDecodeStepArgs a) {
    constexpr int W = T / 32;
    __shared__ float2 s_red[W];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = a.D, M = D / 2, nch = D / 8;
    const size_t b = SPLIT ? blockIdx.x / (unsigned)a.parts : blockIdx.x;
    // the first mode of the thread's pairs and the distance between them
    const int m0 = SPLIT ? 2 * ((int)(blockIdx.x % (unsigned)a.parts) * T + tid) : 2 * tid;
    const int mstep = SPLIT ? 2 * T * a.parts : 2 * T;
    const float* wh = a.params;
    const float* misc = a.params + dec_off_misc(D);
    const float* nu = a.params + dec_off_nu(D);
    const float4* modes = reinterpret_cast<const float4*>(a.params + dec_off_modes(D));

    // this thread's mode pairs (2t, 2t+1), (2t + 512, ...): state and w go out
    // first, independent of the token's controls
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(a.w) + b * (size_t)(D / 2);
    uint32_t* yrow = reinterpret_cast<uint32_t*>(a.y) + b * (size_t)(D / 2);
    float4 zs[kDecPairs];
    uint32_t wre[kDecPairs], wim[kDecPairs];
#pragma unroll
    for (int j = 0; j < kDecPairs; ++j) {
        const int m = m0 + j * mstep;
        if (m < M) {
            zs[j] = __ldcs(reinterpret_cast<const float4*>(a.state_in + (b * M + m) * 2));   // re0, im0, re1, im1
            wre[j] = __ldcs(wrow + m / 2);
            wim[j] = __ldcs(wrow + (M + m) / 2);
        }
    }

    // controller: x~ . w_hat for both directions
    const uint4* xr = reinterpret_cast<const uint4*>(a.x) + b * nch;
    f2x pp = 0ull, pr = 0ull;
    for (int c = tid; c < nch; c += T) {
        const uint4 q = __ldcs(xr + c);
        const float4* w0 = reinterpret_cast<const float4*>(wh + 8 * c);                 // w_hat_phi of the chunk
        const float4* wq = reinterpret_cast<const float4*>(wh + dec_row(D) + 8 * c);    // w_hat_r
        const float4 p0 = w0[0], p1 = w0[1], r0 = wq[0], r1 = wq[1];
        const f2x x0 = bf2x(q.x), x1 = bf2x(q.y), x2 = bf2x(q.z), x3 = bf2x(q.w);
        pp = fma2(x0, pk2(p0.x, p0.y), pp);
        pp = fma2(x1, pk2(p0.z, p0.w), pp);
        pp = fma2(x2, pk2(p1.x, p1.y), pp);
        pp = fma2(x3, pk2(p1.z, p1.w), pp);
        pr = fma2(x0, pk2(r0.x, r0.y), pr);
        pr = fma2(x1, pk2(r0.z, r0.w), pr);
        pr = fma2(x2, pk2(r1.x, r1.y), pr);
        pr = fma2(x3, pk2(r1.z, r1.w), pr);
    }
    float a0, a1, b0, b1;
    up2(pp, a0, a1);
    up2(pr, b0, b1);
    float sp = a0 + a1, sr = b0 + b1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sr += __shfl_xor_sync(0xffffffffu, sr, o);
    }
    if (lane == 0) s_red[warp] = make_float2(sp, sr);
    __syncthreads();
    // {E - 1, C, S, reset}: with four warps every warp forms them (lane 0) and
    // broadcasts by shuffle; with eight, thread 0 forms them behind a second
    // barrier (eight copies of the transcendental chain cost more than it)
    constexpr bool kPerWarp = W <= 4;
    __shared__ float4 s_ctl;
    float4 ctl = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kPerWarp ? lane == 0 : tid == 0) {
        float tp = wh[D], tr = wh[dec_row(D) + D];   // the appended constant 1 times the bias weight
        for (int w = 0; w < W; ++w) {
            tp += s_red[w].x;
            tr += s_red[w].y;
        }
        const float p = tanhf(tp), r = tanhf(tr);
        const float d = misc[0] * p, c = misc[1] * (r / (1.0f + r * r));
        float sn, cs;
        sincosf(d, &sn, &cs);
        const float rs = (a.reset != nullptr && a.reset[b] != 0) ? 1.0f : 0.0f;
        ctl = make_float4(expm1f(c), cs, sn, rs);
        if (!kPerWarp) s_ctl = ctl;
    }
    if (kPerWarp) {
        ctl.x = __shfl_sync(0xffffffffu, ctl.x, 0);
        ctl.y = __shfl_sync(0xffffffffu, ctl.y, 0);
        ctl.z = __shfl_sync(0xffffffffu, ctl.z, 0);
        ctl.w = __shfl_sync(0xffffffffu, ctl.w, 0);
    } else {
        __syncthreads();
        ctl = s_ctl;
    }
    Ctl2 ct;
    ct.e = dup2(ctl.x);
    ct.c = dup2(ctl.y);
    ct.s = dup2(ctl.z);
    const bool reset = ctl.w != 0.f;

#pragma unroll
    for (int j = 0; j < kDecPairs; ++j) {
        const int m = m0 + j * mstep;
        if (m >= M) continue;
        const float4 z4 = zs[j];
        const f2x bre = bf2x(wre[j]), bim = bf2x(wim[j]);
        c2x z;
        if (reset) {
            z.re = bre;
            z.im = bim;
        } else {
            const ModePair k = load_modes(modes, nu, m);
            float n0, n1;
            up2(k.nu, n0, n1);
            const float em = fabsf(ctl.x);
            const Lam2 l = (fabsf(n0) * em < kPolyBound && fabsf(n1) * em < kPolyBound) ? samu_lambda2<true>(k, ct)
                                                                                      : samu_lambda2<false>(k, ct);
            const f2x zr = pk2(z4.x, z4.z), zi = pk2(z4.y, z4.w);
            z.re = fma2(l.re, zr, fma2(l.nim, zi, bre));
            z.im = fma2(l.re, zi, fma2(l.im, zr, bim));
        }
        float r0, r1, i0, i1;
        up2(z.re, r0, r1);
        up2(z.im, i0, i1);
        *reinterpret_cast<float4*>(a.state_out + (b * M + m) * 2) = make_float4(r0, i0, r1, i1);
        yrow[m / 2] = x2bf(z.re);
        yrow[(M + m) / 2] = x2bf(z.im);
        if (a.y32 != nullptr) {
            float* y32 = a.y32 + b * (size_t)D;
            *reinterpret_cast<float2*>(y32 + m) = make_float2(r0, r1);
            *reinterpret_cast<float2*>(y32 + M + m) = make_float2(i0, i1);
        }
    }
}

cudaError_t launch_samu_decode_prepare(const SamuDecodePrepArgs& args, cudaStream_t s) {
    const int M = args.D / 2;
    const unsigned blocks = 1 + (unsigned)((M + kDecThreads - 1) / kDecThreads);
    samu_decode_prepare_kernel<<<blocks, kDecThreads, 0, s>>>(args);
    return cudaGetLastError();
}

// CTAs per sequence: P >= 2 when B P still fits the CTAs resident at once
// (at most the mode-pair groups of T, and 8); otherwise one.
template <int T>
cudaError_t launch_step(SamuDecodeStepArgs a, cudaStream_t s) {
    // resident CTAs per device, asked once per device (a decode step is one
    // launch per token: no per-call queries)
    static std::atomic<long long> resident_cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    long long resident = resident_cache[dev].load(std::memory_order_relaxed);
    if (resident < 1) {
        int sms = 1, per = 1;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, samu_decode_step_kernel<T, true>, T, 0) !=
                cudaSuccess ||
            per < 1)
            per = 1;
        resident = (long long)sms * per;
        resident_cache[dev].store(resident, std::memory_order_relaxed);
    }
    const long long groups = (a.D / 4 + T - 1) / T;   // groups of T mode pairs
    const long long P = std::min<long long>({a.B > 0 ? resident / a.B : 1LL, groups, 8LL});
    if (P >= 2) {
        a.parts = (int)P;
        samu_decode_step_kernel<T, true><<<(unsigned)(a.B * P), T, 0, s>>>(a);
    } else {
        a.parts = 1;
        samu_decode_step_kernel<T, false><<<(unsigned)a.B, T, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_samu_decode_step(const SamuDecodeStepArgs& args, cudaStream_t s) {
    if (args.D <= 1024) return launch_step<128>(args, s);
    return launch_step<kDecThreads>(args, s);
}

}  // namespace lrs

// SAMU controller on sm_103a: FP64 parameter prep, fused controller forward,
// controller backward and the deterministic parameter reductions.
//
// Equations: SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比"), section 05:
// x~ = [x_sel; 1], w_hat = w/||w||, p = tanh(x~ . w_hat_phi), r = tanh(x~ . w_hat_r),
// q(r) = r/(1+r^2), d = tanh(a_phi)/sqrt(M) p, c = tanh(a_r)/sqrt(M) q(r);
// E = e^c, C = cos d, S = sin d once per token (reused by all M modes);
// backward: pbar = dbar tanh(a_phi)/sqrt(M), rbar = cbar tanh(a_r)/sqrt(M)
// (1-r^2)/(1+r^2)^2, the chain rule through tanh, the amplitudes and the
// direction normalisation, using the cached p, r; the per-token partials are
// reduced in a fixed order ("SAMU strengthened-baseline H800 report",
// "Reverse complex backward": deterministic FP32 second stage).
#include "kernels.cuh"

namespace lrs {

// ---------------------------------------------------------------------------
// Streaming layout shared by the controller forward and backward.
//
// Every streaming CTA owns a contiguous run of stages of cg.stage_tok tokens.
// Warp 0 is the producer: lane 0 copies each stage's x_sel rows (contiguous
// in memory) into a ring of cg.ring shared-memory slots with one 1-D bulk
// copy, and the warp does the per-token scalar work.  Warps 1..C are the
// consumers: thread (warp, lane) owns channels 8v .. 8v+7, v = 32 (warp-1) +
// lane, with its unit-direction weights in registers.
//
// Shared memory: ring[slot][token][D] BF16 | per-slot exchange buffer |
// mbarriers.
// ---------------------------------------------------------------------------
constexpr int kCtrlRingMax = 8;                 // ring slots (at most)
constexpr int kCtrlRingBytes = 192 * 1024;      // shared memory for the ring
constexpr int kCtrlMaxThreads = 32 * (1 + 16);   // D = 4096: 16 consumer warps
constexpr int kModeThreads = 32;    // active threads of a mode CTA

struct CtrlSmem {
    uint8_t* ring;
    float* xbuf;        // forward: partial dots [slot][consumer][32]; backward: float2 scalars [slot][token]
    uint64_t* full;     // x rows landed (producer arrival + bytes)
    uint64_t* ready;    // forward: partials written (consumers); backward: scalars written (producer)
    uint64_t* empty;    // backward: slot consumed (consumers)
};

// Bytes between consecutive x_sel rows in a ring slot: the backward keeps
// rows packed; the forward pads each row by 16 bytes so that the eight rows
// an ldmatrix reads fall in distinct banks.
__host__ __device__ inline size_t ctrl_row_bytes(int D, bool backward) { return 2 * (size_t)D + (backward ? 0 : 16); }

__host__ __device__ inline size_t ctrl_slot_bytes(const CtrlGeom& cg, int D, bool backward) {
    return (size_t)cg.stage_tok * ctrl_row_bytes(D, backward);
}

__host__ __device__ inline size_t ctrl_ring_bytes(const CtrlGeom& cg, int D, bool backward) {
    return (size_t)cg.ring * ctrl_slot_bytes(cg, D, backward);
}

__host__ __device__ inline size_t ctrl_xbuf_bytes(const CtrlGeom& cg, bool backward) {
    return backward ? (size_t)cg.max_cta_tok * 8 : (size_t)cg.ring * cg.consumers * 32 * 16;
}

__device__ __forceinline__ CtrlSmem ctrl_smem(uint8_t* base, const CtrlGeom& cg, int D, bool backward) {
    CtrlSmem sm;
    sm.ring = base;
    const size_t rb = ctrl_ring_bytes(cg, D, backward);
    sm.xbuf = reinterpret_cast<float*>(base + rb);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + rb + ((ctrl_xbuf_bytes(cg, backward) + 15) & ~size_t(15)));
    sm.full = bars;
    sm.ready = bars + cg.ring;
    sm.empty = bars + 2 * cg.ring;
    return sm;
}

// Stages [s0, s1) of the streaming CTA `cta`.
__device__ __forceinline__ void ctrl_stage_range(const CtrlGeom& cg, int cta, long long& s0, long long& s1) {
    s0 = cg.n_stages * cta / cg.n_ctas;
    s1 = cg.n_stages * (cta + 1) / cg.n_ctas;
}

// Producer lane 0: the rows of stage (token t0, n tokens) into ring slot
// `slot`, as one bulk copy (packed rows) or one per row (padded rows).
__device__ __forceinline__ void ctrl_issue(const CtrlSmem& sm, int slot, const uint4* x, long long t0, int n, int D,
                                           const CtrlGeom& cg, bool backward) {
    const uint32_t row = 2u * (uint32_t)D;
    uint8_t* dst = sm.ring + (size_t)slot * ctrl_slot_bytes(cg, D, backward);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x) + (size_t)t0 * row;
    fence_proxy_async();
    mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)n * row);
    if (backward) {
        bulk_load(dst, src, (uint32_t)n * row, &sm.full[slot]);
    } else {
        const size_t pitch = ctrl_row_bytes(D, false);
        for (int i = 0; i < n; ++i) bulk_load(dst + (size_t)i * pitch, src + (size_t)i * row, row, &sm.full[slot]);
    }
}

__device__ __forceinline__ void unpack8(const uint4 q, float (&x)[8]) {
    float2 f;
    f = bf2_to_f2(q.x); x[0] = f.x; x[1] = f.y;
    f = bf2_to_f2(q.y); x[2] = f.x; x[3] = f.y;
    f = bf2_to_f2(q.z); x[4] = f.x; x[5] = f.y;
    f = bf2_to_f2(q.w); x[6] = f.x; x[7] = f.y;
}

__device__ __forceinline__ void mode_constants(const float* __restrict__ nu, const float* __restrict__ theta,
                                               int M, float4* __restrict__ modes, int m) {
    if (m >= M) return;
    const double r = exp(-(double)nu[m]);
    double sn, cs;
    sincos((double)theta[m], &sn, &cs);
    const double re = r * cs, im = r * sn;
    const float hr = (float)re, hi = (float)im;
    modes[m] = make_float4(hr, hi, (float)(re - (double)hr), (float)(im - (double)hi));
}

// ---------------------------------------------------------------------------
// Controller forward, with the parameter preparation folded in.
//  - Mode CTAs (the first n_mode_ctas, 32 active threads each): the per-mode
//    transition constant lbar_m = e^{-nu_m} e^{i theta_m} as a double-float
//    (hi, lo) in FP64.
//  - Streaming CTAs: the norms ||w_phi||, ||w_r|| over all D+1 entries (FP32,
//    fixed-order tree, the same in every CTA).  The dot products x~ . w_hat of
//    a stage of 16 tokens are one tensor-core contraction [16 tokens x D] x
//    [D x 8]: consumer warp c takes the 16-channel k-steps 16c .. 16c+15
//    (mma.sync m16n8k16, BF16 operands, FP32 accumulation), A is the x_sel
//    rows in shared memory (ldmatrix), B holds per channel the exact
//    three-way BF16 split w_hat = hi + mid + lo of both directions in columns
//    0-2 (phi) and 3-5 (r), so each product is exact and the sum is FP32.
//    The producer adds the consumers' partial tiles and the three split
//    columns in a fixed order and evaluates p = tanh(s_phi), r = tanh(s_r),
//    q(r), d, c, and E - 1 = expm1(c), C = cos d, S = sin d, one token per
//    lane.  The first streaming CTA stores w_hat and the amplitude factors
//    for the backward.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// c += A B for one m16n8k16 tile (BF16 A row-major, B column-major, FP32 c).
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// w = hi + mid + lo with each part a BF16 value (exactly, up to 2^-24 |w|):
// every subtraction is exact.  part 0, 1 or 2.
__device__ __forceinline__ float bf16_part(float w, int part) {
    const float h = __bfloat162float(__float2bfloat16_rn(w));
    if (part == 0) return h;
    const float r1 = w - h;
    const float m = __bfloat162float(__float2bfloat16_rn(r1));
    if (part == 1) return m;
    return __bfloat162float(__float2bfloat16_rn(r1 - m));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) { return f2_to_bf2(lo, hi); }

constexpr int kCtrlKMax = 16;   // k-steps (16 channels each) per consumer warp

template <int N>
__device__ __forceinline__ void ctrl_fwd_consumer(const SamuCtrlFwdArgs& a, const CtrlSmem& sm, long long s0,
                                                  long long s1, int cw, int lane, float inv_phi, float inv_r) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    const int ks0 = kCtrlKMax * cw;
    const int nk = min(kCtrlKMax, D / 16 - ks0);
    // B fragments: thread (g, t) holds column n = g at k = 2t, 2t+1 (b0) and
    // 2t+8, 2t+9 (b1) of every k-step
    const int g = lane >> 2, t = lane & 3;
    uint32_t bf[kCtrlKMax][2];
#pragma unroll
    for (int j = 0; j < kCtrlKMax; ++j) {
        bf[j][0] = 0u;
        bf[j][1] = 0u;
        if (j < nk && g < 6) {
            const float* w = g < 3 ? a.w_phi : a.w_r;
            const float inv = g < 3 ? inv_phi : inv_r;
            const int part = g % 3;
            const int c0 = 16 * (ks0 + j) + 2 * t;
            bf[j][0] = pack_bf16(bf16_part(w[c0] * inv, part), bf16_part(w[c0 + 1] * inv, part));
            bf[j][1] = pack_bf16(bf16_part(w[c0 + 8] * inv, part), bf16_part(w[c0 + 9] * inv, part));
        }
    }
    const uint32_t pitch = (uint32_t)ctrl_row_bytes(D, false);
    // ldmatrix row of this lane: token lane % 16 (rows past the stage's
    // token count repeat earlier rows; their results are not used), channel
    // half lane / 16 of each k-step
    const uint32_t lane_off = (uint32_t)((lane & 15) % N) * pitch + (uint32_t)(lane >> 4) * 16u;
    float4* xb = reinterpret_cast<float4*>(sm.xbuf);
    for (long long st = s0; st < s1; ++st) {
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        if (!mbar_wait_bounded(&sm.full[slot], (uint32_t)(k / cg.ring) & 1u)) {
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            return;
        }
        const uint32_t base = smem_u32(sm.ring + (size_t)slot * ctrl_slot_bytes(cg, D, false)) + lane_off;
        float ce[4] = {0.f, 0.f, 0.f, 0.f}, co[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kCtrlKMax; j += 2) {
            if (j < nk) {
                uint32_t fa[4];
                ldsm_x4(base + (uint32_t)(ks0 + j) * 32u, fa);
                mma_16816(ce, fa, bf[j][0], bf[j][1]);
            }
            if (j + 1 < nk) {
                uint32_t fa[4];
                ldsm_x4(base + (uint32_t)(ks0 + j + 1) * 32u, fa);
                mma_16816(co, fa, bf[j + 1][0], bf[j + 1][1]);
            }
        }
        xb[((size_t)slot * cg.consumers + cw) * 32 + lane] =
            make_float4(ce[0] + co[0], ce[1] + co[1], ce[2] + co[2], ce[3] + co[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ready[slot]);
    }
}

template <int N>
__device__ __forceinline__ void ctrl_fwd_producer(const SamuCtrlFwdArgs& a, const CtrlSmem& sm, long long s0,
                                                  long long s1, int lane, float bias_p, float bias_r, float k_phi,
                                                  float k_r) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    if (lane == 0)
        for (long long st = s0; st < s1 && st < s0 + cg.ring; ++st)
            ctrl_issue(sm, (int)(st - s0), a.x, st * N, (int)min((long long)N, a.BL - st * N), D, cg, false);
    const float4* xb = reinterpret_cast<const float4*>(sm.xbuf);
    // token i = lane (i < N): row i of the partial tiles is held by lanes
    // 4 (i mod 8) + {0, 1, 2} (columns {0,1}, {2,3}, {4,5}), in the first two
    // values for rows 0-7 and the last two for rows 8-15
    const int i = lane;
    const int src = 4 * (i & 7);
    const bool upper = (i & 8) != 0;
    for (long long st = s0; st < s1; ++st) {
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        const long long t0 = st * N;
        const int n = (int)min((long long)N, a.BL - t0);
        if (!mbar_wait_bounded(&sm.ready[slot], (uint32_t)(k / cg.ring) & 1u)) {
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            return;
        }
        float s_phi = 0.f, s_r = 0.f;
        if (i < N) {
            for (int c = 0; c < cg.consumers; ++c) {
                const float4* tile = xb + ((size_t)slot * cg.consumers + c) * 32 + src;
                const float4 p01 = tile[0], p23 = tile[1], p45 = tile[2];
                const float c0 = upper ? p01.z : p01.x, c1 = upper ? p01.w : p01.y;
                const float c2 = upper ? p23.z : p23.x, c3 = upper ? p23.w : p23.y;
                const float c4 = upper ? p45.z : p45.x, c5 = upper ? p45.w : p45.y;
                s_phi += (c0 + c1) + c2;
                s_r += (c3 + c4) + c5;
            }
        }
        __syncwarp();
        const long long nxt = st + cg.ring;
        if (lane == 0 && nxt < s1)
            ctrl_issue(sm, slot, a.x, nxt * N, (int)min((long long)N, a.BL - nxt * N), D, cg, false);
        if (i < n) {
            const long long t = t0 + i;
            const float p = tanhf(s_phi + bias_p);
            const float r = tanhf(s_r + bias_r);
            const float qr = r / (1.0f + r * r);
            const float d = k_phi * p;
            const float c = k_r * qr;
            float sn, cs;
            sincosf(d, &sn, &cs);
            const float rs = (a.reset != nullptr && a.reset[t] != 0) ? 1.0f : 0.0f;
            a.p[t] = p;
            a.r[t] = r;
            const float em1 = expm1f(c);
            a.ctrl[2 * t] = make_float4(em1, em1, cs, cs);
            a.ctrl[2 * t + 1] = make_float4(sn, sn, rs, rs);
        }
    }
}

__global__ void __launch_bounds__(kCtrlMaxThreads) samu_ctrl_fwd_kernel(SamuCtrlFwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float s_red[2][kCtrlMaxThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int D = a.D;
    const int M = D / 2;
    if ((int)blockIdx.x < a.n_mode_ctas) {
        if (tid < kModeThreads) mode_constants(a.nu, a.theta, M, a.modes, blockIdx.x * kModeThreads + tid);
        return;
    }
    const int cta = blockIdx.x - a.n_mode_ctas;
    const CtrlGeom& cg = a.cg;
    const int n = D + 1;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nwarps = blockDim.x >> 5;
    const CtrlSmem sm = ctrl_smem(smem_raw, cg, D, false);
    if (tid == 0) {
        for (int i = 0; i < cg.ring; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.ready[i], cg.consumers);
        }
    }

    // norms (FP32, fixed order: per-thread strided sum, warp tree, warp-order sum)
    float sp = 0.f, sr = 0.f;
    for (int j = tid; j < n; j += blockDim.x) {
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
    for (int w = 0; w < nwarps; ++w) {
        tp += s_red[0][w];
        tr += s_red[1][w];
    }
    const float nphi = sqrtf(tp), nr = sqrtf(tr);
    const float inv_phi = 1.0f / nphi, inv_r = 1.0f / nr;
    const float ta = tanhf(a.a_phi[0]), tra = tanhf(a.a_r[0]);
    const float ism = 1.0f / sqrtf((float)M);
    const float k_phi = ta * ism, k_r = tra * ism;
    if (cta == 0) {
        for (int j = tid; j < n; j += blockDim.x) {
            a.wh[j] = a.w_phi[j] * inv_phi;
            a.wh[n + j] = a.w_r[j] * inv_r;
        }
        for (int j = tid; j < a.n_counters; j += blockDim.x) a.counters[j] = 0u;
        if (tid == 0) {
            a.misc[0] = k_phi;
            a.misc[1] = k_r;
            a.misc[2] = nphi;
            a.misc[3] = nr;
            a.misc[4] = ta;
            a.misc[5] = tra;
            a.misc[6] = ism;
        }
    }
    long long s0, s1;
    ctrl_stage_range(cg, cta, s0, s1);
    if (warp == 0) {
        const float bias_p = a.w_phi[D] * inv_phi, bias_r = a.w_r[D] * inv_r;
        if (cg.stage_tok == 16)
            ctrl_fwd_producer<16>(a, sm, s0, s1, lane, bias_p, bias_r, k_phi, k_r);
        else
            ctrl_fwd_producer<8>(a, sm, s0, s1, lane, bias_p, bias_r, k_phi, k_r);
    } else {
        if (cg.stage_tok == 16)
            ctrl_fwd_consumer<16>(a, sm, s0, s1, warp - 1, lane, inv_phi, inv_r);
        else
            ctrl_fwd_consumer<8>(a, sm, s0, s1, warp - 1, lane, inv_phi, inv_r);
    }
}

// ---------------------------------------------------------------------------
// Controller backward.  First, every thread of the CTA takes tokens of the
// CTA's range in turn:  dbar = sum over the mode groups of the Im-kappa
// partials, cbar = E * sum of the (-nu Re kappa) partials (E = e^c);
// pbar = dbar tanh(a_phi)/sqrt(M); rbar = cbar tanh(a_r)/sqrt(M)
// (1 - r^2)/(1 + r^2)^2; through tanh: sbar_phi = pbar (1 - p^2),
// sbar_r = rbar (1 - r^2), kept in shared memory for the whole range; the
// bias column (sum sbar) and the amplitude partials (sum dbar p,
// sum cbar q(r)) are reduced over the CTA in a fixed order.  Then the
// producer streams the x_sel rows and the consumers, per token and channel,
// form dx_sel = sbar_phi w_hat_phi[:D] + sbar_r w_hat_r[:D] and accumulate
// dw_hat += sbar x~.  One partial row per CTA.
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void ctrl_bwd_producer(const SamuCtrlBwdArgs& a, const CtrlSmem& sm, long long s0,
                                                  long long s1, int lane) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    if (lane != 0) return;
    for (long long st = s0; st < s1; ++st) {
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        const long long t0 = st * N;
        const int n = (int)min((long long)N, a.BL - t0);
        if (k >= cg.ring && !mbar_wait_bounded(&sm.empty[slot], (uint32_t)(k / cg.ring - 1) & 1u)) {
            atomicOr(a.status, kStatusTimeout);
            return;
        }
        ctrl_issue(sm, slot, a.x, t0, n, D, cg, true);
    }
}

template <int N>
__device__ __forceinline__ void ctrl_bwd_consumer(const SamuCtrlBwdArgs& a, const CtrlSmem& sm, long long s0,
                                                  long long s1, int cw, int lane, int cta) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    const int vecs = D / 8;
    const int v_idx = 32 * cw + lane;
    const bool col_ok = v_idx < vecs;
    float wp[8], wr[8], accp[8], accr[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        wp[c] = col_ok ? a.wh[8 * v_idx + c] : 0.f;
        wr[c] = col_ok ? a.wh[(D + 1) + 8 * v_idx + c] : 0.f;
        accp[c] = 0.f;
        accr[c] = 0.f;
    }
    const float2* sc = reinterpret_cast<const float2*>(sm.xbuf);
    for (long long st = s0; st < s1; ++st) {
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        const long long t0 = st * N;
        const int n = (int)min((long long)N, a.BL - t0);
        if (!mbar_wait_bounded(&sm.full[slot], (uint32_t)(k / cg.ring) & 1u)) {
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            return;
        }
        if (col_ok) {
            const uint4* rows = reinterpret_cast<const uint4*>(sm.ring + (size_t)slot * N * 2 * D);
            const float2* scs = sc + (size_t)k * N;
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                float x[8];
                unpack8(rows[(size_t)i * vecs + v_idx], x);
                const float2 s = scs[i];
                float dx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    dx[c] = fmaf(s.x, wp[c], s.y * wr[c]);
                    accp[c] = fmaf(s.x, x[c], accp[c]);
                    accr[c] = fmaf(s.y, x[c], accr[c]);
                }
                const long long t = t0 + i;
                if (a.grad_fp32) {
                    float4* o = reinterpret_cast<float4*>(a.dx) + (t * vecs + v_idx) * 2;
                    __stcs(o, make_float4(dx[0], dx[1], dx[2], dx[3]));
                    __stcs(o + 1, make_float4(dx[4], dx[5], dx[6], dx[7]));
                } else {
                    uint4 o;
                    o.x = f2_to_bf2(dx[0], dx[1]);
                    o.y = f2_to_bf2(dx[2], dx[3]);
                    o.z = f2_to_bf2(dx[4], dx[5]);
                    o.w = f2_to_bf2(dx[6], dx[7]);
                    __stcs(reinterpret_cast<uint4*>(a.dx) + t * vecs + v_idx, o);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    if (col_ok) {
        float* row = a.dwh_part + (size_t)cta * 2 * (D + 1);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            row[8 * v_idx + c] = accp[c];
            row[(D + 1) + 8 * v_idx + c] = accr[c];
        }
    }
}

__global__ void __launch_bounds__(kCtrlMaxThreads) samu_ctrl_bwd_kernel(SamuCtrlBwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float4 s_red[kCtrlMaxThreads / 32];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int cta = blockIdx.x;
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    const CtrlSmem sm = ctrl_smem(smem_raw, cg, D, true);
    if (tid == 0) {
        for (int i = 0; i < cg.ring; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], cg.consumers);
        }
    }
    long long s0, s1;
    ctrl_stage_range(cg, cta, s0, s1);
    const long long tb = s0 * cg.stage_tok;
    const long long te = min(a.BL, s1 * cg.stage_tok);

    // per-token scalars of the whole range, and the bias / amplitude partials
    const float k_phi = a.misc[0];
    const float k_r = a.misc[1];
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);   // sum sbar_phi, sum sbar_r, sum dbar p, sum cbar q(r)
    float2* sc = reinterpret_cast<float2*>(sm.xbuf);
    for (long long t = tb + tid; t < te; t += blockDim.x) {
        const float2* kp = a.kpart + t * a.n_groups;
        float dbar = 0.f, ebar = 0.f;
#pragma unroll 8
        for (int g = 0; g < a.n_groups; ++g) {
            const float2 v = __ldcs(kp + g);
            dbar += v.x;
            ebar += v.y;
        }
        const float E = 1.0f + a.ctrl[2 * t].x;   // the control word starts with E - 1
        const float p = a.p[t];
        const float r = a.r[t];
        const float cbar = ebar * E;
        const float opr = 1.0f + r * r;
        const float pbar = dbar * k_phi;
        const float rbar = cbar * k_r * (1.0f - r * r) / (opr * opr);
        const float2 s = make_float2(pbar * (1.0f - p * p), rbar * (1.0f - r * r));
        sc[t - tb] = s;
        part.x += s.x;
        part.y += s.y;
        part.z = fmaf(dbar, p, part.z);
        part.w = fmaf(cbar, r / opr, part.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        part.x += __shfl_xor_sync(0xffffffffu, part.x, o);
        part.y += __shfl_xor_sync(0xffffffffu, part.y, o);
        part.z += __shfl_xor_sync(0xffffffffu, part.z, o);
        part.w += __shfl_xor_sync(0xffffffffu, part.w, o);
    }
    if (lane == 0) s_red[warp] = part;
    __syncthreads();
    if (tid == 0) {
        float4 t4 = s_red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
            t4.x += s_red[w].x;
            t4.y += s_red[w].y;
            t4.z += s_red[w].z;
            t4.w += s_red[w].w;
        }
        float* row = a.dwh_part + (size_t)cta * 2 * (D + 1);
        row[D] = t4.x;
        row[(D + 1) + D] = t4.y;
        a.amp_part[cta] = make_float2(t4.z, t4.w);
    }
    if (warp == 0) {
        if (cg.stage_tok == 16)
            ctrl_bwd_producer<16>(a, sm, s0, s1, lane);
        else
            ctrl_bwd_producer<8>(a, sm, s0, s1, lane);
    } else {
        if (cg.stage_tok == 16)
            ctrl_bwd_consumer<16>(a, sm, s0, s1, warp - 1, lane, cta);
        else
            ctrl_bwd_consumer<8>(a, sm, s0, s1, warp - 1, lane, cta);
    }
}

// ---------------------------------------------------------------------------
// Parameter reductions (fixed order, deterministic), one launch:
//  - CTAs [0, ceil(M/32)): 32 modes each; warp w sums the per-segment
//    (dnu, dtheta) rows w, w+32, ...; the 32 warp sums are added in order;
//  - the next 2*ceil((D+1)/32) CTAs: 32 columns of dw_hat_phi or dw_hat_r
//    each, summed the same way over the controller-backward partial rows
//    (one per controller-backward CTA);
//  - the CTA that arrives last (threadfence + counter) computes the
//    unit-direction projection dw = (dw_hat - w_hat (w_hat . dw_hat)) / ||w||
//    and the amplitude gradients da = (sum of partials) / sqrt(M) (1 - tanh(a)^2),
//    and clears the counter for the next call.
// ---------------------------------------------------------------------------
constexpr int kParamWarps = 32;
constexpr int kParamThreads = kParamWarps * 32;

// Block-wide sum of four values, fixed order; every thread gets the totals.
__device__ __forceinline__ float4 block_sum4(float4 v, float4 (*s_w)[1]) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
    }
    if (lane == 0) s_w[warp][0] = v;
    __syncthreads();
    float4 t = s_w[0][0];
    for (int w = 1; w < kParamWarps; ++w) {
        const float4 u = s_w[w][0];
        t.x += u.x;
        t.y += u.y;
        t.z += u.z;
        t.w += u.w;
    }
    return t;
}

__global__ void __launch_bounds__(kParamThreads) samu_params_kernel(SamuParamArgs a) {
    __shared__ float2 s_red[kParamWarps][32];
    __shared__ float4 s_w[kParamWarps][1];
    __shared__ int s_last;
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int M = a.D / 2;
    const int n = a.D + 1;
    const int n_num = (M + 31) / 32;
    if ((int)blockIdx.x < n_num) {
        const int m = blockIdx.x * 32 + lane;
        const int rows = a.B * a.n_part;
        float2 sum = make_float2(0.f, 0.f);
        if (m < M) {
            int r = warp;
            for (; r + 3 * kParamWarps < rows; r += 4 * kParamWarps) {
                float2 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = __ldcg(a.numod + (size_t)(r + q * kParamWarps) * M + m);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sum.x += v[q].x;
                    sum.y += v[q].y;
                }
            }
            for (; r < rows; r += kParamWarps) {
                const float2 v = __ldcg(a.numod + (size_t)r * M + m);
                sum.x += v.x;
                sum.y += v.y;
            }
        }
        s_red[warp][lane] = sum;
        __syncthreads();
        if (warp == 0 && m < M) {
            float2 t = s_red[0][lane];
            for (int w = 1; w < kParamWarps; ++w) {
                t.x += s_red[w][lane].x;
                t.y += s_red[w][lane].y;
            }
            a.dnu[m] = t.x;
            a.dtheta[m] = t.y;
        }
    } else {
        const int cb = blockIdx.x - n_num;
        const int which = cb & 1;
        const int j = (cb >> 1) * 32 + lane;
        float sum = 0.f;
        if (j < n) {
            int r = warp;
            for (; r + 3 * kParamWarps < a.n_rows; r += 4 * kParamWarps) {
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = __ldcg(a.dwh_part + ((size_t)(r + q * kParamWarps) * 2 + which) * n + j);
#pragma unroll
                for (int q = 0; q < 4; ++q) sum += v[q];
            }
            for (; r < a.n_rows; r += kParamWarps) sum += __ldcg(a.dwh_part + ((size_t)r * 2 + which) * n + j);
        }
        s_red[warp][lane].x = sum;
        __syncthreads();
        if (warp == 0 && j < n) {
            float t = s_red[0][lane].x;
            for (int w = 1; w < kParamWarps; ++w) t += s_red[w][lane].x;
            a.dwh[(size_t)which * n + j] = t;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);   // w_hat . dw_hat (phi, r), amplitude sums (phi, r)
    for (int j = threadIdx.x; j < n; j += kParamThreads) {
        v.x = fmaf(a.wh[j], __ldcg(a.dwh + j), v.x);
        v.y = fmaf(a.wh[n + j], __ldcg(a.dwh + n + j), v.y);
    }
    for (int k = threadIdx.x; k < a.n_rows; k += kParamThreads) {
        const float2 u = __ldcg(a.amp_part + k);
        v.z += u.x;
        v.w += u.y;
    }
    const float4 t = block_sum4(v, s_w);
    const float nphi = a.misc[2];
    const float nr = a.misc[3];
    for (int j = threadIdx.x; j < n; j += kParamThreads) {
        a.dw_phi[j] = (__ldcg(a.dwh + j) - a.wh[j] * t.x) / nphi;
        a.dw_r[j] = (__ldcg(a.dwh + n + j) - a.wh[n + j] * t.y) / nr;
    }
    if (threadIdx.x == 0) {
        const float ta = a.misc[4], tr = a.misc[5], ism = a.misc[6];
        a.da_phi[0] = t.z * ism * (1.0f - ta * ta);
        a.da_r[0] = t.w * ism * (1.0f - tr * tr);
        *a.counter = 0u;
    }
}

namespace {

struct CtrlOcc {
    bool done = false;
    int sms = 0;
};
CtrlOcc g_ctrl_occ[64];

int ctrl_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    CtrlOcc& o = g_ctrl_occ[dev];
    if (!o.done) {
        int v = 0;
        o.sms = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 1;
        o.done = true;
    }
    return o.sms;
}

}  // namespace

CtrlGeom samu_ctrl_geom(long long BL, int D, bool backward) {
    CtrlGeom cg;
    // stages of 16 tokens (8 when 16 rows exceed 64 KB), as many slots as fit
    // in kCtrlRingBytes
    cg.stage_tok = 2 * D * 16 <= 64 * 1024 ? 16 : 8;
    int ring = (int)(kCtrlRingBytes / ((size_t)cg.stage_tok * ctrl_row_bytes(D, backward)));
    if (ring > kCtrlRingMax) ring = kCtrlRingMax;
    if (ring < 2) ring = 2;
    cg.ring = ring;
    cg.consumers = (D / 8 + 31) / 32;
    if (cg.consumers < 1) cg.consumers = 1;
    cg.threads = 32 * (1 + cg.consumers);
    cg.n_stages = (BL + cg.stage_tok - 1) / cg.stage_tok;
    {   // tokens of the longest CTA range: there are at least min(stages, SMs) CTAs
        const long long fewest = cg.n_stages < ctrl_sms() ? cg.n_stages : ctrl_sms();
        cg.max_cta_tok = (int)((cg.n_stages + fewest - 1) / fewest * cg.stage_tok);
    }
    const size_t xb = (ctrl_xbuf_bytes(cg, backward) + 15) & ~size_t(15);
    cg.smem = (int)(ctrl_ring_bytes(cg, D, backward) + xb + 3 * cg.ring * sizeof(uint64_t));
    int per_sm = (int)((227 * 1024) / (cg.smem + 1024));
    const int by_threads = 2048 / cg.threads;
    if (per_sm > by_threads) per_sm = by_threads;
    if (per_sm > 4) per_sm = 4;
    if (per_sm < 1) per_sm = 1;
    long long ctas = (long long)ctrl_sms() * per_sm;
    if (ctas > cg.n_stages) ctas = cg.n_stages;
    if (ctas > kCtrlRowsMax) ctas = kCtrlRowsMax;
    cg.n_ctas = (int)ctas;
    return cg;
}

cudaError_t launch_samu_ctrl_fwd(const SamuCtrlFwdArgs& args_in, cudaStream_t s, bool pdl) {
    SamuCtrlFwdArgs a = args_in;
    const int M = a.D / 2;
    a.n_mode_ctas = (M + kModeThreads - 1) / kModeThreads;
    a.cg = samu_ctrl_geom(a.BL, a.D, false);
    const cudaError_t e =
        cudaFuncSetAttribute(samu_ctrl_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, a.cg.smem);
    if (e != cudaSuccess) return e;
    return launch_ex(samu_ctrl_fwd_kernel, a.n_mode_ctas + a.cg.n_ctas, a.cg.threads, (size_t)a.cg.smem, s, pdl, a);
}

cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s, bool pdl) {
    const cudaError_t e =
        cudaFuncSetAttribute(samu_ctrl_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, args.cg.smem);
    if (e != cudaSuccess) return e;
    return launch_ex(samu_ctrl_bwd_kernel, args.cg.n_ctas, args.cg.threads, (size_t)args.cg.smem, s, pdl, args);
}

cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s, bool pdl) {
    const int M = args.D / 2;
    const int blocks = (M + 31) / 32 + 2 * ((args.D + 1 + 31) / 32);
    return launch_ex(samu_params_kernel, blocks, kParamThreads, 0, s, pdl, args);
}

}  // namespace lrs

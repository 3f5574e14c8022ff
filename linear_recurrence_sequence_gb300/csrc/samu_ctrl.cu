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
#include <mutex>

#include "kernels.cuh"

namespace lrs {

// ---------------------------------------------------------------------------
// Streaming layout of the controller backward.
//
// Every CTA owns a contiguous run of stages of cg.stage_tok tokens.  Warp 0
// is the producer: lane 0 copies each stage's x_sel rows (contiguous in
// memory) into a ring of cg.ring shared-memory slots with one 1-D bulk copy.
// Warp 1 is the reducer (per-mode parameter sums).  Warps 2..C+1 are the
// consumers: thread (warp, lane) owns channels 8v .. 8v+7, v = 32 (warp-2) +
// lane, with its unit-direction weights in registers.
//
// Shared memory: ring[slot][token][D] BF16 | per-token scalars of the range |
// mbarriers.
// ---------------------------------------------------------------------------
constexpr int kCtrlRingMax = 8;                        // ring slots (at most)
constexpr size_t kCtrlBwdSmemMax = 200 * 1024;          // leaves room for the reduction CTAs
constexpr int kCtrlBwdMaxThreads = 32 * (2 + 14);       // 14 consumer warps + producer + reducer
constexpr int kCtrlBwdNarrowVecs = 32 * 14;             // 8-channel chunks with one chunk per consumer lane

struct CtrlSmem {
    uint8_t* ring;
    float* xbuf;        // float2 scalars [token of the range]
    uint64_t* full;     // x rows landed (producer arrival + bytes)
    uint64_t* empty;    // slot consumed (consumers)
};

__host__ __device__ inline size_t ctrl_slot_bytes(const CtrlGeom& cg, int D) {
    return (size_t)cg.stage_tok * 2 * (size_t)D;
}

__host__ __device__ inline size_t ctrl_ring_bytes(const CtrlGeom& cg, int D) { return (size_t)cg.ring * ctrl_slot_bytes(cg, D); }

__host__ __device__ inline size_t ctrl_xbuf_bytes(const CtrlGeom& cg) { return (size_t)cg.max_cta_tok * 8; }

__device__ __forceinline__ CtrlSmem ctrl_smem(uint8_t* base, const CtrlGeom& cg, int D) {
    CtrlSmem sm;
    sm.ring = base;
    const size_t rb = ctrl_ring_bytes(cg, D);
    sm.xbuf = reinterpret_cast<float*>(base + rb);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + rb + ((ctrl_xbuf_bytes(cg) + 15) & ~size_t(15)));
    sm.full = bars;
    sm.empty = bars + cg.ring;
    return sm;
}

// Stages [s0, s1) of the CTA `cta`.
__device__ __forceinline__ void ctrl_stage_range(const CtrlGeom& cg, int cta, long long& s0, long long& s1) {
    s0 = cg.n_stages * cta / cg.n_ctas;
    s1 = cg.n_stages * (cta + 1) / cg.n_ctas;
}

// Producer lane 0: the rows of stage (token t0, n tokens) into ring slot
// `slot` as one bulk copy.
__device__ __forceinline__ void ctrl_issue(const CtrlSmem& sm, int slot, const uint4* x, long long t0, int n, int D,
                                           const CtrlGeom& cg) {
    const uint32_t row = 2u * (uint32_t)D;
    uint8_t* dst = sm.ring + (size_t)slot * ctrl_slot_bytes(cg, D);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x) + (size_t)t0 * row;
    fence_proxy_async();
    mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)n * row);
    bulk_load(dst, src, (uint32_t)n * row, &sm.full[slot]);
}

__device__ __forceinline__ void unpack8(const uint4 q, float (&x)[8]) {
    float2 f;
    f = bf2_to_f2(q.x); x[0] = f.x; x[1] = f.y;
    f = bf2_to_f2(q.y); x[2] = f.x; x[3] = f.y;
    f = bf2_to_f2(q.z); x[4] = f.x; x[5] = f.y;
    f = bf2_to_f2(q.w); x[6] = f.x; x[7] = f.y;
}

// ---------------------------------------------------------------------------
// Controller forward, with the parameter preparation folded in.
//  - Every CTA stages the raw directions w_phi, w_r (first D entries) in
//    shared memory as one 80-byte block per 8-channel chunk {phi 0-7, r 0-7,
//    pad} and computes the norms ||w_phi||, ||w_r|| over all D+1 entries
//    (FP32: per-thread strided sums, warp xor tree, warp-order sum; the same
//    in every CTA).
//  - A warp takes groups of kCfTok consecutive tokens (group g, g + W, ...
//    for its global warp index g out of W).  Lane l owns the chunks l, l+32,
//    ... of every token of the group: 16-byte loads straight from x_sel (one
//    warp load = 512 contiguous bytes of one row), paired FP32 dot products
//    with the raw directions (even and odd channels summed apart, then
//    added), then a fixed-order reduce-scatter of the 2 kCfTok sums
//    across the lanes.  One lane per token scales by 1/||w||, adds the bias
//    entry and evaluates p = tanh(s_phi), r = tanh(s_r), q(r), d, c, and
//    E - 1 = expm1(c), C = cos d, S = sin d.
//  - The last ceil(M/32) warps of the grid (those with the fewest groups)
//    first compute the per-mode transition constants
//    lbar_m = e^{-nu_m} e^{i theta_m} as double-floats (hi, lo) in FP64.
//  - CTA 0 stores w_hat and the amplitude factors for the backward.
// ---------------------------------------------------------------------------
constexpr int kCfWarps = 8;
constexpr int kCfThreads = 32 * kCfWarps;
constexpr int kCfTok = 4;      // tokens per warp group
constexpr int kCfBatch = 4;    // chunks per lane per load batch
constexpr int kCfBlock = 5;    // float4 per staged weight chunk (80 bytes: conflict-free for 8 distinct chunks)

// Sums of the 8 channels of chunk q (BF16) against both staged directions,
// as paired FP32 (even and odd channels in the two halves of each pair).
__device__ __forceinline__ void dot8(const uint4 q, const float4* __restrict__ wb, f2x& sp, f2x& sr) {
    const float4 p0 = wb[0], p1 = wb[1], r0 = wb[2], r1 = wb[3];
    const f2x x0 = bf2x(q.x), x1 = bf2x(q.y), x2 = bf2x(q.z), x3 = bf2x(q.w);
    sp = fma2(x0, pk2(p0.x, p0.y), sp);
    sp = fma2(x1, pk2(p0.z, p0.w), sp);
    sp = fma2(x2, pk2(p1.x, p1.y), sp);
    sp = fma2(x3, pk2(p1.z, p1.w), sp);
    sr = fma2(x0, pk2(r0.x, r0.y), sr);
    sr = fma2(x1, pk2(r0.z, r0.w), sr);
    sr = fma2(x2, pk2(r1.x, r1.y), sr);
    sr = fma2(x3, pk2(r1.z, r1.w), sr);
}

// The per-token scalars from the two dot products (raw directions).
// Returns E - 1 and d of the token in em1_out, d_out and whether it is a
// segment start.
__device__ __forceinline__ bool ctrl_fwd_token(const SamuCtrlFwdArgs& a, long long t, float dp, float dr,
                                               float inv_phi, float inv_r, float bias_p, float bias_r, float k_phi,
                                               float k_r, float& em1_out, float& d_out) {
    const float p = tanhf(fmaf(dp, inv_phi, bias_p));
    const float r = tanhf(fmaf(dr, inv_r, bias_r));
    const float qr = r / (1.0f + r * r);
    const float d = k_phi * p;
    const float c = k_r * qr;
    float sn, cs;
    sincosf(d, &sn, &cs);
    a.p[t] = p;
    a.r[t] = r;
    const float em1 = expm1f(c);
    // R = -E, or +0 at a reset; d for the closed-form item transitions
    const bool rst = a.reset != nullptr && a.reset[t] != 0;
    const float rw = rst ? 0.0f : -(1.0f + em1);
    a.ctrl[2 * t] = make_float4(em1, em1, cs, cs);
    a.ctrl[2 * t + 1] = make_float4(sn, sn, rw, d);
    em1_out = em1;
    d_out = d;
    return rst;
}

__global__ void __launch_bounds__(kCfThreads, 2) samu_ctrl_fwd_kernel(SamuCtrlFwdArgs a) {
    extern __shared__ __align__(16) float4 wsm[];   // [D/8][kCfBlock]
    __shared__ float s_red[2][kCfWarps];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The call's status word starts at zero.  This kernel is the call's first
    // and an ordinary launch; the scan kernels record failures only after
    // their dependency wait, which ends once this kernel has completed.
    if (blockIdx.x == 0 && tid == 0 && a.status != nullptr) *a.status = 0u;
    const int D = a.D, M = D / 2, n = D + 1, nch = D / 8;
    const long long W = (long long)gridDim.x * kCfWarps;
    const long long gw = (long long)blockIdx.x * kCfWarps + warp;
    const long long n_items = (long long)a.B * samu_items_per_row(a.L);
    const int cpl = (nch + 31) / 32;   // chunks per lane

    // staged raw directions and the norms
    float sp = 0.f, sr = 0.f;
    for (int j = tid; j < n; j += kCfThreads) {
        const float x = a.w_phi[j], y = a.w_r[j];
        sp = fmaf(x, x, sp);
        sr = fmaf(y, y, sr);
        if (j < D) {
            float* blk = reinterpret_cast<float*>(wsm + (size_t)(j >> 3) * kCfBlock);
            blk[j & 7] = x;
            blk[8 + (j & 7)] = y;
        }
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
    for (int w = 0; w < kCfWarps; ++w) {
        tp += s_red[0][w];
        tr += s_red[1][w];
    }
    const float nphi = sqrtf(tp), nr = sqrtf(tr);
    const float inv_phi = 1.0f / nphi, inv_r = 1.0f / nr;
    const float ta = tanhf(a.a_phi[0]), tra = tanhf(a.a_r[0]);
    const float ism = 1.0f / sqrtf((float)M);
    const float k_phi = ta * ism, k_r = tra * ism;
    const float bias_p = a.w_phi[D] * inv_phi, bias_r = a.w_r[D] * inv_r;
    if (blockIdx.x == 0) {
        for (int j = tid; j < n; j += kCfThreads) {
            a.wh[j] = a.w_phi[j] * inv_phi;
            a.wh[n + j] = a.w_r[j] * inv_r;
        }
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
    {   // per-mode constants: the last warps of the grid, 32 modes each
        const long long nmw = (M + 31) / 32;
        const long long first = W > nmw ? W - nmw : 0;
        for (long long mw = gw - first; gw >= first && mw < nmw; mw += W - first) {
            const int m = (int)mw * 32 + lane;
            mode_constants(a.nu, a.theta, M, a.modes, m);
            mode_power_constants(a.nu, a.theta, M, kMapRows, a.modes + M, m);
        }
    }

    // Items of kMapRows tokens of each batch row (t = 0, 16, ... of the row),
    // one per warp at a time, as kMapRows / kCfTok groups of kCfTok tokens;
    // the item's record (G, cos D, sin D, max |E - 1| or not-simple) is
    // formed from the per-token scalars.
    const uint4* x = a.x;
    const int ipr = samu_items_per_row(a.L);
    for (long long it = gw; it < n_items; it += W) {
        const long long b = it / ipr;
        const int ii = (int)(it - b * ipr);
        const long long tb = b * a.L + (long long)ii * kMapRows;
        const long long te = b * a.L + min((long long)(ii + 1) * kMapRows, (long long)a.L);
        float iG = 0.f, iD = 0.f, iemax = 0.f;
        bool irst = false;
        // The scalars of a group (tanh, sincos, expm1 in one lane per token)
        // are formed after the next group's loads have been issued, so that
        // their latency overlaps the loads; the item's last group follows
        // the loop.
        float pend_p = 0.f, pend_r = 0.f;
        long long pend_t = -1;
        auto scalars = [&](float s_p, float s_r, long long tg) {
            const int k = lane >> 3;
            if ((lane & 7) == 0 && tg + k < te) {
                float em1, d;
                irst = ctrl_fwd_token(a, tg + k, s_p, s_r, inv_phi, inv_r, bias_p, bias_r, k_phi, k_r, em1, d) || irst;
                iG += em1;
                iD += d;
                iemax = fmaxf(iemax, fabsf(em1));
            }
        };
        for (long long t0 = tb; t0 < te; t0 += kCfTok) {
            f2x pacc[2 * kCfTok];   // {token k: phi, r} as even/odd-channel pairs
#pragma unroll
            for (int v = 0; v < 2 * kCfTok; ++v) pacc[v] = 0ull;
            for (int i0 = 0; i0 < cpl; i0 += kCfBatch) {
                uint4 xv[kCfBatch][kCfTok];
#pragma unroll
                for (int b4 = 0; b4 < kCfBatch; ++b4) {
                    const int c = lane + 32 * (i0 + b4);
#pragma unroll
                    for (int k = 0; k < kCfTok; ++k) {
                        const bool ok = i0 + b4 < cpl && c < nch && t0 + k < te;
                        xv[b4][k] = ok ? __ldg(x + (size_t)(t0 + k) * nch + c) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (i0 == 0 && pend_t >= 0) {   // the previous group's scalars under this group's first loads
                    scalars(pend_p, pend_r, pend_t);
                    pend_t = -1;
                }
#pragma unroll
                for (int b4 = 0; b4 < kCfBatch; ++b4) {
                    const int c = lane + 32 * (i0 + b4);
                    if (i0 + b4 < cpl && c < nch) {
                        const float4* wb = wsm + (size_t)c * kCfBlock;
#pragma unroll
                        for (int k = 0; k < kCfTok; ++k) dot8(xv[b4][k], wb, pacc[2 * k], pacc[2 * k + 1]);
                    }
                }
            }
            float acc[2 * kCfTok];
#pragma unroll
            for (int v = 0; v < 2 * kCfTok; ++v) {
                float lo, hi;
                up2(pacc[v], lo, hi);
                acc[v] = lo + hi;
            }
            // reduce-scatter of the 8 sums {token k: phi, r} over the lanes:
            // halving exchanges at distances 16, 8, 4 (lane bit b keeps the upper
            // half), then full sums at distances 2, 1.  Lane L ends with value
            // 4 bit4(L) + 2 bit3(L) + bit2(L): lanes 8k hold s_phi of token k,
            // lanes 8k + 4 its s_r.
#pragma unroll
            for (int o = 16, h = kCfTok; o >= 4; o >>= 1, h >>= 1) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int j = 0; j < h; ++j) {
                    const float send = up ? acc[j] : acc[j + h];
                    const float keep = up ? acc[j + h] : acc[j];
                    acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            float sv = acc[0];
            sv += __shfl_xor_sync(0xffffffffu, sv, 2);
            sv += __shfl_xor_sync(0xffffffffu, sv, 1);
            pend_p = sv;
            pend_r = __shfl_down_sync(0xffffffffu, sv, 4);
            pend_t = t0;
        }
        if (pend_t >= 0) scalars(pend_p, pend_r, pend_t);
        // lanes 0, 8, 16, 24 hold the sums over tokens k, k+4, ... of the
        // item: combined in a fixed order, ((l0 + l8) + (l16 + l24)), in lane 0
#pragma unroll
        for (int o = 8; o <= 16; o <<= 1) {
            iG += __shfl_xor_sync(0xffffffffu, iG, o);
            iD += __shfl_xor_sync(0xffffffffu, iD, o);
            iemax = fmaxf(iemax, __shfl_xor_sync(0xffffffffu, iemax, o));
            irst = __shfl_xor_sync(0xffffffffu, (int)irst, o) != 0 || irst;
        }
        if (lane == 0) {
            float sn, cs;
            sincosf(iD, &sn, &cs);
            const bool simple = !irst && te - tb == kMapRows;
            a.items[it] = make_float4(iG, cs, sn, simple ? iemax : -iemax - 1.0f);
        }
    }
}

// ---------------------------------------------------------------------------
// Controller backward.  Thread 0 starts the first x_sel copies; then every
// thread of the CTA takes tokens of the CTA's range in turn:  dbar = sum over the mode groups of the Im-kappa
// partials, cbar = E * sum of the (-nu Re kappa) partials (E = e^c);
// pbar = dbar tanh(a_phi)/sqrt(M); rbar = cbar tanh(a_r)/sqrt(M)
// (1 - r^2)/(1 + r^2)^2; through tanh: sbar_phi = pbar (1 - p^2),
// sbar_r = rbar (1 - r^2), kept in shared memory for the whole range; the
// bias column (sum sbar) and the amplitude partials (sum dbar p,
// sum cbar q(r)) are reduced over the CTA in a fixed order.  Then the
// producer streams the x_sel rows and the consumers, per token and channel,
// form dx_sel = sbar_phi w_hat_phi[:D] + sbar_r w_hat_r[:D] and accumulate
// dw_hat += sbar x~.  One partial row per CTA.  Meanwhile a reducer warp sums
// the reverse replay's per-segment (dnu, dtheta) rows for the CTA's share of
// the modes.  Warps: 0 producer, 1 reducer, 2.. consumers.
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void ctrl_bwd_producer(const SamuCtrlBwdArgs& a, const CtrlSmem& sm, long long s0,
                                                  long long s1, int lane) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    if (lane != 0) return;
    for (long long st = s0 + cg.ring; st < s1; ++st) {   // the first cg.ring stages went out at the start
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        const long long t0 = st * N;
        const int n = (int)min((long long)N, a.BL - t0);
        if (!mbar_wait_bounded(&sm.empty[slot], (uint32_t)(k / cg.ring - 1) & 1u)) {
            atomicOr(a.status, kStatusTimeout);
            break;
        }
        ctrl_issue(sm, slot, a.x, t0, n, D, cg);
    }
}

// Returns the thread's share of the partial row's projection on w_hat:
// (sum_c w_hat_phi[c] dw_hat_phi[c], sum_c w_hat_r[c] dw_hat_r[c]) over its
// channels: CH chunks of eight, columns 32 cw + lane + 32 consumers j.
template <int N, int CH>
__device__ __forceinline__ float2 ctrl_bwd_consumer(const SamuCtrlBwdArgs& a, const CtrlSmem& sm, long long s0,
                                                    long long s1, int cw, int lane, int cta) {
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    const int vecs = D / 8;
    int v_idx[CH];
    bool col_ok[CH];
    float wp[CH][8], wr[CH][8], accp[CH][8], accr[CH][8];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        v_idx[j] = 32 * (cw + j * cg.consumers) + lane;
        col_ok[j] = v_idx[j] < vecs;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            wp[j][c] = col_ok[j] ? a.wh[8 * v_idx[j] + c] : 0.f;
            wr[j][c] = col_ok[j] ? a.wh[(D + 1) + 8 * v_idx[j] + c] : 0.f;
            accp[j][c] = 0.f;
            accr[j][c] = 0.f;
        }
    }
    const float2* sc = reinterpret_cast<const float2*>(sm.xbuf);
    for (long long st = s0; st < s1; ++st) {
        const int k = (int)(st - s0);
        const int slot = k % cg.ring;
        const long long t0 = st * N;
        const int n = (int)min((long long)N, a.BL - t0);
        if (!mbar_wait_bounded(&sm.full[slot], (uint32_t)(k / cg.ring) & 1u)) {
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            break;   // status set; the CTA still reaches its barriers
        }
        const uint4* rows = reinterpret_cast<const uint4*>(sm.ring + (size_t)slot * N * 2 * D);
        const float2* scs = sc + (size_t)k * N;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (!col_ok[j]) continue;
#pragma unroll 4
            for (int i = 0; i < n; ++i) {
                float x[8];
                unpack8(rows[(size_t)i * vecs + v_idx[j]], x);
                const float2 s = scs[i];
                float dx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    dx[c] = fmaf(s.x, wp[j][c], s.y * wr[j][c]);
                    accp[j][c] = fmaf(s.x, x[c], accp[j][c]);
                    accr[j][c] = fmaf(s.y, x[c], accr[j][c]);
                }
                const long long t = t0 + i;
                if (a.grad_fp32) {
                    float4* o = reinterpret_cast<float4*>(a.dx) + (t * vecs + v_idx[j]) * 2;
                    __stcs(o, make_float4(dx[0], dx[1], dx[2], dx[3]));
                    __stcs(o + 1, make_float4(dx[4], dx[5], dx[6], dx[7]));
                } else {
                    uint4 o;
                    o.x = f2_to_bf2(dx[0], dx[1]);
                    o.y = f2_to_bf2(dx[2], dx[3]);
                    o.z = f2_to_bf2(dx[4], dx[5]);
                    o.w = f2_to_bf2(dx[6], dx[7]);
                    __stcs(reinterpret_cast<uint4*>(a.dx) + t * vecs + v_idx[j], o);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    const int ns = ctrl_half_stride(D);
    float4* row = reinterpret_cast<float4*>(a.dwh_part + (size_t)cta * 2 * ns);
    float2 d = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        if (col_ok[j]) {
            const int v = v_idx[j];
            row[2 * v] = make_float4(accp[j][0], accp[j][1], accp[j][2], accp[j][3]);
            row[2 * v + 1] = make_float4(accp[j][4], accp[j][5], accp[j][6], accp[j][7]);
            row[ns / 4 + 2 * v] = make_float4(accr[j][0], accr[j][1], accr[j][2], accr[j][3]);
            row[ns / 4 + 2 * v + 1] = make_float4(accr[j][4], accr[j][5], accr[j][6], accr[j][7]);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            d.x = fmaf(wp[j][c], accp[j][c], d.x);
            d.y = fmaf(wr[j][c], accr[j][c], d.y);
        }
    }
    return d;
}

// The reducer warp: the CTA's share of the modes, (dnu, dtheta) summed over
// the per-segment rows of the reverse replay.  Lanes split the rows of up to
// 32 modes into 32 / (modes) interleaved phases; the phase sums are added in
// phase order.  Fixed order throughout.
__device__ __forceinline__ void ctrl_bwd_modes(const SamuCtrlBwdArgs& a, int cta, int lane, float2* s_nm) {
    const int M = a.D / 2;
    const int m0 = (int)((long long)M * cta / a.cg.n_ctas), m1 = (int)((long long)M * (cta + 1) / a.cg.n_ctas);
    const int rows = a.numod_rows;
    for (int mc = m0; mc < m1; mc += 32) {
        const int nm = min(32, m1 - mc);
        const int q = 32 / nm;
        const int mi = lane % nm, ph = lane / nm;
        float2 acc = make_float2(0.f, 0.f);
        if (ph < q) {
            const float2* col = a.numod + mc + mi;
            int r = ph;
            for (; r + 3 * q < rows; r += 4 * q) {
                float2 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = __ldcg(col + (size_t)(r + u * q) * M);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x += v[u].x;
                    acc.y += v[u].y;
                }
            }
            for (; r < rows; r += q) {
                const float2 v = __ldcg(col + (size_t)r * M);
                acc.x += v.x;
                acc.y += v.y;
            }
        }
        s_nm[lane] = acc;
        __syncwarp();
        if (lane < nm) {
            float2 t = s_nm[lane];
            for (int p = 1; p < q; ++p) {
                t.x += s_nm[p * nm + lane].x;
                t.y += s_nm[p * nm + lane].y;
            }
            a.dnu[mc + lane] = t.x;
            a.dtheta[mc + lane] = t.y;
        }
        __syncwarp();
    }
}

// Block-wide sum of four values, fixed order; every thread gets the totals.
__device__ __forceinline__ float4 block_sum4(float4 v, float4* s_w) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
    }
    __syncthreads();
    if (lane == 0) s_w[warp] = v;
    __syncthreads();
    float4 t = s_w[0];
    for (int w = 1; w < nwarps; ++w) {
        const float4 u = s_w[w];
        t.x += u.x;
        t.y += u.y;
        t.z += u.z;
        t.w += u.w;
    }
    return t;
}

template <int CH>
__device__ __forceinline__ void ctrl_bwd_body(const SamuCtrlBwdArgs& a, uint8_t* smem_raw, float4* s_red, float2* s_nm) {
    pdl_trigger();
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int cta = blockIdx.x;
    const CtrlGeom& cg = a.cg;
    const int D = a.D;
    const CtrlSmem sm = ctrl_smem(smem_raw, cg, D);
    long long s0, s1;
    ctrl_stage_range(cg, cta, s0, s1);
    if (tid == 0) {   // the first stages go out before the dependency wait and the scalar phase
        for (int i = 0; i < cg.ring; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], cg.consumers);
        }
        for (long long st = s0; st < s1 && st < s0 + cg.ring; ++st) {
            const int nn = cg.stage_tok;
            ctrl_issue(sm, (int)(st - s0), a.x, st * nn, (int)min((long long)nn, a.BL - st * nn), D, cg);
        }
    }
    pdl_wait();   // x_sel is an input; everything below reads the earlier kernels' results
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
        const float2 sv = make_float2(pbar * (1.0f - p * p), rbar * (1.0f - r * r));
        sc[t - tb] = sv;
        part.x += sv.x;
        part.y += sv.y;
        part.z = fmaf(dbar, p, part.z);
        part.w = fmaf(cbar, r / opr, part.w);
    }
    const float4 tot = block_sum4(part, s_red);
    if (tid == 0) {
        float* row = a.dwh_part + (size_t)cta * 2 * ctrl_half_stride(D);
        row[D] = tot.x;
        row[ctrl_half_stride(D) + D] = tot.y;
        a.amp_part[cta] = make_float2(tot.z, tot.w);
    }
    float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);   // this thread's share of w_hat . (partial row)
    if (warp == 0) {
        if (cg.stage_tok == 16)
            ctrl_bwd_producer<16>(a, sm, s0, s1, lane);
        else
            ctrl_bwd_producer<8>(a, sm, s0, s1, lane);
        if (lane == 0) {   // the bias column
            dv.x = a.wh[D] * tot.x;
            dv.y = a.wh[2 * D + 1] * tot.y;
        }
    } else if (warp == 1) {
        ctrl_bwd_modes(a, cta, lane, s_nm);
    } else {
        const float2 d = cg.stage_tok == 16 ? ctrl_bwd_consumer<16, CH>(a, sm, s0, s1, warp - 2, lane, cta)
                                            : ctrl_bwd_consumer<8, CH>(a, sm, s0, s1, warp - 2, lane, cta);
        dv.x = d.x;
        dv.y = d.y;
    }
    // w_hat . (this CTA's partial row), fixed order; summed over the CTAs by
    // the parameter reduction (sum_r w_hat . row_r = w_hat . dw_hat)
    const float4 dt = block_sum4(dv, s_red);
    if (tid == 0) a.dot_part[cta] = make_float2(dt.x, dt.y);
}

// One chunk of eight channels per consumer lane (D <= 3584: at most 14
// consumer warps, 16 warps of 112 registers in all).
__global__ void __maxnreg__(112) samu_ctrl_bwd_kernel(SamuCtrlBwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float4 s_red[kCtrlBwdMaxThreads / 32];
    __shared__ float2 s_nm[32];
    ctrl_bwd_body<1>(a, smem_raw, s_red, s_nm);
}

// Two chunks per consumer lane for the widest rows (D up to 4096: 8 consumer
// warps, 10 warps in all); the per-lane accumulators double, so the register
// cap is higher (three warps of 168 registers per SM sub-partition).
__global__ void __maxnreg__(168) samu_ctrl_bwd_wide_kernel(SamuCtrlBwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ float4 s_red[kCtrlBwdMaxThreads / 32];
    __shared__ float2 s_nm[32];
    ctrl_bwd_body<2>(a, smem_raw, s_red, s_nm);
}

// ---------------------------------------------------------------------------
// Parameter-gradient reductions, one launch right after the controller
// backward (it waits for it with griddepcontrol.wait; its CTAs are small
// enough to be resident beside it).  The controller backward's partial rows
// (one per CTA; phi and r halves of ns = D+1 rounded up to 4 floats) are
// summed column by column: warps 1..7 of CTA c take float4 columns of the
// CTA's slice, lane l the rows l, l+32, ... in order, and the 32 lane sums
// are combined by a fixed xor butterfly.  Warp 0 meanwhile sums the CTAs'
// shares of w_hat . dw_hat (the same fixed order in every CTA), so each
// column is projected onto the unit sphere's tangent at once,
// dw = (dw_hat - w_hat (w_hat . dw_hat)) / ||w||; CTA 0 also forms the
// amplitude gradients da = (sum of partials) / sqrt(M) (1 - tanh(a)^2).
// ---------------------------------------------------------------------------
constexpr int kParamWarps = 8;
constexpr int kParamThreads = 32 * kParamWarps;
constexpr int kParamColWarps = kParamWarps - 1;

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ __forceinline__ float4 shfl_xor4(float4 v, int o) {
    v.x = __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y = __shfl_xor_sync(0xffffffffu, v.y, o);
    v.z = __shfl_xor_sync(0xffffffffu, v.z, o);
    v.w = __shfl_xor_sync(0xffffffffu, v.w, o);
    return v;
}

// Sum of src[0 .. count) over one warp: lane l adds elements l, l+32, ... in
// order, then a fixed xor butterfly; every lane gets the total.
__device__ __forceinline__ float2 warp_sum2(const float2* __restrict__ src, int count, int lane) {
    float2 acc = make_float2(0.f, 0.f);
    int i = lane;
    for (; i + 96 < count; i += 128) {
        float2 x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = __ldcg(src + i + 32 * q);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc.x += x[q].x;
            acc.y += x[q].y;
        }
    }
    for (; i < count; i += 32) {
        const float2 x = __ldcg(src + i);
        acc.x += x.x;
        acc.y += x.y;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
    }
    return acc;
}

// Column v (float4) of the [rows][nv] partial rows, summed over the rows as
// above; every lane gets the total.
__device__ __forceinline__ float4 column_sum(const float4* __restrict__ rows, int n_rows, int nv, int v, int lane) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int r = lane;
    for (; r + 224 < n_rows; r += 256) {
        float4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = __ldcg(rows + (size_t)(r + 32 * q) * nv + v);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc = add4(acc, x[q]);
    }
    {
        float4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            x[q] = r + 32 * q < n_rows ? __ldcg(rows + (size_t)(r + 32 * q) * nv + v) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (r + 32 * q < n_rows) acc = add4(acc, x[q]);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) acc = add4(acc, shfl_xor4(acc, o));
    return acc;
}

__device__ __forceinline__ void project_column(const SamuParamArgs& a, int v, float4 acc, float2 t, int n, int ns) {
    const float c[4] = {acc.x, acc.y, acc.z, acc.w};
    const float nphi = a.misc[2], nr = a.misc[3];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int j = 4 * v + e;   // position in the flattened [2][ns] row
        if (j < n)
            a.dw_phi[j] = (c[e] - a.wh[j] * t.x) / nphi;
        else if (j >= ns && j - ns < n)
            a.dw_r[j - ns] = (c[e] - a.wh[n + (j - ns)] * t.y) / nr;
    }
}

__global__ void __launch_bounds__(kParamThreads) samu_params_kernel(SamuParamArgs a) {
    __shared__ float2 s_t;
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.D + 1;
    const int ns = ctrl_half_stride(a.D);
    const int nv = ns / 2;   // float4 columns per row (2 ns floats)
    const int cta = blockIdx.x, nc = gridDim.x;
    const int v_lo = (int)((long long)nv * cta / nc), v_hi = (int)((long long)nv * (cta + 1) / nc);
    const float4* rows = reinterpret_cast<const float4*>(a.dwh_part);
    if (warp == 0) {
        const float2 t = warp_sum2(a.dot_part, a.n_rows, lane);
        if (lane == 0) s_t = t;
        if (cta == 0) {
            const float2 am = warp_sum2(a.amp_part, a.n_rows, lane);
            if (lane == 0) {
                const float ta = a.misc[4], tr = a.misc[5], ism = a.misc[6];
                a.da_phi[0] = am.x * ism * (1.0f - ta * ta);
                a.da_r[0] = am.y * ism * (1.0f - tr * tr);
            }
        }
    }
    const int v0 = v_lo + warp - 1;
    const bool own = warp > 0 && v0 < v_hi;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (own) acc0 = column_sum(rows, a.n_rows, nv, v0, lane);
    __syncthreads();
    const float2 t = s_t;
    if (own && lane == 0) project_column(a, v0, acc0, t, n, ns);
    if (warp > 0) {
        for (int v = v0 + kParamColWarps; v < v_hi; v += kParamColWarps) {
            const float4 acc = column_sum(rows, a.n_rows, nv, v, lane);
            if (lane == 0) project_column(a, v, acc, t, n, ns);
        }
    }
}

namespace {

struct CtrlOcc {
    bool done = false;
    int sms = 0;
};
CtrlOcc g_ctrl_occ[64];
std::mutex g_ctrl_occ_mutex;   // calls may come from several host threads

int ctrl_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    CtrlOcc& o = g_ctrl_occ[dev];
    std::lock_guard<std::mutex> lock(g_ctrl_occ_mutex);
    if (!o.done) {
        int v = 0;
        o.sms = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 1;
        o.done = true;
    }
    return o.sms;
}

}  // namespace

CtrlGeom samu_ctrl_geom(long long BL, int D) {
    CtrlGeom cg;
    // stages of 16 tokens, or 8 when 16 rows exceed 72 KB
    cg.stage_tok = 16 * 2 * (size_t)D <= 72 * 1024 ? 16 : 8;
    // one 8-channel chunk per consumer lane, two beyond 14 consumer warps
    cg.chunks = D / 8 <= kCtrlBwdNarrowVecs ? 1 : 2;
    cg.consumers = (D / 8 + 32 * cg.chunks - 1) / (32 * cg.chunks);
    if (cg.consumers < 1) cg.consumers = 1;
    cg.threads = 32 * (2 + cg.consumers);   // producer, reducer, consumers
    cg.n_stages = (BL + cg.stage_tok - 1) / cg.stage_tok;
    {   // tokens of the longest CTA range: there are at least min(stages, SMs) CTAs
        const long long fewest = cg.n_stages < ctrl_sms() ? cg.n_stages : ctrl_sms();
        cg.max_cta_tok = (int)((cg.n_stages + fewest - 1) / fewest * cg.stage_tok);
    }
    // as many ring slots (2 .. kCtrlRingMax) as fit with the scalar buffer and
    // the barriers
    for (cg.ring = kCtrlRingMax;; --cg.ring) {
        const size_t xb = (ctrl_xbuf_bytes(cg) + 15) & ~size_t(15);
        cg.smem = (int)(ctrl_ring_bytes(cg, D) + xb + 2 * cg.ring * sizeof(uint64_t));
        if ((size_t)cg.smem <= kCtrlBwdSmemMax || cg.ring == 2) break;
    }
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

cudaError_t launch_samu_ctrl_fwd(const SamuCtrlFwdArgs& a, cudaStream_t s, bool pdl) {
    // two CTAs per SM (one wave), fewer for short inputs; the warps past the
    // items form the per-mode constants
    const long long items = (long long)a.B * samu_items_per_row(a.L);
    long long ctas = (long long)ctrl_sms() * 2;
    const long long need = (items + (a.D / 2 + 31) / 32 + kCfWarps - 1) / kCfWarps;
    if (ctas > need) ctas = need;
    if (ctas < 1) ctas = 1;
    const size_t smem = (size_t)(a.D / 8) * kCfBlock * sizeof(float4);
    const cudaError_t e =
        cudaFuncSetAttribute(samu_ctrl_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_ex(samu_ctrl_fwd_kernel, (unsigned)ctas, kCfThreads, smem, s, pdl, a);
}

cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s, bool pdl) {
    // one float4 column per column warp
    const int nv = ctrl_half_stride(args.D) / 2;
    const int ctas = (nv + kParamColWarps - 1) / kParamColWarps;
    return launch_ex(samu_params_kernel, ctas, kParamThreads, 0, s, pdl, args);
}

cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s, bool pdl) {
    auto* fn = args.cg.chunks == 1 ? samu_ctrl_bwd_kernel : samu_ctrl_bwd_wide_kernel;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, args.cg.smem);
    if (e != cudaSuccess) return e;
    return launch_ex(fn, args.cg.n_ctas, args.cg.threads, (size_t)args.cg.smem, s, pdl, args);
}


}  // namespace lrs

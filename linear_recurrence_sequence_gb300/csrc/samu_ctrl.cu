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
// Controller forward, with the parameter preparation folded in.
//
// Grid = n_mode CTAs followed by controller CTAs.
//  - Mode CTAs (32 active threads each): the per-mode transition constant
//    lbar_m = e^{-nu_m} e^{i theta_m} as a double-float (hi, lo) in FP64; they
//    run alongside the streaming CTAs, off the critical path.
//  - Controller CTAs: the norms ||w_phi||, ||w_r|| over all D+1 entries (FP32,
//    fixed-order tree, recomputed identically by every CTA); each thread then
//    owns 8 consecutive channels with its 16 unit-direction weights in
//    registers, and the CTA walks its token range in batches of 8 tokens: one
//    16-byte load of x_sel per token per thread, 16 partial dot products per
//    thread, a 16-shuffle reduce-scatter inside each warp, a fixed-order sum
//    over the warps, and 8 threads evaluate p, r, q(r), d, c and the shared
//    E - 1 = expm1(c), C = cos d, S = sin d for the 8 tokens in parallel.
//    The first controller CTA stores w_hat and the amplitude factors for the
//    backward.
// ---------------------------------------------------------------------------
constexpr int kCfTok = 8;              // tokens per batch
constexpr int kModeThreads = 32;       // active threads of a mode CTA

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

__global__ void __launch_bounds__(512) samu_ctrl_fwd_kernel(SamuCtrlFwdArgs a) {
    __shared__ float s_red[2][512 / 32];
    __shared__ float s_part[512 / 32][2 * kCfTok];
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
    const int n = D + 1;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nwarps = blockDim.x >> 5;

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
    const int vecs = D / 8;
    const bool col_ok = tid < vecs;
    float wp[8], wr[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        wp[k] = col_ok ? a.w_phi[8 * tid + k] * inv_phi : 0.f;
        wr[k] = col_ok ? a.w_r[8 * tid + k] * inv_r : 0.f;
    }
    const float bias_p = a.w_phi[D] * inv_phi, bias_r = a.w_r[D] * inv_r;
    if (cta == 0) {
        for (int j = tid; j < n; j += blockDim.x) {
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

    const long long BL = a.BL;
    const long long per = (BL + a.n_tok_ctas - 1) / a.n_tok_ctas;
    const long long tb = (long long)cta * per;
    const long long te = min(BL, tb + per);
    for (long long t0 = tb; t0 < te; t0 += kCfTok) {
        uint4 q[kCfTok];
#pragma unroll
        for (int u = 0; u < kCfTok; ++u)
            q[u] = (col_ok && t0 + u < te) ? __ldcs(a.x + (t0 + u) * vecs + tid) : make_uint4(0u, 0u, 0u, 0u);
        float v[2 * kCfTok];   // v[2u] = phi partial of token u, v[2u+1] = r partial
#pragma unroll
        for (int u = 0; u < kCfTok; ++u) {
            float2 f;
            float ap = 0.f, ar = 0.f;
            f = bf2_to_f2(q[u].x); ap = fmaf(f.x, wp[0], ap); ap = fmaf(f.y, wp[1], ap); ar = fmaf(f.x, wr[0], ar); ar = fmaf(f.y, wr[1], ar);
            f = bf2_to_f2(q[u].y); ap = fmaf(f.x, wp[2], ap); ap = fmaf(f.y, wp[3], ap); ar = fmaf(f.x, wr[2], ar); ar = fmaf(f.y, wr[3], ar);
            f = bf2_to_f2(q[u].z); ap = fmaf(f.x, wp[4], ap); ap = fmaf(f.y, wp[5], ap); ar = fmaf(f.x, wr[4], ar); ar = fmaf(f.y, wr[5], ar);
            f = bf2_to_f2(q[u].w); ap = fmaf(f.x, wp[6], ap); ap = fmaf(f.y, wp[7], ap); ar = fmaf(f.x, wr[6], ar); ar = fmaf(f.y, wr[7], ar);
            v[2 * u] = ap;
            v[2 * u + 1] = ar;
        }
        // reduce-scatter of 16 values over the warp: after it, lanes 2i and
        // 2i+1 both hold the warp sum of value sel(i)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const bool hi = lane & 16;
            const float send = hi ? v[k] : v[k + 8];
            const float keep = hi ? v[k + 8] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool hi = lane & 8;
            const float send = hi ? v[k] : v[k + 4];
            const float keep = hi ? v[k + 4] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool hi = lane & 4;
            const float send = hi ? v[k] : v[k + 2];
            const float keep = hi ? v[k + 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
            const bool hi = lane & 2;
            const float send = hi ? v[0] : v[1];
            const float keep = hi ? v[1] : v[0];
            v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        if ((lane & 1) == 0) {
            const int sel = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
            s_part[warp][sel] = v[0];
        }
        __syncthreads();
        if (tid < kCfTok && t0 + tid < te) {
            const long long t = t0 + tid;
            float s_phi = 0.f, s_r = 0.f;
            for (int w = 0; w < nwarps; ++w) {
                s_phi += s_part[w][2 * tid];
                s_r += s_part[w][2 * tid + 1];
            }
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
            a.ctrl[t] = make_float4(expm1f(c), cs, sn, rs);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Controller backward.  A fixed grid of kCtrlBwdCtas CTAs, each owning a
// contiguous token range, processed in blocks of kCbTokBlock tokens; the CTA
// is two halves, each half owning one half of every block, and within a half
// each thread owns 8 consecutive channels.
// Per token:  dbar = sum_slices Im-kappa partials, cbar = E * sum_slices
// (-nu Re kappa) partials (E = e^c);  pbar = dbar tanh(a_phi)/sqrt(M);
// rbar = cbar tanh(a_r)/sqrt(M) (1 - r^2)/(1 + r^2)^2;  through tanh:
// sbar_phi = pbar (1 - p^2), sbar_r = rbar (1 - r^2);
// dx_sel = sbar_phi w_hat_phi[:D] + sbar_r w_hat_r[:D];
// dw_hat += sbar x~ (per-half partial rows, bias column included);
// amplitude partials sum dbar p and sum cbar q(r).
// ---------------------------------------------------------------------------
constexpr int kCbTokBlock = 128;
constexpr int kCbUnroll = 2;

__global__ void __launch_bounds__(512, 2) samu_ctrl_bwd_kernel(SamuCtrlBwdArgs a) {
    __shared__ float s_sphi[kCbTokBlock];
    __shared__ float s_sr[kCbTokBlock];
    __shared__ float s_red[4][kCbTokBlock];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x;
    const int D = a.D;
    const int vecs = D / 8;
    const int cols = max((vecs + 31) / 32 * 32, kCbTokBlock / 2);   // threads per half
    const int halves = blockDim.x / cols;                           // 1 or 2
    const int half = tid / cols;
    const int col = tid - half * cols;
    const long long BL = (long long)a.B * a.L;
    const long long per = (BL + kCtrlBwdCtas - 1) / kCtrlBwdCtas;
    const long long tb = (long long)blockIdx.x * per;
    const long long te = min(BL, tb + per);
    const float k_phi = a.misc[0];
    const float k_r = a.misc[1];
    const bool col_ok = col < vecs;

    float wp[8], wr[8], accp[8], accr[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        wp[k] = col_ok ? a.wh[8 * col + k] : 0.f;
        wr[k] = col_ok ? a.wh[(D + 1) + 8 * col + k] : 0.f;
        accp[k] = 0.f;
        accr[k] = 0.f;
    }
    float bias_p = 0.f, bias_r = 0.f, amp_p = 0.f, amp_r = 0.f;   // threads < kCbTokBlock

    for (long long blk = tb; blk < te; blk += kCbTokBlock) {
        const int nb = (int)min((long long)kCbTokBlock, te - blk);
        if (tid < nb) {
            const long long t = blk + tid;
            const float2* kp = a.kpart + t * a.n_groups;
            float dbar = 0.f, ebar = 0.f;
            for (int s2 = 0; s2 < a.n_groups; ++s2) {
                const float2 v = kp[s2];
                dbar += v.x;
                ebar += v.y;
            }
            const float E = 1.0f + a.ctrl[t].x;   // ctrl.x holds E - 1
            const float p = a.p[t];
            const float r = a.r[t];
            const float cbar = ebar * E;
            const float opr = 1.0f + r * r;
            const float pbar = dbar * k_phi;
            const float rbar = cbar * k_r * (1.0f - r * r) / (opr * opr);
            const float sp = pbar * (1.0f - p * p);
            const float sr = rbar * (1.0f - r * r);
            s_sphi[tid] = sp;
            s_sr[tid] = sr;
            bias_p += sp;
            bias_r += sr;
            amp_p = fmaf(dbar, p, amp_p);
            amp_r = fmaf(cbar, r / opr, amp_r);
        }
        __syncthreads();
        const int h0 = halves == 2 ? (nb + 1) / 2 : nb;
        const int i0 = half == 0 ? 0 : h0;
        const int i1 = half == 0 ? h0 : nb;
        if (col_ok) {
            for (int i = i0; i < i1; i += kCbUnroll) {
                uint4 q[kCbUnroll];
#pragma unroll
                for (int u = 0; u < kCbUnroll; ++u)
                    q[u] = (i + u < i1) ? __ldcs(a.x + (blk + i + u) * vecs + col) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < kCbUnroll; ++u) {
                    if (i + u < i1) {
                        const long long t = blk + i + u;
                        const float sp = s_sphi[i + u];
                        const float sr = s_sr[i + u];
                        float xv[8];
                        float2 f;
                        f = bf2_to_f2(q[u].x); xv[0] = f.x; xv[1] = f.y;
                        f = bf2_to_f2(q[u].y); xv[2] = f.x; xv[3] = f.y;
                        f = bf2_to_f2(q[u].z); xv[4] = f.x; xv[5] = f.y;
                        f = bf2_to_f2(q[u].w); xv[6] = f.x; xv[7] = f.y;
                        float dx[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            dx[k] = fmaf(sp, wp[k], sr * wr[k]);
                            accp[k] = fmaf(sp, xv[k], accp[k]);
                            accr[k] = fmaf(sr, xv[k], accr[k]);
                        }
                        if (a.grad_fp32) {
                            float4* o = reinterpret_cast<float4*>(a.dx) + (t * vecs + col) * 2;
                            __stcs(o, make_float4(dx[0], dx[1], dx[2], dx[3]));
                            __stcs(o + 1, make_float4(dx[4], dx[5], dx[6], dx[7]));
                        } else {
                            uint4 o;
                            o.x = f2_to_bf2(dx[0], dx[1]);
                            o.y = f2_to_bf2(dx[2], dx[3]);
                            o.z = f2_to_bf2(dx[4], dx[5]);
                            o.w = f2_to_bf2(dx[6], dx[7]);
                            __stcs(reinterpret_cast<uint4*>(a.dx) + t * vecs + col, o);
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    // partial rows: (cta, half); a single-half CTA leaves its second row zero
    float* part = a.dwh_part + ((size_t)blockIdx.x * 2 + half) * 2 * (D + 1);
    if (halves == 1) {
        float* other = a.dwh_part + ((size_t)blockIdx.x * 2 + 1) * 2 * (D + 1);
        for (int j = tid; j < 2 * (D + 1); j += blockDim.x) other[j] = 0.f;
    }
    if (col_ok) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            part[8 * col + k] = accp[k];
            part[(D + 1) + 8 * col + k] = accr[k];
        }
    }
    // fixed-order tree over the token-scalar threads for the bias column and amplitudes
    if (tid < kCbTokBlock) {
        s_red[0][tid] = bias_p;
        s_red[1][tid] = bias_r;
        s_red[2][tid] = amp_p;
        s_red[3][tid] = amp_r;
    }
    __syncthreads();
    for (int s2 = kCbTokBlock / 2; s2 > 0; s2 >>= 1) {
        if (tid < s2) {
#pragma unroll
            for (int q = 0; q < 4; ++q) s_red[q][tid] += s_red[q][tid + s2];
        }
        __syncthreads();
    }
    if (tid == 0) {
        float* p0 = a.dwh_part + (size_t)blockIdx.x * 2 * 2 * (D + 1);          // half-0 row
        float* p1 = p0 + 2 * (D + 1);                                           // half-1 row
        p0[D] = s_red[0][0];
        p0[(D + 1) + D] = s_red[1][0];
        p1[D] = 0.f;
        p1[(D + 1) + D] = 0.f;
        a.amp_part[blockIdx.x] = make_float2(s_red[2][0], s_red[3][0]);
    }
}

// ---------------------------------------------------------------------------
// Parameter reductions (fixed order, deterministic), one launch:
//  - CTAs [0, ceil(M/32)): 32 modes each; warp w sums the per-segment
//    (dnu, dtheta) rows w, w+32, ...; the 32 warp sums are added in order;
//  - the next 2*ceil((D+1)/32) CTAs: 32 columns of dw_hat_phi or dw_hat_r
//    each, summed the same way over the controller-backward partial rows;
//  - the CTA that arrives last (threadfence + counter) computes the
//    unit-direction projection dw = (dw_hat - w_hat (w_hat . dw_hat)) / ||w||
//    and the amplitude gradients da = (sum of partials) / sqrt(M) (1 - tanh(a)^2),
//    and clears the counter for the next call.
// ---------------------------------------------------------------------------
constexpr int kParamWarps = 32;
constexpr int kParamThreads = kParamWarps * 32;
constexpr int kColRows = 2 * kCtrlBwdCtas;   // (CTA, token half) partial rows

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
            for (; r + 3 * kParamWarps < kColRows; r += 4 * kParamWarps) {
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = __ldcg(a.dwh_part + ((size_t)(r + q * kParamWarps) * 2 + which) * n + j);
#pragma unroll
                for (int q = 0; q < 4; ++q) sum += v[q];
            }
            for (; r < kColRows; r += kParamWarps) sum += __ldcg(a.dwh_part + ((size_t)r * 2 + which) * n + j);
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
    for (int k = threadIdx.x; k < kCtrlBwdCtas; k += kParamThreads) {
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

cudaError_t launch_samu_ctrl_fwd(const SamuCtrlFwdArgs& args_in, cudaStream_t s, bool pdl) {
    SamuCtrlFwdArgs a = args_in;
    const int M = a.D / 2;
    int cols = ((a.D / 8) + 31) / 32 * 32;
    if (cols < 64) cols = 64;
    a.n_mode_ctas = (M + kModeThreads - 1) / kModeThreads;
    const long long want = (a.BL + kCfTok - 1) / kCfTok;
    a.n_tok_ctas = (int)(want < 152LL * 4 ? want : 152LL * 4);
    return launch_ex(samu_ctrl_fwd_kernel, a.n_mode_ctas + a.n_tok_ctas, cols, 0, s, pdl, a);
}

cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s, bool pdl) {
    int cols = ((args.D / 8) + 31) / 32 * 32;
    if (cols < kCbTokBlock / 2) cols = kCbTokBlock / 2;
    const int threads = 2 * cols <= 512 ? 2 * cols : cols;   // two token halves when they fit
    return launch_ex(samu_ctrl_bwd_kernel, kCtrlBwdCtas, threads, 0, s, pdl, args);
}

cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s, bool pdl) {
    const int M = args.D / 2;
    const int blocks = (M + 31) / 32 + 2 * ((args.D + 1 + 31) / 32);
    return launch_ex(samu_params_kernel, blocks, kParamThreads, 0, s, pdl, args);
}

}  // namespace lrs

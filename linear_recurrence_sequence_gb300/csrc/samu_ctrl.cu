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
// Prep (FP64, once per forward).  CTA 0: unit directions w_hat = w / ||w||
// (norm over all D+1 entries) and the amplitude factors tanh(a)/sqrt(M).
// CTAs 1..: the per-mode transition constant lbar_m = e^{-nu_m} e^{i theta_m}
// as a double-float (hi, lo), one mode per thread.  Small CTAs spread the
// FP64 work over many SMs.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 32;

__global__ void __launch_bounds__(kPrepThreads) samu_prep_kernel(
    const float* __restrict__ w_phi, const float* __restrict__ w_r, const float* __restrict__ a_phi,
    const float* __restrict__ a_r, const float* __restrict__ nu, const float* __restrict__ theta, int D,
    float* __restrict__ wh, float* __restrict__ misc, float4* __restrict__ modes) {
    const int M = D / 2;
    const int tid = threadIdx.x;
    if (blockIdx.x > 0) {
        const int m = (blockIdx.x - 1) * kPrepThreads + tid;
        if (m < M) {
            const double r = exp(-(double)nu[m]);
            double sn, cs;
            sincos((double)theta[m], &sn, &cs);
            const double re = r * cs, im = r * sn;
            const float hr = (float)re, hi = (float)im;
            modes[m] = make_float4(hr, hi, (float)(re - (double)hr), (float)(im - (double)hi));
        }
        return;
    }
    __shared__ double s_sum[2][kPrepThreads];
    const int n = D + 1;
    double sp = 0.0, sr = 0.0;
    for (int j = tid; j < n; j += kPrepThreads) {
        const double x = w_phi[j], y = w_r[j];
        sp = fma(x, x, sp);
        sr = fma(y, y, sr);
    }
    s_sum[0][tid] = sp;
    s_sum[1][tid] = sr;
    __syncwarp();
    for (int s2 = kPrepThreads / 2; s2 > 0; s2 >>= 1) {
        if (tid < s2) {
            s_sum[0][tid] += s_sum[0][tid + s2];
            s_sum[1][tid] += s_sum[1][tid + s2];
        }
        __syncwarp();
    }
    const double nphi = sqrt(s_sum[0][0]);
    const double nr = sqrt(s_sum[1][0]);
    const double inv_phi = 1.0 / nphi;
    const double inv_r = 1.0 / nr;
    for (int j = tid; j < n; j += kPrepThreads) {
        wh[j] = (float)((double)w_phi[j] * inv_phi);
        wh[n + j] = (float)((double)w_r[j] * inv_r);
    }
    if (tid == 0) {
        const double inv_sqrt_m = 1.0 / sqrt((double)M);
        const double ta = tanh((double)a_phi[0]);
        const double tr = tanh((double)a_r[0]);
        misc[0] = (float)(ta * inv_sqrt_m);
        misc[1] = (float)(tr * inv_sqrt_m);
        misc[2] = (float)nphi;
        misc[3] = (float)nr;
        misc[4] = (float)ta;
        misc[5] = (float)tr;
        misc[6] = (float)inv_sqrt_m;
    }
}

// ---------------------------------------------------------------------------
// Controller forward: one warp per token, grid-stride over tokens.  The row
// x_sel[t, :] is read once with 16-byte loads (all of a lane's vectors in
// flight together); both projections accumulate in FP32; the lanes then
// evaluate tanh, q(r), d, c and the shared special functions E - 1 =
// expm1(c), C = cos d, S = sin d, and lane 0 stores them.
// ---------------------------------------------------------------------------
constexpr int kCtrlWarps = 8;

template <int VPL>
__global__ void __launch_bounds__(kCtrlWarps * 32) samu_ctrl_fwd_kernel(
    const uint4* __restrict__ x, const uint8_t* __restrict__ reset, const float* __restrict__ wh,
    const float* __restrict__ misc, long long BL, int D, float* __restrict__ p_out,
    float* __restrict__ r_out, float4* __restrict__ ctrl) {
    extern __shared__ __align__(16) float s_w[];   // [2][stride]: w_hat_phi, w_hat_r
    const int n = D + 1;
    const int stride = (n + 3) & ~3;                 // keeps both rows 16-byte aligned
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        s_w[j] = wh[j];
        s_w[stride + j] = wh[n + j];
    }
    __syncthreads();
    const float* s_phi = s_w;
    const float* s_r = s_w + stride;
    const float k_phi = misc[0];
    const float k_r = misc[1];
    const float bias_phi = s_phi[D];   // x~ carries a constant 1 against the bias weight
    const float bias_r = s_r[D];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int vecs = D / 8;
    const long long nwarps = (long long)gridDim.x * kCtrlWarps;
    for (long long t = (long long)blockIdx.x * kCtrlWarps + warp; t < BL; t += nwarps) {
        const uint4* row = x + t * vecs;
        uint4 q[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            q[k] = (v < vecs) ? __ldcs(row + v) : make_uint4(0u, 0u, 0u, 0u);
        }
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            if (v < vecs) {
                const float2 x01 = bf2_to_f2(q[k].x), x23 = bf2_to_f2(q[k].y);
                const float2 x45 = bf2_to_f2(q[k].z), x67 = bf2_to_f2(q[k].w);
                const float4 p0 = *reinterpret_cast<const float4*>(s_phi + 8 * v);
                const float4 p1 = *reinterpret_cast<const float4*>(s_phi + 8 * v + 4);
                const float4 r0 = *reinterpret_cast<const float4*>(s_r + 8 * v);
                const float4 r1 = *reinterpret_cast<const float4*>(s_r + 8 * v + 4);
                a0 = fmaf(x01.x, p0.x, a0); a1 = fmaf(x01.y, p0.y, a1);
                a0 = fmaf(x23.x, p0.z, a0); a1 = fmaf(x23.y, p0.w, a1);
                a0 = fmaf(x45.x, p1.x, a0); a1 = fmaf(x45.y, p1.y, a1);
                a0 = fmaf(x67.x, p1.z, a0); a1 = fmaf(x67.y, p1.w, a1);
                b0 = fmaf(x01.x, r0.x, b0); b1 = fmaf(x01.y, r0.y, b1);
                b0 = fmaf(x23.x, r0.z, b0); b1 = fmaf(x23.y, r0.w, b1);
                b0 = fmaf(x45.x, r1.x, b0); b1 = fmaf(x45.y, r1.y, b1);
                b0 = fmaf(x67.x, r1.z, b0); b1 = fmaf(x67.y, r1.w, b1);
            }
        }
        float sphi = a0 + a1;
        float sr = b0 + b1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sphi += __shfl_xor_sync(0xffffffffu, sphi, o);
            sr += __shfl_xor_sync(0xffffffffu, sr, o);
        }
        if (lane == 0) {
            const float p = tanhf(sphi + bias_phi);
            const float r = tanhf(sr + bias_r);
            const float qr = r / (1.0f + r * r);
            const float d = k_phi * p;
            const float c = k_r * qr;
            float sn, cs;
            sincosf(d, &sn, &cs);
            const float em1 = expm1f(c);
            const float rs = (reset != nullptr && reset[t] != 0) ? 1.0f : 0.0f;
            p_out[t] = p;
            r_out[t] = r;
            ctrl[t] = make_float4(em1, cs, sn, rs);
        }
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
constexpr int kCbUnroll = 8;

__global__ void __launch_bounds__(512) samu_ctrl_bwd_kernel(SamuCtrlBwdArgs a) {
    __shared__ float s_sphi[kCbTokBlock];
    __shared__ float s_sr[kCbTokBlock];
    __shared__ float s_red[4][kCbTokBlock];
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
// Parameter reductions (fixed order, deterministic).
// ---------------------------------------------------------------------------
// stage 1: per-tile (dnu, dtheta) partials, rows = B*CT, into kReduceGroups groups
__global__ void __launch_bounds__(256) samu_numod_stage1_kernel(const float2* __restrict__ numod,
                                                                float2* __restrict__ numod2,
                                                                int rows, int M) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    const int gidx = blockIdx.y;
    if (m >= M) return;
    const int per = (rows + kReduceGroups - 1) / kReduceGroups;
    const int r0 = gidx * per;
    const int r1 = min(rows, r0 + per);
    float sx = 0.f, sy = 0.f;
    int r = r0;
    for (; r + 8 <= r1; r += 8) {
        float2 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcs(numod + (size_t)(r + k) * M + m);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            sx += v[k].x;
            sy += v[k].y;
        }
    }
    for (; r < r1; ++r) {
        const float2 v = __ldcs(numod + (size_t)r * M + m);
        sx += v.x;
        sy += v.y;
    }
    numod2[(size_t)gidx * M + m] = make_float2(sx, sy);
}

// column sums of the controller-backward partial rows: dwh[which][j].  A CTA
// takes 32 columns; its 8 warps each sum a strided set of rows, then the 8
// warp sums are added in a fixed order.
constexpr int kColRows = 2 * kCtrlBwdCtas;

__global__ void __launch_bounds__(256) samu_dwh_colsum_kernel(const float* __restrict__ part,
                                                              float* __restrict__ dwh, int D) {
    __shared__ float s_part[8][32];
    const int n = D + 1;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int j = blockIdx.x * 32 + lane;
    const int which = blockIdx.y;
    float s = 0.f;
    if (j < n) {
        int k = warp;
        for (; k + 8 * 3 < kColRows; k += 8 * 4) {
            const float v0 = part[((size_t)k * 2 + which) * n + j];
            const float v1 = part[((size_t)(k + 8) * 2 + which) * n + j];
            const float v2 = part[((size_t)(k + 16) * 2 + which) * n + j];
            const float v3 = part[((size_t)(k + 24) * 2 + which) * n + j];
            s += v0;
            s += v1;
            s += v2;
            s += v3;
        }
        for (; k < kColRows; k += 8) s += part[((size_t)k * 2 + which) * n + j];
    }
    s_part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && j < n) {
        float t = s_part[0][lane];
#pragma unroll
        for (int w = 1; w < 8; ++w) t += s_part[w][lane];
        dwh[which * n + j] = t;
    }
}

// final: dnu, dtheta; the unit-direction projection dw = (dw_hat - w_hat (w_hat . dw_hat)) / ||w||;
// the amplitude gradients da = (sum partials) / sqrt(M) * (1 - tanh(a)^2).
__global__ void __launch_bounds__(256) samu_param_final_kernel(SamuParamArgs a) {
    __shared__ float s_dot[2][256];
    __shared__ float s_amp[2][256];
    const int tid = threadIdx.x;
    const int D = a.D;
    const int M = D / 2;
    const int n = D + 1;
    for (int m = tid; m < M; m += blockDim.x) {
        float sx = 0.f, sy = 0.f;
        for (int gi = 0; gi < kReduceGroups; ++gi) {
            const float2 v = a.numod2[(size_t)gi * M + m];
            sx += v.x;
            sy += v.y;
        }
        a.dnu[m] = sx;
        a.dtheta[m] = sy;
    }
    float dp = 0.f, dr = 0.f;
    for (int j = tid; j < n; j += blockDim.x) {
        dp = fmaf(a.wh[j], a.dwh[j], dp);
        dr = fmaf(a.wh[n + j], a.dwh[n + j], dr);
    }
    float ap = 0.f, ar = 0.f;
    for (int k = tid; k < kCtrlBwdCtas; k += blockDim.x) {
        const float2 v = a.amp_part[k];
        ap += v.x;
        ar += v.y;
    }
    s_dot[0][tid] = dp;
    s_dot[1][tid] = dr;
    s_amp[0][tid] = ap;
    s_amp[1][tid] = ar;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (tid < s) {
            s_dot[0][tid] += s_dot[0][tid + s];
            s_dot[1][tid] += s_dot[1][tid + s];
            s_amp[0][tid] += s_amp[0][tid + s];
            s_amp[1][tid] += s_amp[1][tid + s];
        }
        __syncthreads();
    }
    const float dot_p = s_dot[0][0];
    const float dot_r = s_dot[1][0];
    const float nphi = a.misc[2];
    const float nr = a.misc[3];
    for (int j = tid; j < n; j += blockDim.x) {
        a.dw_phi[j] = (a.dwh[j] - a.wh[j] * dot_p) / nphi;
        a.dw_r[j] = (a.dwh[n + j] - a.wh[n + j] * dot_r) / nr;
    }
    if (tid == 0) {
        const float ta = a.misc[4], tr = a.misc[5], ism = a.misc[6];
        a.da_phi[0] = s_amp[0][0] * ism * (1.0f - ta * ta);
        a.da_r[0] = s_amp[1][0] * ism * (1.0f - tr * tr);
    }
}

cudaError_t launch_samu_prep(const float* w_phi, const float* w_r, const float* a_phi,
                             const float* a_r, const float* nu, const float* theta, int D,
                             float* wh, float* misc, float4* modes, cudaStream_t s) {
    const int M = D / 2;
    const int grid = 1 + (M + kPrepThreads - 1) / kPrepThreads;
    samu_prep_kernel<<<grid, kPrepThreads, 0, s>>>(w_phi, w_r, a_phi, a_r, nu, theta, D, wh, misc, modes);
    return cudaGetLastError();
}

template <int VPL>
static cudaError_t launch_ctrl_fwd_t(const void* x, const uint8_t* reset, const float* wh,
                                     const float* misc, long long BL, int D, float* p, float* r,
                                     float4* ctrl, cudaStream_t s) {
    const size_t smem = (size_t)2 * ((D + 1 + 3) & ~3) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(samu_ctrl_fwd_kernel<VPL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const long long want = (BL + kCtrlWarps - 1) / kCtrlWarps;
    const long long grid = want < 152LL * 4 ? want : 152LL * 4;
    samu_ctrl_fwd_kernel<VPL><<<(unsigned)grid, kCtrlWarps * 32, smem, s>>>(
        reinterpret_cast<const uint4*>(x), reset, wh, misc, BL, D, p, r, ctrl);
    return cudaGetLastError();
}

cudaError_t launch_samu_ctrl_fwd(const void* x, const uint8_t* reset, const float* wh,
                                 const float* misc, long long BL, int D, float* p, float* r,
                                 float4* ctrl, cudaStream_t s) {
    const int need = (D / 8 + 31) / 32;   // 16-byte vectors per lane
    if (need <= 1) return launch_ctrl_fwd_t<1>(x, reset, wh, misc, BL, D, p, r, ctrl, s);
    if (need <= 2) return launch_ctrl_fwd_t<2>(x, reset, wh, misc, BL, D, p, r, ctrl, s);
    if (need <= 4) return launch_ctrl_fwd_t<4>(x, reset, wh, misc, BL, D, p, r, ctrl, s);
    if (need <= 8) return launch_ctrl_fwd_t<8>(x, reset, wh, misc, BL, D, p, r, ctrl, s);
    return launch_ctrl_fwd_t<16>(x, reset, wh, misc, BL, D, p, r, ctrl, s);
}

cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s) {
    int cols = ((args.D / 8) + 31) / 32 * 32;
    if (cols < kCbTokBlock / 2) cols = kCbTokBlock / 2;
    const int threads = 2 * cols <= 512 ? 2 * cols : cols;   // two token halves when they fit
    samu_ctrl_bwd_kernel<<<kCtrlBwdCtas, threads, 0, s>>>(args);
    return cudaGetLastError();
}

cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s) {
    const int M = args.D / 2;
    const int rows = args.B * args.CT;
    dim3 g1((M + 255) / 256, kReduceGroups);
    samu_numod_stage1_kernel<<<g1, 256, 0, s>>>(args.numod, args.numod2, rows, M);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2((args.D + 1 + 31) / 32, 2);
    samu_dwh_colsum_kernel<<<g2, 256, 0, s>>>(args.dwh_part, args.dwh, args.D);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    samu_param_final_kernel<<<1, 256, 0, s>>>(args);
    return cudaGetLastError();
}

}  // namespace lrs

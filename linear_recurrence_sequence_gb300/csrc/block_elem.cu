// Element-wise and row-wise kernels of the RecurrentBlock around the mixer
// ("SAMU 与 RG-LRU 的 H800 训练性能对比", section 03: normalisation, per-channel
// convolution, join with the gate branch; the SAMU project page: the block's
// wide input branch is the mixer's write).  The readings of what the pages
// leave open are stated where each kernel is defined.
//
// All tensors are row-major [B L][width] BF16 with FP32 arithmetic; widths
// are multiples of 256, so a thread works on 8 consecutive channels (one
// 16-byte load).
#include "kernels.cuh"

namespace lrs {

namespace {

constexpr float kNormEps = 1e-6f;
constexpr float kGeluC = 0.7978845608028654f;   // sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ float gelu_fwd(float x) {
    const float u = kGeluC * (x + kGeluA * x * x * x);
    return 0.5f * x * (1.f + tanhf(u));
}

__device__ __forceinline__ void unpack8(const uint4 q, float (&v)[8]) {
    float2 f;
    f = bf2_to_f2(q.x); v[0] = f.x; v[1] = f.y;
    f = bf2_to_f2(q.y); v[2] = f.x; v[3] = f.y;
    f = bf2_to_f2(q.z); v[4] = f.x; v[5] = f.y;
    f = bf2_to_f2(q.w); v[6] = f.x; v[7] = f.y;
}
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 q;
    q.x = f2_to_bf2(v[0], v[1]);
    q.y = f2_to_bf2(v[2], v[3]);
    q.z = f2_to_bf2(v[4], v[5]);
    q.w = f2_to_bf2(v[6], v[7]);
    return q;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// RMSNorm forward (reading: scale gamma, eps 1e-6):
//   rstd = 1 / sqrt(mean_c x^2 + eps), h = (x rstd) gamma, one warp per row.
// status_clear (optional): the word is cleared by thread 0 of CTA 0 (the
// first kernel of a block call).
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(const uint4* __restrict__ x, const float* __restrict__ gamma,
                                                          uint4* __restrict__ h, float* __restrict__ rstd,
                                                          long long rows, int W, uint32_t* status_clear) {
    pdl_trigger();
    pdl_wait();
    if (status_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status_clear = 0u;
    const int lane = threadIdx.x & 31;
    const int nv = W / 8;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((long long)gridDim.x * blockDim.x) >> 5) {
        const uint4* xr = x + (size_t)row * nv;
        float ss = 0.f;
        for (int v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(__ldg(xr + v), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
        }
        ss = warp_sum(ss);
        const float r = 1.f / sqrtf(ss / (float)W + kNormEps);
        if (lane == 0) rstd[row] = r;
        for (int v = lane; v < nv; v += 32) {
            float f[8];
            unpack8(__ldg(xr + v), f);
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v);
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v + 1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = f[i] * r * g[i];
            h[(size_t)row * nv + v] = pack8(f);
        }
    }
}

// RMSNorm backward with the residual gradient added:
//   n = x rstd, g = dh gamma, dx = dres + rstd (g - n mean_c(g n)),
//   dgamma partial (per CTA) = sum over the CTA's rows of dh n.
// One thread per 8 channels (blockDim = W / 8), the CTA walks rows
// [r0, r1) four at a time; each row's mean is reduced across the CTA.
constexpr int kNormRowsPerStep = 4;
__global__ void __launch_bounds__(512) rmsnorm_bwd_kernel(const uint4* __restrict__ x, const float* __restrict__ gamma,
                                                          const float* __restrict__ rstd, const uint4* __restrict__ dh,
                                                          const uint4* __restrict__ dres, uint4* __restrict__ dx,
                                                          float* __restrict__ dgamma_part, long long rows, int W,
                                                          uint32_t* status_clear) {
    __shared__ float red[kNormRowsPerStep][16];
    pdl_trigger();
    pdl_wait();
    if (status_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status_clear = 0u;
    const int v = threadIdx.x;   // channels 8 v .. 8 v + 7
    const int nv = W / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const long long r0 = rows * blockIdx.x / gridDim.x, r1 = rows * (blockIdx.x + 1) / gridDim.x;
    float gm[8], dg[8];
    {
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v + 1);
        gm[0] = g0.x; gm[1] = g0.y; gm[2] = g0.z; gm[3] = g0.w;
        gm[4] = g1.x; gm[5] = g1.y; gm[6] = g1.z; gm[7] = g1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) dg[i] = 0.f;
    for (long long rb = r0; rb < r1; rb += kNormRowsPerStep) {
        float nn[kNormRowsPerStep][8], gg[kNormRowsPerStep][8], part[kNormRowsPerStep], rs[kNormRowsPerStep];
#pragma unroll
        for (int k = 0; k < kNormRowsPerStep; ++k) {
            const long long row = rb + k;
            part[k] = 0.f;
            rs[k] = 0.f;
            if (row < r1) {
                float xv[8], hv[8];
                unpack8(__ldg(x + (size_t)row * nv + v), xv);
                unpack8(__ldg(dh + (size_t)row * nv + v), hv);
                rs[k] = __ldg(rstd + row);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    nn[k][i] = xv[i] * rs[k];
                    gg[k][i] = hv[i] * gm[i];
                    part[k] = fmaf(gg[k][i], nn[k][i], part[k]);
                    dg[i] = fmaf(hv[i], nn[k][i], dg[i]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kNormRowsPerStep; ++k) {
            const float s = warp_sum(part[k]);
            if (lane == 0) red[k][warp] = s;
        }
        __syncthreads();
        float mean[kNormRowsPerStep];
#pragma unroll
        for (int k = 0; k < kNormRowsPerStep; ++k) {
            float s = 0.f;
            for (int w = 0; w < nwarps; ++w) s += red[k][w];
            mean[k] = s / (float)W;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kNormRowsPerStep; ++k) {
            const long long row = rb + k;
            if (row < r1) {
                float rv[8], o[8];
                unpack8(__ldg(dres + (size_t)row * nv + v), rv);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = rv[i] + rs[k] * (gg[k][i] - nn[k][i] * mean[k]);
                dx[(size_t)row * nv + v] = pack8(o);
            }
        }
    }
    float4* dp = reinterpret_cast<float4*>(dgamma_part + (size_t)blockIdx.x * W + 8 * v);
    dp[0] = make_float4(dg[0], dg[1], dg[2], dg[3]);
    dp[1] = make_float4(dg[4], dg[5], dg[6], dg[7]);
}

// Causal depthwise convolution of width 4 (reading): u[t] = kb + sum_{j<4}
// k[j] v[t - j] over the taps that stay inside t's segment (a reset at t' > t
// - j, t' <= t cuts the taps before it; t = 0 starts every row).  v is the
// recurrent half (columns D .. 2D - 1) of the input projection's [B L][2 D]
// output.  One thread per (token, 8 channels).
__global__ void __launch_bounds__(256) conv_fwd_kernel(const uint16_t* __restrict__ gv, const float* __restrict__ k,
                                                       const float* __restrict__ kb, const uint8_t* __restrict__ reset,
                                                       uint4* __restrict__ u, int B, int L, int D) {
    pdl_trigger();
    pdl_wait();
    const int nv = D / 8;
    const long long n = (long long)B * L * nv;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(e % nv);
        const long long bt = e / nv;
        const int t = (int)(bt % L);
        float acc[8];
        {
            const float4 b0 = __ldg(reinterpret_cast<const float4*>(kb) + 2 * v);
            const float4 b1 = __ldg(reinterpret_cast<const float4*>(kb) + 2 * v + 1);
            acc[0] = b0.x; acc[1] = b0.y; acc[2] = b0.z; acc[3] = b0.w;
            acc[4] = b1.x; acc[5] = b1.y; acc[6] = b1.z; acc[7] = b1.w;
        }
        bool live = true;   // tap j still inside t's segment
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j > 0) live = live && t - j >= 0 && !(reset != nullptr && reset[bt - j + 1]);
            if (live) {
                float f[8];
                unpack8(__ldg(reinterpret_cast<const uint4*>(gv + (size_t)(bt - j) * 2 * D + D) + v), f);
                const float4 k0 = __ldg(reinterpret_cast<const float4*>(k + (size_t)j * D) + 2 * v);
                const float4 k1 = __ldg(reinterpret_cast<const float4*>(k + (size_t)j * D) + 2 * v + 1);
                const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(kk[i], f[i], acc[i]);
            }
        }
        u[(size_t)bt * nv + v] = pack8(acc);
    }
}

// Adjoint of conv_fwd_kernel with du = dx_sel + dw (the mixer reads x_sel =
// w = u, so both gradients reach u):
//   dv[t] = sum_j k[j] du[t + j] over the taps of t + j that reach t,
//   dk[j] += du[t] v[t - j], dkb += du[t] (per-chunk partials, reduced in a
//   fixed order by sum_parts).
// Thread: 8 channels of one chunk of kConvChunk tokens of one row.  The
// mixer's status word is OR-ed into the block's (thread 0 of CTA 0).
constexpr int kConvChunk = 64;
__global__ void __launch_bounds__(256) conv_bwd_kernel(const uint16_t* __restrict__ gv, const float* __restrict__ k,
                                                       const uint8_t* __restrict__ reset,
                                                       const uint16_t* __restrict__ dxs, const uint16_t* __restrict__ dwm,
                                                       uint16_t* __restrict__ dgv, float* __restrict__ part, int B,
                                                       int L, int D, uint32_t* status, const uint32_t* mixer_status) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0 && mixer_status != nullptr) {
        const uint32_t m = *mixer_status;
        if (m != 0u) atomicOr(status, m);
    }
    const int nv = D / 8;
    const int chunks = (L + kConvChunk - 1) / kConvChunk;
    const long long n = (long long)B * chunks * nv;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const int v = (int)(e % nv);
        const long long bc = e / nv;   // row b, chunk c: partial slot
        const int c = (int)(bc % chunks);
        const int b = (int)(bc / chunks);
        float kk[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 k0 = __ldg(reinterpret_cast<const float4*>(k + (size_t)j * D) + 2 * v);
            const float4 k1 = __ldg(reinterpret_cast<const float4*>(k + (size_t)j * D) + 2 * v + 1);
            kk[j][0] = k0.x; kk[j][1] = k0.y; kk[j][2] = k0.z; kk[j][3] = k0.w;
            kk[j][4] = k1.x; kk[j][5] = k1.y; kk[j][6] = k1.z; kk[j][7] = k1.w;
        }
        float dk[5][8];
#pragma unroll
        for (int j = 0; j < 5; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) dk[j][i] = 0.f;
        const int t0 = c * kConvChunk, t1 = min(L, t0 + kConvChunk);
        const size_t row0 = (size_t)b * L;
        auto du_at = [&](int t, float (&o)[8]) {
            float a[8], w[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(dxs + (row0 + t) * D) + v), a);
            unpack8(__ldg(reinterpret_cast<const uint4*>(dwm + (row0 + t) * D) + v), w);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = a[i] + w[i];
        };
        for (int t = t0; t < t1; ++t) {
            float dut[8];
            du_at(t, dut);
            // parameter partials: du[t] v[t - j] over t's live taps
            bool live = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j > 0) live = live && t - j >= 0 && !(reset != nullptr && reset[row0 + t - j + 1]);
                if (live) {
                    float f[8];
                    unpack8(__ldg(reinterpret_cast<const uint4*>(gv + (row0 + t - j) * 2 * D + D) + v), f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dk[j][i] = fmaf(dut[i], f[i], dk[j][i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) dk[4][i] += dut[i];
            // dv[t] = sum_j k[j] du[t + j] over the outputs t + j whose tap j reaches t
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = kk[0][i] * dut[i];
            bool reach = true;
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                reach = reach && t + j < L && !(reset != nullptr && reset[row0 + t + j]);
                if (reach) {
                    float d2[8];
                    du_at(t + j, d2);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(kk[j][i], d2[i], acc[i]);
                }
            }
            *reinterpret_cast<uint4*>(dgv + (row0 + t) * 2 * D + D + 8 * v) = pack8(acc);
        }
        float* p = part + (size_t)bc * 5 * D;
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            float4* q = reinterpret_cast<float4*>(p + (size_t)j * D + 8 * v);
            q[0] = make_float4(dk[j][0], dk[j][1], dk[j][2], dk[j][3]);
            q[1] = make_float4(dk[j][4], dk[j][5], dk[j][6], dk[j][7]);
        }
    }
}

// Join with the gate branch: j = GeLU(g) y_mixer (BF16), g the gate half
// (columns 0 .. D - 1) of the input projection's output.  The mixer's status
// word is OR-ed into the block's (thread 0 of CTA 0).
__global__ void __launch_bounds__(256) join_fwd_kernel(const uint16_t* __restrict__ gv, const uint4* __restrict__ ym,
                                                       uint4* __restrict__ j, long long BL, int D, uint32_t* status,
                                                       const uint32_t* mixer_status) {
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0 && mixer_status != nullptr) {
        const uint32_t m = *mixer_status;
        if (m != 0u) atomicOr(status, m);
    }
    const int nv = D / 8;
    const long long n = BL * nv;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const long long t = e / nv;
        const int v = (int)(e % nv);
        float g[8], y[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(gv + (size_t)t * 2 * D) + v), g);
        unpack8(__ldg(ym + e), y);
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = gelu_fwd(g[i]) * y[i];
        j[e] = pack8(g);
    }
}

unsigned grid_for(long long n, int threads) {
    long long b = (n + threads - 1) / threads;
    if (b > 8192) b = 8192;
    return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

int block_norm_bwd_ctas(long long rows) {
    long long c = 2LL * 152;
    if (c > rows) c = rows;
    return (int)(c < 1 ? 1 : c);
}

int block_conv_parts(int B, int L) { return B * ((L + kConvChunk - 1) / kConvChunk); }

cudaError_t launch_rmsnorm_fwd(const void* x, const float* gamma, void* h, float* rstd, long long rows, int W,
                               uint32_t* status_clear, cudaStream_t s, bool pdl) {
    return launch_ex(rmsnorm_fwd_kernel, grid_for(rows * 32, 256), 256, 0, s, pdl, static_cast<const uint4*>(x),
                     gamma, static_cast<uint4*>(h), rstd, rows, W, status_clear);
}

cudaError_t launch_rmsnorm_bwd(const void* x, const float* gamma, const float* rstd, const void* dh, const void* dres,
                               void* dx, float* dgamma_part, long long rows, int W, uint32_t* status_clear,
                               cudaStream_t s, bool pdl) {
    return launch_ex(rmsnorm_bwd_kernel, (unsigned)block_norm_bwd_ctas(rows), (unsigned)(W / 8), 0, s, pdl,
                     static_cast<const uint4*>(x), gamma, rstd, static_cast<const uint4*>(dh),
                     static_cast<const uint4*>(dres), static_cast<uint4*>(dx), dgamma_part, rows, W, status_clear);
}

cudaError_t launch_conv_fwd(const void* gv, const float* k, const float* kb, const uint8_t* reset, void* u, int B,
                            int L, int D, cudaStream_t s, bool pdl) {
    return launch_ex(conv_fwd_kernel, grid_for((long long)B * L * (D / 8), 256), 256, 0, s, pdl,
                     static_cast<const uint16_t*>(gv), k, kb, reset, static_cast<uint4*>(u), B, L, D);
}

cudaError_t launch_conv_bwd(const void* gv, const float* k, const uint8_t* reset, const void* dxs, const void* dwm,
                            void* dgv, float* part, int B, int L, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl) {
    return launch_ex(conv_bwd_kernel, grid_for((long long)block_conv_parts(B, L) * (D / 8), 256), 256, 0, s, pdl,
                     static_cast<const uint16_t*>(gv), k, reset, static_cast<const uint16_t*>(dxs),
                     static_cast<const uint16_t*>(dwm), static_cast<uint16_t*>(dgv), part, B, L, D, status,
                     mixer_status);
}

cudaError_t launch_join_fwd(const void* gv, const void* ym, void* j, long long BL, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl) {
    return launch_ex(join_fwd_kernel, grid_for(BL * (D / 8), 256), 256, 0, s, pdl, static_cast<const uint16_t*>(gv),
                     static_cast<const uint4*>(ym), static_cast<uint4*>(j), BL, D, status, mixer_status);
}

}  // namespace lrs

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
#include "block_math.cuh"

namespace lrs {

namespace {

constexpr float kNormEps = 1e-6f;
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

// The same for W <= 1024 (more channels per lane would spill), one warp per row: lane l owns the 8-channel groups
// l + 32 k (k < NK = W / 256) and keeps the row's x, dh and dres in registers
// (3 NK independent 16-byte loads), the row mean is a warp sum.  gamma and
// the per-warp dgamma rows live in shared memory (dgamma accumulates per
// lane over the warp's rows there), which keeps two CTAs per SM; the CTA's
// 8192 / W warps share its contiguous row range and their dgamma rows are
// added in warp order into the CTA's partial row.
template <int NK>
__global__ void __launch_bounds__(256, 2) rmsnorm_bwd_warp_kernel(const uint4* __restrict__ x,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ rstd,
                                                                  const uint4* __restrict__ dh,
                                                                  const uint4* __restrict__ dres,
                                                                  uint4* __restrict__ dx,
                                                                  float* __restrict__ dgamma_part, long long rows) {
    constexpr int W = 256 * NK, nv = W / 8, WPC = 8192 / W > 8 ? 8 : 8192 / W;
    __shared__ __align__(16) float red[WPC][W];
    __shared__ __align__(16) float s_g[W];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long r0 = rows * blockIdx.x / gridDim.x, r1 = rows * (blockIdx.x + 1) / gridDim.x;
    for (int c = threadIdx.x; c < W; c += blockDim.x) s_g[c] = __ldg(gamma + c);
    if (warp < WPC)
        for (int c = lane; c < W; c += 32) red[warp][c] = 0.f;
    __syncthreads();
    float4* dgw = reinterpret_cast<float4*>(red[warp < WPC ? warp : 0]);
    const float4* gw = reinterpret_cast<const float4*>(s_g);
    for (long long row = r0 + warp; row < r1; row += WPC) {
        uint4 qx[NK], qh[NK], qr[NK];
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const size_t o = (size_t)row * nv + lane + 32 * k;
            qx[k] = __ldg(x + o);
            qh[k] = __ldg(dh + o);
            qr[k] = __ldg(dres + o);
        }
        const float rs = __ldg(rstd + row);
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const int v = lane + 32 * k;
            float xv[8], hv[8];
            unpack8(qx[k], xv);
            unpack8(qh[k], hv);
            const float4 g0 = gw[2 * v], g1 = gw[2 * v + 1];
            const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            float4 d0 = dgw[2 * v], d1 = dgw[2 * v + 1];
            float dg[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float n = xv[i] * rs;
                part = fmaf(hv[i] * gm[i], n, part);
                dg[i] = fmaf(hv[i], n, dg[i]);
            }
            dgw[2 * v] = make_float4(dg[0], dg[1], dg[2], dg[3]);
            dgw[2 * v + 1] = make_float4(dg[4], dg[5], dg[6], dg[7]);
        }
        const float mean = warp_sum(part) / (float)W;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const int v = lane + 32 * k;
            float xv[8], hv[8], rv[8], o[8];
            unpack8(qx[k], xv);
            unpack8(qh[k], hv);
            unpack8(qr[k], rv);
            const float4 g0 = gw[2 * v], g1 = gw[2 * v + 1];
            const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float n = xv[i] * rs;
                o[i] = rv[i] + rs * (hv[i] * gm[i] - n * mean);
            }
            dx[(size_t)row * nv + lane + 32 * k] = pack8(o);
        }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < W; c += blockDim.x) {
        float sum = 0.f;
        for (int w = 0; w < WPC; ++w) sum += red[w][c];
        dgamma_part[(size_t)blockIdx.x * W + c] = sum;
    }
}

// Causal depthwise convolution of width 4 (reading): u[t] = kb + sum_{j<4}
// k[j] v[t - j] over the taps that stay inside t's segment (a segment start
// at t - j + 1 .. t cuts tap j; t = 0 starts every row).  v is the recurrent
// half (columns D .. 2D - 1) of the input projection's [B L][2 D] output.
// Thread: 4 channels of kConvRun consecutive tokens; it loads every row its
// window needs first (kConvRun + 3 independent 8-byte loads), then forms the
// outputs.  A warp covers 128 channels of one run (256 contiguous bytes per
// row).
constexpr int kConvRun = 16;

__device__ __forceinline__ void unpack4(const uint2 q, float (&v)[4]) {
    float2 f;
    f = bf2_to_f2(q.x); v[0] = f.x; v[1] = f.y;
    f = bf2_to_f2(q.y); v[2] = f.x; v[3] = f.y;
}
__device__ __forceinline__ uint2 pack4(const float (&v)[4]) {
    uint2 q;
    q.x = f2_to_bf2(v[0], v[1]);
    q.y = f2_to_bf2(v[2], v[3]);
    return q;
}
__device__ __forceinline__ void load_k4(const float* __restrict__ k, const float* __restrict__ kb, int D, int q,
                                        float (&kk)[4][4], float (&bb)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 kv = __ldg(reinterpret_cast<const float4*>(k + (size_t)j * D) + q);
        kk[j][0] = kv.x; kk[j][1] = kv.y; kk[j][2] = kv.z; kk[j][3] = kv.w;
    }
    if (kb != nullptr) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(kb) + q);
        bb[0] = b.x; bb[1] = b.y; bb[2] = b.z; bb[3] = b.w;
    }
}

__global__ void __launch_bounds__(256) conv_fwd_kernel(const uint16_t* __restrict__ gv, const float* __restrict__ k,
                                                       const float* __restrict__ kb, const uint8_t* __restrict__ reset,
                                                       uint16_t* __restrict__ u, int B, int L, int D) {
    pdl_trigger();
    pdl_wait();
    const int nq = D / 4;
    const int runs = (L + kConvRun - 1) / kConvRun;
    const long long n = (long long)B * runs * nq;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
        const int q = (int)(e % nq);
        const long long br = e / nq;
        const int b = (int)(br / runs), t0 = (int)(br % runs) * kConvRun;
        const size_t row0 = (size_t)b * L;
        uint2 rows[kConvRun + 3];   // v[t0 - 3 + i]
#pragma unroll
        for (int i = 0; i < kConvRun + 3; ++i) {
            const int t = t0 - 3 + i;
            rows[i] = (t >= 0 && t < L) ? __ldg(reinterpret_cast<const uint2*>(gv + (row0 + t) * 2 * D + D) + q)
                                        : make_uint2(0u, 0u);
        }
        float kk[4][4], bb[4];
        load_k4(k, kb, D, q, kk, bb);
        // bit i: a segment starts at t0 - 3 + i
        uint32_t st = 0u;
        if (reset != nullptr)
#pragma unroll
            for (int i = 0; i < kConvRun + 3; ++i) {
                const int t = t0 - 3 + i;
                if (t >= 0 && t < L && reset[row0 + t] != 0) st |= 1u << i;
            }
#pragma unroll
        for (int r = 0; r < kConvRun; ++r) {
            const int t = t0 + r;
            if (t >= L) break;
            float acc[4] = {bb[0], bb[1], bb[2], bb[3]};
            bool live = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j > 0) live = live && t - j >= 0 && !((st >> (r + 4 - j)) & 1u);
                if (live) {
                    float f[4];
                    unpack4(rows[r + 3 - j], f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(kk[j][i], f[i], acc[i]);
                }
            }
            *reinterpret_cast<uint2*>(u + (row0 + t) * D + 4 * q) = pack4(acc);
        }
    }
}

// Adjoint of conv_fwd_kernel with du = dx_sel + dw (the SAMU mixer reads
// x_sel = w = u, so both gradients reach u; dwm == nullptr: du = dx_sel, the
// RG-LRU mixer's single input gradient):
//   dv[t] = sum_j k[j] du[t + j] over the outputs t + j whose tap j reaches t
//           (no segment start at t + 1 .. t + j),
//   dk[j] += du[t] v[t - j] over t's live taps, dkb += du[t].
// CTA: a tile of kConvTile = 4 kConvRun tokens of one row and 256 channels;
// thread (run r, channel group g): channels 4 g .. 4 g + 3 of the span and
// the run's tokens, with every row it needs loaded first (du rows t .. t + 3
// and v rows t - 3 .. t of the run: 2 (kConvRun + 3) independent 8-byte
// loads) and the run's segment starts as bits of one word.  The k and bias contributions of the four runs are added in run
// order through shared memory: one partial row per tile, reduced in a fixed
// order by sum_parts.  The mixer's status word is OR-ed into the block's
// (thread 0 of CTA 0).
constexpr int kConvTile = 4 * kConvRun;

__global__ void __launch_bounds__(256) conv_bwd_kernel(const uint16_t* __restrict__ gv, const float* __restrict__ k,
                                                       const uint8_t* __restrict__ reset,
                                                       const uint16_t* __restrict__ dxs, const uint16_t* __restrict__ dwm,
                                                       uint16_t* __restrict__ dgv, float* __restrict__ part, int B,
                                                       int L, int D, uint32_t* status, const uint32_t* mixer_status) {
    __shared__ float red[4][5][256];
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && mixer_status != nullptr) {
        const uint32_t m = *mixer_status;
        if (m != 0u) atomicOr(status, m);
    }
    const int g = threadIdx.x & 63, run = threadIdx.x >> 6;
    const int tiles = (L + kConvTile - 1) / kConvTile;
    const int b = blockIdx.x / tiles, tile = blockIdx.x % tiles;
    const int q = blockIdx.y * 64 + g;   // channels 4 q .. 4 q + 3
    const int t0 = tile * kConvTile + run * kConvRun;
    const size_t row0 = (size_t)b * L;
    float du[kConvRun + 3][4];   // du[t0 + i]
    uint2 vr[kConvRun + 3];      // v[t0 - 3 + i]
    {
        uint2 ra[kConvRun + 3], rw[kConvRun + 3];
#pragma unroll
        for (int i = 0; i < kConvRun + 3; ++i) {
            const int t = t0 + i;
            const bool ok = t < L;
            ra[i] = ok ? __ldg(reinterpret_cast<const uint2*>(dxs + (row0 + t) * D) + q) : make_uint2(0u, 0u);
            rw[i] = (ok && dwm != nullptr) ? __ldg(reinterpret_cast<const uint2*>(dwm + (row0 + t) * D) + q)
                                           : make_uint2(0u, 0u);
            const int tv = t0 - 3 + i;
            vr[i] = (tv >= 0 && tv < L) ? __ldg(reinterpret_cast<const uint2*>(gv + (row0 + tv) * 2 * D + D) + q)
                                        : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kConvRun + 3; ++i) {
            float a[4], w[4];
            unpack4(ra[i], a);
            unpack4(rw[i], w);
#pragma unroll
            for (int c = 0; c < 4; ++c) du[i][c] = a[c] + w[c];
        }
    }
    float kk[4][4], unused[4];
    load_k4(k, nullptr, D, q, kk, unused);
    // bit i: a segment starts at t0 - 3 + i (i < kConvRun + 6)
    uint32_t st = 0u;
    if (reset != nullptr)
#pragma unroll
        for (int i = 0; i < kConvRun + 6; ++i) {
            const int t = t0 - 3 + i;
            if (t >= 0 && t < L && reset[row0 + t] != 0) st |= 1u << i;
        }
    float c[5][4];
#pragma unroll
    for (int j = 0; j < 5; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[j][i] = 0.f;
    // a run whose window holds no segment start and no row edge: every tap
    // counts (the same operations in the same order, without the tests)
    const bool clean = st == 0u && t0 >= 3 && t0 + kConvRun + 3 <= L;
    if (clean) {
#pragma unroll
        for (int r = 0; r < kConvRun; ++r) {
            const int t = t0 + r;
            float acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = kk[0][i] * du[r][i];
#pragma unroll
            for (int j = 1; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = fmaf(kk[j][i], du[r + j][i], acc[i]);
            *reinterpret_cast<uint2*>(dgv + (row0 + t) * 2 * D + D + 4 * q) = pack4(acc);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float f[4];
                unpack4(vr[r + 3 - j], f);
#pragma unroll
                for (int i = 0; i < 4; ++i) c[j][i] = fmaf(du[r][i], f[i], c[j][i]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[4][i] += du[r][i];
        }
    }
#pragma unroll
    for (int r = 0; r < kConvRun && !clean; ++r) {
        const int t = t0 + r;
        if (t < L) {
            float acc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = kk[0][i] * du[r][i];
            bool reach = true;
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                reach = reach && t + j < L && !((st >> (r + 3 + j)) & 1u);
                if (reach)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(kk[j][i], du[r + j][i], acc[i]);
            }
            *reinterpret_cast<uint2*>(dgv + (row0 + t) * 2 * D + D + 4 * q) = pack4(acc);
            bool live = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j > 0) live = live && t - j >= 0 && !((st >> (r + 4 - j)) & 1u);
                if (live) {
                    float f[4];
                    unpack4(vr[r + 3 - j], f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[j][i] = fmaf(du[r][i], f[i], c[j][i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[4][i] += du[r][i];
        }
    }
#pragma unroll
    for (int j = 0; j < 5; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[run][j][4 * g + i] = c[j][i];
    __syncthreads();
    float* p = part + (size_t)blockIdx.x * 5 * D + (size_t)blockIdx.y * 256;
    for (int e = threadIdx.x; e < 5 * 256; e += blockDim.x) {
        const int j = e / 256, ch = e % 256;
        p[(size_t)j * D + ch] = ((red[0][j][ch] + red[1][j][ch]) + red[2][j][ch]) + red[3][j][ch];
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
    long long c = 8LL * 152;
    if (c > rows) c = rows;
    return (int)(c < 1 ? 1 : c);
}

int block_conv_parts(int B, int L) { return B * ((L + kConvTile - 1) / kConvTile); }

cudaError_t launch_rmsnorm_fwd(const void* x, const float* gamma, void* h, float* rstd, long long rows, int W,
                               uint32_t* status_clear, cudaStream_t s, bool pdl) {
    return launch_ex(rmsnorm_fwd_kernel, grid_for(rows * 32, 256), 256, 0, s, pdl, static_cast<const uint4*>(x),
                     gamma, static_cast<uint4*>(h), rstd, rows, W, status_clear);
}

cudaError_t launch_rmsnorm_bwd(const void* x, const float* gamma, const float* rstd, const void* dh, const void* dres,
                               void* dx, float* dgamma_part, long long rows, int W, uint32_t* status_clear,
                               cudaStream_t s, bool pdl) {
    const unsigned ctas = (unsigned)block_norm_bwd_ctas(rows);
    const uint4* xx = static_cast<const uint4*>(x);
    const uint4* hh = static_cast<const uint4*>(dh);
    const uint4* rr = static_cast<const uint4*>(dres);
    uint4* oo = static_cast<uint4*>(dx);
    if (status_clear == nullptr && W <= 1024) {
        const unsigned threads = 32u * (unsigned)(8192 / W > 8 ? 8 : 8192 / W);
        switch (W / 256) {
            case 1: return launch_ex(rmsnorm_bwd_warp_kernel<1>, ctas, threads, 0, s, pdl, xx, gamma, rstd, hh, rr, oo,
                                     dgamma_part, rows);
            case 2: return launch_ex(rmsnorm_bwd_warp_kernel<2>, ctas, threads, 0, s, pdl, xx, gamma, rstd, hh, rr, oo,
                                     dgamma_part, rows);
            case 4: return launch_ex(rmsnorm_bwd_warp_kernel<4>, ctas, threads, 0, s, pdl, xx, gamma, rstd, hh, rr, oo,
                                     dgamma_part, rows);
            default: break;
        }
    }
    return launch_ex(rmsnorm_bwd_kernel, ctas, (unsigned)(W / 8), 0, s, pdl, xx, gamma, rstd, hh, rr, oo, dgamma_part,
                     rows, W, status_clear);
}

cudaError_t launch_conv_fwd(const void* gv, const float* k, const float* kb, const uint8_t* reset, void* u, int B,
                            int L, int D, cudaStream_t s, bool pdl) {
    const long long n = (long long)B * ((L + kConvRun - 1) / kConvRun) * (D / 4);
    return launch_ex(conv_fwd_kernel, grid_for(n, 256), 256, 0, s, pdl, static_cast<const uint16_t*>(gv), k, kb, reset,
                     static_cast<uint16_t*>(u), B, L, D);
}

cudaError_t launch_conv_bwd(const void* gv, const float* k, const uint8_t* reset, const void* dxs, const void* dwm,
                            void* dgv, float* part, int B, int L, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl) {
    const dim3 grid((unsigned)block_conv_parts(B, L), (unsigned)(D / 256));
    return launch_ex(conv_bwd_kernel, grid, 256, 0, s, pdl, static_cast<const uint16_t*>(gv), k, reset,
                     static_cast<const uint16_t*>(dxs), static_cast<const uint16_t*>(dwm), static_cast<uint16_t*>(dgv),
                     part, B, L, D, status, mixer_status);
}

cudaError_t launch_join_fwd(const void* gv, const void* ym, void* j, long long BL, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl) {
    return launch_ex(join_fwd_kernel, grid_for(BL * (D / 8), 256), 256, 0, s, pdl, static_cast<const uint16_t*>(gv),
                     static_cast<const uint4*>(ym), static_cast<uint4*>(j), BL, D, status, mixer_status);
}

}  // namespace lrs

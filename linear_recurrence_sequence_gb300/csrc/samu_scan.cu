// SAMU mixer chunked complex affine scan on sm_103a: forward and reverse.
//
// Equations: SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比"), section 05:
// z_{t,m} = lambda_{t,m} z_{t-1,m} + b_{t,m} with lambda rebuilt in registers
// from the shared per-token E, C, S and the static spectrum (no [B,L,M]
// transition tensor); chunk summaries S_c = T_e o ... o T_s under
// (l2,b2) o (l1,b1) = (l2 l1, l2 b1 + b2); replay from the chunk entry state
// with the visible output fused; the backward runs the conjugate transition
// in reverse time, zbar_{t-1} += conj(lambda_t) zbar_t, bbar_t = zbar_t, and
// rebuilds lambda instead of storing it.
//
// Tiling (GB300): a chain is one (batch row, group of 64 modes); a CTA owns
// one 128-token tile of a chain, staged into shared memory by TMA
// (cp.async.bulk.tensor, one 16 KB box per BF16 half).  Its 8 warps take
// 16-token sub-chunks; lane l owns modes 2l, 2l+1 of the group.  Warp maps
// are combined in shared memory, and tiles of a chain are linked by a
// decoupled look-back (tile ids from an atomic counter, so every awaited tile
// is already resident; all waits bounded).  Every state in the chain is
// produced by the same capply sequence, so results equal the serial
// chunk-entry propagation bit for bit, whatever the timing.
#include "kernels.cuh"

namespace lrs {

// Warp-uniform choice of the lambda variant for one sub-chunk: the polynomial
// path when |nu| max|E - 1| < kPolyBound for every lane's modes.
__device__ __forceinline__ bool use_fast_lambda(const float4* sc, int lane, const ModeConst& k0,
                                                const ModeConst& k1) {
    float e = 0.f;
    if (lane < kSub) {
        const float4 ct = sc[lane];
        if (ct.w == kTokNormal) e = fabsf(ct.x);
    }
    const float emax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(e)));
    const bool ok = fabsf(k0.nu) * emax < kPolyBound && fabsf(k1.nu) * emax < kPolyBound;
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// Forward: sub-chunk summary and replay.  sc = the warp's 16 control words,
// wre/wim = the lane's column of the staged w box (row stride kGroup/2 words).
// ---------------------------------------------------------------------------
template <bool FAST>
__device__ __forceinline__ void fwd_summary(const float4* sc, const uint32_t* wre, const uint32_t* wim,
                                            const ModeConst& k0, const ModeConst& k1, float4& S0, float4& S1) {
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
        const float4 ct = sc[i];
        if (ct.w == kTokPad) break;
        const float2 br = bf2_to_f2(wre[i * (kGroup / 2)]);
        const float2 bi = bf2_to_f2(wim[i * (kGroup / 2)]);
        if (ct.w == kTokNormal) {
            S0 = compose_step(samu_lambda<FAST>(k0, ct), make_float2(br.x, bi.x), S0);
            S1 = compose_step(samu_lambda<FAST>(k1, ct), make_float2(br.y, bi.y), S1);
        } else {   // segment start: lambda = 0
            S0 = make_float4(0.f, 0.f, br.x, bi.x);
            S1 = make_float4(0.f, 0.f, br.y, bi.y);
        }
    }
}

template <bool FAST>
__device__ __forceinline__ void fwd_replay(const float4* sc, const uint32_t* wre, const uint32_t* wim,
                                           const ModeConst& k0, const ModeConst& k1, float2& z0, float2& z1,
                                           uint32_t* yp, float* y32p, bool active, size_t row_words, int half_words) {
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
        const float4 ct = sc[i];
        if (ct.w == kTokPad) break;
        const float2 br = bf2_to_f2(wre[i * (kGroup / 2)]);
        const float2 bi = bf2_to_f2(wim[i * (kGroup / 2)]);
        if (ct.w == kTokNormal) {
            z0 = step_state(samu_lambda<FAST>(k0, ct), make_float2(br.x, bi.x), z0);
            z1 = step_state(samu_lambda<FAST>(k1, ct), make_float2(br.y, bi.y), z1);
        } else {
            z0 = make_float2(br.x, bi.x);
            z1 = make_float2(br.y, bi.y);
        }
        if (active) {
            uint32_t* o = yp + (size_t)i * row_words;
            __stcs(o, f2_to_bf2(z0.x, z1.x));
            __stcs(o + half_words, f2_to_bf2(z0.y, z1.y));
            if (y32p != nullptr) {
                float* f = y32p + (size_t)i * 2 * row_words;
                *reinterpret_cast<float2*>(f) = make_float2(z0.x, z1.x);
                *reinterpret_cast<float2*>(f + 2 * half_words) = make_float2(z0.y, z1.y);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanThreads, 3)
    samu_scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_w, SamuScanFwdArgs a) {
    __shared__ __align__(128) uint32_t s_wre[kTile][kGroup / 2];
    __shared__ __align__(128) uint32_t s_wim[kTile][kGroup / 2];
    __shared__ float4 s_ctrl[kTile];
    __shared__ float4 s_map[kScanWarps][32][2];
    __shared__ float4 s_ent[kScanWarps][32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint32_t s_tile;
    __shared__ int s_err;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        s_tile = atomicAdd(a.counter, 1u);
        mbar_init(&s_bar, 1);
    }
    __syncthreads();
    const ScanGeom& g = a.g;
    const long long tile = s_tile;
    const int chain = (int)(tile % g.n_chains);
    const int c = (int)(tile / g.n_chains);
    const int b = chain / g.n_groups;
    const int grp = chain % g.n_groups;
    const int M = g.lanes;
    const int L = g.L;
    const int CT = g.CT;
    const size_t D = 2 * (size_t)M;
    const int t0 = c * kTile;
    const int m = grp * kGroup + 2 * lane;
    const bool active = m < M;
    uint32_t* fl = a.flags + (size_t)chain * CT;

    if (tid == 0) {
        mbar_arrive_expect_tx(&s_bar, 2 * kBoxBytes);
        tma_load_3d(&s_wre[0][0], &tm_w, grp * kGroup, t0, b, &s_bar);
        tma_load_3d(&s_wim[0][0], &tm_w, M + grp * kGroup, t0, b, &s_bar);
    }
    if (tid < kTile) {
        const int t = t0 + tid;
        float4 ct = make_float4(0.f, 1.f, 0.f, kTokPad);
        if (t < L) {
            ct = a.ctrl[(size_t)b * L + t];
            ct.w = ct.w != 0.f ? kTokReset : kTokNormal;
        }
        s_ctrl[tid] = ct;
    }
    ModeConst k0 = {0.f, 0.f, 0.f, 0.f, 0.f}, k1 = k0;
    if (active) {
        k0 = load_mode(a.modes, a.nu, m);
        k1 = load_mode(a.modes, a.nu, m + 1);
    }
    const int r0 = warp * kSub;
    const int nsub = max(0, min(kSub, L - t0 - r0));
    const bool landed = mbar_wait_bounded(&s_bar, 0);
    if (!__syncthreads_and(landed)) {
        if (tid == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        mbar_wait_bounded(&s_bar, 0);
        return;
    }
    const float4* sc = s_ctrl + r0;
    const uint32_t* wre = &s_wre[r0][lane];
    const uint32_t* wim = &s_wim[r0][lane];
    const bool fast = use_fast_lambda(sc, lane, k0, k1);

    // sub-chunk summary S_w = T_e o ... o T_s
    float4 S0 = make_float4(1.f, 0.f, 0.f, 0.f), S1 = S0;
    if (fast)
        fwd_summary<true>(sc, wre, wim, k0, k1, S0, S1);
    else
        fwd_summary<false>(sc, wre, wim, k0, k1, S0, S1);
    s_map[warp][lane][0] = S0;
    s_map[warp][lane][1] = S1;
    __syncthreads();

    // warp 0: tile map, entry state (directly from the previous tile when its
    // state is already out, else by look-back), publish, sub-chunk entries
    if (warp == 0) {
        float4 A0 = s_map[0][lane][0], A1 = s_map[0][lane][1];
#pragma unroll
        for (int w = 1; w < kScanWarps; ++w) {
            A0 = compose_maps(s_map[w][lane][0], A0);
            A1 = compose_maps(s_map[w][lane][1], A1);
        }
        float2 h0v = make_float2(0.f, 0.f), h1v = h0v;
        bool err = false;
        const size_t hb = (size_t)b * g.CS;
        if (c == 0) {
            if (active && a.h0 != nullptr) {
                const float4 hv = *reinterpret_cast<const float4*>(a.h0 + ((size_t)b * M + m) * 2);
                h0v = make_float2(hv.x, hv.y);
                h1v = make_float2(hv.z, hv.w);
            }
        } else {
            int j = -1;
            if (ld_acquire_gpu(fl + c - 1) == kFlagIncl) {
                j = c - 1;
            } else {
                if (active) {
                    float4* ag = a.agg + ((size_t)b * CT + c) * M + m;
                    ag[0] = A0;
                    ag[1] = A1;
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(fl + c, kFlagAgg);
                j = lookback_find_warp(fl, c, CT, -1);
            }
            if (j < 0) {
                err = true;
            } else if (active) {
                const float4 hv = ldcg4(reinterpret_cast<const float4*>(
                    a.hsub + (hb + (size_t)(j + 1) * kScanWarps) * M + m));
                h0v = make_float2(hv.x, hv.y);
                h1v = make_float2(hv.z, hv.w);
                for (int i = j + 1; i < c; i += 4) {   // maps of tiles j+1 .. c-1, in time order
                    float4 T[4][2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i + q < c) {
                            const float4* ag = a.agg + ((size_t)b * CT + i + q) * M + m;
                            T[q][0] = ldcg4(ag);
                            T[q][1] = ldcg4(ag + 1);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i + q < c) {
                            h0v = capply(T[q][0], h0v);
                            h1v = capply(T[q][1], h1v);
                        }
                    }
                }
            }
        }
        if (!err) {
            if (active) {
                const float2 i0 = capply(A0, h0v);
                const float2 i1 = capply(A1, h1v);
                *reinterpret_cast<float4*>(a.hsub + (hb + (size_t)(c + 1) * kScanWarps) * M + m) =
                    make_float4(i0.x, i0.y, i1.x, i1.y);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(fl + c, kFlagIncl);
            // entry states of the sub-chunks (also kept for the backward)
            float2 e0 = h0v, e1 = h1v;
#pragma unroll
            for (int w = 0; w < kScanWarps; ++w) {
                s_ent[w][lane] = make_float4(e0.x, e0.y, e1.x, e1.y);
                if (active && (w > 0 || c == 0))
                    *reinterpret_cast<float4*>(a.hsub + (hb + (size_t)c * kScanWarps + w) * M + m) =
                        make_float4(e0.x, e0.y, e1.x, e1.y);
                e0 = capply(s_map[w][lane][0], e0);
                e1 = capply(s_map[w][lane][1], e1);
            }
        } else if (lane == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        if (lane == 0) s_err = err ? 1 : 0;
    }
    __syncthreads();
    if (s_err) return;

    // replay the sub-chunk from its entry state and write y
    const float4 e = s_ent[warp][lane];
    float2 z0 = make_float2(e.x, e.y), z1 = make_float2(e.z, e.w);
    const size_t yrow = (((size_t)b * L + t0 + r0) * D + m) / 2;
    uint32_t* yp = a.y + yrow;
    float* y32p = a.y32 != nullptr ? a.y32 + 2 * yrow : nullptr;
    if (fast)
        fwd_replay<true>(sc, wre, wim, k0, k1, z0, z1, yp, y32p, active, D / 2, M / 2);
    else
        fwd_replay<false>(sc, wre, wim, k0, k1, z0, z1, yp, y32p, active, D / 2, M / 2);
    if (active && nsub > 0 && t0 + r0 + nsub == L)
        *reinterpret_cast<float4*>(a.hT + ((size_t)b * M + m) * 2) = make_float4(z0.x, z0.y, z1.x, z1.y);
}

// ---------------------------------------------------------------------------
// Backward: forward sweep (rebuild u_t = lambda_t z_{t-1} and the reverse map
// of the sub-chunk) and reverse sweep (adjoint, dw, kappa sums).
// ---------------------------------------------------------------------------
template <bool FAST>
__device__ __forceinline__ void bwd_forward_sweep(const float4* sc, const uint32_t* wre, const uint32_t* wim,
                                                  const uint32_t* gre, const uint32_t* gim, const ModeConst& k0,
                                                  const ModeConst& k1, float2 z0, float2 z1, float4 (&u)[kSub],
                                                  float4& F0, float4& F1) {
    float2 P0 = make_float2(1.f, 0.f), P1 = P0;
    float2 q0 = make_float2(0.f, 0.f), q1 = q0;
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
        u[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 ct = sc[i];
        if (ct.w == kTokPad) continue;
        const float2 br = bf2_to_f2(wre[i * (kGroup / 2)]);
        const float2 bi = bf2_to_f2(wim[i * (kGroup / 2)]);
        if (ct.w == kTokNormal) {
            const float2 gr = bf2_to_f2(gre[i * (kGroup / 2)]);
            const float2 gi = bf2_to_f2(gim[i * (kGroup / 2)]);
            const float2 l0 = samu_lambda<FAST>(k0, ct);
            const float2 l1 = samu_lambda<FAST>(k1, ct);
            float2 u0, u1;
            z0 = step_state(l0, make_float2(br.x, bi.x), z0, &u0);
            z1 = step_state(l1, make_float2(br.y, bi.y), z1, &u1);
            u[i] = make_float4(u0.x, u0.y, u1.x, u1.y);
            P0 = cmul(l0, P0);
            P1 = cmul(l1, P1);
            const float2 c0 = cmulc(P0, make_float2(gr.x, gi.x));
            const float2 c1 = cmulc(P1, make_float2(gr.y, gi.y));
            q0 = make_float2(q0.x + c0.x, q0.y + c0.y);
            q1 = make_float2(q1.x + c1.x, q1.y + c1.y);
        } else {   // segment start: lambda = 0, nothing later reaches back past it
            z0 = make_float2(br.x, bi.x);
            z1 = make_float2(br.y, bi.y);
            P0 = make_float2(0.f, 0.f);
            P1 = P0;
        }
    }
    F0 = make_float4(P0.x, -P0.y, q0.x, q0.y);
    F1 = make_float4(P1.x, -P1.y, q1.x, q1.y);
}

template <bool FAST>
__device__ __forceinline__ void bwd_reverse_sweep(const float4* sc, const uint32_t* gre, const uint32_t* gim,
                                                  const ModeConst& k0, const ModeConst& k1, const float4 (&u)[kSub],
                                                  float2& A0, float2& A1, float4& acc, uint32_t* dwb, float* dwf,
                                                  bool fp32, bool active, size_t row_words, int half_words,
                                                  float2* kp, int kp_stride, int lane) {
#pragma unroll
    for (int i = kSub - 1; i >= 0; --i) {
        const float4 ct = sc[i];
        if (ct.w == kTokPad) continue;
        const float2 gr = bf2_to_f2(gre[i * (kGroup / 2)]);
        const float2 gi = bf2_to_f2(gim[i * (kGroup / 2)]);
        A0 = make_float2(A0.x + gr.x, A0.y + gi.x);
        A1 = make_float2(A1.x + gr.y, A1.y + gi.y);
        if (active) {
            if (fp32) {
                float* p = dwf + 2 * (size_t)i * row_words;
                *reinterpret_cast<float2*>(p) = make_float2(A0.x, A1.x);
                *reinterpret_cast<float2*>(p + 2 * half_words) = make_float2(A0.y, A1.y);
            } else {
                uint32_t* p = dwb + (size_t)i * row_words;
                __stcs(p, f2_to_bf2(A0.x, A1.x));
                __stcs(p + half_words, f2_to_bf2(A0.y, A1.y));
            }
        }
        if (ct.w == kTokNormal) {
            // kappa = A conj(u)
            const float4 uu = u[i];
            const float kr0 = __fmaf_rn(A0.x, uu.x, __fmul_rn(A0.y, uu.y));
            const float ki0 = __fmaf_rn(A0.y, uu.x, -__fmul_rn(A0.x, uu.y));
            const float kr1 = __fmaf_rn(A1.x, uu.z, __fmul_rn(A1.y, uu.w));
            const float ki1 = __fmaf_rn(A1.y, uu.z, -__fmul_rn(A1.x, uu.w));
            const float Et = 1.0f + ct.x;   // ct.x holds E - 1
            acc.x = __fmaf_rn(-Et, kr0, acc.x);   // dnu_m
            acc.y += ki0;                         // dtheta_m
            acc.z = __fmaf_rn(-Et, kr1, acc.z);
            acc.w += ki1;
            float td = ki0 + ki1;
            float te = -__fmaf_rn(k0.nu, kr0, __fmul_rn(k1.nu, kr1));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                td += __shfl_xor_sync(0xffffffffu, td, o);
                te += __shfl_xor_sync(0xffffffffu, te, o);
            }
            if (lane == 0) kp[(size_t)i * kp_stride] = make_float2(td, te);
            A0 = cmulc(samu_lambda<FAST>(k0, ct), A0);
            A1 = cmulc(samu_lambda<FAST>(k1, ct), A1);
        } else {   // segment start: no controller terms, the adjoint stops here
            if (lane == 0) kp[(size_t)i * kp_stride] = make_float2(0.f, 0.f);
            A0 = make_float2(0.f, 0.f);
            A1 = A0;
        }
    }
}

// Tiles in reverse time order.  Forward sweep of each sub-chunk from its saved
// entry state rebuilds lambda_t, u_t = lambda_t z_{t-1} (kept in registers for
// kappa) and z_t, and accumulates the prefix product P_t = lambda_s..lambda_t
// and q = sum_t conj(P_t) dy_t: the sub-chunk maps an adjoint R arriving at its
// last token to the adjoint leaving it towards the past, R' = conj(P_e) R + q.
// Warp 0 composes the 8 sub-chunk maps, takes the incoming adjoint from the
// next tile (or by look-back), and hands each sub-chunk its incoming adjoint.
// Reverse sweep: A_t = dy_t + (adjoint from t+1); dw_t = A_t;
// kappa_t = A_t conj(u_t);  dtheta_m += Im kappa, dnu_m += -E_t Re kappa,
// dbar_t += Im kappa, Ebar_t += -nu_m Re kappa (reduced over the 64 modes of
// the warp: one per-token partial per mode group).
__global__ void __launch_bounds__(kScanThreads, 2)
    samu_scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_w,
                         SamuScanBwdArgs a) {
    extern __shared__ __align__(128) uint8_t s_dyn[];   // boxes: dy re, dy im, w re, w im
    uint32_t (*s_gre)[kGroup / 2] = reinterpret_cast<uint32_t (*)[kGroup / 2]>(s_dyn);
    uint32_t (*s_gim)[kGroup / 2] = reinterpret_cast<uint32_t (*)[kGroup / 2]>(s_dyn + kBoxBytes);
    uint32_t (*s_wre)[kGroup / 2] = reinterpret_cast<uint32_t (*)[kGroup / 2]>(s_dyn + 2 * kBoxBytes);
    uint32_t (*s_wim)[kGroup / 2] = reinterpret_cast<uint32_t (*)[kGroup / 2]>(s_dyn + 3 * kBoxBytes);
    __shared__ float4 s_ctrl[kTile];
    __shared__ float4 s_map[kScanWarps][32][2];
    __shared__ float4 s_ent[kScanWarps][32];
    __shared__ float4 s_acc[kScanWarps][32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint32_t s_tile;
    __shared__ int s_err;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        s_tile = atomicAdd(a.counter, 1u);
        mbar_init(&s_bar, 1);
    }
    __syncthreads();
    const ScanGeom& g = a.g;
    const long long tile = s_tile;
    const int chain = (int)(tile % g.n_chains);
    const int CT = g.CT;
    const int c = CT - 1 - (int)(tile / g.n_chains);
    const int b = chain / g.n_groups;
    const int grp = chain % g.n_groups;
    const int M = g.lanes;
    const int L = g.L;
    const size_t D = 2 * (size_t)M;
    const int t0 = c * kTile;
    const int m = grp * kGroup + 2 * lane;
    const bool active = m < M;
    uint32_t* fl = a.flags + (size_t)chain * CT;
    const size_t hb = (size_t)b * g.CS;

    if (tid == 0) {
        mbar_arrive_expect_tx(&s_bar, 4 * kBoxBytes);
        tma_load_3d(&s_gre[0][0], &tm_dy, grp * kGroup, t0, b, &s_bar);
        tma_load_3d(&s_gim[0][0], &tm_dy, M + grp * kGroup, t0, b, &s_bar);
        tma_load_3d(&s_wre[0][0], &tm_w, grp * kGroup, t0, b, &s_bar);
        tma_load_3d(&s_wim[0][0], &tm_w, M + grp * kGroup, t0, b, &s_bar);
    }
    if (tid < kTile) {
        const int t = t0 + tid;
        float4 ct = make_float4(0.f, 1.f, 0.f, kTokPad);
        if (t < L) {
            ct = a.ctrl[(size_t)b * L + t];
            ct.w = ct.w != 0.f ? kTokReset : kTokNormal;
        }
        s_ctrl[tid] = ct;
    }
    ModeConst k0 = {0.f, 0.f, 0.f, 0.f, 0.f}, k1 = k0;
    const int r0 = warp * kSub;
    const int nsub = max(0, min(kSub, L - t0 - r0));
    float2 z0 = make_float2(0.f, 0.f), z1 = z0;
    if (active) {
        k0 = load_mode(a.modes, a.nu, m);
        k1 = load_mode(a.modes, a.nu, m + 1);
        if (nsub > 0) {
            const float4 hv = ldcg4(reinterpret_cast<const float4*>(
                a.hsub + (hb + (size_t)c * kScanWarps + warp) * M + m));
            z0 = make_float2(hv.x, hv.y);
            z1 = make_float2(hv.z, hv.w);
        }
    }
    const bool landed = mbar_wait_bounded(&s_bar, 0);
    if (!__syncthreads_and(landed)) {
        if (tid == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        mbar_wait_bounded(&s_bar, 0);
        return;
    }
    const float4* sc = s_ctrl + r0;
    const uint32_t* wre = &s_wre[r0][lane];
    const uint32_t* wim = &s_wim[r0][lane];
    const uint32_t* gre = &s_gre[r0][lane];
    const uint32_t* gim = &s_gim[r0][lane];
    const bool fast = use_fast_lambda(sc, lane, k0, k1);

    float4 u[kSub];   // {u_m, u_m+1} per token
    float4 F0, F1;
    if (fast)
        bwd_forward_sweep<true>(sc, wre, wim, gre, gim, k0, k1, z0, z1, u, F0, F1);
    else
        bwd_forward_sweep<false>(sc, wre, wim, gre, gim, k0, k1, z0, z1, u, F0, F1);
    s_map[warp][lane][0] = F0;
    s_map[warp][lane][1] = F1;
    __syncthreads();

    // warp 0: reverse tile map F_0 o F_1 o ... o F_7 (F_7 first), incoming adjoint, hand-out
    if (warp == 0) {
        float4 A0 = s_map[kScanWarps - 1][lane][0], A1 = s_map[kScanWarps - 1][lane][1];
#pragma unroll
        for (int w = kScanWarps - 2; w >= 0; --w) {
            A0 = compose_maps(s_map[w][lane][0], A0);
            A1 = compose_maps(s_map[w][lane][1], A1);
        }
        float2 R0 = make_float2(0.f, 0.f), R1 = R0;
        bool err = false;
        if (c == CT - 1) {
            if (active && a.dhT != nullptr) {
                const float4 v = *reinterpret_cast<const float4*>(a.dhT + ((size_t)b * M + m) * 2);
                R0 = make_float2(v.x, v.y);
                R1 = make_float2(v.z, v.w);
            }
        } else {
            int j = -1;
            if (ld_acquire_gpu(fl + c + 1) == kFlagIncl) {
                j = c + 1;
            } else {
                if (active) {
                    float4* ag = a.agg + ((size_t)b * CT + c) * M + m;
                    ag[0] = A0;
                    ag[1] = A1;
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(fl + c, kFlagAgg);
                j = lookback_find_warp(fl, c, CT, +1);
            }
            if (j < 0) {
                err = true;
            } else if (active) {
                const float4 rv = ldcg4(reinterpret_cast<const float4*>(a.rin + ((size_t)b * CT + j) * M + m));
                R0 = make_float2(rv.x, rv.y);
                R1 = make_float2(rv.z, rv.w);
                for (int i = j - 1; i > c; i -= 4) {   // maps of tiles j-1 .. c+1 (later first)
                    float4 T[4][2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i - q > c) {
                            const float4* ag = a.agg + ((size_t)b * CT + i - q) * M + m;
                            T[q][0] = ldcg4(ag);
                            T[q][1] = ldcg4(ag + 1);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i - q > c) {
                            R0 = capply(T[q][0], R0);
                            R1 = capply(T[q][1], R1);
                        }
                    }
                }
            }
        }
        if (!err) {
            if (active) {
                const float2 o0 = capply(A0, R0);
                const float2 o1 = capply(A1, R1);
                *reinterpret_cast<float4*>(a.rin + ((size_t)b * CT + c) * M + m) = make_float4(o0.x, o0.y, o1.x, o1.y);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(fl + c, kFlagIncl);
            float2 r0v = R0, r1v = R1;
#pragma unroll
            for (int w = kScanWarps - 1; w >= 0; --w) {
                s_ent[w][lane] = make_float4(r0v.x, r0v.y, r1v.x, r1v.y);
                r0v = capply(s_map[w][lane][0], r0v);
                r1v = capply(s_map[w][lane][1], r1v);
            }
        } else if (lane == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        if (lane == 0) s_err = err ? 1 : 0;
    }
    __syncthreads();
    if (s_err) return;

    // reverse sweep
    const float4 e = s_ent[warp][lane];
    float2 A0 = make_float2(e.x, e.y), A1 = make_float2(e.z, e.w);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);   // dnu_m, dtheta_m, dnu_m+1, dtheta_m+1
    const size_t row = (((size_t)b * L + t0 + r0) * D + m) / 2;
    uint32_t* dwb = reinterpret_cast<uint32_t*>(a.dw) + row;
    float* dwf = reinterpret_cast<float*>(a.dw) + 2 * row;
    float2* kp = a.kpart + ((size_t)b * L + t0 + r0) * g.n_groups + grp;
    if (fast)
        bwd_reverse_sweep<true>(sc, gre, gim, k0, k1, u, A0, A1, acc, dwb, dwf, a.grad_fp32 != 0, active, D / 2,
                                M / 2, kp, g.n_groups, lane);
    else
        bwd_reverse_sweep<false>(sc, gre, gim, k0, k1, u, A0, A1, acc, dwb, dwf, a.grad_fp32 != 0, active, D / 2,
                                 M / 2, kp, g.n_groups, lane);
    if (c == 0 && warp == 0 && active)
        *reinterpret_cast<float4*>(a.dh0 + ((size_t)b * M + m) * 2) = make_float4(A0.x, A0.y, A1.x, A1.y);
    s_acc[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && active) {
        float4 s = s_acc[0][lane];
#pragma unroll
        for (int w = 1; w < kScanWarps; ++w) {
            const float4 v = s_acc[w][lane];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        *reinterpret_cast<float4*>(a.numod + ((size_t)b * CT + c) * M + m) = s;
    }
}

// ---------------------------------------------------------------------------
cudaError_t launch_samu_scan_fwd(const CUtensorMap& tm_w, const SamuScanFwdArgs& args, cudaStream_t s) {
    samu_scan_fwd_kernel<<<(unsigned)args.g.n_tiles, kScanThreads, 0, s>>>(tm_w, args);
    return cudaGetLastError();
}

cudaError_t launch_samu_scan_bwd(const CUtensorMap& tm_dy, const CUtensorMap& tm_w,
                                 const SamuScanBwdArgs& args, cudaStream_t s) {
    const int smem = 4 * kBoxBytes;
    cudaError_t e = cudaFuncSetAttribute(samu_scan_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    samu_scan_bwd_kernel<<<(unsigned)args.g.n_tiles, kScanThreads, smem, s>>>(tm_dy, tm_w, args);
    return cudaGetLastError();
}

}  // namespace lrs

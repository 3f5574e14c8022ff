// RG-LRU real scan on the same tiled look-back engine (comparison path).
//
// Equations: SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比"), section 04:
// g^x = sigmoid(l^x), g^a = sigmoid(l^a), a_t = exp(-8 g^a softplus(alpha)),
// b_t = x_t g^x sqrt(max(1 - a_t^2, 0)), h_t = a_t h_{t-1} + b_t, with the gate
// preparation fused into the scan (no materialised a/b tensors) and, at a
// segment start, a_t = 0 and a unit normaliser ("Griffin 第 4、5 节 H800 对照
// 协议", "RG-LRU 的固定方程").  1 - a^2 is evaluated as -expm1(2 log a) so the
// normaliser keeps full FP32 relative accuracy when a is close to 1.  The
// gate functions use the SFU's approximations (sigmoid, square roots) and a
// short series for expm1: the IEEE-rounded library forms cost several times
// the instructions and the recurrence does not amplify these errors.
//
// Tiling as in the SAMU scan: a chain is (batch row, 64 channels), a CTA owns
// a 128-token tile (x, l^x, l^a and, backward, dy staged by TMA), 8 warps of
// 16-token sub-chunks, lane l owns channels 2l, 2l+1 (paired FP32 arithmetic),
// decoupled look-back between tiles.
//
// The same kernels serve the mixer with its two 16-block block-diagonal gate
// projections (logit modes 1 and 2 below; the "PL" variants): the logits are
// x W (+ the biases, added on reading), FP32 products of the library's
// tensor-core contraction kernel or, in the forward, formed per tile on the
// tensor cores inside the scan.
#include <algorithm>
#include <atomic>

#include "kernels.cuh"
#include "umma.cuh"

namespace lrs {

constexpr int kRgThreads = kRgWarps * 32;
constexpr int kRgBoxBytes = kRgTile * kRowBytes;   // one BF16 [128 x 64] box

// Where the gate logits come from (the kernels' LM parameter):
//   0  BF16 [128 x 64] boxes of the raw l^x, l^a inputs;
//   1  FP32 [128 x 64] boxes of the products x W (tensor-core contraction
//      kernel), biases added on reading;
//   2  computed in the kernel on the tensor cores (forward): the tile's x box
//      (TMA, 128-byte swizzle) times the group's packed weights (both gates),
//      FP32 accumulators in tensor memory, staged to shared memory one gate
//      at a time as [128 tokens][kStageRow] FP32; biases added on reading.
//      (One gate's staging area keeps the CTA at two per SM.)
constexpr int kStageRow = 68;                              // padded row: conflict-free staging stores
constexpr int kStageBytes = kRgTile * kStageRow * 4;       // one gate
constexpr int kWimgBytes = 2 * kGroup * kGroup * 2;        // both gates' [64 x 64] BF16 weight images

template <int LM>
struct RgLogits {
    static constexpr int kBoxBytes = LM == 2 ? 0 : (LM == 1 ? 2 * kRgBoxBytes : kRgBoxBytes);
    static constexpr int kSlotBytes = LM == 2 ? kRgBoxBytes + kWimgBytes : kRgBoxBytes + 2 * kBoxBytes;
};

// Logits mode 2: one gate's [128 tokens x 64] FP32 products from tensor memory
// to the staging area [128][kStageRow]; warp w drains tokens 32 (w % 4) .. + 31
// (the tensor-memory lanes it may read), columns 32 (w / 4) .. + 31.
__device__ __forceinline__ void rg_stage_gate(uint32_t tmem, uint8_t* s_stage, int gt, int warp, int lane) {
    const int q = warp & 3, ch = 32 * (warp >> 2);
    float* st = reinterpret_cast<float*>(s_stage) + (size_t)(32 * q + lane) * kStageRow;
#pragma unroll
    for (int col = 0; col < 32; col += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(gt * kGroup + ch + col), v);
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(st + ch + col + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
}

// The lane's two logits of token row r (biases added for LM >= 1).
template <int LM>
__device__ __forceinline__ float2 rg_logit(const uint8_t* box, int r, int lane, float2 bias) {
    if (LM >= 1) {
        const float2 v = LM == 2 ? reinterpret_cast<const float2*>(box)[(r * kStageRow) / 2 + lane]
                                 : reinterpret_cast<const float2*>(box)[r * 32 + lane];
        return make_float2(v.x + bias.x, v.y + bias.y);
    }
    return bf2_to_f2(reinterpret_cast<const uint32_t*>(box)[r * 32 + lane]);
}

// The lane's two x values of token row r (the box is 128-byte swizzled for LM 2:
// the 16-byte chunk j of row r sits at chunk j ^ (r % 8)).
template <int LM>
__device__ __forceinline__ float2 rg_x(const uint8_t* box, int r, int lane) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(box);
    if (LM == 2) return bf2_to_f2(w[r * 32 + ((((lane >> 2) ^ (r & 7))) << 2) + (lane & 3)]);
    return bf2_to_f2(w[r * 32 + lane]);
}

// Gate arithmetic for the lane's two channels at once, as FP32 pairs (paired
// f32x2 instructions; the SFU approximations run per element).
//  - sigmoid(v) = 1 / (1 + e^{-v}) from two SFU operations.  Its ~2^-22
//    relative error only scales the write gate and, through
//    log a = g^a (-8 softplus), moves log a by at most ~1e-8 absolute:
//    nothing accumulates through the recurrence.
//  - e^v - 1: for |v| < 1/4 its Taylor series through v^8 (coefficients 1/k!;
//    the remainder is below 1e-10 relative there), so that 1 - a^2 keeps full
//    relative accuracy when a is close to 1; otherwise e^v - 1 from ex2, where
//    the cancellation costs at most a factor 4.
//  - a = e^{log a}, u = 1 - a^2 = -(e^{2 log a} - 1), n = sqrt(max(u, 0));
//    at a segment start a = 0 and n = 1.
struct RgGate2 {
    f2x a, n, u, gx, ga;   // retention, write normaliser, 1 - a^2, sigmoid(l^x), sigmoid(l^a)
};

__device__ __forceinline__ f2x sfu_ex2(f2x t) {
    float t0, t1;
    up2(t, t0, t1);
    return pk2(ex2_approx(t0), ex2_approx(t1));
}

__device__ __forceinline__ f2x sigmoid2(f2x v) {
    float d0, d1;
    up2(add2(dup2(1.0f), sfu_ex2(mul2(v, dup2(-kLog2e)))), d0, d1);
    return pk2(rcp_approx(d0), rcp_approx(d1));
}

__device__ __forceinline__ f2x expm1_2(f2x v) {
    f2x p = fma2(v, dup2(1.0f / 40320.0f), dup2(1.0f / 5040.0f));
    p = fma2(v, p, dup2(1.0f / 720.0f));
    p = fma2(v, p, dup2(1.0f / 120.0f));
    p = fma2(v, p, dup2(1.0f / 24.0f));
    p = fma2(v, p, dup2(1.0f / 6.0f));
    p = fma2(v, p, dup2(0.5f));
    p = fma2(v, p, dup2(1.0f));
    const f2x series = mul2(v, p);
    float v0, v1;
    up2(v, v0, v1);
    if (fabsf(v0) < 0.25f && fabsf(v1) < 0.25f) return series;
    float s0, s1;
    up2(series, s0, s1);
    return pk2(fabsf(v0) < 0.25f ? s0 : ex2_approx(v0 * kLog2e) - 1.0f,
               fabsf(v1) < 0.25f ? s1 : ex2_approx(v1 * kLog2e) - 1.0f);
}

// The keep gate's part (everything but g^x) from l^a.
__device__ __forceinline__ RgGate2 rg_keep_gate2(f2x la, f2x nsp, bool is_reset) {
    RgGate2 gt;
    gt.gx = 0ull;
    gt.ga = sigmoid2(la);
    const f2x lg = mul2(gt.ga, nsp);   // log a
    gt.a = sfu_ex2(mul2(lg, dup2(kLog2e)));
    gt.u = sub2(0ull, expm1_2(mul2(dup2(2.0f), lg)));
    float u0, u1;
    up2(gt.u, u0, u1);
    gt.n = pk2(sqrt_approx(fmaxf(u0, 0.0f)), sqrt_approx(fmaxf(u1, 0.0f)));
    if (is_reset) {
        gt.a = 0ull;
        gt.n = dup2(1.0f);
    }
    return gt;
}

__device__ __forceinline__ RgGate2 rg_gate2(f2x lx, f2x la, f2x nsp, bool is_reset) {
    RgGate2 gt = rg_keep_gate2(la, nsp, is_reset);
    gt.gx = sigmoid2(lx);
    return gt;
}

__device__ __forceinline__ float softplus_f(float v) {
    return v > 0.f ? v + log1pf(expf(-v)) : log1pf(expf(v));
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
// Thread 0: the boxes of `tile` into ring slot `slot` (LM 2: the x box and
// the group's weight images).
template <int LM>
__device__ __forceinline__ void rg_fwd_issue(uint8_t* slot_base, uint64_t* bar, const CUtensorMap* tm_x,
                                             const CUtensorMap* tm_lx, const CUtensorMap* tm_la,
                                             const uint8_t* wimg, const ScanGeom& g, long long tile) {
    constexpr int LB = RgLogits<LM>::kBoxBytes;
    const int chain = (int)(tile % g.n_chains);
    const int c = (int)(tile / g.n_chains);
    const int b = chain / g.n_groups, grp = chain % g.n_groups;
    fence_proxy_async();
    mbar_arrive_expect_tx(bar, RgLogits<LM>::kSlotBytes);
    tma_load_3d(slot_base, tm_x, grp * kGroup, c * kRgTile, b, bar);
    if (LM == 2) {
        bulk_load(slot_base + kRgBoxBytes, wimg + (size_t)grp * kWimgBytes, kWimgBytes, bar);
    } else {
        tma_load_3d(slot_base + kRgBoxBytes, tm_lx, grp * kGroup, c * kRgTile, b, bar);
        tma_load_3d(slot_base + kRgBoxBytes + LB, tm_la, grp * kGroup, c * kRgTile, b, bar);
    }
}

// Persistent CTAs: each takes tiles in ticket order (atomic counter) and keeps
// the next ticket's boxes in flight in the second slot of a two-slot ring
// while it works on the current one.  Tickets are taken in increasing order
// by every CTA and each CTA finishes its current tile before its prefetched
// one, so the smallest tile in progress always finds its predecessors done.
template <int LM>
__global__ void __launch_bounds__(kRgThreads, 2)
    rglru_scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_lx,
                          const __grid_constant__ CUtensorMap tm_la, RglruScanFwdArgs a) {
    constexpr bool PL = LM >= 1;
    constexpr int LB = RgLogits<LM>::kBoxBytes;
    constexpr int SB = RgLogits<LM>::kSlotBytes;
    constexpr uint32_t kIdesc = umma_idesc_bf16(kRgTile, kGroup);
    extern __shared__ __align__(1024) uint8_t s_raw[];   // [slot][x, l^x, l^a boxes] (+ LM 2 staging)
    __shared__ uint8_t s_rst[kRgTile];
    __shared__ float4 s_map[kRgWarps][32];
    __shared__ float2 s_ent[kRgWarps][32];
    __shared__ __align__(8) uint64_t s_bars[2];
    __shared__ __align__(8) uint64_t s_mma_bar;
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_tick[2];
    __shared__ int s_err;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const ScanGeom& g = a.g;
    const uint32_t n_tiles = (uint32_t)g.n_tiles;
    // the slots start on a 1024-byte boundary (the 128-byte swizzle's atom; one
    // spare kilobyte of dynamic shared memory is requested for this)
    uint8_t* s_dyn = s_raw + ((1024u - (smem_u32(s_raw) & 1023u)) & 1023u);
    uint8_t* s_stage = s_dyn + 2 * SB;
    if (LM == 2 && warp == 0) {   // two gates x 64 FP32 columns of tensor memory
        tmem_alloc(&s_tmem, 2 * kGroup);
        tmem_fence_before_sync();
    }
    if (tid == 0) {
        mbar_init(&s_bars[0], 1);
        mbar_init(&s_bars[1], 1);
        if (LM == 2) mbar_init(&s_mma_bar, 1);
        s_tick[0] = atomicAdd(a.counter, 1u);
        if (s_tick[0] < n_tiles) rg_fwd_issue<LM>(s_dyn, &s_bars[0], &tm_x, &tm_lx, &tm_la, a.wimg, g, s_tick[0]);
    }
    __syncthreads();
    if (LM == 2) tmem_fence_after_sync();
    const uint32_t tmem = LM == 2 ? s_tmem : 0u;
    int pend = -1;       // iteration whose prefetched copy is outstanding when the loop is left early
    int mma_lost = -1;   // LM 2: iteration whose MMA completion was not seen
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    const uint32_t tile_u = s_tick[slot];
    if (tile_u >= n_tiles) break;
    if (tid == 0) {   // the next ticket into the other slot (free since the end of the previous tile)
        s_tick[slot ^ 1] = atomicAdd(a.counter, 1u);
        if (s_tick[slot ^ 1] < n_tiles)
            rg_fwd_issue<LM>(s_dyn + (size_t)(slot ^ 1) * SB, &s_bars[slot ^ 1], &tm_x, &tm_lx, &tm_la, a.wimg, g,
                             s_tick[slot ^ 1]);
    }
    uint8_t* sb = s_dyn + (size_t)slot * SB;
    const uint8_t* s_x = sb;
    const uint8_t* s_lx = LM == 2 ? s_stage : sb + kRgBoxBytes;
    const uint8_t* s_la = LM == 2 ? s_stage : sb + kRgBoxBytes + LB;   // LM 2: the same area, one gate at a time
    const long long tile = tile_u;
    const int chain = (int)(tile % g.n_chains);
    const int c = (int)(tile / g.n_chains);
    const int b = chain / g.n_groups;
    const int grp = chain % g.n_groups;
    const int D = g.lanes;
    const int L = g.L;
    const int CT = g.CT;
    const int t0 = c * kRgTile;
    const int d = grp * kGroup + 2 * lane;
    const bool active = d < D;
    uint32_t* fl = a.flags + (size_t)chain * CT;
    const size_t hb = (size_t)b * g.CS;

    if (tid < kRgTile) {
        const int t = t0 + tid;
        s_rst[tid] = (t < L && a.reset != nullptr && a.reset[(size_t)b * L + t] != 0) ? 1 : 0;
    }
    float nsp0 = 0.f, nsp1 = 0.f;
    float2 bxv = make_float2(0.f, 0.f), bav = bxv;
    if (active) {
        nsp0 = -8.0f * softplus_f(a.alpha[d]);
        nsp1 = -8.0f * softplus_f(a.alpha[d + 1]);
        if (PL) {
            bxv = *reinterpret_cast<const float2*>(a.bx + d);
            bav = *reinterpret_cast<const float2*>(a.ba + d);
        }
    }
    const int r0 = warp * kSub;
    const int nsub = max(0, min(kSub, L - t0 - r0));
    const bool landed = mbar_wait_bounded(&s_bars[slot], (uint32_t)(it >> 1) & 1u);
    if (!__syncthreads_and(landed)) {
        if (tid == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        pend = it + 1;
        break;
    }
    if (LM == 2) {
        // logits of the tile: D_gate[128 x 64] = x[128 x 64] . Wimg_gate[64 x 64]^T,
        // four K = 16 steps per gate, issued by one thread
        if (tid == 0) {
            tmem_fence_after_sync();
            const uint32_t xa = smem_u32(sb), wa = smem_u32(sb + kRgBoxBytes);
#pragma unroll
            for (int gt = 0; gt < 2; ++gt)
#pragma unroll
                for (int ks = 0; ks < kGroup / 16; ++ks)
                    umma_bf16(tmem + (uint32_t)(gt * kGroup), umma_desc_sw128(xa + 32u * ks),
                              umma_desc_sw128(wa + (uint32_t)(gt * kGroup * kGroup * 2) + 32u * ks), kIdesc, ks > 0);
            umma_commit(&s_mma_bar);
        }
        const bool done = mbar_wait_bounded(&s_mma_bar, (uint32_t)it & 1u);
        if (!__syncthreads_and(done)) {
            if (tid == 0) {
                st_release_gpu(fl + c, kFlagErr);
                atomicOr(a.status, kStatusTimeout);
            }
            pend = it + 1;
            mma_lost = it;
            break;
        }
        tmem_fence_after_sync();
    }

    // the lane's two channels as pairs: a_t, b_t per token; the sub-chunk map (SA, SB)
    f2x av[kSub], bv[kSub];
    f2x SA = dup2(1.0f), SB = 0ull;
    const f2x nsp = pk2(nsp0, nsp1);
    if (LM == 2) {
        // gate 0 (write gate) staged: x g^x per token; then gate 1 (keep gate) into
        // the same area: a, the normaliser n and b = (x g^x) n
#pragma unroll
        for (int gt = 0; gt < 2; ++gt) {
            rg_stage_gate(tmem, s_stage, gt, warp, lane);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kSub; ++i) {
                if (gt == 0) {
                    av[i] = dup2(1.0f);
                    bv[i] = 0ull;
                }
                if (i < nsub) {
                    if (gt == 0) {
                        const float2 xx = rg_x<LM>(s_x, r0 + i, lane);
                        const float2 gl = rg_logit<LM>(s_lx, r0 + i, lane, bxv);
                        bv[i] = mul2(pk2(xx.x, xx.y), sigmoid2(pk2(gl.x, gl.y)));
                    } else {
                        const float2 al = rg_logit<LM>(s_la, r0 + i, lane, bav);
                        const RgGate2 kg = rg_keep_gate2(pk2(al.x, al.y), nsp, s_rst[r0 + i] != 0);
                        av[i] = kg.a;
                        bv[i] = mul2(bv[i], kg.n);
                        SA = mul2(av[i], SA);                // (a, b) o (A, B) = (a A, a B + b)
                        SB = fma2(av[i], SB, bv[i]);
                    }
                }
            }
            if (gt == 0) __syncthreads();   // every warp has read gate 0 before gate 1 overwrites it
        }
        tmem_fence_before_sync();
    } else {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            av[i] = dup2(1.0f);
            bv[i] = 0ull;
            if (i < nsub) {
                const bool rs = s_rst[r0 + i] != 0;
                const float2 xx = rg_x<LM>(s_x, r0 + i, lane);
                const float2 gl = rg_logit<LM>(s_lx, r0 + i, lane, bxv);
                const float2 al = rg_logit<LM>(s_la, r0 + i, lane, bav);
                const RgGate2 gt = rg_gate2(pk2(gl.x, gl.y), pk2(al.x, al.y), nsp, rs);
                av[i] = gt.a;
                bv[i] = mul2(mul2(pk2(xx.x, xx.y), gt.gx), gt.n);
                SA = mul2(av[i], SA);                // (a, b) o (A, B) = (a A, a B + b)
                SB = fma2(av[i], SB, bv[i]);
            }
        }
    }
    {
        float A0, A1, B0, B1;
        up2(SA, A0, A1);
        up2(SB, B0, B1);
        s_map[warp][lane] = make_float4(A0, B0, A1, B1);
    }
    // the previous tile's flag, read while the other warps finish their maps
    const uint32_t pflag = (warp == 0 && lane == 0 && c > 0) ? ld_acquire_gpu(fl + c - 1) : 0u;
    __syncthreads();

    if (warp == 0) {
        float4 A = s_map[0][lane];
#pragma unroll
        for (int w = 1; w < kRgWarps; ++w) {
            const float4 Sw = s_map[w][lane];
            const float2 t0v = rcompose(make_float2(Sw.x, Sw.y), make_float2(A.x, A.y));
            const float2 t1v = rcompose(make_float2(Sw.z, Sw.w), make_float2(A.z, A.w));
            A = make_float4(t0v.x, t0v.y, t1v.x, t1v.y);
        }
        float h0v = 0.f, h1v = 0.f;
        bool err = false;
        if (c == 0) {
            if (active && a.h0 != nullptr) {
                const float2 hv = *reinterpret_cast<const float2*>(a.h0 + (size_t)b * D + d);
                h0v = hv.x;
                h1v = hv.y;
            }
        } else {
            // the neighbouring tile already inclusive: its state
            // is the entry and this tile's map need not be published
            int j = __shfl_sync(0xffffffffu, pflag, 0) == kFlagIncl ? c - 1 : -2;
            if (j == -2) {
                if (active)
                    *reinterpret_cast<float4*>(a.agg + ((size_t)b * CT + c) * D + d) = A;
                __syncwarp();
                if (lane == 0) st_release_gpu(fl + c, kFlagAgg);
                j = lookback_find_warp(fl, c, CT, -1);
            }
            if (j < 0) {
                err = true;
            } else if (active) {
                const float2 hv = __ldcg(reinterpret_cast<const float2*>(
                    a.hsub + (hb + (size_t)(j + 1) * kRgWarps) * D + d));
                h0v = hv.x;
                h1v = hv.y;
                for (int i = j + 1; i < c; i += 4) {
                    float4 T[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (i + q < c)
                            T[q] = ldcg4(reinterpret_cast<const float4*>(a.agg + ((size_t)b * CT + i + q) * D + d));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i + q < c) {
                            h0v = rapply(make_float2(T[q].x, T[q].y), h0v);
                            h1v = rapply(make_float2(T[q].z, T[q].w), h1v);
                        }
                    }
                }
            }
        }
        if (!err) {
            float e0 = h0v, e1 = h1v;
#pragma unroll
            for (int w = 0; w < kRgWarps; ++w) {
                s_ent[w][lane] = make_float2(e0, e1);
                if (active && (w > 0 || c == 0))
                    *reinterpret_cast<float2*>(a.hsub + (hb + (size_t)c * kRgWarps + w) * D + d) = make_float2(e0, e1);
                const float4 Sw = s_map[w][lane];
                e0 = rapply(make_float2(Sw.x, Sw.y), e0);
                e1 = rapply(make_float2(Sw.z, Sw.w), e1);
            }
            if (active)
                *reinterpret_cast<float2*>(a.hsub + (hb + (size_t)(c + 1) * kRgWarps) * D + d) =
                    make_float2(rapply(make_float2(A.x, A.y), h0v), rapply(make_float2(A.z, A.w), h1v));
        } else if (lane == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        if (lane == 0) s_err = err ? 1 : 0;
    }
    __syncthreads();
    if (s_err) {
        pend = it + 1;
        break;
    }
    if (warp == 0) {   // the state after the tile, published while the other warps replay
        __syncwarp();
        if (lane == 0) st_release_gpu(fl + c, kFlagIncl);
    }

    const float2 e = s_ent[warp][lane];
    f2x z = pk2(e.x, e.y);
    const size_t row = (((size_t)b * L + t0 + r0) * D + d) / 2;
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
        if (i < nsub) {
            z = fma2(av[i], z, bv[i]);
            if (active) {
                const size_t o = row + (size_t)i * (D / 2);
                float z0, z1;
                up2(z, z0, z1);
                __stcs(a.y + o, f2_to_bf2(z0, z1));
                if (a.y32 != nullptr) *reinterpret_cast<float2*>(a.y32 + 2 * o) = make_float2(z0, z1);
            }
        }
    }
    if (active && nsub > 0 && t0 + r0 + nsub == L) {
        float z0, z1;
        up2(z, z0, z1);
        *reinterpret_cast<float2*>(a.hT + (size_t)b * D + d) = make_float2(z0, z1);
    }
    __syncthreads();   // this slot and s_rst free; the next ticket visible
  }
    // leaving early (a failed wait): the next ticket's copy, or the tile's
    // MMA, may still be in flight
    if (tid == 0 && pend >= 0 && s_tick[pend & 1] < n_tiles)
        mbar_wait_bounded(&s_bars[pend & 1], (uint32_t)(pend >> 1) & 1u);
    if (LM == 2) {
        if (tid == 0 && mma_lost >= 0) mbar_wait_bounded(&s_mma_bar, (uint32_t)mma_lost & 1u);
        __syncthreads();
        if (warp == 0) {
            tmem_fence_after_sync();
            tmem_dealloc(tmem, 2 * kGroup);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward.  Forward sweep from the saved sub-chunk entry: h_{t-1} (kept in
// registers), the prefix product P_t = a_s..a_t and q = sum_t P_t dy_t; the
// sub-chunk maps an adjoint R arriving at its last token to R' = P_e R + q.
// Warp 0 composes, looks back over later tiles and hands out incoming
// adjoints.  Reverse sweep with the gate derivatives:
//   H_t = dy_t + a_{t+1} H_{t+1};  dx = H g^x n;  dl^x = H x n g^x (1 - g^x);
//   abar = H h_{t-1} + H x g^x (-2 a) / sqrt(max(4 (1 - a^2), 1e-6));
//   dl^a = abar (-8 softplus(alpha)) a g^a (1 - g^a);
//   dalpha += abar (-8 g^a) sigmoid(alpha) a.
// ---------------------------------------------------------------------------
// The leading BF16 pair of (v0, v1) and the BF16 pair of the remainders.
__device__ __forceinline__ void split_bf2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    hi = f2_to_bf2(v0, v1);
    const float2 h = bf2_to_f2(hi);
    lo = f2_to_bf2(v0 - h.x, v1 - h.y);
}

// Logits mode 2 (gate logits formed in the kernel): dynamic shared memory is
// [x box, 128-byte swizzle][weight images, then g^x per token][dy box][staging];
// the write gate's products are staged first and turned into g^x (kept in
// shared memory for the reverse sweep), then the keep gate's, which stay in the
// staging area for both sweeps.
constexpr int kBwdGxOff = kRgBoxBytes;                       // the weight images' slot, reused
constexpr int kBwdGxBytes = kRgTile * kGroup * 4;            // g^x [128][64] FP32
constexpr int kBwdDyOff = kBwdGxOff + kBwdGxBytes;
constexpr int kBwdStageOff = kBwdDyOff + kRgBoxBytes;
constexpr int kBwdFusedBytes = kBwdStageOff + kStageBytes;
static_assert(kWimgBytes <= kBwdGxBytes, "the weight images fit the g^x area");

template <int LM>
__global__ void __launch_bounds__(kRgThreads, 2)
    rglru_scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_lx, const __grid_constant__ CUtensorMap tm_la,
                          RglruScanBwdArgs a) {
    constexpr bool PL = LM >= 1;
    constexpr int LB = RgLogits<LM>::kBoxBytes;
    constexpr uint32_t kIdesc = umma_idesc_bf16(kRgTile, kGroup);
    // LM 0/1 boxes: dy, x, l^x, l^a; LM 2: see above (1024-byte aligned for the swizzle)
    extern __shared__ __align__(1024) uint8_t s_raw[];
    uint8_t* s_dyn = LM == 2 ? s_raw + ((1024u - (smem_u32(s_raw) & 1023u)) & 1023u) : s_raw;
    uint32_t (*s_g)[kGroup / 2] =
        reinterpret_cast<uint32_t (*)[kGroup / 2]>(LM == 2 ? s_dyn + kBwdDyOff : s_dyn);
    const uint8_t* s_x = LM == 2 ? s_dyn : s_dyn + kRgBoxBytes;
    uint8_t* s_stage = s_dyn + kBwdStageOff;
    float2* s_gx = reinterpret_cast<float2*>(s_dyn + kBwdGxOff);   // LM 2: [128][32] pairs
    const uint8_t* s_lx = LM == 2 ? s_stage : s_dyn + 2 * kRgBoxBytes;
    const uint8_t* s_la = LM == 2 ? s_stage : s_dyn + 2 * kRgBoxBytes + LB;
    __shared__ uint8_t s_rst[kRgTile];
    __shared__ float4 s_map[kRgWarps][32];
    __shared__ float2 s_ent[kRgWarps][32];
    __shared__ float2 s_acc[kRgWarps][32];
    __shared__ float4 s_bacc[PL ? kRgWarps : 1][32];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ __align__(8) uint64_t s_mma_bar;
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_tile;
    __shared__ int s_err;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (LM == 2 && warp == 0) {   // two gates x 64 FP32 columns of tensor memory
        tmem_alloc(&s_tmem, 2 * kGroup);
        tmem_fence_before_sync();
    }
    if (tid == 0) {
        s_tile = atomicAdd(a.counter, 1u);
        mbar_init(&s_bar, 1);
        if (LM == 2) mbar_init(&s_mma_bar, 1);
    }
    __syncthreads();
    if (LM == 2) tmem_fence_after_sync();
    const uint32_t tmem = LM == 2 ? s_tmem : 0u;
    const ScanGeom& g = a.g;
    const long long tile = s_tile;
    const int chain = (int)(tile % g.n_chains);
    const int CT = g.CT;
    const int c = CT - 1 - (int)(tile / g.n_chains);
    const int b = chain / g.n_groups;
    const int grp = chain % g.n_groups;
    const int D = g.lanes;
    const int L = g.L;
    const int t0 = c * kRgTile;
    const int d = grp * kGroup + 2 * lane;
    const bool active = d < D;
    uint32_t* fl = a.flags + (size_t)chain * CT;
    const size_t hb = (size_t)b * g.CS;

    if (tid == 0) {
        if (LM == 2) {
            mbar_arrive_expect_tx(&s_bar, 2 * kRgBoxBytes + kWimgBytes);
            tma_load_3d(s_dyn, &tm_x, grp * kGroup, t0, b, &s_bar);
            bulk_load(s_dyn + kBwdGxOff, a.wimg + (size_t)grp * kWimgBytes, kWimgBytes, &s_bar);
            tma_load_3d(&s_g[0][0], &tm_dy, grp * kGroup, t0, b, &s_bar);
        } else {
            mbar_arrive_expect_tx(&s_bar, 2 * kRgBoxBytes + 2 * LB);
            tma_load_3d(&s_g[0][0], &tm_dy, grp * kGroup, t0, b, &s_bar);
            tma_load_3d(s_dyn + kRgBoxBytes, &tm_x, grp * kGroup, t0, b, &s_bar);
            tma_load_3d(s_dyn + 2 * kRgBoxBytes, &tm_lx, grp * kGroup, t0, b, &s_bar);
            tma_load_3d(s_dyn + 2 * kRgBoxBytes + LB, &tm_la, grp * kGroup, t0, b, &s_bar);
        }
    }
    if (tid < kRgTile) {
        const int t = t0 + tid;
        s_rst[tid] = (t < L && a.reset != nullptr && a.reset[(size_t)b * L + t] != 0) ? 1 : 0;
    }
    const int r0 = warp * kSub;
    const int nsub = max(0, min(kSub, L - t0 - r0));
    float nsp0 = 0.f, nsp1 = 0.f, sa0 = 0.f, sa1 = 0.f;
    float h0v = 0.f, h1v = 0.f;
    float2 bxv = make_float2(0.f, 0.f), bav = bxv;
    if (active) {
        if (PL) {
            bxv = *reinterpret_cast<const float2*>(a.bx + d);
            bav = *reinterpret_cast<const float2*>(a.ba + d);
        }
        const float al0 = a.alpha[d], al1 = a.alpha[d + 1];
        nsp0 = -8.0f * softplus_f(al0);
        nsp1 = -8.0f * softplus_f(al1);
        sa0 = 1.0f / (1.0f + expf(-al0));
        sa1 = 1.0f / (1.0f + expf(-al1));
        if (nsub > 0) {
            const float2 hv = __ldcg(reinterpret_cast<const float2*>(
                a.hsub + (hb + (size_t)c * kRgWarps + warp) * D + d));
            h0v = hv.x;
            h1v = hv.y;
        }
    }
    bool ok = mbar_wait_bounded(&s_bar, 0);
    if (!__syncthreads_and(ok)) {
        if (tid == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
            mbar_wait_bounded(&s_bar, 0);
        }
        if (LM == 2) {
            __syncthreads();
            if (warp == 0) tmem_dealloc(tmem, 2 * kGroup);
        }
        return;
    }
    if (LM == 2) {
        // logits of the tile: D_gate[128 x 64] = x[128 x 64] . Wimg_gate[64 x 64]^T
        if (tid == 0) {
            tmem_fence_after_sync();
            const uint32_t xa = smem_u32(s_dyn), wa = smem_u32(s_dyn + kBwdGxOff);
#pragma unroll
            for (int gt = 0; gt < 2; ++gt)
#pragma unroll
                for (int ks = 0; ks < kGroup / 16; ++ks)
                    umma_bf16(tmem + (uint32_t)(gt * kGroup), umma_desc_sw128(xa + 32u * ks),
                              umma_desc_sw128(wa + (uint32_t)(gt * kGroup * kGroup * 2) + 32u * ks), kIdesc, ks > 0);
            umma_commit(&s_mma_bar);
        }
        ok = mbar_wait_bounded(&s_mma_bar, 0);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                st_release_gpu(fl + c, kFlagErr);
                atomicOr(a.status, kStatusTimeout);
                mbar_wait_bounded(&s_mma_bar, 0);
            }
            __syncthreads();
            if (warp == 0) {
                tmem_fence_after_sync();
                tmem_dealloc(tmem, 2 * kGroup);
            }
            return;
        }
        tmem_fence_after_sync();
    }

    // the lane's two channels as pairs (the same IEEE operations per element)
    const f2x nsp = pk2(nsp0, nsp1);
    f2x hp[kSub];   // h_{t-1} per token
    f2x hv = pk2(h0v, h1v), P = dup2(1.0f), q = 0ull;
    if (LM == 2) {
        // write gate: g^x kept for the reverse sweep, x g^x in hp[] until the keep gate is staged
        rg_stage_gate(tmem, s_stage, 0, warp, lane);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            hp[i] = 0ull;
            if (i < nsub) {
                const float2 xx = rg_x<LM>(s_x, r0 + i, lane);
                const float2 gl = rg_logit<LM>(s_lx, r0 + i, lane, bxv);
                const f2x gx = sigmoid2(pk2(gl.x, gl.y));
                float g0, g1;
                up2(gx, g0, g1);
                s_gx[(r0 + i) * 32 + lane] = make_float2(g0, g1);
                hp[i] = mul2(pk2(xx.x, xx.y), gx);
            }
        }
        __syncthreads();   // every warp has read the write gate before the keep gate replaces it
        rg_stage_gate(tmem, s_stage, 1, warp, lane);
        tmem_fence_before_sync();
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            if (i < nsub) {
                const float2 al = rg_logit<LM>(s_la, r0 + i, lane, bav);
                const float2 gg = bf2_to_f2(s_g[r0 + i][lane]);
                const RgGate2 kg = rg_keep_gate2(pk2(al.x, al.y), nsp, s_rst[r0 + i] != 0);
                const f2x bt = mul2(hp[i], kg.n);
                hp[i] = hv;
                hv = fma2(kg.a, hv, bt);
                P = mul2(P, kg.a);
                q = fma2(P, pk2(gg.x, gg.y), q);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
            hp[i] = 0ull;
            if (i < nsub) {
                const bool rs = s_rst[r0 + i] != 0;
                const float2 xx = rg_x<LM>(s_x, r0 + i, lane);
                const float2 gl = rg_logit<LM>(s_lx, r0 + i, lane, bxv);
                const float2 al = rg_logit<LM>(s_la, r0 + i, lane, bav);
                const float2 gg = bf2_to_f2(s_g[r0 + i][lane]);
                const RgGate2 gt = rg_gate2(pk2(gl.x, gl.y), pk2(al.x, al.y), nsp, rs);
                hp[i] = hv;
                hv = fma2(gt.a, hv, mul2(mul2(pk2(xx.x, xx.y), gt.gx), gt.n));
                P = mul2(P, gt.a);
                q = fma2(P, pk2(gg.x, gg.y), q);
            }
        }
    }
    {
        float P0, P1, q0, q1;
        up2(P, P0, P1);
        up2(q, q0, q1);
        s_map[warp][lane] = make_float4(P0, q0, P1, q1);
    }
    // the next tile's flag, read while the other warps finish their maps
    const uint32_t pflag = (warp == 0 && lane == 0 && c < CT - 1) ? ld_acquire_gpu(fl + c + 1) : 0u;
    __syncthreads();
    if (LM == 2 && warp == 0) {   // the tile's tensor memory is no longer read
        tmem_fence_after_sync();
        tmem_dealloc(tmem, 2 * kGroup);
    }

    if (warp == 0) {
        float4 A = s_map[kRgWarps - 1][lane];
#pragma unroll
        for (int w = kRgWarps - 2; w >= 0; --w) {
            const float4 Fw = s_map[w][lane];
            const float2 t0v = rcompose(make_float2(Fw.x, Fw.y), make_float2(A.x, A.y));
            const float2 t1v = rcompose(make_float2(Fw.z, Fw.w), make_float2(A.z, A.w));
            A = make_float4(t0v.x, t0v.y, t1v.x, t1v.y);
        }
        float R0 = 0.f, R1 = 0.f;
        bool err = false;
        if (c == CT - 1) {
            if (active && a.dhT != nullptr) {
                const float2 v = *reinterpret_cast<const float2*>(a.dhT + (size_t)b * D + d);
                R0 = v.x;
                R1 = v.y;
            }
        } else {
            // the neighbouring tile already inclusive: its state
            // is the entry and this tile's map need not be published
            int j = __shfl_sync(0xffffffffu, pflag, 0) == kFlagIncl ? c + 1 : -2;
            if (j == -2) {
                if (active)
                    *reinterpret_cast<float4*>(a.agg + ((size_t)b * CT + c) * D + d) = A;
                __syncwarp();
                if (lane == 0) st_release_gpu(fl + c, kFlagAgg);
                j = lookback_find_warp(fl, c, CT, +1);
            }
            if (j < 0) {
                err = true;
            } else if (active) {
                const float2 rv = __ldcg(reinterpret_cast<const float2*>(a.rin + ((size_t)b * CT + j) * D + d));
                R0 = rv.x;
                R1 = rv.y;
                for (int i = j - 1; i > c; i -= 4) {
                    float4 T[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (i - q > c)
                            T[q] = ldcg4(reinterpret_cast<const float4*>(a.agg + ((size_t)b * CT + i - q) * D + d));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (i - q > c) {
                            R0 = rapply(make_float2(T[q].x, T[q].y), R0);
                            R1 = rapply(make_float2(T[q].z, T[q].w), R1);
                        }
                    }
                }
            }
        }
        if (!err) {
            float v0 = R0, v1 = R1;
#pragma unroll
            for (int w = kRgWarps - 1; w >= 0; --w) {
                s_ent[w][lane] = make_float2(v0, v1);
                const float4 Fw = s_map[w][lane];
                v0 = rapply(make_float2(Fw.x, Fw.y), v0);
                v1 = rapply(make_float2(Fw.z, Fw.w), v1);
            }
            if (active)
                *reinterpret_cast<float2*>(a.rin + ((size_t)b * CT + c) * D + d) =
                    make_float2(rapply(make_float2(A.x, A.y), R0), rapply(make_float2(A.z, A.w), R1));
        } else if (lane == 0) {
            st_release_gpu(fl + c, kFlagErr);
            atomicOr(a.status, kStatusTimeout);
        }
        if (lane == 0) s_err = err ? 1 : 0;
    }
    __syncthreads();
    if (s_err) return;
    if (warp == 0) {   // the state after the tile, published while the other warps replay
        __syncwarp();
        if (lane == 0) st_release_gpu(fl + c, kFlagIncl);
    }

    const float2 e = s_ent[warp][lane];
    f2x H = pk2(e.x, e.y), da = 0ull;
    const f2x m8sa = mul2(dup2(-8.0f), pk2(sa0, sa1));   // -8 sigmoid(alpha)
    f2x bsx = 0ull, bsa = 0ull;   // PL: sums of dl^x, dl^a over the lane's tokens
    const size_t row = (((size_t)b * L + t0 + r0) * D + d) / 2;
#pragma unroll
    for (int i = kSub - 1; i >= 0; --i) {
        if (i < nsub) {
            const bool rs = s_rst[r0 + i] != 0;
            const float2 xf = rg_x<LM>(s_x, r0 + i, lane);
            const float2 al = rg_logit<LM>(s_la, r0 + i, lane, bav);
            const float2 gg = bf2_to_f2(s_g[r0 + i][lane]);
            RgGate2 gt;
            if (LM == 2) {
                gt = rg_keep_gate2(pk2(al.x, al.y), nsp, rs);
                const float2 gx = s_gx[(r0 + i) * 32 + lane];
                gt.gx = pk2(gx.x, gx.y);
            } else {
                const float2 gl = rg_logit<LM>(s_lx, r0 + i, lane, bxv);
                gt = rg_gate2(pk2(gl.x, gl.y), pk2(al.x, al.y), nsp, rs);
            }
            const f2x xx = pk2(xf.x, xf.y);
            H = add2(H, pk2(gg.x, gg.y));
            const f2x Hxg = mul2(mul2(H, xx), gt.gx);
            const f2x dx2 = mul2(mul2(H, gt.gx), gt.n);
            const f2x dlx2 = mul2(mul2(Hxg, gt.n), sub2(dup2(1.0f), gt.gx));
            f2x dla2 = 0ull;
            if (!rs) {
                float u0, u1;
                up2(mul2(dup2(4.0f), gt.u), u0, u1);
                const f2x rq = pk2(rsqrt_approx(fmaxf(u0, 1e-6f)), rsqrt_approx(fmaxf(u1, 1e-6f)));
                const f2x ab = fma2(H, hp[i], mul2(mul2(Hxg, mul2(dup2(-2.0f), gt.a)), rq));
                const f2x aga = mul2(gt.a, gt.ga);
                dla2 = mul2(mul2(ab, mul2(nsp, aga)), sub2(dup2(1.0f), gt.ga));
                da = fma2(ab, mul2(aga, m8sa), da);
            }
            if (PL) {
                bsx = add2(bsx, dlx2);
                bsa = add2(bsa, dla2);
            }
            float dx0, dx1, dlx0, dlx1, dla0, dla1;
            up2(dx2, dx0, dx1);
            up2(dlx2, dlx0, dlx1);
            up2(dla2, dla0, dla1);
            if (PL && active) {
                // token t, channels d, d+1 of block h at offset ob: parts p at gp + p * dk / 2
                uint32_t* gp = a.gparts + ((((size_t)b * L + t0 + r0 + i) * D) * 6 + (size_t)(d / a.dk) * 6 * a.dk +
                                           d % a.dk) / 2;
                const int ps = a.dk / 2;
                uint32_t hi, lo;
                split_bf2(dlx0, dlx1, hi, lo);
                __stcs(gp, hi);
                __stcs(gp + ps, lo);
                split_bf2(dla0, dla1, hi, lo);
                __stcs(gp + 2 * ps, hi);
                __stcs(gp + 3 * ps, lo);
                split_bf2(dx0, dx1, hi, lo);
                __stcs(gp + 4 * ps, hi);
                __stcs(gp + 5 * ps, lo);
            } else if (active) {
                const size_t o = row + (size_t)i * (D / 2);
                if (a.grad_fp32) {
                    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.dx) + 2 * o) = make_float2(dx0, dx1);
                    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.dlx) + 2 * o) = make_float2(dlx0, dlx1);
                    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.dla) + 2 * o) = make_float2(dla0, dla1);
                } else {
                    __stcs(reinterpret_cast<uint32_t*>(a.dx) + o, f2_to_bf2(dx0, dx1));
                    __stcs(reinterpret_cast<uint32_t*>(a.dlx) + o, f2_to_bf2(dlx0, dlx1));
                    __stcs(reinterpret_cast<uint32_t*>(a.dla) + o, f2_to_bf2(dla0, dla1));
                }
            }
            H = mul2(H, gt.a);
        }
    }
    float H0, H1, da0, da1;
    up2(H, H0, H1);
    up2(da, da0, da1);
    if (c == 0 && warp == 0 && active) *reinterpret_cast<float2*>(a.dh0 + (size_t)b * D + d) = make_float2(H0, H1);
    s_acc[warp][lane] = make_float2(da0, da1);
    if (PL) {
        float x0, x1, y0, y1;
        up2(bsx, x0, x1);
        up2(bsa, y0, y1);
        s_bacc[warp][lane] = make_float4(x0, x1, y0, y1);
    }
    __syncthreads();
    if (warp == 0 && active) {
        float2 s = s_acc[0][lane];
#pragma unroll
        for (int w = 1; w < kRgWarps; ++w) {
            s.x += s_acc[w][lane].x;
            s.y += s_acc[w][lane].y;
        }
        *reinterpret_cast<float2*>(a.apart + ((size_t)b * CT + c) * D + d) = s;
    }
    if (PL && warp == 1 && active) {   // the tile's bias-gradient partials, warps in order
        float4 s = s_bacc[0][lane];
#pragma unroll
        for (int w = 1; w < kRgWarps; ++w) {
            const float4 v = s_bacc[w][lane];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        const size_t o = ((size_t)b * CT + c) * D + d;
        *reinterpret_cast<float2*>(a.bxpart + o) = make_float2(s.x, s.y);
        *reinterpret_cast<float2*>(a.bapart + o) = make_float2(s.z, s.w);
    }
}

// dalpha: two fixed-order stages over the per-tile partials [rows][D]
__global__ void __launch_bounds__(256) rglru_alpha_stage1_kernel(const float* __restrict__ apart,
                                                                 float* __restrict__ apart2, int rows, int D) {
    const int d = blockIdx.x * blockDim.x + threadIdx.x;
    const int gidx = blockIdx.y;
    if (d >= D) return;
    const int per = (rows + kReduceGroups - 1) / kReduceGroups;
    const int r0 = gidx * per;
    const int r1 = min(rows, r0 + per);
    float s = 0.f;
    int r = r0;
    for (; r + 8 <= r1; r += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcs(apart + (size_t)(r + k) * D + d);
#pragma unroll
        for (int k = 0; k < 8; ++k) s += v[k];
    }
    for (; r < r1; ++r) s += __ldcs(apart + (size_t)r * D + d);
    apart2[(size_t)gidx * D + d] = s;
}

__global__ void __launch_bounds__(256) rglru_alpha_stage2_kernel(const float* __restrict__ apart2,
                                                                 float* __restrict__ dalpha, int D) {
    const int d = blockIdx.x * blockDim.x + threadIdx.x;
    if (d >= D) return;
    float s = 0.f;
    for (int gi = 0; gi < kReduceGroups; ++gi) s += apart2[(size_t)gi * D + d];
    dalpha[d] = s;
}

// Weight images for the in-kernel logits: group g, gate q, output n, input k
// (channels 64 g + n, 64 g + k) hold W_q[h][i][o] when both channels lie in
// diagonal block h (i, o their offsets in it), else 0; stored K-major with the
// 128-byte swizzle (row n: 128 bytes, chunk k / 8 at k / 8 ^ n % 8).
__global__ void __launch_bounds__(256) rglru_proj_wimg_kernel(const uint16_t* __restrict__ w_x,
                                                              const uint16_t* __restrict__ w_a,
                                                              uint16_t* __restrict__ img, int D) {
    const int dk = D / kProjBlocks;
    const size_t n_el = (size_t)(D / kGroup) * 2 * kGroup * kGroup;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_el; e += (size_t)gridDim.x * blockDim.x) {
        const int k = (int)(e % kGroup);
        const int n = (int)(e / kGroup % kGroup);
        const int q = (int)(e / (kGroup * kGroup) % 2);
        const size_t grp = e / (2 * kGroup * kGroup);
        const int co = (int)grp * kGroup + n, ci = (int)grp * kGroup + k;
        const int h = co / dk;
        uint16_t v = 0;
        if (ci / dk == h) {
            const uint16_t* w = q == 0 ? w_x : w_a;
            v = w[((size_t)h * dk + (ci - h * dk)) * dk + (co - h * dk)];
        }
        img[(grp * 2 + q) * kGroup * kGroup + (size_t)n * kGroup + ((((k >> 3) ^ (n & 7))) << 3) + (k & 7)] = v;
    }
}

cudaError_t launch_rglru_proj_wimg(const void* w_x, const void* w_a, void* wimg, int D, cudaStream_t s) {
    const size_t n = (size_t)(D / kGroup) * 2 * kGroup * kGroup;
    rglru_proj_wimg_kernel<<<(unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, s>>>(
        static_cast<const uint16_t*>(w_x), static_cast<const uint16_t*>(w_a), static_cast<uint16_t*>(wimg), D);
    return cudaGetLastError();
}

// Persistent grid: as many CTAs as are resident at once, at most one per tile.
// Residency is counted from the kernel's registers and shared memory against
// the SM's (the occupancy query answers one CTA per SM for a kernel that
// allocates tensor memory whatever its size, while two of the forward's fit).
// Tickets go out in the order CTAs start, so a CTA only ever waits on tiles
// held by CTAs already running: a grid larger than what is resident is slower,
// never stuck.
// (The count is asked once per device and logits mode.)
template <int LM, typename K>
unsigned rg_grid(K kernel, int smem, long long n_tiles) {
    static std::atomic<long long> resident_cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    const long long cached = resident_cache[dev].load(std::memory_order_relaxed);
    if (cached > 0) return (unsigned)(cached < n_tiles ? cached : (n_tiles > 0 ? n_tiles : 1));
    int sms = 1, per = 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kRgThreads, smem) != cudaSuccess || per < 1)
        per = 1;
    cudaFuncAttributes fa{};
    int smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0;
    if (cudaFuncGetAttributes(&fa, kernel) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) == cudaSuccess) {
        const long long cta_smem = (long long)fa.sharedSizeBytes + smem + reserved;
        const long long warp_regs = ((long long)fa.numRegs * 32 + 255) / 256 * 256;   // 256-register units
        const long long cta_regs = warp_regs * (kRgThreads / 32);
        long long fit = threads_sm / kRgThreads;
        if (cta_smem > 0) fit = std::min(fit, (long long)smem_sm / cta_smem);
        if (cta_regs > 0) fit = std::min(fit, (long long)regs_sm / cta_regs);
        if (fit > per) per = (int)fit;
    }
    const long long n = (long long)sms * per;
    resident_cache[dev].store(n, std::memory_order_relaxed);
    return (unsigned)(n < n_tiles ? n : (n_tiles > 0 ? n_tiles : 1));
}

template <int LM>
cudaError_t launch_fwd(const CUtensorMap& tm_x, const CUtensorMap& tm_lx, const CUtensorMap& tm_la,
                       const RglruScanFwdArgs& args, cudaStream_t s) {
    // two slots, the staging area (LM 2) and a spare kilobyte for 1024-byte alignment
    const int smem = 2 * RgLogits<LM>::kSlotBytes + (LM == 2 ? kStageBytes : 0) + 1024;
    cudaError_t e = cudaFuncSetAttribute(rglru_scan_fwd_kernel<LM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    rglru_scan_fwd_kernel<LM><<<rg_grid<LM>(rglru_scan_fwd_kernel<LM>, smem, args.g.n_tiles), kRgThreads, smem, s>>>(
        tm_x, tm_lx, tm_la, args);
    return cudaGetLastError();
}

cudaError_t launch_rglru_scan_fwd(const CUtensorMap& tm_x, const CUtensorMap& tm_lx, const CUtensorMap& tm_la,
                                  const RglruScanFwdArgs& args, cudaStream_t s, int logits) {
    if (logits == 2) return launch_fwd<2>(tm_x, tm_lx, tm_la, args, s);
    if (logits == 1) return launch_fwd<1>(tm_x, tm_lx, tm_la, args, s);
    return launch_fwd<0>(tm_x, tm_lx, tm_la, args, s);
}

template <int LM>
cudaError_t launch_bwd(const CUtensorMap& tm_dy, const CUtensorMap& tm_x, const CUtensorMap& tm_lx,
                       const CUtensorMap& tm_la, const RglruScanBwdArgs& args, cudaStream_t s) {
    // LM 2: a spare kilobyte for the 1024-byte alignment of the swizzled boxes
    const int smem = LM == 2 ? kBwdFusedBytes + 1024 : 2 * kRgBoxBytes + 2 * RgLogits<LM>::kBoxBytes;
    cudaError_t e = cudaFuncSetAttribute(rglru_scan_bwd_kernel<LM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    rglru_scan_bwd_kernel<LM><<<(unsigned)args.g.n_tiles, kRgThreads, smem, s>>>(tm_dy, tm_x, tm_lx, tm_la, args);
    return cudaGetLastError();
}

cudaError_t launch_rglru_scan_bwd(const CUtensorMap& tm_dy, const CUtensorMap& tm_x, const CUtensorMap& tm_lx,
                                  const CUtensorMap& tm_la, const RglruScanBwdArgs& args, cudaStream_t s,
                                  int logits) {
    if (logits == 2) return launch_bwd<2>(tm_dy, tm_x, tm_lx, tm_la, args, s);
    if (logits == 1) return launch_bwd<1>(tm_dy, tm_x, tm_lx, tm_la, args, s);
    return launch_bwd<0>(tm_dy, tm_x, tm_lx, tm_la, args, s);
}

cudaError_t launch_rglru_alpha(const float* apart, float* apart2, float* dalpha, int rows, int D,
                               cudaStream_t s) {
    dim3 g1((D + 255) / 256, kReduceGroups);
    rglru_alpha_stage1_kernel<<<g1, 256, 0, s>>>(apart, apart2, rows, D);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    rglru_alpha_stage2_kernel<<<(D + 255) / 256, 256, 0, s>>>(apart2, dalpha, D);
    return cudaGetLastError();
}

}  // namespace lrs

// SAMU mixer chunked complex affine scan on sm_103a: forward and reverse.
//
// Equations: SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比"), section 05:
// z_{t,m} = lambda_{t,m} z_{t-1,m} + b_{t,m} with lambda rebuilt in registers
// from the shared per-token E, C, S and the static spectrum (no [B,L,M]
// transition tensor); chunk summaries under (l2,b2) o (l1,b1) =
// (l2 l1, l2 b1 + b2); a chunk prefix gives every chunk its entry state; the
// replay from the entry state emits the visible output.  The backward runs
// the conjugate transition in reverse time,
// zbar_{t-1} = conj(lambda_t) zbar_t + dy_{t-1}, with the same three steps,
// and rebuilds lambda and z instead of storing them.
//
// GB300 organisation.  A chain is one (batch row, group of 64 modes); lane l
// of a warp owns modes 2l, 2l+1.  Each chain is cut into NS segments (a
// multiple of 16 tokens each), one per warp, NS chosen on the host so that
// the segments of all chains run at once on the resident warps: one wave,
// equal work per warp.  A warp walks its segment 16 tokens at a time through
// a private ring of two shared-memory slots that TMA fills one sub-chunk
// ahead (a [16 x 64] BF16 box per half plus the 16 control words).
//
// Each direction is two launches with no waits between CTAs:
//  1. maps:    every warp composes its segment's affine map, walking the
//              segment in the opposite time direction to step 2, and a CTA
//              (8 consecutive segments of one chain) composes its CTA map;
//              a full 16-token item without a reset gets its transition in
//              closed form from two per-item statistics (by default; see
//              item_transition) and its affine part by Horner's rule;
//  2. replay:  every CTA first folds the chain's earlier (later) CTA maps into
//              its entry state (adjoint), every warp applies the earlier
//              (later) segment maps of its CTA and replays its segment.
// Step 2 starts each segment where step 1 finished it, so its first reads of
// w (forward) or dy (backward) hit in L2.  Every composition runs in a fixed
// order: results are bitwise reproducible from run to run.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kernels.cuh"

namespace lrs {

constexpr int kEngineWarps = 8;                     // warps per CTA (each on its own segment)
constexpr int kEngineThreads = kEngineWarps * 32;
constexpr int kWords = kGroup / 2;                  // BF16 pairs per box row
constexpr int kCtlBytes = 32;                       // one token's control word (two float4)
static_assert(kEngineWarps == kSegPerCta, "a CTA holds the segments of one chain");

// One warp's staging ring of S items of R tokens: a [R x 64] BF16 box per
// half of the warp's 64 modes plus the R control words.  Every TMA
// destination starts on a 128-byte boundary (box sizes are multiples of 128
// bytes).
template <int R, int S>
struct alignas(128) WarpRingT {
    static constexpr int kRows = R;
    static constexpr int kSlots = S;
    static constexpr int kItemBytes = 2 * R * kRowBytes + R * kCtlBytes;
    uint32_t box[S][2][R][kWords];   // [slot][re, im][token][pair]
    float4 ctrl[S][2 * R];           // [slot][token: two float4]
    uint64_t full[S];
};
// The maps and replay kernels stage kMapRows-token items, kMapSlots per warp
// (the reverse replay's ring, one slot per 8-token unit, is defined with it).
using MapRing = WarpRingT<kMapRows, kMapSlots>;
constexpr int kWarpSmem = (int)sizeof(MapRing);
constexpr int kEngineSmem = kEngineWarps * kWarpSmem;

template <class Ring>
__device__ __forceinline__ Ring& warp_ring(uint8_t* smem_raw, int warp) {
    return *reinterpret_cast<Ring*>(smem_raw + (size_t)warp * kWarpSmem);
}

// The segment of one warp.
struct SegTask {
    int b, grp, s;
    int t_begin, t_end;   // tokens [t_begin, t_end)
    int nsc;              // kMapRows-token items
};

__device__ __forceinline__ SegTask seg_task(const SegGeom& g, long long gw) {
    SegTask T;
    const int chain = (int)(gw / g.NS);
    T.s = (int)(gw % g.NS);
    T.b = chain / g.n_groups;
    T.grp = chain % g.n_groups;
    T.t_begin = T.s * g.seg;
    T.t_end = min(g.L, T.t_begin + g.seg);
    T.nsc = T.t_end > T.t_begin ? (T.t_end - T.t_begin + kMapRows - 1) / kMapRows : 0;   // 0: a segment past L
    return T;
}

// Warp-uniform facts about N consecutive tokens that select the code path:
//  fast:   |nu| max|E - 1| < kPolyBound for every lane's modes (polynomial
//          lambda instead of ex2.approx);
//  simple: all N tokens present and none of them a reset (no per-token
//          checks).
struct SubKind {
    bool fast, simple;
};

template <int N>
__device__ __forceinline__ SubKind sub_kind(const float4* sc, int nsub, int lane, const ModePair& k) {
    const int i = lane & (N - 1);
    const float em1 = sc[2 * i].x;
    const float rst = sc[2 * i + 1].z;
    const bool mine = lane < nsub;
    const float e = mine ? fabsf(em1) : 0.f;
    const float emax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(e)));
    float n0, n1;
    up2(k.nu, n0, n1);
    const bool ok = fabsf(n0) * emax < kPolyBound && fabsf(n1) * emax < kPolyBound;
    SubKind kd;
    kd.fast = __all_sync(0xffffffffu, ok);
    kd.simple = nsub == N && !__any_sync(0xffffffffu, mine && is_reset_word(rst));
    return kd;
}

// Calls FN<FAST, SIMPLE>(args...) for the sub-chunk kind.
#define LRS_SUB_DISPATCH(kd, FN, ...)                  \
    do {                                               \
        if (kd.fast) {                                 \
            if (kd.simple)                             \
                FN<true, true>(__VA_ARGS__);           \
            else                                       \
                FN<true, false>(__VA_ARGS__);          \
        } else {                                       \
            if (kd.simple)                             \
                FN<false, true>(__VA_ARGS__);          \
            else                                       \
                FN<false, false>(__VA_ARGS__);         \
        }                                              \
    } while (0)

// The same for FN<N, FAST, SIMPLE> and FN<N, FAST, SIMPLE, X>.
#define LRS_SUB_DISPATCH_N(kd, FN, N, ...)             \
    do {                                               \
        if (kd.fast) {                                 \
            if (kd.simple)                             \
                FN<N, true, true>(__VA_ARGS__);        \
            else                                       \
                FN<N, true, false>(__VA_ARGS__);       \
        } else {                                       \
            if (kd.simple)                             \
                FN<N, false, true>(__VA_ARGS__);       \
            else                                       \
                FN<N, false, false>(__VA_ARGS__);      \
        }                                              \
    } while (0)
#define LRS_SUB_DISPATCH_NX(kd, FN, N, X, ...)         \
    do {                                               \
        if (kd.fast) {                                 \
            if (kd.simple)                             \
                FN<N, true, true, X>(__VA_ARGS__);     \
            else                                       \
                FN<N, true, false, X>(__VA_ARGS__);    \
        } else {                                       \
            if (kd.simple)                             \
                FN<N, false, true, X>(__VA_ARGS__);    \
            else                                       \
                FN<N, false, false, X>(__VA_ARGS__);   \
        }                                              \
    } while (0)

// Per-item plan of one warp's segment, 32 items at a time, from the
// controller forward's item records (one float4 per 16-token item of a batch
// row: G = sum (E - 1), cos D, sin D, and max |E - 1| with its sign marking
// an item that is not simple): lane j describes item 32 q + j of the segment
// (its tokens t_begin + 16 (32 q + j) ...):
//  simple (bit j): all 16 tokens present and none a reset;
//  fast (bit j):   numax max|E - 1| < kPolyBound, numax = max |nu| over the
//                  warp's modes (the same test as sub_kind);
//  G, c, s:        the closed-form transition's statistics.
// One coalesced 16-byte load per lane and 32 items replaces the per-item
// votes, sums and sincosf.
struct ItemPlan {
    unsigned fast, simple;
    float G, c, s;
    int q;   // batch held, -1 before the first
};

// max |nu| over the warp's modes
__device__ __forceinline__ float warp_numax(const ModePair& k) {
    float n0, n1;
    up2(k.nu, n0, n1);
    const float v = fmaxf(fabsf(n0), fabsf(n1));
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

__device__ __forceinline__ float record_emax(float v) { return v >= 0.f ? v : -v - 1.f; }

// Batch q of the plan of the segment T of a sequence of length L.  The
// records are read through L2 (the controller forward may have run beside
// this kernel before its dependency wait).
template <bool STATS>
__device__ __forceinline__ void plan_batch(ItemPlan& P, const float4* __restrict__ items, const SegTask& T, int L,
                                           int q, const ModePair& k, int lane) {
    const float numax = warp_numax(k);
    const int idx = 32 * q + lane;
    const bool ok = idx < T.nsc;
    float4 r = make_float4(0.f, 1.f, 0.f, 0.f);
    if (ok) r = __ldcg(items + (size_t)T.b * samu_items_per_row(L) + T.t_begin / kMapRows + idx);
    P.fast = __ballot_sync(0xffffffffu, numax * record_emax(r.w) < kPolyBound);
    P.simple = __ballot_sync(0xffffffffu, ok && r.w >= 0.f);
    if (STATS) {
        P.G = r.x;
        P.c = r.y;
        P.s = r.z;
    }
    P.q = q;
}

__device__ __forceinline__ float4 identity_map() { return make_float4(1.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ c2x czero() {
    c2x z;
    z.re = 0ull;
    z.im = 0ull;
    return z;
}

// A lane's two modes of an [.., M, 2] FP32 array (re, im per mode) as pairs.
__device__ __forceinline__ c2x load_c2(const float* p) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    c2x z;
    z.re = pk2(v.x, v.z);
    z.im = pk2(v.y, v.w);
    return z;
}
__device__ __forceinline__ void store_c2(float* p, const c2x& z) {
    float r0, r1, i0, i1;
    up2(z.re, r0, r1);
    up2(z.im, i0, i1);
    *reinterpret_cast<float4*>(p) = make_float4(r0, i0, r1, i1);
}
// An affine map of each of the two modes, as stored per mode {l.re, l.im, b.re, b.im}.
__device__ __forceinline__ void store_map2(float4* p, const c2x& l, const c2x& bb) {
    float lr0, lr1, li0, li1, br0, br1, bi0, bi1;
    up2(l.re, lr0, lr1);
    up2(l.im, li0, li1);
    up2(bb.re, br0, br1);
    up2(bb.im, bi0, bi1);
    p[0] = make_float4(lr0, li0, br0, bi0);
    p[1] = make_float4(lr1, li1, br1, bi1);
}

// Lane 0: stage the item at token ts of tensor `tm` (both halves of the
// warp's 64 modes) and its control words into ring slot `slot`.  The warp has
// finished reading the slot (__syncwarp before the call).
// The item's two boxes (the slot's expected bytes include the control words,
// so the slot completes only once ring_issue_ctrl has been issued too).
template <class Ring>
__device__ __forceinline__ void ring_issue_data(Ring& R, int slot, const CUtensorMap* tm, int x_re, int x_im, int ts,
                                                int b) {
    fence_proxy_async();
    mbar_arrive_expect_tx(&R.full[slot], Ring::kItemBytes);
    tma_load_3d(&R.box[slot][0][0][0], tm, x_re, ts, b, &R.full[slot]);
    tma_load_3d(&R.box[slot][1][0][0], tm, x_im, ts, b, &R.full[slot]);
}
template <class Ring>
__device__ __forceinline__ void ring_issue_ctrl(Ring& R, int slot, const CUtensorMap* tm_ctrl, int ts, int b) {
    tma_load_3d(&R.ctrl[slot][0], tm_ctrl, 0, ts, b, &R.full[slot]);
}
template <class Ring>
__device__ __forceinline__ void ring_issue(Ring& R, int slot, const CUtensorMap* tm, const CUtensorMap* tm_ctrl,
                                           int x_re, int x_im, int ts, int b) {
    ring_issue_data(R, slot, tm, x_re, x_im, ts, b);
    ring_issue_ctrl(R, slot, tm_ctrl, ts, b);
}

template <class Ring>
__device__ __forceinline__ void ring_init(Ring& R, int lane) {
    if (lane == 0) {
        for (int i = 0; i < Ring::kSlots; ++i) mbar_init(&R.full[i], 1);
    }
    __syncwarp();
}

// Waits for item k of the ring (n_items in all).  If the copy never lands:
// records the failure, waits (bounded) for the later items already issued,
// and returns false so that the warp can leave.
template <class Ring>
__device__ __forceinline__ bool ring_wait(Ring& R, int k, int n_items, uint32_t* status, int lane) {
    constexpr int S = Ring::kSlots;
    if (mbar_wait_bounded(&R.full[k % S], (uint32_t)(k / S) & 1u)) return true;
    if (lane == 0) atomicOr(status, kStatusTimeout);
    for (int j = k + 1; j < k + S && j < n_items; ++j) mbar_wait_bounded(&R.full[j % S], (uint32_t)(j / S) & 1u);
    return false;
}

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
// Appends the sub-chunk's tokens, latest first, to the map H = (P, beta) of
// the tokens after them: H o T_t = (P lambda_t, P b_t + beta).
template <int N, bool FAST, bool SIMPLE>
__device__ __forceinline__ void fwd_maps_sub(const float4* sc, const uint32_t* wre, const uint32_t* wim, int nsub,
                                             const ModePair& k, c2x& P, c2x& be) {
#pragma unroll
    for (int i = N - 1; i >= 0; --i) {
        if (SIMPLE || i < nsub) {
            const Ctl2 ct = load_ctl(sc, i);
            const uint32_t wr = wre[i * kWords], wi = wim[i * kWords];
            c2x bb;
            bb.re = bf2x(wr);
            bb.im = bf2x(wi);
            be = cfma2(P, bb, nbf2x(wi), be);
            if (SIMPLE || !is_reset(ct))
                P = cmul2(samu_lambda2<FAST>(k, ct), P);
            else   // segment start: nothing before it reaches past it
                P = czero();
        }
    }
}

// ---------------------------------------------------------------------------
// Closed-form item transitions (SAMU GPU page, section 05, "exact chunk closed
// form"): over tokens without a reset the product of the transitions is
//   prod_t lambda_{t,m} = lbar_m^K e^{-nu_m G} e^{i D},
//   G = sum_t (E_t - 1),  D = sum_t d_t,
// two statistics per item shared by all modes.  lbar_m^K is the FP64-formed
// double-float of mode_power_constants (the phase K theta_m is never rounded
// to FP32), so the product is one rounding away from exact instead of K.
// An item's map is then its affine part by Horner's rule (four paired FMAs
// per token, against eight for the running product and the affine part)
// and this product, composed with the maps of the other items as before.
// ---------------------------------------------------------------------------
__device__ __forceinline__ c2x cmulx(const c2x& a, const c2x& b) {   // a b
    c2x r;
    r.re = fma2(a.re, b.re, mul2(sub2(0ull, a.im), b.im));
    r.im = fma2(a.re, b.im, mul2(a.im, b.re));
    return r;
}

// The transition of one full item of N tokens, none a reset, for the lane's
// two modes (zero for an inactive lane), from the item's G and cos D, sin D
// (ItemPlan).
template <int N>
__device__ __forceinline__ c2x item_transition(float G, float cs, float sn, const float4* __restrict__ modes_n,
                                               const ModePair& k, int m, bool active) {
    static_assert(N == kMapRows, "the plan's statistics cover kMapRows tokens");
    float n0, n1;
    up2(k.nu, n0, n1);
    const float x0 = n0 * G, x1 = n1 * G;   // nu G
    f2x q;                                   // e^{-nu G}
    if (fabsf(x0) < kPolyBound && fabsf(x1) < kPolyBound) {
        const f2x x = pk2(x0, x1);
        q = fma2(x, fma2(x, fma2(x, dup2(-1.0f / 6.0f), dup2(0.5f)), dup2(-1.0f)), dup2(1.0f));
    } else {
        q = pk2(ex2_approx(__fmul_rn(-x0, kLog2e)), ex2_approx(__fmul_rn(-x1, kLog2e)));
    }
    const f2x dr = mul2(q, dup2(cs)), di = mul2(q, dup2(sn));
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (active) {
        v0 = modes_n[m];
        v1 = modes_n[m + 1];
    }
    const f2x hr = pk2(v0.x, v1.x), hi = pk2(v0.y, v1.y), lr = pk2(v0.z, v1.z), li = pk2(v0.w, v1.w);
    // (hi + lo)(dr + i di), the lo products added first
    c2x L;
    L.re = fma2(hr, dr, fma2(sub2(0ull, hi), di, fma2(lr, dr, mul2(sub2(0ull, li), di))));
    L.im = fma2(hr, di, fma2(hi, dr, fma2(lr, di, mul2(li, dr))));
    return L;
}

// A full item of the forward maps (N tokens, none a reset), appended to the
// map H = (P, beta) of the tokens after it: H o T_item = (P L, P h + beta),
// h = lambda_{N-1}(... (lambda_1 b_0 + b_1) ...) + b_{N-1}.
template <int N, bool FAST>
__device__ __forceinline__ void fwd_maps_item_cf(const float4* sc, const uint32_t* wre, const uint32_t* wim,
                                                 const ModePair& k, const float4* __restrict__ modes_n, int m,
                                                 bool active, float G, float cs, float sn, c2x& P, c2x& be) {
    c2x h;
    h.re = bf2x(wre[0]);
    h.im = bf2x(wim[0]);
#pragma unroll
    for (int i = 1; i < N; ++i) {
        const Ctl2 ct = load_ctl(sc, i);
        const f2x bre = bf2x(wre[i * kWords]);
        const f2x bim = bf2x(wim[i * kWords]);
        const Lam2 l = samu_lambda2<FAST>(k, ct);
        const f2x hr = fma2(l.re, h.re, fma2(l.nim, h.im, bre));
        const f2x hi = fma2(l.re, h.im, fma2(l.im, h.re, bim));
        h.re = hr;
        h.im = hi;
    }
    const c2x L = item_transition<N>(G, cs, sn, modes_n, k, m, active);
    const c2x Ph = cmulx(P, h);
    be.re = add2(be.re, Ph.re);
    be.im = add2(be.im, Ph.im);
    P = cmulx(P, L);
}

// hs: the item's first state checkpoint (the state entering its first
// token); the states entering its tokens 8, 16, ... go to the following
// checkpoints (the backward restarts there); written by active lanes only.
// The step z <- lambda z + b is one complex fused multiply-add (four paired
// FMAs).
template <int N, bool FAST, bool SIMPLE, bool Y32>
__device__ __forceinline__ void fwd_replay_sub(const float4* sc, const uint32_t* wre, const uint32_t* wim, int nsub,
                                               const ModePair& k, c2x& z, uint32_t* yp, float* y32p, bool active,
                                               size_t row, int half, f2x* hs, int M) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (i > 0 && i % kHalf == 0 && active && (SIMPLE || i < nsub)) {
            f2x* h = hs + (size_t)(i / kHalf) * M;
            h[0] = z.re;
            h[1] = z.im;
        }
        if (SIMPLE || i < nsub) {
            const Ctl2 ct = load_ctl(sc, i);
            const f2x bre = bf2x(wre[i * kWords]);
            const f2x bim = bf2x(wim[i * kWords]);
            if (SIMPLE || !is_reset(ct)) {
                const Lam2 l = samu_lambda2<FAST>(k, ct);
                const f2x zr = fma2(l.re, z.re, fma2(l.nim, z.im, bre));
                const f2x zi = fma2(l.re, z.im, fma2(l.im, z.re, bim));
                z.re = zr;
                z.im = zi;
            } else {
                z.re = bre;
                z.im = bim;
            }
            if (active) {
                uint32_t* o = yp + (size_t)i * row;
                __stcs(o, x2bf(z.re));
                __stcs(o + half, x2bf(z.im));
                if (Y32) {
                    f2x* f = reinterpret_cast<f2x*>(y32p + (size_t)i * 2 * row);
                    f[0] = z.re;
                    f[half] = z.im;   // M floats further: the imaginary half
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Chain prefix, run by every replay CTA for itself at its start: its
// kEngineWarps warps take equal ranges of the earlier (forward) or later
// (backward) CTA maps of the chain, compose them, and the partial maps are
// applied in a fixed order.  Maps are per mode {l.re, l.im, b.re, b.im}; lane
// l handles modes m, m+1 (cm points at mode m, CTA 0).
// ---------------------------------------------------------------------------
constexpr int kFoldChunk = 4;

template <int N>
__device__ __forceinline__ void ld_maps(const float4* __restrict__ cm, int M, int i0, int lo, int hi, int dir,
                                        float4 (&T)[N][2]) {
#pragma unroll
    for (int q = 0; q < N; ++q) {
        const int i = i0 + dir * q;
        if (i >= lo && i < hi) {
            T[q][0] = __ldcg(cm + (size_t)i * M);
            T[q][1] = __ldcg(cm + (size_t)i * M + 1);
        }
    }
}

// The state entering CTA cc of a chain, C_{cc-1} o ... o C_0 (h0), formed by
// the CTA's kEngineWarps warps: warp w composes the CTA maps of its range
// [cc w / 8, cc (w+1) / 8) in order (one batch of loads per kFoldChunk maps)
// and leaves the result in `xch(w)` (per lane 2 float4); after a CTA
// barrier every warp applies the 8 partial maps to h0 in warp order.  cm
// points at CTA 0's map of the lane's first mode; xch(w) must not be written
// by anything else meanwhile.  Fixed order; every warp gets the same bits.
template <class Xch>
__device__ __forceinline__ c2x cta_entry_fwd(const float4* __restrict__ cm, int cc, int M, const float* h0p, Xch xch,
                                             int warp, int lane, bool active) {
    const int lo = cc * warp / kEngineWarps, hi = cc * (warp + 1) / kEngineWarps;
    float4 P0 = identity_map(), P1 = P0;
    if (active) {
        for (int i0 = lo; i0 < hi; i0 += kFoldChunk) {
            float4 T[kFoldChunk][2];
            ld_maps(cm, M, i0, lo, hi, 1, T);
#pragma unroll
            for (int q = 0; q < kFoldChunk; ++q) {
                if (i0 + q < hi) {
                    P0 = compose_maps(T[q][0], P0);
                    P1 = compose_maps(T[q][1], P1);
                }
            }
        }
    }
    xch(warp)[2 * lane] = P0;
    xch(warp)[2 * lane + 1] = P1;
    __syncthreads();
    float2 z0 = make_float2(0.f, 0.f), z1 = z0;
    if (active && h0p != nullptr) {
        const float4 hv = *reinterpret_cast<const float4*>(h0p);
        z0 = make_float2(hv.x, hv.y);
        z1 = make_float2(hv.z, hv.w);
    }
#pragma unroll
    for (int v = 0; v < kEngineWarps; ++v) {
        z0 = capply(xch(v)[2 * lane], z0);
        z1 = capply(xch(v)[2 * lane + 1], z1);
    }
    __syncthreads();   // the exchange areas are free again
    c2x z;
    z.re = pk2(z0.x, z1.x);
    z.im = pk2(z0.y, z1.y);
    return z;
}

// Shared memory of the maps kernels' last phase, on top of the drained
// staging rings: the CTA's segment maps sit in the box area of warp 0's
// ring, never on a ring's mbarriers (whose memory is not reused).
struct EpilogueSmem {
    float4 (*seg)[32][2];
};
static_assert(sizeof(float4) * kEngineWarps * 32 * 2 <= sizeof(((MapRing*)nullptr)->box),
              "segment maps must fit a ring's box area");

__device__ __forceinline__ EpilogueSmem epilogue_smem(uint8_t* smem_raw) {
    EpilogueSmem e;
    e.seg = reinterpret_cast<float4 (*)[32][2]>(&warp_ring<MapRing>(smem_raw, 0).box[0][0][0][0]);
    return e;
}

__global__ void __launch_bounds__(kEngineThreads, 3)
    samu_fwd_maps_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ctrl,
                         SamuScanFwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    MapRing& R = warp_ring<MapRing>(smem_raw, warp);
    constexpr int kRing = MapRing::kSlots;
    constexpr int kN = MapRing::kRows;
    const SegGeom& g = a.g;
    const long long gw = (long long)blockIdx.x * kEngineWarps + warp;   // < n_chains * NS: whole CTAs
    const SegTask T = seg_task(g, gw);
    const int M = g.M;
    const int m = T.grp * kGroup + 2 * lane;
    const bool active = m < M;
    const int x_re = T.grp * kGroup, x_im = M + T.grp * kGroup;
    ring_init(R, lane);
    pdl_trigger();
    // item k is sub-chunk nsc-1-k: the segment from its end backwards.  w is an
    // input no earlier kernel of the call writes: its first boxes go out
    // before the wait for the controller forward; the control words after it.
    if (lane == 0)
        for (int k = 0; k < kRing && k < T.nsc; ++k)
            ring_issue_data(R, k, &tm_w, x_re, x_im, T.t_begin + (T.nsc - 1 - k) * kN, T.b);
    pdl_wait();
    if (lane == 0)
        for (int k = 0; k < kRing && k < T.nsc; ++k)
            ring_issue_ctrl(R, k, &tm_ctrl, T.t_begin + (T.nsc - 1 - k) * kN, T.b);
    const ModePair k = active ? load_modes(a.modes, a.nu, m) : zero_modes();
    ItemPlan plan;
    plan.q = -1;
    c2x P;
    P.re = dup2(1.f);
    P.im = 0ull;
    c2x be = czero();
    for (int it = 0; it < T.nsc; ++it) {
        const int slot = it % kRing;
        const int idx = T.nsc - 1 - it;   // the item's place in the segment
        const int ts = T.t_begin + idx * kN;
        const int nsub = min(kN, T.t_end - ts);
        if ((idx >> 5) != plan.q) plan_batch<true>(plan, a.items, T, g.L, idx >> 5, k, lane);
        SubKind kd;
        kd.fast = (plan.fast >> (idx & 31)) & 1u;
        kd.simple = (plan.simple >> (idx & 31)) & 1u;
        const float iG = __shfl_sync(0xffffffffu, plan.G, idx & 31);
        const float ic = __shfl_sync(0xffffffffu, plan.c, idx & 31);
        const float is = __shfl_sync(0xffffffffu, plan.s, idx & 31);
        if (!ring_wait(R, it, T.nsc, a.status, lane)) break;   // status set; the CTA still reaches its barriers
        const float4* sc = R.ctrl[slot];
        const uint32_t* wre = &R.box[slot][0][0][lane];
        const uint32_t* wim = &R.box[slot][1][0][lane];
        if (a.closed_form && kd.simple) {
            if (kd.fast)
                fwd_maps_item_cf<kN, true>(sc, wre, wim, k, a.modes + M, m, active, iG, ic, is, P, be);
            else
                fwd_maps_item_cf<kN, false>(sc, wre, wim, k, a.modes + M, m, active, iG, ic, is, P, be);
        } else {
            LRS_SUB_DISPATCH_N(kd, fwd_maps_sub, kN, sc, wre, wim, nsub, k, P, be);
        }
        __syncwarp();
        if (lane == 0 && it + kRing < T.nsc)
            ring_issue(R, slot, &tm_w, &tm_ctrl, x_re, x_im, T.t_begin + (T.nsc - 1 - it - kRing) * kN, T.b);
    }
    if (active) store_map2(a.smap + ((size_t)T.b * g.NS + T.s) * M + m, P, be);

    // CTA map: its segments composed in time order
    __syncthreads();   // rings drained
    const EpilogueSmem E = epilogue_smem(smem_raw);
    store_map2(&E.seg[warp][lane][0], P, be);
    __syncthreads();
    if (warp == 0) {
        const int cc = blockIdx.x % g.NC;
        float4 A0 = E.seg[0][lane][0], A1 = E.seg[0][lane][1];
#pragma unroll
        for (int w = 1; w < kEngineWarps; ++w) {
            A0 = compose_maps(E.seg[w][lane][0], A0);
            A1 = compose_maps(E.seg[w][lane][1], A1);
        }
        if (active) {
            float4* cm = a.cmap + ((size_t)T.b * g.NC + cc) * M + m;
            cm[0] = A0;
            cm[1] = A1;
        }
    }
}

template <bool Y32>
__global__ void __launch_bounds__(kEngineThreads, 3)
    samu_fwd_replay_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ctrl,
                           SamuScanFwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    MapRing& R = warp_ring<MapRing>(smem_raw, warp);
    constexpr int kRing = MapRing::kSlots;
    constexpr int kN = MapRing::kRows;
    const SegGeom& g = a.g;
    const long long gw = (long long)blockIdx.x * kEngineWarps + warp;   // < n_chains * NS: whole CTAs
    const SegTask T = seg_task(g, gw);
    const int M = g.M;
    const int L = g.L;
    const size_t D = 2 * (size_t)M;
    const int m = T.grp * kGroup + 2 * lane;
    const bool active = m < M;
    const int x_re = T.grp * kGroup, x_im = M + T.grp * kGroup;
    ring_init(R, lane);
    pdl_trigger();
    if (lane == 0)   // w (an input) before the wait for the maps kernel, control words after it
        for (int k = 0; k < kRing && k < T.nsc; ++k) ring_issue_data(R, k, &tm_w, x_re, x_im, T.t_begin + k * kN, T.b);
    pdl_wait();
    // the CTA's entry state from the earlier CTAs' maps (the rings' control-word
    // areas, not yet filled, carry the warps' partial maps)
    const int cc = T.s / kSegPerCta;
    const c2x e0 = cta_entry_fwd(
        a.cmap + (size_t)T.b * g.NC * M + m, cc, M, a.h0 != nullptr ? a.h0 + ((size_t)T.b * M + m) * 2 : nullptr,
        [&](int w) { return &warp_ring<MapRing>(smem_raw, w).ctrl[0][0]; }, warp, lane, active);
    if (lane == 0) {
        fence_proxy_async();
        for (int k = 0; k < kRing && k < T.nsc; ++k) ring_issue_ctrl(R, k, &tm_ctrl, T.t_begin + k * kN, T.b);
    }
    const ModePair k = active ? load_modes(a.modes, a.nu, m) : zero_modes();
    ItemPlan plan;
    plan.q = -1;
    c2x z = czero();
    if (active) {   // entry: the CTA's entry state through the maps of the earlier segments of the CTA
        float2 z0, z1;
        up2(e0.re, z0.x, z1.x);
        up2(e0.im, z0.y, z1.y);
        for (int v0 = cc * kSegPerCta; v0 < T.s; v0 += 4) {   // the CTA's earlier segments, 4 loads at a time
            float4 Tm[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (v0 + q < T.s) {
                    const float4* sm = a.smap + ((size_t)T.b * g.NS + v0 + q) * M + m;
                    Tm[q][0] = sm[0];
                    Tm[q][1] = sm[1];
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (v0 + q < T.s) {
                    z0 = capply(Tm[q][0], z0);
                    z1 = capply(Tm[q][1], z1);
                }
            }
        }
        z.re = pk2(z0.x, z1.x);
        z.im = pk2(z0.y, z1.y);
    }
    for (int it = 0; it < T.nsc; ++it) {
        const int slot = it % kRing;
        const int ts = T.t_begin + it * kN;
        const int nsub = min(kN, T.t_end - ts);
        // checkpoints (pairs {re, im}): the state entering token ts here, those
        // entering ts + 8, ... inside the item
        f2x* hs = active ? reinterpret_cast<f2x*>(a.hsub + ((size_t)T.b * g.CS + ts / kHalf) * M + m) : nullptr;
        if (active) {
            hs[0] = z.re;
            hs[1] = z.im;
        }

        if (!ring_wait(R, it, T.nsc, a.status, lane)) return;
        const float4* sc = R.ctrl[slot];
        const uint32_t* wre = &R.box[slot][0][0][lane];
        const uint32_t* wim = &R.box[slot][1][0][lane];
        const size_t row0 = (((size_t)T.b * L + ts) * D + m) / 2;
        float* y32p = Y32 ? a.y32 + 2 * row0 : nullptr;
        if ((it >> 5) != plan.q) plan_batch<false>(plan, a.items, T, L, it >> 5, k, lane);
        SubKind kd;
        kd.fast = (plan.fast >> (it & 31)) & 1u;
        kd.simple = (plan.simple >> (it & 31)) & 1u;
        LRS_SUB_DISPATCH_NX(kd, fwd_replay_sub, kN, Y32, sc, wre, wim, nsub, k, z, a.y + row0, y32p, active, D / 2,
                            M / 2, hs, M);
        __syncwarp();
        if (lane == 0 && it + kRing < T.nsc)
            ring_issue(R, slot, &tm_w, &tm_ctrl, x_re, x_im, T.t_begin + (it + kRing) * kN, T.b);
    }
    if (active && T.nsc > 0 && T.t_end == L) store_c2(a.hT + ((size_t)T.b * M + m) * 2, z);
}

// ---------------------------------------------------------------------------
// Backward.  The adjoint R arriving at a span's last token from later tokens
// leaves the span towards the past as Q R + beta, Q = conj(product of the
// span's lambdas); stored as {Q, beta} so that capply() applies it.  For one
// token, R -> conj(lambda_t) (R + dy_t).
// ---------------------------------------------------------------------------
// Appends the sub-chunk's tokens, earliest first, to the map G of the tokens
// before them: G o F_t = (Q conj(lambda_t), beta + Q conj(lambda_t) dy_t).
template <int N, bool FAST, bool SIMPLE>
__device__ __forceinline__ void bwd_maps_sub(const float4* sc, const uint32_t* gre, const uint32_t* gim, int nsub,
                                             const ModePair& k, c2x& Q, c2x& be) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        if (SIMPLE || i < nsub) {
            const Ctl2 ct = load_ctl(sc, i);
            const uint32_t gr = gre[i * kWords], gi = gim[i * kWords];
            if (SIMPLE || !is_reset(ct)) {
                Q = cmulc2(samu_lambda2<FAST>(k, ct), Q);
                c2x gg;
                gg.re = bf2x(gr);
                gg.im = bf2x(gi);
                be = cfma2(Q, gg, nbf2x(gi), be);
            } else {   // segment start: nothing reaches back past it
                Q = czero();
            }
        }
    }
}

// A full item of the adjoint maps (N tokens, none a reset), appended to the
// map G = (Q, beta) of the tokens before it: G o F_item = (Q conj(L), beta + Q x),
// x = conj(lambda_0) y_0 with y_{N-1} = g_{N-1} and
// y_i = g_i + conj(lambda_{i+1}) y_{i+1} (four paired FMAs per token).
template <int N, bool FAST>
__device__ __forceinline__ void bwd_maps_item_cf(const float4* sc, const uint32_t* gre, const uint32_t* gim,
                                                 const ModePair& k, const float4* __restrict__ modes_n, int m,
                                                 bool active, float G, float cs, float sn, c2x& Q, c2x& be) {
    c2x y;
    y.re = bf2x(gre[(N - 1) * kWords]);
    y.im = bf2x(gim[(N - 1) * kWords]);
#pragma unroll
    for (int i = N - 1; i > 0; --i) {
        const Lam2 l = samu_lambda2<FAST>(k, load_ctl(sc, i));
        const f2x gr = bf2x(gre[(i - 1) * kWords]);
        const f2x gi = bf2x(gim[(i - 1) * kWords]);
        const f2x yr = fma2(l.re, y.re, fma2(l.im, y.im, gr));
        const f2x yi = fma2(l.re, y.im, fma2(l.nim, y.re, gi));
        y.re = yr;
        y.im = yi;
    }
    const c2x x = cmulc2(samu_lambda2<FAST>(k, load_ctl(sc, 0)), y);
    c2x L = item_transition<N>(G, cs, sn, modes_n, k, m, active);
    L.im = sub2(0ull, L.im);   // conj
    const c2x Qx = cmulx(Q, x);
    be.re = add2(be.re, Qx.re);
    be.im = add2(be.im, Qx.im);
    Q = cmulx(Q, L);
}

// The adjoint arriving at the last token of CTA cc of a chain,
// C_{cc+1} o ... o C_{n-1} (dhT), formed like cta_entry_fwd over the later
// CTAs [cc+1, n): warp w composes its range from the latest map down.
template <class Xch>
__device__ __forceinline__ c2x cta_entry_bwd(const float4* __restrict__ cm, int cc, int n, int M, const float* dhTp,
                                             Xch xch, int warp, int lane, bool active) {
    const int cnt = n - 1 - cc;
    const int lo = cc + 1 + cnt * warp / kEngineWarps, hi = cc + 1 + cnt * (warp + 1) / kEngineWarps;
    float4 P0 = identity_map(), P1 = P0;
    if (active) {
        for (int i0 = hi - 1; i0 >= lo; i0 -= kFoldChunk) {
            float4 T[kFoldChunk][2];
            ld_maps(cm, M, i0, lo, hi, -1, T);
#pragma unroll
            for (int q = 0; q < kFoldChunk; ++q) {
                if (i0 - q >= lo) {
                    P0 = compose_maps(T[q][0], P0);
                    P1 = compose_maps(T[q][1], P1);
                }
            }
        }
    }
    xch(warp)[2 * lane] = P0;
    xch(warp)[2 * lane + 1] = P1;
    __syncthreads();
    float2 r0 = make_float2(0.f, 0.f), r1 = r0;
    if (active && dhTp != nullptr) {
        const float4 v = *reinterpret_cast<const float4*>(dhTp);
        r0 = make_float2(v.x, v.y);
        r1 = make_float2(v.z, v.w);
    }
#pragma unroll
    for (int v = kEngineWarps - 1; v >= 0; --v) {
        r0 = capply(xch(v)[2 * lane], r0);
        r1 = capply(xch(v)[2 * lane + 1], r1);
    }
    __syncthreads();
    c2x A;
    A.re = pk2(r0.x, r1.x);
    A.im = pk2(r0.y, r1.y);
    return A;
}

__global__ void __launch_bounds__(kEngineThreads, 3)
    samu_bwd_maps_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_ctrl,
                         SamuScanBwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    MapRing& R = warp_ring<MapRing>(smem_raw, warp);
    constexpr int kRing = MapRing::kSlots;
    constexpr int kN = MapRing::kRows;
    const SegGeom& g = a.g;
    const long long gw = (long long)blockIdx.x * kEngineWarps + warp;   // < n_chains * NS: whole CTAs
    const SegTask T = seg_task(g, gw);
    const int M = g.M;
    const int m = T.grp * kGroup + 2 * lane;
    const bool active = m < M;
    const int x_re = T.grp * kGroup, x_im = M + T.grp * kGroup;
    ring_init(R, lane);
    pdl_trigger();
    // item k is sub-chunk k: the segment from its start forwards (dy, an
    // input, before the dependency wait; control words after it)
    if (lane == 0)
        for (int k = 0; k < kRing && k < T.nsc; ++k) ring_issue_data(R, k, &tm_dy, x_re, x_im, T.t_begin + k * kN, T.b);
    pdl_wait();
    if (lane == 0)
        for (int k = 0; k < kRing && k < T.nsc; ++k) ring_issue_ctrl(R, k, &tm_ctrl, T.t_begin + k * kN, T.b);
    const ModePair k = active ? load_modes(a.modes, a.nu, m) : zero_modes();
    ItemPlan plan;
    plan.q = -1;
    c2x Q;
    Q.re = dup2(1.f);
    Q.im = 0ull;
    c2x be = czero();
    for (int it = 0; it < T.nsc; ++it) {
        const int slot = it % kRing;
        const int ts = T.t_begin + it * kN;
        const int nsub = min(kN, T.t_end - ts);
        if ((it >> 5) != plan.q) plan_batch<true>(plan, a.items, T, g.L, it >> 5, k, lane);
        SubKind kd;
        kd.fast = (plan.fast >> (it & 31)) & 1u;
        kd.simple = (plan.simple >> (it & 31)) & 1u;
        const float iG = __shfl_sync(0xffffffffu, plan.G, it & 31);
        const float ic = __shfl_sync(0xffffffffu, plan.c, it & 31);
        const float is = __shfl_sync(0xffffffffu, plan.s, it & 31);
        if (!ring_wait(R, it, T.nsc, a.status, lane)) break;   // status set; the CTA still reaches its barriers
        const float4* sc = R.ctrl[slot];
        const uint32_t* gre = &R.box[slot][0][0][lane];
        const uint32_t* gim = &R.box[slot][1][0][lane];
        if (a.closed_form && kd.simple) {
            if (kd.fast)
                bwd_maps_item_cf<kN, true>(sc, gre, gim, k, a.modes + M, m, active, iG, ic, is, Q, be);
            else
                bwd_maps_item_cf<kN, false>(sc, gre, gim, k, a.modes + M, m, active, iG, ic, is, Q, be);
        } else {
            LRS_SUB_DISPATCH_N(kd, bwd_maps_sub, kN, sc, gre, gim, nsub, k, Q, be);
        }
        __syncwarp();
        if (lane == 0 && it + kRing < T.nsc)
            ring_issue(R, slot, &tm_dy, &tm_ctrl, x_re, x_im, T.t_begin + (it + kRing) * kN, T.b);
    }
    if (active) store_map2(a.smap + ((size_t)T.b * g.NS + T.s) * M + m, Q, be);

    // adjoint CTA map (the latest segment applied first)
    __syncthreads();   // rings drained
    const EpilogueSmem E = epilogue_smem(smem_raw);
    store_map2(&E.seg[warp][lane][0], Q, be);
    __syncthreads();
    if (warp == 0) {
        const int cc = blockIdx.x % g.NC;
        float4 A0 = E.seg[kEngineWarps - 1][lane][0], A1 = E.seg[kEngineWarps - 1][lane][1];
#pragma unroll
        for (int w = kEngineWarps - 2; w >= 0; --w) {
            A0 = compose_maps(E.seg[w][lane][0], A0);
            A1 = compose_maps(E.seg[w][lane][1], A1);
        }
        if (active) {
            float4* cm = a.cmap + ((size_t)T.b * g.NC + cc) * M + m;
            cm[0] = A0;
            cm[1] = A1;
        }
    }
}

// ---------------------------------------------------------------------------
// Reverse replay.  It walks each segment backwards in units of 8 tokens, the
// distance between the forward's state checkpoints.  One ring slot holds a
// whole unit: its w rows, its dy rows (overwritten by its dw rows when dw
// leaves by TMA) and its control words, so a unit costs one wait and one
// refill.  The forward sweep rebuilds the unit's states from the checkpoint
// with the forward replay's own step (the same bits) and keeps lambda_t and
// the state z_{t-1} entering every token in registers; the reverse sweep
// then runs the adjoint.
// ---------------------------------------------------------------------------
template <int S>
struct alignas(128) RevRingT {
    static constexpr int kSlots = S;
    static constexpr int kUnitBytes = 4 * kHalf * kRowBytes + kHalf * kCtlBytes;
    uint32_t w[S][2][kHalf][kWords];   // [slot][re, im][token][pair]
    uint32_t g[S][2][kHalf][kWords];   // dy rows, then (TMA variant) dw rows
    float4 ctrl[S][2 * kHalf];         // [slot][token: two float4]
    float4 ck[2][32];                  // two units' checkpoints, {re, re, im, im} per lane (per-lane async copies)
    uint64_t full[S];
};
using RevRing = RevRingT<3>;
constexpr int kRevSmem = kEngineWarps * (int)sizeof(RevRing);
static_assert(sizeof(float4) * 2 * 32 <= sizeof(((RevRing*)nullptr)->w[0]),
              "a slot's w rows hold the prologue's partial maps");

__device__ __forceinline__ RevRing& rev_ring(uint8_t* smem_raw, int warp) {
    return *reinterpret_cast<RevRing*>(smem_raw + (size_t)warp * sizeof(RevRing));
}

// Per-lane asynchronous 16-byte copy global -> shared (cp.async, no register
// staging); each lane waits for its own copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Lane 0: the w and dy rows of the unit at token ts into `slot` (the slot's
// expected bytes include the control words: it completes once
// rev_issue_ctrl has been issued too).
__device__ __forceinline__ void rev_issue_data(RevRing& R, int slot, const CUtensorMap* tm_w, const CUtensorMap* tm_dy,
                                               int x_re, int x_im, int ts, int b) {
    fence_proxy_async();
    mbar_arrive_expect_tx(&R.full[slot], RevRing::kUnitBytes);
    tma_load_3d(&R.w[slot][0][0][0], tm_w, x_re, ts, b, &R.full[slot]);
    tma_load_3d(&R.w[slot][1][0][0], tm_w, x_im, ts, b, &R.full[slot]);
    tma_load_3d(&R.g[slot][0][0][0], tm_dy, x_re, ts, b, &R.full[slot]);
    tma_load_3d(&R.g[slot][1][0][0], tm_dy, x_im, ts, b, &R.full[slot]);
}
__device__ __forceinline__ void rev_issue_ctrl(RevRing& R, int slot, const CUtensorMap* tm_ctrl, int ts, int b) {
    tma_load_3d(&R.ctrl[slot][0], tm_ctrl, 0, ts, b, &R.full[slot]);
}

// Forward sweep of one unit from its entry state z: for every token lambda_t
// and the state z_{t-1} entering it; z_t = lambda_t z_{t-1} + b_t with the
// forward replay's expression.  A reset token gets lambda_t = 0 (z_t = b_t).
template <bool FAST, bool SIMPLE>
__device__ __forceinline__ void rev_forward_sweep(const float4* sc, const uint32_t* wre, const uint32_t* wim, int nh,
                                                  const ModePair& k, c2x z, c2x (&zp)[kHalf], f2x (&lre)[kHalf],
                                                  f2x (&lim)[kHalf]) {
#pragma unroll
    for (int i = 0; i < kHalf; ++i) {
        zp[i] = z;
        lre[i] = 0ull;
        lim[i] = 0ull;
        if (SIMPLE || i < nh) {
            const Ctl2 ct = load_ctl(sc, i);
            const f2x bre = bf2x(wre[i * kWords]);
            const f2x bim = bf2x(wim[i * kWords]);
            if (SIMPLE || !is_reset(ct)) {
                const Lam2 l = samu_lambda2<FAST>(k, ct);
                const f2x zr = fma2(l.re, z.re, fma2(l.nim, z.im, bre));
                const f2x zi = fma2(l.re, z.im, fma2(l.im, z.re, bim));
                z.re = zr;
                z.im = zi;
                lre[i] = l.re;
                lim[i] = l.im;
            } else {
                z.re = bre;
                z.im = bim;
            }
        }
    }
}

// Sums v[k] over the 32 lanes for every k of 16 values at once: halving
// exchanges inside each 16-lane half, then one exchange across the halves.
// On return lane L holds the total of v[L mod 16].  Fixed order.
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const float send = up ? v[j] : v[j + o];
            const float keep = up ? v[j + o] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// How the reverse replay writes dw.
enum DwStore { kDwBf16 = 0, kDwFp32 = 1, kDwBf16Tma = 2 };

// Reverse sweep of one unit: A_t = dy_t + (adjoint from t+1); dw_t = A_t;
// A'_t = conj(lambda_t) A_t, the adjoint passed to t-1; then
// kappa_t = A_t conj(lambda_t z_{t-1}) = A'_t conj(z_{t-1});
// dtheta_m += Im kappa, dnu_m += -E_t Re kappa; per token dbar += Im kappa
// and Ebar += -nu_m Re kappa summed over the 64 modes of the warp (written
// to kp[token * kp_row + {0, 1}]).  DW == kDwBf16Tma: dw_t replaces dy_t in
// the staged rows (every lane active), stored by TMA afterwards.
template <bool SIMPLE, int DW>
__device__ __forceinline__ void rev_reverse_sweep(const float4* sc, uint32_t* gre, uint32_t* gim, int nh,
                                                  float nu0, float nu1, const c2x (&zp)[kHalf],
                                                  const f2x (&lre)[kHalf], const f2x (&lim)[kHalf], c2x& A,
                                                  f2x& acc_nu, f2x& acc_th, uint32_t* dwb, float* dwf,
                                                  bool active, size_t row, int half, float* kp, size_t kp_row,
                                                  int lane) {
    float v[2 * kHalf];
#pragma unroll
    for (int i = kHalf - 1; i >= 0; --i) {
        v[2 * i] = 0.f;
        v[2 * i + 1] = 0.f;
        if (SIMPLE || i < nh) {
            const float rw = sc[2 * i + 1].z;   // -E, or +0 at a segment start
            A.re = add2(A.re, bf2x(gre[i * kWords]));
            A.im = add2(A.im, bf2x(gim[i * kWords]));
            if (DW == kDwBf16Tma) {
                gre[i * kWords] = x2bf(A.re);
                gim[i * kWords] = x2bf(A.im);
            } else if (active) {
                if (DW == kDwFp32) {
                    f2x* p = reinterpret_cast<f2x*>(dwf + 2 * (size_t)i * row);
                    p[0] = A.re;
                    p[half] = A.im;   // M floats further: the imaginary half
                } else {
                    uint32_t* p = dwb + (size_t)i * row;
                    __stcs(p, x2bf(A.re));
                    __stcs(p + half, x2bf(A.im));
                }
            }
            if (SIMPLE || !is_reset_word(rw)) {
                // A' = conj(lambda) A
                const f2x ar = fma2(lre[i], A.re, mul2(lim[i], A.im));
                const f2x ai = fma2(lre[i], A.im, mul2(sub2(0ull, lim[i]), A.re));
                // kappa = A' conj(z_{t-1})
                const f2x kr = fma2(ar, zp[i].re, mul2(ai, zp[i].im));
                const f2x ki = fma2(ai, zp[i].re, mul2(sub2(0ull, ar), zp[i].im));
                acc_nu = fma2(dup2(rw), kr, acc_nu);   // -E_t Re kappa
                acc_th = add2(acc_th, ki);
                float ki0, ki1, kr0, kr1;
                up2(ki, ki0, ki1);
                up2(kr, kr0, kr1);
                v[2 * i] = ki0 + ki1;
                v[2 * i + 1] = -__fmaf_rn(nu0, kr0, __fmul_rn(nu1, kr1));
                A.re = ar;
                A.im = ai;
            } else {   // segment start: no controller terms, the adjoint stops here
                A = czero();
            }
        }
    }
    const float tot = warp_reduce_scatter16(v, lane);
    if (lane < 2 * kHalf && (lane >> 1) < nh) kp[(size_t)(lane >> 1) * kp_row + (lane & 1)] = tot;
}

// One unit (forward sweep, reverse sweep) of kind <FAST, SIMPLE>.
template <bool FAST, bool SIMPLE, int DW>
__device__ __forceinline__ void rev_unit(RevRing& R, int slot, int nh, const ModePair& k, float nu0, float nu1,
                                         const c2x& z, c2x& A, f2x& acc_nu, f2x& acc_th, uint32_t* dwb, float* dwf,
                                         bool active, size_t row, int half, float* kp, size_t kp_row, int lane) {
    const float4* sc = R.ctrl[slot];
    c2x zp[kHalf];
    f2x lre[kHalf], lim[kHalf];
    rev_forward_sweep<FAST, SIMPLE>(sc, &R.w[slot][0][0][lane], &R.w[slot][1][0][lane], nh, k, z, zp, lre, lim);
    rev_reverse_sweep<SIMPLE, DW>(sc, &R.g[slot][0][0][lane], &R.g[slot][1][0][lane], nh, nu0, nu1, zp, lre, lim, A,
                                  acc_nu, acc_th, dwb, dwf, active, row, half, kp, kp_row, lane);
}

// Warp-uniform facts about the whole segment, from the forward's item
// records: simple (every item full and free of resets) and fast
// (|nu| max|E - 1| < kPolyBound for every lane's modes).  A segment that is
// both runs every unit on the branch-free polynomial path; one that is not
// decides per unit (sub_kind), as the forward replay does per item.
__device__ __forceinline__ SubKind segment_kind(const float4* __restrict__ items, const SegTask& T, int L, int lane,
                                                const ModePair& k) {
    const int n_it = (T.t_end - T.t_begin + kMapRows - 1) / kMapRows;
    float emax = 0.f;
    bool simple = true;
    for (int i = lane; i < n_it; i += 32) {
        const float v = __ldcg(&items[(size_t)T.b * samu_items_per_row(L) + T.t_begin / kMapRows + i].w);
        emax = fmaxf(emax, record_emax(v));
        simple = simple && v >= 0.f;
    }
    SubKind kd;
    kd.fast = warp_numax(k) * __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(emax))) < kPolyBound;
    kd.simple = __all_sync(0xffffffffu, simple);
    return kd;
}

template <int DW>
__global__ void __launch_bounds__(kEngineThreads, 2)
    samu_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ CUtensorMap tm_ctrl, const __grid_constant__ CUtensorMap tm_dw,
                         SamuScanBwdArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    RevRing& R = rev_ring(smem_raw, warp);
    constexpr int kS = RevRing::kSlots;
    const SegGeom& g = a.g;
    const long long gw = (long long)blockIdx.x * kEngineWarps + warp;
    const SegTask T = seg_task(g, gw);
    const int M = g.M;
    const int L = g.L;
    const size_t D = 2 * (size_t)M;
    const int m = T.grp * kGroup + 2 * lane;
    const bool active = m < M;
    const int x_re = T.grp * kGroup, x_im = M + T.grp * kGroup;
    const int n_units = T.t_end > T.t_begin ? (T.t_end - T.t_begin + kHalf - 1) / kHalf : 0;
    // unit u: tokens from ts(u), the segment from its end backwards
    auto unit_ts = [&](int u) { return T.t_begin + (n_units - 1 - u) * kHalf; };
    // the forward's checkpoint of unit u (the state entering its first token),
    // fetched one unit ahead by per-lane asynchronous copies
    auto ckpt_src = [&](int u) {
        return reinterpret_cast<const float4*>(a.hsub + ((size_t)T.b * g.CS + unit_ts(u) / kHalf) * M + m);
    };
    if (lane == 0)
        for (int s = 0; s < kS; ++s) mbar_init(&R.full[s], 1);
    __syncwarp();
    pdl_trigger();
    // w, dy (inputs) and the forward's control words and checkpoints (written
    // before the previous, ordinary launch) are read before the dependency
    // wait; slot kS - 1's w rows carry the prologue's partial maps, so its
    // unit goes out after the fold.
    if (lane == 0)
        for (int u = 0; u < kS - 1 && u < n_units; ++u) rev_issue_data(R, u, &tm_w, &tm_dy, x_re, x_im, unit_ts(u), T.b);
    const ModePair k = active ? load_modes(a.modes, a.nu, m) : zero_modes();
    float nu0, nu1;
    up2(k.nu, nu0, nu1);
    const SubKind seg_kd = segment_kind(a.items, T, L, lane, k);
    if (active && n_units > 0) cp_async16(&R.ck[0][lane], ckpt_src(0));
    cp_async_commit();
    pdl_wait();
    // the adjoint arriving at the CTA from the later CTAs' maps
    const int cc = T.s / kSegPerCta;
    const c2x a0 = cta_entry_bwd(
        a.cmap + (size_t)T.b * g.NC * M + m, cc, g.NC, M, a.dhT != nullptr ? a.dhT + ((size_t)T.b * M + m) * 2 : nullptr,
        [&](int w) { return reinterpret_cast<float4*>(&rev_ring(smem_raw, w).w[kS - 1][0][0][0]); }, warp, lane,
        active);
    if (lane == 0) {
        if (kS - 1 < n_units) rev_issue_data(R, kS - 1, &tm_w, &tm_dy, x_re, x_im, unit_ts(kS - 1), T.b);
        for (int u = 0; u < kS && u < n_units; ++u) rev_issue_ctrl(R, u, &tm_ctrl, unit_ts(u), T.b);
    }
    c2x A = czero();
    if (active) {   // the adjoint arriving at the CTA through the maps of the later segments of the CTA
        float2 r0, r1;
        up2(a0.re, r0.x, r1.x);
        up2(a0.im, r0.y, r1.y);
        for (int v1 = (cc + 1) * kSegPerCta - 1; v1 > T.s; v1 -= 4) {   // the CTA's later segments, latest first
            float4 Tm[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (v1 - q > T.s) {
                    const float4* sm = a.smap + ((size_t)T.b * g.NS + v1 - q) * M + m;
                    Tm[q][0] = sm[0];
                    Tm[q][1] = sm[1];
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (v1 - q > T.s) {
                    r0 = capply(Tm[q][0], r0);
                    r1 = capply(Tm[q][1], r1);
                }
            }
        }
        A.re = pk2(r0.x, r1.x);
        A.im = pk2(r0.y, r1.y);
    }
    f2x acc_nu = 0ull, acc_th = 0ull;
    const size_t kp_row = 2 * (size_t)g.n_groups;
    int slot = 0;
    uint32_t phase = 0;
    for (int u = 0; u < n_units; ++u) {
        const int ts = unit_ts(u);
        const int nh = min(kHalf, T.t_end - ts);
        c2x z = czero();   // the forward's checkpoint: the state entering token ts
        cp_async_wait_all();
        if (active) {
            const float4 c4 = R.ck[u & 1][lane];
            z.re = pk2(c4.x, c4.y);
            z.im = pk2(c4.z, c4.w);
        }
        if (active && u + 1 < n_units) cp_async16(&R.ck[(u + 1) & 1][lane], ckpt_src(u + 1));
        cp_async_commit();
        const size_t row0 = (((size_t)T.b * L + ts) * D + m) / 2;
        uint32_t* dwb = reinterpret_cast<uint32_t*>(a.dw) + row0;
        float* dwf = reinterpret_cast<float*>(a.dw) + 2 * row0;
        float* kp = reinterpret_cast<float*>(a.kpart + ((size_t)T.b * L + ts) * g.n_groups + T.grp);
        if (!mbar_wait_bounded(&R.full[slot], phase)) {
            cp_async_wait_all();   // this lane's checkpoint copy lands before the CTA may exit
            if (lane == 0) {
                atomicOr(a.status, kStatusTimeout);
                if (DW == kDwBf16Tma) bulk_wait_all();
            }
            // the copies still in flight: units up to u + kS - 1 (the TMA-store
            // variant refills one unit later: up to max(kS - 1, u + 1))
            const int last = DW == kDwBf16Tma ? max(kS - 1, u + 1) : u + kS - 1;
            for (int j = u + 1; j <= last && j < n_units; ++j)
                mbar_wait_bounded(&R.full[j % kS], (uint32_t)(j / kS) & 1u);
            return;
        }
        if (seg_kd.fast && seg_kd.simple) {
            rev_unit<true, true, DW>(R, slot, nh, k, nu0, nu1, z, A, acc_nu, acc_th, dwb, dwf, active, D / 2, M / 2,
                                     kp, kp_row, lane);
        } else {
            const SubKind kd = sub_kind<kHalf>(R.ctrl[slot], nh, lane, k);
            if (kd.fast) {
                if (kd.simple)
                    rev_unit<true, true, DW>(R, slot, nh, k, nu0, nu1, z, A, acc_nu, acc_th, dwb, dwf, active, D / 2,
                                             M / 2, kp, kp_row, lane);
                else
                    rev_unit<true, false, DW>(R, slot, nh, k, nu0, nu1, z, A, acc_nu, acc_th, dwb, dwf, active, D / 2,
                                              M / 2, kp, kp_row, lane);
            } else {
                if (kd.simple)
                    rev_unit<false, true, DW>(R, slot, nh, k, nu0, nu1, z, A, acc_nu, acc_th, dwb, dwf, active,
                                              D / 2, M / 2, kp, kp_row, lane);
                else
                    rev_unit<false, false, DW>(R, slot, nh, k, nu0, nu1, z, A, acc_nu, acc_th, dwb, dwf, active,
                                               D / 2, M / 2, kp, kp_row, lane);
            }
        }
        if (DW == kDwBf16Tma) {
            // the unit's dw rows are in this slot: TMA-store them, then refill
            // the previous unit's slot once its store has read it
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&tm_dw, x_re, ts, T.b, &R.g[slot][0][0][0]);
                tma_store_3d(&tm_dw, x_im, ts, T.b, &R.g[slot][1][0][0]);
                bulk_commit();
                const int j = u - 1 + kS;
                if (u >= 1 && j < n_units) {
                    bulk_wait_read<1>();
                    const int ps = slot == 0 ? kS - 1 : slot - 1;
                    rev_issue_data(R, ps, &tm_w, &tm_dy, x_re, x_im, unit_ts(j), T.b);
                    rev_issue_ctrl(R, ps, &tm_ctrl, unit_ts(j), T.b);
                }
            }
        } else {
            __syncwarp();
            if (lane == 0 && u + kS < n_units) {
                rev_issue_data(R, slot, &tm_w, &tm_dy, x_re, x_im, unit_ts(u + kS), T.b);
                rev_issue_ctrl(R, slot, &tm_ctrl, unit_ts(u + kS), T.b);
            }
        }
        if (++slot == kS) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (DW == kDwBf16Tma && lane == 0) bulk_wait_all();
    if (active) {
        float n0, n1, t0, t1;
        up2(acc_nu, n0, n1);
        up2(acc_th, t0, t1);
        *reinterpret_cast<float4*>(a.numod + ((size_t)T.b * g.NS + T.s) * M + m) = make_float4(n0, t0, n1, t1);
        if (T.s == 0) store_c2(a.dh0 + ((size_t)T.b * M + m) * 2, A);
    }
}

// ---------------------------------------------------------------------------
// Host side.
namespace {

struct EngineOccupancy {
    bool done = false;
    int sms = 0;
    int fwd = 0;   // resident CTAs per SM for the forward pair (maps, replay)
    int bwd = 0;   // ... and for the backward pair (maps, main)
};

// Per device, filled once under g_occ_mutex (calls may come from several
// host threads).
EngineOccupancy g_occ[64];
std::mutex g_occ_mutex;

bool set_smem(const void* fn, int smem) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
}

int occupancy(const void* fn, int smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kEngineThreads, smem) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

const EngineOccupancy& engine_occupancy() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    EngineOccupancy& o = g_occ[dev];
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (!o.done) {
        int v = 0;
        o.sms = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 1;
        const void* fwd[] = {reinterpret_cast<const void*>(samu_fwd_maps_kernel),
                             reinterpret_cast<const void*>(samu_fwd_replay_kernel<false>),
                             reinterpret_cast<const void*>(samu_fwd_replay_kernel<true>)};
        const void* bwd[] = {reinterpret_cast<const void*>(samu_bwd_maps_kernel),
                             reinterpret_cast<const void*>(samu_bwd_main_kernel<kDwBf16>),
                             reinterpret_cast<const void*>(samu_bwd_main_kernel<kDwFp32>),
                             reinterpret_cast<const void*>(samu_bwd_main_kernel<kDwBf16Tma>)};
        const int bwd_smem[] = {kEngineSmem, kRevSmem, kRevSmem, kRevSmem};
        o.fwd = 1 << 30;
        for (const void* f : fwd) {
            set_smem(f, kEngineSmem);
            o.fwd = std::min(o.fwd, occupancy(f, kEngineSmem));
        }
        o.bwd = 1 << 30;
        for (int i = 0; i < 4; ++i) {
            set_smem(bwd[i], bwd_smem[i]);
            o.bwd = std::min(o.bwd, occupancy(bwd[i], bwd_smem[i]));
        }
        o.done = true;
    }
    return o;
}

unsigned engine_grid(const SegGeom& g) {
    const long long warps = (long long)g.n_chains * g.NS;
    return (unsigned)((warps + kEngineWarps - 1) / kEngineWarps);
}

}  // namespace

SegGeom samu_scan_geom(int B, int L, int M, bool backward) {
    const EngineOccupancy& o = engine_occupancy();
    const long long warps = (long long)(backward ? o.bwd : o.fwd) * kEngineWarps * o.sms;
    return samu_seg_geom(B, L, M, warps);
}

cudaError_t launch_samu_fwd_maps(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                 cudaStream_t s, bool pdl) {
    return launch_ex(samu_fwd_maps_kernel, engine_grid(args.g), kEngineThreads, kEngineSmem, s, pdl, tm_w, tm_ctrl,
                     args);
}

cudaError_t launch_samu_fwd_replay(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                   cudaStream_t s, bool pdl) {
    if (args.y32 != nullptr)
        return launch_ex(samu_fwd_replay_kernel<true>, engine_grid(args.g), kEngineThreads, kEngineSmem, s, pdl, tm_w,
                         tm_ctrl, args);
    return launch_ex(samu_fwd_replay_kernel<false>, engine_grid(args.g), kEngineThreads, kEngineSmem, s, pdl, tm_w,
                     tm_ctrl, args);
}

cudaError_t launch_samu_bwd_maps(const CUtensorMap& tm_dy, const CUtensorMap& tm_ctrl, const SamuScanBwdArgs& args,
                                 cudaStream_t s, bool pdl) {
    return launch_ex(samu_bwd_maps_kernel, engine_grid(args.g), kEngineThreads, kEngineSmem, s, pdl, tm_dy, tm_ctrl,
                     args);
}

cudaError_t launch_samu_bwd_main(const CUtensorMap& tm_dy, const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl,
                                 const CUtensorMap& tm_dw, const SamuScanBwdArgs& args, cudaStream_t s, bool pdl) {
    const unsigned grid = engine_grid(args.g);
    if (args.grad_fp32)
        return launch_ex(samu_bwd_main_kernel<kDwFp32>, grid, kEngineThreads, kRevSmem, s, pdl, tm_dy, tm_w, tm_ctrl,
                         tm_dw, args);
    if (args.g.M % kGroup == 0)
        return launch_ex(samu_bwd_main_kernel<kDwBf16Tma>, grid, kEngineThreads, kRevSmem, s, pdl, tm_dy, tm_w,
                         tm_ctrl, tm_dw, args);
    return launch_ex(samu_bwd_main_kernel<kDwBf16>, grid, kEngineThreads, kRevSmem, s, pdl, tm_dy, tm_w, tm_ctrl,
                     tm_dw, args);
}

}  // namespace lrs

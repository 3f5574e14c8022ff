// Kernel argument blocks, shared per-step device functions and launcher
// declarations of the CUDA library.
#pragma once

#include "common.cuh"
#include "layout.cuh"

namespace lrs {

constexpr float kLog2e = 1.4426950408889634f;

// Per-mode constants of the transition.  lambda_{t,m} = e^{-nu_m E_t} e^{i(theta_m + d_t)}
// (SAMU GPU page, section 05, transition equation) is evaluated as
//   lambda_{t,m} = lbar_m * delta_{t,m},  lbar_m = e^{-nu_m} e^{i theta_m},
//   delta_{t,m} = e^{-nu_m (E_t - 1)} (C_t + i S_t),
// which is the same number.  lbar_m is held as a double-float (hi + lo, formed
// once in FP64), so no per-mode rounding of e^{-nu}, cos theta or sin theta
// biases every step of a long chain; delta is close to 1 and formed per step
// in FP32 from E_t - 1 = expm1(c_t) and the shared C_t, S_t.
struct ModeConst {
    float hr, hi, lr, li;   // lbar: hi part (re, im), lo part (re, im)
    float nu;
};

__device__ __forceinline__ ModeConst load_mode(const float4* __restrict__ modes,
                                               const float* __restrict__ nu, int m) {
    const float4 v = modes[m];
    ModeConst k;
    k.hr = v.x;
    k.hi = v.y;
    k.lr = v.z;
    k.li = v.w;
    k.nu = nu[m];
    return k;
}

// Per-token control word, written by the controller forward and staged into
// shared memory by TMA: {E_t - 1, C_t, S_t, reset_t} with reset_t 1 at a
// segment start (lambda = 0) and 0 elsewhere.  It is the same for every lane,
// so the branches on it are warp-uniform.

// Bound on |nu (E - 1)| under which the degree-3 polynomial below is exact to
// < 2e-11 relative (the truncation term x^4/24), checked once per warp and tile.
constexpr float kPolyBound = 1.0f / 64.0f;

// lambda_{t,m} for a token that is not a reset: lbar_m * e^{-nu (E-1)} (C + iS).
// FAST: e^{-x} by its degree-3 Taylor polynomial (valid for |x| < kPolyBound;
// its rounding errors carry no per-mode bias); otherwise ex2.approx, whose
// ~1e-7 error matters little for the short-memory modes that need it.
// Every pass that needs lambda calls this, so the forward and the backward
// rebuild the same bits.
template <bool FAST>
__device__ __forceinline__ float2 samu_lambda(const ModeConst& k, float4 ctl) {
    const float x = __fmul_rn(k.nu, ctl.x);                 // nu (E - 1)
    float q;                                                 // e^{-x}
    if (FAST) {
        q = __fmaf_rn(x, __fmaf_rn(x, __fmaf_rn(x, -1.0f / 6.0f, 0.5f), -1.0f), 1.0f);
    } else {
        q = ex2_approx(__fmul_rn(-x, kLog2e));
    }
    const float dr = __fmul_rn(q, ctl.y);
    const float di = __fmul_rn(q, ctl.z);
    return make_float2(__fmaf_rn(k.hr, dr, __fmaf_rn(-k.hi, di, k.lr)),
                       __fmaf_rn(k.hr, di, __fmaf_rn(k.hi, dr, k.li)));
}

// One state step z' = lambda z + b, formed as u = lambda z then u + b.  The
// backward keeps u = lambda z_{t-1} for kappa, so both directions use this form.
__device__ __forceinline__ float2 step_state(float2 l, float2 bb, float2 z, float2* u_out = nullptr) {
    const float2 u = cmul(l, z);
    if (u_out) *u_out = u;
    return make_float2(__fadd_rn(u.x, bb.x), __fadd_rn(u.y, bb.y));
}

// S <- T_t o S for T_t(h) = l h + bb, S = {Lambda, beta}.
__device__ __forceinline__ float4 compose_step(float2 l, float2 bb, float4 S) {
    const float2 L = cmul(l, make_float2(S.x, S.y));
    const float2 Bv = capply(make_float4(l.x, l.y, bb.x, bb.y), make_float2(S.z, S.w));
    return make_float4(L.x, L.y, Bv.x, Bv.y);
}

// Forward scan over segments: segment maps, chain prefix, replay.  w and
// the control words reach the kernels through TMA tensor maps (16-token
// boxes); everything indexed by segment is [B][NS][M] (per mode).
struct SamuScanFwdArgs {
    SegGeom g;
    const float4* modes;    // [M] lbar hi/lo
    const float* nu;
    const float* h0;        // [B,M,2] or null
    uint32_t* y;            // BF16 pairs of y
    float* y32;             // optional
    float* hT;              // [B,M,2]
    float2* hsub;           // [B][CS][M] entry state of every 16-token sub-chunk
    float4* smap;           // [B][NS][M] segment maps
    float2* sent;           // [B][NS][M] segment entry states
    uint32_t* status;       // cleared by the maps kernel
};

// Backward scan over segments: adjoint segment maps, reverse chain prefix,
// reverse replay.  sent holds the adjoint arriving at each segment's last
// token from later tokens.
struct SamuScanBwdArgs {
    SegGeom g;
    const float4* modes;
    const float* nu;
    const float* dhT;       // [B,M,2] or null
    const float2* hsub;     // [B][CS][M] (the forward's sub-chunk entry states)
    void* dw;               // BF16 pairs or FP32
    int grad_fp32;
    float* dh0;             // [B,M,2]
    float4* smap;           // [B][NS][M] adjoint segment maps
    float2* sent;           // [B][NS][M] incoming adjoints
    float2* kpart;          // [B*L][n_groups] {sum Im kappa, sum -nu Re kappa}
    float2* numod;          // [B][NS][M] {dnu, dtheta} per segment
    uint32_t* status;
};

// Controller streaming geometry: every CTA owns a contiguous run of
// `stage_tok`-token stages of x_sel (and of dx_sel), staged through a ring of
// `ring` shared-memory slots by 1-D bulk copies; one producer warp plus
// `consumers` warps of 32 threads, each thread owning 8 channels.
struct CtrlGeom {
    int stage_tok;          // tokens per stage (16, or 8 when 16 rows exceed 64 KB)
    int ring;               // slots (at most 8, filling up to 192 KB)
    int consumers;          // consumer warps
    int threads;            // 32 * (1 + consumers)
    int smem;               // dynamic shared memory bytes
    int n_ctas;             // streaming CTAs
    long long n_stages;     // ceil(B*L / stage_tok)
    int max_cta_tok;        // tokens of the longest CTA range (backward scalar buffer)
};

CtrlGeom samu_ctrl_geom(long long BL, int D, bool backward);

struct SamuCtrlBwdArgs {
    long long BL;
    int D, n_groups;
    CtrlGeom cg;
    const uint4* x;         // BF16 x_sel as 16-byte vectors
    const float2* kpart;
    const float* p;
    const float* r;
    const float4* ctrl;
    const float* wh;        // [2][D+1]
    const float* misc;
    void* dx;               // BF16 or FP32
    int grad_fp32;
    float* dwh_part;        // [cg.n_ctas][2][D+1]
    float2* amp_part;       // [cg.n_ctas]
    uint32_t* status;
};

struct SamuParamArgs {
    int B, L, D;
    int n_part;             // numod rows per batch row
    int n_rows;             // rows of dwh_part / amp_part
    const float2* numod;    // [B*n_part][M]
    const float* dwh_part;  // [n_rows][2][D+1]
    const float2* amp_part;
    float* dwh;             // [2][D+1] column sums of dwh_part
    uint32_t* counter;      // CTA arrival counter, zero on entry, left zero
    const float* wh;
    const float* misc;
    float* dnu;
    float* dtheta;
    float* dw_phi;
    float* dw_r;
    float* da_phi;
    float* da_r;
};

struct SamuCtrlFwdArgs {
    long long BL;
    int D;
    int n_mode_ctas;               // filled by the launcher
    CtrlGeom cg;                   // filled by the launcher
    const uint4* x;                // BF16 x_sel as 16-byte vectors
    const uint8_t* reset;
    const float* w_phi;
    const float* w_r;
    const float* a_phi;
    const float* a_r;
    const float* nu;
    const float* theta;
    float* p;
    float* r;
    float4* ctrl;                  // {E - 1, C, S, reset}
    float* wh;                     // [2][D+1]
    float* misc;
    float4* modes;                 // [M] lbar hi/lo
    uint32_t* status;
};

cudaError_t launch_samu_ctrl_fwd(const SamuCtrlFwdArgs& args, cudaStream_t s, bool pdl);
// Segment geometry of the forward (backward = false) or backward scan on the
// current device: every segment of every chain resident at once.
SegGeom samu_scan_geom(int B, int L, int M, bool backward);
// Forward: maps (w read backwards in time), prefix, replay (forwards).
// pdl: launch as a programmatic dependent of the previous kernel on s.
cudaError_t launch_samu_fwd_maps(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                 cudaStream_t s, bool pdl);
cudaError_t launch_samu_fwd_prefix(const SamuScanFwdArgs& args, cudaStream_t s, bool pdl);
cudaError_t launch_samu_fwd_replay(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                   cudaStream_t s, bool pdl);
// Backward: maps (dy read forwards in time, 16-row boxes), prefix, main
// (backwards, 8-row boxes).
cudaError_t launch_samu_bwd_maps(const CUtensorMap& tm_dy, const CUtensorMap& tm_ctrl, const SamuScanBwdArgs& args,
                                 cudaStream_t s, bool pdl);
cudaError_t launch_samu_bwd_prefix(const SamuScanBwdArgs& args, cudaStream_t s, bool pdl);
cudaError_t launch_samu_bwd_main(const CUtensorMap& tm_dy, const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl,
                                 const SamuScanBwdArgs& args, cudaStream_t s, bool pdl);
cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s, bool pdl);
cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------------------
// RG-LRU
// ---------------------------------------------------------------------------
struct RglruScanFwdArgs {
    ScanGeom g;
    const float* alpha;
    const uint8_t* reset;
    const float* h0;        // [B,D] or null
    uint32_t* y;
    float* y32;
    float* hT;
    float* hsub;            // [B][CS][D]
    float2* agg;            // [B][CT][D] {a, b}
    uint32_t* flags;
    uint32_t* counter;
    uint32_t* status;
};

struct RglruScanBwdArgs {
    ScanGeom g;
    const float* alpha;
    const uint8_t* reset;
    const float* dhT;
    const float* hsub;
    void* dx;
    void* dlx;
    void* dla;
    int grad_fp32;
    float* dh0;
    float2* agg;
    float* rin;
    float* apart;           // [B*CT][D]
    uint32_t* flags;
    uint32_t* counter;
    uint32_t* status;
};

cudaError_t launch_rglru_scan_fwd(const CUtensorMap& tm_x, const CUtensorMap& tm_lx, const CUtensorMap& tm_la,
                                  const RglruScanFwdArgs& args, cudaStream_t s);
cudaError_t launch_rglru_scan_bwd(const CUtensorMap& tm_dy, const CUtensorMap& tm_x, const CUtensorMap& tm_lx,
                                  const CUtensorMap& tm_la, const RglruScanBwdArgs& args, cudaStream_t s);
cudaError_t launch_rglru_alpha(const float* apart, float* apart2, float* dalpha, int rows, int D,
                               cudaStream_t s);

}  // namespace lrs

// Kernel argument blocks, shared per-step device functions and launcher
// declarations of the CUDA library.
#pragma once

#include "common.cuh"
#include "layout.cuh"

namespace lrs {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Paired FP32 arithmetic.  Each lane of a scan warp owns the two adjacent
// modes m, m+1; their values travel as one pair {mode m, mode m+1} in a
// 64-bit register pair, and each arithmetic step on them is one paired
// instruction (PTX fma/mul/add/sub.rn.f32x2): per element exactly the IEEE
// round-to-nearest operation of the scalar form.
// ---------------------------------------------------------------------------
typedef unsigned long long f2x;

__device__ __forceinline__ f2x pk2(float lo, float hi) {
    f2x r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2x dup2(float v) { return pk2(v, v); }
__device__ __forceinline__ void up2(f2x v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2x fma2(f2x a, f2x b, f2x c) {
    f2x d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2x mul2(f2x a, f2x b) {
    f2x d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2x add2(f2x a, f2x b) {
    f2x d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2x sub2(f2x a, f2x b) {
    f2x d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// A BF16 pair word (low half mode m, high half mode m+1) as an FP32 pair;
// nbf2x gives the negated pair (sign bits flipped before widening).
__device__ __forceinline__ f2x bf2x(uint32_t w) {
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ f2x nbf2x(uint32_t w) { return bf2x(w ^ 0x80008000u); }
// An FP32 pair rounded to a BF16 pair word (round to nearest even).
__device__ __forceinline__ uint32_t x2bf(f2x v) {
    float a, b;
    up2(v, a, b);
    return f2_to_bf2(a, b);
}

// Complex values of the two modes: real-part pair and imaginary-part pair.
struct c2x {
    f2x re, im;
};

// Per-mode constants of the transition.  lambda_{t,m} = e^{-nu_m E_t} e^{i(theta_m + d_t)}
// (SAMU GPU page, section 05, transition equation) is evaluated as
//   lambda_{t,m} = lbar_m * delta_{t,m},  lbar_m = e^{-nu_m} e^{i theta_m},
//   delta_{t,m} = e^{-nu_m (E_t - 1)} (C_t + i S_t),
// which is the same number.  lbar_m is held as a double-float (hi + lo, formed
// once in FP64), so no per-mode rounding of e^{-nu}, cos theta or sin theta
// biases every step of a long chain; delta is close to 1 and formed per step
// in FP32 from E_t - 1 = expm1(c_t) and the shared C_t, S_t.
struct ModePair {
    f2x hr, hi, nhi, lr, li;   // lbar hi part (re, im, -im), lo part (re, im)
    f2x nu;
};

__device__ __forceinline__ ModePair load_modes(const float4* __restrict__ modes, const float* __restrict__ nu,
                                               int m) {
    const float4 v0 = modes[m], v1 = modes[m + 1];
    ModePair k;
    k.hr = pk2(v0.x, v1.x);
    k.hi = pk2(v0.y, v1.y);
    k.nhi = pk2(-v0.y, -v1.y);
    k.lr = pk2(v0.z, v1.z);
    k.li = pk2(v0.w, v1.w);
    k.nu = pk2(nu[m], nu[m + 1]);
    return k;
}

// lbar_m = e^{-nu_m} e^{i theta_m} in FP64, stored as the double-float
// {hi.re, hi.im, lo.re, lo.im} (hi the FP32 rounding, lo the FP32 rounding of
// the remainder) that samu_lambda2 consumes.
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

// lbar_m^K = e^{-K nu_m} e^{i K theta_m}, formed in FP64 (K theta_m is exact
// there, and the reduction of the phase, up to 2 pi K, is done in FP64 too) and
// stored as the same double-float: the closed-form transition of K
// consecutive tokens is lbar_m^K e^{-nu_m G} e^{i D} (G, D below).
__device__ __forceinline__ void mode_power_constants(const float* __restrict__ nu, const float* __restrict__ theta,
                                                     int M, int K, float4* __restrict__ out, int m) {
    if (m >= M) return;
    const double r = exp(-(double)K * (double)nu[m]);
    double sn, cs;
    sincos((double)K * (double)theta[m], &sn, &cs);
    const double re = r * cs, im = r * sn;
    const float hr = (float)re, hi = (float)im;
    out[m] = make_float4(hr, hi, (float)(re - (double)hr), (float)(im - (double)hi));
}

__device__ __forceinline__ ModePair zero_modes() {
    ModePair k;
    k.hr = k.hi = k.nhi = k.lr = k.li = k.nu = 0ull;
    return k;
}

// Per-token control word, written by the controller forward and staged into
// shared memory by TMA, each value duplicated so that it loads as a pair:
// {E-1, E-1, C, C}, {S, S, R, d} (two float4), R = -E for an ordinary token
// and R = +0 at a segment start (lambda = 0); E = e^c > 0, so the sign tells
// them apart.  It is the same for every lane, so the branches on it are
// warp-uniform.
struct Ctl2 {
    f2x e, c, s;   // E - 1, C, S
    f2x ne;        // -E (ordinary tokens)
    float rflag;   // R
};

__device__ __forceinline__ Ctl2 load_ctl(const float4* sc, int i) {
    const float4 a = sc[2 * i], b = sc[2 * i + 1];
    Ctl2 ct;
    ct.e = pk2(a.x, a.y);
    ct.c = pk2(a.z, a.w);
    ct.s = pk2(b.x, b.y);
    ct.ne = pk2(b.z, b.z);
    ct.rflag = b.z;
    return ct;
}

__device__ __forceinline__ bool is_reset_word(float r) { return r >= 0.f; }
__device__ __forceinline__ bool is_reset(const Ctl2& ct) { return is_reset_word(ct.rflag); }

// Bound on |nu (E - 1)| under which the degree-3 polynomial below is exact to
// < 2.5e-9 relative (the truncation term x^4/24, about 0.04 FP32 ulp),
// checked once per warp and sub-chunk.
constexpr float kPolyBound = 1.0f / 64.0f;

// lambda of both modes for a token that is not a reset:
// lbar * e^{-nu (E-1)} (C + iS), with its negated imaginary part.  FAST:
// e^{-x} by its degree-3 Taylor polynomial (valid for |x| < kPolyBound; its
// rounding errors carry no per-mode bias); otherwise ex2.approx, whose ~1e-7
// error matters little for the short-memory modes that need it.  Every pass
// that needs lambda calls this, so the forward and the backward rebuild the
// same bits.
struct Lam2 {
    f2x re, im, nim;
};

template <bool FAST>
__device__ __forceinline__ Lam2 samu_lambda2(const ModePair& k, const Ctl2& ct) {
    const f2x x = mul2(k.nu, ct.e);   // nu (E - 1)
    f2x q;                            // e^{-x}
    if (FAST) {
        q = fma2(x, fma2(x, fma2(x, dup2(-1.0f / 6.0f), dup2(0.5f)), dup2(-1.0f)), dup2(1.0f));
    } else {
        float a, b;
        up2(x, a, b);
        q = pk2(ex2_approx(__fmul_rn(-a, kLog2e)), ex2_approx(__fmul_rn(-b, kLog2e)));
    }
    const f2x dr = mul2(q, ct.c);
    const f2x di = mul2(q, ct.s);
    Lam2 l;
    l.re = fma2(k.hr, dr, fma2(k.nhi, di, k.lr));
    l.im = fma2(k.hr, di, fma2(k.hi, dr, k.li));
    l.nim = sub2(0ull, l.im);
    return l;
}

// lambda z
__device__ __forceinline__ c2x cmul2(const Lam2& l, const c2x& z) {
    c2x r;
    r.re = fma2(l.re, z.re, mul2(l.nim, z.im));
    r.im = fma2(l.re, z.im, mul2(l.im, z.re));
    return r;
}

// conj(lambda) z
__device__ __forceinline__ c2x cmulc2(const Lam2& l, const c2x& z) {
    c2x r;
    r.re = fma2(l.re, z.re, mul2(l.im, z.im));
    r.im = fma2(l.re, z.im, mul2(l.nim, z.re));
    return r;
}

// acc + P b, given -Im b
__device__ __forceinline__ c2x cfma2(const c2x& P, const c2x& bb, f2x nb_im, const c2x& acc) {
    c2x r;
    r.re = fma2(P.re, bb.re, fma2(P.im, nb_im, acc.re));
    r.im = fma2(P.re, bb.im, fma2(P.im, bb.re, acc.im));
    return r;
}

// Forward scan over segments: segment maps, chain prefix, replay.  w and
// the control words reach the kernels through TMA tensor maps (16-token
// boxes); everything indexed by segment is [B][NS][M] (per mode).
struct SamuScanFwdArgs {
    SegGeom g;
    const float4* items;    // [B][items per row] the controller's item records (per-item plan)
    const float4* modes;    // [2][M] lbar, lbar^16 (hi/lo)
    const float* nu;
    int closed_form;        // full items without a reset: closed-form transition
    const float* h0;        // [B,M,2] or null
    uint32_t* y;            // BF16 pairs of y
    float* y32;             // optional
    float* hT;              // [B,M,2]
    float2* hsub;           // [B][CS][M] the state every 8 tokens
    float4* smap;           // [B][NS][M] segment maps
    float4* cmap;           // [B][NC][M] CTA maps (four consecutive segments)
    uint32_t* status;       // cleared by the controller forward
};

// Backward scan over segments: adjoint segment maps, reverse chain prefix,
// reverse replay.  sent holds the adjoint arriving at each segment's last
// token from later tokens.
struct SamuScanBwdArgs {
    SegGeom g;
    const float4* items;    // [B][items per row] the forward's item records (per-item plan, per-segment kind)
    const float4* modes;    // [2][M] lbar, lbar^16 (hi/lo)
    const float* nu;
    int closed_form;        // full items without a reset: closed-form transition
    const float* dhT;       // [B,M,2] or null
    const float2* hsub;     // [B][CS][M] (the forward's sub-chunk entry states)
    void* dw;               // BF16 pairs or FP32
    int grad_fp32;
    float* dh0;             // [B,M,2]
    float4* smap;           // [B][NS][M] adjoint segment maps
    float4* cmap;           // [B][NC][M] adjoint CTA maps
    float2* kpart;          // [B*L][n_groups] {sum Im kappa, sum -nu Re kappa}
    float2* numod;          // [B][NS][M] {dnu, dtheta} per segment
    uint32_t* status;
};

// Controller-backward streaming geometry: every CTA owns a contiguous run of
// `stage_tok`-token stages of x_sel (and of dx_sel), staged through a ring of
// `ring` shared-memory slots by 1-D bulk copies; a producer warp, a reducer
// warp and `consumers` warps of 32 threads, each thread owning 8 channels.
struct CtrlGeom {
    int stage_tok;          // tokens per stage (16, or 8 when 16 rows exceed 72 KB)
    int ring;               // slots (2 to 8, as many as fit)
    int chunks;             // 8-channel chunks per consumer lane (1, or 2 for D > 3584)
    int consumers;          // consumer warps
    int threads;            // 32 * (2 + consumers)
    int smem;               // dynamic shared memory bytes
    int n_ctas;             // streaming CTAs
    long long n_stages;     // ceil(B*L / stage_tok)
    int max_cta_tok;        // tokens of the longest CTA range (scalar buffer)
};

CtrlGeom samu_ctrl_geom(long long BL, int D);

struct SamuCtrlBwdArgs {
    long long BL;
    int D, n_groups;
    CtrlGeom cg;
    const uint4* x;         // BF16 x_sel as 16-byte vectors
    const float2* kpart;
    const float* p;
    const float* r;
    const float4* ctrl;     // [B*L][2] control words
    const float* wh;        // [2][D+1]
    const float* misc;
    const float2* numod;    // [numod_rows][M] per-segment (dnu, dtheta)
    int numod_rows;
    void* dx;               // BF16 or FP32
    int grad_fp32;
    float* dwh_part;        // [cg.n_ctas][2][ns], ns = ctrl_half_stride(D)
    float2* amp_part;       // [cg.n_ctas]
    float2* dot_part;       // [cg.n_ctas] w_hat . (partial row), phi and r
    float* dnu;
    float* dtheta;
    uint32_t* status;
};

struct SamuParamArgs {
    int D;
    int n_rows;             // rows of dwh_part / amp_part / dot_part (controller-backward CTAs)
    const float* dwh_part;  // [n_rows][2][ns]
    const float2* amp_part;
    const float2* dot_part;
    const float* wh;
    const float* misc;
    float* dw_phi;
    float* dw_r;
    float* da_phi;
    float* da_r;
};

struct SamuCtrlFwdArgs {
    long long BL;
    int B, L;
    int D;
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
    float4* ctrl;                  // [B*L][2] {E-1, E-1, C, C}, {S, S, R, d}
    float4* items;                 // [B][items per row] item records (samu_items_per_row)
    float* wh;                     // [2][D+1]
    float* misc;
    float4* modes;                 // [2][M] lbar, lbar^16 hi/lo
    uint32_t* status;
};

cudaError_t launch_samu_ctrl_fwd(const SamuCtrlFwdArgs& args, cudaStream_t s, bool pdl);
// Segment geometry of the forward (backward = false) or backward scan on the
// current device: every segment of every chain resident at once.
SegGeom samu_scan_geom(int B, int L, int M, bool backward);
// Forward: maps (w read backwards in time; the last CTA of each chain folds
// the chain's CTA maps into entry states), replay (forwards).
// pdl: launch as a programmatic dependent of the previous kernel on s.
cudaError_t launch_samu_fwd_maps(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                 cudaStream_t s, bool pdl);
cudaError_t launch_samu_fwd_replay(const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl, const SamuScanFwdArgs& args,
                                   cudaStream_t s, bool pdl);
// Backward: maps (dy read forwards in time, 16-row boxes; the last CTA of
// each chain folds the adjoint CTA maps), main (backwards, 8-row boxes).
cudaError_t launch_samu_bwd_maps(const CUtensorMap& tm_dy, const CUtensorMap& tm_ctrl, const SamuScanBwdArgs& args,
                                 cudaStream_t s, bool pdl);
// tm_dw: an 8-row map over dw (BF16 gradients; used when M is a multiple of
// 64, the rows are then written by TMA from shared memory).
cudaError_t launch_samu_bwd_main(const CUtensorMap& tm_dy, const CUtensorMap& tm_w, const CUtensorMap& tm_ctrl,
                                 const CUtensorMap& tm_dw, const SamuScanBwdArgs& args, cudaStream_t s, bool pdl);
// Controller backward (with the (dnu, dtheta) reductions), then the
// reductions of the unit-direction and amplitude gradients.
cudaError_t launch_samu_ctrl_bwd(const SamuCtrlBwdArgs& args, cudaStream_t s, bool pdl);
cudaError_t launch_samu_params(const SamuParamArgs& args, cudaStream_t s, bool pdl);
// The status word of samu_forward_noalloc's fixed array in the current
// context (its address looked up as that entry point does).
int noalloc_status_word(uint32_t** out);

// ---------------------------------------------------------------------------
// SAMU single-token decode step
// ---------------------------------------------------------------------------
struct SamuDecodePrepArgs {
    int D;
    const float* nu;
    const float* theta;
    const float* w_phi;
    const float* w_r;
    const float* a_phi;
    const float* a_r;
    float* params;          // samu_decode_params_floats(D) floats, 16-byte aligned
};

struct SamuDecodeStepArgs {
    long long B;
    int D;
    const uint16_t* x;      // [B][D] BF16
    const uint16_t* w;      // [B][D] BF16
    const float* state_in;  // [B][M][2]
    float* state_out;       // [B][M][2] (may be state_in)
    const uint8_t* reset;   // [B] or null
    const float* params;
    uint16_t* y;            // [B][D] BF16
    float* y32;             // [B][D] or null
    int parts;              // CTAs per sequence (set by the launcher)
};

size_t samu_decode_params_floats(int D);
cudaError_t launch_samu_decode_prepare(const SamuDecodePrepArgs& args, cudaStream_t s);
cudaError_t launch_samu_decode_step(const SamuDecodeStepArgs& args, cudaStream_t s);

// ---------------------------------------------------------------------------
// RG-LRU
// ---------------------------------------------------------------------------
// With projected gates (logit modes 1 and 2, the "PL" variants) l^x and l^a are FP32
// [B,L,D] (x W without the bias) and bx, ba the biases added on reading.
struct RglruScanFwdArgs {
    ScanGeom g;
    const float* alpha;
    const float* bx;        // [D], PL only
    const float* ba;
    const uint8_t* wimg;    // logits mode 2: the groups' weight images
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

// PL variant: the token's gradients go to gparts [B*L][16][6][dk] BF16 as
// leading BF16 parts and BF16 remainders (v = hi + lo to 16 significant
// bits): parts 0/1 dl^x, 2/3 dl^a, 4/5 dx through the write term; bxpart /
// bapart receive the per-tile sums of the gate gradients (the bias
// gradients' partials).
struct RglruScanBwdArgs {
    ScanGeom g;
    const float* alpha;
    const float* bx;
    const float* ba;
    const uint8_t* reset;
    const float* dhT;
    const float* hsub;
    void* dx;
    void* dlx;
    void* dla;
    uint32_t* gparts;       // PL only
    int dk;                 // PL only: D / 16
    const uint8_t* wimg;    // logits mode 2: the groups' weight images
    float* bxpart;          // [B*CT][D]
    float* bapart;
    int grad_fp32;
    float* dh0;
    float2* agg;
    float* rin;
    float* apart;           // [B*CT][D]
    uint32_t* flags;
    uint32_t* counter;
    uint32_t* status;
};

// logits: 0 raw BF16 l^x, l^a; 1 FP32 products x W (+ biases); 2 products
// formed in the kernel on the tensor cores from args.wimg (+ biases); for 2,
// tm_x must be the 128-byte-swizzled map of x and tm_lx, tm_la are unused.
cudaError_t launch_rglru_scan_fwd(const CUtensorMap& tm_x, const CUtensorMap& tm_lx, const CUtensorMap& tm_la,
                                  const RglruScanFwdArgs& args, cudaStream_t s, int logits = 0);
// The groups' weight images for logits mode 2: per 64-channel group and gate the
// [64 outputs][64 inputs] BF16 matrix (zero outside the diagonal blocks;
// dk = D/16 must divide 64) in the K-major 128-byte-swizzled layout.
cudaError_t launch_rglru_proj_wimg(const void* w_x, const void* w_a, void* wimg, int D, cudaStream_t s);
// logits as for the forward: 0 raw BF16 l^x, l^a (dx, dl^x, dl^a out); 1 FP32
// products x W, 2 products formed in the kernel from args.wimg (both: the
// projected gradient parts out; for 2, tm_x is the 128-byte-swizzled map of x
// and tm_lx, tm_la are unused).
cudaError_t launch_rglru_scan_bwd(const CUtensorMap& tm_dy, const CUtensorMap& tm_x, const CUtensorMap& tm_lx,
                                  const CUtensorMap& tm_la, const RglruScanBwdArgs& args, cudaStream_t s,
                                  int logits = 0);
cudaError_t launch_rglru_alpha(const float* apart, float* apart2, float* dalpha, int rows, int D,
                               cudaStream_t s);
// The gate projections' contractions on the tensor cores (proj_gemm.cu):
// operand images of W_x, W_a (logits) and of the packed Wcat (dx); the FP32
// logits x W_q of both gates; dx from the gradient parts; dW_x, dW_a from the
// gradient parts and x (token splits added in a fixed order).  status: the
// call's device status word (bounded waits).
cudaError_t launch_proj_pack(const void* w_x, const void* w_a, void* wt, void* wc, const ProjDims& d, cudaStream_t s);
cudaError_t launch_proj_logits(const void* x, const void* wt, float* lx, float* la, int D, const ProjDims& d,
                               uint32_t* status, cudaStream_t s, bool pdl);
cudaError_t launch_proj_dx(const void* gparts, const void* wc, void* dx, bool dx_fp32, int D, const ProjDims& d,
                           uint32_t* status, cudaStream_t s, bool pdl);
int proj_dw_splits(const ProjDims& d);
cudaError_t launch_proj_dw(const void* gparts, const void* x, float* part, float* dw_x, float* dw_a, int D,
                           const ProjDims& d, uint32_t* status, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------------------
// RecurrentBlock around the SAMU mixer (block_gemm.cu, block_elem.cu).
// ---------------------------------------------------------------------------
// Operand layouts of the dense contraction C(m, n) = sum_k A(m, k) B(n, k):
//   NT: A [M][K], B [N][K] (forward, y = x W^T);
//   NN: A [M][K], B [K][N] (dX, dx = dy W);
//   TN: A [K][M], B [K][N] (dW = dy^T x, K = tokens, split into FP32 partials).
enum BgLayoutKind { kBgNT = 0, kBgNN = 1, kBgTN = 2 };
// Fused epilogues (see block_gemm.cu).
enum BgEpiKind { kEpiStore = 0, kEpiResid = 1, kEpiGlu = 2, kEpiGluBwd = 3, kEpiJoinBwd = 4, kEpiF32 = 5 };
constexpr int kBlockGemmSplitsMax = 16;
constexpr int kBlockSmsBound = 256;   // SMs assumed when sizing the split partials (GB300: 152)

struct BlockGemmArgs {
    int layout, epi;
    int M, N, K;                 // glu: N = F hidden units (the B rows f and F + f pair up)
    int m_tiles, n_tiles, splits, ksteps, n_items;   // filled by launch_block_gemm (splits: TN only, in)
    int n_pairs;                 // filled: items of the two-CTA clusters (row-block pairs)
    uint16_t* out;  int ldo;     // BF16 output (store, resid: C; glu: q; glu_bwd: [da | db]; join_bwd: dy_mixer)
    const uint16_t* r; int ldr;  // resid: the residual added to C
    uint16_t* out2; int ld2;     // glu: [a | b]; join_bwd: dg (the gate half of [dg | dv])
    const uint16_t* e0; int lde0;   // glu_bwd: [a | b]; join_bwd: [g | v]
    const uint16_t* e1; int lde1;   // join_bwd: y_mixer
    int F;                       // glu, glu_bwd: offset of the b (db) half
    float* part;                 // f32: [splits][M][N]
    uint32_t* status;
};

// Token splits of a TN contraction of an M x N weight gradient over K tokens
// on `sms` SMs (block_gemm_sms(): this device's, capped at kBlockSmsBound),
// and the largest count any SM count up to kBlockSmsBound can choose (the
// split partials' workspace is sized for it).
int block_gemm_sms();
int block_gemm_splits(int M, int N, long long K, int sms);
int block_gemm_splits_bound(int M, int N, long long K);
cudaError_t launch_block_gemm(const BlockGemmArgs& a, const void* A, const void* B, cudaStream_t s, bool pdl);
// out[i] = sum_{p < parts} part[p * stride + i] in order, i < n.
cudaError_t launch_sum_parts(const float* part, long long stride, int parts, long long n, float* out, cudaStream_t s,
                             bool pdl);
int block_norm_bwd_ctas(long long rows);
int block_conv_parts(int B, int L);
cudaError_t launch_rmsnorm_fwd(const void* x, const float* gamma, void* h, float* rstd, long long rows, int W,
                               uint32_t* status_clear, cudaStream_t s, bool pdl);
cudaError_t launch_rmsnorm_bwd(const void* x, const float* gamma, const float* rstd, const void* dh, const void* dres,
                               void* dx, float* dgamma_part, long long rows, int W, uint32_t* status_clear,
                               cudaStream_t s, bool pdl);
cudaError_t launch_conv_fwd(const void* gv, const float* k, const float* kb, const uint8_t* reset, void* u, int B,
                            int L, int D, cudaStream_t s, bool pdl);
cudaError_t launch_conv_bwd(const void* gv, const float* k, const uint8_t* reset, const void* dxs, const void* dwm,
                            void* dgv, float* part, int B, int L, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl);
cudaError_t launch_join_fwd(const void* gv, const void* ym, void* j, long long BL, int D, uint32_t* status,
                            const uint32_t* mixer_status, cudaStream_t s, bool pdl);

}  // namespace lrs

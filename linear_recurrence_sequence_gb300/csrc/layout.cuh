// Workspace layouts and launch geometry shared by the host entry points and
// the kernels.  All offsets are in bytes from the start of the caller's
// `saved` or `scratch` buffer and are 256-byte aligned.
#pragma once

#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace lrs {

constexpr size_t kAlign = 256;
constexpr int kCtrlRowsMax = 608;    // partial-sum rows of the controller backward (CTAs)
constexpr int kReduceGroups = 64;     // first-stage groups of the RG-LRU per-tile alpha partials
constexpr int kStatusBlock = 64;      // bytes at the start of scratch: status word + arrival counter

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Floats per half (phi, r) of a controller-backward partial row: D + 1
// rounded up to a multiple of 4, so that rows are float4 arrays.
__host__ __device__ inline int ctrl_half_stride(int D) { return (D + 1 + 3) & ~3; }

// Tile shapes.  RG-LRU: a tile is 128 tokens of one chain, one 16-token
// sub-chunk per warp.
constexpr int kRgWarps = 8;                        // RG-LRU: 8 warps
constexpr int kRgTile = kRgWarps * kSub;           // 128 tokens

// Geometry of one chunked scan over [B, L, lanes] (lanes = M modes for SAMU,
// D channels for RG-LRU).  A chain is one (batch row, group of kGroup lanes);
// its tiles are `tile` consecutive tokens.
struct ScanGeom {
    int B, L, lanes;
    int tile;              // tokens per tile
    int subs;              // 16-token sub-chunks per tile
    int n_groups;          // ceil(lanes / kGroup)
    int n_chains;          // B * n_groups
    int CT;                // tiles per chain, ceil(L / tile)
    int CS;                // entry-state slots per batch row (slot = t / 16, with slack)
    long long n_tiles;     // n_chains * CT
};

inline ScanGeom make_geom(int B, int L, int lanes, int tile) {
    ScanGeom g;
    g.B = B;
    g.L = L;
    g.lanes = lanes;
    g.tile = tile;
    g.subs = tile / kSub;
    g.n_groups = (lanes + kGroup - 1) / kGroup;
    g.n_chains = B * g.n_groups;
    g.CT = (L + tile - 1) / tile;
    g.CS = (L + kSub - 1) / kSub + g.subs + 1;
    g.n_tiles = (long long)g.n_chains * g.CT;
    return g;
}

// SAMU segments.  Every chain is cut into NS segments of `seg` tokens (a
// multiple of 16; the last one ends at L), one per warp, with NS chosen so
// that all segments of all chains run at once on the resident warps.  The
// scratch arrays indexed by segment are sized for the most segments any
// device can ask for: at least kSegMinTok tokens each and at most
// kMaxSegWarps segments in all.
constexpr int kSegMinTok = kSub;
constexpr int kHalf = kSub / 2;     // tokens between SAMU state checkpoints
constexpr int kMapRows = 16;        // tokens per staged item of the SAMU maps and replay kernels
constexpr int kMapSlots = 2;        // items in flight per warp there
static_assert(kMapRows % kHalf == 0, "items start on state checkpoints");
constexpr long long kMaxSegWarps = 16384;

struct SegGeom {
    int B, L, M;
    int n_groups, n_chains;
    int seg;               // tokens per segment
    int NS;                // segments per chain (a multiple of kSegPerCta)
    int NC;                // CTAs per chain, NS / kSegPerCta
    int NSmax;             // bound on NS for this (B, L, M) on any device
    int CS;                // state checkpoints per batch row (slot = t / 8)
};

// Segments (warps) per CTA of the scan engine; the segments of a CTA are
// consecutive segments of one chain.
constexpr int kSegPerCta = 8;

inline int round_up16(long long v) { return (int)((v + kSub - 1) / kSub * kSub); }
inline int round_up_cta(long long v) { return (int)((v + kSegPerCta - 1) / kSegPerCta * kSegPerCta); }

// seg_min: the shortest segment any device may use for this problem.
inline int seg_min_tokens(int L, int n_chains) {
    const long long need = ((long long)L * n_chains + kMaxSegWarps - 1) / kMaxSegWarps;
    const int s = round_up16(need);
    return s < kSegMinTok ? kSegMinTok : s;
}

// Segment geometry for `warps` resident warps (warps <= 0: the bound only).
// Segments past the end of the sequence (NS is rounded up to whole CTAs) are
// empty.
inline SegGeom samu_seg_geom(int B, int L, int M, long long warps) {
    SegGeom g;
    g.B = B;
    g.L = L;
    g.M = M;
    g.n_groups = (M + kGroup - 1) / kGroup;
    g.n_chains = B * g.n_groups;
    const int smin = seg_min_tokens(L, g.n_chains);
    g.NSmax = round_up_cta((L + smin - 1) / smin);
    int seg = smin;
    if (warps > 0) {
        // whole CTAs of segments per chain that fit at once
        const long long per_chain = warps / g.n_chains / kSegPerCta * kSegPerCta;
        const long long parts = per_chain >= kSegPerCta ? per_chain : kSegPerCta;
        seg = round_up16(((long long)L + parts - 1) / parts);
        if (seg < smin) seg = smin;
    }
    g.seg = seg;
    g.NS = round_up_cta((L + seg - 1) / seg);
    g.NC = g.NS / kSegPerCta;
    g.CS = (L + kHalf - 1) / kHalf + 1;
    return g;
}

// ---------------------------------------------------------------------------
// SAMU
// ---------------------------------------------------------------------------
// misc floats: 0 = tanh(a_phi)/sqrt(M), 1 = tanh(a_r)/sqrt(M), 2 = ||w_phi||,
// 3 = ||w_r||, 4 = tanh(a_phi), 5 = tanh(a_r), 6 = 1/sqrt(M)
constexpr int kMiscFloats = 16;

struct SamuSaved {
    size_t p, r, ctrl, items, hsub, wh, misc, modes, total;
};

// Per-item records of the control words: one float4 per kMapRows-token item
// of each batch row (items start at t = 0, 16, ... of the row):
// {G = sum (E - 1), cos D, sin D with D = sum d, v}, v = max |E - 1| over the
// item's tokens when the item is full and holds no reset, else
// -(max |E - 1|) - 1.
__host__ __device__ inline int samu_items_per_row(int L) { return (L + kMapRows - 1) / kMapRows; }

inline SamuSaved samu_saved_layout(int B, int L, int D) {
    const int M = D / 2;
    const SegGeom g = samu_seg_geom(B, L, M, 0);
    const size_t BL = (size_t)B * L;
    SamuSaved s;
    size_t o = 0;
    s.p = o;      o = align_up(o + BL * 4);                          // p_t
    s.r = o;      o = align_up(o + BL * 4);                          // r_t
    s.ctrl = o;   o = align_up(o + BL * 32);                         // {E-1, E-1, C, C}, {S, S, R, d}, R = -E or +0 at a reset
    s.items = o;  o = align_up(o + (size_t)B * samu_items_per_row(L) * 16);   // item records
    s.hsub = o;   o = align_up(o + (size_t)B * g.CS * M * 8);        // state every 8 tokens
    s.wh = o;     o = align_up(o + (size_t)2 * (D + 1) * 4);         // unit directions
    s.misc = o;   o = align_up(o + kMiscFloats * 4);
    s.modes = o;  o = align_up(o + (size_t)M * 32);                  // [2][M]: lbar, then lbar^16, hi/lo per mode
    s.total = o;
    return s;
}

struct SamuScratch {
    size_t status, smap, cmap, kpart, numod, dwh_part, amp_part, dot_part, total;
    size_t zero_bytes;     // status block: cleared at the start of a backward call
};

inline SamuScratch samu_scratch_layout(int B, int L, int D) {
    const int M = D / 2;
    const SegGeom g = samu_seg_geom(B, L, M, 0);
    const size_t BL = (size_t)B * L;
    const size_t rows = (size_t)B * g.NSmax * M;
    SamuScratch s;
    size_t o = 0;
    s.status = o;   o += kStatusBlock;
    s.zero_bytes = o;
    o = align_up(o);
    const size_t crows = (size_t)B * (g.NSmax / kSegPerCta) * M;
    s.smap = o;     o = align_up(o + rows * 16);                      // segment maps
    s.cmap = o;     o = align_up(o + crows * 16);                     // CTA maps (8 segments)
    s.kpart = o;    o = align_up(o + BL * g.n_groups * 8);            // per-token controller partials
    s.numod = o;    o = align_up(o + rows * 8);                       // per-segment (dnu, dtheta)
    const size_t prow = (size_t)2 * ctrl_half_stride(D) * 4;              // one partial row, bytes
    s.dwh_part = o; o = align_up(o + (size_t)kCtrlRowsMax * prow);        // one row per CTA
    s.amp_part = o; o = align_up(o + (size_t)kCtrlRowsMax * 8);
    s.dot_part = o; o = align_up(o + (size_t)kCtrlRowsMax * 8);           // w_hat . (partial row)
    s.total = o;
    return s;
}

// ---------------------------------------------------------------------------
// RG-LRU
// ---------------------------------------------------------------------------
struct RglruSaved {
    size_t hsub, total;
};

inline RglruSaved rglru_saved_layout(int B, int L, int D) {
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    RglruSaved s;
    size_t o = 0;
    s.hsub = o; o = align_up(o + (size_t)B * g.CS * D * 4);
    s.total = o;
    return s;
}

struct RglruScratch {
    size_t status, flags, agg, rin, apart, apart2, total, memset_bytes;
};

inline RglruScratch rglru_scratch_layout(int B, int L, int D) {
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    RglruScratch s;
    size_t o = 0;
    s.status = o;  o += kStatusBlock;
    s.flags = o;   o = align_up(o + (size_t)g.n_tiles * 4);
    s.memset_bytes = o;
    s.agg = o;     o = align_up(o + (size_t)B * g.CT * D * 8);
    s.rin = o;     o = align_up(o + (size_t)B * g.CT * D * 4);
    s.apart = o;   o = align_up(o + (size_t)B * g.CT * D * 4);
    s.apart2 = o;  o = align_up(o + (size_t)kReduceGroups * D * 4);
    s.total = o;
    return s;
}

// RG-LRU with the block-diagonal gate projections.  Sizes of the
// tensor-core contractions: dk = D/16 channels per block, NP = dk rounded up
// to 16 (the N tile), kp = dk and kp6 = 6 dk rounded up to 64 (the K slices),
// dw_rows = 4 dk rounded up to 128 (the M tiles of the weight gradient).
constexpr int kProjBlocks = 16;                      // diagonal blocks of each gate projection
constexpr int kProjDwSplitsMax = 16;                 // token splits of the weight-gradient contraction

struct ProjDims {
    int BL, dk, NP, kp, kp6, dw_rows;
};

inline ProjDims proj_dims(int B, int L, int D) {
    ProjDims d;
    d.BL = B * L;
    d.dk = D / kProjBlocks;
    d.NP = (d.dk + 15) / 16 * 16;
    d.kp = (d.dk + 63) / 64 * 64;
    d.kp6 = (6 * d.dk + 63) / 64 * 64;
    d.dw_rows = (4 * d.dk + 127) / 128 * 128;
    return d;
}

// The scan's scratch, then the FP32 products x W of both gates, the six BF16
// gradient parts per token and block ([B*L][16][6][dk]), the packed operand
// images of the logits and dx contractions, the weight gradient's per-split
// partial products, the bias-gradient partials and the weight images of the
// in-kernel logits.
struct RglruProjScratch {
    RglruScratch scan;
    size_t lx, la, gparts, wt, wc, dwpart, wimg, bxpart, bapart, total;
};

inline RglruProjScratch rglru_proj_scratch_layout(int B, int L, int D) {
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    const ProjDims pd = proj_dims(B, L, D);
    RglruProjScratch s;
    s.scan = rglru_scratch_layout(B, L, D);
    const size_t bld = (size_t)B * L * D;
    size_t o = s.scan.total;
    s.lx = o;      o = align_up(o + bld * 4);
    s.la = o;      o = align_up(o + bld * 4);
    s.gparts = o;  o = align_up(o + bld * 6 * 2);
    s.wt = o;      o = align_up(o + (size_t)kProjBlocks * 2 * pd.NP * pd.kp * 2);
    s.wc = o;      o = align_up(o + (size_t)kProjBlocks * pd.NP * pd.kp6 * 2);
    s.dwpart = o;  o = align_up(o + (size_t)kProjDwSplitsMax * kProjBlocks * pd.dw_rows * pd.NP * 4);
    s.wimg = o;    o = align_up(o + (size_t)(D / 64) * 2 * 64 * 64 * 2);   // in-kernel logits: weight images
    s.bxpart = o;  o = align_up(o + (size_t)B * g.CT * D * 4);
    s.bapart = o;  o = align_up(o + (size_t)B * g.CT * D * 4);
    s.total = o;
    return s;
}

// ---------------------------------------------------------------------------
// RecurrentBlock around the SAMU mixer: widths Dm (residual stream), D (the
// mixer), F = 3 Dm (MLP hidden units).
// ---------------------------------------------------------------------------
constexpr int kBlockMlpRatio = 3;

// Forward -> backward: the mixer's own saved buffer (SAMU or the RG-LRU with
// its gate projections: mixer_saved bytes), then the block's BF16
// activations and the two norms' FP32 reciprocal RMS per token.
struct BlockSaved {
    size_t mixer, h1, rstd1, gv, u, ym, j, r1, rstd2, h2, ab, q, total;
};

inline BlockSaved block_saved_layout(int B, int L, int Dm, int D, size_t mixer_saved) {
    const size_t BL = (size_t)B * L, F = (size_t)kBlockMlpRatio * Dm;
    BlockSaved s;
    size_t o = 0;
    s.mixer = o;  o = align_up(o + mixer_saved);
    s.h1 = o;     o = align_up(o + BL * Dm * 2);
    s.rstd1 = o;  o = align_up(o + BL * 4);
    s.gv = o;     o = align_up(o + BL * 2 * D * 2);     // [g | v]
    s.u = o;      o = align_up(o + BL * D * 2);
    s.ym = o;     o = align_up(o + BL * D * 2);
    s.j = o;      o = align_up(o + BL * D * 2);
    s.r1 = o;     o = align_up(o + BL * Dm * 2);
    s.rstd2 = o;  o = align_up(o + BL * 4);
    s.h2 = o;     o = align_up(o + BL * Dm * 2);
    s.ab = o;     o = align_up(o + BL * 2 * F * 2);     // [a | b]
    s.q = o;      o = align_up(o + BL * F * 2);
    s.total = o;
    return s;
}

// Scratch: the block's status word, the mixer's scratch, the BF16 gradients
// between layers, the weight-gradient split partials (shared by the four
// weight contractions, one after another), the norm and convolution partials.
struct BlockScratch {
    size_t mixer, dab, dh2, dr1, dym, dgv, dxs, dwm, dh1, wpart, npart, cpart, total;
};

inline BlockScratch block_scratch_layout(int B, int L, int Dm, int D, size_t mixer_scratch, size_t wpart_floats,
                                         size_t npart_floats, size_t cpart_floats) {
    const size_t BL = (size_t)B * L, F = (size_t)kBlockMlpRatio * Dm;
    BlockScratch s;
    size_t o = kAlign;   // [0, kAlign): the block's status word
    s.mixer = o;  o = align_up(o + mixer_scratch);
    s.dab = o;    o = align_up(o + BL * 2 * F * 2);
    s.dh2 = o;    o = align_up(o + BL * Dm * 2);
    s.dr1 = o;    o = align_up(o + BL * Dm * 2);
    s.dym = o;    o = align_up(o + BL * D * 2);
    s.dgv = o;    o = align_up(o + BL * 2 * D * 2);
    s.dxs = o;    o = align_up(o + BL * D * 2);
    s.dwm = o;    o = align_up(o + BL * D * 2);
    s.dh1 = o;    o = align_up(o + BL * Dm * 2);
    s.wpart = o;  o = align_up(o + wpart_floats * 4);
    s.npart = o;  o = align_up(o + npart_floats * 4);
    s.cpart = o;  o = align_up(o + cpart_floats * 4);
    s.total = o;
    return s;
}

}  // namespace lrs

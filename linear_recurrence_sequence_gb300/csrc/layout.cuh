// Workspace layouts and launch geometry shared by the host entry points and
// the kernels.  All offsets are in bytes from the start of the caller's
// `saved` or `scratch` buffer and are 256-byte aligned.
#pragma once

#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace lrs {

constexpr size_t kAlign = 256;
constexpr int kCtrlBwdCtas = 304;     // fixed grid of the controller backward (2 x 152 SMs)
constexpr int kReduceGroups = 64;     // first-stage groups of the per-tile parameter partials
constexpr int kStatusBlock = 64;      // bytes at the start of scratch: status word + tile counter

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Geometry of one chunked scan over [B, L, lanes] (lanes = M modes for SAMU,
// D channels for RG-LRU).  A chain is one (batch row, group of kGroup lanes);
// its tiles are kTile consecutive tokens.
struct ScanGeom {
    int B, L, lanes;
    int n_groups;          // ceil(lanes / kGroup)
    int n_chains;          // B * n_groups
    int CT;                // tiles per chain, ceil(L / kTile)
    int CS;                // entry-state slots per batch row: one per sub-chunk, + 1
    long long n_tiles;     // n_chains * CT
};

inline ScanGeom make_geom(int B, int L, int lanes) {
    ScanGeom g;
    g.B = B;
    g.L = L;
    g.lanes = lanes;
    g.n_groups = (lanes + kGroup - 1) / kGroup;
    g.n_chains = B * g.n_groups;
    g.CT = (L + kTile - 1) / kTile;
    g.CS = g.CT * kScanWarps + 1;
    g.n_tiles = (long long)g.n_chains * g.CT;
    return g;
}

// ---------------------------------------------------------------------------
// SAMU
// ---------------------------------------------------------------------------
// misc floats: 0 = tanh(a_phi)/sqrt(M), 1 = tanh(a_r)/sqrt(M), 2 = ||w_phi||,
// 3 = ||w_r||, 4 = tanh(a_phi), 5 = tanh(a_r), 6 = 1/sqrt(M)
constexpr int kMiscFloats = 16;

struct SamuSaved {
    size_t p, r, ctrl, hsub, wh, misc, modes, total;
};

inline SamuSaved samu_saved_layout(int B, int L, int D) {
    const int M = D / 2;
    const ScanGeom g = make_geom(B, L, M);
    const size_t BL = (size_t)B * L;
    SamuSaved s;
    size_t o = 0;
    s.p = o;      o = align_up(o + BL * 4);                          // p_t
    s.r = o;      o = align_up(o + BL * 4);                          // r_t
    s.ctrl = o;   o = align_up(o + BL * 16);                         // {E-1, C, S, reset}
    s.hsub = o;   o = align_up(o + (size_t)B * g.CS * M * 8);        // sub-chunk entry states
    s.wh = o;     o = align_up(o + (size_t)2 * (D + 1) * 4);         // unit directions
    s.misc = o;   o = align_up(o + kMiscFloats * 4);
    s.modes = o;  o = align_up(o + (size_t)M * 16);                  // lbar hi/lo per mode
    s.total = o;
    return s;
}

struct SamuScratch {
    size_t status, flags, agg, rin, kpart, numod, numod2, dwh_part, amp_part, dwh, total;
    size_t memset_bytes;   // bytes cleared at the start of each call: status block + flags
};

inline SamuScratch samu_scratch_layout(int B, int L, int D) {
    const int M = D / 2;
    const ScanGeom g = make_geom(B, L, M);
    const size_t BL = (size_t)B * L;
    SamuScratch s;
    size_t o = 0;
    s.status = o;   o += kStatusBlock;
    s.flags = o;    o = align_up(o + (size_t)g.n_tiles * 4);
    s.memset_bytes = o;
    s.agg = o;      o = align_up(o + (size_t)B * g.CT * M * 16);      // tile maps
    s.rin = o;      o = align_up(o + (size_t)B * g.CT * M * 8);       // adjoint leaving each tile
    s.kpart = o;    o = align_up(o + BL * g.n_groups * 8);            // per-token controller partials
    s.numod = o;    o = align_up(o + (size_t)B * g.CT * M * 8);       // per-tile (dnu, dtheta)
    s.numod2 = o;   o = align_up(o + (size_t)kReduceGroups * M * 8);
    s.dwh_part = o; o = align_up(o + (size_t)kCtrlBwdCtas * 2 * 2 * (D + 1) * 4);   // (cta, half) rows
    s.amp_part = o; o = align_up(o + (size_t)kCtrlBwdCtas * 8);
    s.dwh = o;      o = align_up(o + (size_t)8 * 2 * (D + 1) * 4);             // column-sum groups
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
    const ScanGeom g = make_geom(B, L, D);
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
    const ScanGeom g = make_geom(B, L, D);
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

}  // namespace lrs

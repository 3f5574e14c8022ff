// Dense BF16 contractions of the RecurrentBlock on the fifth-generation tensor
// cores (sm_103a).
//
// The block around the mixer ("SAMU 与 RG-LRU 的 H800 训练性能对比", section
// 03, single-block table: normalisation, two input projections, per-channel
// convolution, mixer, join and output projection, second normalisation,
// gated MLP, with the input and parameter backward) is made of dense linear
// layers.  One kernel template computes every one of their contractions,
//   C(m, n) = sum_k A(m, k) B(n, k),
// on 128 x 256 tiles with BF16 operands and FP32 accumulators in tensor
// memory, in three operand layouts:
//   NT  forward   y = x W^T:   A = x [rows][K] and B = W [N][K], both K-major;
//   NN  dX        dx = dy W:   A = dy [rows][K] K-major, B(n, k) = W[k][n]
//                              (MN-major: the weight's rows are the K index);
//   TN  dW        dW = dy^T x: A(m, k) = dy[k][m], B(n, k) = x[k][n], both
//                              MN-major (the token index is the row index of
//                              both), split over the tokens with FP32 partials
//                              added in a fixed order by a second kernel.
// Roles: warp 8 streams 64-wide K slices of both operands by TMA (128-byte
// swizzle) into a ring of stages; one thread of warp 9 issues tcgen05.mma
// (M 128, N 256, K 16) and frees each stage with tcgen05.commit; warps 0-7
// drain the accumulator (tcgen05.ld, one row per thread; warp w reads the
// rows of tensor-memory lane quarter w % 4 and column half w / 4) through the
// layer's fused epilogue.  Two accumulators (512 tensor-memory columns) let the
// epilogue of one tile run under the MMAs of the next.  CTAs are persistent
// over the tiles; every wait is bounded and an abort flag ends the other
// roles after a failure.
// Two-CTA clusters (MC): the two CTAs take the tiles of two consecutive row
// blocks with the same columns (and token split) in lockstep; each loads its
// own A slice and one half of the shared B slice, multicast into both CTAs'
// stages, so the L2 delivers B once per pair.  A stage is refilled only after
// the MMAs of both CTAs have read it (each issuer's commit arrives on both
// CTAs' empty barriers).  A row block past the matrix (odd row-block count)
// runs on zero-filled A and stores nothing.
//
// Fused epilogues (row t of the tile, columns n):
//   store     C in BF16;
//   resid     C + R in BF16 (the residual stream);
//   glu       the tile's columns 0..127 are a = h W_1^T, 128..255 b = h W_2^T
//             for the same 128 hidden units: a, b (BF16) and
//             q = GeLU(a) b (BF16, from the rounded a and b);
//   glu_bwd   C = dq: da = dq b GeLU'(a), db = dq GeLU(a) (BF16);
//   join_bwd  C = dj: dy_mixer = dj GeLU(g), dg = dj y_mixer GeLU'(g) (BF16);
//   f32       C in FP32 (dW partials).
// The BF16 results leave by TMA stores from swizzled per-warp staging; the
// operands that resid, glu_bwd and join_bwd read come by TMA into per-warp
// slots two 32-column groups ahead (their results are staged in the slot the
// group's operands came in).  The f32 partials are stored by the threads.
#include <algorithm>
#include <atomic>

#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tmap.cuh"
#include "umma.cuh"
#include "block_math.cuh"

namespace lrs {

namespace {

constexpr int kBgEpiWarps = 8;
constexpr int kBgThreads = 32 * (kBgEpiWarps + 2);   // warps 0-7 epilogue, 8 producer, 9 MMA
constexpr int kBgProducer = kBgEpiWarps, kBgIssuer = kBgEpiWarps + 1;
constexpr int kBgK = 64;          // K per stage (one 128-byte swizzle row of BF16)
constexpr int kBgM = 128;         // tile rows
constexpr int kBgN = 256;         // tile columns (accumulator columns)
constexpr int kBgStages = 4;      // ring stages (3 for the epilogues with operands)
constexpr uint32_t kBgABytes = kBgM * 128;            // 16 KB
constexpr uint32_t kBgBBytes = kBgN * 128;            // 32 KB
constexpr uint32_t kBgStageBytes = kBgABytes + kBgBBytes;
constexpr uint32_t kBgTmemCols = 2 * kBgN;           // two accumulators
// Epilogues that read operands of their own (residual, GLU backward, join
// backward) take them by TMA into shared memory: per epilogue warp two slots,
// each one 32-column group of its 32 rows per operand ([32][32] BF16 boxes,
// 64-byte swizzle), filled two groups ahead.  With two operands the ring gives
// up a stage for them; the residual's one operand fits beside four stages.
__host__ __device__ constexpr bool bg_op_epi(int epi) {
    return epi == kEpiResid || epi == kEpiGluBwd || epi == kEpiJoinBwd;
}
__host__ __device__ constexpr int bg_op_count(int epi) { return !bg_op_epi(epi) ? 0 : epi == kEpiResid ? 1 : 2; }
__host__ __device__ constexpr int bg_stages(int epi) { return bg_op_count(epi) == 2 ? kBgStages - 1 : kBgStages; }
constexpr int kBgOpCols = 32;
constexpr uint32_t kBgOpBox = 32 * kBgOpCols * 2;     // 2 KB
__host__ __device__ constexpr uint32_t bg_op_slot(int epi) { return (uint32_t)bg_op_count(epi) * kBgOpBox; }
// The GLU epilogue writes a, b and q by TMA stores from per-warp staging:
// [32 rows][16 columns] BF16 boxes (32-byte swizzle), one of each.
constexpr uint32_t kBgStBox = 32 * 16 * 2;            // 1 KB
// The plain store's staging: two [32 rows][32 columns] BF16 boxes (64-byte
// swizzle) per warp, alternating.
__host__ __device__ constexpr uint32_t bg_st_warp(int epi) {
    return epi == kEpiGlu ? 3 * kBgStBox : epi == kEpiStore ? 2 * kBgOpBox : 0u;
}
constexpr size_t bg_smem(int epi) {   // + 1 KB for the 1024-byte alignment
    return (size_t)bg_stages(epi) * kBgStageBytes + (size_t)kBgEpiWarps * (2 * bg_op_slot(epi) + bg_st_warp(epi)) +
           1024;
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf_round(float x) {   // value of RNE(x) in BF16, as FP32
    return __bfloat162float(__float2bfloat16_rn(x));
}

// 8 BF16 values from 16 bytes.
__device__ __forceinline__ void unpack8(const uint4 q, float (&v)[8]) {
    v[0] = bf_lo(q.x); v[1] = bf_hi(q.x); v[2] = bf_lo(q.y); v[3] = bf_hi(q.y);
    v[4] = bf_lo(q.z); v[5] = bf_hi(q.z); v[6] = bf_lo(q.w); v[7] = bf_hi(q.w);
}
__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 q;
    q.x = f2_to_bf2(v[0], v[1]);
    q.y = f2_to_bf2(v[2], v[3]);
    q.z = f2_to_bf2(v[4], v[5]);
    q.w = f2_to_bf2(v[6], v[7]);
    return q;
}

struct BgItem {
    int mt, nt, s, k0, k1;
};

// Work item w of a CTA (MC: pair item w, row block 2 (w's row pair) + rank).
__device__ __forceinline__ BgItem bg_item(const BlockGemmArgs& a, int w, bool mc, int rank) {
    BgItem it;
    if (a.layout == kBgTN) {
        it.s = w % a.splits;
        const int r = w / a.splits;
        it.nt = r % a.n_tiles;
        it.mt = mc ? 2 * (r / a.n_tiles) + rank : r / a.n_tiles;
        it.k0 = (int)((long long)a.ksteps * it.s / a.splits);
        it.k1 = (int)((long long)a.ksteps * (it.s + 1) / a.splits);
    } else {
        it.mt = mc ? 2 * (w / a.n_tiles) + rank : w / a.n_tiles;
        it.nt = w % a.n_tiles;
        it.s = 0;
        it.k0 = 0;
        it.k1 = a.ksteps;
    }
    return it;
}

// Epilogue of one accumulator row (row `m` of tile `it`, accumulator columns
// at taddr), column half `half` of the tile (of its 128 hidden units for glu).
template <int EPI>
__device__ __forceinline__ void bg_epilogue(const BlockGemmArgs& a, const BgItem& it, int m, uint32_t taddr, int half) {
    const long long t = (long long)it.mt * kBgM + m;
    const int c0 = half * (kBgN / 2), c1 = c0 + kBgN / 2;
    if (EPI == kEpiF32) {
        float* o = a.part + ((size_t)it.s * a.M + (size_t)t) * a.N + (size_t)it.nt * kBgN;
        for (int c = c0; c < c1; c += 32) {
            float v[2][16];
            tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(c + 16), v[0], v[1]);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(o + c + j) =
                    make_float4(v[j / 16][j % 16], v[j / 16][j % 16 + 1], v[j / 16][j % 16 + 2], v[j / 16][j % 16 + 3]);
        }
        return;
    }
    const bool ok = t < a.M;
    if (EPI == kEpiGlu) {
        const int f0 = it.nt * (kBgN / 2);
        for (int c = half * (kBgN / 4); c < (half + 1) * (kBgN / 4); c += 16) {
            float va[16], vb[16];
            tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(kBgN / 2 + c), va, vb);
            if (!ok) continue;
            float q[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                va[j] = bf_round(va[j]);
                vb[j] = bf_round(vb[j]);
                q[j] = gelu_fwd(va[j]) * vb[j];
            }
            uint16_t* ab = a.out2 + (size_t)t * a.ld2 + f0 + c;
            uint16_t* qo = a.out + (size_t)t * a.ldo + f0 + c;
#pragma unroll
            for (int j = 0; j < 16; j += 8) {
                *reinterpret_cast<uint4*>(ab + j) = pack8(va + j);
                *reinterpret_cast<uint4*>(ab + a.F + j) = pack8(vb + j);
                *reinterpret_cast<uint4*>(qo + j) = pack8(q + j);
            }
        }
        return;
    }
    const int n0 = it.nt * kBgN;
    if (EPI == kEpiStore) {
        for (int c = c0; c < c1; c += 32) {
            float v[2][16];
            tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(c + 16), v[0], v[1]);
            if (!ok) continue;
            uint16_t* o = a.out + (size_t)t * a.ldo + n0 + c;
#pragma unroll
            for (int j = 0; j < 32; j += 8) *reinterpret_cast<uint4*>(o + j) = pack8(v[j / 16] + j % 16);
        }
        return;
    }
    // Epilogues that read operands of their own: the row's operands of 64
    // columns are loaded first (up to 16 independent 16-byte loads in flight
    // per thread), then the accumulator is drained 16 columns at a time.
    constexpr int kChunk = 64;
    for (int cc = c0; cc < c1; cc += kChunk) {
        const int n = n0 + cc;
        uint4 p0[kChunk / 8], p1[kChunk / 8];
        if (ok) {
            const uint16_t* s0 = EPI == kEpiResid ? a.r + (size_t)t * a.ldr + n : a.e0 + (size_t)t * a.lde0 + n;
            const uint16_t* s1 = EPI == kEpiGluBwd ? s0 + a.F : EPI == kEpiJoinBwd ? a.e1 + (size_t)t * a.lde1 + n : s0;
#pragma unroll
            for (int j = 0; j < kChunk / 8; ++j) {
                p0[j] = __ldg(reinterpret_cast<const uint4*>(s0) + j);
                if (EPI != kEpiResid) p1[j] = __ldg(reinterpret_cast<const uint4*>(s1) + j);
            }
        }
        float vq[2][16];   // two groups of 16 accumulator columns per tensor-memory round trip
#pragma unroll
        for (int q = 0; q < kChunk / 16; ++q) {
            if ((q & 1) == 0)
                tmem_ld16x2(taddr + (uint32_t)(cc + 16 * q), taddr + (uint32_t)(cc + 16 * q + 16), vq[0], vq[1]);
            float* v = vq[q & 1];
            if (!ok) continue;
            const size_t col = (size_t)n + 16 * q;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float x0[8], x1[8], r0[8], r1[8];
                unpack8(p0[2 * q + h], x0);
                if (EPI != kEpiResid) unpack8(p1[2 * q + h], x1);
                float* vv = v + 8 * h;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (EPI == kEpiResid) {
                        r0[i] = vv[i] + x0[i];
                    } else if (EPI == kEpiGluBwd) {   // x0 = a, x1 = b: da, db
                        float g, dg;
                        gelu_fwd_grad(x0[i], g, dg);
                        r0[i] = vv[i] * x1[i] * dg;
                        r1[i] = vv[i] * g;
                    } else {                          // x0 = g, x1 = y_mixer: d y_mixer, dg
                        float g, dg;
                        gelu_fwd_grad(x0[i], g, dg);
                        r0[i] = vv[i] * g;
                        r1[i] = vv[i] * x1[i] * dg;
                    }
                }
                if (EPI == kEpiResid) {
                    *reinterpret_cast<uint4*>(a.out + (size_t)t * a.ldo + col + 8 * h) = pack8(r0);
                } else if (EPI == kEpiGluBwd) {
                    uint16_t* o = a.out + (size_t)t * a.ldo + col + 8 * h;   // da at f, db at F + f
                    *reinterpret_cast<uint4*>(o) = pack8(r0);
                    *reinterpret_cast<uint4*>(o + a.F) = pack8(r1);
                } else {
                    *reinterpret_cast<uint4*>(a.out + (size_t)t * a.ldo + col + 8 * h) = pack8(r0);
                    *reinterpret_cast<uint4*>(a.out2 + (size_t)t * a.ld2 + col + 8 * h) = pack8(r1);
                }
            }
        }
    }
}

template <int LAYOUT, int EPI, bool MC>
__global__ void __launch_bounds__(kBgThreads, 1)
    block_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_e0, const __grid_constant__ CUtensorMap tm_e1,
                      const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_s1,
                      BlockGemmArgs a) {
    constexpr int S = bg_stages(EPI);
    constexpr bool OP = bg_op_epi(EPI);
    extern __shared__ uint8_t bg_raw[];
    __shared__ __align__(8) uint64_t s_full[kBgStages], s_empty[kBgStages], s_acc[2], s_free[2], s_fin;
    __shared__ __align__(8) uint64_t s_op[kBgEpiWarps][2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(bg_raw) + 1023u) & ~uintptr_t(1023));

    const int rank = MC ? (int)cluster_ctarank() : 0;
    constexpr uint16_t kPair = 0x3;
    // MC: the CTA's pair items, the same sequence in both CTAs of the cluster
    const int w0 = MC ? (int)blockIdx.x / 2 : (int)blockIdx.x;
    const int wstep = MC ? (int)gridDim.x / 2 : (int)gridDim.x;
    const int n_work = MC ? a.n_pairs : a.n_items;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], MC ? 2 : 1);   // MC: both CTAs' MMAs free a stage
        }
        if (OP)
            for (int i = 0; i < kBgEpiWarps; ++i) {
                mbar_init(&s_op[i][0], 1);
                mbar_init(&s_op[i][1], 1);
            }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_acc[i], 1);
            mbar_init(&s_free[i], kBgEpiWarps);
        }
        mbar_init(&s_fin, 1);
        s_abort = 0;
    }
    if (warp == kBgIssuer) {
        tmem_alloc(&s_tmem, kBgTmemCols);
        tmem_fence_before_sync();
    }
    pdl_trigger();
    pdl_wait();
    __syncthreads();
    if (MC) cluster_sync();   // both CTAs' barriers exist before either reaches the other's
    tmem_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(a.status, kStatusTimeout);
    };

    if (warp == kBgProducer) {
        // producer: every K step of every tile of this CTA, in order
        if (lane == 0) {
            uint32_t n = 0;   // stages issued
            for (int w = w0; w < n_work && !*abort_flag; w += wstep) {
                const BgItem it = bg_item(a, w, MC, rank);
                for (int ks = it.k0; ks < it.k1; ++ks, ++n) {
                    const int slot = (int)(n % S);
                    if (n >= (uint32_t)S && !mbar_wait_bounded(&s_empty[slot], ((n / S) - 1) & 1u)) {
                        fail();
                        break;
                    }
                    if (*abort_flag) break;
                    uint8_t* sa = ring + (size_t)slot * kBgStageBytes;
                    uint8_t* sb = sa + kBgABytes;
                    const int k0 = kBgK * ks;
                    mbar_arrive_expect_tx(&s_full[slot], kBgStageBytes);
                    // B: MC loads half of the slice (rank 0 the first, rank 1 the second) into both CTAs
                    auto load_b = [&](int part, uint8_t* dst, int x, int y) {
                        if (!MC)
                            tma_load_2d(dst, &tm_b, x, y, &s_full[slot]);
                        else if (part == rank)
                            tma_load_2d_mc(dst, &tm_b, x, y, &s_full[slot], kPair);
                    };
                    if (LAYOUT == kBgNT) {
                        tma_load_2d(sa, &tm_a, k0, it.mt * kBgM, &s_full[slot]);
                        const int r0 = EPI == kEpiGlu ? it.nt * (kBgN / 2) : it.nt * kBgN;
                        const int r1 = EPI == kEpiGlu ? a.F + r0 : r0 + kBgN / 2;
                        load_b(0, sb, k0, r0);
                        load_b(1, sb + kBgBBytes / 2, k0, r1);
                    } else if (LAYOUT == kBgNN) {
                        tma_load_2d(sa, &tm_a, k0, it.mt * kBgM, &s_full[slot]);
#pragma unroll
                        for (int j = 0; j < kBgN / 64; ++j)
                            load_b(j / 2, sb + (size_t)j * 8192, it.nt * kBgN + 64 * j, k0);
                    } else {
                        tma_load_2d(sa, &tm_a, it.mt * kBgM, k0, &s_full[slot]);
                        tma_load_2d(sa + 8192, &tm_a, it.mt * kBgM + 64, k0, &s_full[slot]);
#pragma unroll
                        for (int j = 0; j < kBgN / 64; ++j)
                            load_b(j / 2, sb + (size_t)j * 8192, it.nt * kBgN + 64 * j, k0);
                    }
                }
            }
            // copies still in flight land before the CTA may exit (MC: and the
            // other CTA's MMAs have read this CTA's halves of the last stages)
            const uint32_t lo = n > (uint32_t)S ? n - S : 0;
            for (uint32_t j = lo; j < n; ++j) mbar_wait_bounded(&s_full[j % S], (j / S) & 1u);
            if (MC)
                for (uint32_t j = lo; j < n; ++j) mbar_wait_bounded(&s_empty[j % S], (j / S) & 1u);
        }
    } else if (warp == kBgIssuer) {
        // MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(kBgM, kBgN) | (LAYOUT == kBgTN ? (1u << 15) : 0u) |
                                       (LAYOUT != kBgNT ? (1u << 16) : 0u);
            uint32_t n = 0, item = 0;
            for (int w = w0; w < n_work && !*abort_flag; w += wstep, ++item) {
                const BgItem it = bg_item(a, w, MC, rank);
                const uint32_t buf = item & 1u;
                // the epilogue has drained this accumulator's previous tile
                if (item >= 2 && !mbar_wait_bounded(&s_free[buf], ((item >> 1) - 1) & 1u)) {
                    fail();
                    break;
                }
                tmem_fence_after_sync();
                const uint32_t acc_t = tmem + buf * (uint32_t)kBgN;
                bool ok = true;
                for (int ks = it.k0; ks < it.k1; ++ks, ++n) {
                    const int slot = (int)(n % S);
                    if (!mbar_wait_bounded(&s_full[slot], (n / S) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tmem_fence_after_sync();
                    const uint32_t sa = smem_u32(ring + (size_t)slot * kBgStageBytes);
                    const uint32_t sb = sa + kBgABytes;
#pragma unroll
                    for (int kk = 0; kk < kBgK / 16; ++kk) {
                        const bool accum = ks > it.k0 || kk > 0;
                        const uint64_t da = LAYOUT == kBgTN ? umma_desc_sw128_mn(sa + 2048u * kk, 8192u)
                                                            : umma_desc_sw128(sa + 32u * kk);
                        const uint64_t db = LAYOUT == kBgNT ? umma_desc_sw128(sb + 32u * kk)
                                                            : umma_desc_sw128_mn(sb + 2048u * kk, 8192u);
                        umma_bf16(acc_t, da, db, idesc, accum);
                    }
                    // the stage is free once these MMAs have read it (MC: in both CTAs)
                    if (MC)
                        umma_commit_mc(&s_empty[slot], kPair);
                    else
                        umma_commit(&s_empty[slot]);
                }
                if (!ok) break;
                umma_commit(&s_acc[buf]);
            }
            // every MMA issued by this thread has completed before the columns are released
            umma_commit(&s_fin);
            mbar_wait_bounded(&s_fin, 0);
        }
    } else if (OP) {
        // epilogue warps 0-7 with operands: rows 32 (warp % 4) .. + 31, column half warp / 4,
        // in groups of 32 columns whose operand rows arrive by TMA two groups ahead
        const int q4 = warp & 3, hf = warp >> 2;
        constexpr uint32_t kSlot = bg_op_slot(EPI);
        uint8_t* ops = ring + (size_t)S * kBgStageBytes + (size_t)warp * 2 * kSlot;
        constexpr int kG = (kBgN / 2) / kBgOpCols;   // groups per tile
        const uint32_t n_groups = w0 < n_work ? (uint32_t)((n_work - 1 - w0) / wstep + 1) * kG : 0u;
        uint32_t issued = 0;   // lane 0: groups asked for
        auto issue = [&]() {
            const uint32_t gi = issued++;
            const int slot = (int)(gi & 1u);
            const BgItem ig = bg_item(a, w0 + (int)(gi / kG) * wstep, MC, rank);
            const int x = ig.nt * kBgN + hf * (kBgN / 2) + (int)(gi % kG) * kBgOpCols;
            const int y = ig.mt * kBgM + 32 * q4;
            uint8_t* dst = ops + (size_t)slot * kSlot;
            fence_proxy_async();   // the slot's earlier reads (the warp's, before __syncwarp) come first
            mbar_arrive_expect_tx(&s_op[warp][slot], kSlot);
            tma_load_2d(dst, &tm_e0, x, y, &s_op[warp][slot]);
            if (EPI == kEpiGluBwd) tma_load_2d(dst + kBgOpBox, &tm_e0, a.F + x, y, &s_op[warp][slot]);
            if (EPI == kEpiJoinBwd) tma_load_2d(dst + kBgOpBox, &tm_e1, x, y, &s_op[warp][slot]);
        };
        if (lane == 0)
            while (issued < n_groups && issued < 2u) issue();
        uint32_t item = 0, g = 0;   // g: groups consumed
        for (int w = w0; w < n_work && !*abort_flag; w += wstep, ++item) {
            const BgItem it = bg_item(a, w, MC, rank);
            const uint32_t buf = item & 1u;
            if (!mbar_wait_bounded(&s_acc[buf], (item >> 1) & 1u)) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_after_sync();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + buf * (uint32_t)kBgN;
            bool lost = false;
            for (int k = 0; k < kG; ++k, ++g) {
                const int slot = (int)(g & 1u);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_op[warp][slot], (g >> 1) & 1u))) {
                    lost = true;
                    break;
                }
                const int c = hf * (kBgN / 2) + k * kBgOpCols;   // the group's first column in the tile
                float v[2][16];
                tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(c + 16), v[0], v[1]);
                // this row's operands: four 16-byte units of 64 bytes, the unit index
                // XOR-ed with bits 1-2 of the row (the 64-byte swizzle)
                const uint8_t* src = ops + (size_t)slot * kSlot + (size_t)lane * 64;
                uint4 o0[4], o1[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int pu = u ^ ((lane >> 1) & 3);
                    o0[u] = *reinterpret_cast<const uint4*>(src + 16 * pu);
                    if (EPI != kEpiResid) o1[u] = *reinterpret_cast<const uint4*>(src + kBgOpBox + 16 * pu);
                }
                // the group's results, staged in the slot its operands came in and
                // stored by TMA (rows past M are clipped; a row block past the matrix
                // stores nothing), before the slot takes group g + 2
                uint4 w0[4], w1[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float x0[8], x1[8], r0[8], r1[8];
                    unpack8(o0[u], x0);
                    if (EPI != kEpiResid) unpack8(o1[u], x1);
                    const float* vv = v[u >> 1] + 8 * (u & 1);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (EPI == kEpiResid) {
                            r0[i] = vv[i] + x0[i];
                        } else if (EPI == kEpiGluBwd) {   // x0 = a, x1 = b: da, db
                            float gg, dg;
                            gelu_fwd_grad(x0[i], gg, dg);
                            r0[i] = vv[i] * x1[i] * dg;
                            r1[i] = vv[i] * gg;
                        } else {                          // x0 = g, x1 = y_mixer: d y_mixer, dg
                            float gg, dg;
                            gelu_fwd_grad(x0[i], gg, dg);
                            r0[i] = vv[i] * gg;
                            r1[i] = vv[i] * x1[i] * dg;
                        }
                    }
                    w0[u] = pack8(r0);
                    if (EPI != kEpiResid) w1[u] = pack8(r1);
                }
                __syncwarp();   // every lane has read its operands from the slot
                uint8_t* box = ops + (size_t)slot * kSlot;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int pu = u ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4*>(box + (size_t)lane * 64 + 16 * pu) = w0[u];
                    if (EPI != kEpiResid) *reinterpret_cast<uint4*>(box + kBgOpBox + (size_t)lane * 64 + 16 * pu) = w1[u];
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    if (it.mt < a.m_tiles && it.mt * kBgM + 32 * q4 < a.M) {
                        const int x = it.nt * kBgN + c;
                        // resid: out; glu_bwd: da at f, db at F + f of [da | db]; join_bwd: d y_mixer, dg
                        tma_store_2d(&tm_s0, x, it.mt * kBgM + 32 * q4, box);
                        if (EPI == kEpiGluBwd) tma_store_2d(&tm_s0, a.F + x, it.mt * kBgM + 32 * q4, box + kBgOpBox);
                        if (EPI == kEpiJoinBwd) tma_store_2d(&tm_s1, x, it.mt * kBgM + 32 * q4, box + kBgOpBox);
                        bulk_commit();
                        bulk_wait_read<0>();   // the slot is read out before it takes the next group
                    }
                    if (issued < n_groups) issue();
                }
            }
            if (lost) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[buf]);
        }
        // operand groups still in flight land, and the stores complete, before the CTA may exit
        if (lane == 0) {
            for (uint32_t j = g; j < issued; ++j) mbar_wait_bounded(&s_op[warp][j & 1u], (j >> 1) & 1u);
            bulk_wait_all();
        }
    } else if (EPI == kEpiStore) {
        // epilogue warps 0-7 of the plain store: rows 32 (warp % 4) .. + 31, column half
        // warp / 4, 32 columns at a time staged in two alternating boxes and stored by TMA
        const int q4 = warp & 3, hf = warp >> 2;
        uint8_t* stg = ring + (size_t)S * kBgStageBytes + (size_t)warp * bg_st_warp(EPI);
        uint32_t chunk = 0, item = 0;   // every chunk commits one bulk group (empty when nothing is stored)
        for (int w = w0; w < n_work && !*abort_flag; w += wstep, ++item) {
            const BgItem it = bg_item(a, w, MC, rank);
            const uint32_t buf = item & 1u;
            if (!mbar_wait_bounded(&s_acc[buf], (item >> 1) & 1u)) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_after_sync();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + buf * (uint32_t)kBgN;
            const int y = it.mt * kBgM + 32 * q4;
            const bool store = it.mt < a.m_tiles && y < a.M;   // rows past M are clipped by the TMA
#pragma unroll 1
            for (int c = hf * (kBgN / 2); c < (hf + 1) * (kBgN / 2); c += 32, ++chunk) {
                float v[2][16];
                tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(c + 16), v[0], v[1]);
                uint8_t* box = stg + (size_t)(chunk & 1u) * kBgOpBox;
                if (lane == 0 && chunk >= 2) bulk_wait_read<1>();   // the box of two chunks ago is read out
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int pu = u ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4*>(box + (size_t)lane * 64 + 16 * pu) = pack8(v[u >> 1] + 8 * (u & 1));
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    if (store) tma_store_2d(&tm_s0, it.nt * kBgN + c, y, box);
                    bulk_commit();
                }
            }
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[buf]);
        }
        if (lane == 0) bulk_wait_all();   // every store has completed before the CTA may exit
    } else if (EPI == kEpiGlu) {
        // epilogue warps 0-7 of the GLU: rows 32 (warp % 4) .. + 31, hidden units of column
        // half warp / 4, 16 at a time; a, b and q leave by TMA stores (tm_e0: [a | b], tm_e1: q)
        const int q4 = warp & 3, hf = warp >> 2;
        uint8_t* stg = ring + (size_t)S * kBgStageBytes + (size_t)warp * bg_st_warp(EPI);
        bool pending = false;   // lane 0: stores committed whose staging reads may be in flight
        uint32_t item = 0;
        for (int w = w0; w < n_work && !*abort_flag; w += wstep, ++item) {
            const BgItem it = bg_item(a, w, MC, rank);
            const uint32_t buf = item & 1u;
            if (!mbar_wait_bounded(&s_acc[buf], (item >> 1) & 1u)) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_after_sync();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + buf * (uint32_t)kBgN;
            const int f0 = it.nt * (kBgN / 2);
            const int y = it.mt * kBgM + 32 * q4;
            const bool store = it.mt < a.m_tiles && y < a.M;   // rows past M are clipped by the TMA
#pragma unroll 1
            for (int c = hf * (kBgN / 4); c < (hf + 1) * (kBgN / 4); c += 16) {
                float va[16], vb[16];
                tmem_ld16x2(taddr + (uint32_t)c, taddr + (uint32_t)(kBgN / 2 + c), va, vb);
                float q[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    va[j] = bf_round(va[j]);
                    vb[j] = bf_round(vb[j]);
                    q[j] = gelu_fwd(va[j]) * vb[j];
                }
                if (lane == 0 && pending) bulk_wait_read<0>();   // the staging is free again
                __syncwarp();
                // row `lane` of each box: 32 bytes, the 16-byte unit u at u ^ bit 2 of the row
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t off = (uint32_t)lane * 32u + 16u * (uint32_t)(u ^ ((lane >> 2) & 1));
                    *reinterpret_cast<uint4*>(stg + off) = pack8(va + 8 * u);
                    *reinterpret_cast<uint4*>(stg + kBgStBox + off) = pack8(vb + 8 * u);
                    *reinterpret_cast<uint4*>(stg + 2 * kBgStBox + off) = pack8(q + 8 * u);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0 && store) {
                    tma_store_2d(&tm_e0, f0 + c, y, stg);
                    tma_store_2d(&tm_e0, a.F + f0 + c, y, stg + kBgStBox);
                    tma_store_2d(&tm_e1, f0 + c, y, stg + 2 * kBgStBox);
                    bulk_commit();
                    pending = true;
                }
            }
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[buf]);
        }
        if (lane == 0) bulk_wait_all();   // every store has completed before the CTA may exit
    } else {
        // epilogue warps 0-7: accumulator rows 32 (warp % 4) .. + 31, column half warp / 4
        uint32_t item = 0;
        const int row = 32 * (warp & 3) + lane;
        for (int w = w0; w < n_work && !*abort_flag; w += wstep, ++item) {
            const BgItem it = bg_item(a, w, MC, rank);
            const uint32_t buf = item & 1u;
            if (!mbar_wait_bounded(&s_acc[buf], (item >> 1) & 1u)) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_after_sync();
            const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + buf * (uint32_t)kBgN;
            if (it.mt < a.m_tiles) bg_epilogue<EPI>(a, it, row, taddr, warp >> 2);
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[buf]);
        }
    }
    __syncthreads();
    if (warp == kBgIssuer) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem, kBgTmemCols);
    }
    if (MC) cluster_sync();   // neither CTA leaves while the other may still use its stages
}

// Out[i] (i < n) = sum over p < parts of part[p * stride + i], in a fixed
// order.  Few parts: one thread per output, p = 0, 1, ... .  Many parts: 32
// outputs per CTA (one per lane) and 32 groups of parts (one per warp, group g
// taking p = g, g + 32, ... in order), the group sums then added g = 0..31.
constexpr int kSumGroups = 32;
__global__ void __launch_bounds__(256) sum_parts_kernel(const float* __restrict__ part, long long stride, int parts,
                                                        long long n, float* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int p = 0; p < parts; ++p) s += part[(size_t)p * stride + i];
        out[i] = s;
    }
}
// The same with four consecutive outputs per thread (16-byte loads; n, stride
// and the pointers multiples of 4 floats), every part's loads issued before
// the sums, which still run p = 0, 1, ... per output.
__global__ void __launch_bounds__(256) sum_parts4_kernel(const float4* __restrict__ part, long long stride4, int parts,
                                                         long long n4, float4* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        int p = 0;
        for (; p + 4 <= parts; p += 4) {
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = __ldcs(part + (size_t)(p + k) * stride4 + i);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s.x += v[k].x;
                s.y += v[k].y;
                s.z += v[k].z;
                s.w += v[k].w;
            }
        }
        for (; p < parts; ++p) {
            const float4 v = __ldcs(part + (size_t)p * stride4 + i);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        out[i] = s;
    }
}
__global__ void __launch_bounds__(32 * kSumGroups) sum_parts_grouped_kernel(const float* __restrict__ part,
                                                                           long long stride, int parts, long long n,
                                                                           float* __restrict__ out) {
    __shared__ float acc[kSumGroups][33];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    for (long long i0 = (long long)blockIdx.x * 32; i0 < n; i0 += (long long)gridDim.x * 32) {
        const long long i = i0 + lane;
        float s = 0.f;
        if (i < n)
            for (int p = g; p < parts; p += kSumGroups) s += part[(size_t)p * stride + i];
        acc[g][lane] = s;
        __syncthreads();
        if (g == 0 && i < n) {
            float t = 0.f;
            for (int k = 0; k < kSumGroups; ++k) t += acc[k][lane];
            out[i] = t;
        }
        __syncthreads();
    }
}
// 2-D tensor map over a row-major [rows][cols] BF16 matrix, box {64, box_rows},
// 128-byte swizzle (rows past the matrix and columns past cols read as zero).
bool bg_map(CUtensorMap* map, const void* ptr, long long cols, long long rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBgK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int bg_sms() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    return (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 1;
}

// Two-CTA clusters sharing the B slice, when there are row blocks to pair.
template <int LAYOUT, int EPI, bool MC>
cudaError_t bg_launch_as(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& te0, const CUtensorMap& te1,
                         const CUtensorMap& ts0, const CUtensorMap& ts1, const BlockGemmArgs& a, cudaStream_t s,
                         bool pdl) {
    auto* fn = block_gemm_kernel<LAYOUT, EPI, MC>;
    constexpr size_t smem = bg_smem(EPI);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kBgThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (MC) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    long long grid = bg_sms();
    if (MC) {
        // one cluster per pair item at most, as many as fit at once (the
        // occupancy query is slow next to a launch: asked once per device)
        static std::atomic<int> cached[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
        int clusters = cached[dev].load(std::memory_order_relaxed);
        if (clusters < 1) {
            cfg.gridDim = dim3(2);
            if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess || clusters < 1)
                clusters = (int)(grid / 2);
            if (clusters < 1) clusters = 1;
            cached[dev].store(clusters, std::memory_order_relaxed);
        }
        grid = 2LL * std::min<long long>(clusters, a.n_pairs);
    } else if (grid > a.n_items) {
        grid = a.n_items;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.numAttrs = na;
    cfg.gridDim = dim3((unsigned)grid);
    return cudaLaunchKernelEx(&cfg, fn, ta, tb, te0, te1, ts0, ts1, a);
}

// The epilogue operands' tensor maps: [rows][cols] BF16 with row stride ld,
// box 32 x 32, 64-byte swizzle (rows past the matrix read as zero).
bool bg_op_map(CUtensorMap* map, const void* ptr, long long cols, long long rows, long long ld) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBgOpCols, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The GLU's output maps: [rows][cols] BF16 with row stride ld, box 16 x 32,
// 32-byte swizzle (rows past the matrix are not written).
bool bg_st_map(CUtensorMap* map, const void* ptr, long long cols, long long rows, long long ld) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int LAYOUT, int EPI>
cudaError_t bg_launch(const CUtensorMap& ta, const CUtensorMap& tb, const BlockGemmArgs& a, cudaStream_t s, bool pdl) {
    CUtensorMap te0 = ta, te1 = ta, ts0 = ta, ts1 = ta;
    // stores of the plain, residual, GLU backward and join backward epilogues:
    // box 32 x 32, 64-byte swizzle (rows past the matrix are not written)
    if (EPI == kEpiStore || EPI == kEpiResid || EPI == kEpiJoinBwd) {
        if (!bg_op_map(&ts0, a.out, a.N, a.M, a.ldo)) return cudaErrorInvalidValue;
    } else if (EPI == kEpiGluBwd) {   // [da | db]
        if (!bg_op_map(&ts0, a.out, 2LL * a.F, a.M, a.ldo)) return cudaErrorInvalidValue;
    }
    if (EPI == kEpiJoinBwd && !bg_op_map(&ts1, a.out2, a.N, a.M, a.ld2)) return cudaErrorInvalidValue;
    if (EPI == kEpiGlu) {   // stores: [a | b] and q, box 16 x 32, 32-byte swizzle
        if (!bg_st_map(&te0, a.out2, 2LL * a.F, a.M, a.ld2) || !bg_st_map(&te1, a.out, a.F, a.M, a.ldo))
            return cudaErrorInvalidValue;
    } else if (EPI == kEpiResid) {
        if (!bg_op_map(&te0, a.r, a.N, a.M, a.ldr)) return cudaErrorInvalidValue;
    } else if (EPI == kEpiGluBwd) {   // [a | b]: a at column f, b at F + f
        if (!bg_op_map(&te0, a.e0, 2LL * a.F, a.M, a.lde0)) return cudaErrorInvalidValue;
    } else if (EPI == kEpiJoinBwd) {  // g: the first N columns of [g | v]; y_mixer
        if (!bg_op_map(&te0, a.e0, a.N, a.M, a.lde0) || !bg_op_map(&te1, a.e1, a.N, a.M, a.lde1))
            return cudaErrorInvalidValue;
    }
    if (a.m_tiles >= 2) return bg_launch_as<LAYOUT, EPI, true>(ta, tb, te0, te1, ts0, ts1, a, s, pdl);
    return bg_launch_as<LAYOUT, EPI, false>(ta, tb, te0, te1, ts0, ts1, a, s, pdl);
}

}  // namespace

int block_gemm_sms() {
    const int n = bg_sms();
    return n < kBlockSmsBound ? n : kBlockSmsBound;
}

// Token splits of a TN (dW) contraction: the count that minimises the
// estimated time, waves x K steps per item x the time of one K step of a
// 128 x 256 tile (0.48 us, measured at B4 L4K Dm = D = 1024), plus the split
// partials' extra traffic (written, read back, the sum written) at 6 TB/s.
// A count that only fills one wave can leave most of a second wave idle
// (192 items on 152 SMs run as two waves at 63%).
constexpr double kBgStepUs = 0.48;
constexpr double kBgBytesPerUs = 6.0e6;

int block_gemm_splits(int M, int N, long long K, int sms) {
    const long long tiles = (long long)(M / kBgM) * (N / kBgN);
    if (tiles < 1 || sms < 1) return 1;
    const long long steps = (K + kBgK - 1) / kBgK;
    double best = 0.0;
    int best_s = 1;
    for (int sp = 1; sp <= kBlockGemmSplitsMax && sp <= steps; ++sp) {
        const long long waves = (tiles * sp + sms - 1) / sms;
        const double t = (double)waves * (double)((steps + sp - 1) / sp) * kBgStepUs +
                         (sp > 1 ? ((double)sp * 8.0 + 4.0) * (double)M * (double)N / kBgBytesPerUs : 0.0);
        if (sp == 1 || t < best) {
            best = t;
            best_s = sp;
        }
    }
    return best_s;
}

int block_gemm_splits_bound(int M, int N, long long K) {
    int s = 1;
    for (int sms = 1; sms <= kBlockSmsBound; ++sms) s = std::max(s, block_gemm_splits(M, N, K, sms));
    return s;
}

cudaError_t launch_block_gemm(const BlockGemmArgs& args_in, const void* A, const void* Bm, cudaStream_t s, bool pdl) {
    BlockGemmArgs a = args_in;
    CUtensorMap ta, tb;
    const long long M = a.M, N = a.N, K = a.K;
    if (a.layout == kBgNT) {
        // A [M][K]; B [N][K] (glu: [2F][K], tile columns pair rows f and F + f)
        const long long brows = a.epi == kEpiGlu ? 2LL * a.F : N;
        if (!bg_map(&ta, A, K, M, kBgM) || !bg_map(&tb, Bm, K, brows, kBgN / 2)) return cudaErrorInvalidValue;
        a.n_tiles = a.epi == kEpiGlu ? (int)(N / (kBgN / 2)) : (int)(N / kBgN);
        a.m_tiles = (int)((M + kBgM - 1) / kBgM);
        a.splits = 1;
        a.ksteps = (int)(K / kBgK);
    } else if (a.layout == kBgNN) {
        // A [M][K]; B = W [K][N]
        if (!bg_map(&ta, A, K, M, kBgM) || !bg_map(&tb, Bm, N, K, 64)) return cudaErrorInvalidValue;
        a.n_tiles = (int)(N / kBgN);
        a.m_tiles = (int)((M + kBgM - 1) / kBgM);
        a.splits = 1;
        a.ksteps = (int)(K / kBgK);
    } else {
        // A = dy [K][M]; B = x [K][N]; K = tokens (a ragged last step reads zeros)
        if (!bg_map(&ta, A, M, K, 64) || !bg_map(&tb, Bm, N, K, 64)) return cudaErrorInvalidValue;
        a.n_tiles = (int)(N / kBgN);
        a.m_tiles = (int)(M / kBgM);
        a.ksteps = (int)((K + kBgK - 1) / kBgK);
        if (a.splits < 1) a.splits = 1;
    }
    a.n_items = a.m_tiles * a.n_tiles * a.splits;
    a.n_pairs = (a.m_tiles + 1) / 2 * a.n_tiles * a.splits;
    if (a.n_items < 1) return cudaSuccess;
    switch (a.layout * 16 + a.epi) {
        case kBgNT * 16 + kEpiStore: return bg_launch<kBgNT, kEpiStore>(ta, tb, a, s, pdl);
        case kBgNT * 16 + kEpiResid: return bg_launch<kBgNT, kEpiResid>(ta, tb, a, s, pdl);
        case kBgNT * 16 + kEpiGlu: return bg_launch<kBgNT, kEpiGlu>(ta, tb, a, s, pdl);
        case kBgNN * 16 + kEpiStore: return bg_launch<kBgNN, kEpiStore>(ta, tb, a, s, pdl);
        case kBgNN * 16 + kEpiGluBwd: return bg_launch<kBgNN, kEpiGluBwd>(ta, tb, a, s, pdl);
        case kBgNN * 16 + kEpiJoinBwd: return bg_launch<kBgNN, kEpiJoinBwd>(ta, tb, a, s, pdl);
        case kBgTN * 16 + kEpiF32: return bg_launch<kBgTN, kEpiF32>(ta, tb, a, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_sum_parts(const float* part, long long stride, int parts, long long n, float* out, cudaStream_t s,
                             bool pdl) {
    if (parts > 16) {
        long long blocks = (n + 31) / 32;
        if (blocks > 8192) blocks = 8192;
        return launch_ex(sum_parts_grouped_kernel, (unsigned)blocks, 32 * kSumGroups, 0, s, pdl, part, stride, parts,
                         n, out);
    }
    if (n % 4 == 0 && stride % 4 == 0 && reinterpret_cast<uintptr_t>(part) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(out) % 16 == 0) {
        long long blocks = (n / 4 + 255) / 256;
        if (blocks > 8192) blocks = 8192;
        if (blocks < 1) blocks = 1;
        return launch_ex(sum_parts4_kernel, (unsigned)blocks, 256, 0, s, pdl, reinterpret_cast<const float4*>(part),
                         stride / 4, parts, n / 4, reinterpret_cast<float4*>(out));
    }
    long long blocks = (n + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    if (blocks < 1) blocks = 1;
    return launch_ex(sum_parts_kernel, (unsigned)blocks, 256, 0, s, pdl, part, stride, parts, n, out);
}

}  // namespace lrs

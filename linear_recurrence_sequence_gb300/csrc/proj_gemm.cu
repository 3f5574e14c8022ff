// RG-LRU gate projections on the fifth-generation tensor cores (sm_103a).
//
// The RG-LRU mixer's two gate projections are 16-block block-diagonal
// linear layers ("SAMU 与 RG-LRU 的 H800 训练性能对比", section 04, forward: two
// canonical block-diagonal projections produce the write- and keep-gate raw
// values; section 06: parameter count 2 D^2/16 + 3 D).  Per block h
// (dk = D/16 channels) the three contractions of a forward + backward are
//   logits: l_q[t][h dk + o] = sum_i x[t][h dk + i] W_q[h][i][o]      (q = x, a)
//   dx:     dx[t][h dk + i]  = sum_k Wcat[h](i, k) G[t][h][k]          (k < 6 dk)
//   dW:     P[h](k, i)       = sum_t G[t][h][k] x[t][h dk + i]          (k < 4 dk)
// where G [B L][16][6][dk] holds the scan backward's BF16 gradient parts
// (dl^x, dl^a and dx through the write term, each as a leading part and a
// remainder) and Wcat packs W_x, W_x, W_a, W_a and two identity blocks.
//
// One kernel template computes C(m, n) = sum_k A(m, k) B(n, k) on 128 x NP
// tiles (NP = dk rounded up to 16), BF16 operands and FP32 accumulators in
// tensor memory:
//  - a producer warp streams the operands' 64-wide K slices by TMA (128-byte
//    swizzle) into a ring of stages;
//  - one thread of an MMA warp issues tcgen05.mma (M 128, N NP, K 16) and
//    releases each stage with tcgen05.commit;
//  - four epilogue warps read the accumulator rows with tcgen05.ld and store
//    them.
// Logits and dx read both operands K-major (the operands' rows are the M and
// N indices); dW reads both MN-major: its reduction index t is the row index
// of G and of x in memory, so a [64 x 64] box of either is a K-group-major
// tile whose 128-byte rows run along M (or N).  dW is split over the tokens
// and the splits are added in a fixed order by a second kernel.
// Every CTA is persistent over work items; every wait is bounded and a shared
// abort flag ends the other roles' loops after a failure.
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace lrs {

namespace {

constexpr int kPgThreads = 192;   // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kPgK = 64;          // K per stage (one 128-byte swizzle row of BF16)
constexpr int kPgStagesMax = 4;
constexpr size_t kPgSmemBudget = 200 * 1024;

enum { kModeLogit = 0, kModeDx = 1, kModeDw = 2 };

}  // namespace

struct ProjGemmArgs {
    int mode;
    int BL, D, dk, NP;        // tokens, width, block width, N tile (dk rounded up to 16)
    int ksteps;               // K steps per work item (logits, dx); dW: K steps of all tokens
    int n_items;
    int m_tiles;              // logits, dx: token tiles; dW: tiles of the 4 dk part rows
    int splits;               // dW: token splits
    float* out0;              // logits: l_x [BL][D]; dx: dx (FP32) ; dW: partials [splits][16][m_tiles 128][NP]
    float* out1;              // logits: l_a [BL][D]
    uint16_t* out_bf16;       // dx in BF16 (or null)
    uint32_t* status;
};

struct PgGeom {
    int stages;
    uint32_t a_bytes, b_bytes, stage_bytes;
    size_t smem;              // ring + slack
};

__host__ __device__ inline PgGeom pg_geom(int mode, int NP) {
    PgGeom g;
    g.a_bytes = 128u * 128u;   // 128 rows x 128 B (or two 64-row MN chunks)
    if (mode == kModeLogit)
        g.b_bytes = 2u * (uint32_t)NP * 128u;
    else if (mode == kModeDx)
        g.b_bytes = (uint32_t)NP * 128u;
    else
        g.b_bytes = (uint32_t)((NP + 63) / 64) * 64u * 128u;
    g.stage_bytes = g.a_bytes + ((g.b_bytes + 1023u) & ~1023u);
    // slack: 1 KB for the 1024-byte alignment of the ring, and 16 KB after it
    // so that no descriptor of the last stage can address past the allocation
    constexpr size_t kSlack = 1024 + 16 * 1024;
    int s = kPgStagesMax;
    while (s > 2 && (size_t)s * g.stage_bytes + kSlack > kPgSmemBudget) --s;
    g.stages = s;
    g.smem = (size_t)s * g.stage_bytes + kSlack;
    return g;
}

__host__ __device__ inline uint32_t pg_tmem_cols(int mode, int NP) {
    const int need = mode == kModeLogit ? 2 * NP : NP;
    uint32_t c = 32;
    while ((int)c < need) c <<= 1;
    return c;
}

// Work item w: (block h, tile mt[, split s]) and its K-step range.
struct PgItem {
    int h, mt, s, k0, k1;
};

__device__ __forceinline__ PgItem pg_item(const ProjGemmArgs& a, int w) {
    PgItem it;
    if (a.mode == kModeDw) {
        it.s = w % a.splits;
        const int r = w / a.splits;
        it.mt = r % a.m_tiles;
        it.h = r / a.m_tiles;
        it.k0 = (int)((long long)a.ksteps * it.s / a.splits);
        it.k1 = (int)((long long)a.ksteps * (it.s + 1) / a.splits);
    } else {
        it.h = w % kProjBlocks;
        it.mt = w / kProjBlocks;
        it.s = 0;
        it.k0 = 0;
        it.k1 = a.ksteps;
    }
    return it;
}

template <int MODE>
__global__ void __launch_bounds__(kPgThreads, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     ProjGemmArgs a) {
    extern __shared__ uint8_t pg_raw[];
    __shared__ __align__(8) uint64_t s_full[kPgStagesMax], s_empty[kPgStagesMax], s_acc, s_free;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const PgGeom pg = pg_geom(MODE, a.NP);
    const int S = pg.stages;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pg_raw) + 1023u) & ~uintptr_t(1023));
    const uint32_t tcols = pg_tmem_cols(MODE, a.NP);
    const int dk = a.dk, NP = a.NP;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);
        }
        mbar_init(&s_acc, 1);
        mbar_init(&s_free, 4);   // the four epilogue warps
        s_abort = 0;
    }
    if (warp == 5) {
        tmem_alloc(&s_tmem, tcols);
        tmem_fence_before_sync();
    }
    pdl_trigger();
    pdl_wait();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(a.status, kStatusTimeout);
    };

    if (warp == 4) {
        // producer: every K step of every work item of this CTA, in order
        if (lane == 0) {
            uint32_t n = 0;   // stages issued
            for (int w = blockIdx.x; w < a.n_items && !*abort_flag; w += gridDim.x) {
                const PgItem it = pg_item(a, w);
                for (int ks = it.k0; ks < it.k1; ++ks, ++n) {
                    const int slot = (int)(n % S);
                    if (n >= (uint32_t)S && !mbar_wait_bounded(&s_empty[slot], ((n / S) - 1) & 1u)) {
                        fail();
                        break;
                    }
                    if (*abort_flag) break;
                    uint8_t* st = ring + (size_t)slot * pg.stage_bytes;
                    uint8_t* sb = st + pg.a_bytes;
                    mbar_arrive_expect_tx(&s_full[slot], pg.a_bytes + pg.b_bytes);
                    if (MODE == kModeLogit) {
                        tma_load_2d(st, &tm_a, it.h * dk + kPgK * ks, it.mt * 128, &s_full[slot]);
                        tma_load_2d(sb, &tm_b, kPgK * ks, (2 * it.h) * NP, &s_full[slot]);
                        tma_load_2d(sb + (size_t)NP * 128, &tm_b, kPgK * ks, (2 * it.h + 1) * NP, &s_full[slot]);
                    } else if (MODE == kModeDx) {
                        tma_load_2d(st, &tm_a, it.h * 6 * dk + kPgK * ks, it.mt * 128, &s_full[slot]);
                        tma_load_2d(sb, &tm_b, kPgK * ks, it.h * NP, &s_full[slot]);
                    } else {
                        const int t0 = kPgK * ks;
                        const int m0 = it.h * 6 * dk + it.mt * 128;
                        tma_load_2d(st, &tm_a, m0, t0, &s_full[slot]);
                        tma_load_2d(st + 8192, &tm_a, m0 + 64, t0, &s_full[slot]);
                        for (int j = 0; j * 64 < NP; ++j)
                            tma_load_2d(sb + (size_t)j * 8192, &tm_b, it.h * dk + 64 * j, t0, &s_full[slot]);
                    }
                }
            }
            // copies still in flight land before the CTA may exit
            const uint32_t lo = n > (uint32_t)S ? n - S : 0;
            for (uint32_t j = lo; j < n; ++j) mbar_wait_bounded(&s_full[j % S], (j / S) & 1u);
        }
    } else if (warp == 5) {
        // MMA issuer
        if (lane == 0) {
            const uint32_t idesc = MODE == kModeDw ? umma_idesc_bf16_mn(128, NP) : umma_idesc_bf16(128, NP);
            uint32_t n = 0, item = 0;
            bool committed = false;
            for (int w = blockIdx.x; w < a.n_items && !*abort_flag; w += gridDim.x, ++item) {
                const PgItem it = pg_item(a, w);
                if (item > 0 && !mbar_wait_bounded(&s_free, (item - 1) & 1u)) {   // epilogue has read the accumulator
                    fail();
                    break;
                }
                tmem_fence_after_sync();
                bool ok = true;
                for (int ks = it.k0; ks < it.k1; ++ks, ++n) {
                    const int slot = (int)(n % S);
                    if (!mbar_wait_bounded(&s_full[slot], (n / S) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tmem_fence_after_sync();
                    const uint32_t sa = smem_u32(ring + (size_t)slot * pg.stage_bytes);
                    const uint32_t sb = sa + pg.a_bytes;
#pragma unroll
                    for (int kk = 0; kk < kPgK / 16; ++kk) {
                        const bool acc = ks > it.k0 || kk > 0;
                        if (MODE == kModeLogit) {
                            umma_bf16(tmem, umma_desc_sw128(sa + 32u * kk), umma_desc_sw128(sb + 32u * kk), idesc, acc);
                            umma_bf16(tmem + (uint32_t)NP, umma_desc_sw128(sa + 32u * kk),
                                      umma_desc_sw128(sb + (uint32_t)NP * 128u + 32u * kk), idesc, acc);
                        } else if (MODE == kModeDx) {
                            umma_bf16(tmem, umma_desc_sw128(sa + 32u * kk), umma_desc_sw128(sb + 32u * kk), idesc, acc);
                        } else {
                            umma_bf16(tmem, umma_desc_sw128_mn(sa + 2048u * kk, 8192u),
                                      umma_desc_sw128_mn(sb + 2048u * kk, 8192u), idesc, acc);
                        }
                    }
                    umma_commit(&s_empty[slot]);   // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                umma_commit(&s_acc);
                committed = true;
            }
            (void)committed;
        }
    } else {
        // epilogue warps 0-3: accumulator rows 32 warp .. 32 warp + 31
        uint32_t item = 0;
        for (int w = blockIdx.x; w < a.n_items && !*abort_flag; w += gridDim.x, ++item) {
            const PgItem it = pg_item(a, w);
            if (!mbar_wait_bounded(&s_acc, item & 1u)) {
                if (lane == 0) fail();
                break;
            }
            tmem_fence_after_sync();
            const int m = 32 * warp + lane;
            const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
            if (MODE == kModeLogit) {
                const long long t = (long long)it.mt * 128 + m;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float* o = (q == 0 ? a.out0 : a.out1) + (size_t)t * a.D + (size_t)it.h * dk;
                    for (int c = 0; c < NP; c += 16) {
                        float v[16];
                        tmem_ld16(trow + (uint32_t)(q * NP + c), v);
                        if (t < a.BL) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                if (c + j < dk)
                                    *reinterpret_cast<float4*>(o + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                        }
                    }
                }
            } else if (MODE == kModeDx) {
                const long long t = (long long)it.mt * 128 + m;
                for (int c = 0; c < NP; c += 16) {
                    float v[16];
                    tmem_ld16(trow + (uint32_t)c, v);
                    if (t < a.BL) {
                        const size_t base = (size_t)t * a.D + (size_t)it.h * dk + c;
                        if (a.out_bf16 != nullptr) {
#pragma unroll
                            for (int j = 0; j < 16; j += 8)
                                if (c + j < dk) {
                                    uint4 pk;
                                    pk.x = f2_to_bf2(v[j], v[j + 1]);
                                    pk.y = f2_to_bf2(v[j + 2], v[j + 3]);
                                    pk.z = f2_to_bf2(v[j + 4], v[j + 5]);
                                    pk.w = f2_to_bf2(v[j + 6], v[j + 7]);
                                    *reinterpret_cast<uint4*>(a.out_bf16 + base + j) = pk;
                                }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                if (c + j < dk)
                                    *reinterpret_cast<float4*>(a.out0 + base + j) =
                                        make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                        }
                    }
                }
            } else {
                const int row = it.mt * 128 + m;   // part row p dk + o
                float* o = a.out0 + (((size_t)it.s * kProjBlocks + it.h) * (size_t)(a.m_tiles * 128) + row) * NP;
                for (int c = 0; c < NP; c += 16) {
                    float v[16];
                    tmem_ld16(trow + (uint32_t)c, v);
                    if (row < 4 * dk) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(o + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    }
                }
            }
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free);
        }
    }
    __syncthreads();
    if (warp == 5) {
        // the MMAs of an aborted item may still be running: wait (bounded) for
        // the last commit before the accumulator columns are released
        if (*abort_flag && lane == 0) {
            for (int i = 0; i < S; ++i) mbar_wait_bounded(&s_empty[i], 0);
        }
        __syncwarp();
        tmem_fence_after_sync();
        tmem_dealloc(tmem, tcols);
    }
}

// Packed operand images (BF16, K-major, zero outside the blocks):
//  wt[h][q][n][k] = W_q[h][k][n]                   (logits: B(n, k), K padded to kp)
//  wc[h][n][k]    = Wcat[h](n, k): W_x[h][n][o] (k = p dk + o, p = 0, 1),
//                   W_a (p = 2, 3), [n == o] (p = 4, 5)   (dx: B(n, k), K padded to kp6)
__global__ void __launch_bounds__(256) proj_pack_kernel(const uint16_t* __restrict__ w_x,
                                                        const uint16_t* __restrict__ w_a, uint16_t* __restrict__ wt,
                                                        uint16_t* __restrict__ wc, int dk, int NP, int kp, int kp6) {
    const size_t n_t = (size_t)kProjBlocks * 2 * NP * kp;
    const size_t n_c = (size_t)kProjBlocks * NP * kp6;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_t + n_c; e += (size_t)gridDim.x * blockDim.x) {
        if (e < n_t) {
            const int k = (int)(e % kp);
            const int n = (int)(e / kp % NP);
            const int q = (int)(e / ((size_t)kp * NP) % 2);
            const int h = (int)(e / ((size_t)kp * NP * 2));
            uint16_t v = 0;
            if (n < dk && k < dk) v = (q == 0 ? w_x : w_a)[((size_t)h * dk + k) * dk + n];
            wt[e] = v;
        } else {
            const size_t f = e - n_t;
            const int k = (int)(f % kp6);
            const int n = (int)(f / kp6 % NP);
            const int h = (int)(f / ((size_t)kp6 * NP));
            uint16_t v = 0;
            if (n < dk && k < 6 * dk) {
                const int p = k / dk, o = k % dk;
                if (p < 2)
                    v = w_x[((size_t)h * dk + n) * dk + o];
                else if (p < 4)
                    v = w_a[((size_t)h * dk + n) * dk + o];
                else
                    v = n == o ? (uint16_t)0x3F80u : (uint16_t)0;   // BF16 1.0 and 0.0
            }
            wc[f] = v;
        }
    }
}

// dW_x[h][i][o] = sum over the splits, in order, of P(o, i) + P(dk + o, i);
// dW_a likewise from the part rows 2 dk + o and 3 dk + o.
__global__ void __launch_bounds__(256) proj_dw_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw_x,
                                                             float* __restrict__ dw_a, int dk, int NP, int rows,
                                                             int splits) {
    pdl_trigger();
    pdl_wait();
    const size_t n = (size_t)kProjBlocks * dk * dk;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const int o = (int)(e % dk);
        const int i = (int)(e / dk % dk);
        const size_t h = e / ((size_t)dk * dk);
        float sx = 0.f, sa = 0.f;
        for (int s = 0; s < splits; ++s) {
            const float* p = part + ((size_t)s * kProjBlocks + h) * (size_t)rows * NP;
            sx += p[(size_t)o * NP + i] + p[(size_t)(dk + o) * NP + i];
            sa += p[(size_t)(2 * dk + o) * NP + i] + p[(size_t)(3 * dk + o) * NP + i];
        }
        dw_x[e] = sx;
        dw_a[e] = sa;
    }
}

namespace {

// 2-D tensor map over a row-major [rows][cols] BF16 matrix, box {64, box_rows},
// 128-byte swizzle (rows past the matrix and columns past cols read as zero).
bool make_2d_sw128(CUtensorMap* map, const void* ptr, long long cols, long long rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kPgK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int pg_sms() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    return (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 1;
}

template <int MODE>
cudaError_t launch_pg(const CUtensorMap& ta, const CUtensorMap& tb, const ProjGemmArgs& a, cudaStream_t s, bool pdl) {
    const PgGeom pg = pg_geom(MODE, a.NP);
    const cudaError_t e =
        cudaFuncSetAttribute(proj_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pg.smem);
    if (e != cudaSuccess) return e;
    int grid = pg_sms();
    if (grid > a.n_items) grid = a.n_items;
    return launch_ex(proj_gemm_kernel<MODE>, (unsigned)grid, kPgThreads, pg.smem, s, pdl, ta, tb, a);
}

}  // namespace

cudaError_t launch_proj_pack(const void* w_x, const void* w_a, void* wt, void* wc, const ProjDims& d, cudaStream_t s) {
    const size_t n = (size_t)kProjBlocks * d.NP * (2 * d.kp + d.kp6);
    proj_pack_kernel<<<(unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, s>>>(
        static_cast<const uint16_t*>(w_x), static_cast<const uint16_t*>(w_a), static_cast<uint16_t*>(wt),
        static_cast<uint16_t*>(wc), d.dk, d.NP, d.kp, d.kp6);
    return cudaGetLastError();
}

cudaError_t launch_proj_logits(const void* x, const void* wt, float* lx, float* la, int D, const ProjDims& d,
                               uint32_t* status, cudaStream_t s, bool pdl) {
    CUtensorMap ta, tb;
    if (!make_2d_sw128(&ta, x, D, d.BL, 128) || !make_2d_sw128(&tb, wt, d.kp, (long long)kProjBlocks * 2 * d.NP, d.NP))
        return cudaErrorInvalidValue;
    ProjGemmArgs a{};
    a.mode = kModeLogit;
    a.BL = d.BL;
    a.D = D;
    a.dk = d.dk;
    a.NP = d.NP;
    a.ksteps = d.kp / kPgK;
    a.m_tiles = (d.BL + 127) / 128;
    a.n_items = a.m_tiles * kProjBlocks;
    a.splits = 1;
    a.out0 = lx;
    a.out1 = la;
    a.status = status;
    return launch_pg<kModeLogit>(ta, tb, a, s, pdl);
}

cudaError_t launch_proj_dx(const void* gparts, const void* wc, void* dx, bool dx_fp32, int D, const ProjDims& d,
                           uint32_t* status, cudaStream_t s, bool pdl) {
    CUtensorMap ta, tb;
    if (!make_2d_sw128(&ta, gparts, 6LL * D, d.BL, 128) ||
        !make_2d_sw128(&tb, wc, d.kp6, (long long)kProjBlocks * d.NP, d.NP))
        return cudaErrorInvalidValue;
    ProjGemmArgs a{};
    a.mode = kModeDx;
    a.BL = d.BL;
    a.D = D;
    a.dk = d.dk;
    a.NP = d.NP;
    a.ksteps = d.kp6 / kPgK;
    a.m_tiles = (d.BL + 127) / 128;
    a.n_items = a.m_tiles * kProjBlocks;
    a.splits = 1;
    a.out0 = dx_fp32 ? static_cast<float*>(dx) : nullptr;
    a.out_bf16 = dx_fp32 ? nullptr : static_cast<uint16_t*>(dx);
    a.status = status;
    return launch_pg<kModeDx>(ta, tb, a, s, pdl);
}

int proj_dw_splits(const ProjDims& d) {
    const int tiles = kProjBlocks * (d.dw_rows / 128);
    int s = (pg_sms() + tiles - 1) / tiles;
    const int steps = (d.BL + kPgK - 1) / kPgK;
    if (s > kProjDwSplitsMax) s = kProjDwSplitsMax;
    if (s > steps) s = steps;
    return s < 1 ? 1 : s;
}

cudaError_t launch_proj_dw(const void* gparts, const void* x, float* part, float* dw_x, float* dw_a, int D,
                           const ProjDims& d, uint32_t* status, cudaStream_t s, bool pdl) {
    CUtensorMap ta, tb;
    if (!make_2d_sw128(&ta, gparts, 6LL * D, d.BL, kPgK) || !make_2d_sw128(&tb, x, D, d.BL, kPgK))
        return cudaErrorInvalidValue;
    ProjGemmArgs a{};
    a.mode = kModeDw;
    a.BL = d.BL;
    a.D = D;
    a.dk = d.dk;
    a.NP = d.NP;
    a.ksteps = (d.BL + kPgK - 1) / kPgK;
    a.m_tiles = d.dw_rows / 128;
    a.splits = proj_dw_splits(d);
    a.n_items = kProjBlocks * a.m_tiles * a.splits;
    a.out0 = part;
    a.status = status;
    cudaError_t e = launch_pg<kModeDw>(ta, tb, a, s, pdl);
    if (e != cudaSuccess) return e;
    const size_t n = (size_t)kProjBlocks * d.dk * d.dk;
    return launch_ex(proj_dw_reduce_kernel, (unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024), 256, 0, s,
                     true, static_cast<const float*>(part), dw_x, dw_a, d.dk, d.NP, d.dw_rows, a.splits);
}

}  // namespace lrs

// extern "C" entry points declared in include/samu.h: argument checks,
// workspace carving and kernel launches.  No allocation, no synchronisation
// (except lrs_device_status, which documents that it synchronises).
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include "kernels.cuh"
#include "tmap.cuh"

using namespace lrs;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int L, int D) {
    if (B < 1 || L < 1 || D < 2 || (D & 1)) return LRS_ERR_ARG;
    const long long BL = (long long)B * L;
    if (BL * (long long)D > (1LL << 40)) return LRS_ERR_UNSUPPORTED;
    return LRS_OK;
}

int check_samu_shape(int B, int L, int D) {
    int st = check_common(B, L, D);
    if (st != LRS_OK) return st;
    if (D % 16 != 0 || D > 4096) return LRS_ERR_UNSUPPORTED;
    const SegGeom g = samu_seg_geom(B, L, D / 2, 0);
    if ((long long)g.n_chains * g.NSmax > 0x7fffffffLL) return LRS_ERR_UNSUPPORTED;
    return LRS_OK;
}

int check_rglru_shape(int B, int L, int D) {
    int st = check_common(B, L, D);
    if (st != LRS_OK) return st;
    if (D % 8 != 0) return LRS_ERR_UNSUPPORTED;
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    if (g.n_tiles > 0x7fffffffLL) return LRS_ERR_UNSUPPORTED;
    return LRS_OK;
}

// Required pointer: non-null and 16-byte aligned.
bool req(const void* p) { return p != nullptr && aligned16(p); }
// Optional pointer: null, or 16-byte aligned.
bool opt(const void* p) { return p == nullptr || aligned16(p); }

// Opt-in per-kernel event timing (lrs_profile_*): a fixed pool of CUDA event
// pairs recorded on the launching stream around each kernel.
struct Profiler {
    bool on = false;
    int cap = 0;
    int n = 0;
    cudaEvent_t* ev = nullptr;   // 2 * cap events
    int* ids = nullptr;
} g_prof;

void prof_begin(int id, cudaStream_t s) {
    if (!g_prof.on || g_prof.n >= g_prof.cap) return;
    g_prof.ids[g_prof.n] = id;
    cudaEventRecord(g_prof.ev[2 * g_prof.n], s);
}

void prof_end(cudaStream_t s) {
    if (!g_prof.on || g_prof.n >= g_prof.cap) return;
    cudaEventRecord(g_prof.ev[2 * g_prof.n + 1], s);
    ++g_prof.n;
}

// Launches after the first of a call overlap their start with the previous
// kernel (programmatic dependent launch), except while per-kernel timing is
// on, so that every kernel's events bracket it alone.
bool pdl_ok() { return !g_prof.on; }

// samu_set_chunk_transition (read once by each call, from any host thread)
std::atomic<int> g_transition{LRS_TRANSITION_CLOSED_FORM};

// Kernel ids reported by lrs_profile_end.
enum {
    KID_SAMU_CTRL_FWD = 2, KID_SAMU_SCAN_FWD, KID_SAMU_SCAN_BWD, KID_SAMU_CTRL_BWD,
    KID_SAMU_PARAMS, KID_RGLRU_SCAN_FWD, KID_RGLRU_SCAN_BWD, KID_RGLRU_ALPHA, KID_SAMU_FWD_MAPS,
    KID_SAMU_BWD_MAPS, KID_SAMU_DECODE_PREP, KID_SAMU_DECODE_STEP, KID_RGLRU_PROJ_FWD, KID_RGLRU_PROJ_BWD,
    KID_RGLRU_PROJ_PACK, KID_BLOCK_GEMM, KID_BLOCK_NORM, KID_BLOCK_CONV, KID_BLOCK_JOIN, KID_BLOCK_SUM
};

#define LRS_LAUNCH(id, stream, expr)            \
    do {                                        \
        prof_begin((id), (stream));             \
        cudaError_t e_ = (expr);                \
        prof_end(stream);                       \
        if (e_ != cudaSuccess) return LRS_ERR_CUDA; \
    } while (0)

int check_rglru_proj_shape(int B, int L, int D) {
    const int st = check_rglru_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (D % kProjBlocks != 0 || (D / kProjBlocks) % 8 != 0) return LRS_ERR_UNSUPPORTED;
    if ((long long)B * L > 0x7fffffffLL) return LRS_ERR_UNSUPPORTED;
    return LRS_OK;
}

// Failure-path self-test: one warp waits, bounded, on an mbarrier that nothing
// completes; the wait gives up at its deadline and records the timeout in the
// status word, exactly as a stalled copy would in the scan kernels.
__global__ void lrs_selftest_wait_kernel(uint32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        *status = 0u;
        mbar_init(&bar, 1);
    }
    __syncthreads();
    if (!mbar_wait_bounded(&bar, 0) && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T>
const T* at(const void* base, size_t off) {
    return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

}  // namespace

extern "C" {

const char* lrs_status_string(int status) {
    switch (status) {
        case LRS_OK: return "ok";
        case LRS_ERR_ARG: return "invalid argument (null or misaligned pointer, bad shape)";
        case LRS_ERR_UNSUPPORTED: return "unsupported shape";
        case LRS_ERR_CUDA: return "CUDA launch failed";
        case LRS_ERR_TIMEOUT: return "a bounded device-side wait gave up";
        case LRS_ERR_TOO_LARGE: return "problem too large for the fixed no-allocation workspace";
        default: return "unknown status";
    }
}

const char* samu_status_string(int status) { return lrs_status_string(status); }

int lrs_version(void) { return 101; }

int samu_set_chunk_transition(int kind) {
    if (kind != LRS_TRANSITION_CHAINED && kind != LRS_TRANSITION_CLOSED_FORM) return LRS_ERR_ARG;
    g_transition.store(kind);
    return LRS_OK;
}

int samu_get_chunk_transition(void) { return g_transition.load(); }

int lrs_profile_begin(int capacity) {
    if (capacity < 1) return LRS_ERR_ARG;
    if (g_prof.cap < capacity) {
        for (int i = 0; i < 2 * g_prof.cap; ++i) cudaEventDestroy(g_prof.ev[i]);
        delete[] g_prof.ev;
        delete[] g_prof.ids;
        g_prof.ev = new cudaEvent_t[2 * capacity];
        g_prof.ids = new int[capacity];
        for (int i = 0; i < 2 * capacity; ++i) {
            if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
                g_prof.cap = 0;
                return LRS_ERR_CUDA;
            }
        }
        g_prof.cap = capacity;
    }
    g_prof.n = 0;
    g_prof.on = true;
    return LRS_OK;
}

int lrs_profile_end(int* kernel_ids, float* ms, int capacity, int* count) {
    if (count == nullptr) return LRS_ERR_ARG;
    g_prof.on = false;
    const int n = g_prof.n < capacity ? g_prof.n : capacity;
    for (int i = 0; i < n; ++i) {
        if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return LRS_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) return LRS_ERR_CUDA;
        if (kernel_ids) kernel_ids[i] = g_prof.ids[i];
        if (ms) ms[i] = t;
    }
    *count = g_prof.n;
    return LRS_OK;
}

int lrs_selftest_wait_timeout(void* scratch, cudaStream_t stream) {
    uint32_t* word = static_cast<uint32_t*>(scratch);
    if (scratch == nullptr) {   // the no-allocation forward's fixed array
        const int st = noalloc_status_word(&word);
        if (st != LRS_OK) return st;
    } else if (!req(scratch)) {
        return LRS_ERR_ARG;
    }
    lrs_selftest_wait_kernel<<<1, 32, 0, stream>>>(word);
    return cudaGetLastError() == cudaSuccess ? LRS_OK : LRS_ERR_CUDA;
}

int lrs_device_status(void* scratch, int* status, cudaStream_t stream) {
    if (scratch == nullptr || status == nullptr) return LRS_ERR_ARG;
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return LRS_ERR_CUDA;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return LRS_ERR_CUDA;
    *status = (v & kStatusLayout) ? LRS_ERR_CUDA : (v & (kStatusTimeout | kStatusUpstream)) ? LRS_ERR_TIMEOUT : LRS_OK;
    return LRS_OK;
}

// ---------------------------------------------------------------------------
// SAMU
// ---------------------------------------------------------------------------
int samu_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes) {
    const int st = check_samu_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (saved_bytes) *saved_bytes = samu_saved_layout(B, L, D).total;
    if (scratch_bytes) *scratch_bytes = samu_scratch_layout(B, L, D).total;
    return LRS_OK;
}

int samu_forward(const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                 const float* nu, const float* theta, const float* w_phi, const float* w_r,
                 const float* a_phi, const float* a_r, int B, int L, int D,
                 void* y, float* y32, float* hT, void* saved, void* scratch,
                 cudaStream_t stream) {
    const int st = check_samu_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (!req(x_sel) || !req(w) || !opt(h0) || !req(nu) || !req(theta) || !req(w_phi) ||
        !req(w_r) || a_phi == nullptr || a_r == nullptr || !req(y) || !opt(y32) || !req(hT) ||
        !req(saved) || !req(scratch))
        return LRS_ERR_ARG;
    const int M = D / 2;
    const SamuSaved sv = samu_saved_layout(B, L, D);
    const SamuScratch sc = samu_scratch_layout(B, L, D);
    const long long BL = (long long)B * L;

    float* wh = at<float>(saved, sv.wh);
    float* misc = at<float>(saved, sv.misc);
    float* p = at<float>(saved, sv.p);
    float* r = at<float>(saved, sv.r);
    float4* ctrl = at<float4>(saved, sv.ctrl);
    float4* items = at<float4>(saved, sv.items);

    float4* modes = at<float4>(saved, sv.modes);
    SamuCtrlFwdArgs cf;
    cf.BL = BL;
    cf.B = B;
    cf.L = L;
    cf.D = D;
    cf.x = static_cast<const uint4*>(x_sel);
    cf.reset = reset;
    cf.w_phi = w_phi;
    cf.w_r = w_r;
    cf.a_phi = a_phi;
    cf.a_r = a_r;
    cf.nu = nu;
    cf.theta = theta;
    cf.p = p;
    cf.r = r;
    cf.ctrl = ctrl;
    cf.items = items;
    cf.wh = wh;
    cf.misc = misc;
    cf.modes = modes;
    cf.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_SAMU_CTRL_FWD, stream, launch_samu_ctrl_fwd(cf, stream, false));

    const SegGeom g = samu_scan_geom(B, L, M, false);
    CUtensorMap tm_w, tm_ctrl;
    if (!make_bf16_map(&tm_w, w, B, L, D, kMapRows) || !make_ctrl_map(&tm_ctrl, ctrl, B, L, kMapRows)) return LRS_ERR_CUDA;
    SamuScanFwdArgs a;
    a.g = g;
    a.items = items;
    a.modes = modes;
    a.nu = nu;
    a.closed_form = g_transition.load() == LRS_TRANSITION_CLOSED_FORM;
    a.h0 = h0;
    a.y = static_cast<uint32_t*>(y);
    a.y32 = y32;
    a.hT = hT;
    a.hsub = at<float2>(saved, sv.hsub);
    a.smap = at<float4>(scratch, sc.smap);
    a.cmap = at<float4>(scratch, sc.cmap);
    a.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_SAMU_FWD_MAPS, stream, launch_samu_fwd_maps(tm_w, tm_ctrl, a, stream, pdl_ok()));
    LRS_LAUNCH(KID_SAMU_SCAN_FWD, stream, launch_samu_fwd_replay(tm_w, tm_ctrl, a, stream, pdl_ok()));
    return LRS_OK;
}

int samu_backward(const void* dy, const float* dhT,
                  const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                  const float* nu, const float* theta, const float* w_phi, const float* w_r,
                  const float* a_phi, const float* a_r, int B, int L, int D,
                  const void* saved, void* dx_sel, void* dw, int grad_dtype,
                  float* dh0, float* dnu, float* dtheta, float* dw_phi, float* dw_r,
                  float* da_phi, float* da_r, void* scratch, cudaStream_t stream) {
    (void)h0;
    (void)w_phi;
    (void)w_r;
    (void)a_phi;
    (void)a_r;
    const int st = check_samu_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (grad_dtype != LRS_GRAD_BF16 && grad_dtype != LRS_GRAD_FP32) return LRS_ERR_ARG;
    if (!req(dy) || !opt(dhT) || !req(x_sel) || !req(w) || !req(nu) || !req(theta) ||
        !req(saved) || !req(dx_sel) || !req(dw) || !req(dh0) || !req(dnu) || !req(dtheta) ||
        !req(dw_phi) || !req(dw_r) || da_phi == nullptr || da_r == nullptr || !req(scratch))
        return LRS_ERR_ARG;
    const int M = D / 2;
    const SamuSaved sv = samu_saved_layout(B, L, D);
    const SamuScratch sc = samu_scratch_layout(B, L, D);
    const SegGeom g = samu_scan_geom(B, L, M, true);
    const int fp32 = grad_dtype == LRS_GRAD_FP32 ? 1 : 0;

    const float4* ctrl = at<float4>(saved, sv.ctrl);
    // the status word starts at zero
    if (cudaMemsetAsync(scratch, 0, sc.zero_bytes, stream) != cudaSuccess) return LRS_ERR_CUDA;
    // 16-row boxes for the adjoint maps, 8-row boxes for the reverse replay
    CUtensorMap tm_dy, tm_ctrl, tm_dy8, tm_w8, tm_ctrl8;
    if (!make_bf16_map(&tm_dy, dy, B, L, D, kMapRows) || !make_ctrl_map(&tm_ctrl, ctrl, B, L, kMapRows) ||
        !make_bf16_map(&tm_dy8, dy, B, L, D, kHalf) || !make_bf16_map(&tm_w8, w, B, L, D, kHalf) ||
        !make_ctrl_map(&tm_ctrl8, ctrl, B, L, kHalf))
        return LRS_ERR_CUDA;
    SamuScanBwdArgs s;
    s.g = g;
    s.items = at<float4>(saved, sv.items);
    s.modes = at<float4>(saved, sv.modes);
    s.nu = nu;
    s.closed_form = g_transition.load() == LRS_TRANSITION_CLOSED_FORM;
    s.dhT = dhT;
    s.hsub = at<float2>(saved, sv.hsub);
    s.dw = dw;
    s.grad_fp32 = fp32;
    s.dh0 = dh0;
    s.smap = at<float4>(scratch, sc.smap);
    s.cmap = at<float4>(scratch, sc.cmap);
    s.kpart = at<float2>(scratch, sc.kpart);
    s.numod = at<float2>(scratch, sc.numod);
    s.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_SAMU_BWD_MAPS, stream, launch_samu_bwd_maps(tm_dy, tm_ctrl, s, stream, false));
    CUtensorMap tm_dw8{};
    if (!fp32 && !make_bf16_map(&tm_dw8, dw, B, L, D, kHalf)) return LRS_ERR_CUDA;
    LRS_LAUNCH(KID_SAMU_SCAN_BWD, stream, launch_samu_bwd_main(tm_dy8, tm_w8, tm_ctrl8, tm_dw8, s, stream, pdl_ok()));

    SamuCtrlBwdArgs cb;
    cb.BL = (long long)B * L;
    cb.D = D;
    cb.n_groups = g.n_groups;
    cb.cg = samu_ctrl_geom(cb.BL, D);
    cb.status = s.status;
    cb.x = static_cast<const uint4*>(x_sel);
    cb.kpart = s.kpart;
    cb.p = at<float>(saved, sv.p);
    cb.r = at<float>(saved, sv.r);
    cb.ctrl = ctrl;
    cb.wh = at<float>(saved, sv.wh);
    cb.misc = at<float>(saved, sv.misc);
    cb.dx = dx_sel;
    cb.grad_fp32 = fp32;
    cb.numod = s.numod;
    cb.numod_rows = B * g.NS;
    cb.dwh_part = at<float>(scratch, sc.dwh_part);
    cb.amp_part = at<float2>(scratch, sc.amp_part);
    cb.dot_part = at<float2>(scratch, sc.dot_part);
    cb.dnu = dnu;
    cb.dtheta = dtheta;
    LRS_LAUNCH(KID_SAMU_CTRL_BWD, stream, launch_samu_ctrl_bwd(cb, stream, pdl_ok()));

    SamuParamArgs pa;
    pa.D = D;
    pa.n_rows = cb.cg.n_ctas;
    pa.dwh_part = cb.dwh_part;
    pa.amp_part = cb.amp_part;
    pa.dot_part = cb.dot_part;
    pa.wh = cb.wh;
    pa.misc = cb.misc;
    pa.dw_phi = dw_phi;
    pa.dw_r = dw_r;
    pa.da_phi = da_phi;
    pa.da_r = da_r;
    LRS_LAUNCH(KID_SAMU_PARAMS, stream, launch_samu_params(pa, stream, pdl_ok()));
    return LRS_OK;
}

// ---------------------------------------------------------------------------
// SAMU decode step
// ---------------------------------------------------------------------------
int samu_decode_params_floats(int D, size_t* floats) {
    if (floats == nullptr) return LRS_ERR_ARG;
    const int st = check_samu_shape(1, 1, D);
    if (st != LRS_OK) return st;
    *floats = samu_decode_params_floats(D);
    return LRS_OK;
}

int samu_decode_prepare(const float* nu, const float* theta, const float* w_phi, const float* w_r,
                        const float* a_phi, const float* a_r, int D, float* params, cudaStream_t stream) {
    const int st = check_samu_shape(1, 1, D);
    if (st != LRS_OK) return st;
    if (!req(nu) || !req(theta) || !req(w_phi) || !req(w_r) || a_phi == nullptr || a_r == nullptr || !req(params))
        return LRS_ERR_ARG;
    SamuDecodePrepArgs a;
    a.D = D;
    a.nu = nu;
    a.theta = theta;
    a.w_phi = w_phi;
    a.w_r = w_r;
    a.a_phi = a_phi;
    a.a_r = a_r;
    a.params = params;
    LRS_LAUNCH(KID_SAMU_DECODE_PREP, stream, launch_samu_decode_prepare(a, stream));
    return LRS_OK;
}

int samu_decode_step(const void* x_sel, const void* w, const float* state_in, float* state_out,
                     const uint8_t* reset, const float* params, int B, int D, void* y, float* y32,
                     cudaStream_t stream) {
    const int st = check_samu_shape(B, 1, D);
    if (st != LRS_OK) return st;
    if (!req(x_sel) || !req(w) || !req(state_in) || !req(state_out) || !req(params) || !req(y) || !opt(y32))
        return LRS_ERR_ARG;
    SamuDecodeStepArgs a;
    a.B = B;
    a.D = D;
    a.x = static_cast<const uint16_t*>(x_sel);
    a.w = static_cast<const uint16_t*>(w);
    a.state_in = state_in;
    a.state_out = state_out;
    a.reset = reset;
    a.params = params;
    a.y = static_cast<uint16_t*>(y);
    a.y32 = y32;
    LRS_LAUNCH(KID_SAMU_DECODE_STEP, stream, launch_samu_decode_step(a, stream));
    return LRS_OK;
}

// ---------------------------------------------------------------------------
// RG-LRU
// ---------------------------------------------------------------------------
int rglru_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes) {
    const int st = check_rglru_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (saved_bytes) *saved_bytes = rglru_saved_layout(B, L, D).total;
    if (scratch_bytes) *scratch_bytes = rglru_scratch_layout(B, L, D).total;
    return LRS_OK;
}

int rglru_forward(const void* x, const void* lx, const void* la, const float* alpha,
                  const float* h0, const uint8_t* reset, int B, int L, int D,
                  void* y, float* y32, float* hT, void* saved, void* scratch,
                  cudaStream_t stream) {
    const int st = check_rglru_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (!req(x) || !req(lx) || !req(la) || !req(alpha) || !opt(h0) || !req(y) || !opt(y32) ||
        !req(hT) || !req(saved) || !req(scratch))
        return LRS_ERR_ARG;
    const RglruSaved sv = rglru_saved_layout(B, L, D);
    const RglruScratch sc = rglru_scratch_layout(B, L, D);
    cudaError_t e = cudaMemsetAsync(scratch, 0, sc.memset_bytes, stream);
    if (e != cudaSuccess) return LRS_ERR_CUDA;
    CUtensorMap tm_x, tm_lx, tm_la;
    if (!make_bf16_map(&tm_x, x, B, L, D, kRgTile) || !make_bf16_map(&tm_lx, lx, B, L, D, kRgTile) ||
        !make_bf16_map(&tm_la, la, B, L, D, kRgTile))
        return LRS_ERR_CUDA;
    RglruScanFwdArgs a{};
    a.g = make_geom(B, L, D, kRgTile);
    a.alpha = alpha;
    a.reset = reset;
    a.h0 = h0;
    a.y = static_cast<uint32_t*>(y);
    a.y32 = y32;
    a.hT = hT;
    a.hsub = at<float>(saved, sv.hsub);
    a.agg = at<float2>(scratch, sc.agg);
    a.flags = at<uint32_t>(scratch, sc.flags);
    a.counter = at<uint32_t>(scratch, sc.status + 4);
    a.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_RGLRU_SCAN_FWD, stream, launch_rglru_scan_fwd(tm_x, tm_lx, tm_la, a, stream));
    return LRS_OK;
}

int rglru_backward(const void* dy, const float* dhT, const void* x, const void* lx,
                   const void* la, const float* alpha, const float* h0, const uint8_t* reset,
                   int B, int L, int D, const void* saved, void* dx, void* dlx, void* dla,
                   int grad_dtype, float* dalpha, float* dh0, void* scratch,
                   cudaStream_t stream) {
    (void)h0;
    const int st = check_rglru_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (grad_dtype != LRS_GRAD_BF16 && grad_dtype != LRS_GRAD_FP32) return LRS_ERR_ARG;
    if (!req(dy) || !opt(dhT) || !req(x) || !req(lx) || !req(la) || !req(alpha) || !req(saved) ||
        !req(dx) || !req(dlx) || !req(dla) || !req(dalpha) || !req(dh0) || !req(scratch))
        return LRS_ERR_ARG;
    const RglruSaved sv = rglru_saved_layout(B, L, D);
    const RglruScratch sc = rglru_scratch_layout(B, L, D);
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    cudaError_t e = cudaMemsetAsync(scratch, 0, sc.memset_bytes, stream);
    if (e != cudaSuccess) return LRS_ERR_CUDA;
    CUtensorMap tm_dy, tm_x, tm_lx, tm_la;
    if (!make_bf16_map(&tm_dy, dy, B, L, D, kRgTile) || !make_bf16_map(&tm_x, x, B, L, D, kRgTile) ||
        !make_bf16_map(&tm_lx, lx, B, L, D, kRgTile) || !make_bf16_map(&tm_la, la, B, L, D, kRgTile))
        return LRS_ERR_CUDA;
    RglruScanBwdArgs a{};
    a.g = g;
    a.alpha = alpha;
    a.reset = reset;
    a.dhT = dhT;
    a.hsub = at<float>(saved, sv.hsub);
    a.dx = dx;
    a.dlx = dlx;
    a.dla = dla;
    a.grad_fp32 = grad_dtype == LRS_GRAD_FP32 ? 1 : 0;
    a.dh0 = dh0;
    a.agg = at<float2>(scratch, sc.agg);
    a.rin = at<float>(scratch, sc.rin);
    a.apart = at<float>(scratch, sc.apart);
    a.flags = at<uint32_t>(scratch, sc.flags);
    a.counter = at<uint32_t>(scratch, sc.status + 4);
    a.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_RGLRU_SCAN_BWD, stream, launch_rglru_scan_bwd(tm_dy, tm_x, tm_lx, tm_la, a, stream));
    LRS_LAUNCH(KID_RGLRU_ALPHA, stream,
               launch_rglru_alpha(a.apart, at<float>(scratch, sc.apart2), dalpha, B * g.CT, D, stream));
    return LRS_OK;
}

int rglru_proj_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes) {
    const int st = check_rglru_proj_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (saved_bytes) *saved_bytes = rglru_saved_layout(B, L, D).total;
    if (scratch_bytes) *scratch_bytes = rglru_proj_scratch_layout(B, L, D).total;
    return LRS_OK;
}

int rglru_proj_forward(const void* x, const void* w_x, const float* b_x, const void* w_a, const float* b_a,
                       const float* alpha, const float* h0, const uint8_t* reset, int B, int L, int D,
                       void* y, float* y32, float* hT, void* saved, void* scratch, cudaStream_t stream) {
    const int st = check_rglru_proj_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (!req(x) || !req(w_x) || !req(b_x) || !req(w_a) || !req(b_a) || !req(alpha) || !opt(h0) || !req(y) ||
        !opt(y32) || !req(hT) || !req(saved) || !req(scratch))
        return LRS_ERR_ARG;
    const RglruSaved sv = rglru_saved_layout(B, L, D);
    const RglruProjScratch ps = rglru_proj_scratch_layout(B, L, D);
    const RglruScratch& sc = ps.scan;
    float* lx = at<float>(scratch, ps.lx);
    float* la = at<float>(scratch, ps.la);
    // in-kernel logits on the tensor cores when the diagonal blocks tile the
    // 64-channel groups (D/16 divides 64); otherwise the GEMM path
    const bool fused = 64 % (D / kProjBlocks) == 0;
    if (cudaMemsetAsync(scratch, 0, sc.memset_bytes, stream) != cudaSuccess) return LRS_ERR_CUDA;
    CUtensorMap tm_x, tm_lx, tm_la;
    if (fused) {
        LRS_LAUNCH(KID_RGLRU_PROJ_PACK, stream, launch_rglru_proj_wimg(w_x, w_a, at<void>(scratch, ps.wimg), D, stream));
        if (!make_bf16_map_sw128(&tm_x, x, B, L, D, kRgTile)) return LRS_ERR_CUDA;
        tm_lx = tm_x;
        tm_la = tm_x;
    } else {
        const ProjDims pd = proj_dims(B, L, D);
        LRS_LAUNCH(KID_RGLRU_PROJ_PACK, stream,
                   launch_proj_pack(w_x, w_a, at<void>(scratch, ps.wt), at<void>(scratch, ps.wc), pd, stream));
        LRS_LAUNCH(KID_RGLRU_PROJ_FWD, stream,
                   launch_proj_logits(x, at<void>(scratch, ps.wt), lx, la, D, pd, at<uint32_t>(scratch, sc.status),
                                      stream, false));
        if (!make_bf16_map(&tm_x, x, B, L, D, kRgTile) || !make_f32_map(&tm_lx, lx, B, L, D, kRgTile) ||
            !make_f32_map(&tm_la, la, B, L, D, kRgTile))
            return LRS_ERR_CUDA;
    }
    RglruScanFwdArgs a{};
    a.g = make_geom(B, L, D, kRgTile);
    a.alpha = alpha;
    a.bx = b_x;
    a.ba = b_a;
    a.wimg = at<uint8_t>(scratch, ps.wimg);
    a.reset = reset;
    a.h0 = h0;
    a.y = static_cast<uint32_t*>(y);
    a.y32 = y32;
    a.hT = hT;
    a.hsub = at<float>(saved, sv.hsub);
    a.agg = at<float2>(scratch, sc.agg);
    a.flags = at<uint32_t>(scratch, sc.flags);
    a.counter = at<uint32_t>(scratch, sc.status + 4);
    a.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_RGLRU_SCAN_FWD, stream, launch_rglru_scan_fwd(tm_x, tm_lx, tm_la, a, stream, fused ? 2 : 1));
    return LRS_OK;
}

int rglru_proj_backward(const void* dy, const float* dhT, const void* x, const void* w_x, const float* b_x,
                        const void* w_a, const float* b_a, const float* alpha, const float* h0,
                        const uint8_t* reset, int B, int L, int D, const void* saved, void* dx, int grad_dtype,
                        float* dw_x, float* db_x, float* dw_a, float* db_a, float* dalpha, float* dh0,
                        void* scratch, cudaStream_t stream) {
    (void)h0;
    const int st = check_rglru_proj_shape(B, L, D);
    if (st != LRS_OK) return st;
    if (grad_dtype != LRS_GRAD_BF16 && grad_dtype != LRS_GRAD_FP32) return LRS_ERR_ARG;
    if (!req(dy) || !opt(dhT) || !req(x) || !req(w_x) || !req(b_x) || !req(w_a) || !req(b_a) || !req(alpha) ||
        !req(saved) || !req(dx) || !req(dw_x) || !req(db_x) || !req(dw_a) || !req(db_a) || !req(dalpha) ||
        !req(dh0) || !req(scratch))
        return LRS_ERR_ARG;
    const RglruSaved sv = rglru_saved_layout(B, L, D);
    const RglruProjScratch ps = rglru_proj_scratch_layout(B, L, D);
    const RglruScratch& sc = ps.scan;
    const ScanGeom g = make_geom(B, L, D, kRgTile);
    float* lx = at<float>(scratch, ps.lx);
    float* la = at<float>(scratch, ps.la);
    const bool fp32 = grad_dtype == LRS_GRAD_FP32;
    const ProjDims pd = proj_dims(B, L, D);
    const int dk = pd.dk;
    uint32_t* status = at<uint32_t>(scratch, sc.status);
    // the logits formed again in the scan kernel on the tensor cores when the
    // diagonal blocks tile the 64-channel groups, as in the forward; otherwise
    // by the logits contraction
    const bool fused = 64 % dk == 0;
    if (cudaMemsetAsync(scratch, 0, sc.memset_bytes, stream) != cudaSuccess) return LRS_ERR_CUDA;
    LRS_LAUNCH(KID_RGLRU_PROJ_PACK, stream,
               launch_proj_pack(w_x, w_a, at<void>(scratch, ps.wt), at<void>(scratch, ps.wc), pd, stream));
    CUtensorMap tm_dy, tm_x, tm_lx, tm_la;
    if (!make_bf16_map(&tm_dy, dy, B, L, D, kRgTile)) return LRS_ERR_CUDA;
    if (fused) {
        LRS_LAUNCH(KID_RGLRU_PROJ_PACK, stream, launch_rglru_proj_wimg(w_x, w_a, at<void>(scratch, ps.wimg), D, stream));
        if (!make_bf16_map_sw128(&tm_x, x, B, L, D, kRgTile)) return LRS_ERR_CUDA;
        tm_lx = tm_x;
        tm_la = tm_x;
    } else {
        LRS_LAUNCH(KID_RGLRU_PROJ_FWD, stream,
                   launch_proj_logits(x, at<void>(scratch, ps.wt), lx, la, D, pd, status, stream, false));
        if (!make_bf16_map(&tm_x, x, B, L, D, kRgTile) || !make_f32_map(&tm_lx, lx, B, L, D, kRgTile) ||
            !make_f32_map(&tm_la, la, B, L, D, kRgTile))
            return LRS_ERR_CUDA;
    }
    RglruScanBwdArgs a{};
    a.g = g;
    a.alpha = alpha;
    a.bx = b_x;
    a.ba = b_a;
    a.reset = reset;
    a.dhT = dhT;
    a.hsub = at<float>(saved, sv.hsub);
    a.dx = nullptr;
    a.dlx = nullptr;
    a.dla = nullptr;
    a.gparts = at<uint32_t>(scratch, ps.gparts);
    a.dk = dk;
    a.wimg = at<uint8_t>(scratch, ps.wimg);
    a.bxpart = at<float>(scratch, ps.bxpart);
    a.bapart = at<float>(scratch, ps.bapart);
    a.grad_fp32 = 1;
    a.dh0 = dh0;
    a.agg = at<float2>(scratch, sc.agg);
    a.rin = at<float>(scratch, sc.rin);
    a.apart = at<float>(scratch, sc.apart);
    a.flags = at<uint32_t>(scratch, sc.flags);
    a.counter = at<uint32_t>(scratch, sc.status + 4);
    a.status = at<uint32_t>(scratch, sc.status);
    LRS_LAUNCH(KID_RGLRU_SCAN_BWD, stream, launch_rglru_scan_bwd(tm_dy, tm_x, tm_lx, tm_la, a, stream, fused ? 2 : 1));
    float* apart2 = at<float>(scratch, sc.apart2);
    LRS_LAUNCH(KID_RGLRU_ALPHA, stream, launch_rglru_alpha(a.apart, apart2, dalpha, B * g.CT, D, stream));
    LRS_LAUNCH(KID_RGLRU_ALPHA, stream, launch_rglru_alpha(a.bxpart, apart2, db_x, B * g.CT, D, stream));
    LRS_LAUNCH(KID_RGLRU_ALPHA, stream, launch_rglru_alpha(a.bapart, apart2, db_a, B * g.CT, D, stream));
    LRS_LAUNCH(KID_RGLRU_PROJ_BWD, stream,
               launch_proj_dx(a.gparts, at<void>(scratch, ps.wc), dx, fp32, D, pd, status, stream, false));
    LRS_LAUNCH(KID_RGLRU_PROJ_BWD, stream,
               launch_proj_dw(a.gparts, x, at<float>(scratch, ps.dwpart), dw_x, dw_a, D, pd, status, stream, false));
    return LRS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// RecurrentBlock around a mixer: SAMU (samu_block_*) or, for the pages'
// comparison, the RG-LRU with its gate projections (rglru_block_*).  The
// block's own layers are the same; only the mixer calls differ.
// ---------------------------------------------------------------------------
namespace {

int check_block_widths(int B, int L, int Dm, int D) {
    if (Dm % 256 != 0 || D % 256 != 0 || Dm > 4096) return LRS_ERR_UNSUPPORTED;
    if ((long long)B * L >= (1LL << 31)) return LRS_ERR_UNSUPPORTED;
    return LRS_OK;
}

int check_block_shape(int B, int L, int Dm, int D) {
    if (Dm < 1) return LRS_ERR_ARG;
    const int st = check_samu_shape(B, L, D);
    return st != LRS_OK ? st : check_block_widths(B, L, Dm, D);
}

int check_rglru_block_shape(int B, int L, int Dm, int D) {
    if (Dm < 1) return LRS_ERR_ARG;
    const int st = check_rglru_proj_shape(B, L, D);
    return st != LRS_OK ? st : check_block_widths(B, L, Dm, D);
}

// The block's own parameters and their gradients (both block kinds).
struct BlockCore {
    const float* gamma1;
    const void* w_in;
    const float* conv_k;
    const float* conv_b;
    const void* w_o;
    const float* gamma2;
    const void* w_mlp_in;
    const void* w_mlp_out;
};
struct BlockCoreGrads {
    float *dgamma1, *dw_in, *dconv_k, *dconv_b, *dw_o, *dgamma2, *dw_mlp_in, *dw_mlp_out;
};

bool core_ok(const BlockCore& p) {
    return req(p.gamma1) && req(p.w_in) && req(p.conv_k) && req(p.conv_b) && req(p.w_o) && req(p.gamma2) &&
           req(p.w_mlp_in) && req(p.w_mlp_out);
}
bool core_grads_ok(const BlockCoreGrads& g) {
    return req(g.dgamma1) && req(g.dw_in) && req(g.dconv_k) && req(g.dconv_b) && req(g.dw_o) && req(g.dgamma2) &&
           req(g.dw_mlp_in) && req(g.dw_mlp_out);
}

// The mixer's buffers inside the block's: its saved and scratch bytes and
// the offset of its status word in its scratch.
struct MixerSizes {
    size_t saved, scratch, status;
};
MixerSizes samu_mixer_sizes(int B, int L, int D) {
    return {samu_saved_layout(B, L, D).total, samu_scratch_layout(B, L, D).total, samu_scratch_layout(B, L, D).status};
}
MixerSizes rglru_mixer_sizes(int B, int L, int D) {
    const RglruProjScratch ps = rglru_proj_scratch_layout(B, L, D);
    return {rglru_saved_layout(B, L, D).total, ps.total, ps.scan.status};
}

// The four weight-gradient contractions (rows M x columns N of the gradient).
struct BlockDw {
    int M, N;
};
void block_dws(int Dm, int D, BlockDw (&w)[4]) {
    const int F = kBlockMlpRatio * Dm;
    w[0] = {Dm, F};        // w_mlp_out
    w[1] = {2 * F, Dm};    // w_mlp_in
    w[2] = {Dm, D};        // w_o
    w[3] = {2 * D, Dm};    // w_in
}

BlockScratch block_scratch(int B, int L, int Dm, int D, size_t mixer_scratch) {
    BlockDw w[4];
    block_dws(Dm, D, w);
    size_t wp = 0;
    for (const BlockDw& d : w) {
        const int sp = block_gemm_splits_bound(d.M, d.N, (long long)B * L);
        if (sp > 1) wp = std::max(wp, (size_t)sp * d.M * d.N);
    }
    const size_t np = (size_t)block_norm_bwd_ctas((long long)B * L) * Dm;
    const size_t cp = (size_t)block_conv_parts(B, L) * 5 * D;
    return block_scratch_layout(B, L, Dm, D, mixer_scratch, wp, np, cp);
}

BlockGemmArgs gemm_args(int layout, int epi, int M, int N, int K, uint32_t* status) {
    BlockGemmArgs g{};
    g.layout = layout;
    g.epi = epi;
    g.M = M;
    g.N = N;
    g.K = K;
    g.splits = 1;
    g.status = status;
    return g;
}

// dW [M][N] = A^T B over the tokens: split partials into wpart and a fixed-order
// sum, or straight into dw with one split.
int block_weight_grad(const void* A, const void* Bm, int M, int N, long long BL, float* dw, float* wpart,
                      uint32_t* status, cudaStream_t stream) {
    BlockGemmArgs g = gemm_args(kBgTN, kEpiF32, M, N, (int)BL, status);
    g.splits = block_gemm_splits(M, N, BL, block_gemm_sms());
    g.part = g.splits > 1 ? wpart : dw;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, A, Bm, stream, pdl_ok()));
    if (g.splits > 1)
        LRS_LAUNCH(KID_BLOCK_SUM, stream,
                   launch_sum_parts(wpart, (long long)M * N, g.splits, (long long)M * N, dw, stream, pdl_ok()));
    return LRS_OK;
}

// Block forward around mix(u, y_mixer, mixer saved, mixer scratch) -> status.
template <class Mix>
int block_forward_impl(const BlockCore& p, const void* x, const uint8_t* reset, int B, int L, int Dm, int D,
                       void* out, void* saved, void* scratch, const MixerSizes& ms, Mix mix, cudaStream_t stream) {
    const long long BL = (long long)B * L;
    const int F = kBlockMlpRatio * Dm;
    const BlockSaved sv = block_saved_layout(B, L, Dm, D, ms.saved);
    const BlockScratch sc = block_scratch(B, L, Dm, D, ms.scratch);
    uint32_t* status = at<uint32_t>(scratch, 0);
    void* msaved = at<void>(saved, sv.mixer);
    void* mscratch = at<void>(scratch, sc.mixer);
    const uint32_t* mstatus = at<uint32_t>(mscratch, ms.status);
    void* h1 = at<void>(saved, sv.h1);
    float* rstd1 = at<float>(saved, sv.rstd1);
    void* gv = at<void>(saved, sv.gv);
    void* u = at<void>(saved, sv.u);
    void* ym = at<void>(saved, sv.ym);
    void* j = at<void>(saved, sv.j);
    void* r1 = at<void>(saved, sv.r1);
    float* rstd2 = at<float>(saved, sv.rstd2);
    void* h2 = at<void>(saved, sv.h2);
    void* ab = at<void>(saved, sv.ab);
    void* q = at<void>(saved, sv.q);

    // h1 = RMSNorm(x); [g | v] = h1 w_in^T; u = conv(v)
    LRS_LAUNCH(KID_BLOCK_NORM, stream, launch_rmsnorm_fwd(x, p.gamma1, h1, rstd1, BL, Dm, status, stream, false));
    BlockGemmArgs g = gemm_args(kBgNT, kEpiStore, (int)BL, 2 * D, Dm, status);
    g.out = static_cast<uint16_t*>(gv);
    g.ldo = 2 * D;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, h1, p.w_in, stream, pdl_ok()));
    LRS_LAUNCH(KID_BLOCK_CONV, stream, launch_conv_fwd(gv, p.conv_k, p.conv_b, reset, u, B, L, D, stream, pdl_ok()));
    const int st = mix(u, ym, msaved, mscratch);
    if (st != LRS_OK) return st;
    // j = GeLU(g) y_mix; r1 = x + j w_o^T
    LRS_LAUNCH(KID_BLOCK_JOIN, stream, launch_join_fwd(gv, ym, j, BL, D, status, mstatus, stream, pdl_ok()));
    g = gemm_args(kBgNT, kEpiResid, (int)BL, Dm, D, status);
    g.out = static_cast<uint16_t*>(r1);
    g.ldo = Dm;
    g.r = static_cast<const uint16_t*>(x);
    g.ldr = Dm;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, j, p.w_o, stream, pdl_ok()));
    // h2 = RMSNorm(r1); [a | b] = h2 w_mlp_in^T, q = GeLU(a) b; out = r1 + q w_mlp_out^T
    LRS_LAUNCH(KID_BLOCK_NORM, stream, launch_rmsnorm_fwd(r1, p.gamma2, h2, rstd2, BL, Dm, nullptr, stream, pdl_ok()));
    g = gemm_args(kBgNT, kEpiGlu, (int)BL, F, Dm, status);
    g.out = static_cast<uint16_t*>(q);
    g.ldo = F;
    g.out2 = static_cast<uint16_t*>(ab);
    g.ld2 = 2 * F;
    g.F = F;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, h2, p.w_mlp_in, stream, pdl_ok()));
    g = gemm_args(kBgNT, kEpiResid, (int)BL, Dm, F, status);
    g.out = static_cast<uint16_t*>(out);
    g.ldo = Dm;
    g.r = static_cast<const uint16_t*>(r1);
    g.ldr = Dm;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, q, p.w_mlp_out, stream, pdl_ok()));
    return LRS_OK;
}

// Block backward around mixb(dy_mixer, u, mixer saved, dxs, dwm, mixer
// scratch) -> status, which writes the mixer's input gradient(s) w.r.t. u:
// dxs, and dwm when two_grads (SAMU: x_sel = w = u).
template <class MixB>
int block_backward_impl(const BlockCore& p, const BlockCoreGrads& gr, const void* x, const uint8_t* reset,
                        const void* dout, int B, int L, int Dm, int D, const void* saved, void* dx, void* scratch,
                        const MixerSizes& ms, bool two_grads, MixB mixb, cudaStream_t stream) {
    const long long BL = (long long)B * L;
    const int F = kBlockMlpRatio * Dm;
    const BlockSaved sv = block_saved_layout(B, L, Dm, D, ms.saved);
    const BlockScratch sc = block_scratch(B, L, Dm, D, ms.scratch);
    uint32_t* status = at<uint32_t>(scratch, 0);
    const void* msaved = at<void>(saved, sv.mixer);
    void* mscratch = at<void>(scratch, sc.mixer);
    const uint32_t* mstatus = at<uint32_t>(mscratch, ms.status);
    const void* h1 = at<void>(saved, sv.h1);
    const float* rstd1 = at<float>(saved, sv.rstd1);
    const void* gv = at<void>(saved, sv.gv);
    const void* u = at<void>(saved, sv.u);
    const void* ym = at<void>(saved, sv.ym);
    const void* j = at<void>(saved, sv.j);
    const void* r1 = at<void>(saved, sv.r1);
    const float* rstd2 = at<float>(saved, sv.rstd2);
    const void* h2 = at<void>(saved, sv.h2);
    const void* ab = at<void>(saved, sv.ab);
    const void* q = at<void>(saved, sv.q);
    void* dab = at<void>(scratch, sc.dab);
    void* dh2 = at<void>(scratch, sc.dh2);
    void* dr1 = at<void>(scratch, sc.dr1);
    void* dym = at<void>(scratch, sc.dym);
    void* dgv = at<void>(scratch, sc.dgv);
    void* dxs = at<void>(scratch, sc.dxs);
    void* dwm = at<void>(scratch, sc.dwm);
    void* dh1 = at<void>(scratch, sc.dh1);
    float* wpart = at<float>(scratch, sc.wpart);
    float* npart = at<float>(scratch, sc.npart);
    float* cpart = at<float>(scratch, sc.cpart);
    const int ncta = block_norm_bwd_ctas(BL);
    int st;

    if (cudaMemsetAsync(status, 0, 16, stream) != cudaSuccess) return LRS_ERR_CUDA;
    // gated MLP: dq = dout w_mlp_out -> [da | db]; dW_mlp_out = dout^T q
    BlockGemmArgs g = gemm_args(kBgNN, kEpiGluBwd, (int)BL, F, Dm, status);
    g.out = static_cast<uint16_t*>(dab);
    g.ldo = 2 * F;
    g.e0 = static_cast<const uint16_t*>(ab);
    g.lde0 = 2 * F;
    g.F = F;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, dout, p.w_mlp_out, stream, false));
    if ((st = block_weight_grad(dout, q, Dm, F, BL, gr.dw_mlp_out, wpart, status, stream)) != LRS_OK) return st;
    // dh2 = [da | db] w_mlp_in; dW_mlp_in = [da | db]^T h2
    g = gemm_args(kBgNN, kEpiStore, (int)BL, Dm, 2 * F, status);
    g.out = static_cast<uint16_t*>(dh2);
    g.ldo = Dm;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, dab, p.w_mlp_in, stream, pdl_ok()));
    if ((st = block_weight_grad(dab, h2, 2 * F, Dm, BL, gr.dw_mlp_in, wpart, status, stream)) != LRS_OK) return st;
    // dr1 = dout + RMSNorm'(dh2)
    LRS_LAUNCH(KID_BLOCK_NORM, stream,
               launch_rmsnorm_bwd(r1, p.gamma2, rstd2, dh2, dout, dr1, npart, BL, Dm, nullptr, stream, pdl_ok()));
    LRS_LAUNCH(KID_BLOCK_SUM, stream, launch_sum_parts(npart, Dm, ncta, Dm, gr.dgamma2, stream, pdl_ok()));
    // join: dj = dr1 w_o -> dy_mix, dg; dW_o = dr1^T j
    g = gemm_args(kBgNN, kEpiJoinBwd, (int)BL, D, Dm, status);
    g.out = static_cast<uint16_t*>(dym);
    g.ldo = D;
    g.out2 = static_cast<uint16_t*>(dgv);
    g.ld2 = 2 * D;
    g.e0 = static_cast<const uint16_t*>(gv);
    g.lde0 = 2 * D;
    g.e1 = static_cast<const uint16_t*>(ym);
    g.lde1 = D;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, dr1, p.w_o, stream, pdl_ok()));
    if ((st = block_weight_grad(dr1, j, Dm, D, BL, gr.dw_o, wpart, status, stream)) != LRS_OK) return st;
    // the mixer: its input gradient(s) w.r.t. u
    st = mixb(dym, u, msaved, dxs, dwm, mscratch);
    if (st != LRS_OK) return st;
    // convolution: dv (the recurrent half of [dg | dv]), dconv_k, dconv_b
    const int cparts = block_conv_parts(B, L);
    LRS_LAUNCH(KID_BLOCK_CONV, stream,
               launch_conv_bwd(gv, p.conv_k, reset, dxs, two_grads ? dwm : nullptr, dgv, cpart, B, L, D, status,
                               mstatus, stream, pdl_ok()));
    LRS_LAUNCH(KID_BLOCK_SUM, stream,
               launch_sum_parts(cpart, 5LL * D, cparts, 4LL * D, gr.dconv_k, stream, pdl_ok()));
    LRS_LAUNCH(KID_BLOCK_SUM, stream,
               launch_sum_parts(cpart + 4 * (size_t)D, 5LL * D, cparts, D, gr.dconv_b, stream, pdl_ok()));
    // dh1 = [dg | dv] w_in; dW_in = [dg | dv]^T h1
    g = gemm_args(kBgNN, kEpiStore, (int)BL, Dm, 2 * D, status);
    g.out = static_cast<uint16_t*>(dh1);
    g.ldo = Dm;
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, dgv, p.w_in, stream, pdl_ok()));
    if ((st = block_weight_grad(dgv, h1, 2 * D, Dm, BL, gr.dw_in, wpart, status, stream)) != LRS_OK) return st;
    // dx = dr1 + RMSNorm'(dh1)
    LRS_LAUNCH(KID_BLOCK_NORM, stream,
               launch_rmsnorm_bwd(x, p.gamma1, rstd1, dh1, dr1, dx, npart, BL, Dm, nullptr, stream, pdl_ok()));
    LRS_LAUNCH(KID_BLOCK_SUM, stream, launch_sum_parts(npart, Dm, ncta, Dm, gr.dgamma1, stream, pdl_ok()));
    return LRS_OK;
}

BlockCore core_of(const samu_block_params* p) {
    return {p->gamma1, p->w_in, p->conv_k, p->conv_b, p->w_o, p->gamma2, p->w_mlp_in, p->w_mlp_out};
}
BlockCore core_of(const rglru_block_params* p) {
    return {p->gamma1, p->w_in, p->conv_k, p->conv_b, p->w_o, p->gamma2, p->w_mlp_in, p->w_mlp_out};
}
BlockCoreGrads core_of(const samu_block_grads* g) {
    return {g->dgamma1, g->dw_in, g->dconv_k, g->dconv_b, g->dw_o, g->dgamma2, g->dw_mlp_in, g->dw_mlp_out};
}
BlockCoreGrads core_of(const rglru_block_grads* g) {
    return {g->dgamma1, g->dw_in, g->dconv_k, g->dconv_b, g->dw_o, g->dgamma2, g->dw_mlp_in, g->dw_mlp_out};
}

}  // namespace

extern "C" {

int samu_block_workspace_bytes(int B, int L, int Dm, int D, size_t* saved_bytes, size_t* scratch_bytes) {
    const int st = check_block_shape(B, L, Dm, D);
    if (st != LRS_OK) return st;
    const MixerSizes ms = samu_mixer_sizes(B, L, D);
    if (saved_bytes != nullptr) *saved_bytes = block_saved_layout(B, L, Dm, D, ms.saved).total;
    if (scratch_bytes != nullptr) *scratch_bytes = block_scratch(B, L, Dm, D, ms.scratch).total;
    return LRS_OK;
}

int samu_block_forward(const samu_block_params* p, const void* x, const float* h0, const uint8_t* reset, int B,
                       int L, int Dm, int D, void* out, float* hT, void* saved, void* scratch, cudaStream_t stream) {
    const int st0 = check_block_shape(B, L, Dm, D);
    if (st0 != LRS_OK) return st0;
    if (p == nullptr || !core_ok(core_of(p)) || !req(p->nu) || !req(p->theta) || !req(p->w_phi) || !req(p->w_r) ||
        p->a_phi == nullptr || p->a_r == nullptr || !req(x) || !opt(h0) || !req(out) || !req(hT) || !req(saved) ||
        !req(scratch))
        return LRS_ERR_ARG;
    // the mixer on x_sel = w = u
    auto mix = [&](const void* u, void* ym, void* msaved, void* mscratch) {
        return samu_forward(u, u, h0, reset, p->nu, p->theta, p->w_phi, p->w_r, p->a_phi, p->a_r, B, L, D, ym,
                            nullptr, hT, msaved, mscratch, stream);
    };
    return block_forward_impl(core_of(p), x, reset, B, L, Dm, D, out, saved, scratch, samu_mixer_sizes(B, L, D), mix,
                              stream);
}

int samu_block_backward(const samu_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                        const void* dout, const float* dhT, int B, int L, int Dm, int D, const void* saved, void* dx,
                        float* dh0, const samu_block_grads* gr, void* scratch, cudaStream_t stream) {
    const int st0 = check_block_shape(B, L, Dm, D);
    if (st0 != LRS_OK) return st0;
    if (p == nullptr || gr == nullptr || !core_ok(core_of(p)) || !core_grads_ok(core_of(gr)) || !req(p->nu) ||
        !req(p->theta) || !req(p->w_phi) || !req(p->w_r) || p->a_phi == nullptr || p->a_r == nullptr ||
        !req(gr->dnu) || !req(gr->dtheta) || !req(gr->dw_phi) || !req(gr->dw_r) || gr->da_phi == nullptr ||
        gr->da_r == nullptr || !req(x) || !opt(h0) || !req(dout) || !opt(dhT) || !req(saved) || !req(dx) ||
        !req(dh0) || !req(scratch))
        return LRS_ERR_ARG;
    // the mixer (x_sel = w = u): both of its input gradients reach u
    auto mixb = [&](const void* dym, const void* u, const void* msaved, void* dxs, void* dwm, void* mscratch) {
        return samu_backward(dym, dhT, u, u, h0, reset, p->nu, p->theta, p->w_phi, p->w_r, p->a_phi, p->a_r, B, L,
                             D, msaved, dxs, dwm, LRS_GRAD_BF16, dh0, gr->dnu, gr->dtheta, gr->dw_phi, gr->dw_r,
                             gr->da_phi, gr->da_r, mscratch, stream);
    };
    return block_backward_impl(core_of(p), core_of(gr), x, reset, dout, B, L, Dm, D, saved, dx, scratch,
                               samu_mixer_sizes(B, L, D), true, mixb, stream);
}

int rglru_block_workspace_bytes(int B, int L, int Dm, int D, size_t* saved_bytes, size_t* scratch_bytes) {
    const int st = check_rglru_block_shape(B, L, Dm, D);
    if (st != LRS_OK) return st;
    const MixerSizes ms = rglru_mixer_sizes(B, L, D);
    if (saved_bytes != nullptr) *saved_bytes = block_saved_layout(B, L, Dm, D, ms.saved).total;
    if (scratch_bytes != nullptr) *scratch_bytes = block_scratch(B, L, Dm, D, ms.scratch).total;
    return LRS_OK;
}

int rglru_block_forward(const rglru_block_params* p, const void* x, const float* h0, const uint8_t* reset, int B,
                        int L, int Dm, int D, void* out, float* hT, void* saved, void* scratch, cudaStream_t stream) {
    const int st0 = check_rglru_block_shape(B, L, Dm, D);
    if (st0 != LRS_OK) return st0;
    if (p == nullptr || !core_ok(core_of(p)) || !req(p->w_x) || !req(p->b_x) || !req(p->w_a) || !req(p->b_a) ||
        !req(p->alpha) || !req(x) || !opt(h0) || !req(out) || !req(hT) || !req(saved) || !req(scratch))
        return LRS_ERR_ARG;
    auto mix = [&](const void* u, void* ym, void* msaved, void* mscratch) {
        return rglru_proj_forward(u, p->w_x, p->b_x, p->w_a, p->b_a, p->alpha, h0, reset, B, L, D, ym, nullptr, hT,
                                  msaved, mscratch, stream);
    };
    return block_forward_impl(core_of(p), x, reset, B, L, Dm, D, out, saved, scratch, rglru_mixer_sizes(B, L, D), mix,
                              stream);
}

int rglru_block_backward(const rglru_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                         const void* dout, const float* dhT, int B, int L, int Dm, int D, const void* saved, void* dx,
                         float* dh0, const rglru_block_grads* gr, void* scratch, cudaStream_t stream) {
    const int st0 = check_rglru_block_shape(B, L, Dm, D);
    if (st0 != LRS_OK) return st0;
    if (p == nullptr || gr == nullptr || !core_ok(core_of(p)) || !core_grads_ok(core_of(gr)) || !req(p->w_x) ||
        !req(p->b_x) || !req(p->w_a) || !req(p->b_a) || !req(p->alpha) || !req(gr->dw_x) || !req(gr->db_x) ||
        !req(gr->dw_a) || !req(gr->db_a) || !req(gr->dalpha) || !req(x) || !opt(h0) || !req(dout) || !opt(dhT) ||
        !req(saved) || !req(dx) || !req(dh0) || !req(scratch))
        return LRS_ERR_ARG;
    auto mixb = [&](const void* dym, const void* u, const void* msaved, void* dxs, void*, void* mscratch) {
        return rglru_proj_backward(dym, dhT, u, p->w_x, p->b_x, p->w_a, p->b_a, p->alpha, h0, reset, B, L, D,
                                   msaved, dxs, LRS_GRAD_BF16, gr->dw_x, gr->db_x, gr->dw_a, gr->db_a, gr->dalpha,
                                   dh0, mscratch, stream);
    };
    return block_backward_impl(core_of(p), core_of(gr), x, reset, dout, B, L, Dm, D, saved, dx, scratch,
                               rglru_mixer_sizes(B, L, D), false, mixb, stream);
}

int lrs_dense_gemm(int layout, const void* A, const void* Bm, void* C, int M, int N, int K, void* scratch,
                   cudaStream_t stream) {
    if (!req(A) || !req(Bm) || !req(C) || !req(scratch) || M < 1 || N < 1 || K < 1) return LRS_ERR_ARG;
    if (layout != LRS_GEMM_NT && layout != LRS_GEMM_NN && layout != LRS_GEMM_TN) return LRS_ERR_ARG;
    if (N % 256 != 0) return LRS_ERR_UNSUPPORTED;
    if (layout != LRS_GEMM_TN && K % 64 != 0) return LRS_ERR_UNSUPPORTED;
    if (layout == LRS_GEMM_TN && M % 128 != 0) return LRS_ERR_UNSUPPORTED;
    uint32_t* status = at<uint32_t>(scratch, 0);
    if (cudaMemsetAsync(status, 0, 16, stream) != cudaSuccess) return LRS_ERR_CUDA;
    BlockGemmArgs g = gemm_args(layout == LRS_GEMM_NT ? kBgNT : layout == LRS_GEMM_NN ? kBgNN : kBgTN,
                                layout == LRS_GEMM_TN ? kEpiF32 : kEpiStore, M, N, K, status);
    if (layout == LRS_GEMM_TN) {
        g.part = static_cast<float*>(C);
    } else {
        g.out = static_cast<uint16_t*>(C);
        g.ldo = N;
    }
    LRS_LAUNCH(KID_BLOCK_GEMM, stream, launch_block_gemm(g, A, Bm, stream, false));
    return LRS_OK;
}

}  // extern "C"

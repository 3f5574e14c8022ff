// samu_forward_noalloc: the SAMU forward for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at all and have no spare device buffer
// to lend as `saved`/`scratch`: a host application whose device memory is
// owned by its own pooled allocator (a direct cudaMalloc would bypass or
// fragment the pool), or a latency-critical loop where cudaMalloc's implicit
// device synchronisation is not acceptable.  For them this entry point runs
// the same forward kernels as samu_forward with every intermediate (the
// controller cache, the per-mode constants, the sub-chunk entry states, and
// the segment maps and entry states) placed in one fixed array in device
// memory, declared below.  The array is part of the library's device image:
// every GPU that loads the library holds LRS_NOALLOC_BYTES for it until the
// process exits.  The paper describes no such entry point.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the one part that must start at zero, the status word, is
// cleared by each call's first kernel (the controller forward, which ends
// before any later kernel of the call can record a failure there).  Two
// calls whose work overlaps on the GPU (different streams, or different host
// threads) race on the array and give undefined results.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "tmap.cuh"

using namespace lrs;

namespace {

// The fixed workspace.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_noalloc_ws[LRS_NOALLOC_BYTES];

// Device addresses of the workspace, one per CUDA context that has called
// in.  Contexts are told apart by their driver-assigned unique id (never
// reused within a process), so a context created after cudaDeviceReset, or a
// caller's own non-primary context, gets its own look-up instead of a stale
// address.
constexpr int kMaxContexts = 64;
struct CtxAddr {
    unsigned long long id;
    void* ptr;
};
std::mutex g_noalloc_mutex;
CtxAddr g_noalloc_addr[kMaxContexts];
int g_noalloc_n = 0;

PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
    static PFN_cuCtxGetCurrent_v4000 fn = []() -> PFN_cuCtxGetCurrent_v4000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    return fn;
}

PFN_cuCtxGetId_v12000 ctx_id_fn() {
    static PFN_cuCtxGetId_v12000 fn = []() -> PFN_cuCtxGetId_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    }();
    return fn;
}

// Unique id of the current context; false if there is none yet or the
// driver entry points are unavailable.
bool current_ctx_id(unsigned long long* id) {
    PFN_cuCtxGetCurrent_v4000 cur = ctx_current_fn();
    PFN_cuCtxGetId_v12000 gid = ctx_id_fn();
    if (cur == nullptr || gid == nullptr) return false;
    CUcontext ctx = nullptr;
    if (cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return gid(ctx, id) == CUDA_SUCCESS;
}

// Device address of the workspace in the current context.  The first call in
// a context does the set-up: one cudaGetSymbolAddress with that context
// current (which also binds the device's primary context if none was
// current), its return code checked, the address remembered under the
// context's id.
int noalloc_workspace(void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    unsigned long long id = 0;
    const bool have_id = current_ctx_id(&id);
    if (have_id) {
        for (int i = 0; i < g_noalloc_n; ++i) {
            if (g_noalloc_addr[i].id == id) {
                *out = g_noalloc_addr[i].ptr;
                return LRS_OK;
            }
        }
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return LRS_ERR_CUDA;
    // the look-up may have made the primary context current: read the id again
    if (have_id || current_ctx_id(&id)) {
        if (g_noalloc_n < kMaxContexts) g_noalloc_addr[g_noalloc_n++] = CtxAddr{id, p};
    }
    *out = p;
    return LRS_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Layout of the fixed array: the status word at offset 0 (a fixed place, so
// that samu_forward_noalloc_status needs no shape), samu_forward's saved
// layout from kAlign on, then the forward part of its scratch layout (segment
// maps, CTA maps).
constexpr size_t kNoallocStatus = 0;
constexpr size_t kNoallocSaved = kAlign;
size_t noalloc_scratch_offset(int B, int L, int D) {
    return kNoallocSaved + align_up(samu_saved_layout(B, L, D).total);
}

size_t noalloc_need(int B, int L, int D) {
    const int M = D / 2;
    const SamuScratch sc = samu_scratch_layout(B, L, D);
    return noalloc_scratch_offset(B, L, D) + sc.cmap +
           (size_t)B * (samu_seg_geom(B, L, M, 0).NSmax / kSegPerCta) * M * 16;
}

}  // namespace

extern "C" int samu_forward_noalloc(const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                                    const float* nu, const float* theta, const float* w_phi, const float* w_r,
                                    const float* a_phi, const float* a_r, int B, int L, int D, void* y,
                                    float* y32, float* hT, cudaStream_t stream) {
    if (B < 1 || L < 1 || D < 2 || (D & 1)) return LRS_ERR_ARG;
    if (D % 16 != 0 || D > 4096) return LRS_ERR_UNSUPPORTED;
    const auto req = [](const void* p) { return p != nullptr && al16(p); };
    const auto opt = [](const void* p) { return p == nullptr || al16(p); };
    if (!req(x_sel) || !req(w) || !opt(h0) || !req(nu) || !req(theta) || !req(w_phi) || !req(w_r) ||
        a_phi == nullptr || a_r == nullptr || !req(y) || !opt(y32) || !req(hT))
        return LRS_ERR_ARG;
    if (noalloc_need(B, L, D) > (size_t)LRS_NOALLOC_BYTES) return LRS_ERR_TOO_LARGE;

    // the same layout as samu_forward's saved + the forward part of its scratch
    const int M = D / 2;
    const SamuSaved sv = samu_saved_layout(B, L, D);
    const SamuScratch sc = samu_scratch_layout(B, L, D);
    void* base = nullptr;
    const int st = noalloc_workspace(&base);
    if (st != LRS_OK) return st;
    unsigned char* saved = static_cast<unsigned char*>(base) + kNoallocSaved;
    unsigned char* scratch = static_cast<unsigned char*>(base) + noalloc_scratch_offset(B, L, D);
    uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(base) + kNoallocStatus);

    float* wh = reinterpret_cast<float*>(saved + sv.wh);
    float* misc = reinterpret_cast<float*>(saved + sv.misc);
    float4* modes = reinterpret_cast<float4*>(saved + sv.modes);
    float* p = reinterpret_cast<float*>(saved + sv.p);
    float* r = reinterpret_cast<float*>(saved + sv.r);
    float4* ctrl = reinterpret_cast<float4*>(saved + sv.ctrl);
    float4* items = reinterpret_cast<float4*>(saved + sv.items);

    SamuCtrlFwdArgs cf;
    cf.BL = (long long)B * L;
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
    cf.status = status;
    if (launch_samu_ctrl_fwd(cf, stream, false) != cudaSuccess) return LRS_ERR_CUDA;

    CUtensorMap tm_w, tm_ctrl;
    if (!make_bf16_map(&tm_w, w, B, L, D, kMapRows) || !make_ctrl_map(&tm_ctrl, ctrl, B, L, kMapRows)) return LRS_ERR_CUDA;
    SamuScanFwdArgs a;
    a.g = samu_scan_geom(B, L, M, false);
    a.items = items;
    a.modes = modes;
    a.nu = nu;
    a.closed_form = samu_get_chunk_transition() == LRS_TRANSITION_CLOSED_FORM;
    a.h0 = h0;
    a.y = static_cast<uint32_t*>(y);
    a.y32 = y32;
    a.hT = hT;
    a.hsub = reinterpret_cast<float2*>(saved + sv.hsub);
    a.smap = reinterpret_cast<float4*>(scratch + sc.smap);
    a.cmap = reinterpret_cast<float4*>(scratch + sc.cmap);
    a.status = status;
    if (launch_samu_fwd_maps(tm_w, tm_ctrl, a, stream, true) != cudaSuccess) return LRS_ERR_CUDA;
    if (launch_samu_fwd_replay(tm_w, tm_ctrl, a, stream, true) != cudaSuccess) return LRS_ERR_CUDA;
    return LRS_OK;
}

// The status word of the most recent samu_forward_noalloc in the current
// context, read through the same cached address.
extern "C" int samu_forward_noalloc_status(int* status, cudaStream_t stream) {
    if (status == nullptr) return LRS_ERR_ARG;
    void* base = nullptr;
    const int st = noalloc_workspace(&base);
    if (st != LRS_OK) return st;
    return lrs_device_status(static_cast<unsigned char*>(base) + kNoallocStatus, status, stream);
}

namespace lrs {
// The status word of the fixed array in the current context (for the
// failure-path self-test, lrs_selftest_wait_timeout with no scratch).
int noalloc_status_word(uint32_t** out) {
    void* base = nullptr;
    const int st = noalloc_workspace(&base);
    if (st != LRS_OK) return st;
    *out = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(base) + kNoallocStatus);
    return LRS_OK;
}
}  // namespace lrs

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
// cleared by each call's first scan kernel.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on the array and give undefined results.
#include <mutex>

#include "kernels.cuh"
#include "tmap.cuh"

using namespace lrs;

namespace {

// The fixed workspace.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_noalloc_ws[LRS_NOALLOC_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the workspace on the current device, looked up once per
// device (the first call on a device does this set-up).
int noalloc_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LRS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LRS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return LRS_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LRS_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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

    // the same layout as samu_forward's saved + the forward part of its scratch
    const int M = D / 2;
    const SamuSaved sv = samu_saved_layout(B, L, D);
    const SamuScratch sc = samu_scratch_layout(B, L, D);
    const size_t scratch_off = align_up(sv.total);
    const size_t need = scratch_off + sc.cmap + (size_t)B * (samu_seg_geom(B, L, M, 0).NSmax / kSegPerCta) * M * 16;
    if (need > (size_t)LRS_NOALLOC_BYTES) return LRS_ERR_TOO_LARGE;

    void* base = nullptr;
    const int st = noalloc_workspace(&base);
    if (st != LRS_OK) return st;
    unsigned char* saved = static_cast<unsigned char*>(base);
    unsigned char* scratch = saved + scratch_off;

    float* wh = reinterpret_cast<float*>(saved + sv.wh);
    float* misc = reinterpret_cast<float*>(saved + sv.misc);
    float4* modes = reinterpret_cast<float4*>(saved + sv.modes);
    float* p = reinterpret_cast<float*>(saved + sv.p);
    float* r = reinterpret_cast<float*>(saved + sv.r);
    float4* ctrl = reinterpret_cast<float4*>(saved + sv.ctrl);

    SamuCtrlFwdArgs cf;
    cf.BL = (long long)B * L;
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
    cf.wh = wh;
    cf.misc = misc;
    cf.modes = modes;
    cf.status = reinterpret_cast<uint32_t*>(scratch + sc.status);
    if (launch_samu_ctrl_fwd(cf, stream, false) != cudaSuccess) return LRS_ERR_CUDA;

    CUtensorMap tm_w, tm_ctrl;
    if (!make_bf16_map(&tm_w, w, B, L, D, kMapRows) || !make_ctrl_map(&tm_ctrl, ctrl, B, L, kMapRows)) return LRS_ERR_CUDA;
    SamuScanFwdArgs a;
    a.g = samu_scan_geom(B, L, M, false);
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
    a.status = reinterpret_cast<uint32_t*>(scratch + sc.status);
    if (launch_samu_fwd_maps(tm_w, tm_ctrl, a, stream, true) != cudaSuccess) return LRS_ERR_CUDA;
    if (launch_samu_fwd_replay(tm_w, tm_ctrl, a, stream, true) != cudaSuccess) return LRS_ERR_CUDA;
    return LRS_OK;
}

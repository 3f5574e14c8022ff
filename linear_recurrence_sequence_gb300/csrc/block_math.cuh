// GeLU of the RecurrentBlock (tanh form, a reading: the pages name a gated
// MLP and a gate branch but print no activation), shared by its contraction
// epilogues and element-wise kernels.
//   GeLU(x) = x (1 + tanh u) / 2,  u = sqrt(2/pi) (x + 0.044715 x^3),
// through the logistic function: (1 + tanh u) / 2 = s = 1 / (1 + e^{-2u}) and
// 1 - tanh^2 u = 4 s (1 - s) with 1 - s = e^{-2u} s (no cancellation), so
//   GeLU(x) = x s,  GeLU'(x) = s + 2 x s (1 - s) sqrt(2/pi) (1 + 3 0.044715 x^2).
// e^{-2u} comes from __expf with its argument clamped at 80 (beyond it s is
// below 2e-35 either way, and e s stays finite).  The reciprocal of 1 + e >= 1
// is correctly rounded in GeLU itself and from the SFU (rcp.approx, about
// 2^-23 relative) in the form with the derivative: measured in the
// contraction epilogues, the SFU form made the two backward epilogues faster
// (223 against 239 us and 77 against 85 us per launch at B4 L4K Dm 1024)
// and the forward GLU epilogue slower (247 against 202 us).  Relative error
// about 2^-20 over |2u| <= 20 either way, far below a BF16 ulp.
#pragma once

#include "common.cuh"

namespace lrs {

constexpr float kGeluC = 0.7978845608028654f;   // sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ void gelu_fwd_grad(float x, float& g, float& dg) {
    const float u = kGeluC * (x + kGeluA * x * x * x);
    const float e = __expf(fminf(-2.f * u, 80.f));
    const float sg = rcp_approx(1.f + e);
    const float om = e * sg;
    g = x * sg;
    dg = sg + 2.f * x * sg * om * kGeluC * (1.f + 3.f * kGeluA * x * x);
}

__device__ __forceinline__ float gelu_fwd(float x) {
    const float u = kGeluC * (x + kGeluA * x * x * x);
    return x * __frcp_rn(1.f + __expf(fminf(-2.f * u, 80.f)));
}

}  // namespace lrs

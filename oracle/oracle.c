/*
 * FP64 CPU oracle for the SAMU recurrent mixer and the RG-LRU scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Every routine is the plain, sequential definition written out in double
 * precision: one token after another, one mode (or channel) after another,
 * with no chunking, no prefix hierarchy and no fusion.  Sources, cited by
 * page title and section:
 *   [SAMU page]   "SAMU 与 RG-LRU 的 H800 训练性能对比" (SAMU_GPU index page),
 *                 section 05 "SAMU 在 GPU 上如何运行" (controller, transition,
 *                 recurrence and adjoint equations) and section 04
 *                 "RG-LRU 在 GPU 上如何运行" (gate, recurrence, reset rule).
 *   [Protocol]    "Griffin 第 4、5 节 H800 对照协议", section "SAMU 的固定方程"
 *                 (M complex modes = 2M real states; wide branch split into
 *                 real and imaginary parts as w_t) and "RG-LRU 的固定方程"
 *                 (segment_pos == 0 cuts the old state and cancels the
 *                 first-token normalisation multiplier).
 *
 * Layout conventions (all arrays row-major, doubles unless stated):
 *   x_sel, w, dy, y, dx_sel, dw : [B][L][D];  channel m < M is the real part
 *                                 of mode m, channel M+m its imaginary part.
 *   h0, hT, dh0, dhT (SAMU)     : [B][M][2]  (re, im)
 *   reset                       : [B][L] bytes, nonzero = segment start, or NULL
 *   nu, theta                   : [M];  w_phi, w_r : [D+1] (last = bias weight)
 * Complex cotangents follow dL/dRe + i dL/dIm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Rounding helper for expected BF16 outputs.                               */
/* ------------------------------------------------------------------------ */

/* Round a double to the nearest bfloat16 value (8 significant bits, ties to
 * even) directly from double, and return its 16-bit pattern.  No detour
 * through float, so there is no double rounding. */
uint16_t oracle_bf16_rne(double v)
{
    if (v != v) return 0x7fc0;                       /* NaN */
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    int e;
    frexp(a, &e);                                     /* a = f * 2^e, f in [0.5,1) */
    int ulp_exp = (e - 1) - 7;                        /* 8 significant bits */
    if (ulp_exp < -133) ulp_exp = -133;               /* subnormal spacing */
    double q = ldexp(a, -ulp_exp);                    /* exact scaling */
    double r = nearbyint(q);                          /* default mode: ties to even */
    double m = ldexp(r, ulp_exp);
    float f = (m > 3.3895313892515355e38) ? INFINITY : (float)m;  /* exact */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t h = (uint16_t)(bits >> 16);
    if (signbit(v)) h |= 0x8000;
    return h;
}

void oracle_bf16_rne_array(const double* v, uint16_t* out, long n)
{
    for (long i = 0; i < n; ++i) out[i] = oracle_bf16_rne(v[i]);
}

/* ------------------------------------------------------------------------ */
/* SAMU controller ([SAMU page] section 05, controller equations).           */
/* ------------------------------------------------------------------------ */

/* Unit direction w_hat = w / ||w||_2, norm over all D+1 entries (bias
 * included), as in the definition of w_hat_phi and w_hat_r. */
static double unit_direction(const double* w, int n, double* w_hat)
{
    double s = 0.0;
    for (int j = 0; j < n; ++j) s += w[j] * w[j];
    double nrm = sqrt(s);
    for (int j = 0; j < n; ++j) w_hat[j] = w[j] / nrm;
    return nrm;
}

/* Per-token controls.  x_tilde = [x_sel; 1]; p = tanh(x_tilde . w_hat_phi),
 * r = tanh(x_tilde . w_hat_r); q(r) = r / (1 + r^2);
 * d = tanh(a_phi)/sqrt(M) * p;  c = tanh(a_r)/sqrt(M) * q(r);
 * E = e^c, C = cos d, S = sin d.   ctrl rows hold {p, r, E, C, S}. */
static void samu_controller(int L, int D, const double* x /* [L][D] */,
                            const double* wh_phi, const double* wh_r,
                            double a_phi, double a_r, double* ctrl /* [L][5] */)
{
    const int M = D / 2;
    const double amp_phi = tanh(a_phi) / sqrt((double)M);
    const double amp_r = tanh(a_r) / sqrt((double)M);
    for (int t = 0; t < L; ++t) {
        const double* xt = x + (size_t)t * D;
        double s_phi = wh_phi[D];   /* the appended constant 1 times the bias weight */
        double s_r = wh_r[D];
        for (int j = 0; j < D; ++j) {
            s_phi += xt[j] * wh_phi[j];
            s_r += xt[j] * wh_r[j];
        }
        double p = tanh(s_phi);
        double r = tanh(s_r);
        double q = r / (1.0 + r * r);
        double d = amp_phi * p;
        double c = amp_r * q;
        double* o = ctrl + (size_t)t * 5;
        o[0] = p;
        o[1] = r;
        o[2] = exp(c);
        o[3] = cos(d);
        o[4] = sin(d);
    }
}

/* Transition lambda_{t,m} = e^{-nu_m E_t} [(cos th C - sin th S) + i (sin th C + cos th S)]
 * ([SAMU page] section 05, transition equation).  A reset position has lambda = 0. */
static void samu_lambda(double nu, double th, const double* ctl, int is_reset,
                        double* lr, double* li)
{
    if (is_reset) { *lr = 0.0; *li = 0.0; return; }
    double E = ctl[2], C = ctl[3], S = ctl[4];
    double rho = exp(-nu * E);
    *lr = rho * (cos(th) * C - sin(th) * S);
    *li = rho * (sin(th) * C + cos(th) * S);
}

/* Forward: z_{t,m} = lambda_{t,m} z_{t-1,m} + b_{t,m}, b = w[t,m] + i w[t,M+m],
 * z_{-1} = h0, y_t = z_t (same halves layout as w), hT = z_{L-1}.
 * ctrl_out (optional) receives {p, r, E, C, S} per token: [B][L][5]. */
void oracle_samu_forward(int B, int L, int D,
                         const double* x_sel, const double* w,
                         const double* h0, const uint8_t* reset,
                         const double* nu, const double* theta,
                         const double* w_phi, const double* w_r,
                         double a_phi, double a_r,
                         double* y, double* hT, double* ctrl_out)
{
    const int M = D / 2;
    double* wh_phi = malloc(sizeof(double) * (D + 1));
    double* wh_r = malloc(sizeof(double) * (D + 1));
    double* ctrl = malloc(sizeof(double) * 5 * (size_t)(L > 0 ? L : 1));
    unit_direction(w_phi, D + 1, wh_phi);
    unit_direction(w_r, D + 1, wh_r);
    for (int b = 0; b < B; ++b) {
        const double* xb = x_sel + (size_t)b * L * D;
        const double* wb = w + (size_t)b * L * D;
        double* yb = y + (size_t)b * L * D;
        samu_controller(L, D, xb, wh_phi, wh_r, a_phi, a_r, ctrl);
        if (ctrl_out) memcpy(ctrl_out + (size_t)b * L * 5, ctrl, sizeof(double) * 5 * L);
        for (int m = 0; m < M; ++m) {
            double zr = h0 ? h0[((size_t)b * M + m) * 2 + 0] : 0.0;
            double zi = h0 ? h0[((size_t)b * M + m) * 2 + 1] : 0.0;
            for (int t = 0; t < L; ++t) {
                int rs = reset ? (reset[(size_t)b * L + t] != 0) : 0;
                double lr, li;
                samu_lambda(nu[m], theta[m], ctrl + (size_t)t * 5, rs, &lr, &li);
                double br = wb[(size_t)t * D + m];
                double bi = wb[(size_t)t * D + M + m];
                double nr = lr * zr - li * zi + br;
                double ni = lr * zi + li * zr + bi;
                zr = nr;
                zi = ni;
                yb[(size_t)t * D + m] = zr;
                yb[(size_t)t * D + M + m] = zi;
            }
            hT[((size_t)b * M + m) * 2 + 0] = zr;
            hT[((size_t)b * M + m) * 2 + 1] = zi;
        }
    }
    free(wh_phi);
    free(wh_r);
    free(ctrl);
}

/* Backward, by the hand-derived adjoint ([SAMU page] section 05, reverse
 * equations: zbar_{t-1} += conj(lambda_t) zbar_t, bbar_t = zbar_t;
 * cbar_t = sum_m cbar_{t,m}, dbar_t = sum_m dbar_{t,m};
 * pbar = dbar tanh(a_phi)/sqrt(M);  rbar = cbar tanh(a_r)/sqrt(M) (1-r^2)/(1+r^2)^2).
 *
 * With kappa_{t,m} = A_{t,m} conj(lambda_{t,m} z_{t-1,m}), A the total adjoint
 * of z_t, and lambda = exp(-nu E + i(theta + d)):
 *   dtheta_m += Im kappa,  dnu_m += -E_t Re kappa,
 *   dbar_t   += Im kappa,  Ebar_t += -nu_m Re kappa,  cbar_t = Ebar_t E_t.
 * Reset positions (lambda = 0, not a function of any input) contribute nothing
 * and cut the adjoint.  The controller chain rule runs through tanh, the
 * amplitudes and the unit-direction normalisation:
 *   dw = (dw_hat - w_hat (w_hat . dw_hat)) / ||w||.
 * All outputs are overwritten. */
void oracle_samu_backward(int B, int L, int D,
                          const double* x_sel, const double* w,
                          const double* h0, const uint8_t* reset,
                          const double* nu, const double* theta,
                          const double* w_phi, const double* w_r,
                          double a_phi, double a_r,
                          const double* dy, const double* dhT,
                          double* dx_sel, double* dw, double* dh0,
                          double* dnu, double* dtheta,
                          double* dw_phi, double* dw_r,
                          double* da_phi, double* da_r)
{
    const int M = D / 2;
    const size_t Ls = (size_t)(L > 0 ? L : 1);
    double* wh_phi = malloc(sizeof(double) * (D + 1));
    double* wh_r = malloc(sizeof(double) * (D + 1));
    double* dwh_phi = calloc(D + 1, sizeof(double));
    double* dwh_r = calloc(D + 1, sizeof(double));
    double* ctrl = malloc(sizeof(double) * 5 * Ls);
    double* zr = malloc(sizeof(double) * (Ls + 1));   /* z_{t-1} at index t */
    double* zi = malloc(sizeof(double) * (Ls + 1));
    double* dbar = malloc(sizeof(double) * Ls);
    double* Ebar = malloc(sizeof(double) * Ls);
    double n_phi = unit_direction(w_phi, D + 1, wh_phi);
    double n_r = unit_direction(w_r, D + 1, wh_r);
    const double sqM = sqrt((double)M);
    const double amp_phi = tanh(a_phi) / sqM;
    const double amp_r = tanh(a_r) / sqM;
    double acc_aphi = 0.0, acc_ar = 0.0;

    for (int m = 0; m < M; ++m) { dnu[m] = 0.0; dtheta[m] = 0.0; }

    for (int b = 0; b < B; ++b) {
        const double* xb = x_sel + (size_t)b * L * D;
        const double* wb = w + (size_t)b * L * D;
        const double* gb = dy + (size_t)b * L * D;
        const uint8_t* rb = reset ? reset + (size_t)b * L : NULL;
        samu_controller(L, D, xb, wh_phi, wh_r, a_phi, a_r, ctrl);
        for (int t = 0; t < L; ++t) { dbar[t] = 0.0; Ebar[t] = 0.0; }

        for (int m = 0; m < M; ++m) {
            /* forward states of this mode */
            zr[0] = h0 ? h0[((size_t)b * M + m) * 2 + 0] : 0.0;
            zi[0] = h0 ? h0[((size_t)b * M + m) * 2 + 1] : 0.0;
            for (int t = 0; t < L; ++t) {
                double lr, li;
                samu_lambda(nu[m], theta[m], ctrl + (size_t)t * 5, rb ? rb[t] != 0 : 0, &lr, &li);
                zr[t + 1] = lr * zr[t] - li * zi[t] + wb[(size_t)t * D + m];
                zi[t + 1] = lr * zi[t] + li * zr[t] + wb[(size_t)t * D + M + m];
            }
            /* reverse sweep */
            double Ar = dhT ? dhT[((size_t)b * M + m) * 2 + 0] : 0.0;
            double Ai = dhT ? dhT[((size_t)b * M + m) * 2 + 1] : 0.0;
            for (int t = L - 1; t >= 0; --t) {
                Ar += gb[(size_t)t * D + m];
                Ai += gb[(size_t)t * D + M + m];
                dw[((size_t)b * L + t) * D + m] = Ar;
                dw[((size_t)b * L + t) * D + M + m] = Ai;
                int rs = rb ? rb[t] != 0 : 0;
                if (rs) { Ar = 0.0; Ai = 0.0; continue; }
                double lr, li;
                samu_lambda(nu[m], theta[m], ctrl + (size_t)t * 5, 0, &lr, &li);
                /* u = lambda z_{t-1};  kappa = A conj(u) */
                double ur = lr * zr[t] - li * zi[t];
                double ui = lr * zi[t] + li * zr[t];
                double kr = Ar * ur + Ai * ui;
                double ki = Ai * ur - Ar * ui;
                double E = ctrl[(size_t)t * 5 + 2];
                dtheta[m] += ki;
                dnu[m] += -E * kr;
                dbar[t] += ki;
                Ebar[t] += -nu[m] * kr;
                /* A <- conj(lambda) A */
                double nr = lr * Ar + li * Ai;
                double ni = lr * Ai - li * Ar;
                Ar = nr;
                Ai = ni;
            }
            dh0[((size_t)b * M + m) * 2 + 0] = Ar;
            dh0[((size_t)b * M + m) * 2 + 1] = Ai;
        }

        /* controller backward, token by token */
        for (int t = 0; t < L; ++t) {
            const double* c5 = ctrl + (size_t)t * 5;
            double p = c5[0], r = c5[1], E = c5[2];
            double cbar = Ebar[t] * E;                      /* E = e^c */
            double pbar = dbar[t] * amp_phi;
            double opr = 1.0 + r * r;
            double rbar = cbar * amp_r * (1.0 - r * r) / (opr * opr);
            double sphi_bar = pbar * (1.0 - p * p);         /* through tanh */
            double sr_bar = rbar * (1.0 - r * r);
            const double* xt = xb + (size_t)t * D;
            double* dxt = dx_sel + ((size_t)b * L + t) * D;
            for (int j = 0; j < D; ++j) {
                dxt[j] = sphi_bar * wh_phi[j] + sr_bar * wh_r[j];
                dwh_phi[j] += sphi_bar * xt[j];
                dwh_r[j] += sr_bar * xt[j];
            }
            dwh_phi[D] += sphi_bar;
            dwh_r[D] += sr_bar;
            acc_aphi += dbar[t] * p / sqM;
            acc_ar += cbar * (r / opr) / sqM;
        }
    }

    /* through the unit-direction normalisation */
    double dot_phi = 0.0, dot_r = 0.0;
    for (int j = 0; j <= D; ++j) {
        dot_phi += wh_phi[j] * dwh_phi[j];
        dot_r += wh_r[j] * dwh_r[j];
    }
    for (int j = 0; j <= D; ++j) {
        dw_phi[j] = (dwh_phi[j] - wh_phi[j] * dot_phi) / n_phi;
        dw_r[j] = (dwh_r[j] - wh_r[j] * dot_r) / n_r;
    }
    double ta = tanh(a_phi), tr = tanh(a_r);
    *da_phi = acc_aphi * (1.0 - ta * ta);
    *da_r = acc_ar * (1.0 - tr * tr);

    free(wh_phi); free(wh_r); free(dwh_phi); free(dwh_r);
    free(ctrl); free(zr); free(zi); free(dbar); free(Ebar);
}

/* ------------------------------------------------------------------------ */
/* RG-LRU ([SAMU page] section 04; [Protocol] "RG-LRU 的固定方程").           */
/* ------------------------------------------------------------------------ */

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }
static double softplus(double v) { return v > 0 ? v + log1p(exp(-v)) : log1p(exp(v)); }

/* Derivative of the write normaliser sqrt(u), u = 1 - a^2, bounded at 1000
 * (the clipped square-root derivative of the canonical reference; the bound
 * itself is not printed on the pages). */
static double dsqrt_clipped(double u)
{
    double four_u = 4.0 * u;
    if (four_u < 1e-6) four_u = 1e-6;
    return 1.0 / sqrt(four_u);
}

/* Forward: g^x = sigmoid(l^x), g^a = sigmoid(l^a),
 * a = exp(-8 g^a softplus(alpha)), b = x g^x sqrt(max(1 - a^2, 0)),
 * h_t = a h_{t-1} + b.  At a segment start a = 0 and the normaliser is 1.
 * h0, hT : [B][D]. */
void oracle_rglru_forward(int B, int L, int D,
                          const double* x, const double* lx, const double* la,
                          const double* alpha, const double* h0, const uint8_t* reset,
                          double* y, double* hT)
{
    for (int b = 0; b < B; ++b) {
        for (int d = 0; d < D; ++d) {
            double sp = softplus(alpha[d]);
            double h = h0 ? h0[(size_t)b * D + d] : 0.0;
            for (int t = 0; t < L; ++t) {
                size_t i = ((size_t)b * L + t) * D + d;
                int rs = reset ? reset[(size_t)b * L + t] != 0 : 0;
                double gx = sigmoid(lx[i]);
                double ga = sigmoid(la[i]);
                double a = exp(-8.0 * ga * sp);
                double u = 1.0 - a * a;
                double nrm = sqrt(u > 0.0 ? u : 0.0);
                if (rs) { a = 0.0; nrm = 1.0; }
                h = a * h + x[i] * gx * nrm;
                y[i] = h;
            }
            hT[(size_t)b * D + d] = h;
        }
    }
}

/* Backward: H_t = dy_t + a_{t+1} H_{t+1} (H_{L-1} = dy + dhT);
 * dx = H g^x n;  dl^x = H x n g^x (1 - g^x);
 * abar = H h_{t-1} + H x g^x dn/da, dn/da = -2a dsqrt(1 - a^2) (not at resets);
 * dl^a = abar (-8 softplus(alpha)) a g^a (1 - g^a);
 * dalpha_d = sum abar (-8 g^a) sigmoid(alpha) a;  dh0 = a_0 H_0.
 * h0 may be NULL (zero).  dhT may be NULL (zero). */
void oracle_rglru_backward(int B, int L, int D,
                           const double* x, const double* lx, const double* la,
                           const double* alpha, const double* h0, const uint8_t* reset,
                           const double* dy, const double* dhT,
                           double* dx, double* dlx, double* dla,
                           double* dalpha, double* dh0)
{
    const size_t Ls = (size_t)(L > 0 ? L : 1);
    double* hs = malloc(sizeof(double) * (Ls + 1));    /* h_{t-1} at index t */
    for (int d = 0; d < D; ++d) dalpha[d] = 0.0;
    for (int b = 0; b < B; ++b) {
        for (int d = 0; d < D; ++d) {
            double sp = softplus(alpha[d]);
            double sa = sigmoid(alpha[d]);
            hs[0] = h0 ? h0[(size_t)b * D + d] : 0.0;
            for (int t = 0; t < L; ++t) {
                size_t i = ((size_t)b * L + t) * D + d;
                int rs = reset ? reset[(size_t)b * L + t] != 0 : 0;
                double gx = sigmoid(lx[i]);
                double ga = sigmoid(la[i]);
                double a = exp(-8.0 * ga * sp);
                double u = 1.0 - a * a;
                double nrm = sqrt(u > 0.0 ? u : 0.0);
                if (rs) { a = 0.0; nrm = 1.0; }
                hs[t + 1] = a * hs[t] + x[i] * gx * nrm;
            }
            double H = dhT ? dhT[(size_t)b * D + d] : 0.0;
            for (int t = L - 1; t >= 0; --t) {
                size_t i = ((size_t)b * L + t) * D + d;
                int rs = reset ? reset[(size_t)b * L + t] != 0 : 0;
                H += dy[i];
                double gx = sigmoid(lx[i]);
                double ga = sigmoid(la[i]);
                double a = exp(-8.0 * ga * sp);
                double u = 1.0 - a * a;
                double nrm = rs ? 1.0 : sqrt(u > 0.0 ? u : 0.0);
                dx[i] = H * gx * nrm;
                dlx[i] = H * x[i] * nrm * gx * (1.0 - gx);
                if (rs) {
                    dla[i] = 0.0;
                    H = 0.0;
                    continue;
                }
                double abar = H * hs[t] + H * x[i] * gx * (-2.0 * a) * dsqrt_clipped(u);
                dla[i] = abar * (-8.0 * sp) * a * ga * (1.0 - ga);
                dalpha[d] += abar * (-8.0 * ga) * sa * a;
                H = a * H;
            }
            dh0[(size_t)b * D + d] = H;
        }
    }
    free(hs);
}

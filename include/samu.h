/*
 * samu.h — C ABI of the GB300 (sm_103a) chunked affine scan library for the
 * SAMU recurrent mixer and the real RG-LRU scan.
 *
 * Sources (cited by page title and section):
 *   [SAMU page]  "SAMU 与 RG-LRU 的 H800 训练性能对比" (SAMU_GPU index page):
 *                section 05 "SAMU 在 GPU 上如何运行" — controller, transition
 *                lambda_{t,m}, complex recurrence, affine composition, forward
 *                and reverse (conjugate) passes, shared-control reduction;
 *                section 04 "RG-LRU 在 GPU 上如何运行" — gates, recurrence,
 *                reset rule, backward; section 02 glossary — "前向+反向" scope
 *                (backward returns the input, initial-state and all parameter
 *                gradients from a dense output cotangent).
 *   [Protocol]   "Griffin 第 4、5 节 H800 对照协议", "SAMU 的固定方程" (M complex
 *                modes = 2M real states, wide branch split into real and
 *                imaginary parts) and "RG-LRU 的固定方程" (segment start cuts
 *                the old state and cancels the normaliser).
 *   [Report]     "SAMU strengthened-baseline H800 report", "Reverse complex
 *                backward" (two shared controller-gradient partials per token,
 *                deterministic FP32 second stage).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA
 *    storage), row-major, contiguous, at least 16-byte aligned.
 *  - Shapes: B batch, L sequence length, D real state width, M = D / 2 complex
 *    modes.  [B,L,D] tensors put the real part of mode m in channel m and its
 *    imaginary part in channel M + m ("halves" layout).
 *  - BF16 tensors are passed as `const void*` / `void*` (IEEE bfloat16 bits).
 *    Complex FP32 states ([B,M,2]) are interleaved (re, im).
 *  - Ownership: the caller allocates every buffer, including `saved` (written
 *    by the forward, read by the backward) and `scratch`; sizes come from the
 *    *_workspace_bytes query.  The library never allocates, never frees and
 *    never synchronises the stream.
 *  - Every call is asynchronous on `stream`; outputs are overwritten, never
 *    accumulated.  A scratch buffer must not be used by two calls that may
 *    run concurrently.  `saved` must come from a forward with the same inputs.
 *  - Errors: the return value is a status code (LRS_OK = 0).  Argument checks
 *    happen on the host before anything is launched.  A device-side bounded
 *    wait that gives up is recorded in the scratch status word and reported by
 *    lrs_device_status() (LRS_ERR_TIMEOUT); the affected outputs are then
 *    undefined.  No C++ exception crosses this ABI.
 *  - Supported shapes: B >= 1, L >= 1.  SAMU: D % 16 == 0 and D <= 4096;
 *    RG-LRU: D % 8 == 0 (every measured width satisfies both).  Other even D
 *    return LRS_ERR_UNSUPPORTED: the tiles are fetched by TMA, whose innermost
 *    box coordinate must fall on a 16-byte boundary.
 */
#ifndef LRS_SAMU_H
#define LRS_SAMU_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define LRS_OK 0
#define LRS_ERR_ARG 1          /* null pointer, bad shape, misaligned pointer */
#define LRS_ERR_UNSUPPORTED 2  /* valid but unsupported shape (see "Supported shapes") */
#define LRS_ERR_CUDA 3         /* a kernel launch or memset failed */
#define LRS_ERR_TIMEOUT 4      /* a bounded device-side wait gave up */
#define LRS_ERR_TOO_LARGE 5    /* problem does not fit the fixed no-allocation workspace */

/* Gradient output dtype selector for the backward calls. */
#define LRS_GRAD_BF16 0
#define LRS_GRAD_FP32 1

/* Human-readable text for a status code (static storage).  samu_status_string
 * is the same function under the name the SAMU calls' documentation uses. */
const char* lrs_status_string(int status);
const char* samu_status_string(int status);

/* ABI version (major * 100 + minor). */
int lrs_version(void);

/* Reads the device status word kept in `scratch` (a buffer last used by one
 * of the calls below; every call clears the word when it starts, so it covers
 * the most recent call).  SYNCHRONISES `stream`.  *status receives LRS_OK or
 * LRS_ERR_TIMEOUT (LRS_ERR_CUDA if a kernel found its shared memory
 * misaligned and copied nothing).  Returns LRS_ERR_ARG / LRS_ERR_CUDA on failure. */
int lrs_device_status(void* scratch, int* status, cudaStream_t stream);

/* Self-test of the failure path of the bounded device-side waits: launches
 * one kernel whose wait on an mbarrier that nothing completes gives up at the
 * same deadline as the library's own waits (about 0.2 s), clears and then
 * sets the status word at the start of `scratch` (a buffer of at least 64
 * bytes, 16-byte aligned), and returns.  lrs_device_status then reports
 * LRS_ERR_TIMEOUT, and the context stays usable.  With scratch NULL the
 * kernel uses the status word of samu_forward_noalloc's fixed array in the
 * current context instead (samu_forward_noalloc_status then reports the
 * timeout).  Asynchronous on `stream`.
 * Errors: LRS_ERR_ARG (scratch misaligned), LRS_ERR_CUDA. */
int lrs_selftest_wait_timeout(void* scratch, cudaStream_t stream);

/* Opt-in per-kernel timing for benchmarks (not needed for computing).
 * lrs_profile_begin creates (once) `capacity` pairs of CUDA events and, until
 * lrs_profile_end, records one pair on the launching stream around every
 * kernel that the calls below launch (at most `capacity`).  lrs_profile_end
 * waits for the recorded events and writes, for the first min(count,
 * capacity) kernels, their id (2 controller forward, 3 SAMU forward replay,
 * 4 SAMU backward main, 5 controller backward, 6 SAMU parameter reductions,
 * 7 RG-LRU scan forward, 8 RG-LRU scan backward, 9 RG-LRU alpha reduction,
 * 10 SAMU forward maps, 11 SAMU backward maps, 12 SAMU decode prepare,
 * 13 SAMU decode step, 14 RG-LRU gate-projection GEMMs, 15 RG-LRU projection
 * backward GEMMs, 16 RG-LRU weight packing and dW combination, 17 RecurrentBlock
 * contractions, 18 RecurrentBlock RMSNorm (forward and backward), 19 its
 * convolution, 20 its join, 21 its fixed-order gradient sums; 9 also covers
 * the bias-gradient reductions) and duration in
 * milliseconds; *count receives the number of
 * kernels launched while profiling was on.  Not thread-safe: one profiling
 * session per process.  Errors: LRS_ERR_ARG (capacity < 1 or count NULL),
 * LRS_ERR_CUDA. */
int lrs_profile_begin(int capacity);
int lrs_profile_end(int* kernel_ids, float* ms, int capacity, int* count);

/* ======================================================================== */
/* SAMU mixer                                                                */
/* ======================================================================== */

/* How the SAMU maps kernels form the transition of a 16-token item.
 * CHAINED multiplies the per-token transitions one by one.  CLOSED_FORM uses
 * the item's two shared statistics instead ([SAMU page] section 05, "exact
 * chunk closed form"): prod_t lambda_{t,m} = lbar_m^16 e^{-nu_m G} e^{i D},
 * with G = sum_t (E_t - 1) and D = sum_t d_t over the item's tokens, and
 * lbar_m^16 formed in FP64.  An item that holds a reset, or is cut short by
 * the end of the sequence, is always chained.  Both give the same function
 * within FP32 rounding.  The setting is process-wide.  It applies to the
 * samu_forward / samu_backward calls made after it, including CUDA graphs
 * captured after it (a captured graph keeps the form it was captured with).
 * Any host thread may call it; each SAMU call reads the setting once.
 * Errors: LRS_ERR_ARG for an unknown kind. */
#define LRS_TRANSITION_CHAINED 0
#define LRS_TRANSITION_CLOSED_FORM 1
int samu_set_chunk_transition(int kind);
/* The current setting (LRS_TRANSITION_CLOSED_FORM unless changed). */
int samu_get_chunk_transition(void);

/* Bytes of the caller-owned `saved` buffer (forward -> backward) and of the
 * `scratch` buffer for problems of shape (B, L, D).  Either output pointer may
 * be NULL.  Pure host function. */
int samu_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes);

/* SAMU mixer forward ([SAMU page] section 05, forward):
 *   x~_t = [x_sel_t; 1]; w^_phi = w_phi/||w_phi||, w^_r = w_r/||w_r|| (norms over
 *   all D+1 entries); p_t = tanh(x~_t . w^_phi), r_t = tanh(x~_t . w^_r);
 *   d_t = tanh(a_phi)/sqrt(M) p_t; c_t = tanh(a_r)/sqrt(M) r_t/(1+r_t^2);
 *   E_t = e^{c_t}, C_t = cos d_t, S_t = sin d_t (once per token);
 *   lambda_{t,m} = e^{-nu_m E_t} [(cos th_m C_t - sin th_m S_t) + i(sin th_m C_t + cos th_m S_t)]
 *   (lambda = 0 where reset[b,t] != 0);
 *   z_{t,m} = lambda_{t,m} z_{t-1,m} + b_{t,m},  b_{t,m} = w[t,m] + i w[t,M+m],  z_{-1} = h0;
 *   y_t = z_t in the halves layout;  hT = z_{L-1}.
 *
 *   x_sel, w   [B,L,D] BF16 (in)
 *   h0         [B,M,2] FP32 (in) or NULL for zero
 *   reset      [B,L] uint8, nonzero = segment start (in) or NULL for none
 *   nu, theta  [M] FP32 (in);  w_phi, w_r [D+1] FP32 (in; last entry = bias)
 *   a_phi, a_r device pointers to one FP32 each (in)
 *   y          [B,L,D] BF16 (out, round to nearest even from the FP32 state)
 *   y32        [B,L,D] FP32 (out, optional: the pre-rounding value) or NULL
 *   hT         [B,M,2] FP32 (out)
 *   saved      samu_workspace_bytes().saved bytes (out: controller cache p, r,
 *              E/C/S, normalised directions and chunk entry states)
 *   scratch    samu_workspace_bytes().scratch bytes (temporary)
 * Errors: LRS_ERR_ARG for a NULL required pointer, non-positive shape, odd D,
 * or a tensor pointer not 16-byte aligned; LRS_ERR_UNSUPPORTED for
 * D % 16 != 0 or D > 4096; LRS_ERR_CUDA if a launch fails. */
int samu_forward(const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                 const float* nu, const float* theta, const float* w_phi, const float* w_r,
                 const float* a_phi, const float* a_r, int B, int L, int D,
                 void* y, float* y32, float* hT, void* saved, void* scratch,
                 cudaStream_t stream);

/* SAMU mixer backward ([SAMU page] section 05, backward; [Report] "Reverse
 * complex backward"): the conjugate reverse scan zbar_{t-1} += conj(lambda_t)
 * zbar_t with bbar_t = zbar_t, the per-token shared-control gradients
 * cbar_t = sum_m cbar_{t,m}, dbar_t = sum_m dbar_{t,m} (two FP32 partials per
 * mode slice, reduced in a fixed order), and the controller chain rule down to
 * x_sel and the parameters.
 *
 *   dy          [B,L,D] BF16 dense output cotangent (in)
 *   dhT         [B,M,2] FP32 cotangent of hT (in) or NULL for zero
 *   x_sel ... a_r, B, L, D: exactly the forward's inputs (in)
 *   saved       the forward's saved buffer (in)
 *   dx_sel, dw  [B,L,D] (out) in BF16 (grad_dtype = LRS_GRAD_BF16) or FP32
 *   dh0         [B,M,2] FP32 (out)
 *   dnu, dtheta [M] FP32 (out);  dw_phi, dw_r [D+1] FP32 (out)
 *   da_phi, da_r device pointers to one FP32 each (out)
 *   scratch     as for the forward (temporary)
 * Parameter gradients are deterministic (fixed reduction order).
 * Errors: as samu_forward, plus LRS_ERR_ARG for an unknown grad_dtype. */
int samu_backward(const void* dy, const float* dhT,
                  const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                  const float* nu, const float* theta, const float* w_phi, const float* w_r,
                  const float* a_phi, const float* a_r, int B, int L, int D,
                  const void* saved, void* dx_sel, void* dw, int grad_dtype,
                  float* dh0, float* dnu, float* dtheta, float* dw_phi, float* dw_r,
                  float* da_phi, float* da_r, void* scratch, cudaStream_t stream);

/* ======================================================================== */
/* SAMU single-token decode step                                              */
/* ======================================================================== */

/* Floats of the caller-owned decode parameter block for width D (pure host
 * function; the block must be 16-byte aligned).  Errors: LRS_ERR_ARG
 * (floats NULL), LRS_ERR_UNSUPPORTED (D as for samu_forward). */
int samu_decode_params_floats(int D, size_t* floats);

/* Prepares the per-parameter part of the decode step ([SAMU page] section 05:
 * w_hat = w / ||w|| over all D+1 entries, the amplitude factors
 * tanh(a)/sqrt(M), and lbar_m = e^{-nu_m} e^{i theta_m} formed in FP64) into
 * `params` (device, samu_decode_params_floats(D) floats).  Inputs as for
 * samu_forward.  Call again whenever the parameters change.  One launch,
 * asynchronous on `stream`. */
int samu_decode_prepare(const float* nu, const float* theta, const float* w_phi, const float* w_r,
                        const float* a_phi, const float* a_r, int D, float* params, cudaStream_t stream);

/* One token of each of B sequences ([SAMU page] section 05 applied to one
 * token with the carried state as z_{t-1}):  p, r, d, c, E, C, S from the
 * token's x_sel row; z_m <- lambda_m z_m + b_m (lambda = 0 where reset[b] != 0);
 * y = z in the halves layout.  Applying it token after token equals
 * samu_forward over the sequence.
 *
 *   x_sel, w    [B,D] BF16 (in): the token of every sequence
 *   state_in    [B,M,2] FP32 (in): z_{t-1};  state_out [B,M,2] FP32 (out),
 *               may be the same buffer as state_in (updated in place)
 *   reset       [B] uint8 (in) or NULL
 *   params      prepared by samu_decode_prepare (in)
 *   y           [B,D] BF16 (out);  y32 [B,D] FP32 (out) or NULL
 * One launch (one CTA per sequence), asynchronous on `stream`.
 * Errors: LRS_ERR_ARG (null or misaligned pointer, B < 1), LRS_ERR_UNSUPPORTED
 * (D as for samu_forward), LRS_ERR_CUDA. */
int samu_decode_step(const void* x_sel, const void* w, const float* state_in, float* state_out,
                     const uint8_t* reset, const float* params, int B, int D, void* y, float* y32,
                     cudaStream_t stream);

/* ======================================================================== */
/* RG-LRU (comparison path on the same engine)                               */
/* ======================================================================== */

int rglru_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes);

/* RG-LRU forward ([SAMU page] section 04; [Protocol] "RG-LRU 的固定方程"):
 *   g^x = sigmoid(lx), g^a = sigmoid(la), a_t = exp(-8 g^a softplus(alpha)),
 *   b_t = x_t g^x sqrt(max(1 - a_t^2, 0)); at a segment start a_t = 0 and the
 *   normaliser is 1; h_t = a_t h_{t-1} + b_t, h_{-1} = h0; y_t = h_t; hT = h_{L-1}.
 *
 *   x, lx, la  [B,L,D] BF16 (in);  alpha [D] FP32 (in)
 *   h0         [B,D] FP32 (in) or NULL;  reset [B,L] uint8 (in) or NULL
 *   y          [B,L,D] BF16 (out);  y32 [B,L,D] FP32 (out, optional) or NULL
 *   hT         [B,D] FP32 (out);  saved, scratch: rglru_workspace_bytes()
 * Errors: as samu_forward. */
int rglru_forward(const void* x, const void* lx, const void* la, const float* alpha,
                  const float* h0, const uint8_t* reset, int B, int L, int D,
                  void* y, float* y32, float* hT, void* saved, void* scratch,
                  cudaStream_t stream);

/* RG-LRU backward ([SAMU page] section 04, backward): reverse real affine scan,
 * gates recomputed, square-root derivative bounded at 1000 (the clipped
 * derivative of the canonical reference), dalpha reduced over batch and chunks
 * to [D] in a fixed order.
 *
 *   dy [B,L,D] BF16 (in);  dhT [B,D] FP32 (in) or NULL
 *   x, lx, la, alpha, h0, reset, B, L, D: the forward's inputs (in)
 *   saved: the forward's saved buffer (in)
 *   dx, dlx, dla [B,L,D] BF16 or FP32 by grad_dtype (out)
 *   dalpha [D] FP32 (out);  dh0 [B,D] FP32 (out)
 * Errors: as samu_backward. */
int rglru_backward(const void* dy, const float* dhT, const void* x, const void* lx,
                   const void* la, const float* alpha, const float* h0, const uint8_t* reset,
                   int B, int L, int D, const void* saved, void* dx, void* dlx, void* dla,
                   int grad_dtype, float* dalpha, float* dh0, void* scratch,
                   cudaStream_t stream);

/* ======================================================================== */
/* RG-LRU with its block-diagonal gate projections                           */
/* ======================================================================== */

/* The RG-LRU mixer's two gate projections ahead of the scan ([SAMU page]
 * section 04, forward: "two canonical block-diagonal projections produce the
 * write- and keep-gate raw values"; [Protocol] "RG-LRU 的固定方程": 16-block
 * block-diagonal linear layers; section 06 parameter count 2 D^2/16 + 3 D):
 *   lx_t[h dk + o] = sum_i x_t[h dk + i] w_x[h][i][o] + b_x[h dk + o],
 *   la_t likewise with w_a, b_a;  h = 0..15, dk = D/16,
 * then the RG-LRU scan of rglru_forward on (x, lx, la).  The products are
 * formed from the BF16 x and BF16 weights with FP32 accumulation on the
 * tensor cores (inside the scan kernel when D/16 divides 64, else by a
 * separate contraction kernel) and stay in FP32 (no rounding of the logits).
 *
 *   x           [B,L,D] BF16 (in)
 *   w_x, w_a    [16][dk][dk] BF16 (in), row i = input channel, column o = output
 *   b_x, b_a    [D] FP32 (in);  alpha [D] FP32 (in)
 *   h0, reset, y, y32, hT: as rglru_forward
 *   saved, scratch: rglru_proj_workspace_bytes() (scratch holds the FP32
 *               logits, the gradient parts and the packed weight images)
 * Errors: as rglru_forward, plus LRS_ERR_UNSUPPORTED unless D is a multiple
 * of 128 (dk a multiple of 8). */
int rglru_proj_workspace_bytes(int B, int L, int D, size_t* saved_bytes, size_t* scratch_bytes);
int rglru_proj_forward(const void* x, const void* w_x, const float* b_x, const void* w_a, const float* b_a,
                       const float* alpha, const float* h0, const uint8_t* reset, int B, int L, int D,
                       void* y, float* y32, float* hT, void* saved, void* scratch, cudaStream_t stream);

/* Backward of rglru_proj_forward: the scan backward with the logits
 * recomputed (inside the scan kernel on the tensor cores when D/16 divides
 * 64, else by the contraction kernel), then dx = dx_scan + dlx W_x^T +
 * dla W_a^T per block,
 * dW_x = x^T dlx, dW_a = x^T dla, db = sum over tokens of dl.  The gate
 * gradients and dx_scan enter the two tensor-core contractions (one for dx
 * with K = 6 D/16, one for dW with K = B L, split over the tokens and added in
 * a fixed order) as BF16 leading parts plus BF16 remainders (16 significant
 * bits); the bias and alpha gradients are fixed-order sums.
 *
 *   dy, dhT, x, w_x, b_x, w_a, b_a, alpha, h0, reset, B, L, D, saved: as above
 *   dx          [B,L,D] BF16 or FP32 by grad_dtype (out)
 *   dw_x, dw_a  [16][dk][dk] FP32 (out);  db_x, db_a, dalpha [D] FP32 (out)
 *   dh0         [B,D] FP32 (out)
 * Errors: as rglru_backward. */
int rglru_proj_backward(const void* dy, const float* dhT, const void* x, const void* w_x, const float* b_x,
                        const void* w_a, const float* b_a, const float* alpha, const float* h0,
                        const uint8_t* reset, int B, int L, int D, const void* saved, void* dx, int grad_dtype,
                        float* dw_x, float* db_x, float* dw_a, float* db_a, float* dalpha, float* dh0,
                        void* scratch, cudaStream_t stream);

/* ======================================================================== */
/* One RecurrentBlock around the SAMU mixer                                  */
/* ======================================================================== */

/* The mixer inside one complete block ([SAMU page] section 03, single-block
 * table and the glossary entry on the complete block: normalisation, two
 * input projections, per-channel convolution, the mixer, the join and output
 * projection, a second normalisation and a gated MLP, with the input and
 * parameter backward; the SAMU project page: the block's wide input branch,
 * split into real and imaginary halves, is the mixer's write w).  Widths: Dm
 * (the residual stream), D (the mixer, M = D/2 modes), F = 3 Dm (the MLP).
 * The pages leave the layers' details open; this library reads them as:
 *   h1 = RMSNorm(x; gamma1)          RMSNorm(x; g) = x / sqrt(mean(x^2) + 1e-6) * g
 *   [g | v] = h1 w_in^T              g: gate branch, v: recurrent branch (D each)
 *   u[t] = conv_b + sum_{j<4} conv_k[j] v[t-j]   causal, per channel; taps before
 *                                    the start of t's segment (reset) are zero
 *   (y_mix, hT) = SAMU(x_sel = u, w = u, h0, reset)   exactly samu_forward
 *   r1 = x + (GeLU(g) y_mix) w_o^T   GeLU(x) = x/2 (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))
 *   h2 = RMSNorm(r1; gamma2)
 *   [a | b] = h2 w_mlp_in^T;  out = r1 + (GeLU(a) b) w_mlp_out^T
 * Every activation between layers is stored in BF16 (round to nearest even)
 * and every contraction accumulates in FP32 on the tensor cores.
 *
 * Parameters (device pointers in a host struct; BF16 matrices are row-major
 * [out][in], FP32 vectors contiguous): */
typedef struct {
    const float* gamma1;     /* [Dm] */
    const void* w_in;        /* [2D][Dm] BF16: rows 0..D-1 gate branch, D..2D-1 recurrent branch */
    const float* conv_k;     /* [4][D]: tap j multiplies v[t-j] */
    const float* conv_b;     /* [D] */
    const float* nu;         /* [M]  the mixer's parameters, as samu_forward */
    const float* theta;      /* [M] */
    const float* w_phi;      /* [D+1] */
    const float* w_r;        /* [D+1] */
    const float* a_phi;      /* one FP32 */
    const float* a_r;        /* one FP32 */
    const void* w_o;         /* [Dm][D] BF16 */
    const float* gamma2;     /* [Dm] */
    const void* w_mlp_in;    /* [2F][Dm] BF16: rows 0..F-1 the GeLU branch a, F..2F-1 the linear branch b */
    const void* w_mlp_out;   /* [Dm][F] BF16 */
} samu_block_params;

/* Parameter gradients (FP32, the parameters' shapes; every one overwritten). */
typedef struct {
    float* dgamma1; float* dw_in; float* dconv_k; float* dconv_b;
    float* dnu; float* dtheta; float* dw_phi; float* dw_r; float* da_phi; float* da_r;
    float* dw_o; float* dgamma2; float* dw_mlp_in; float* dw_mlp_out;
} samu_block_grads;

/* Bytes of `saved` (the mixer's saved buffer plus the block's BF16
 * activations) and `scratch` for shape (B, L, Dm, D).  Pure host function.
 * Errors: LRS_ERR_ARG / LRS_ERR_UNSUPPORTED as samu_block_forward. */
int samu_block_workspace_bytes(int B, int L, int Dm, int D, size_t* saved_bytes, size_t* scratch_bytes);

/* Block forward.
 *   p          parameters (host struct of device pointers; every field required)
 *   x          [B,L,Dm] BF16 (in)
 *   h0         [B,M,2] FP32 (in) or NULL;  reset [B,L] uint8 (in) or NULL
 *   out        [B,L,Dm] BF16 (out);  hT [B,M,2] FP32 (out)
 *   saved, scratch: samu_block_workspace_bytes()
 * lrs_device_status(scratch) reports the whole call (the mixer included).
 * Errors: LRS_ERR_ARG (null or misaligned pointer, bad shape),
 * LRS_ERR_UNSUPPORTED unless Dm and D are multiples of 256 with Dm <= 4096,
 * D <= 4096 and B*L < 2^31, LRS_ERR_CUDA. */
int samu_block_forward(const samu_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                       int B, int L, int Dm, int D, void* out, float* hT, void* saved, void* scratch,
                       cudaStream_t stream);

/* Block backward for the cotangents dout [B,L,Dm] BF16 and dhT [B,M,2] FP32
 * (or NULL): dx [B,L,Dm] BF16 (out), dh0 [B,M,2] FP32 (out) and every
 * parameter gradient in g (out).  Gradients between layers are BF16; the
 * weight gradients are FP32 contractions over the tokens (split over the
 * tokens and added in a fixed order: deterministic).  The inputs must be the
 * forward's and `saved` its saved buffer.  Errors: as samu_block_forward. */
int samu_block_backward(const samu_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                        const void* dout, const float* dhT, int B, int L, int Dm, int D, const void* saved,
                        void* dx, float* dh0, const samu_block_grads* g, void* scratch, cudaStream_t stream);

/* The same block around the RG-LRU mixer with its two 16-block gate
 * projections, the comparison the [SAMU page] section 03 single-block table
 * makes: identical layers, with (y_mix, hT) = rglru_proj_forward(x = u, ...)
 * in place of the SAMU mixer (h0, hT, dhT, dh0 are [B,D] FP32).  Parameters:
 * the block's own as in samu_block_params, then the mixer's as
 * rglru_proj_forward takes them.  Errors: as samu_block_forward, with the
 * mixer's width rules of rglru_proj_forward in place of samu_forward's. */
typedef struct {
    const float* gamma1; const void* w_in; const float* conv_k; const float* conv_b;
    const void* w_x;         /* [16][D/16][D/16] BF16 */
    const float* b_x;        /* [D] */
    const void* w_a;         /* [16][D/16][D/16] BF16 */
    const float* b_a;        /* [D] */
    const float* alpha;      /* [D] */
    const void* w_o; const float* gamma2; const void* w_mlp_in; const void* w_mlp_out;
} rglru_block_params;

typedef struct {
    float* dgamma1; float* dw_in; float* dconv_k; float* dconv_b;
    float* dw_x; float* db_x; float* dw_a; float* db_a; float* dalpha;
    float* dw_o; float* dgamma2; float* dw_mlp_in; float* dw_mlp_out;
} rglru_block_grads;

int rglru_block_workspace_bytes(int B, int L, int Dm, int D, size_t* saved_bytes, size_t* scratch_bytes);
int rglru_block_forward(const rglru_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                        int B, int L, int Dm, int D, void* out, float* hT, void* saved, void* scratch,
                        cudaStream_t stream);
int rglru_block_backward(const rglru_block_params* p, const void* x, const float* h0, const uint8_t* reset,
                         const void* dout, const float* dhT, int B, int L, int Dm, int D, const void* saved,
                         void* dx, float* dh0, const rglru_block_grads* g, void* scratch, cudaStream_t stream);

/* The block's tensor-core contraction on its own (for tests), layouts:
 *   LRS_GEMM_NT  C [M][N] BF16 = A [M][K] . B [N][K]^T
 *   LRS_GEMM_NN  C [M][N] BF16 = A [M][K] . B [K][N]
 *   LRS_GEMM_TN  C [M][N] FP32 = A [K][M]^T . B [K][N]   (one split)
 * FP32 accumulation, BF16 results rounded to nearest even.  N must be a
 * multiple of 256 and K of 64 (NT, NN); M a multiple of 128 (TN); other
 * sizes return LRS_ERR_UNSUPPORTED.  scratch: 256 bytes (the status word).
 * Errors: LRS_ERR_ARG, LRS_ERR_UNSUPPORTED, LRS_ERR_CUDA. */
#define LRS_GEMM_NT 0
#define LRS_GEMM_NN 1
#define LRS_GEMM_TN 2
int lrs_dense_gemm(int layout, const void* A, const void* Bm, void* C, int M, int N, int K, void* scratch,
                   cudaStream_t stream);

/* ======================================================================== */
/* SAMU forward without allocation                                           */
/* ======================================================================== */

/* Size of the fixed device workspace used by samu_forward_noalloc (64 MiB).
 * Every GPU that loads this library holds this much device memory for it
 * until the process exits. */
#define LRS_NOALLOC_BYTES (64u << 20)

/* samu_forward for callers that cannot allocate device memory and have no
 * spare buffer to lend as `saved`/`scratch` (for example an application whose
 * device memory belongs to its own pooled allocator, or a latency-critical
 * loop that must not take cudaMalloc's implicit synchronisation).  The paper
 * has no counterpart; it exists for such callers.
 *
 * Same computation and same arguments as samu_forward without `saved` and
 * `scratch`: the caller still passes every input and output (x_sel, w, h0,
 * reset, nu, theta, w_phi, w_r, a_phi, a_r, y, y32, hT, as documented there).
 * The intermediates live in one fixed device array of LRS_NOALLOC_BYTES that
 * the library declares; nothing is allocated or freed (no cudaMalloc,
 * cudaFree or allocating library routine).  There is no matching backward:
 * the controller cache and entry states are overwritten by the next call.
 *
 * - The first call in each CUDA context (the device's primary context, or a
 *   context of the caller's own) looks up the array's device address in that
 *   context (one cudaGetSymbolAddress, with that context current) and keeps
 *   it under the context's unique id; make that first call before any stream
 *   capture in the context.
 * - Every call on a device shares the array and leaves its contents behind;
 *   each call clears what must start at zero (the status word).  Calls whose
 *   GPU work overlaps (other streams, other host threads) race on the array:
 *   serialise them.
 * - Problems whose intermediates exceed LRS_NOALLOC_BYTES are rejected with
 *   LRS_ERR_TOO_LARGE before anything is launched.  B=1, L=32768, D=2048 uses
 *   about 52 MiB (the entry states every 8 tokens alone take 32 MiB there);
 *   B=1, L=131072, D=1024 (87 MiB) is refused.
 * - A bounded device-side wait that gives up is recorded in the array's
 *   status word; samu_forward_noalloc_status reads it.
 * Errors: as samu_forward, plus LRS_ERR_TOO_LARGE. */
int samu_forward_noalloc(const void* x_sel, const void* w, const float* h0, const uint8_t* reset,
                         const float* nu, const float* theta, const float* w_phi, const float* w_r,
                         const float* a_phi, const float* a_r, int B, int L, int D,
                         void* y, float* y32, float* hT, cudaStream_t stream);

/* The device status word of the most recent samu_forward_noalloc in the
 * current context (the same word samu_forward keeps in its scratch buffer):
 * *status receives LRS_OK, or LRS_ERR_TIMEOUT if a bounded device-side wait
 * of that call gave up (its outputs are then undefined).  SYNCHRONISES
 * `stream`.  Allocates nothing; the first call in a context does the same
 * address look-up as samu_forward_noalloc.  The paper has no counterpart.
 * Errors: LRS_ERR_ARG (status NULL), LRS_ERR_CUDA. */
int samu_forward_noalloc_status(int* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LRS_SAMU_H */

"""One RecurrentBlock around the SAMU mixer: CUDA path (tcgen05 contractions,
norms, convolution, the mixer) through the C ABI vs the FP64 block oracle
(oracle/block.py, BF16 store points emulated), element by element, plus the
block's tensor-core contraction on its own vs an FP64 matmul of the same BF16
operands.

Tolerances.  Every tensor the block stores is BF16 (relative spacing 2^-8).
The CUDA path and the oracle round the same quantities at the same points;
they differ by FP32 (tensor-core accumulation, tanhf, the mixer's FP32 scan)
against FP64 arithmetic, which moves a stored value across a BF16 rounding
boundary now and then.  Each flip is one ulp of one element, but the next
layer's K-term sums carry it into all of their outputs: when a fraction phi
of a row's inputs flipped, about sqrt(phi) of the sums' own roundings flip.
So the share of elements one or more ulps apart grows along the chain of
stores (a few percent for out, 10-25 percent for dx, which sits behind more
than ten of them), while the size of the difference stays at the level of
BF16 rounding noise.  Checked:
  - out: relative L2 error <= 2^-8 (one BF16 ulp RMS); dx, behind the whole
    backward chain: <= 2^-7;
  - every element of out and dx within 2^-4 of the tensor's RMS: a wrong row,
    tap or tile shows up at the level of the RMS itself;
  - the CUDA result is as accurate as BF16 storage allows: its relative L2
    error against the plain FP64 block (no BF16 points) is at most 1.25 times
    the emulated oracle's own, plus 2^-12;
  - FP32 results (hT, dh0, parameter gradients), sums of BF16 products over
    the tokens: relative L2 error <= 2^-7; the mixer's final state hT
    (FP32 end to end from BF16 inputs): <= 2^-8; the two scalar amplitude
    gradients, sums over every token of terms of both signs: within 2^-7 of
    the larger of their own size and the RMS element of the mixer's
    parameter gradients (their relative error is unbounded near cancellation).
"""
import numpy as np
import pytest
import torch

from linear_recurrence_sequence_gb300 import api, synth
from oracle import block as ob

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _bf16_ulp(v):
    """Spacing of BF16 numbers at |v| (2^(e - 7) for |v| in [2^e, 2^(e + 1)))."""
    a = np.maximum(np.abs(v), 1e-30)
    return np.exp2(np.floor(np.log2(a)) - 7)


def _check_bf16(name, got, ref, exact, rel_max):
    rel = _rel(got, ref)
    rms = np.sqrt(np.mean(ref * ref))
    err = np.abs(got - ref)
    acc_gpu, acc_ref = _rel(got, exact), _rel(ref, exact)
    print(f"{name}: rel {rel:.2e}, max |err|/rms {err.max() / rms:.2e}, "
          f"elements beyond 1 ulp {(err > _bf16_ulp(ref)).mean():.2e}, "
          f"error vs plain FP64 {acc_gpu:.2e} (emulated oracle {acc_ref:.2e})")
    assert rel <= rel_max, (name, rel)
    assert err.max() <= 2.0 ** -4 * rms, (name, float(err.max() / rms))
    assert acc_gpu <= 1.25 * acc_ref + 2.0 ** -12, (name, acc_gpu, acc_ref)


def _oracle_params(inp):
    """The oracle's per-layer parameters from the library's stacked ones:
    w_in = [W_g; W_v], w_mlp_in = [W_1; W_2], w_mlp_out = W_3."""
    p = {}
    for n in (synth.BLOCK_PARAMS if inp["mixer"] == "samu" else synth.RGLRU_BLOCK_PARAMS):
        v = inp[n]
        p[n] = synth.bf16_bits_to_f64(v) if n in synth.BLOCK_BF16_PARAMS else np.asarray(v, dtype=np.float64)
    D, F = inp["D"], 3 * inp["Dm"]
    p["w_g"], p["w_v"] = p["w_in"][:D], p["w_in"][D:]
    p["w_1"], p["w_2"] = p["w_mlp_in"][:F], p["w_mlp_in"][F:]
    p["w_3"] = p["w_mlp_out"]
    if inp["mixer"] == "samu":
        p["a_phi"] = float(inp["a_phi"])
        p["a_r"] = float(inp["a_r"])
    return p


def _stacked_grads(gr):
    """The oracle's gradients in the library's stacked layout."""
    out = dict(gr)
    out["dw_in"] = np.concatenate([gr["dw_g"], gr["dw_v"]])
    out["dw_mlp_in"] = np.concatenate([gr["dw_1"], gr["dw_2"]])
    out["dw_mlp_out"] = gr["dw_3"]
    return out


def _run_block(inp):
    t = api.block_tensors_from_numpy(inp, DEV)
    f = api.samu_block_forward(t["x"], t["params"], t["h0"], t["reset"])
    g = api.samu_block_backward(t["dout"], t["dhT"], t["x"], t["params"], t["h0"], t["reset"], f["saved"])
    torch.cuda.synchronize()
    assert api.device_status(f["scratch"]) == 0
    assert api.device_status(g["scratch"]) == 0
    return f, g


CASES = {
    # ragged L (not a multiple of the 128-row tiles or of the 16-token items), resets, h0
    "small_ragged": dict(B=2, L=300, Dm=256, D=256, seed=21, reset_p=0.01),
    # several N tiles in every contraction (F = 1536), two mixer chains
    "two_tiles": dict(B=1, L=640, Dm=512, D=512, seed=22, reset_p=0.0),
    # mixer wider than the residual stream
    "wide_mixer": dict(B=1, L=256, Dm=256, D=768, seed=23, reset_p=0.02),
    # the same block around the RG-LRU mixer with its gate projections (the pages' comparison)
    "rglru_small_ragged": dict(B=2, L=300, Dm=256, D=256, seed=31, reset_p=0.01, mixer="rglru"),
    "rglru_two_tiles": dict(B=1, L=640, Dm=512, D=512, seed=32, reset_p=0.0, mixer="rglru"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_block_forward_backward_matches_oracle(case):
    c = CASES[case]
    mixer = c.get("mixer", "samu")
    inp = synth.block_inputs(c["B"], c["L"], c["Dm"], c["D"], c["seed"], h0=True, reset_p=c["reset_p"], mixer=mixer)
    f, g = _run_block(inp)
    p = _oracle_params(inp)
    x = synth.bf16_bits_to_f64(inp["x"])
    dout = synth.bf16_bits_to_f64(inp["dout"])
    h0 = inp["h0"].astype(np.float64)
    dhT = inp["dhT"].astype(np.float64)
    ref = ob.samu_block_forward(x, p, h0, inp["reset"], bf16=True, mixer=mixer)
    exact = ob.samu_block_forward(x, p, h0, inp["reset"], bf16=False, mixer=mixer)
    _check_bf16("out", _f64(f["out"]), ref["out"], exact["out"], 2.0 ** -8)
    rel_hT = _rel(_f64(f["hT"]), ref["hT"])
    print(f"hT: rel {rel_hT:.2e}")
    assert rel_hT <= 2.0 ** -8
    gr = _stacked_grads(ob.samu_block_backward(x, p, dout, h0, inp["reset"], dhT, bf16=True, mixer=mixer))
    gx = ob.samu_block_backward(x, p, dout, h0, inp["reset"], dhT, bf16=False, mixer=mixer)
    _check_bf16("dx", _f64(g["dx"]), gr["dx"], gx["dx"], 2.0 ** -7)
    mixer_group = (["dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"] if mixer == "samu"
                   else ["dw_x", "db_x", "dw_a", "db_a", "dalpha"])
    group_rms = np.sqrt(np.mean(np.concatenate([np.ravel(gr[k]) for k in mixer_group]) ** 2))
    names = synth.BLOCK_PARAMS if mixer == "samu" else synth.RGLRU_BLOCK_PARAMS
    for k in ["dh0"] + ["d" + n for n in names]:
        ref_k = np.asarray(gr[k], dtype=np.float64)
        got = _f64(g[k]).reshape(np.shape(ref_k))
        if ref_k.size == 1:
            # the amplitude gradients are single sums over every token of terms of
            # both signs: near cancellation their relative error is unbounded, so
            # the difference is measured against the mixer gradients' RMS element
            err = float(abs(got.ravel()[0] - ref_k.ravel()[0]))
            print(f"{k}: {float(got.ravel()[0]):.4e} vs {float(ref_k.ravel()[0]):.4e}, "
                  f"|err| / group RMS {err / group_rms:.2e}")
            assert err <= 2.0 ** -7 * max(abs(float(ref_k.ravel()[0])), group_rms), (k, err)
            continue
        rel = _rel(got, ref_k)
        print(f"{k}: rel {rel:.2e}")
        assert rel <= 2.0 ** -7, (k, rel)


def test_block_backward_is_bitwise_reproducible():
    inp = synth.block_inputs(2, 300, 256, 256, 24, h0=True, reset_p=0.01)
    t = api.block_tensors_from_numpy(inp, DEV)
    f = api.samu_block_forward(t["x"], t["params"], t["h0"], t["reset"])
    g1 = api.samu_block_backward(t["dout"], t["dhT"], t["x"], t["params"], t["h0"], t["reset"], f["saved"])
    g1 = {k: v.clone() for k, v in g1.items() if k != "scratch"}
    f2 = api.samu_block_forward(t["x"], t["params"], t["h0"], t["reset"])
    assert torch.equal(f2["out"], f["out"])
    g2 = api.samu_block_backward(t["dout"], t["dhT"], t["x"], t["params"], t["h0"], t["reset"], f2["saved"])
    for k, v in g1.items():
        assert torch.equal(v, g2[k]), k


@pytest.mark.parametrize("layout,M,N,K", [
    (api.LRS_GEMM_NT, 300, 512, 192),     # ragged M
    (api.LRS_GEMM_NT, 128, 256, 64),      # one tile, one K step
    (api.LRS_GEMM_NN, 300, 768, 320),
    (api.LRS_GEMM_TN, 256, 512, 300),     # ragged K (tokens)
    (api.LRS_GEMM_TN, 384, 256, 1000),
])
def test_dense_gemm_matches_fp64_matmul(layout, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K + layout)
    ash = (K, M) if layout == api.LRS_GEMM_TN else (M, K)
    bsh = (N, K) if layout == api.LRS_GEMM_NT else (K, N)
    a_bits = synth.f32_to_bf16_bits(rng.standard_normal(ash, dtype=np.float32))
    b_bits = synth.f32_to_bf16_bits(rng.standard_normal(bsh, dtype=np.float32))
    A = api._bf16(a_bits, DEV)
    B = api._bf16(b_bits, DEV)
    C = api.dense_gemm(layout, A, B, M, N, K)
    torch.cuda.synchronize()
    a = synth.bf16_bits_to_f64(a_bits)
    b = synth.bf16_bits_to_f64(b_bits)
    ref = a.T @ b if layout == api.LRS_GEMM_TN else (a @ b.T if layout == api.LRS_GEMM_NT else a @ b)
    got = _f64(C)
    if layout == api.LRS_GEMM_TN:
        # FP32 accumulation of K unit-variance products on the tensor cores (not a
        # sequential IEEE sum): error of order 1e-6 sqrt(K) per output, measured
        # maximum over 10^5 outputs 5.5e-6 sqrt(K)
        err = np.abs(got - ref).max() / np.sqrt(K)
        assert err <= 2e-5, err
    else:
        # BF16 results: at most one rounding step from RNE of the exact sum
        err = np.abs(got - ref)
        assert np.all(err <= _bf16_ulp(ref) + 1e-6 * np.sqrt(K)), float((err / _bf16_ulp(ref)).max())

"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and quantises them; it holds none of the
method's arithmetic.  Both the CUDA path and the FP64 oracle receive the exact
same bits: BF16 tensors as uint16 bit patterns, FP32 parameters as float32.

Draw order (one numpy PCG64 stream per seed):
    SAMU  : x_sel, w, nu, theta, w_phi, w_r, a_phi, a_r, h0, reset, dy, dhT
    RG-LRU: x, lx, la, alpha, h0, reset, dy, dhT
    Block : x, then the block's own parameters, the mixer's (as SAMU, or the
            projected RG-LRU's), h0, reset, dout, dhT (see block_inputs)

Value distributions follow the workloads of the SAMU GPU page's measurements:
BF16 N(0,1) activations and cotangents; nu_m = -ln U[0.9, 0.999];
theta_m ~ U[0, 2 pi); w_phi, w_r ~ N(0,1) of length D+1; a_phi, a_r ~ U[-1, 1];
complex h0 with N(0, 0.1^2) real and imaginary parts; Bernoulli resets.
RG-LRU: softplus(alpha) = -ln U[0.9, 0.999] / 8 and resets at segment starts
with gaps U{256..4096} (t = 0 is always a start).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "bf16_bits_to_f64",
    "samu_inputs", "rglru_inputs", "block_inputs", "BLOCK_PARAMS", "WORKLOADS", "Workload",
]


def f32_to_bf16_bits(a) -> np.ndarray:
    """Quantise to bfloat16 (round to nearest, ties to even) via float32; returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    # ties-to-even rounding of the low 16 bits; finite inputs cannot overflow
    # 32 bits here (NaN inputs are not produced by these generators)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def _normal_bf16(rng, shape):
    # draw in float32 directly to keep the cost of large tensors modest
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def samu_inputs(B: int, L: int, D: int, seed: int, *, h0: bool = True,
                reset_p: float = 0.0, zero_amplitudes: bool = False) -> dict:
    """Seeded SAMU mixer inputs.  Returns numpy arrays:

    x_sel, w, dy : uint16 BF16 bits [B,L,D]
    nu, theta    : float32 [M];  w_phi, w_r : float32 [D+1];  a_phi, a_r : float32 scalars
    h0, dhT      : float32 [B,M,2] (h0 None when h0=False)
    reset        : uint8 [B,L] (None when reset_p == 0)
    """
    if D % 2:
        raise ValueError("D must be even")
    M = D // 2
    rng = np.random.default_rng(seed)
    x_sel = _normal_bf16(rng, (B, L, D))
    w = _normal_bf16(rng, (B, L, D))
    nu = (-np.log(rng.uniform(0.9, 0.999, size=M))).astype(np.float32)
    theta = rng.uniform(0.0, 2.0 * math.pi, size=M).astype(np.float32)
    w_phi = rng.standard_normal(D + 1).astype(np.float32)
    w_r = rng.standard_normal(D + 1).astype(np.float32)
    a_phi = np.float32(rng.uniform(-1.0, 1.0))
    a_r = np.float32(rng.uniform(-1.0, 1.0))
    h0_arr = (0.1 * rng.standard_normal((B, M, 2))).astype(np.float32)
    rmask = (rng.random((B, L)) < reset_p).astype(np.uint8) if reset_p > 0 else None
    dy = _normal_bf16(rng, (B, L, D))
    dhT = rng.standard_normal((B, M, 2)).astype(np.float32)
    if zero_amplitudes:
        a_phi = np.float32(0.0)
        a_r = np.float32(0.0)
    return {
        "x_sel": x_sel, "w": w, "nu": nu, "theta": theta, "w_phi": w_phi, "w_r": w_r,
        "a_phi": a_phi, "a_r": a_r, "h0": h0_arr if h0 else None, "reset": rmask,
        "dy": dy, "dhT": dhT, "B": B, "L": L, "D": D,
    }


# Parameters of one RecurrentBlock, in the order of the C struct samu_block_params.
BLOCK_PARAMS = ("gamma1", "w_in", "conv_k", "conv_b", "nu", "theta", "w_phi", "w_r", "a_phi", "a_r",
                "w_o", "gamma2", "w_mlp_in", "w_mlp_out")
BLOCK_BF16_PARAMS = ("w_in", "w_o", "w_mlp_in", "w_mlp_out", "w_x", "w_a")
# The same block around the RG-LRU mixer with its gate projections (the
# pages' comparison), in the order of the C struct rglru_block_params.
RGLRU_BLOCK_PARAMS = ("gamma1", "w_in", "conv_k", "conv_b", "w_x", "b_x", "w_a", "b_a", "alpha",
                      "w_o", "gamma2", "w_mlp_in", "w_mlp_out")


def block_inputs(B: int, L: int, Dm: int, D: int, seed: int, *, h0: bool = True,
                 reset_p: float = 0.0, mixer: str = "samu") -> dict:
    """Seeded inputs of one RecurrentBlock (widths Dm, D, F = 3 Dm) around
    the SAMU mixer, or with mixer="rglru" around the RG-LRU with its gate
    projections.  BF16 tensors as uint16 bits: x, dout [B,L,Dm] ~ N(0,1);
    the dense weights ~ N(0, 1/fan_in): w_in [2D,Dm], w_o [Dm,D],
    w_mlp_in [2F,Dm], w_mlp_out [Dm,F].  FP32: gamma1, gamma2 ~ 1 + 0.1 N(0,1);
    conv_k [4,D] ~ N(0, 1/4), conv_b [D] ~ 0.1 N(0,1); the mixer's parameters
    drawn as samu_inputs (or rglru_proj_inputs) draws them; h0, dhT [B,M,2]
    (RG-LRU: [B,D]); Bernoulli resets."""
    if D % 2:
        raise ValueError("D must be even")
    M, F = D // 2, 3 * Dm
    rng = np.random.default_rng(seed)

    def dense(rows, cols):
        return f32_to_bf16_bits(rng.standard_normal(size=(rows, cols), dtype=np.float32) / np.float32(math.sqrt(cols)))

    x = _normal_bf16(rng, (B, L, Dm))
    out = {"x": x}
    out["gamma1"] = (1.0 + 0.1 * rng.standard_normal(Dm)).astype(np.float32)
    out["w_in"] = dense(2 * D, Dm)
    out["conv_k"] = (0.5 * rng.standard_normal((4, D))).astype(np.float32)
    out["conv_b"] = (0.1 * rng.standard_normal(D)).astype(np.float32)
    if mixer == "samu":
        out["nu"] = (-np.log(rng.uniform(0.9, 0.999, size=M))).astype(np.float32)
        out["theta"] = rng.uniform(0.0, 2.0 * math.pi, size=M).astype(np.float32)
        out["w_phi"] = rng.standard_normal(D + 1).astype(np.float32)
        out["w_r"] = rng.standard_normal(D + 1).astype(np.float32)
        out["a_phi"] = np.float32(rng.uniform(-1.0, 1.0))
        out["a_r"] = np.float32(rng.uniform(-1.0, 1.0))
    else:
        dk = D // PROJ_BLOCKS
        out["w_x"] = f32_to_bf16_bits(rng.standard_normal((PROJ_BLOCKS, dk, dk)) / math.sqrt(dk))
        out["w_a"] = f32_to_bf16_bits(rng.standard_normal((PROJ_BLOCKS, dk, dk)) / math.sqrt(dk))
        out["b_x"] = (0.1 * rng.standard_normal(D)).astype(np.float32)
        out["b_a"] = (0.1 * rng.standard_normal(D)).astype(np.float32)
        sp = -np.log(rng.uniform(0.9, 0.999, size=D)) / 8.0          # softplus(alpha)
        out["alpha"] = np.log(np.expm1(sp)).astype(np.float32)
    out["w_o"] = dense(Dm, D)
    out["gamma2"] = (1.0 + 0.1 * rng.standard_normal(Dm)).astype(np.float32)
    out["w_mlp_in"] = dense(2 * F, Dm)
    out["w_mlp_out"] = dense(Dm, F)
    state = (B, M, 2) if mixer == "samu" else (B, D)
    h0_arr = (0.1 * rng.standard_normal(state)).astype(np.float32)
    out["h0"] = h0_arr if h0 else None
    out["reset"] = (rng.random((B, L)) < reset_p).astype(np.uint8) if reset_p > 0 else None
    out["dout"] = _normal_bf16(rng, (B, L, Dm))
    out["dhT"] = rng.standard_normal(state).astype(np.float32)
    out.update({"B": B, "L": L, "Dm": Dm, "D": D, "mixer": mixer})
    return out


def segment_starts(rng, B: int, L: int, lo: int = 256, hi: int = 4096) -> np.ndarray:
    """Reset mask with a segment start at t = 0 and gaps drawn from U{lo..hi}."""
    mask = np.zeros((B, L), dtype=np.uint8)
    for b in range(B):
        t = 0
        while t < L:
            mask[b, t] = 1
            t += int(rng.integers(lo, hi + 1))
    return mask


def rglru_inputs(B: int, L: int, D: int, seed: int, *, h0: bool = False,
                 resets: str = "segments") -> dict:
    """Seeded RG-LRU inputs.  x, lx, la, dy: uint16 BF16 bits [B,L,D]; alpha float32 [D];
    h0, dhT float32 [B,D] (h0 None when h0=False); reset uint8 [B,L] or None.

    resets: "segments" (gaps U{256..4096}, start at t=0), "none", or a float
    probability for Bernoulli resets.
    """
    rng = np.random.default_rng(seed)
    x = _normal_bf16(rng, (B, L, D))
    lx = _normal_bf16(rng, (B, L, D))
    la = _normal_bf16(rng, (B, L, D))
    sp = -np.log(rng.uniform(0.9, 0.999, size=D)) / 8.0          # softplus(alpha)
    alpha = np.log(np.expm1(sp)).astype(np.float32)               # inverse softplus, fp64
    h0_arr = (0.1 * rng.standard_normal((B, D))).astype(np.float32)
    if resets == "segments":
        rmask = segment_starts(rng, B, L)
    elif resets == "none":
        rmask = None
    else:
        rmask = (rng.random((B, L)) < float(resets)).astype(np.uint8)
    dy = _normal_bf16(rng, (B, L, D))
    dhT = rng.standard_normal((B, D)).astype(np.float32)
    return {"x": x, "lx": lx, "la": la, "alpha": alpha, "h0": h0_arr if h0 else None,
            "reset": rmask, "dy": dy, "dhT": dhT, "B": B, "L": L, "D": D}


PROJ_BLOCKS = 16   # diagonal blocks of each RG-LRU gate projection


def rglru_proj_inputs(B: int, L: int, D: int, seed: int, *, h0: bool = False,
                      resets: str = "segments") -> dict:
    """Seeded inputs of the RG-LRU mixer with its two block-diagonal gate
    projections.  x, dy: uint16 BF16 bits [B,L,D]; w_x, w_a: uint16 BF16 bits
    [16][D/16][D/16] with entries N(0, 1/(D/16)) (so that the logits x W are
    about N(0,1) like the raw-logit workloads); b_x, b_a float32 [D] N(0, 0.1^2);
    alpha, h0, reset, dhT as rglru_inputs.  Draw order: x, w_x, w_a, b_x, b_a,
    alpha, h0, reset, dy, dhT."""
    rng = np.random.default_rng(seed)
    dk = D // PROJ_BLOCKS
    x = _normal_bf16(rng, (B, L, D))
    w_x = f32_to_bf16_bits(rng.standard_normal((PROJ_BLOCKS, dk, dk)) / math.sqrt(dk))
    w_a = f32_to_bf16_bits(rng.standard_normal((PROJ_BLOCKS, dk, dk)) / math.sqrt(dk))
    b_x = (0.1 * rng.standard_normal(D)).astype(np.float32)
    b_a = (0.1 * rng.standard_normal(D)).astype(np.float32)
    sp = -np.log(rng.uniform(0.9, 0.999, size=D)) / 8.0          # softplus(alpha)
    alpha = np.log(np.expm1(sp)).astype(np.float32)
    h0_arr = (0.1 * rng.standard_normal((B, D))).astype(np.float32)
    if resets == "segments":
        rmask = segment_starts(rng, B, L)
    elif resets == "none":
        rmask = None
    else:
        rmask = (rng.random((B, L)) < float(resets)).astype(np.uint8)
    dy = _normal_bf16(rng, (B, L, D))
    dhT = rng.standard_normal((B, D)).astype(np.float32)
    return {"x": x, "w_x": w_x, "w_a": w_a, "b_x": b_x, "b_a": b_a, "alpha": alpha,
            "h0": h0_arr if h0 else None, "reset": rmask, "dy": dy, "dhT": dhT, "B": B, "L": L, "D": D}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "samu" or "rglru"
    B: int
    L: int
    D: int
    seeds: tuple = (0,)
    h0: bool = True
    reset_p: float = 0.0
    extra: dict = field(default_factory=dict)

    def make(self, seed=None) -> dict:
        s = self.seeds[0] if seed is None else seed
        if self.kind == "samu":
            return samu_inputs(self.B, self.L, self.D, s, h0=self.h0, reset_p=self.reset_p)
        if self.kind == "rglru_proj":
            return rglru_proj_inputs(self.B, self.L, self.D, s, h0=self.h0,
                                     resets=self.extra.get("resets", "segments"))
        return rglru_inputs(self.B, self.L, self.D, s, h0=self.h0,
                            resets=self.extra.get("resets", "segments"))


# The five measured workload families (shapes, generators and seeds).
WORKLOADS = {
    "tiny": Workload("tiny", "samu", 2, 2048, 256, (0,), h0=True, reset_p=1 / 512),
    "short": Workload("short", "samu", 4, 4096, 1024, (1, 2, 3), h0=False, reset_p=0.0),
    "length_8k": Workload("length_8k", "samu", 1, 8192, 1024, (0,), h0=True, reset_p=1 / 8192),
    "length_32k": Workload("length_32k", "samu", 1, 32768, 1024, (0,), h0=True, reset_p=1 / 8192),
    "length_64k": Workload("length_64k", "samu", 1, 65536, 1024, (0,), h0=True, reset_p=1 / 8192),
    "length_128k": Workload("length_128k", "samu", 1, 131072, 1024, (0,), h0=True, reset_p=1 / 8192),
    "width_1024": Workload("width_1024", "samu", 1, 32768, 1024, (0,), h0=False),
    "width_1536": Workload("width_1536", "samu", 1, 32768, 1536, (0,), h0=False),
    "width_2048": Workload("width_2048", "samu", 1, 32768, 2048, (0,), h0=False),
    "width_2560": Workload("width_2560", "samu", 1, 32768, 2560, (0,), h0=False),
    "medium_8k_2560": Workload("medium_8k_2560", "samu", 1, 8192, 2560, (0,), h0=False),
    "rglru_2k": Workload("rglru_2k", "rglru", 8, 2048, 1024, (0,), h0=False),
    "rglru_4k": Workload("rglru_4k", "rglru", 8, 4096, 1024, (0,), h0=False),
    "rglru_8k": Workload("rglru_8k", "rglru", 8, 8192, 1024, (0,), h0=False),
    "rglru_16k": Workload("rglru_16k", "rglru", 8, 16384, 1024, (0,), h0=False),
    # the RG-LRU mixer with its 16-block gate projections (the pages' mixer scope)
    "rglru_proj_8k": Workload("rglru_proj_8k", "rglru_proj", 8, 8192, 1024, (0,), h0=False),
    # the pages' headline comparison shape: B1 L8192 D1024, RG-LRU with its gate projections
    "rglru_proj_b1_8k": Workload("rglru_proj_b1_8k", "rglru_proj", 1, 8192, 1024, (0,), h0=False),
    "rglru_proj_16k": Workload("rglru_proj_16k", "rglru_proj", 8, 16384, 1024, (0,), h0=False),
}

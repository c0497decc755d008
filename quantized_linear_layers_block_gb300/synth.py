"""Seeded synthetic inputs for the ternary linear layer.

This module only draws random numbers in the shapes and distributions of the
layer's workloads. It holds none of the layer's arithmetic (no rotation, no
quantisation, no packing, no GEMM), so both the CPU oracle and the CUDA path
can consume its output without sharing any method code.

Source of the shapes: the Qwen-family 27B ternary model served in the Qiita
articles "RTX 5070 ×2 / WSL2 で Ternary-Bonsai-2-27B を vLLM TP=2 で本番運用"
(item ecc183fae033565af7cb): hidden size 5120 (a 256-token all-reduce of
2.6 MB in bf16, §6 "部品ごとに測る"), intermediate size 17408 (the down_proj
input width, §1 "TP=2 への移植"), 64 layers, weights in {-1, 0, +1} with one
fp16 scale per 128 elements (前提).

Recipe (every draw from numpy's PCG64 seeded with the given seed):
  * codes: ternary, P(0) = p0, +1 and -1 equally likely (uniform means p0=1/3),
    drawn as one uniform u per element: u < p0 -> 0, else sign by u's half.
  * scales: exp(N(mu, sigma)) rounded to fp16, one per (row, 128-column group).
  * x: bf16 (round-to-nearest-even of the fp32 draw, after any outlier scaling),
    either N(0,1) with chosen outlier channels scaled, or Student-t(df=3)
    drawn as Z / sqrt(chi2_3 / 3), chi2_3 a sum of three squared normals.
"""

from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "LayerInputs",
    "ternary_codes",
    "group_scales",
    "bf16_bits_from_f32",
    "bf16_bits_to_f32",
    "activations_gauss_outliers",
    "activations_student_t",
    "make_layer",
    "CONFIGS",
    "config_inputs",
]


@dataclasses.dataclass
class LayerInputs:
    """One layer's inputs: codes int8 [N,K], s fp16 [N,K/128], x bf16 bits uint16 [M,K]."""

    codes: np.ndarray
    s: np.ndarray
    x_bits: np.ndarray

    @property
    def M(self) -> int:
        return int(self.x_bits.shape[0])

    @property
    def N(self) -> int:
        return int(self.codes.shape[0])

    @property
    def K(self) -> int:
        return int(self.codes.shape[1])


def ternary_codes(rng: np.random.Generator, n: int, k: int, p0: float) -> np.ndarray:
    """int8 [n,k] in {-1,0,+1}: P(0)=p0, +1/-1 equiprobable."""
    out = np.empty((n, k), dtype=np.int8)
    rows = max(1, (1 << 24) // max(k, 1))
    for r0 in range(0, n, rows):
        u = rng.random((min(rows, n - r0), k), dtype=np.float32)
        c = np.where(u < p0, 0, np.where(u < p0 + (1.0 - p0) * 0.5, 1, -1))
        out[r0:r0 + c.shape[0]] = c.astype(np.int8)
    return out


def group_scales(rng: np.random.Generator, n: int, k: int, mu: float, sigma: float) -> np.ndarray:
    """fp16 [n, k/128]: exp(N(mu, sigma)) rounded to fp16."""
    g = k // 128
    return np.exp(rng.normal(mu, sigma, size=(n, g))).astype(np.float16)


def bf16_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the uint16 bit patterns.

    Used only to produce bf16 inputs; the values are finite by construction.
    """
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations_gauss_outliers(rng: np.random.Generator, m: int, k: int, n_outliers: int,
                               factor: float) -> np.ndarray:
    """bf16 bits [m,k]: N(0,1) with n_outliers channels (chosen without replacement) scaled."""
    x = rng.standard_normal((m, k), dtype=np.float32)
    if n_outliers > 0:
        ch = rng.choice(k, size=n_outliers, replace=False)
        x[:, ch] *= np.float32(factor)
    return bf16_bits_from_f32(x)


def activations_student_t(rng: np.random.Generator, m: int, k: int) -> np.ndarray:
    """bf16 bits [m,k]: Student-t with 3 degrees of freedom, Z / sqrt(chi2_3 / 3)."""
    z = rng.standard_normal((m, k))
    chi2 = (rng.standard_normal((3, m, k)) ** 2).sum(axis=0)
    return bf16_bits_from_f32((z / np.sqrt(chi2 / 3.0)).astype(np.float32))


def make_layer(seed: int, M: int, K: int, N: int, *, p0: float, mu: float, sigma: float,
               x_kind: str, n_outliers: int = 0, outlier_factor: float = 1.0) -> LayerInputs:
    """Draw one layer's inputs; the order of draws is codes, scales, x."""
    if K % 1024 or N % 128:
        raise ValueError("K must be a multiple of 1024 and N a multiple of 128")
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = ternary_codes(rng, N, K, p0)
    s = group_scales(rng, N, K, mu, sigma)
    if x_kind == "gauss":
        xb = activations_gauss_outliers(rng, M, K, n_outliers, outlier_factor)
    elif x_kind == "t3":
        xb = activations_student_t(rng, M, K)
    else:
        raise ValueError(x_kind)
    return LayerInputs(codes=codes, s=s, x_bits=xb)


# The five workloads. Seed: 0 for the tiny layer; 1000*config + layer otherwise.
CONFIGS = {
    "tiny": dict(M=16, K=2048, N=256, p0=1.0 / 3.0, mu=-4.0, sigma=0.5,
                 x_kind="gauss", n_outliers=4, outlier_factor=20.0, cfg=1),
    "decode": dict(M=1, K=5120, N=17408, p0=0.4, mu=-4.0, sigma=0.5, x_kind="t3", cfg=2),
    "decode16": dict(M=16, K=5120, N=17408, p0=0.4, mu=-4.0, sigma=0.5, x_kind="t3", cfg=2),
    "down_proj": dict(M=256, K=17408, N=5120, p0=1.0 / 3.0, mu=-4.0, sigma=0.5,
                      x_kind="gauss", n_outliers=174, outlier_factor=30.0, cfg=3),
    "gate_up": dict(M=512, K=5120, N=34816, p0=0.33, mu=-4.0, sigma=0.7, x_kind="t3", cfg=4),
    "sweep_up": dict(M=None, K=5120, N=17408, p0=0.4, mu=-4.0, sigma=0.5, x_kind="t3", cfg=5),
    "sweep_down": dict(M=None, K=17408, N=5120, p0=0.4, mu=-4.0, sigma=0.5, x_kind="t3", cfg=5),
}

SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 4096)

# The int8 128-group codec's payload: one bf16 part per rank of the row-parallel
# all-reduce of the 5120-wide hidden state (P1 §6: 256 tokens, 2.6 MB; P3 §5:
# 1584-row payloads). Each part is N(0,1) with the same few outlier channels
# (0.2 % of H, scaled by 20) in every part, rounded to bf16.
CODEC = dict(R=1584, H=5120, parts=2, outlier_frac=0.002, outlier_factor=20.0, seed=6000)


def codec_parts(seed: int, R: int, H: int, parts: int, outlier_frac: float = 0.002,
                outlier_factor: float = 20.0) -> list:
    """bf16 bits [R, H] for each of `parts` ranks; the outlier channels are drawn first."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_out = int(round(outlier_frac * H))
    ch = rng.choice(H, size=n_out, replace=False) if n_out > 0 else np.zeros(0, dtype=np.int64)
    out = []
    for _ in range(parts):
        x = rng.standard_normal((R, H), dtype=np.float32)
        x[:, ch] *= np.float32(outlier_factor)
        out.append(bf16_bits_from_f32(x))
    return out


def config_seed(name: str, layer: int = 0) -> int:
    cfg = CONFIGS[name]["cfg"]
    return 0 if cfg == 1 else 1000 * cfg + layer


def config_inputs(name: str, layer: int = 0, M: int | None = None, N: int | None = None,
                  K: int | None = None) -> LayerInputs:
    """Inputs of a named workload; M, N, K may be overridden (e.g. a row sample, a sweep M)."""
    c = dict(CONFIGS[name])
    c.pop("cfg")
    if M is not None:
        c["M"] = M
    if N is not None:
        c["N"] = N
    if K is not None:
        c["K"] = K
    if c["M"] is None:
        raise ValueError("sweep configs need an explicit M")
    return make_layer(config_seed(name, layer), **c)


# --------------------------------------------------------------------------
# Device-side generation of many layers for benchmarking (same recipe, drawn
# with torch's CUDA generator so that 64 layer buffers take seconds, not
# minutes). Parity tests use the numpy generator above.
# --------------------------------------------------------------------------

def torch_layer(seed: int, M: int, K: int, N: int, *, p0: float, mu: float, sigma: float,
                x_kind: str, n_outliers: int = 0, outlier_factor: float = 1.0,
                device: str = "cuda"):
    """(codes int8 [N,K], s fp16 [N,K/128], x bf16 [M,K]) on `device`, seeded."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    codes = torch.empty((N, K), dtype=torch.int8, device=device)
    rows = max(1, (1 << 26) // K)
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        u = torch.rand((r1 - r0, K), generator=g, device=device)
        c = torch.where(u < p0, 0, torch.where(u < p0 + (1.0 - p0) * 0.5, 1, -1))
        codes[r0:r1] = c.to(torch.int8)
    s = torch.exp(torch.randn((N, K // 128), generator=g, device=device) * sigma + mu).to(torch.float16)
    if x_kind == "gauss":
        x = torch.randn((M, K), generator=g, device=device)
        if n_outliers > 0:
            ch = torch.randperm(K, generator=g, device=device)[:n_outliers]
            x[:, ch] *= outlier_factor
    elif x_kind == "t3":
        z = torch.randn((M, K), generator=g, device=device)
        chi2 = (torch.randn((3, M, K), generator=g, device=device) ** 2).sum(0)
        x = z / torch.sqrt(chi2 / 3.0)
    else:
        raise ValueError(x_kind)
    return codes, s, x.to(torch.bfloat16)


def torch_config_layer(name: str, layer: int, M: int | None = None, device: str = "cuda"):
    """A named workload's layer drawn on the device (see torch_layer)."""
    c = dict(CONFIGS[name])
    c.pop("cfg")
    if M is not None:
        c["M"] = M
    return torch_layer(config_seed(name, layer), device=device, **c)


def torch_codec_parts(seed: int, R: int, H: int, parts: int, outlier_frac: float = 0.002,
                      outlier_factor: float = 20.0, device: str = "cuda") -> list:
    """Device-side draws of the codec payload (same recipe, torch's generator), bf16 tensors."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    n_out = int(round(outlier_frac * H))
    ch = torch.randperm(H, generator=g, device=device)[:n_out]
    out = []
    for _ in range(parts):
        x = torch.randn((R, H), generator=g, device=device, dtype=torch.float32)
        x[:, ch] *= outlier_factor
        out.append(x.to(torch.bfloat16))
    return out


"""CPU oracle for the int8 128-group codec — TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this module. The product path never calls it.

What it computes, from the pages:

  [P1] Qiita item ecc183fae033565af7cb, §6 "最後に残った問題", paragraph
       "通信を減らす・隠す、は全部だめだった": the row-parallel all-reduce
       payload is compressed to int8 with one scale per 128 elements, the
       compressed parts are all-gathered, and each rank adds its own part
       in bf16 (uncompressed) to the decompressed parts of the others.
  [P3] Qiita item 66e136acefd5a54b2f1d, §5 "解説: 長文を読む速度(prefill)":
       the same codec as two GPU kernels, "compress" and "decompress and
       add", on 1584-row payloads of the 5120-wide hidden state.

Readings where the pages are silent (listed in the design notes):
  * Compression follows the activation quantiser of the layer, per group of
    128 consecutive elements of a row: a = max |x| over the group (x is bf16,
    widened exactly to fp32); inv = fl32(127 / a);
    q = clamp(rne(fl32(x inv)), -127, 127); scale = fl32(a / 127), stored as
    fp32; a group with a = 0 gives q = 0 and scale = 0.
  * Decompress-and-add accumulates in fp32, starting from the rank's own bf16
    part and adding the peers' parts fl32(q scale) in rank order, each product
    and each sum rounded to fp32 (no fused multiply-add); the sum is rounded
    once to bf16 (round to nearest even).
  * A group whose maximum a is below 127 / FLT_MAX (about 3.7e-37, bf16
    subnormals and the smallest normals) overflows inv to +inf; its non-zero
    elements then code to +-127 and its zeros to 0 (the NaN of 0 * inf
    converts to 0, as an fp32 -> integer conversion does).
  * Layouts are row-major: x, q and the output [R, H]; scale [R, H/128];
    the peers' parts are stacked as [P-1, R, H] and [P-1, R, H/128].

The collective itself (all-gather across GPUs) is out of scope: the codec is
what runs on one GPU before and after it.

Pins (tests/test_oracle_codec.py): integer payloads whose group maximum is
127 round-trip exactly and add exactly (one and two peers); the round-trip
error bound scale/2 (1 + 1e-4); the largest element of every non-zero group
codes to +-127; a per-group, not per-row, scale; zero groups; the own part
passes uncompressed; the pages' 1.5 % error figure as an upper bound for the
workload's payloads.
"""

from __future__ import annotations

import numpy as np

from .ternary_linear import bf16_to_f32, f32_to_bf16_bits

CODEC_GROUP = 128     # elements per scale (P1 §6)
CODEC_QMAX = 127


def quantize_groups(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Compress a bf16 payload [R, H] (uint16 bit patterns) to int8 codes
    [R, H] and fp32 scales [R, H/128] (P1 §6; reading: the layer's symmetric
    quantiser applied per 128-element group)."""
    x = bf16_to_f32(np.asarray(x_bits, dtype=np.uint16))
    R, H = x.shape
    if H % CODEC_GROUP:
        raise ValueError("H must be a multiple of 128")
    xg = x.reshape(R, H // CODEC_GROUP, CODEC_GROUP)
    a = np.max(np.abs(xg), axis=2)                                # fp32, exact
    nz = a > 0
    safe = np.where(nz, a, np.float32(1))
    with np.errstate(over="ignore"):
        inv = np.where(nz, np.float32(CODEC_QMAX) / safe, np.float32(0)).astype(np.float32)
    scale = np.where(nz, safe / np.float32(CODEC_QMAX), np.float32(0)).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        t = (xg * inv[:, :, None]).astype(np.float32)             # one fp32 multiply
    # A group whose maximum is below 127 / FLT_MAX makes inv overflow to +inf:
    # its non-zero elements then code to +-127 and its exact zeros (0 * inf =
    # NaN) to 0, the value an fp32 -> int conversion gives a NaN.
    t = np.where(np.isnan(t), np.float32(0), t)
    q = np.clip(np.rint(t), -CODEC_QMAX, CODEC_QMAX).astype(np.int8)   # rint: half to even
    return q.reshape(R, H), scale


def dequantize_groups(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """fl32(q scale) per element, [R, H] fp32."""
    R, H = q.shape
    qg = q.astype(np.float32).reshape(R, H // CODEC_GROUP, CODEC_GROUP)
    return (qg * scale[:, :, None].astype(np.float32)).astype(np.float32).reshape(R, H)


def dequant_add(own_bits: np.ndarray, q_peers: np.ndarray, scale_peers: np.ndarray) -> np.ndarray:
    """Decompress the peers' parts and add them to the own bf16 part
    (P1 §6: own part kept in bf16). fp32 accumulation in rank order, one
    rounding to bf16 at the end. Returns bf16 bit patterns [R, H]."""
    acc = bf16_to_f32(np.asarray(own_bits, dtype=np.uint16)).astype(np.float32)
    q_peers = np.asarray(q_peers)
    scale_peers = np.asarray(scale_peers)
    if q_peers.ndim == 2:
        q_peers = q_peers[None]
        scale_peers = scale_peers[None]
    for p in range(q_peers.shape[0]):
        acc = (acc + dequantize_groups(q_peers[p], scale_peers[p])).astype(np.float32)
    return f32_to_bf16_bits(acc)


def allreduce_fp64(parts_bits: list[np.ndarray]) -> np.ndarray:
    """The exact sum of the ranks' bf16 parts, in fp64 (what the compressed
    all-reduce approximates)."""
    return sum(bf16_to_f32(np.asarray(p, dtype=np.uint16)).astype(np.float64) for p in parts_bits)

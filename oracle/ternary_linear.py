"""CPU oracle for the ternary linear layer — TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this module. The product path (the CUDA library and its
binding) never calls it and shares no code with it.

What it computes, step by step, in the order of the source pages:

  [P1] Qiita item ecc183fae033565af7cb, "RTX 5070 (12GB) ×2 / WSL2 で
       Ternary-Bonsai-2-27B を vLLM TP=2 で本番運用するまでの記録"
       - 前提: weights are {-1,0,+1} codes in 2 bits plus one fp16 scale per
         128 elements; a block-wise Hadamard rotation sits on the input side.
       - §1 "TP=2 への移植": the Sylvester recursion
         H1024 [a; b] = [H512 a + H512 b; H512 a - H512 b].
       - §4 "効いた高速化" (prefill linear layers as an int8 GEMM):
         q[n,g] = round(127 s[n,g] / smax[n]); W_int8[n,k] = code[n,k] q[n,k/128]
         fits exactly in int8; activations are quantised to int8 per token
         after the rotation; one int8 GEMM; rescale per row and per token.

Readings where the pages are silent (each one is listed in the design notes):
  * H is the Sylvester matrix in natural order, H[i,j] = (-1)^popcount(i&j),
    scaled by 1/sqrt(1024) = 1/32 so that the rotation is orthonormal.
  * The fp32 rotation is the fast Walsh-Hadamard transform with butterfly
    strides 1, 2, 4, ..., 512 in that order, (a, b) -> (a + b, a - b), each an
    IEEE fp32 add/sub; the 1/32 scale is applied after the last stage.
  * smax[n] = max_g |s[n,g]|; t = fl32(fl32(127 s) / smax); q = round-half-even(t);
    sw[n] = fl32(smax / 127); a zero row gives q = 0 and sw = 0.
  * Activation quantisation is symmetric over the whole token:
    a = max_k |xr|; inv = fl32(127 / a); xq = clamp(rne(fl32(xr inv)), -127, 127);
    sx = fl32(a / 127); a token with a = 0 gives xq = 0, sx = 0. A token with
    0 < a < 127/FLT_MAX (bf16 subnormals) overflows inv to +inf: its non-zero
    elements code to +-127 and its exact zeros (0 * inf = NaN) to 0.
  * The rotated activations stay fp32 (no bf16 rounding before quantisation).
  * Epilogue: y = fl32(fl32(fl32(acc) sw[n]) sx[m]); optional rne to bf16.
  * The 2-bit packed layout is this library's own format (the pages only say
    "2-bit representation"): uint32 words [N][K/16], little endian; word w of
    row n covers k in [16w, 16w+16); the 2-bit field at bit 16h + 2j holds
    e = code[n, 16w + 2j + h] + 1, for j in 0..7 and h in {0, 1}.

Pins (tests/test_oracle_pins.py): H H^T = 1024 I in integers, the §1
recursion, scipy's Sylvester Hadamard, involution and Parseval, the §1
rank-swap negative control (~sqrt 2; the page measured 1.44), |code q| <= 127,
brute-force integer GEMM on tiny shapes, hand-derived one-hot examples, and the
layer-level relative error against the unquantised fp64 ternary matmul.
"""

from __future__ import annotations

import numpy as np

BLOCK = 1024          # Hadamard block size (P1 前提 "ブロック単位のアダマール回転")
GROUP = 128           # elements per fp16 weight scale (P1 前提, §4)
QMAX = 127            # symmetric int8 range used by §4's q and the activations
INV_SQRT_BLOCK = np.float32(1.0 / 32.0)


# --------------------------------------------------------------------------
# Hadamard rotation
# --------------------------------------------------------------------------

def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (a power of two), natural order.

    Closed form H[i,j] = (-1)^popcount(i & j); equal to the P1 §1 recursion
    H_2n = [[H_n, H_n], [H_n, -H_n]].
    """
    i = np.arange(n, dtype=np.int64)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.zeros_like(bits)
    while np.any(bits):
        pop += bits & 1
        bits >>= 1
    return np.where(pop % 2 == 0, 1, -1).astype(np.int64)


def fwht(v: np.ndarray, dtype=np.float32) -> np.ndarray:
    """Unscaled Walsh-Hadamard transform of the last axis (a power of two) in `dtype`.

    Butterfly stages with strides 1, 2, 4, ... in that order; each stage maps
    the pair (v[i], v[i + h]) with i & h == 0 to (v[i] + v[i+h], v[i] - v[i+h]).
    """
    v = np.array(v, dtype=dtype, copy=True)
    n = v.shape[-1]
    lead = v.shape[:-1]
    h = 1
    while h < n:
        w = v.reshape(lead + (n // (2 * h), 2, h))
        a = w[..., 0, :].copy()
        b = w[..., 1, :].copy()
        w[..., 0, :] = a + b
        w[..., 1, :] = a - b
        v = w.reshape(lead + (n,))
        h *= 2
    return v


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rotate_fp32(x_bits: np.ndarray, signs: np.ndarray | None = None) -> np.ndarray:
    """xr = (1/32) H1024 (signs * x) per 1024-block of each token, in fp32 (P1 前提)."""
    x = bf16_to_f32(x_bits)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 1024")
    if signs is not None:
        x = x * np.asarray(signs, dtype=np.float32)[None, :]
    blocks = x.reshape(M, K // BLOCK, BLOCK)
    r = fwht(blocks, np.float32) * INV_SQRT_BLOCK
    return r.reshape(M, K).astype(np.float32)


def rotate_fp64(x_bits: np.ndarray, signs: np.ndarray | None = None) -> np.ndarray:
    """The same rotation in fp64, by the explicit matrix product with H/32."""
    x = bf16_to_f32(x_bits).astype(np.float64)
    M, K = x.shape
    if signs is not None:
        x = x * np.asarray(signs, dtype=np.float64)[None, :]
    H = hadamard(BLOCK).astype(np.float64) / 32.0
    blocks = x.reshape(M, K // BLOCK, BLOCK)
    return np.einsum("ij,mbj->mbi", H, blocks).reshape(M, K)


# --------------------------------------------------------------------------
# Per-token activation quantisation (P1 §4)
# --------------------------------------------------------------------------

def quantize_per_token(xr: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Symmetric per-token int8: returns xq int8 [M,K] and sx fp32 [M]."""
    xr = np.asarray(xr, dtype=np.float32)
    M, K = xr.shape
    xq = np.zeros((M, K), dtype=np.int8)
    sx = np.zeros(M, dtype=np.float32)
    for m in range(M):
        a = np.max(np.abs(xr[m]))
        if a == 0:
            continue
        # a below 127 / FLT_MAX (about 3.7e-37; a token of bf16 subnormals)
        # makes the fp32 quotient overflow to +inf
        with np.errstate(over="ignore"):
            inv = np.float32(np.float32(QMAX) / a)
        with np.errstate(over="ignore", invalid="ignore"):
            t = (xr[m] * inv).astype(np.float32)
        # Reading for that case: a non-zero element times +inf is +-inf and
        # clamps to +-127; an exact zero times +inf is NaN and codes to 0, the
        # value an fp32 -> int conversion gives a NaN. Finite products are
        # rounded half to even and clamped as usual.
        t = np.where(np.isnan(t), np.float32(0), t)
        xq[m] = np.clip(np.rint(t), -QMAX, QMAX).astype(np.int8)
        sx[m] = np.float32(a / np.float32(QMAX))
    return xq, sx


def rotate_quant(x_bits: np.ndarray, signs: np.ndarray | None = None):
    """Rotation followed by per-token quantisation: (xq int8 [M,K], sx fp32 [M])."""
    return quantize_per_token(rotate_fp32(x_bits, signs))


# --------------------------------------------------------------------------
# Weight decomposition and packing (P1 §4 and 前提)
# --------------------------------------------------------------------------

def row_scale_decompose(s: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """s fp16 [N,G] -> (q int8 [N,G], sw fp32 [N], smax fp32 [N]).

    q[n,g] = rne(fl32(fl32(127 s[n,g]) / smax[n])) with smax[n] = max_g |s[n,g]|.
    """
    sf = np.asarray(s, dtype=np.float16).astype(np.float32)
    N, G = sf.shape
    smax = np.max(np.abs(sf), axis=1).astype(np.float32)
    q = np.zeros((N, G), dtype=np.int8)
    nz = smax > 0
    num = (np.float32(QMAX) * sf[nz]).astype(np.float32)
    t = (num / smax[nz][:, None]).astype(np.float32)
    q[nz] = np.rint(t).astype(np.int8)
    sw = np.where(nz, smax / np.float32(QMAX), np.float32(0)).astype(np.float32)
    return q, sw, smax


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """codes int8 [N,K] in {-1,0,1} -> packed uint8 [N,K/4] (layout in the module header)."""
    c = np.asarray(codes)
    N, K = c.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if np.any((c < -1) | (c > 1)):
        raise ValueError("codes must be in {-1, 0, 1}")
    e = (c.astype(np.int64) + 1).reshape(N, K // 16, 8, 2)    # [n, w, j, h]
    words = np.zeros((N, K // 16), dtype=np.uint64)
    for j in range(8):
        for h in range(2):
            words |= e[:, :, j, h].astype(np.uint64) << np.uint64(16 * h + 2 * j)
    return words.astype("<u4").view(np.uint8).reshape(N, K // 4)


def unpack_codes(packed: np.ndarray, K: int) -> np.ndarray:
    """Inverse of pack_codes."""
    N = packed.shape[0]
    words = np.ascontiguousarray(packed, dtype=np.uint8).view("<u4").reshape(N, K // 16)
    words = words.astype(np.uint64)
    e = np.zeros((N, K // 16, 8, 2), dtype=np.int64)
    for j in range(8):
        for h in range(2):
            e[:, :, j, h] = (words >> np.uint64(16 * h + 2 * j)) & np.uint64(3)
    return (e.reshape(N, K) - 1).astype(np.int8)


def pack_weights(codes: np.ndarray, s: np.ndarray):
    """The load-time step: (packed uint8 [N,K/4], qT int8 [G,N], sw fp32 [N])."""
    q, sw, _ = row_scale_decompose(s)
    return pack_codes(codes), np.ascontiguousarray(q.T), sw


def expand_w_int8(codes: np.ndarray, q: np.ndarray) -> np.ndarray:
    """W_int8[n,k] = code[n,k] * q[n, k // 128] as int16 (P1 §4)."""
    c = np.asarray(codes, dtype=np.int16)
    N, K = c.shape
    return c * np.repeat(np.asarray(q, dtype=np.int16), GROUP, axis=1)[:, :K]


# --------------------------------------------------------------------------
# Integer GEMM and epilogue (P1 §4)
# --------------------------------------------------------------------------

def int_gemm(xq: np.ndarray, w_int8: np.ndarray) -> np.ndarray:
    """acc[m,n] = sum_k xq[m,k] W_int8[n,k], exact.

    Evaluated as an fp64 matmul: every product is an integer of magnitude
    <= 127*127 and every partial sum stays below 2^53, so the result is exact
    whatever order the library sums in.
    """
    a = np.asarray(xq, dtype=np.float64)
    b = np.asarray(w_int8, dtype=np.float64)
    return (a @ b.T).astype(np.int64)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 by round-to-nearest-even, as uint16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def epilogue(acc: np.ndarray, sw: np.ndarray, sx: np.ndarray) -> np.ndarray:
    """y[m,n] = fl32(fl32(fl32(acc) sw[n]) sx[m]) in fp32 (P1 §4 row/token rescale)."""
    a = np.asarray(acc, dtype=np.int64).astype(np.float32)
    t = (a * np.asarray(sw, dtype=np.float32)[None, :]).astype(np.float32)
    return (t * np.asarray(sx, dtype=np.float32)[:, None]).astype(np.float32)


def layer(x_bits, codes, s, signs=None, rows: np.ndarray | None = None) -> dict:
    """The whole quantised layer; `rows` restricts the output features computed.

    Returns a dict with xq, sx, q, sw, acc (int64), y32 (fp32), ybf (bf16 bits).
    """
    xq, sx = rotate_quant(x_bits, signs)
    q, sw, _ = row_scale_decompose(s)
    if rows is not None:
        codes = np.asarray(codes)[rows]
        q = q[rows]
        sw = sw[rows]
    acc = int_gemm(xq, expand_w_int8(codes, q))
    y32 = epilogue(acc, sw, sx)
    return dict(xq=xq, sx=sx, q=q, sw=sw, acc=acc, y32=y32, ybf=f32_to_bf16_bits(y32))


def reference_fp64(x_bits, codes, s, signs=None, rows: np.ndarray | None = None) -> np.ndarray:
    """The unquantised ternary layer in fp64: y = rot(x) (code * s)^T."""
    xr = rotate_fp64(x_bits, signs)
    c = np.asarray(codes, dtype=np.float64)
    sf = np.asarray(s, dtype=np.float16).astype(np.float64)
    if rows is not None:
        c = c[rows]
        sf = sf[rows]
    W = c * np.repeat(sf, GROUP, axis=1)[:, :c.shape[1]]
    return xr @ W.T


def rel_fro(y: np.ndarray, ref: np.ndarray) -> float:
    """Relative Frobenius error ||y - ref||_F / ||ref||_F."""
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(np.asarray(y, dtype=np.float64) - ref) / np.linalg.norm(ref))


# --------------------------------------------------------------------------
# Float-activation decode (P1 §5): the same ternary layer without activation
# quantisation, accumulated in floating point.
# --------------------------------------------------------------------------

def layer_float_act(x_bits, codes, s, signs=None, rows: np.ndarray | None = None) -> dict:
    """y[m,n] = sum_g s[n,g] sum_{k in g} code[n,k] xr[m,k] with xr the fp32
    rotation (bit-identical to the library's) and s the fp16 group scales.

    P1 §5 "効かなかったもの" contrasts the int8 dp4a decode GEMV with the
    production decode, which keeps the activations in floating point and was
    the more accurate of the two. Reading: the rotated activations stay fp32,
    the weights are code * s with the original fp16 scales (no int8 q), and
    the result is the plain definition evaluated in fp64 (every product is
    exact in fp64; the sums carry fp64 rounding only, far below the fp32
    tolerance a GPU evaluation is held to).

    Returns y64 [M,N] (fp64) and T [M,N] = sum_g |s| sum_k |code xr|, the sum
    of the absolute terms that bounds the rounding error of any fp32
    evaluation order.
    """
    xr = rotate_fp32(x_bits, signs).astype(np.float64)
    c = np.asarray(codes, dtype=np.float64)
    sf = np.asarray(s, dtype=np.float16).astype(np.float64)
    if rows is not None:
        c = c[rows]
        sf = sf[rows]
    N, K = c.shape
    W = c * np.repeat(sf, GROUP, axis=1)[:, :K]
    y64 = xr @ W.T
    T = np.abs(xr) @ np.abs(W).T
    return dict(xr=xr.astype(np.float32), y64=y64, T=T)

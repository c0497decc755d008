"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each pin_* function checks the oracle against something the source pages or
mathematics fix: a library's Sylvester Hadamard, integer identities, the
recursion and rank-swap control of the TP port, hand-derived one-hot examples,
brute-force loops on tiny shapes, and the layer error level the pages print.
The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU, via monkeypatch) and check that some pin catches each one.

Pages: [P1] Qiita item ecc183fae033565af7cb (Ternary-Bonsai-2-27B on
2× RTX 5070 with vLLM TP=2): 前提 (format), §1 "TP=2 への移植" (recursion and
the CPU mock: 2.6e-3 vs TP=1, 1.44 with ranks swapped), §4 "効いた高速化"
(q, W_int8, per-token int8, per-layer error 2.4e-3 -> 9.5e-3).
"""

import json
import os
import warnings

import numpy as np
import pytest
import scipy.linalg

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth

# a pin that overflows or divides by zero somewhere unplanned fails loudly
pytestmark = pytest.mark.filterwarnings("error::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pages():
    with open(os.path.join(GOLDEN, "pages_numbers.json")) as f:
        return json.load(f)


def _bf16(v):
    return synth.bf16_bits_from_f32(np.asarray(v, dtype=np.float32))


# ------------------------------------------------------------------ pins

def pin_hadamard():
    H = O.hadamard(1024)
    assert np.array_equal(H @ H.T, 1024 * np.eye(1024, dtype=np.int64))
    for n in (2, 4, 8, 64, 512, 1024):
        assert np.array_equal(O.hadamard(n), scipy.linalg.hadamard(n))


def pin_fwht_vs_library():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((3, 1024))
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    got = O.fwht(v, np.float64)
    ref = v @ H.T
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def pin_sylvester_recursion():
    """P1 §1: H1024 [a; b] = [H512 a + H512 b; H512 a - H512 b]."""
    rng = np.random.default_rng(2)
    for _ in range(4):
        a, b = rng.standard_normal(512), rng.standard_normal(512)
        full = O.fwht(np.concatenate([a, b]), np.float64)
        ha = scipy.linalg.hadamard(512) @ a
        hb = scipy.linalg.hadamard(512) @ b
        split = np.concatenate([ha + hb, ha - hb])
        assert np.max(np.abs(full - split)) <= 1e-11 * np.max(np.abs(full))


def pin_rank_swap_control():
    """P1 §1: swapping the two ranks' sum/difference is detected (page: 1.44).

    For the exact rotation the swapped result differs by [-2 H b; 2 H b], a
    relative error of 2|Hb| / sqrt(|Ha|^2 + |Hb|^2), about sqrt(2) for halves
    of equal energy.
    """
    pages = _pages()
    rng = np.random.default_rng(3)
    errs = []
    for _ in range(8):
        a, b = rng.standard_normal(512), rng.standard_normal(512)
        full = O.fwht(np.concatenate([a, b]), np.float64)
        ha = O.fwht(a, np.float64)
        hb = O.fwht(b, np.float64)
        swapped = np.concatenate([ha - hb, ha + hb])
        e = np.linalg.norm(swapped - full) / np.linalg.norm(full)
        closed = 2 * np.linalg.norm(hb) / np.sqrt(np.linalg.norm(ha) ** 2 + np.linalg.norm(hb) ** 2)
        assert abs(e - closed) <= 1e-12
        errs.append(e)
    assert abs(np.mean(errs) - np.sqrt(2.0)) < 0.1
    assert abs(pages["tp_split_rank_swap_rel_error"]["value"] - np.sqrt(2.0)) < 0.1


def pin_tp_split_bf16_level():
    """P1 §1: the split evaluated with bf16 tensors is off only at bf16 rounding level (2.6e-3)."""
    pages = _pages()
    rng = np.random.default_rng(4)

    def r16(v):
        return synth.bf16_bits_to_f32(_bf16(v)).astype(np.float64)

    errs = []
    for _ in range(16):
        x = r16(rng.standard_normal(1024))
        tp1 = r16(O.fwht(x, np.float64) / 32.0)
        ha = r16(O.fwht(x[:512], np.float64) / 32.0)
        hb = r16(O.fwht(x[512:], np.float64) / 32.0)
        tp2 = np.concatenate([r16(ha + hb), r16(ha - hb)])
        errs.append(np.linalg.norm(tp2 - tp1) / np.linalg.norm(tp1))
    lvl = pages["tp_split_rel_error_vs_tp1"]["value"]
    assert lvl / 4 < np.mean(errs) < lvl * 2


def pin_rotation_orthonormal():
    rng = np.random.default_rng(5)
    xb = _bf16(rng.standard_normal((2, 2048)))
    xr = O.rotate_fp64(xb)
    x = synth.bf16_bits_to_f32(xb).astype(np.float64)
    assert np.allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    # (H/32)^2 = I: rotating the rotated vector returns the input.
    H = scipy.linalg.hadamard(1024) / 32.0
    back = np.concatenate([xr[:, :1024] @ H.T, xr[:, 1024:] @ H.T], axis=1)
    assert np.max(np.abs(back - x)) < 1e-12 * np.max(np.abs(x))


def pin_rotate_fp32_near_fp64():
    rng = np.random.default_rng(6)
    xb = _bf16(rng.standard_normal((4, 3072)) * 3)
    r32 = O.rotate_fp32(xb).astype(np.float64)
    r64 = O.rotate_fp64(xb)
    # ten butterfly stages, each one fp32 rounding of a value bounded by the block's L1 norm
    x = synth.bf16_bits_to_f32(xb).astype(np.float64).reshape(4, 3, 1024)
    bound = 10 * 2.0 ** -24 * np.abs(x).sum(axis=2) / 32.0
    err = np.abs(r32 - r64).reshape(4, 3, 1024).max(axis=2)
    assert np.all(err <= bound)


def pin_quant_one_hot():
    """Hand-derived: x = 2.0 at channel j0 of block 0, zero elsewhere.

    xr = (2/32) H[:, j0] = +-1/16 on block 0 and 0 on block 1, so a = 1/16,
    127/a = 2032 exactly, xq = 127 H[:, j0] on block 0, 0 on block 1.
    """
    for j0 in (0, 5, 777):
        x = np.zeros((1, 2048), dtype=np.float32)
        x[0, j0] = 2.0
        xq, sx = O.rotate_quant(_bf16(x))
        want = np.zeros(2048, dtype=np.int64)
        want[:1024] = 127 * scipy.linalg.hadamard(1024)[:, j0]
        assert np.array_equal(xq[0].astype(np.int64), want)
        assert sx[0] == np.float32(1.0 / 16.0) / np.float32(127.0)
        assert abs(float(sx[0]) * 127 * 16 - 1) < 1e-7


def pin_quant_properties():
    rng = np.random.default_rng(7)
    xb = _bf16(rng.standard_normal((5, 2048)))
    xb[3] = 0  # an all-zero token (bf16 +0)
    xr = O.rotate_fp32(xb)
    xq, sx = O.quantize_per_token(xr)
    for m in range(5):
        if m == 3:
            assert sx[m] == 0 and not np.any(xq[m])
            continue
        assert np.max(np.abs(xq[m].astype(np.int64))) == 127
        assert np.min(xq[m].astype(np.int64)) >= -127
        err = np.abs(xq[m].astype(np.float64) * sx[m] - xr[m])
        assert np.all(err <= 0.5 * float(sx[m]) * (1 + 1e-5))


def pin_quant_tiny_token():
    """Hand-derived: tokens of bf16 subnormals, where fl32(127 / a) overflows to +inf.

    Token 0: x[0] = 2^-133 (bf16 bits 0x0001), x[1] = 2^-132 (0x0002), zero
    elsewhere, K = 2048. Block 0 rotates to (2^-133 + 2^-132) / 32 = 3 2^-138 at
    even i and (2^-133 - 2^-132) / 32 = -2^-138 at odd i, all exact fp32
    subnormals; block 1 is zero. a = 3 2^-138 < 127 / FLT_MAX, so inv = +inf:
    block 0 codes to +127 / -127 (even / odd i), block 1's zeros to 0, and
    sx = fl32(3 2^-138 / 127) = 48 2^-149 (3 2^11 / 127 = 48.38 rounds to 48).
    Token 1: x[0] = 2^-133 alone: block 0 is 2^-138 everywhere -> +127,
    block 1 -> 0, sx = fl32(2^-138 / 127) = 16 2^-149 (2^11 / 127 = 16.13).
    """
    x = np.zeros((2, 2048), dtype=np.uint16)
    x[0, 0], x[0, 1] = 0x0001, 0x0002
    x[1, 0] = 0x0001
    xr = O.rotate_fp32(x)
    tiny = np.float32(2.0 ** -138)
    assert np.all(xr[0, 0:1024:2] == np.float32(3) * tiny)
    assert np.all(xr[0, 1:1024:2] == -tiny) and not np.any(xr[0, 1024:])
    with np.errstate(over="ignore"):
        assert np.float32(127) / (np.float32(3) * tiny) == np.inf
    xq, sx = O.quantize_per_token(xr)
    want0 = np.zeros(2048, dtype=np.int64)
    want0[0:1024:2], want0[1:1024:2] = 127, -127
    want1 = np.zeros(2048, dtype=np.int64)
    want1[:1024] = 127
    assert np.array_equal(xq[0].astype(np.int64), want0)
    assert np.array_equal(xq[1].astype(np.int64), want1)
    assert sx[0] == np.float32(48 * 2.0 ** -149) and sx[1] == np.float32(16 * 2.0 ** -149)
    # the boundary: just above 127 / FLT_MAX the quotient is finite and the
    # ordinary rule applies (one element reaches 127, the half-ulp bound holds)
    a = np.float32(np.float32(127) / np.finfo(np.float32).max)
    a_up = np.nextafter(np.nextafter(a, np.float32(1)), np.float32(1))
    xr2 = np.array([[a_up, -a_up / 2, 0, a_up / 4] + [0] * 1020], dtype=np.float32)
    xq2, sx2 = O.quantize_per_token(xr2)
    assert xq2[0, :4].tolist() == [127, -64, 0, 32]


def pin_pack_layout_handworked():
    """One 16-code word worked by hand (layout: field at bit 16h+2j holds code[2j+h]+1).

    codes  = [1,-1,0,1, 0,0,-1,-1, 1,1,0,-1, -1,0,1,0]
    even k -> e = [2,1,1,0,2,1,0,2] -> low half  0x8616
    odd k  -> e = [0,2,1,0,2,0,1,1] -> high half 0x5218
    """
    codes = np.array([[1, -1, 0, 1, 0, 0, -1, -1, 1, 1, 0, -1, -1, 0, 1, 0]], dtype=np.int8)
    packed = O.pack_codes(codes)
    assert packed.tolist() == [[0x16, 0x86, 0x18, 0x52]]
    assert np.array_equal(O.unpack_codes(packed, 16), codes)


def pin_pack_roundtrip():
    rng = np.random.default_rng(8)
    c = synth.ternary_codes(rng, 8, 2048, 0.4)
    assert np.array_equal(O.unpack_codes(O.pack_codes(c), 2048), c)


def pin_row_scale_decompose():
    """P1 §4: W_int8 = code q fits exactly in int8; the row's max group has |q| = 127."""
    rng = np.random.default_rng(9)
    s = synth.group_scales(rng, 64, 4096, -4.0, 0.7)
    s[5, :] = 0                                   # an all-zero row
    s[6, 3] = -2 * np.max(np.abs(s[6]))            # a negative scale of largest magnitude
    s[7, :] = np.float16(2.0 ** -20)               # tiny but normal scales, all equal
    q, sw, smax = O.row_scale_decompose(s)
    sf = s.astype(np.float64)
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    for n in range(64):
        if n == 5:
            assert not np.any(q[n]) and sw[n] == 0
            continue
        assert np.max(np.abs(q[n].astype(np.int64))) == 127
        err = np.abs(q[n].astype(np.float64) * float(sw[n]) - sf[n])
        assert np.all(err <= float(smax[n]) / 254.0 * (1 + 2.0 ** -20))
    assert q[6, 3] == -127 and np.all(q[7] == 127)
    # brute force on a few rows: the nearest integer to 127 s / smax, ties to even
    for n in (0, 1, 6):
        for g in range(s.shape[1]):
            t = float(np.float32(np.float32(127.0) * np.float32(s[n, g])) / np.float32(smax[n]))
            lo = np.floor(t)
            want = lo + 1 if (t - lo > 0.5 or (t - lo == 0.5 and lo % 2 == 1)) else lo
            assert q[n, g] == want


def pin_int_gemm_bruteforce():
    rng = np.random.default_rng(10)
    for (M, N, K) in ((1, 3, 1024), (3, 4, 1024), (2, 2, 2048)):
        xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        codes = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
        q = rng.integers(-127, 128, size=(N, K // 128)).astype(np.int8)
        got = O.int_gemm(xq, O.expand_w_int8(codes, q))
        for m in range(M):
            for n in range(N):
                acc = 0
                for k in range(K):
                    acc += int(xq[m, k]) * int(codes[n, k]) * int(q[n, k // 128])
                assert got[m, n] == acc


def pin_int_gemm_extremes():
    K = 1024
    xq = np.full((2, K), 127, dtype=np.int8)
    xq[1, 1::2] = -127
    codes = np.ones((2, K), dtype=np.int8)
    q = np.full((2, K // 128), 127, dtype=np.int8)
    acc = O.int_gemm(xq, O.expand_w_int8(codes, q))
    assert acc[0, 0] == 16_516_096 and acc[1, 0] == 0
    codes[1, 1::2] = -1
    acc = O.int_gemm(xq, O.expand_w_int8(codes, q))
    assert acc[1, 1] == 16_516_096 and acc[0, 1] == 0


def pin_epilogue_closed_form():
    rng = np.random.default_rng(11)
    acc = rng.integers(-(2 ** 28), 2 ** 28, size=(4, 8))
    sw = rng.random(8).astype(np.float32) * 1e-3
    sx = rng.random(4).astype(np.float32) * 1e-2
    y = O.epilogue(acc, sw, sx).astype(np.float64)
    exact = acc.astype(np.float64) * sw.astype(np.float64)[None, :] * sx.astype(np.float64)[:, None]
    assert np.all(np.abs(y - exact) <= 3 * 2.0 ** -24 * np.abs(exact))
    bits = O.f32_to_bf16_bits(np.array([1.0, 1.00390625, 1.01171875, -3.0], dtype=np.float32))
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3 * 2^-8 is a tie -> even (1 + 2^-6)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC040]


def pin_layer_one_hot_exact():
    """Whole layer on hand-derived inputs where quantisation is lossless.

    x = 2.0 at channel j0, row n codes = H[j0, :] on block 0 (0 on block 1),
    all scales 2^-4: y = sum_i (2/32) H[i,j0]^2 2^-4 = 1024 / 256 = 4.
    """
    j0 = 5
    x = np.zeros((1, 2048), dtype=np.float32)
    x[0, j0] = 2.0
    codes = np.zeros((2, 2048), dtype=np.int8)
    codes[0, :1024] = scipy.linalg.hadamard(1024)[j0]
    codes[1, :1024] = 1
    s = np.full((2, 16), 2.0 ** -4, dtype=np.float16)
    r = O.layer(_bf16(x), codes, s)
    assert r["acc"][0, 0] == 127 * 127 * 1024
    assert r["acc"][0, 1] == 0
    assert abs(float(r["y32"][0, 0]) - 4.0) < 4.0 * 1e-6
    ref = O.reference_fp64(_bf16(x), codes, s)
    assert abs(ref[0, 0] - 4.0) < 1e-12


def pin_layer_error_level():
    """P1 §4: the int8 path's per-layer error is about 9.5e-3; the bound used is 1.5e-2."""
    pages = _pages()
    L = synth.config_inputs("tiny")
    r = O.layer(L.x_bits, L.codes, L.s)
    e = O.rel_fro(r["y32"], O.reference_fp64(L.x_bits, L.codes, L.s))
    assert pages["int8_path_layer_rel_error"]["value"] / 3 < e < 1.5e-2


PINS = [pin_hadamard, pin_fwht_vs_library, pin_sylvester_recursion, pin_rank_swap_control,
        pin_tp_split_bf16_level, pin_rotation_orthonormal, pin_rotate_fp32_near_fp64,
        pin_quant_one_hot, pin_quant_properties, pin_quant_tiny_token,
        pin_pack_layout_handworked, pin_pack_roundtrip,
        pin_row_scale_decompose, pin_int_gemm_bruteforce, pin_int_gemm_extremes,
        pin_epilogue_closed_form, pin_layer_one_hot_exact, pin_layer_error_level]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ------------------------------------------------------------------ planted mistakes

def _fwht_wrong_sign(v, dtype=np.float32):
    v = np.array(v, dtype=dtype, copy=True)
    n = v.shape[-1]
    lead = v.shape[:-1]
    h = 1
    while h < n:
        w = v.reshape(lead + (n // (2 * h), 2, h))
        a, b = w[..., 0, :].copy(), w[..., 1, :].copy()
        w[..., 0, :] = a - b          # planted: sum and difference exchanged
        w[..., 1, :] = a + b
        v = w.reshape(lead + (n,))
        h *= 2
    return v


def _expand_shifted_group(codes, q):
    c = np.asarray(codes, dtype=np.int16)
    qq = np.roll(np.asarray(q, dtype=np.int16), 1, axis=1)   # planted: off-by-one group
    return c * np.repeat(qq, 128, axis=1)


def _expand_rows_reversed(codes, q):
    c = np.asarray(codes, dtype=np.int16)
    qq = np.asarray(q, dtype=np.int16)[::-1]                 # planted: q rows reversed
    return c * np.repeat(qq, 128, axis=1)


def _quant_128(xr):
    xr = np.asarray(xr, dtype=np.float32)
    a = np.max(np.abs(xr), axis=1)
    inv = np.float32(128) / a                                # planted: 128 levels
    xq = np.clip(np.rint(xr * inv[:, None]), -128, 127).astype(np.int8)
    return xq, (a / np.float32(128)).astype(np.float32)


def _quant_nan_unhandled(xr):
    xr = np.asarray(xr, dtype=np.float32)
    a = np.max(np.abs(xr), axis=1)
    inv = (np.float32(127) / a).astype(np.float32)
    t = xr * inv[:, None]
    # planted: NaN (0 * inf) left to the int8 cast, +-inf clamped, as a naive port would
    xq = np.clip(np.rint(np.nan_to_num(t, nan=127.0)), -127, 127).astype(np.int8)
    return xq, (a / np.float32(127)).astype(np.float32)


def _decompose_no_abs(s):
    sf = np.asarray(s, dtype=np.float16).astype(np.float32)
    smax = np.max(sf, axis=1)                                # planted: max without |.|
    q = np.rint(np.float32(127) * sf / smax[:, None]).clip(-128, 127).astype(np.int8)
    return q, smax / np.float32(127), smax


def _pack_swapped_halves(codes):
    c = np.asarray(codes)
    N, K = c.shape
    e = (c.astype(np.int64) + 1).reshape(N, K // 16, 8, 2)
    words = np.zeros((N, K // 16), dtype=np.uint64)
    for j in range(8):
        for h in range(2):
            words |= e[:, :, j, 1 - h].astype(np.uint64) << np.uint64(16 * h + 2 * j)
    return words.astype("<u4").view(np.uint8).reshape(N, K // 4)


def _epilogue_no_token_scale(acc, sw, sx):
    a = np.asarray(acc, dtype=np.int64).astype(np.float32)
    return (a * np.asarray(sw, dtype=np.float32)[None, :]).astype(np.float32)   # planted: sx dropped


MUTATIONS = [
    ("fwht", _fwht_wrong_sign, [pin_fwht_vs_library, pin_quant_one_hot]),
    ("expand_w_int8", _expand_shifted_group, [pin_int_gemm_bruteforce]),
    ("expand_w_int8", _expand_rows_reversed, [pin_int_gemm_bruteforce]),
    ("quantize_per_token", _quant_128, [pin_quant_one_hot]),
    ("quantize_per_token", _quant_nan_unhandled, [pin_quant_tiny_token]),
    ("row_scale_decompose", _decompose_no_abs, [pin_row_scale_decompose]),
    ("pack_codes", _pack_swapped_halves, [pin_pack_layout_handworked]),
    ("epilogue", _epilogue_no_token_scale, [pin_epilogue_closed_form]),
]


@pytest.mark.parametrize("name,fake,pins", MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fake, pins):
    monkeypatch.setattr(O, name, fake)
    caught = []
    for pin in pins:
        with warnings.catch_warnings():
            warnings.simplefilter("ignore", RuntimeWarning)   # the planted versions may overflow
            try:
                pin()
            except (AssertionError, ValueError, IndexError):
                caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake in {name}"


def test_all_pins_hold_unpatched():
    for pin in PINS:
        pin()

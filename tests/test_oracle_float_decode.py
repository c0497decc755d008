"""Pins of the float-activation decode oracle (oracle.ternary_linear.layer_float_act).

Page: Qiita item ecc183fae033565af7cb §5 "効かなかったもの" (the production
decode keeps floating-point activations; the int8 dp4a GEMV was less exact).
The pins fix it to closed forms and to independent computations:
  * codes all +1 and unit scales: y = sum_k xr_k = 32 sum_b x[1024 b] (the
    Hadamard row sums vanish except for column 0 of each block);
  * a one-hot code at k0: y = s[n, k0/128] xr[k0] exactly;
  * negating the codes negates y; scaling s by 2 doubles y exactly;
  * the explicit fp64 matrix product of the rotation (reference_fp64) agrees
    to 1e-6 relative (only the fp32 rounding of xr differs);
  * it is closer to the unquantised reference than the int8 layer is.
"""

import numpy as np

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth


def _x(M, K, seed=5):
    rng = np.random.default_rng(seed)
    return synth.bf16_bits_from_f32(rng.standard_normal((M, K)).astype(np.float32))


def test_all_plus_one_closed_form():
    M, K, N = 3, 3072, 4
    xb = _x(M, K)
    codes = np.ones((N, K), dtype=np.int8)
    s = np.ones((N, K // 128), dtype=np.float16)
    y = O.layer_float_act(xb, codes, s)["y64"]
    x = O.bf16_to_f32(xb).astype(np.float64)
    closed = 32.0 * x[:, ::1024].sum(axis=1)
    assert np.allclose(y, closed[:, None], rtol=1e-6, atol=1e-6)


def test_one_hot_is_exact():
    M, K, N = 2, 2048, 3
    xb = _x(M, K, 6)
    codes = np.zeros((N, K), dtype=np.int8)
    k0 = [5, 1030, 2047]
    for n, k in enumerate(k0):
        codes[n, k] = 1 if n != 1 else -1
    s = np.full((N, K // 128), 0.5, dtype=np.float16)
    s[2, 2047 // 128] = 0.125
    out = O.layer_float_act(xb, codes, s)
    xr = out["xr"].astype(np.float64)
    for n, k in enumerate(k0):
        expect = (1 if n != 1 else -1) * float(s[n, k // 128]) * xr[:, k]
        assert np.array_equal(out["y64"][:, n], expect)


def test_sign_and_scale_symmetry():
    inp = synth.config_inputs("tiny", M=2, N=128)
    a = O.layer_float_act(inp.x_bits, inp.codes, inp.s)["y64"]
    b = O.layer_float_act(inp.x_bits, -inp.codes, inp.s)["y64"]
    c = O.layer_float_act(inp.x_bits, inp.codes, (inp.s.astype(np.float32) * 2).astype(np.float16))["y64"]
    assert np.array_equal(b, -a)
    assert np.array_equal(c, 2 * a)


def test_matches_fp64_rotation_reference():
    inp = synth.config_inputs("tiny", M=4, N=128)
    y = O.layer_float_act(inp.x_bits, inp.codes, inp.s)["y64"]
    ref = O.reference_fp64(inp.x_bits, inp.codes, inp.s)
    assert O.rel_fro(y, ref) < 1e-6


def test_more_accurate_than_the_int8_layer():
    inp = synth.config_inputs("tiny", M=8, N=128)
    ref = O.reference_fp64(inp.x_bits, inp.codes, inp.s)
    yf = O.layer_float_act(inp.x_bits, inp.codes, inp.s)["y64"]
    yi = O.layer(inp.x_bits, inp.codes, inp.s)["y32"]
    assert O.rel_fro(yf, ref) < 1e-3 * O.rel_fro(yi, ref)


def test_abs_sum_bounds_the_value():
    inp = synth.config_inputs("tiny", M=2, N=128)
    out = O.layer_float_act(inp.x_bits, inp.codes, inp.s)
    assert np.all(np.abs(out["y64"]) <= out["T"] * (1 + 1e-12))

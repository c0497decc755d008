"""GPU parity of the tensor-core decode (tl_linear_decode_tc), through the C ABI.

The int32 accumulator must equal the oracle's (Qiita item ecc183fae033565af7cb
§4) and the dp4a decode's bit for bit; fp32 y within 1e-3 of the oracle (equal
in practice), bf16 within one ulp. The cases cover M = 1..32 (one to four
8-token MMA tiles, partly filled), clusters of CTAs splitting K, the smallest
and the deepest K, and the largest accumulator.
"""

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth

pytestmark = pytest.mark.gpu

SENT = -(2 ** 31)


@pytest.fixture(scope="module")
def tl():
    from quantized_linear_layers_block_gb300 import build
    build.build()
    from quantized_linear_layers_block_gb300 import tl as _tl
    _tl.lib()
    assert _tl.tl_get_status() == _tl.TL_OK
    return _tl


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).cuda()


def x_dev(xb):
    return dev(xb.view(np.int16), torch.bfloat16)


def pack(tl, L):
    return tl.tl_pack_weights(dev(L.codes), dev(L.s.view(np.int16), torch.float16))


def _run_tc(tl, L, packed, qT, sw, y_dtype=4, signs=None):
    xq, sx = tl.tl_rotate_quant_act(x_dev(L.x_bits), signs=signs, xq_dtype=tl.TL_F16)
    acc = torch.full((L.M, L.N), SENT, dtype=torch.int32, device="cuda")
    y = tl.tl_linear_decode_tc(packed, qT, sw, xq, sx, L.N, L.K, y_dtype, acc_dbg=acc)
    assert tl.tl_get_status() == tl.TL_OK
    return acc.cpu().numpy().astype(np.int64), y


def _rows(N, n=160, seed=0):
    return None if N <= 1024 else np.sort(np.random.default_rng(seed).choice(N, size=n, replace=False))


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 13, 16, 17, 24, 25, 31, 32])
def test_decode_tc_matches_oracle_and_dp4a(tl, M):
    L = synth.config_inputs("decode", M=M, N=640, K=3072)
    packed, qT, sw = pack(tl, L)
    acc, y = _run_tc(tl, L, packed, qT, sw)
    r = O.layer(L.x_bits, L.codes, L.s)
    assert np.array_equal(acc, r["acc"])
    yv = y.cpu().numpy()
    assert np.max(np.abs(yv - r["y32"])) <= 1e-3 * np.max(np.abs(r["y32"]))
    xq, sx = tl.tl_rotate_quant_act(x_dev(L.x_bits), xq_dtype=tl.TL_I8)
    acc2 = torch.empty((M, L.N), dtype=torch.int32, device="cuda")
    y2 = tl.tl_linear_decode(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=acc2)
    assert tl.tl_get_status() == tl.TL_OK
    assert np.array_equal(acc2.cpu().numpy(), acc)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("M,N,K", [(1, 17408, 5120), (16, 17408, 5120), (32, 17408, 5120),
                                   (1, 5120, 17408), (8, 5120, 17408), (32, 5120, 17408),
                                   (4, 128, 1024), (2, 256, 32768), (7, 34816, 5120),
                                   (32, 384, 1024)])
def test_decode_tc_shapes(tl, M, N, K):
    """The MLP shapes (each K split over a cluster of 2 or 4 CTAs), the smallest
    and the deepest layers, and a wide gate+up layer; sampled rows."""
    L = synth.config_inputs("decode", M=M, N=N, K=K)
    packed, qT, sw = pack(tl, L)
    acc, y = _run_tc(tl, L, packed, qT, sw, y_dtype=3)
    rows = _rows(N)
    r = O.layer(L.x_bits, L.codes, L.s, rows=rows)
    sel = slice(None) if rows is None else rows
    assert np.array_equal(acc[:, sel], r["acc"])
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)[:, sel].astype(np.int32)
    ref = r["ybf"].astype(np.int32)
    a = np.where(yb & 0x8000, 0x8000 - yb, yb)
    b = np.where(ref & 0x8000, 0x8000 - ref, ref)
    assert np.max(np.abs(a - b)) <= 1


def test_decode_tc_extremes(tl):
    """The largest accumulator: x one-hot per block rotates to xq = 127 everywhere;
    all codes +1 and equal scales (q = 127) give 127 * 127 * K; alternating codes
    cancel to 0; a zero token, a negative-max token."""
    K, N, M = 8192, 256, 4
    x = np.zeros((M, K), dtype=np.float32)
    x[0, ::1024] = 2.0
    x[1, ::1024] = -2.0
    x[3, 5] = 7.0
    codes = np.ones((N, K), dtype=np.int8)
    codes[1::2, 1::2] = -1
    codes[2] = 0
    s = np.full((N, K // 128), 2.0 ** -4, dtype=np.float16)
    xb = synth.bf16_bits_from_f32(x)
    packed, qT, sw = tl.tl_pack_weights(dev(codes), dev(s.view(np.int16), torch.float16))
    xq, sx = tl.tl_rotate_quant_act(x_dev(xb), xq_dtype=tl.TL_F16)
    acc = torch.full((M, N), SENT, dtype=torch.int32, device="cuda")
    tl.tl_linear_decode_tc(packed, qT, sw, xq, sx, N, K, 4, acc_dbg=acc)
    assert tl.tl_get_status() == tl.TL_OK
    r = O.layer(xb, codes, s)
    a = acc.cpu().numpy().astype(np.int64)
    assert np.array_equal(a, r["acc"])
    assert a[0, 0] == 127 * 127 * K and a[1, 0] == -127 * 127 * K and a[0, 1] == 0
    assert not np.any(a[2])


def test_decode_tc_tiny_tokens_and_signs(tl):
    K, N = 2048, 256
    x = np.zeros((3, K), dtype=np.uint16)
    x[0, 0], x[0, 1] = 0x0001, 0x0002
    x[1, 0] = 0x0001
    x[2] = synth.bf16_bits_from_f32(np.random.default_rng(2).standard_normal(K).astype(np.float32))
    L = synth.config_inputs("decode", M=3, N=N, K=K)
    L.x_bits = x
    packed, qT, sw = pack(tl, L)
    acc, y = _run_tc(tl, L, packed, qT, sw)
    r = O.layer(x, L.codes, L.s)
    assert np.array_equal(acc, r["acc"])
    assert np.array_equal(y.cpu().numpy().view(np.uint32), r["y32"].view(np.uint32))
    signs = np.where(np.random.default_rng(9).random(K) < 0.5, -1, 1).astype(np.int8)
    acc_s, _ = _run_tc(tl, L, packed, qT, sw, signs=dev(signs))
    assert np.array_equal(acc_s, O.layer(x, L.codes, L.s, signs=signs)["acc"])


def test_decode_tc_argument_errors(tl):
    L = synth.config_inputs("decode", M=2, N=128, K=1024)
    packed, qT, sw = pack(tl, L)
    xf, sx = tl.tl_rotate_quant_act(x_dev(L.x_bits), xq_dtype=tl.TL_F16)
    y = torch.empty((2, 128), dtype=torch.float32, device="cuda")
    lib = tl.lib()
    P = lambda t: t.data_ptr()  # noqa: E731
    st = torch.cuda.current_stream().cuda_stream
    assert lib.tl_linear_decode_tc(P(packed), P(qT), P(sw), P(xf), P(sx), 33, 128, 1024, P(y), 4,
                                   None, st) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode_tc(P(packed), P(qT), P(sw), None, P(sx), 2, 128, 1024, P(y), 4,
                                   None, st) == tl.TL_EINVAL
    assert lib.tl_linear_decode_tc(P(packed), P(qT), P(sw), P(xf) + 4, P(sx), 2, 128, 1024, P(y), 4,
                                   None, st) == tl.TL_EINVAL
    assert lib.tl_linear_decode_tc(P(packed), P(qT), P(sw), P(xf), P(sx), 2, 100, 1024, P(y), 4,
                                   None, st) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode_tc(P(packed), P(qT), P(sw), P(xf), P(sx), 0, 128, 1024, P(y), 4,
                                   None, st) == tl.TL_OK
    assert tl.tl_get_status() == tl.TL_OK

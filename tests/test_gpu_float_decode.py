"""GPU parity of the float-activation decode (tl_rotate_act, tl_linear_decode_f32act)
against the oracle (oracle.ternary_linear.layer_float_act).

The rotation is bit-exact. The GEMV sums in fp32 in the kernel's own order;
every product code * xr is exact, and each term passes through at most
K/1024 + 23 roundings (16 FMAs in a chunk partial, the even/odd add, the
scale FMA, one FMA per chunk step of the lane, 5 shuffle-tree adds), so
|y - y64| <= gamma_d * T with T = sum |s code xr| and gamma_d = d u / (1 - d u),
u = 2^-24: at most 3.3e-6 T for K <= 32768. The test holds it to 4e-6 T
(plus 2^-8 |y| for a bf16 output).

Page: Qiita item ecc183fae033565af7cb §5 "効かなかったもの".
"""

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth
from quantized_linear_layers_block_gb300 import tl

pytestmark = pytest.mark.gpu

TOL = 4e-6


def _dev(inp, signs=None):
    codes = torch.from_numpy(inp.codes).cuda()
    s = torch.from_numpy(inp.s).cuda()
    x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    packed, _, _ = tl.tl_pack_weights(codes, s)
    sg = None if signs is None else torch.from_numpy(signs).cuda()
    xr = tl.tl_rotate_act(x, signs=sg)
    return packed, s, xr


@pytest.mark.parametrize("M,K", [(1, 1024), (3, 2048), (2, 17408), (5, 5120)])
def test_rotate_act_is_bit_exact(M, K):
    inp = synth.config_inputs("tiny", M=M, K=K, N=128)
    rng = np.random.default_rng(K)
    signs = rng.choice(np.array([-1, 1], dtype=np.int8), size=K)
    for sg in (None, signs):
        _, _, xr = _dev(inp, sg)
        torch.cuda.synchronize()
        assert np.array_equal(xr.cpu().numpy().view(np.uint32), O.rotate_fp32(inp.x_bits, sg).view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(1, 256, 1024), (1, 128, 2048), (2, 384, 3072), (3, 256, 5120),
                                   (4, 128, 8192), (1, 256, 32768), (2, 128, 17408)])
@pytest.mark.parametrize("y_dtype", [tl.TL_F32, tl.TL_BF16])
def test_f32act_within_rounding_bound(M, N, K, y_dtype):
    inp = synth.config_inputs("tiny", M=M, K=K, N=N)
    packed, s, xr = _dev(inp)
    y = tl.tl_linear_decode_f32act(packed, s, xr, N, K, y_dtype)
    torch.cuda.synchronize()
    assert tl.tl_get_status() == tl.TL_OK
    ref = O.layer_float_act(inp.x_bits, inp.codes, inp.s)
    yg = y.float().cpu().numpy().astype(np.float64)
    bound = TOL * ref["T"] + 1e-30
    if y_dtype == tl.TL_BF16:
        bound = bound + 2.0 ** -8 * np.abs(ref["y64"])
    assert np.all(np.abs(yg - ref["y64"]) <= bound)


def test_f32act_full_decode_shape_sampled_rows():
    """M = 1, K = 5120, N = 17408 (the decode workload), 256 sampled rows."""
    inp = synth.config_inputs("decode")
    packed, s, xr = _dev(inp)
    y = tl.tl_linear_decode_f32act(packed, s, xr, 17408, 5120, tl.TL_F32)
    torch.cuda.synchronize()
    rows = np.random.default_rng(3).choice(17408, size=256, replace=False)
    ref = O.layer_float_act(inp.x_bits, inp.codes, inp.s, rows=rows)
    yg = y.cpu().numpy()[:, rows].astype(np.float64)
    assert np.all(np.abs(yg - ref["y64"]) <= TOL * ref["T"] + 1e-30)


def test_f32act_is_more_exact_than_int8():
    inp = synth.config_inputs("tiny", M=1, K=4096, N=512)
    packed, s, xr = _dev(inp)
    yf = tl.tl_linear_decode_f32act(packed, s, xr, 512, 4096, tl.TL_F32)
    lay = tl.TernaryLinear(torch.from_numpy(inp.codes), torch.from_numpy(inp.s), y_dtype=tl.TL_F32)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    yi = lay.forward(x)
    torch.cuda.synchronize()
    ref = O.reference_fp64(inp.x_bits, inp.codes, inp.s)
    ef = O.rel_fro(yf.cpu().numpy(), ref)
    ei = O.rel_fro(yi.cpu().numpy(), ref)
    assert ef < 1e-5 and ei > 1e-3


def test_f32act_zero_inputs():
    inp = synth.config_inputs("tiny", M=2, K=2048, N=128)
    packed, s, _ = _dev(inp)
    xr = torch.zeros((2, 2048), dtype=torch.float32, device="cuda")
    y = tl.tl_linear_decode_f32act(packed, s, xr, 128, 2048, tl.TL_F32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0

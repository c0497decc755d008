"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Tiers (Qiita item ecc183fae033565af7cb §4 "効いた高速化" defines the layer):
  1. bytes and integers bit-exact: packed codes, qT, sw, xq, sx, the int32
     accumulator (acc_dbg) of both the decode and the prefill kernels;
  2. fp32 outputs within max|y - r| / max|r| <= 1e-3 of the oracle (the pinned
     operation order makes them equal), bf16 outputs within one bf16 ulp of the
     oracle's rne(fp32);
  3. the layer within 1.5e-2 relative Frobenius error of the unquantised fp64
     ternary matmul (the page reports about 9.5e-3 per layer).
Full-size workloads compare sampled output rows that the oracle computes alone.
"""

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-3
FRO_TOL = 1.5e-2
ACC_SENTINEL = -(2 ** 31)   # |acc| <= 127*127*K < 2^31 - 1, so never a real value


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
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def x_dev(L):
    return dev(L.x_bits.view(np.int16), torch.bfloat16)


def pack_dev(tl, L):
    return tl.tl_pack_weights(dev(L.codes), dev(L.s.view(np.int16), torch.float16))


def bf16_ulp_diff(a_bits, b_bits):
    """|difference| in bf16 ulps between two arrays of bf16 bit patterns (same sign assumed)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, 0x8000 - a, a)
    b = np.where(b & 0x8000, 0x8000 - b, b)
    return np.abs(a - b)


def check_status(tl):
    assert tl.tl_get_status() == tl.TL_OK


# ------------------------------------------------------------------ K0 pack

@pytest.mark.parametrize("name,N", [("tiny", None), ("decode", 1024), ("down_proj", 256)])
def test_pack_bitexact(tl, name, N):
    L = synth.config_inputs(name, N=N, M=1)
    s = L.s.copy()
    s[0, :] = 0                                   # all-zero row
    s[1, 2] = -2 * np.abs(s[1]).max()             # negative scale of largest magnitude
    s[2, :] = np.float16(2.0 ** -14)              # all equal tiny scales
    L.s = s
    packed, qT, sw = pack_dev(tl, L)
    check_status(tl)
    p_ref, qT_ref, sw_ref = O.pack_weights(L.codes, L.s)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(qT.cpu().numpy(), qT_ref)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), sw_ref.view(np.uint32))


def test_pack_flags_bad_codes(tl):
    L = synth.config_inputs("tiny")
    codes = L.codes.copy()
    codes[3, 17] = 2
    tl.tl_pack_weights(dev(codes), dev(L.s.view(np.int16), torch.float16))
    assert tl.tl_get_status() == tl.TL_EDATA
    assert tl.tl_get_status() == tl.TL_OK      # cleared by the read


def test_weights_used_right_after_packing(tl):
    """The GEMM kernels load weights before they wait on the preceding kernel;
    tl_pack_weights' outputs are used by the very next launches on the same
    stream, with no synchronisation in between, and must give the oracle's result."""
    L = synth.config_inputs("decode", M=1, N=2048, K=5120)
    r = O.layer(L.x_bits, L.codes, L.s)
    codes = dev(L.codes)
    s = dev(L.s.view(np.int16), torch.float16)
    x = x_dev(L)
    xq8, sx8 = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8)
    xq16, sx16 = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
    torch.cuda.synchronize()
    N, K = L.N, L.K
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    qT = torch.empty((K // 128, N), dtype=torch.int8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for path in ("fused", "decode", "prefill"):
        for _ in range(3):
            acc = torch.full((1, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
            # stale contents that would give a different result if read early
            packed.fill_(0x55)
            qT.fill_(127)
            sw.fill_(1.0)
            assert tl.lib().tl_pack_weights(codes.data_ptr(), s.data_ptr(), N, K, packed.data_ptr(),
                                            qT.data_ptr(), sw.data_ptr(), stream) == tl.TL_OK
            # no synchronisation: the next launch on the stream consumes the weights
            if path == "fused":
                tl.tl_linear_decode_fused(packed, qT, sw, x, L.N, L.K, 4, acc_dbg=acc)
            elif path == "decode":
                tl.tl_linear_decode(packed, qT, sw, xq8, sx8, L.N, L.K, 4, acc_dbg=acc)
            else:
                tl.tl_linear_prefill(packed, qT, sw, xq16, sx16, L.N, L.K, 4, acc_dbg=acc)
            check_status(tl)
            assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"]), path


# ------------------------------------------------------------------ K1 rotate + quantise

def _rq_cases():
    rng = np.random.default_rng(123)
    cases = []
    L = synth.config_inputs("tiny")
    cases.append(("tiny", L.x_bits, None))
    xb = synth.activations_gauss_outliers(rng, 3, 17408, 174, 30.0)
    xb[1] = 0                                               # an all-zero token
    cases.append(("k17408_zero_token", xb, None))
    x = np.zeros((2, 2048), dtype=np.float32)
    x[0, 5] = 2.0
    x[1, 1024 + 777] = -3.0
    cases.append(("one_hot", synth.bf16_bits_from_f32(x), None))
    xb = synth.activations_student_t(rng, 5, 5120)
    signs = np.where(rng.random(5120) < 0.5, -1, 1).astype(np.int8)
    cases.append(("t3_signs", xb, signs))
    return cases


@pytest.mark.parametrize("name,xb,signs", _rq_cases(), ids=[c[0] for c in _rq_cases()])
def test_rotate_quant_bitexact(tl, name, xb, signs):
    xq_ref, sx_ref = O.rotate_quant(xb, signs)
    xd = dev(xb.view(np.int16), torch.bfloat16)
    sd = None if signs is None else dev(signs)
    xq, sx = tl.tl_rotate_quant_act(xd, signs=sd, xq_dtype=tl.TL_I8)
    xh, sx2 = tl.tl_rotate_quant_act(xd, signs=sd, xq_dtype=tl.TL_F16)
    check_status(tl)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(xh.cpu().numpy().astype(np.int64), xq_ref.astype(np.int64))
    assert np.array_equal(sx2.cpu().numpy(), sx.cpu().numpy())


@pytest.mark.parametrize("K", [1024, 3072, 5120, 17408, 20480, 21504])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_rotate_quant_sizes(tl, M, K):
    """K1 over odd and even token counts and block counts from 1 to 21, with and
    without signs, both images, bit-exact."""
    rng = np.random.default_rng(1000 * M + K // 1024)
    xb = synth.activations_student_t(rng, M, K)
    xq_ref, sx_ref = O.rotate_quant(xb)
    signs = np.where(rng.random(K) < 0.5, -1, 1).astype(np.int8)
    xq_s, sx_s = O.rotate_quant(xb, signs)
    xd = dev(xb.view(np.int16), torch.bfloat16)
    for sg, (xr, sr) in ((None, (xq_ref, sx_ref)), (dev(signs), (xq_s, sx_s))):
        xq, sx = tl.tl_rotate_quant_act(xd, signs=sg, xq_dtype=tl.TL_I8)
        xh, sx2 = tl.tl_rotate_quant_act(xd, signs=sg, xq_dtype=tl.TL_F16)
        check_status(tl)
        assert np.array_equal(xq.cpu().numpy(), xr)
        assert np.array_equal(xh.cpu().numpy().astype(np.int64), xr.astype(np.int64))
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sr.view(np.uint32))
        assert np.array_equal(sx2.cpu().numpy().view(np.uint32), sr.view(np.uint32))


def _tiny_tokens(K=2048):
    """Tokens of bf16 subnormals whose largest rotated value is below 127 / FLT_MAX,
    so that fl32(127 / a) overflows to +inf (the oracle's reading: non-zero
    elements code to +-127, exact zeros to 0), next to an ordinary token."""
    x = np.zeros((4, K), dtype=np.uint16)
    x[0, 0], x[0, 1] = 0x0001, 0x0002            # two subnormals: +-127 over block 0, zeros after
    x[1, 0] = 0x0001                             # one subnormal: block 0 all +127, the rest exact zeros
    x[2] = synth.bf16_bits_from_f32(np.random.default_rng(5).standard_normal(K).astype(np.float32))
    x[3, 3], x[3, K - 1] = 0x8005, 0x0003        # subnormals of both signs in the first and last block
    return x


def test_tiny_token_quantiser(tl):
    """The subnormal-token case through K1 (int8 and fp16 images), the decode and
    prefill GEMMs and the fused decode, bit-exact against the oracle."""
    K, N = 2048, 256
    xb = _tiny_tokens(K)
    xq_ref, sx_ref = O.rotate_quant(xb)
    assert np.any(sx_ref[[0, 1, 3]] < np.float32(1e-40))      # the overflow case is reached
    xd = dev(xb.view(np.int16), torch.bfloat16)
    xq, sx = tl.tl_rotate_quant_act(xd, xq_dtype=tl.TL_I8)
    xh, sx2 = tl.tl_rotate_quant_act(xd, xq_dtype=tl.TL_F16)
    check_status(tl)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(xh.cpu().numpy().astype(np.int64), xq_ref.astype(np.int64))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(sx2.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))

    L = synth.config_inputs("decode", M=4, N=N, K=K)
    L.x_bits = xb
    packed, qT, sw = pack_dev(tl, L)
    r = O.layer(L.x_bits, L.codes, L.s)
    for path in ("decode", "prefill"):
        acc, y = _run(tl, path, L, packed, qT, sw, 4)
        assert np.array_equal(acc.astype(np.int64), r["acc"]), path
        assert np.array_equal(y.cpu().numpy().view(np.uint32), r["y32"].view(np.uint32)), path
    for M in (1, 4):
        acc = torch.full((M, N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
        xq1 = torch.zeros((M, K), dtype=torch.int8, device="cuda")
        sx1 = torch.zeros((M,), dtype=torch.float32, device="cuda")
        tl.tl_linear_decode_fused(packed, qT, sw, xd[:M].contiguous(), N, K, 4, acc_dbg=acc,
                                  xq_out=xq1, sx_out=sx1)
        check_status(tl)
        assert np.array_equal(xq1.cpu().numpy(), xq_ref[:M])
        assert np.array_equal(sx1.cpu().numpy().view(np.uint32), sx_ref[:M].view(np.uint32))
        assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"][:M])


# ------------------------------------------------------------------ K2 / K3 layer parity

def _run(tl, path, L, packed, qT, sw, y_dtype):
    xd = x_dev(L)
    M = L.M
    acc = torch.full((M, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    if path == "decode":
        xq, sx = tl.tl_rotate_quant_act(xd, xq_dtype=tl.TL_I8)
        y = tl.tl_linear_decode(packed, qT, sw, xq, sx, L.N, L.K, y_dtype, acc_dbg=acc)
    else:
        xq, sx = tl.tl_rotate_quant_act(xd, xq_dtype=tl.TL_F16)
        need = tl.tl_prefill_workspace_size(M, L.N, L.K)
        ws = torch.zeros((max(need, 16),), dtype=torch.uint8, device="cuda") if need else None
        y = tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, y_dtype, acc_dbg=acc, workspace=ws)
    check_status(tl)
    return acc.cpu().numpy(), y


def _compare(L, acc, y, y_dtype, rows=None, frobenius=True):
    r = O.layer(L.x_bits, L.codes, L.s, rows=rows)
    sel = slice(None) if rows is None else rows
    acc_s = acc[:, sel]
    assert np.array_equal(acc_s.astype(np.int64), r["acc"]), "int32 accumulator differs"
    yv = y.float().cpu().numpy()[:, sel] if y_dtype == 4 else None
    if y_dtype == 4:
        err = np.max(np.abs(yv - r["y32"])) / max(np.max(np.abs(r["y32"])), 1e-30)
        assert err <= FP32_TOL
    else:
        yb = y.view(torch.int16).cpu().numpy().view(np.uint16)[:, sel]
        assert np.max(bf16_ulp_diff(yb, r["ybf"])) <= 1
        yv = synth.bf16_bits_to_f32(yb)
    if frobenius:
        ref = O.reference_fp64(L.x_bits, L.codes, L.s, rows=rows)
        assert O.rel_fro(yv, ref) <= FRO_TOL


@pytest.mark.parametrize("path", ["decode", "prefill"])
@pytest.mark.parametrize("y_dtype", [3, 4], ids=["bf16", "f32"])
def test_tiny_layer(tl, path, y_dtype):
    L = synth.config_inputs("tiny")
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, path, L, packed, qT, sw, y_dtype)
    _compare(L, acc, y, y_dtype)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 13, 16, 17, 31, 32])
def test_decode_prefill_agree(tl, M):
    L = synth.config_inputs("decode", M=M, N=512, K=3072)
    packed, qT, sw = pack_dev(tl, L)
    acc_d, y_d = _run(tl, "decode", L, packed, qT, sw, 4)
    acc_p, y_p = _run(tl, "prefill", L, packed, qT, sw, 4)
    assert np.array_equal(acc_d, acc_p)
    assert torch.equal(y_d, y_p)
    _compare(L, acc_d, y_d, 4, frobenius=False)


@pytest.mark.parametrize("K", [1024, 3072, 6144, 8192, 16384, 17408])
def test_decode_m1_shapes(tl, K):
    """M = 1 runs a kernel specialised on K / 1024 for the common depths, a generic one otherwise."""
    L = synth.config_inputs("decode", M=1, N=384, K=K)
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, "decode", L, packed, qT, sw, 4)
    _compare(L, acc, y, 4)


@pytest.mark.parametrize("K", [1024, 2048, 3072, 5120, 6144, 7168, 8192])
@pytest.mark.parametrize("signed", [False, True], ids=["plain", "signs"])
def test_decode_fused_matches_two_step(tl, K, signed):
    """One launch (rotate + quantise + decode) equals the two-kernel path bit for bit."""
    L = synth.config_inputs("decode", M=1, N=256, K=K)
    packed, qT, sw = pack_dev(tl, L)
    x = x_dev(L)
    signs = None
    if signed:
        signs = dev(np.where(np.random.default_rng(K).random(K) < 0.5, -1, 1).astype(np.int8))
    acc2 = torch.empty((1, L.N), dtype=torch.int32, device="cuda")
    xq, sx = tl.tl_rotate_quant_act(x, signs=signs, xq_dtype=tl.TL_I8)
    y2 = tl.tl_linear_decode(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=acc2)
    acc1 = torch.full((1, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    xq1 = torch.zeros((1, K), dtype=torch.int8, device="cuda")
    sx1 = torch.zeros((1,), dtype=torch.float32, device="cuda")
    y1 = tl.tl_linear_decode_fused(packed, qT, sw, x, L.N, L.K, 4, signs=signs, acc_dbg=acc1,
                                   xq_out=xq1, sx_out=sx1)
    check_status(tl)
    assert torch.equal(xq1, xq) and torch.equal(sx1, sx)
    assert torch.equal(acc1, acc2) and torch.equal(y1, y2)
    if not signed:
        _compare(L, acc1.cpu().numpy(), y1, 4)


@pytest.mark.parametrize("K", [1024, 5120, 8192])
def test_decode_fused_clusters_of_four(tl, K):
    """N / 32 not a multiple of 8 (N = 384: 12 CTAs) runs the fused kernel in clusters of 4."""
    L = synth.config_inputs("decode", M=1, N=384, K=K)
    packed, qT, sw = pack_dev(tl, L)
    x = x_dev(L)
    acc2 = torch.empty((1, L.N), dtype=torch.int32, device="cuda")
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8)
    y2 = tl.tl_linear_decode(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=acc2)
    acc1 = torch.full((1, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    y1 = tl.tl_linear_decode_fused(packed, qT, sw, x, L.N, L.K, 4, acc_dbg=acc1)
    check_status(tl)
    assert torch.equal(acc1, acc2) and torch.equal(y1, y2)
    _compare(L, acc1.cpu().numpy(), y1, 4)


@pytest.mark.parametrize("M,K,N,signed", [(2, 1024, 256, False), (3, 5120, 256, True), (4, 17408, 256, False),
                                           (5, 8192, 384, False), (8, 5120, 256, True),
                                           (9, 4096, 256, False), (16, 2048, 384, True), (16, 4096, 256, False)])
def test_decode_fused_multi_token(tl, M, K, N, signed):
    """2 <= M <= 16 tokens (M K <= 72 K) in one launch equal the two-kernel path bit for bit,
    including the quantised tokens and their scales."""
    L = synth.config_inputs("decode", M=M, N=N, K=K)
    packed, qT, sw = pack_dev(tl, L)
    x = x_dev(L)
    signs = None
    if signed:
        signs = dev(np.where(np.random.default_rng(K + M).random(K) < 0.5, -1, 1).astype(np.int8))
    acc2 = torch.empty((M, L.N), dtype=torch.int32, device="cuda")
    xq, sx = tl.tl_rotate_quant_act(x, signs=signs, xq_dtype=tl.TL_I8)
    y2 = tl.tl_linear_decode(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=acc2)
    acc1 = torch.full((M, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    xq1 = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx1 = torch.zeros((M,), dtype=torch.float32, device="cuda")
    y1 = tl.tl_linear_decode_fused(packed, qT, sw, x, L.N, L.K, 4, signs=signs, acc_dbg=acc1,
                                   xq_out=xq1, sx_out=sx1)
    check_status(tl)
    assert torch.equal(xq1, xq) and torch.equal(sx1, sx)
    assert torch.equal(acc1, acc2) and torch.equal(y1, y2)
    if not signed:
        _compare(L, acc1.cpu().numpy(), y1, 4, frobenius=False)


def test_decode_fused_full_size(tl):
    L = synth.config_inputs("decode")
    packed, qT, sw = pack_dev(tl, L)
    acc = torch.full((1, L.N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    y = tl.tl_linear_decode_fused(packed, qT, sw, x_dev(L), L.N, L.K, 3, acc_dbg=acc)
    check_status(tl)
    _compare(L, acc.cpu().numpy(), y, 3, rows=_sample_rows(L.N))


@pytest.mark.parametrize("M,K", [(2, 17408), (7, 17408), (16, 17408), (32, 17408), (32, 1024)])
def test_decode_slabs(tl, M, K):
    """M * K beyond one shared-memory slab: K is processed in slabs with partial sums."""
    L = synth.config_inputs("down_proj", M=M, N=256, K=K)
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, "decode", L, packed, qT, sw, 4)
    _compare(L, acc, y, 4)


@pytest.mark.parametrize("M,N,K", [(300, 384, 2048), (129, 256, 1024), (1, 128, 1024),
                                   (256, 640, 4096), (777, 128, 3072)])
def test_prefill_ragged(tl, M, N, K):
    L = synth.config_inputs("gate_up", M=M, N=N, K=K)
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, "prefill", L, packed, qT, sw, 3)
    _compare(L, acc, y, 3)


def test_prefill_split_k_matches_unsplit(tl):
    """Few tiles -> K split across CTAs; the int32 result must not depend on it."""
    L = synth.config_inputs("down_proj", M=64, N=256, K=17408)
    packed, qT, sw = pack_dev(tl, L)
    xq, sx = tl.tl_rotate_quant_act(x_dev(L), xq_dtype=tl.TL_F16)
    need = tl.tl_prefill_workspace_size(L.M, L.N, L.K)
    assert need > 0
    ws = torch.zeros((need,), dtype=torch.uint8, device="cuda")
    a1 = torch.empty((L.M, L.N), dtype=torch.int32, device="cuda")
    a2 = torch.empty_like(a1)
    y1 = tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=a1, workspace=ws)
    y2 = tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=a2, workspace=None)
    check_status(tl)
    assert torch.equal(a1, a2) and torch.equal(y1, y2)
    _compare(L, a1.cpu().numpy(), y1, 4)
    # the call returned the workspace to zero: the next call needs no clearing
    assert not torch.any(ws)
    a3 = torch.empty_like(a1)
    tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=a3, workspace=ws)
    check_status(tl)
    assert torch.equal(a3, a1) and not torch.any(ws)


@pytest.mark.parametrize("M,N,K", [(1, 17408, 5120), (16, 5120, 17408), (9, 384, 2048),
                                   (32, 17408, 5120), (20, 640, 8192), (64, 5120, 17408),
                                   (48, 1152, 3072)])
def test_prefill_narrow_tiles(tl, M, N, K):
    """Batches of at most 16, 32 and 64 tokens run on tiles of that many tokens
    (split along K where the tiles are fewer than the SMs): the int32 result
    equals the oracle's on every row, the workspace is left zero, and the
    128-token-tile kernel (a batch padded to 65 tokens) gives the same rows."""
    L = synth.config_inputs("decode", M=M, N=N, K=K)
    packed, qT, sw = pack_dev(tl, L)
    rows = None if N <= 2048 else _sample_rows(N)
    acc, y = _run(tl, "prefill", L, packed, qT, sw, 4)
    _compare(L, acc, y, 4, rows=rows, frobenius=False)
    xb = np.zeros((65, K), dtype=np.uint16)
    xb[:M] = L.x_bits
    xq, sx = tl.tl_rotate_quant_act(dev(xb.view(np.int16), torch.bfloat16), xq_dtype=tl.TL_F16)
    a65 = torch.empty((65, N), dtype=torch.int32, device="cuda")
    tl.tl_linear_prefill(packed, qT, sw, xq, sx, N, K, 4, acc_dbg=a65, workspace=None)
    check_status(tl)
    assert np.array_equal(a65[:M].cpu().numpy(), acc)


def test_prefill_repeatable_after_sync(tl):
    """Whole tiles of 17 chunks on two CTAs, each call started on an idle GPU and
    compared with the oracle: a shared-memory slot refilled by TMA while the
    expansion warps' ordinary loads of it were still pending made rows of the
    result wrong in some runs (fixed by a proxy fence before the slot's release)."""
    L = synth.config_inputs("down_proj", M=64, N=256, K=17408)
    packed, qT, sw = pack_dev(tl, L)
    xq, sx = tl.tl_rotate_quant_act(x_dev(L), xq_dtype=tl.TL_F16)
    ref = O.layer(L.x_bits, L.codes, L.s)["acc"]
    for _ in range(8):
        torch.cuda.synchronize()
        a = torch.full((L.M, L.N), -7, dtype=torch.int32, device="cuda")
        tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, 4, acc_dbg=a, workspace=None)
        torch.cuda.synchronize()
        assert np.array_equal(a.cpu().numpy().astype(np.int64), ref)
    check_status(tl)


def test_exactness_adversarial(tl):
    """Chunk sums at the integer-exact fp32 limit, cancellation and +-1 terms.

    x = 2.0 at channel 0 of every 1024-block rotates to xr = 1/16 everywhere,
    so xq = 127 in every column; with all scales equal q = 127. Row patterns:
      0: all +1  -> 127*127*1024 per block (> 2^24 over the two blocks)
      1: alternating +-1 -> 0, partial sums oscillate
      2: all +1 but one -1 per block
      3: first half +1, second half -1 per block -> partial sums rise to 8.3e6 then fall
      4: random codes
    """
    K, N, M = 2048, 128, 2
    x = np.zeros((M, K), dtype=np.float32)
    x[:, 0] = 2.0
    x[:, 1024] = 2.0
    x[1, 1024] = -2.0
    codes = np.zeros((N, K), dtype=np.int8)
    codes[0] = 1
    codes[1, 0::2], codes[1, 1::2] = 1, -1
    codes[2] = 1
    codes[2, 511], codes[2, 1024 + 3] = -1, -1
    codes[3, :] = 1
    codes[3, 512:1024], codes[3, 1536:] = -1, -1
    codes[4:] = np.random.default_rng(5).integers(-1, 2, size=(N - 4, K))
    s = np.full((N, K // 128), 2.0 ** -4, dtype=np.float16)
    L = synth.LayerInputs(codes=codes, s=s, x_bits=synth.bf16_bits_from_f32(x))
    packed, qT, sw = pack_dev(tl, L)
    for path in ("prefill", "decode"):
        acc, y = _run(tl, path, L, packed, qT, sw, 4)
        r = O.layer(L.x_bits, L.codes, L.s)
        assert int(r["acc"][0, 0]) == 2 * 127 * 127 * 1024
        assert np.array_equal(acc.astype(np.int64), r["acc"])


def test_exactness_largest_accumulator(tl):
    """K = 32768 with every term at +-127*127: |acc| = 127*127*32768 = 528,515,072, the largest
    the layer can produce (below 2^31). x = 2.0 at channel 0 of every block gives xq = 127
    everywhere (as above); row 0 all +1, row 1 all -1, row 2 the sign flipping every block,
    the rest random."""
    K, N, M = 32768, 128, 1
    x = np.zeros((M, K), dtype=np.float32)
    x[:, 0::1024] = 2.0
    codes = np.random.default_rng(6).integers(-1, 2, size=(N, K)).astype(np.int8)
    codes[0] = 1
    codes[1] = -1
    codes[2] = np.repeat(np.where(np.arange(K // 1024) % 2 == 0, 1, -1), 1024)
    s = np.full((N, K // 128), 2.0 ** -4, dtype=np.float16)
    L = synth.LayerInputs(codes=codes, s=s, x_bits=synth.bf16_bits_from_f32(x))
    packed, qT, sw = pack_dev(tl, L)
    r = O.layer(L.x_bits, L.codes, L.s)
    assert int(r["acc"][0, 0]) == 127 * 127 * K and int(r["acc"][0, 1]) == -127 * 127 * K
    assert int(r["acc"][0, 2]) == 0
    for path in ("prefill", "decode"):
        acc, y = _run(tl, path, L, packed, qT, sw, 4)
        assert np.array_equal(acc.astype(np.int64), r["acc"]), path


def test_bounded_inputs_extreme_values(tl):
    """Saturated scales and activations at bf16 range edges stay exact."""
    rng = np.random.default_rng(77)
    M, N, K = 40, 256, 2048
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0] *= 1e30
    x[1] *= 1e-30
    x[2, :] = 0
    codes = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    s = np.exp(rng.normal(-4, 3.0, size=(N, K // 128))).astype(np.float16)
    s[7] = np.float16(65504.0)
    L = synth.LayerInputs(codes=codes, s=s, x_bits=synth.bf16_bits_from_f32(x))
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, "prefill", L, packed, qT, sw, 4)
    r = O.layer(L.x_bits, L.codes, L.s)
    assert np.array_equal(acc.astype(np.int64), r["acc"])
    assert np.array_equal(y.cpu().numpy().view(np.uint32), r["y32"].view(np.uint32))


# ------------------------------------------------------------------ full-size workloads, sampled rows

@pytest.mark.parametrize("path,M", [("decode", 1), ("decode", 5), ("decode", 32),
                                    ("prefill", 1), ("prefill", 160)])
def test_largest_k(tl, path, M):
    """K = 32768, the largest the library takes: the one-CTA-per-token rotation runs 1024 threads,
    decode takes its generic K path (and slabs at M = 32), |acc| may reach 127 * 127 * 32768."""
    L = synth.config_inputs("decode", M=M, N=256, K=32768)
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, path, L, packed, qT, sw, 4)
    _compare(L, acc, y, 4, frobenius=False)


def _sample_rows(N, n=192, seed=0):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(N, size=n, replace=False))


@pytest.mark.parametrize("M,N,K", [pytest.param(128, 80 * 128, 17408, id="regions"),
                                   pytest.param(64, 256, 17408, id="atomics"),
                                   pytest.param(1024, 5120, 17408, id="atomics-last-round")])
def test_prefill_cut_tiles_match_whole_tiles(tl, M, N, K):
    """A tile cut along K between CTAs meets through one region per CTA (at most three CTAs
    per tile: 80 tiles of 17 chunks over 152 SMs) or through atomics into one region (more
    CTAs per tile; the 1024-token case cuts only the last partial round of SMs): the int32
    result equals the one with every tile whole (no workspace), and the call leaves the
    workspace zero."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    need = tl.tl_prefill_workspace_size(M, N, K)
    if need == 0:
        pytest.skip(f"with {sms} SMs this shape is not cut")
    codes, s, x = synth.torch_layer(7, M, K, N, p0=0.4, mu=-4.0, sigma=0.5, x_kind="t3")
    packed, qT, sw = tl.tl_pack_weights(codes, s)
    del codes
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
    ws = torch.zeros((need,), dtype=torch.uint8, device="cuda")
    a_cut = torch.full((M, N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    a_whole = torch.full((M, N), ACC_SENTINEL, dtype=torch.int32, device="cuda")
    for _ in range(2):   # the second call reuses the workspace the first one returned to zero
        y_cut = tl.tl_linear_prefill(packed, qT, sw, xq, sx, N, K, tl.TL_F32, acc_dbg=a_cut, workspace=ws)
        check_status(tl)
        assert not torch.any(ws)
    y_whole = tl.tl_linear_prefill(packed, qT, sw, xq, sx, N, K, tl.TL_F32, acc_dbg=a_whole)
    check_status(tl)
    assert not torch.any(a_cut == ACC_SENTINEL)
    assert torch.equal(a_cut, a_whole) and torch.equal(y_cut, y_whole)


@pytest.mark.parametrize("name,path", [("decode", "decode"), ("decode16", "decode"),
                                       ("down_proj", "prefill"), ("gate_up", "prefill")])
def test_full_size_sampled(tl, name, path):
    L = synth.config_inputs(name)
    packed, qT, sw = pack_dev(tl, L)
    acc, y = _run(tl, path, L, packed, qT, sw, 4)
    rows = _sample_rows(L.N)
    _compare(L, acc, y, 4, rows=rows)
    # properties that hold at any size: every output was written, and every
    # output is the epilogue of its own accumulator with the oracle's scales
    assert not np.any(acc == ACC_SENTINEL)
    _, sx_ref = O.rotate_quant(L.x_bits)
    _, sw_ref, _ = O.row_scale_decompose(L.s)
    want = O.epilogue(acc, sw_ref, sx_ref)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_full_size_decode_vs_prefill(tl):
    L = synth.config_inputs("decode16")
    packed, qT, sw = pack_dev(tl, L)
    acc_d, _ = _run(tl, "decode", L, packed, qT, sw, 3)
    acc_p, _ = _run(tl, "prefill", L, packed, qT, sw, 3)
    assert np.array_equal(acc_d, acc_p)


# ------------------------------------------------------------------ boundary behaviour on the device

def test_guard_rows_untouched(tl):
    L = synth.config_inputs("gate_up", M=130, N=256, K=1024)
    packed, qT, sw = pack_dev(tl, L)
    xq, sx = tl.tl_rotate_quant_act(x_dev(L), xq_dtype=tl.TL_F16)
    buf = torch.full((L.M + 2, L.N), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[1:L.M + 1]
    tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, 4, y=y)
    check_status(tl)
    assert torch.all(buf[0] == 12345.0) and torch.all(buf[-1] == 12345.0)
    xq8, sx8 = tl.tl_rotate_quant_act(x_dev(L)[:17].contiguous(), xq_dtype=tl.TL_I8)
    buf.fill_(12345.0)
    tl.tl_linear_decode(packed, qT, sw, xq8, sx8, L.N, L.K, 4, y=buf[1:18])
    check_status(tl)
    assert torch.all(buf[0] == 12345.0) and torch.all(buf[18:] == 12345.0)


def test_argument_errors_launch_nothing(tl):
    L = synth.config_inputs("tiny")
    packed, qT, sw = pack_dev(tl, L)
    xq, sx = tl.tl_rotate_quant_act(x_dev(L), xq_dtype=tl.TL_I8)
    y = torch.zeros((L.M, L.N), dtype=torch.float32, device="cuda")
    lib = tl.lib()
    s = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731
    # misaligned activation pointer
    assert lib.tl_linear_decode(P(packed), P(qT), P(sw), P(xq) + 1, P(sx), L.M, L.N, L.K, P(y), 4, None, s) == tl.TL_EINVAL
    # M > 32 on decode
    assert lib.tl_linear_decode(P(packed), P(qT), P(sw), P(xq), P(sx), 33, L.N, L.K, P(y), 4, None, s) == tl.TL_EUNSUPPORTED
    # K not a multiple of 1024, N not a multiple of 128
    assert lib.tl_linear_prefill(P(packed), P(qT), P(sw), P(xq), P(sx), 16, L.N, 1536, P(y), 4, None, None, 0, s) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_prefill(P(packed), P(qT), P(sw), P(xq), P(sx), 16, 200, L.K, P(y), 4, None, None, 0, s) == tl.TL_EUNSUPPORTED
    # bad dtype, NULL output
    assert lib.tl_linear_prefill(P(packed), P(qT), P(sw), P(xq), P(sx), 16, L.N, L.K, P(y), 9, None, None, 0, s) == tl.TL_EINVAL
    assert lib.tl_linear_decode(P(packed), P(qT), P(sw), P(xq), P(sx), 16, L.N, L.K, None, 4, None, s) == tl.TL_EINVAL
    # empty problems are valid and launch nothing
    assert lib.tl_linear_decode(P(packed), P(qT), P(sw), P(xq), P(sx), 0, L.N, L.K, P(y), 4, None, s) == tl.TL_OK
    assert lib.tl_linear_prefill(None, None, None, None, None, 0, L.N, L.K, None, 4, None, None, 0, s) == tl.TL_OK
    assert lib.tl_rotate_quant_act(None, 0, 1024, None, None, 1, None, s) == tl.TL_OK
    assert torch.all(y == 0)
    check_status(tl)


@pytest.mark.parametrize("K", [5120, 17408])
@pytest.mark.parametrize("M", [1, 3, 4, 5, 12, 16, 17, 40])
def test_forward_every_route(tl, M, K):
    """TernaryLinear.forward on each side of its kernel boundary (dp4a decode,
    prefill) matches the oracle: bf16 y within one ulp of the oracle's, f32 y
    identical."""
    L = synth.config_inputs("decode", M=M, N=384, K=K)
    lay = tl.TernaryLinear(torch.from_numpy(L.codes), torch.from_numpy(L.s))
    lay32 = tl.TernaryLinear(torch.from_numpy(L.codes), torch.from_numpy(L.s), y_dtype=tl.TL_F32)
    x = torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    y = lay.forward(x)
    y32 = lay32.forward(x)
    torch.cuda.synchronize()
    check_status(tl)
    r = O.layer(L.x_bits, L.codes, L.s)
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.max(bf16_ulp_diff(yb, r["ybf"])) <= 1, lay.kernel_for(M)
    assert np.array_equal(y32.cpu().numpy().view(np.uint32), r["y32"].view(np.uint32)), lay.kernel_for(M)


def test_host_pipeline_matches_forward(tl):
    """tl.HostPipeline (copies overlapped with the kernels on three streams) gives the
    same bytes as TernaryLinear.forward on device tensors, for decode and prefill sizes."""
    outs = []
    pipe = tl.HostPipeline("cuda", depth=2)
    cases = []
    for li, M in enumerate((1, 64, 3, 130, 16)):
        L = synth.config_inputs("tiny", M=M)
        lay = tl.TernaryLinear(torch.from_numpy(L.codes), torch.from_numpy(L.s))
        xh = torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        yh = torch.empty((M, L.N), dtype=torch.bfloat16).pin_memory()
        pipe.submit(lay, xh, yh)
        cases.append((lay, xh, yh))
    pipe.synchronize()
    for lay, xh, yh in cases:
        ref = lay.forward(xh.cuda())
        torch.cuda.synchronize()
        assert torch.equal(yh, ref.cpu())
    check_status(tl)


def test_graph_step_matches_forward(tl):
    """tl.GraphStep (one copy in, the layers, one copy out, captured in a CUDA graph)
    gives the same bytes as TernaryLinear.forward, on every replay, with new inputs."""
    layers, ms, xs = [], [], []
    for li, M in enumerate((1, 2, 16)):
        L = synth.config_inputs("tiny", M=M)
        layers.append(tl.TernaryLinear(torch.from_numpy(L.codes), torch.from_numpy(L.s)))
        ms.append(M)
        xs.append(torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16))
    step = tl.GraphStep(layers, ms)
    for rep in range(3):
        for x, xin in zip(xs, step.inputs):
            xin.copy_(x if rep < 2 else -x)
        step.run()
        for lay, xin, yout in zip(layers, step.inputs, step.outputs):
            ref = lay.forward(xin.cuda())
            torch.cuda.synchronize()
            assert torch.equal(yout, ref.cpu())
    check_status(tl)

"""tl_linear_prefill_noalloc: the prefill layer for callers that cannot allocate.

Some hosts cannot hand this library a device workspace: their device memory
already belongs to their own pool, or they must not call cudaMalloc in the
middle of a step because it synchronises the device. For them the library
keeps a fixed split-K scratch array of its own. These tests call that entry
point through the C ABI and check it against tl_linear_prefill with a
caller-provided workspace, twice in a row (the second call must not see the
first call's partial sums), and that a problem too large for the array is
refused. The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from quantized_linear_layers_block_gb300 import synth

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-3


@pytest.fixture(scope="module")
def tl():
    from quantized_linear_layers_block_gb300 import build
    build.build()
    from quantized_linear_layers_block_gb300 import tl as _tl
    _tl.lib()
    return _tl


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).cuda()


def test_noalloc_matches_workspace_version_on_two_calls(tl):
    # few output tiles and a long K: the kernel splits K and uses the scratch
    L = synth.config_inputs("down_proj", M=64, N=256, K=17408)
    need = tl.tl_prefill_workspace_size(L.M, L.N, L.K)
    assert 0 < need <= 8 * 1024 * 1024
    packed, qT, sw = tl.tl_pack_weights(_dev(L.codes), _dev(L.s.view(np.int16), torch.float16))
    x = _dev(L.x_bits.view(np.int16), torch.bfloat16)
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    acc_ref = torch.empty((L.M, L.N), dtype=torch.int32, device="cuda")
    y_ref = tl.tl_linear_prefill(packed, qT, sw, xq, sx, L.N, L.K, tl.TL_F32, acc_dbg=acc_ref,
                                 workspace=ws)
    assert tl.tl_get_status() == tl.TL_OK
    r = y_ref.cpu().numpy()
    for _ in range(2):
        acc = torch.full((L.M, L.N), -(2 ** 31), dtype=torch.int32, device="cuda")
        y = tl.tl_linear_prefill_noalloc(packed, qT, sw, xq, sx, L.N, L.K, tl.TL_F32, acc_dbg=acc)
        assert tl.tl_get_status() == tl.TL_OK
        assert torch.equal(acc, acc_ref)
        err = np.max(np.abs(y.cpu().numpy() - r)) / np.max(np.abs(r))
        assert err <= FP32_TOL


def test_noalloc_refuses_problems_beyond_its_scratch(tl):
    limit = 8 * 1024 * 1024
    shape = None
    for M in (1024, 2048, 4096, 8192):
        for N in (1152, 2304, 4608):
            if tl.tl_prefill_workspace_size(M, N, 17408) > limit:
                shape = (M, N)
                break
        if shape:
            break
    if shape is None:
        pytest.skip("no shape on this device needs more split-K scratch than the array holds")
    M, N = shape
    K = 2048   # the refusal happens before any launch; keep the buffers small
    if tl.tl_prefill_workspace_size(M, N, K) <= limit:
        K = 17408
    packed = torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda")
    qT = torch.zeros((K // 128, N), dtype=torch.int8, device="cuda")
    sw = torch.zeros((N,), dtype=torch.float32, device="cuda")
    xq = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    sx = torch.zeros((M,), dtype=torch.float32, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    rc = tl.lib().tl_linear_prefill_noalloc(P(packed.data_ptr()), P(qT.data_ptr()), P(sw.data_ptr()),
                                           P(xq.data_ptr()), P(sx.data_ptr()), M, N, K,
                                           P(y.data_ptr()), tl.TL_F32, None,
                                           P(torch.cuda.current_stream().cuda_stream))
    assert rc == tl.TL_ENOSPACE
    assert tl.tl_get_status() == tl.TL_OK
    assert torch.all(y == 7.0)

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

LIMIT = 16 * 1024 * 1024   # TL_NOALLOC_SCRATCH_BYTES


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
    assert 0 < need <= LIMIT
    packed, qT, sw = tl.tl_pack_weights(_dev(L.codes), _dev(L.s.view(np.int16), torch.float16))
    x = _dev(L.x_bits.view(np.int16), torch.bfloat16)
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
    ws = torch.zeros((need,), dtype=torch.uint8, device="cuda")
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


M_TILE = 128      # a 128-token batch runs on one 128-token tile: 64 KB per split-K region


def _sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def _zeros_layer(M, N, K):
    return (torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda"),
            torch.zeros((K // 128, N), dtype=torch.int8, device="cuda"),
            torch.zeros((N,), dtype=torch.float32, device="cuda"),
            torch.zeros((M, K), dtype=torch.float16, device="cuda"),
            torch.zeros((M,), dtype=torch.float32, device="cuda"))


def _call_raw(tl, packed, qT, sw, xq, sx, M, N, K, y, acc=None):
    P = ctypes.c_void_p
    return tl.lib().tl_linear_prefill_noalloc(P(packed.data_ptr()), P(qT.data_ptr()), P(sw.data_ptr()),
                                             P(xq.data_ptr()), P(sx.data_ptr()), M, N, K,
                                             P(y.data_ptr()), tl.TL_F32,
                                             None if acc is None else P(acc.data_ptr()),
                                             P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_allocates_nothing(tl):
    """After a first call (which loads the kernels), a call changes neither the
    caching allocator's bytes nor the device's free memory."""
    L = synth.config_inputs("down_proj", M=64, N=256, K=17408)
    packed, qT, sw = tl.tl_pack_weights(_dev(L.codes), _dev(L.s.view(np.int16), torch.float16))
    xq, sx = tl.tl_rotate_quant_act(_dev(L.x_bits.view(np.int16), torch.bfloat16), xq_dtype=tl.TL_F16)
    y = torch.empty((L.M, L.N), dtype=torch.float32, device="cuda")
    acc = torch.empty((L.M, L.N), dtype=torch.int32, device="cuda")
    assert _call_raw(tl, packed, qT, sw, xq, sx, L.M, L.N, L.K, y, acc) == tl.TL_OK
    torch.cuda.synchronize()
    first = acc.clone()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        assert _call_raw(tl, packed, qT, sw, xq, sx, L.M, L.N, L.K, y, acc) == tl.TL_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] >= free0
    assert tl.tl_get_status() == tl.TL_OK
    assert torch.equal(acc, first)


def test_noalloc_refuses_problems_beyond_its_scratch(tl):
    """Fewer tiles than SMs with a long K (K is cut) and more split-K scratch
    than the array holds: refused before any launch."""
    sms = _sms()
    M, K = M_TILE, 32768
    shape = None
    for tiles in range(sms - 1, 0, -1):   # 128-row tiles of one 128-token block
        need = tl.tl_prefill_workspace_size(M, tiles * 128, K)
        if need > LIMIT:
            shape = tiles * 128
            break
    if shape is None:
        pytest.skip(f"with {sms} SMs no single-tile-row problem needs more than the array holds")
    N = shape
    assert (N // 128) < sms
    packed, qT, sw, xq, sx = _zeros_layer(M, N, K)
    y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    assert _call_raw(tl, packed, qT, sw, xq, sx, M, N, K, y) == tl.TL_ENOSPACE
    assert tl.tl_get_status() == tl.TL_OK
    assert torch.all(y == 7.0)


def test_noalloc_runs_unsplit_when_tiles_fill_the_gpu(tl):
    """At least as many tiles as SMs, with a short K: whole tiles even though
    the last round fills only part of the GPU; no scratch is needed, and the
    result is the same as tl_linear_prefill's."""
    sms = _sms()
    M, K = M_TILE, 2048
    N = (sms + 140) * 128          # one full round, then 140 tiles left over
    need = tl.tl_prefill_workspace_size(M, N, K)
    assert (N // 128) >= sms and need == 0
    L = synth.config_inputs("gate_up", M=M, N=N, K=K)
    packed, qT, sw = tl.tl_pack_weights(_dev(L.codes), _dev(L.s.view(np.int16), torch.float16))
    xq, sx = tl.tl_rotate_quant_act(_dev(L.x_bits.view(np.int16), torch.bfloat16), xq_dtype=tl.TL_F16)
    acc_ref = torch.empty((M, N), dtype=torch.int32, device="cuda")
    tl.tl_linear_prefill(packed, qT, sw, xq, sx, N, K, tl.TL_F32, acc_dbg=acc_ref)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    acc = torch.full((M, N), -(2 ** 31), dtype=torch.int32, device="cuda")
    assert _call_raw(tl, packed, qT, sw, xq, sx, M, N, K, y, acc) == tl.TL_OK
    assert tl.tl_get_status() == tl.TL_OK
    assert torch.equal(acc, acc_ref)

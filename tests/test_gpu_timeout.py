"""Failure detection without a GPU fault: a device-side wait that nothing ends
gives up after its limit, records TL_ETIMEOUT, and the context stays usable."""

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth, tl


def test_selftest_rejects_bad_limits_without_gpu():
    assert tl.lib().tl_selftest_wait_timeout(0, None) == tl.TL_EINVAL
    assert tl.lib().tl_selftest_wait_timeout(200000, None) == tl.TL_EINVAL


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    assert tl.tl_get_status() == tl.TL_OK
    tl.tl_selftest_wait_timeout(2000)            # 2 ms
    assert tl.tl_get_status() == tl.TL_ETIMEOUT
    assert tl.tl_get_status() == tl.TL_OK        # reading clears it
    # the layer still runs and is still exact
    L = synth.config_inputs("tiny")
    lay = tl.TernaryLinear(torch.from_numpy(L.codes), torch.from_numpy(L.s))
    x = torch.from_numpy(L.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8)
    acc = torch.empty((L.M, L.N), dtype=torch.int32, device="cuda")
    tl.tl_linear_decode(lay.packed, lay.qT, lay.sw, xq, sx, L.N, L.K, tl.TL_F32, acc_dbg=acc)
    assert tl.tl_get_status() == tl.TL_OK
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), O.layer(L.x_bits, L.codes, L.s)["acc"])

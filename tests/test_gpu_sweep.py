"""The M sweep of the workloads: M in {1, 2, 4, ..., 1024, 4096} over the two MLP
shapes (K = 5120 -> N = 17408 and K = 17408 -> N = 5120), through the prefill
kernel at every M and the decode kernel for M <= 32. The int32 accumulator
is compared bit for bit with the oracle on the whole output for M <= 64 and
on 64 seeded sampled rows above; the fp32 output must be identical too."""

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth, tl

pytestmark = pytest.mark.gpu

_CACHE = {}


def _weights(name):
    if name not in _CACHE:
        L = synth.config_inputs(name, M=1)
        codes = torch.from_numpy(L.codes).cuda()
        s = torch.from_numpy(L.s).cuda()
        packed, qT, sw = tl.tl_pack_weights(codes, s)
        torch.cuda.synchronize()
        _CACHE.clear()
        _CACHE[name] = (L.codes, L.s, packed, qT, sw)
    return _CACHE[name]


@pytest.mark.parametrize("name", ["sweep_up", "sweep_down"])
@pytest.mark.parametrize("M", synth.SWEEP_M)
def test_sweep(name, M):
    codes, s, packed, qT, sw = _weights(name)
    N, K = codes.shape
    L = synth.config_inputs(name, M=M, N=128)          # x only (same seed; codes of this draw unused)
    x = torch.from_numpy(L.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    rows = None if M <= 64 else np.sort(np.random.default_rng(M).choice(N, size=64, replace=False))
    ref = O.layer(L.x_bits, codes, s, rows=rows)
    paths = ["prefill"] + (["decode"] if M <= 32 else [])
    for path in paths:
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        if path == "prefill":
            xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_F16)
            ws = tl.tl_prefill_workspace_size(M, N, K)
            wsb = torch.zeros((max(ws, 16),), dtype=torch.uint8, device="cuda")
            y = tl.tl_linear_prefill(packed, qT, sw, xq, sx, N, K, tl.TL_F32, acc_dbg=acc, workspace=wsb)
        else:
            xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8)
            y = tl.tl_linear_decode(packed, qT, sw, xq, sx, N, K, tl.TL_F32, acc_dbg=acc)
        torch.cuda.synchronize()
        assert tl.tl_get_status() == tl.TL_OK
        a = acc.cpu().numpy().astype(np.int64)
        yv = y.cpu().numpy()
        if rows is not None:
            a, yv = a[:, rows], yv[:, rows]
        assert np.array_equal(a, ref["acc"]), path
        assert np.array_equal(yv, ref["y32"]), path

"""TernaryLinear's choice of kernel per batch size (host logic, no GPU): the dp4a
decode up to 4 tokens (while M K <= 72 K), the tensor-core decode for 5-16
tokens while K <= 8192, the tcgen05 prefill kernel otherwise."""

import pytest

from quantized_linear_layers_block_gb300 import tl


def layer(K, N=5120):
    lay = object.__new__(tl.TernaryLinear)   # routing reads only the shape
    lay.N, lay.K = N, K
    return lay


@pytest.mark.parametrize("K,expect", [
    (5120, {1: "decode", 4: "decode", 5: "decode_tc", 8: "decode_tc", 16: "decode_tc",
            17: "prefill", 32: "prefill", 512: "prefill"}),
    (8192, {4: "decode", 5: "decode_tc", 16: "decode_tc", 17: "prefill"}),
    (17408, {1: "decode", 4: "decode", 5: "prefill", 16: "prefill", 256: "prefill"}),
    (32768, {1: "decode", 2: "decode", 3: "prefill", 16: "prefill"}),
])
def test_kernel_for(K, expect):
    lay = layer(K)
    for M, kind in expect.items():
        assert lay.kernel_for(M) == kind, (K, M)


def test_boundaries_follow_the_constants():
    lay = layer(5120)
    assert lay.kernel_for(lay.DECODE_MAX_M) == "decode"
    assert lay.kernel_for(lay.TC_MAX_M) == "decode_tc"
    assert lay.kernel_for(lay.TC_MAX_M + 1) == "prefill"
    deep = layer(lay.TC_MAX_K + 1024)
    assert deep.kernel_for(lay.DECODE_MAX_M + 1) == "prefill"

"""TernaryLinear's choice of kernel per batch size (host logic, no GPU): the dp4a
decode up to 4 tokens while M K <= 64 K, the tcgen05 prefill kernel otherwise."""

import pytest

from quantized_linear_layers_block_gb300 import tl


def layer(K, N=5120):
    lay = object.__new__(tl.TernaryLinear)   # routing reads only the shape
    lay.N, lay.K = N, K
    return lay


@pytest.mark.parametrize("K,expect", [
    (5120, {1: "decode", 4: "decode", 5: "prefill", 8: "prefill", 16: "prefill",
            17: "prefill", 32: "prefill", 512: "prefill"}),
    (8192, {4: "decode", 5: "prefill", 16: "prefill"}),
    (17408, {1: "decode", 3: "decode", 4: "prefill", 16: "prefill", 256: "prefill"}),
    (32768, {1: "decode", 2: "decode", 3: "prefill", 16: "prefill"}),
])
def test_kernel_for(K, expect):
    lay = layer(K)
    for M, kind in expect.items():
        assert lay.kernel_for(M) == kind, (K, M)


def test_boundaries_follow_the_constants():
    lay = layer(5120)
    assert lay.kernel_for(lay.DECODE_MAX_M) == "decode"
    assert lay.kernel_for(lay.DECODE_MAX_M + 1) == "prefill"
    deep = layer(lay.DECODE_MAX_MK // 2 + 1024)
    assert deep.kernel_for(2) == "prefill"
    assert deep.kernel_for(1) == "decode"

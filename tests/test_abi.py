"""The C-ABI library builds, loads and exports every entry point of include/tl.h;
argument errors are returned before any CUDA call (no GPU needed)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "tl.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from quantized_linear_layers_block_gb300 import build
    build.build()
    from quantized_linear_layers_block_gb300 import tl
    return tl.lib()


def test_header_declares_the_four_layer_entry_points():
    names = declared_functions()
    for n in ("tl_pack_weights", "tl_rotate_quant_act", "tl_linear_prefill", "tl_linear_decode"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from quantized_linear_layers_block_gb300 import tl
    assert set(declared_functions()) <= set(tl.SIGNATURES)


def test_strerror_and_version(lib):
    from quantized_linear_layers_block_gb300 import tl
    assert tl.tl_version() >= 10000
    for code in range(7):
        assert tl.tl_strerror(code).startswith("TL_")


def test_packed_sizes(lib):
    from quantized_linear_layers_block_gb300 import tl
    assert tl.tl_packed_sizes(17408, 5120) == (22_282_240, 696_320, 69_632)
    assert tl.tl_packed_sizes(5120, 17408) == (22_282_240, 696_320, 20_480)
    with pytest.raises(tl.TLError):
        tl.tl_packed_sizes(100, 1024)


def test_argument_errors_without_gpu(lib):
    from quantized_linear_layers_block_gb300 import tl
    P = ctypes.c_void_p
    bad = P(16 + 3)   # misaligned, never dereferenced
    ok = P(4096)
    # shapes
    assert lib.tl_linear_decode(ok, ok, ok, ok, ok, 33, 128, 1024, ok, tl.TL_F32, None, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode(ok, ok, ok, ok, ok, 1, 130, 1024, ok, tl.TL_F32, None, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_prefill(ok, ok, ok, ok, ok, 1, 128, 1000, ok, tl.TL_F32, None, None, 0, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_prefill(ok, ok, ok, ok, ok, 1, 128, 33792, ok, tl.TL_F32, None, None, 0, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_rotate_quant_act(ok, 1, 1536, None, ok, tl.TL_I8, ok, None) == tl.TL_EUNSUPPORTED
    # fused decode: M <= 16; M = 1 up to K = 8192; M >= 2 while M (rounded up) * K <= 72 K, on
    # the multi-token kernel's K values
    fused = lib.tl_linear_decode_fused
    assert fused(ok, ok, ok, ok, None, 17, 128, 1024, ok, tl.TL_F32, None, None, None, None) == tl.TL_EUNSUPPORTED
    assert fused(ok, ok, ok, ok, None, 1, 128, 9216, ok, tl.TL_F32, None, None, None, None) == tl.TL_EUNSUPPORTED
    assert fused(ok, ok, ok, ok, None, 16, 128, 5120, ok, tl.TL_F32, None, None, None, None) == tl.TL_EUNSUPPORTED
    assert fused(ok, ok, ok, ok, None, 2, 128, 6144, ok, tl.TL_F32, None, None, None, None) == tl.TL_EUNSUPPORTED
    assert fused(ok, ok, ok, ok, None, 5, 128, 17408, ok, tl.TL_F32, None, None, None, None) == tl.TL_EUNSUPPORTED
    # negative sizes, NULLs, misalignment, dtypes
    assert lib.tl_linear_prefill(ok, ok, ok, ok, ok, -1, 128, 1024, ok, tl.TL_F32, None, None, 0, None) == tl.TL_EINVAL
    assert lib.tl_linear_prefill(ok, ok, ok, None, ok, 4, 128, 1024, ok, tl.TL_F32, None, None, 0, None) == tl.TL_EINVAL
    assert lib.tl_linear_prefill(ok, ok, ok, bad, ok, 4, 128, 1024, ok, tl.TL_F32, None, None, 0, None) == tl.TL_EINVAL
    assert lib.tl_linear_prefill(ok, ok, ok, ok, ok, 4, 128, 1024, ok, 7, None, None, 0, None) == tl.TL_EINVAL
    assert lib.tl_linear_prefill(ok, ok, ok, ok, ok, 4, 128, 1024, ok, tl.TL_F32, bad, None, 0, None) == tl.TL_EINVAL
    assert lib.tl_linear_decode(ok, ok, ok, ok, ok, 4, 128, 1024, None, tl.TL_BF16, None, None) == tl.TL_EINVAL
    assert lib.tl_rotate_quant_act(ok, 2, 1024, bad, ok, tl.TL_I8, ok, None) == tl.TL_EINVAL
    assert lib.tl_rotate_quant_act(ok, 2, 1024, None, ok, tl.TL_BF16, ok, None) == tl.TL_EINVAL
    assert lib.tl_pack_weights(ok, ok, 128, 1024, ok, None, ok, None) == tl.TL_EINVAL
    assert lib.tl_pack_weights(ok, ok, 120, 1024, ok, ok, ok, None) == tl.TL_EUNSUPPORTED
    # empty problems are valid no-ops
    assert lib.tl_linear_decode(None, None, None, None, None, 0, 128, 1024, None, tl.TL_BF16, None, None) == tl.TL_OK
    assert lib.tl_linear_prefill(None, None, None, None, None, 5, 0, 1024, None, tl.TL_BF16, None, None, 0, None) == tl.TL_OK
    assert lib.tl_rotate_quant_act(None, 0, 2048, None, None, tl.TL_F16, None, None) == tl.TL_OK
    sz = ctypes.c_size_t(99)
    assert lib.tl_prefill_workspace_size(0, 128, 1024, ctypes.byref(sz)) == tl.TL_OK and sz.value == 0


def test_codec_argument_errors_without_gpu(lib):
    from quantized_linear_layers_block_gb300 import tl
    P = ctypes.c_void_p
    bad = P(16 + 4)
    ok = P(4096)
    assert lib.tl_codec_quant(ok, 4, 200, ok, ok, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_codec_quant(ok, -1, 256, ok, ok, None) == tl.TL_EINVAL
    assert lib.tl_codec_quant(ok, 4, 0, ok, ok, None) == tl.TL_EINVAL
    assert lib.tl_codec_quant(ok, 4, 256, None, ok, None) == tl.TL_EINVAL
    assert lib.tl_codec_quant(ok, 4, 256, ok, bad, None) == tl.TL_EINVAL
    assert lib.tl_codec_quant(None, 0, 256, None, None, None) == tl.TL_OK
    assert lib.tl_codec_dequant_add(ok, ok, ok, 8, 4, 256, ok, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_codec_dequant_add(ok, ok, ok, -1, 4, 256, ok, None) == tl.TL_EINVAL
    assert lib.tl_codec_dequant_add(ok, ok, ok, 1, 4, 384 + 64, ok, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_codec_dequant_add(ok, None, ok, 1, 4, 256, ok, None) == tl.TL_EINVAL
    assert lib.tl_codec_dequant_add(ok, ok, ok, 1, 4, 256, bad, None) == tl.TL_EINVAL
    assert lib.tl_codec_dequant_add(None, None, None, 1, 0, 256, None, None) == tl.TL_OK


def test_float_decode_argument_errors_without_gpu(lib):
    from quantized_linear_layers_block_gb300 import tl
    P = ctypes.c_void_p
    bad = P(16 + 8)
    ok = P(4096)
    assert lib.tl_linear_decode_f32act(ok, ok, ok, 5, 128, 1024, ok, tl.TL_F32, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode_f32act(ok, ok, ok, 4, 128, 10240, ok, tl.TL_F32, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode_f32act(ok, ok, ok, 1, 128, 1000, ok, tl.TL_F32, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_linear_decode_f32act(ok, None, ok, 1, 128, 1024, ok, tl.TL_F32, None) == tl.TL_EINVAL
    assert lib.tl_linear_decode_f32act(ok, ok, bad, 1, 128, 1024, ok, tl.TL_F32, None) == tl.TL_EINVAL
    assert lib.tl_linear_decode_f32act(ok, ok, ok, 1, 128, 1024, ok, tl.TL_I8, None) == tl.TL_EINVAL
    assert lib.tl_linear_decode_f32act(None, None, None, 0, 128, 1024, None, tl.TL_F32, None) == tl.TL_OK
    assert lib.tl_rotate_act(ok, 1, 1536, None, ok, None) == tl.TL_EUNSUPPORTED
    assert lib.tl_rotate_act(ok, 1, 1024, bad, ok, None) == tl.TL_EINVAL
    assert lib.tl_rotate_act(None, 0, 1024, None, None, None) == tl.TL_OK

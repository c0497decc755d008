"""Pins of the int8 128-group codec oracle (oracle/int8_codec.py) to facts that
do not depend on the oracle itself: exact integer round trips, the rounding
error bound of a symmetric 127-level quantiser, the per-group (not per-row)
scale, zero groups, and the pages' own error figure.

Pages: Qiita item ecc183fae033565af7cb §6 "最後に残った問題" (int8 with one
scale per 128 elements, all-gather, own part added in bf16, "1.5 % error per
call"), and item 66e136acefd5a54b2f1d §5 "解説: 長文を読む速度(prefill)"
(the compress and decompress-and-add kernels, 1584-row payloads).

The mutation tests at the end plant plausible mistakes in the oracle and check
that at least one pin fails for each.
"""

import numpy as np
import pytest

from oracle import int8_codec as C
from oracle.ternary_linear import bf16_to_f32, f32_to_bf16_bits
from quantized_linear_layers_block_gb300 import synth


def _bits(v):
    return f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def _int_payload(rng, R, H, peak=127):
    """Integers in [-peak, peak] with every 128-group holding +-peak somewhere."""
    x = rng.integers(-peak, peak + 1, size=(R, H)).astype(np.float32)
    for g in range(H // 128):
        x[:, 128 * g + rng.integers(0, 128)] = peak * rng.choice([-1.0, 1.0])
    return x


# ------------------------------------------------------------------ pins

def pin_integer_roundtrip_exact():
    """Group max 127 and integer values: scale = 127/127 = 1, so q = x exactly."""
    rng = np.random.default_rng(1)
    x = _int_payload(rng, 3, 384)
    q, s = C.quantize_groups(_bits(x))
    assert np.all(s == 1.0)
    assert np.array_equal(q.astype(np.float32), x)
    assert np.array_equal(C.dequantize_groups(q, s), x)


def pin_integer_add_exact():
    """own + peer with small integers is exact in fp32 and in bf16 (|sum| <= 227 < 256)."""
    rng = np.random.default_rng(2)
    own = rng.integers(-100, 101, size=(2, 256)).astype(np.float32)
    peer = _int_payload(rng, 2, 256)
    q, s = C.quantize_groups(_bits(peer))
    out = bf16_to_f32(C.dequant_add(_bits(own), q, s))
    assert np.array_equal(out, own + peer)


def pin_two_peers_add_exact():
    """Three ranks of integer payloads: the sum of all parts, exactly (|sum| <= 256)."""
    rng = np.random.default_rng(3)
    own = rng.integers(-2, 3, size=(2, 256)).astype(np.float32)
    peers = [_int_payload(rng, 2, 256) for _ in range(2)]
    qs, ss = zip(*(C.quantize_groups(_bits(p)) for p in peers))
    out = bf16_to_f32(C.dequant_add(_bits(own), np.stack(qs), np.stack(ss)))
    assert np.array_equal(out, own + peers[0] + peers[1])


def pin_roundtrip_error_bound():
    """|q scale - x| <= scale/2 (1 + 1e-4) for a nearest-rounding 127-level quantiser."""
    x = synth.codec_parts(11, 8, 1024, 1)[0]
    q, s = C.quantize_groups(x)
    xf = bf16_to_f32(x).astype(np.float64)
    err = np.abs(C.dequantize_groups(q, s).astype(np.float64) - xf).reshape(8, 8, 128)
    assert np.all(err <= (s.astype(np.float64)[:, :, None] / 2) * (1 + 1e-4))


def pin_group_max_reaches_127():
    """The largest element of every non-zero group maps to +-127; none exceeds it."""
    x = synth.codec_parts(12, 8, 1024, 1)[0]
    q, s = C.quantize_groups(x)
    mx = np.abs(q.astype(np.int32)).reshape(8, 8, 128).max(axis=2)
    assert np.all(mx[s > 0] == 127)
    assert np.abs(q.astype(np.int32)).max() <= 127


def pin_scale_is_per_group():
    """An outlier in group 1 leaves group 0's scale alone (a per-row scale would not)."""
    x = np.zeros((1, 256), dtype=np.float32)
    x[0, :128] = np.linspace(-1.0, 1.0, 128, dtype=np.float32)
    x[0, 200] = 1000.0
    q, s = C.quantize_groups(_bits(x))
    assert s[0, 0] == np.float32(1.0) / np.float32(127)
    assert abs(int(q[0, 0])) == 127 and abs(int(q[0, 127])) == 127
    assert s[0, 1] == np.float32(1000.0) / np.float32(127)


def pin_zero_groups():
    """An all-zero group: codes 0, scale 0, and decompress-and-add returns the own part."""
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 128:] = 3.0
    q, s = C.quantize_groups(_bits(x))
    assert np.all(q[0] == 0) and np.all(s[0] == 0) and np.all(q[1, :128] == 0) and s[1, 0] == 0
    own = _bits(np.full((2, 256), 0.5, dtype=np.float32))
    out = bf16_to_f32(C.dequant_add(own, q, s))
    assert np.all(out[0] == 0.5) and np.all(out[1, :128] == 0.5) and np.all(out[1, 128:] == 3.5)


def pin_own_part_is_not_compressed():
    """A peer of zeros: the output is the own part bit for bit, whatever its values."""
    own = synth.codec_parts(13, 4, 512, 1)[0]
    q = np.zeros((4, 512), dtype=np.int8)
    s = np.zeros((4, 4), dtype=np.float32)
    assert np.array_equal(C.dequant_add(own, q, s), own)


def pin_pages_error_figure():
    """The pages report about 1.5 % error per compressed all-reduce; the payload of
    the 1584-row workload (a 64-row sample) stays below that."""
    c = synth.CODEC
    own, peer = synth.codec_parts(c["seed"], 64, c["H"], 2, c["outlier_frac"], c["outlier_factor"])
    q, s = C.quantize_groups(peer)
    y = bf16_to_f32(C.dequant_add(own, q, s)).astype(np.float64)
    ref = C.allreduce_fp64([own, peer])
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 1.5e-2
    assert rel > 1e-4          # it is a lossy codec: far from exact on real payloads


PINS = [pin_integer_roundtrip_exact, pin_integer_add_exact, pin_two_peers_add_exact,
        pin_roundtrip_error_bound, pin_group_max_reaches_127, pin_scale_is_per_group,
        pin_zero_groups, pin_own_part_is_not_compressed, pin_pages_error_figure]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ------------------------------------------------------------------ planted mistakes

_real_quant = C.quantize_groups
_real_deq = C.dequantize_groups


def _quant_per_row(x_bits):
    x = bf16_to_f32(np.asarray(x_bits, dtype=np.uint16))
    R, H = x.shape
    a = np.max(np.abs(x), axis=1, keepdims=True)                  # planted: one scale per row
    inv = np.where(a > 0, np.float32(127) / np.where(a > 0, a, 1), 0).astype(np.float32)
    q = np.clip(np.rint(x * inv), -127, 127).astype(np.int8)
    s = np.repeat(np.where(a > 0, a / np.float32(127), 0).astype(np.float32), H // 128, axis=1)
    return q, s


def _quant_floor(x_bits):
    x = bf16_to_f32(np.asarray(x_bits, dtype=np.uint16))
    R, H = x.shape
    xg = x.reshape(R, H // 128, 128)
    a = np.max(np.abs(xg), axis=2)
    safe = np.where(a > 0, a, 1).astype(np.float32)
    inv = np.where(a > 0, np.float32(127) / safe, 0).astype(np.float32)
    q = np.clip(np.trunc(xg * inv[:, :, None]), -127, 127).astype(np.int8)   # planted: truncation
    return q.reshape(R, H), np.where(a > 0, safe / np.float32(127), 0).astype(np.float32)


def _quant_128_levels(x_bits):
    q, s = _real_quant(x_bits)
    return q, (s * np.float32(127) / np.float32(128)).astype(np.float32)   # planted: a/128


def _deq_group_shift(q, s):
    return _real_deq(q, np.roll(s, 1, axis=1))                       # planted: wrong group index


def _deq_add_compress_own(own_bits, qp, sp):
    qo, so = _real_quant(own_bits)                                   # planted: own part compressed too
    acc = _real_deq(qo, so)
    qp = np.asarray(qp)
    sp = np.asarray(sp)
    if qp.ndim == 2:
        qp, sp = qp[None], sp[None]
    for p in range(qp.shape[0]):
        acc = (acc + _real_deq(qp[p], sp[p])).astype(np.float32)
    return f32_to_bf16_bits(acc)


MUTANTS = [
    ("quantize_groups", _quant_per_row),
    ("quantize_groups", _quant_floor),
    ("quantize_groups", _quant_128_levels),
    ("dequantize_groups", _deq_group_shift),
    ("dequant_add", _deq_add_compress_own),
]


@pytest.mark.parametrize("name,fake", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, fake):
    monkeypatch.setattr(C, name, fake)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake in {name}"


def test_tiny_group_overflowing_inverse():
    """A group of bf16 subnormals: inv = 127/a overflows to +inf; non-zeros code to
    +-127 (x inf = +-inf, clamped) and exact zeros to 0."""
    x = np.zeros((1, 128), dtype=np.uint16)
    x[0, 3] = 0x0001          # +9.2e-41
    x[0, 7] = 0x8002          # -1.8e-40
    q, s = C.quantize_groups(x)
    assert s[0, 0] > 0 and np.isfinite(s[0, 0])
    assert q[0, 3] == 127 and q[0, 7] == -127
    assert np.count_nonzero(q) == 2

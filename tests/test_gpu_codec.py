"""GPU parity of the int8 128-group codec (tl_codec_quant, tl_codec_dequant_add)
against the CPU oracle (oracle/int8_codec.py): bit-exact int8 codes, fp32 scales
and bf16 sums on ragged, small, full-size (1584 x 5120) and edge-case payloads.

Pages: Qiita item ecc183fae033565af7cb §6 "最後に残った問題" and item
66e136acefd5a54b2f1d §5 "解説: 長文を読む速度(prefill)".
"""

import numpy as np
import pytest
import torch

from oracle import int8_codec as C
from quantized_linear_layers_block_gb300 import synth
from quantized_linear_layers_block_gb300 import tl

pytestmark = pytest.mark.gpu


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _quant_both(xb):
    q, s = tl.tl_codec_quant(_dev_bf16(xb))
    torch.cuda.synchronize()
    qo, so = C.quantize_groups(xb)
    return q.cpu().numpy(), s.cpu().numpy(), qo, so


@pytest.mark.parametrize("R,H", [(1, 128), (3, 256), (37, 640), (129, 5120), (5, 17408)])
def test_quant_matches_oracle(R, H):
    xb = synth.codec_parts(100 + R, R, H, 1)[0]
    q, s, qo, so = _quant_both(xb)
    assert np.array_equal(q, qo)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quant_edge_values():
    R, H = 6, 384
    x = synth.codec_parts(7, R, H, 1)[0].copy()
    x[0, :] = 0                                  # zero row
    x[1, :128] = 0x7F7F                          # bf16 max, a whole group
    x[1, 128:256] = np.where(np.arange(128) % 2, 0x7F7F, 0xFF7F)   # +-max alternating
    x[2, :128] = 0                               # one group of subnormals and zeros
    x[2, 5] = 0x0001
    x[2, 9] = 0x8003
    x[3, 256:] = 0x0080                          # smallest normal everywhere
    x[4, :] = 0x3F80                             # all 1.0 (ties of x*inv at exactly 127)
    x[5, ::2] = 0xBF80                           # -1.0 / ... mix
    q, s, qo, so = _quant_both(x)
    assert np.array_equal(q, qo)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("npeers", [0, 1, 2, 3, 7])
@pytest.mark.parametrize("R,H", [(37, 640), (64, 5120)])
def test_dequant_add_matches_oracle(npeers, R, H):
    parts = synth.codec_parts(300 + npeers, R, H, npeers + 1)
    own = parts[0]
    qs, ss = [], []
    for p in parts[1:]:
        q, s = C.quantize_groups(p)
        qs.append(q)
        ss.append(s)
    if npeers:
        qd = torch.from_numpy(np.stack(qs)).cuda()
        sd = torch.from_numpy(np.stack(ss)).cuda()
        ref = C.dequant_add(own, np.stack(qs), np.stack(ss))
    else:
        qd = sd = None
        ref = own
    out = tl.tl_codec_dequant_add(_dev_bf16(own), qd, sd)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), ref)


def test_dequant_add_in_place():
    R, H = 40, 1024
    own, peer = synth.codec_parts(17, R, H, 2)
    q, s = C.quantize_groups(peer)
    buf = _dev_bf16(own)
    tl.tl_codec_dequant_add(buf, torch.from_numpy(q).cuda()[None], torch.from_numpy(s).cuda()[None], out=buf)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(buf), C.dequant_add(own, q, s))


def test_full_size_allreduce_two_ranks():
    """The 1584 x 5120 workload, two ranks emulated on one GPU: each rank compresses
    its part on the GPU, the 'all-gather' is a device copy, each rank adds the
    other's part to its own. Every byte matches the oracle."""
    c = synth.CODEC
    parts = synth.codec_parts(c["seed"], c["R"], c["H"], 2, c["outlier_frac"], c["outlier_factor"])
    dev = [_dev_bf16(p) for p in parts]
    comp = [tl.tl_codec_quant(d) for d in dev]
    outs = [tl.tl_codec_dequant_add(dev[r], comp[1 - r][0][None].contiguous(), comp[1 - r][1][None].contiguous())
            for r in range(2)]
    torch.cuda.synchronize()
    assert tl.tl_get_status() == tl.TL_OK
    for r in range(2):
        qo, so = C.quantize_groups(parts[1 - r])
        assert np.array_equal(comp[1 - r][0].cpu().numpy(), qo)
        assert np.array_equal(_bits(outs[r]), C.dequant_add(parts[r], qo, so))


def test_empty_payload_is_a_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = tl.tl_codec_quant(x)
    out = tl.tl_codec_dequant_add(x, q[None], s[None])
    torch.cuda.synchronize()
    assert q.numel() == 0 and out.numel() == 0

"""The row-parallel (K-split) algebra of the pages, emulated with two ranks.

Qiita item ecc183fae033565af7cb §1 "TP=2 への移植": with the input features
split across two ranks, a 1024-block that straddles the split is rotated with
the Sylvester recursion H1024 [a; b] = [H512 a + H512 b; H512 a - H512 b]: each
rank transforms its 512-half, the halves are exchanged, rank 0 keeps the sum
and rank 1 the difference. The per-token absmax of the quantiser is an
all-reduce(max); the integer accumulator of §4 is an all-reduce(sum) of int32
partial sums, which is exact and independent of the order.

test_ksplit_two_ranks_gloo runs the algebra as two gloo processes on the CPU
(the exchange is a real all_gather, the reductions real all_reduce calls) and
checks xq, acc and y bit for bit against the one-process oracle. The GPU test
splits the layer's K between two halves of the library's own call and checks
that the two int32 partial accumulators add up to the full one.
"""

import os
import socket
import tempfile

import numpy as np
import pytest
import torch

from oracle import ternary_linear as O
from quantized_linear_layers_block_gb300 import synth

M, K, N = 4, 3072, 256        # K/2 = 1536: the middle 1024-block straddles the two ranks


def _inputs():
    return synth.config_inputs("tiny", M=M, K=K, N=N)


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_rotation(x: np.ndarray, rank: int, world: int, swap: bool = False) -> np.ndarray:
    """fp32 rotation of this rank's columns; a block split between ranks goes
    through the §1 recursion with one all_gather of the half transforms."""
    import torch.distributed as dist
    kr = K // world
    c0, c1 = rank * kr, (rank + 1) * kr
    out = np.zeros((M, kr), dtype=np.float32)
    for b in range(K // O.BLOCK):
        b0, b1 = b * O.BLOCK, (b + 1) * O.BLOCK
        lo, hi = max(b0, c0), min(b1, c1)
        whole = lo == b0 and hi == b1
        if whole:
            out[:, lo - c0:hi - c0] = O.fwht(x[:, b0:b1], np.float32) * O.INV_SQRT_BLOCK
            continue
        if lo >= hi:
            continue          # a block of the other rank alone (a split block is touched by both)
        half = O.BLOCK // 2
        mine = O.fwht(x[:, lo:hi], np.float32)                    # H512 of this rank's half
        parts = [torch.empty((M, half), dtype=torch.float32) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(mine)))
        a, bb = parts[0].numpy(), parts[1].numpy()                 # halves in rank order
        first = (lo == b0)                                          # this rank holds the first half
        if swap:
            first = not first                                      # the ranks' halves exchanged
        res = (a + bb) if first else (a - bb)                       # the last butterfly stage (stride 512)
        out[:, lo - c0:hi - c0] = res.astype(np.float32) * O.INV_SQRT_BLOCK
    return out


def _ksplit_worker(rank: int, world: int, port: int, outdir: str, swap: bool) -> None:
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = _inputs()
        x = O.bf16_to_f32(inp.x_bits)
        kr = K // world
        cols = slice(rank * kr, (rank + 1) * kr)
        xr = _rank_rotation(x, rank, world, swap)
        # per-token absmax: all_reduce(max) of the local maxima
        a = torch.from_numpy(np.max(np.abs(xr), axis=1).astype(np.float32))
        dist.all_reduce(a, op=dist.ReduceOp.MAX)
        a = a.numpy()
        xq = np.zeros((M, kr), dtype=np.int8)
        sx = np.zeros(M, dtype=np.float32)
        for m in range(M):
            if a[m] > 0:
                inv = np.float32(O.QMAX) / a[m]
                xq[m] = np.clip(np.rint(xr[m] * inv), -O.QMAX, O.QMAX).astype(np.int8)
                sx[m] = a[m] / np.float32(O.QMAX)
        # the row scales are the full row's (one smax per output feature for all ranks)
        q, sw, _ = O.row_scale_decompose(inp.s)
        g0, g1 = cols.start // O.GROUP, cols.stop // O.GROUP
        acc = O.int_gemm(xq, O.expand_w_int8(inp.codes[:, cols], q[:, g0:g1]))
        acc_t = torch.from_numpy(acc.astype(np.int32))
        dist.all_reduce(acc_t, op=dist.ReduceOp.SUM)                 # the int32 all-reduce
        y = O.epilogue(acc_t.numpy().astype(np.int64), sw, sx)
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), xr=xr, xq=xq, acc=acc_t.numpy(), y=y, sx=sx)
    finally:
        dist.destroy_process_group()


def _run_two_ranks(swap: bool):
    import torch.multiprocessing as mp
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_ksplit_worker, args=(2, _free_port(), d, swap), nprocs=2, join=True)
        return [dict(np.load(os.path.join(d, f"rank{r}.npz"))) for r in range(2)]


def test_ksplit_two_ranks_gloo():
    res = _run_two_ranks(swap=False)
    ref = O.layer(_inputs().x_bits, _inputs().codes, _inputs().s)
    xr_ref = O.rotate_fp32(_inputs().x_bits)
    assert np.array_equal(np.concatenate([r["xr"] for r in res], axis=1), xr_ref)
    assert np.array_equal(np.concatenate([r["xq"] for r in res], axis=1), ref["xq"])
    for r in res:
        assert np.array_equal(r["sx"], ref["sx"])
        assert np.array_equal(r["acc"].astype(np.int64), ref["acc"])
        assert np.array_equal(r["y"], ref["y32"])


def test_ksplit_rank_swap_negative_control():
    """Swapping the sum and difference halves (the mistake the pages describe)
    scrambles the straddled block: its relative error is about sqrt(2) (the
    pages measured 1.44)."""
    res = _run_two_ranks(swap=True)
    xr = np.concatenate([r["xr"] for r in res], axis=1).astype(np.float64)
    ref = O.rotate_fp64(_inputs().x_bits)
    blk = slice(O.BLOCK, 2 * O.BLOCK)
    err = np.linalg.norm(xr[:, blk] - ref[:, blk]) / np.linalg.norm(ref[:, blk])
    assert 1.2 < err < 1.6
    # the blocks that each rank owns whole are untouched
    assert np.allclose(xr[:, :O.BLOCK], ref[:, :O.BLOCK], rtol=0, atol=1e-5)


@pytest.mark.gpu
@pytest.mark.parametrize("Mg", [1, 64])
def test_ksplit_int32_partials_add_up_on_gpu(Mg):
    """Two K-halves through the library: acc(half 0) + acc(half 1) == acc(full),
    bit for bit, for the decode (M = 1) and prefill (M = 64) kernels."""
    from quantized_linear_layers_block_gb300 import tl
    Kg, Ng = 2048, 256
    inp = synth.config_inputs("tiny", M=Mg, K=Kg, N=Ng)
    codes = torch.from_numpy(inp.codes).cuda()
    s = torch.from_numpy(inp.s).cuda()
    x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    packed, qT, sw = tl.tl_pack_weights(codes, s)
    decode = Mg <= 32
    xq, sx = tl.tl_rotate_quant_act(x, xq_dtype=tl.TL_I8 if decode else tl.TL_F16)
    call = tl.tl_linear_decode if decode else tl.tl_linear_prefill
    acc_full = torch.empty((Mg, Ng), dtype=torch.int32, device="cuda")
    call(packed, qT, sw, xq, sx, Ng, Kg, tl.TL_F32, acc_dbg=acc_full)
    parts = []
    h = Kg // 2
    for r in range(2):
        pk = packed[:, r * h // 4:(r + 1) * h // 4].contiguous()
        qr = qT[r * h // 128:(r + 1) * h // 128].contiguous()
        xr = xq[:, r * h:(r + 1) * h].contiguous()
        acc = torch.empty((Mg, Ng), dtype=torch.int32, device="cuda")
        call(pk, qr, sw, xr, sx, Ng, h, tl.TL_F32, acc_dbg=acc)
        parts.append(acc)
    torch.cuda.synchronize()
    assert tl.tl_get_status() == tl.TL_OK
    ref = O.layer(inp.x_bits, inp.codes, inp.s)["acc"]
    assert np.array_equal(acc_full.cpu().numpy().astype(np.int64), ref)
    assert np.array_equal((parts[0] + parts[1]).cpu().numpy().astype(np.int64), ref)

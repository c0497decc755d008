"""Python binding of the C ABI in include/tl.h (argument marshalling only).

Every function here forwards device pointers, sizes and the current CUDA
stream to libtl_gb300.so; all arithmetic of the layer runs in the library's
CUDA kernels. PyTorch only allocates device memory and supplies the stream.
If the library has not been built, loading it raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtl_gb300.so")
_lib = None
_lock = threading.Lock()

TL_OK, TL_EINVAL, TL_EUNSUPPORTED, TL_ECUDA, TL_ETIMEOUT, TL_EDATA, TL_ENOSPACE = range(7)
TL_I8, TL_F16, TL_BF16, TL_F32 = 1, 2, 3, 4
FUSED_DECODE_MAX_K = 8192

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "tl_strerror": (ctypes.c_char_p, [_I]),
    "tl_version": (_I, []),
    "tl_packed_sizes": (_I, [_I, _I, _PSZ, _PSZ, _PSZ]),
    "tl_pack_weights": (_I, [_P, _P, _I, _I, _P, _P, _P, _P]),
    "tl_rotate_quant_act": (_I, [_P, _I, _I, _P, _P, _I, _P, _P]),
    "tl_prefill_workspace_size": (_I, [_I, _I, _I, _PSZ]),
    "tl_linear_prefill": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "tl_linear_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "tl_linear_decode_tc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "tl_linear_prefill_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "tl_linear_decode_fused": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P, _P]),
    "tl_rotate_act": (_I, [_P, _I, _I, _P, _P, _P]),
    "tl_linear_decode_f32act": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _P]),
    "tl_codec_quant": (_I, [_P, _I, _I, _P, _P, _P]),
    "tl_codec_dequant_add": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "tl_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "tl_get_status": (_I, [_P]),
}


class TLError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {tl_strerror(code)}")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m quantized_linear_layers_block_gb300.build` (needs nvcc)")
            handle = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def tl_strerror(code: int) -> str:
    return lib().tl_strerror(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != TL_OK:
        raise TLError(code, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_tensor(t: torch.Tensor, dtype: torch.dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def tl_version() -> int:
    return lib().tl_version()


def tl_packed_sizes(N: int, K: int) -> tuple[int, int, int]:
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().tl_packed_sizes(N, K, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "tl_packed_sizes")
    return a.value, b.value, c.value


def tl_prefill_workspace_size(M: int, N: int, K: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().tl_prefill_workspace_size(M, N, K, ctypes.byref(b)), "tl_prefill_workspace_size")
    return b.value


def tl_pack_weights(codes: torch.Tensor, s: torch.Tensor, stream=None):
    """codes int8 [N,K] and s fp16 [N,K/128] (device) -> (packed uint8 [N,K/4], qT int8 [K/128,N], sw fp32 [N])."""
    _dev_tensor(codes, torch.int8, "codes")
    _dev_tensor(s, torch.float16, "s")
    N, K = codes.shape
    dev = codes.device
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
    qT = torch.empty((K // 128, N), dtype=torch.int8, device=dev)
    sw = torch.empty((N,), dtype=torch.float32, device=dev)
    _check(lib().tl_pack_weights(_ptr(codes), _ptr(s), N, K, _ptr(packed), _ptr(qT), _ptr(sw),
                                 _stream(stream)), "tl_pack_weights")
    return packed, qT, sw


def tl_rotate_quant_act(x: torch.Tensor, signs: torch.Tensor | None = None, xq_dtype: int = TL_I8,
                        xq: torch.Tensor | None = None, sx: torch.Tensor | None = None, stream=None):
    """x bf16 [M,K] (device) -> (xq [M,K] int8 or fp16, sx fp32 [M])."""
    _dev_tensor(x, torch.bfloat16, "x")
    M, K = x.shape
    tdt = torch.int8 if xq_dtype == TL_I8 else torch.float16
    if xq is None:
        xq = torch.empty((M, K), dtype=tdt, device=x.device)
    if sx is None:
        sx = torch.empty((M,), dtype=torch.float32, device=x.device)
    if signs is not None:
        _dev_tensor(signs, torch.int8, "signs")
    _check(lib().tl_rotate_quant_act(_ptr(x), M, K, _ptr(signs), _ptr(xq), xq_dtype, _ptr(sx),
                                     _stream(stream)), "tl_rotate_quant_act")
    return xq, sx


def _linear_out(M, N, y_dtype, dev, y):
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16 if y_dtype == TL_BF16 else torch.float32, device=dev)
    return y


def tl_linear_prefill(packed, qT, sw, xq, sx, N: int, K: int, y_dtype: int = TL_BF16,
                      y: torch.Tensor | None = None, acc_dbg: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Tensor-core layer; xq is the fp16 image of the int8 codes [M,K]. Returns y [M,N]."""
    _dev_tensor(xq, torch.float16, "xq")
    M = xq.shape[0]
    y = _linear_out(M, N, y_dtype, xq.device, y)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tl_linear_prefill(_ptr(packed), _ptr(qT), _ptr(sw), _ptr(xq), _ptr(sx), M, N, K,
                                   _ptr(y), y_dtype, _ptr(acc_dbg), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "tl_linear_prefill")
    return y


def tl_linear_prefill_noalloc(packed, qT, sw, xq, sx, N: int, K: int, y_dtype: int = TL_BF16,
                              y: torch.Tensor | None = None, acc_dbg: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """tl_linear_prefill with the library's own static split-K scratch (no workspace argument).

    For callers that cannot allocate device memory; see include/tl.h. Calls
    that may overlap on the GPU share the scratch and must be serialised.
    """
    _dev_tensor(xq, torch.float16, "xq")
    M = xq.shape[0]
    if y is None:
        y = _linear_out(M, N, y_dtype, xq.device, y)
    _check(lib().tl_linear_prefill_noalloc(_ptr(packed), _ptr(qT), _ptr(sw), _ptr(xq), _ptr(sx), M, N,
                                           K, _ptr(y), y_dtype, _ptr(acc_dbg), _stream(stream)),
           "tl_linear_prefill_noalloc")
    return y


def tl_linear_decode(packed, qT, sw, xq, sx, N: int, K: int, y_dtype: int = TL_BF16,
                     y: torch.Tensor | None = None, acc_dbg: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """CUDA-core layer for M <= 32; xq int8 [M,K]. Returns y [M,N]."""
    _dev_tensor(xq, torch.int8, "xq")
    M = xq.shape[0]
    y = _linear_out(M, N, y_dtype, xq.device, y)
    _check(lib().tl_linear_decode(_ptr(packed), _ptr(qT), _ptr(sw), _ptr(xq), _ptr(sx), M, N, K,
                                  _ptr(y), y_dtype, _ptr(acc_dbg), _stream(stream)), "tl_linear_decode")
    return y


def tl_linear_decode_tc(packed, qT, sw, xq, sx, N: int, K: int, y_dtype: int = TL_BF16,
                        y: torch.Tensor | None = None, acc_dbg: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Tensor-core decode for M <= 32; xq is the fp16 image of the codes [M,K]. Returns y [M,N]."""
    _dev_tensor(xq, torch.float16, "xq")
    M = xq.shape[0]
    y = _linear_out(M, N, y_dtype, xq.device, y)
    _check(lib().tl_linear_decode_tc(_ptr(packed), _ptr(qT), _ptr(sw), _ptr(xq), _ptr(sx), M, N, K,
                                     _ptr(y), y_dtype, _ptr(acc_dbg), _stream(stream)),
           "tl_linear_decode_tc")
    return y


def tl_linear_decode_fused(packed, qT, sw, x, N: int, K: int, y_dtype: int = TL_BF16,
                           signs=None, y: torch.Tensor | None = None,
                           acc_dbg: torch.Tensor | None = None, xq_out: torch.Tensor | None = None,
                           sx_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Up to 16 tokens (x bf16 [M, K]) through rotation, quantisation and the decode GEMV in one
    launch (shapes as tl.h states)."""
    _dev_tensor(x, torch.bfloat16, "x")
    M = x.shape[0]
    y = _linear_out(M, N, y_dtype, x.device, y)
    _check(lib().tl_linear_decode_fused(_ptr(packed), _ptr(qT), _ptr(sw), _ptr(x), _ptr(signs), M, N, K,
                                        _ptr(y), y_dtype, _ptr(acc_dbg), _ptr(xq_out), _ptr(sx_out),
                                        _stream(stream)), "tl_linear_decode_fused")
    return y


def tl_rotate_act(x: torch.Tensor, signs: torch.Tensor | None = None, xr: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """x bf16 [M,K] (device) -> xr fp32 [M,K], the rotation alone."""
    _dev_tensor(x, torch.bfloat16, "x")
    M, K = x.shape
    if xr is None:
        xr = torch.empty((M, K), dtype=torch.float32, device=x.device)
    if signs is not None:
        _dev_tensor(signs, torch.int8, "signs")
    _check(lib().tl_rotate_act(_ptr(x), M, K, _ptr(signs), _ptr(xr), _stream(stream)), "tl_rotate_act")
    return xr


def tl_linear_decode_f32act(packed, s, xr, N: int, K: int, y_dtype: int = TL_F32,
                            y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Float-activation decode (M <= 4): s fp16 [N,K/128], xr fp32 [M,K] -> y [M,N]."""
    _dev_tensor(xr, torch.float32, "xr")
    _dev_tensor(s, torch.float16, "s")
    M = xr.shape[0]
    y = _linear_out(M, N, y_dtype, xr.device, y)
    _check(lib().tl_linear_decode_f32act(_ptr(packed), _ptr(s), _ptr(xr), M, N, K, _ptr(y), y_dtype,
                                         _stream(stream)), "tl_linear_decode_f32act")
    return y


def tl_codec_quant(x: torch.Tensor, q: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                   stream=None):
    """Compress a bf16 payload [R,H] -> (int8 q [R,H], fp32 scale [R,H/128])."""
    _dev_tensor(x, torch.bfloat16, "x")
    R, H = x.shape
    if q is None:
        q = torch.empty((R, H), dtype=torch.int8, device=x.device)
    if scale is None:
        scale = torch.empty((R, H // 128), dtype=torch.float32, device=x.device)
    _check(lib().tl_codec_quant(_ptr(x), R, H, _ptr(q), _ptr(scale), _stream(stream)), "tl_codec_quant")
    return q, scale


def tl_codec_dequant_add(own: torch.Tensor, q_peers: torch.Tensor | None, scale_peers: torch.Tensor | None,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """own bf16 [R,H] + the peers' decompressed parts (q int8 [P,R,H], scale fp32 [P,R,H/128]) -> bf16 [R,H]."""
    _dev_tensor(own, torch.bfloat16, "own")
    R, H = own.shape
    npeers = 0
    if q_peers is not None:
        _dev_tensor(q_peers, torch.int8, "q_peers")
        _dev_tensor(scale_peers, torch.float32, "scale_peers")
        npeers = q_peers.shape[0] if q_peers.dim() == 3 else 1
    if out is None:
        out = torch.empty_like(own)
    _check(lib().tl_codec_dequant_add(_ptr(own), _ptr(q_peers), _ptr(scale_peers), npeers, R, H, _ptr(out),
                                      _stream(stream)), "tl_codec_dequant_add")
    return out


def tl_selftest_wait_timeout(limit_us: int = 2000, stream=None) -> None:
    """Launch the library's wait that cannot complete (see include/tl.h); tl_get_status then reads TL_ETIMEOUT."""
    _check(lib().tl_selftest_wait_timeout(int(limit_us), _stream(stream)), "tl_selftest_wait_timeout")


def tl_get_status(stream=None) -> int:
    return lib().tl_get_status(_stream(stream))


class TernaryLinear:
    """One ternary linear layer held in device memory (the library's public entry).

    Built once from int8 codes [N,K] and fp16 group scales [N,K/128]; forward()
    takes bf16 activations [M,K] on the host or the device and returns y [M,N]
    where it found x. Small M * K (decode) runs rotate+quantise and the CUDA-core
    decode kernel, larger problems rotate+quantise and the tensor-core prefill
    kernel; both give the same integer accumulator and the same y.
    """

    # Which kernel serves a batch of M tokens (measured on GB300 over both MLP
    # shapes, rotate+quantise and the kernel per layer, 8 layer buffers in a
    # CUDA graph): the dp4a CUDA-core decode up to 4 tokens while M K <= 64 K
    # (K = 5120, M = 4: 16.2 against 17.2 us for the prefill kernel; K = 17408,
    # M = 3: 21.5 against 21.6, M = 4: 22.5 against 21.8); the tcgen05 prefill
    # kernel above (K = 5120, M = 5..16: 17.3 us against 18.2-23.4 for the
    # mma.sync tensor-core decode, which tl_linear_decode_tc still offers).
    DECODE_MAX_M = 4
    DECODE_MAX_MK = 64 * 1024

    def kernel_for(self, M: int) -> str:
        """'decode' or 'prefill': the kernel forward() runs for M tokens."""
        if M <= self.DECODE_MAX_M and M * self.K <= self.DECODE_MAX_MK:
            return "decode"
        return "prefill"

    def __init__(self, codes: torch.Tensor, s: torch.Tensor, device="cuda", y_dtype: int = TL_BF16):
        dev = torch.device(device)
        codes = codes.to(dev, non_blocking=False).contiguous()
        s = s.to(dev, non_blocking=False).contiguous()
        self.N, self.K = codes.shape
        self.device = dev
        self.y_dtype = y_dtype
        self.packed, self.qT, self.sw = tl_pack_weights(codes, s)
        _check(tl_get_status(), "tl_pack_weights (device check)")
        self._ws = None

    def _workspace(self, M: int):
        need = tl_prefill_workspace_size(M, self.N, self.K)
        if need == 0:
            return None
        if self._ws is None or self._ws.numel() < need:
            # zeroed once here; every call that completes leaves it zero again
            self._ws = torch.zeros((need,), dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, stream=None, out: torch.Tensor | None = None) -> torch.Tensor:
        """y = layer(x). `out` (device, [M, N], the layer's y dtype) receives y when given.

        The layer keeps one split-K workspace for the prefill kernel (used when a
        batch has few output tiles and a long K): calls on the same layer object
        that can run at the same time on different streams must be ordered by
        the caller (an event), or use one layer object per stream."""
        on_host = not x.is_cuda
        xd = x.to(self.device, non_blocking=True) if on_host else x
        M = xd.shape[0]
        kind = self.kernel_for(M)
        if kind == "decode":
            xq, sx = tl_rotate_quant_act(xd, xq_dtype=TL_I8, stream=stream)
            y = tl_linear_decode(self.packed, self.qT, self.sw, xq, sx, self.N, self.K,
                                 self.y_dtype, y=out, stream=stream)
        else:
            xq, sx = tl_rotate_quant_act(xd, xq_dtype=TL_F16, stream=stream)
            y = tl_linear_prefill(self.packed, self.qT, self.sw, xq, sx, self.N, self.K,
                                  self.y_dtype, y=out, workspace=self._workspace(M), stream=stream)
        if on_host:
            out = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
            out.copy_(y, non_blocking=True)
            torch.cuda.current_stream(self.device).synchronize() if stream is None else stream.synchronize()
            return out
        return y

    __call__ = forward


class HostPipeline:
    """Runs TernaryLinear layers on host (pinned) inputs with the copies overlapped.

    Three CUDA streams: host->device copies, the layer kernels, device->host
    copies. submit() queues one layer call and returns at once; the copy of the
    next input runs while the current layer computes, and the copy-back of a
    result while the next layer computes. `depth` device input buffers rotate so
    that a buffer is reused only after the kernels that read it have finished.
    synchronize() waits for every submitted call; results are then in the pinned
    host tensors given to submit(). The arithmetic is the layers' own (the
    library's kernels); this class only orders copies and launches.
    """

    def __init__(self, device="cuda", depth: int = 3):
        self.device = torch.device(device)
        self.depth = depth
        self.h2d = torch.cuda.Stream(self.device)
        self.comp = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self._xbuf = [None] * depth
        self._free = [None] * depth     # event: the kernels reading buffer i have finished
        self._n = 0

    def submit(self, layer: "TernaryLinear", x_host: torch.Tensor, y_host: torch.Tensor) -> None:
        if x_host.is_cuda or y_host.is_cuda:
            raise ValueError("HostPipeline takes host tensors (pinned for overlap)")
        i = self._n % self.depth
        self._n += 1
        buf = self._xbuf[i]
        if buf is None or buf.shape != x_host.shape or buf.dtype != x_host.dtype:
            buf = self._xbuf[i] = torch.empty(x_host.shape, dtype=x_host.dtype, device=self.device)
        with torch.cuda.stream(self.h2d):
            if self._free[i] is not None:
                self.h2d.wait_event(self._free[i])
            buf.copy_(x_host, non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(self.h2d)
        with torch.cuda.stream(self.comp):
            self.comp.wait_event(copied)
            y = layer.forward(buf, stream=self.comp)
            done = torch.cuda.Event()
            done.record(self.comp)
            self._free[i] = done
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(done)
            y.record_stream(self.d2h)
            y_host.copy_(y, non_blocking=True)

    def synchronize(self) -> None:
        self.d2h.synchronize()
        self.comp.synchronize()
        self.h2d.synchronize()


class GraphStep:
    """One step of layer calls with host I/O, captured in a CUDA graph.

    `layers` are TernaryLinear objects and `ms` their token counts. The step
    owns one pinned host buffer for all inputs and one for all outputs, exposed
    as per-layer views (`inputs[i]` bf16 [M_i, K_i], `outputs[i]` [M_i, N_i]).
    run() replays: one host->device copy of every input, each layer's kernels
    writing into a slice of one device output buffer, one device->host copy of
    every output, then waits. A step costs one launch from the host however many
    layers it holds (the serving pattern for decode, where a layer's kernels take
    a few microseconds). Captured once on a side stream after one eager warm-up.
    """

    def __init__(self, layers, ms, device="cuda"):
        self.device = torch.device(device)
        self.layers = list(layers)
        ms = list(ms)
        dt = {TL_BF16: torch.bfloat16, TL_F32: torch.float32}
        ydts = {l.y_dtype for l in self.layers}
        if len(ydts) != 1:
            raise ValueError("GraphStep layers must share one output dtype")
        ydt = dt[ydts.pop()]
        in_sizes = [m * l.K for l, m in zip(self.layers, ms)]
        out_sizes = [m * l.N for l, m in zip(self.layers, ms)]
        self._in_host = torch.empty(sum(in_sizes), dtype=torch.bfloat16).pin_memory()
        self._out_host = torch.empty(sum(out_sizes), dtype=ydt).pin_memory()
        self._in_dev = torch.empty(sum(in_sizes), dtype=torch.bfloat16, device=self.device)
        self._out_dev = torch.empty(sum(out_sizes), dtype=ydt, device=self.device)

        def views(buf, sizes, shapes):
            out, o = [], 0
            for n, shp in zip(sizes, shapes):
                out.append(buf[o:o + n].view(shp))
                o += n
            return out
        in_shapes = [(m, l.K) for l, m in zip(self.layers, ms)]
        out_shapes = [(m, l.N) for l, m in zip(self.layers, ms)]
        self.inputs = views(self._in_host, in_sizes, in_shapes)
        self.outputs = views(self._out_host, out_sizes, out_shapes)
        self._xd = views(self._in_dev, in_sizes, in_shapes)
        self._yd = views(self._out_dev, out_sizes, out_shapes)
        self._stream = torch.cuda.Stream(self.device)
        with torch.cuda.stream(self._stream):
            self._body()
        self._stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self._stream, capture_error_mode="relaxed"):
            self._body()

    def _body(self):
        self._in_dev.copy_(self._in_host, non_blocking=True)
        for layer, xd, yd in zip(self.layers, self._xd, self._yd):
            layer.forward(xd, out=yd)
        self._out_host.copy_(self._out_dev, non_blocking=True)

    def run(self) -> None:
        self.graph.replay()
        torch.cuda.current_stream(self.device).synchronize()

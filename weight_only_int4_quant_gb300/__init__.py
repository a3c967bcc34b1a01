"""Python binding of libtlq: the GB300 weight-only INT4/INT2 quantized linear layer.

Argument marshalling only.  Every step of the layer runs in the library's CUDA
kernels; torch provides device memory and streams.  The C entry points (see
include/tlq.h) are exposed under the same names; a missing or stale library
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB as _LIB_PATH
from .build import build as _build

__all__ = [
    "TLQError", "load", "build", "EXPORTED",
    "tl_quant_gemm", "tl_pack_weights", "tl_unpack_weights", "tl_loop_block_forward",
    "tl_check_status", "tl_reset_status", "tl_selftest_wait_timeout", "tl_last_error", "tl_version",
    "tl_loop_block_forward_static_scratch", "tl_quant_gemm_batched", "gemm_descs", "quant_gemm", "pack_weights", "unpack_weights", "LoopBlock",
    "tl_requant_int4_to_int2", "tl_requant_int4_to_int2_batched", "requant_int4_to_int2",
    "tl_quant_gemm_swiglu", "tl_interleave_rows", "tl_swiglu_block_forward", "quant_gemm_swiglu",
    "interleave_rows", "SwiGLUBlock", "tl_dequant_fp16", "dequant_fp16",
    "tl_loop_block_forward_chunked", "tl_swiglu_block_forward_chunked", "tl_quant_gemm_batched_host",
    "tl_quant_gemm_ws", "tl_quant_gemm_workspace_size", "tl_quant_gemm_swiglu_ws", "tl_loop_block_to_int2",
    "tl_swiglu_block_to_int2", "gemm_workspace", "requant_descs", "tl_probe_read_bandwidth",
    "tl_loop_block_l2_plan", "tl_prefill_plan",
]

# every symbol include/tlq.h declares
EXPORTED = (
    "tl_last_error", "tl_version", "tl_quant_gemm", "tl_pack_weights", "tl_unpack_weights",
    "tl_loop_block_forward", "tl_check_status", "tl_reset_status", "tl_selftest_wait_timeout",
    "tl_loop_block_forward_static_scratch", "tl_quant_gemm_batched", "tl_requant_int4_to_int2",
    "tl_requant_int4_to_int2_batched", "tl_quant_gemm_swiglu", "tl_interleave_rows", "tl_swiglu_block_forward",
    "tl_dequant_fp16", "tl_loop_block_forward_chunked", "tl_swiglu_block_forward_chunked",
    "tl_quant_gemm_batched_host", "tl_quant_gemm_ws", "tl_quant_gemm_workspace_size", "tl_quant_gemm_swiglu_ws",
    "tl_loop_block_to_int2", "tl_swiglu_block_to_int2", "tl_probe_read_bandwidth", "tl_loop_block_l2_plan",
    "tl_prefill_plan",
)

TLQ_OK, TLQ_EINVAL, TLQ_EUNSUPPORTED, TLQ_ECUDA, TLQ_ETIMEOUT = 0, 1, 2, 3, 4
_STATUS_NAMES = {0: "TLQ_OK", 1: "TLQ_EINVAL", 2: "TLQ_EUNSUPPORTED", 3: "TLQ_ECUDA", 4: "TLQ_ETIMEOUT"}


class TLQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, status), message))
        self.status = status


class _QProj(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("s", ctypes.c_void_p), ("z", ctypes.c_void_p),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("ldw", ctypes.c_int)]


class _GemmDesc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("Wpacked", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("C", ctypes.c_void_p), ("M", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("bits", ctypes.c_int), ("group", ctypes.c_int), ("ldw", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class _RequantDesc(ctypes.Structure):
    _fields_ = [("W4", ctypes.c_void_p), ("s4", ctypes.c_void_p), ("z4", ctypes.c_void_p), ("W2", ctypes.c_void_p),
                ("s2", ctypes.c_void_p), ("z2", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int)]


class _Block(ctypes.Structure):
    _fields_ = [("qkv", _QProj), ("o", _QProj), ("up", _QProj), ("down", _QProj),
                ("bits", ctypes.c_int), ("group", ctypes.c_int), ("D", ctypes.c_int),
                ("h", ctypes.c_void_p), ("qkv_out", ctypes.c_void_p), ("o_out", ctypes.c_void_p),
                ("up_out", ctypes.c_void_p), ("normalize", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class _SwigluBlock(ctypes.Structure):
    _fields_ = [("qkv", _QProj), ("o", _QProj), ("gate_up", _QProj), ("down", _QProj),
                ("bits", ctypes.c_int), ("group", ctypes.c_int), ("D", ctypes.c_int),
                ("h", ctypes.c_void_p), ("qkv_out", ctypes.c_void_p), ("o_out", ctypes.c_void_p),
                ("act_out", ctypes.c_void_p), ("normalize", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libtlq.so for sm_103a (nvcc) and return its path."""
    return _build(force=force, verbose=verbose)


def load():
    """Load libtlq.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        try:  # share the process's CUDA runtime with torch
            import torch  # noqa: F401
        except ImportError:
            pass
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libtlq.so is not built (%s); call weight_only_int4_quant_gb300.build()"
                               % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
        sigs = {
            "tl_last_error": ([], ctypes.c_char_p),
            "tl_version": ([], ctypes.c_char_p),
            "tl_quant_gemm": ([P, P, P, P, P, I, I, I, I, I, P], I),
            "tl_pack_weights": ([P, P, I, I, I, P], I),
            "tl_unpack_weights": ([P, P, I, I, I, P], I),
            "tl_loop_block_forward": ([P, ctypes.POINTER(_Block), I, I, P], I),
            "tl_check_status": ([P], I),
            "tl_reset_status": ([P], I),
            "tl_selftest_wait_timeout": ([U, P], I),
            "tl_loop_block_forward_static_scratch": ([P, ctypes.POINTER(_Block), I, I, P], I),
            "tl_quant_gemm_batched": ([ctypes.POINTER(_GemmDesc), I, P], I),
            "tl_requant_int4_to_int2": ([P, P, P, P, P, P, I, I, I, P], I),
            "tl_requant_int4_to_int2_batched": ([ctypes.POINTER(_RequantDesc), I, I, P], I),
            "tl_quant_gemm_swiglu": ([P, P, P, P, P, I, I, I, I, I, P], I),
            "tl_interleave_rows": ([P, P, P, I, ctypes.c_size_t, P], I),
            "tl_dequant_fp16": ([P, P, P, P, I, I, I, I, P], I),
            "tl_quant_gemm_batched_host": ([ctypes.POINTER(_GemmDesc), I, P, P, ctypes.c_size_t, P, P,
                                            ctypes.c_size_t, P], I),
            "tl_loop_block_forward_chunked": ([P, ctypes.POINTER(_Block), I, I, I, P], I),
            "tl_swiglu_block_forward_chunked": ([P, ctypes.POINTER(_SwigluBlock), I, I, I, P], I),
            "tl_swiglu_block_forward": ([P, ctypes.POINTER(_SwigluBlock), I, I, P], I),
            "tl_quant_gemm_workspace_size": ([I, I, I, I, I], ctypes.c_size_t),
            "tl_prefill_plan": ([P, P, P, P, I, P, P, P], I),
            "tl_quant_gemm_ws": ([P, P, P, P, P, I, I, I, I, I, P, ctypes.c_size_t, P], I),
            "tl_quant_gemm_swiglu_ws": ([P, P, P, P, P, I, I, I, I, I, P, ctypes.c_size_t, P], I),
            "tl_loop_block_to_int2": ([ctypes.POINTER(_Block), ctypes.POINTER(_QProj), P], I),
            "tl_swiglu_block_to_int2": ([ctypes.POINTER(_SwigluBlock), ctypes.POINTER(_QProj), P], I),
            "tl_probe_read_bandwidth": ([P, ctypes.c_size_t, I, P, P], I),
            "tl_loop_block_l2_plan": ([ctypes.POINTER(_Block), I, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)], I),
        }
        for name, (args, res) in sigs.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _raise_if(st: int):
    if st != TLQ_OK:
        raise TLQError(st, load().tl_last_error().decode(errors="replace"))


def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtype, name):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtype:
        raise ValueError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def tl_last_error() -> str:
    return load().tl_last_error().decode(errors="replace")


def tl_version() -> str:
    return load().tl_version().decode()


def tl_quant_gemm(A, W, scales, zeros, C, bits: int, group: int, stream=None) -> None:
    """C[M][N] = fp16(A[M][K] . dequant(W)^T) on the GPU (see include/tlq.h)."""
    import torch

    M, K = A.shape
    N = W.shape[0]
    st = load().tl_quant_gemm(_dev(A, (torch.float16,), "A"), _dev(W, (torch.int32, torch.uint32), "W"),
                              _dev(scales, (torch.float16,), "scales"), _dev(zeros, (torch.float16,), "zeros"),
                              _dev(C, (torch.float16,), "C"), M, N, K, bits, group, _stream(stream))
    _raise_if(st)


def tl_quant_gemm_workspace_size(M: int, N: int, K: int, bits: int, group: int) -> int:
    """Bytes of k-split workspace the tensor-core kernel would use (0: none)."""
    return int(load().tl_quant_gemm_workspace_size(M, N, K, bits, group))


def tl_prefill_plan(shapes, ws_bytes=None, device=None):
    """[(token tiles per CTA, k split)] the library would launch for the
    (M, N, K) problems in ``shapes`` ((0, 0): the decode kernel); several
    problems with M > 16 (up to four) are planned jointly, as a batched call
    runs them.  ``ws_bytes``: the workspace bytes each is given (default 0);
    ``device``: None for the current device, or (sms, clusters with one token
    tile for k splits 1/2/4/8, the same with two) -- then no CUDA call is made."""
    n = len(shapes)
    arr = lambda t, vals: (t * n)(*vals)  # noqa: E731
    Ms = arr(ctypes.c_int, [s[0] for s in shapes])
    Ns = arr(ctypes.c_int, [s[1] for s in shapes])
    Ks = arr(ctypes.c_int, [s[2] for s in shapes])
    ws = arr(ctypes.c_size_t, list(ws_bytes) if ws_bytes is not None else [0] * n)
    dev = None
    if device is not None:
        sms, one, two = device
        dev = (ctypes.c_int * 9)(sms, *one, *two)
    nmt = (ctypes.c_int * n)()
    ks = (ctypes.c_int * n)()
    _raise_if(load().tl_prefill_plan(Ms, Ns, Ks, ws, n, dev, nmt, ks))
    return [(nmt[i], ks[i]) for i in range(n)]


def gemm_workspace(M: int, N: int, K: int, bits: int, group: int, device="cuda"):
    """A caller-owned workspace tensor for one problem (None when the kernel
    would not split K); torch allocates it, the library never does."""
    import torch

    n = tl_quant_gemm_workspace_size(M, N, K, bits, group)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def tl_quant_gemm_ws(A, W, scales, zeros, C, bits: int, group: int, workspace=None, stream=None) -> None:
    """tl_quant_gemm with a caller-owned k-split workspace (uint8 CUDA tensor or None)."""
    import torch

    M, K = A.shape
    N = W.shape[0]
    ws = _dev(workspace, (torch.uint8,), "workspace") if workspace is not None else None
    nb = workspace.numel() if workspace is not None else 0
    st = load().tl_quant_gemm_ws(_dev(A, (torch.float16,), "A"), _dev(W, (torch.int32, torch.uint32), "W"),
                                 _dev(scales, (torch.float16,), "scales"), _dev(zeros, (torch.float16,), "zeros"),
                                 _dev(C, (torch.float16,), "C"), M, N, K, bits, group, ws, nb, _stream(stream))
    _raise_if(st)


def gemm_descs(problems):
    """ctypes descriptor array for tl_quant_gemm_batched from
    (A, W, scales, zeros, C, bits, group[, workspace[, ldw]]) tuples of CUDA
    tensors (workspace: a uint8 tensor or None; ldw: the weight's row stride
    in words, 0 = compact); build it once and reuse it to keep per-call host
    work small (the tuples' tensors must stay alive as long as it is used)."""
    import torch

    arr = (_GemmDesc * len(problems))()
    for i, prob in enumerate(problems):
        A, W, s, z, C, bits, group = prob[:7]
        ws = prob[7] if len(prob) > 7 else None
        ldw = prob[8] if len(prob) > 8 else 0
        M, K = A.shape
        arr[i] = _GemmDesc(_dev(A, (torch.float16,), "A"), _dev(W, (torch.int32, torch.uint32), "W"),
                           _dev(s, (torch.float16,), "scales"), _dev(z, (torch.float16,), "zeros"),
                           _dev(C, (torch.float16,), "C"), M, W.shape[0], K, bits, group, ldw,
                           _dev(ws, (torch.uint8,), "workspace") if ws is not None else None,
                           ws.numel() if ws is not None else 0)
    return arr


def tl_quant_gemm_batched(descs, stream=None) -> None:
    """Run independent quant_gemm problems in as few launches as possible;
    ``descs`` is a list of (A, W, scales, zeros, C, bits, group) tuples or the
    array gemm_descs() returns.  Problems with M > 16 run side by side on the
    library's side streams for ``stream``, joined back before later work on
    ``stream``; capture a graph on a stream that has made one call outside
    capture to keep that in the graph."""
    if not isinstance(descs, ctypes.Array):
        descs = gemm_descs(descs)
    _raise_if(load().tl_quant_gemm_batched(descs, len(descs), _stream(stream)))


def tl_quant_gemm_batched_host(descs, hostA, devA, hostC, devC, stream=None) -> None:
    """The batched call on host buffers: hostA (CPU tensor, pinned) -> devA,
    the GEMMs, devC -> hostC (CPU tensor, pinned), in order on `stream`.
    Every descriptor's A / C must be a view into devA / devC."""
    import torch

    for t, name, cuda in ((hostA, "hostA", False), (hostC, "hostC", False), (devA, "devA", True), (devC, "devC", True)):
        if not isinstance(t, torch.Tensor) or t.is_cuda != cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor" % (name, "CUDA" if cuda else "host"))
    if hostA.numel() * hostA.element_size() != devA.numel() * devA.element_size() or \
            hostC.numel() * hostC.element_size() != devC.numel() * devC.element_size():
        raise ValueError("host and device buffers must have the same sizes")
    if not isinstance(descs, ctypes.Array):
        descs = gemm_descs(descs)
    _raise_if(load().tl_quant_gemm_batched_host(descs, len(descs), hostA.data_ptr(), devA.data_ptr(),
                                                devA.numel() * devA.element_size(), hostC.data_ptr(),
                                                devC.data_ptr(), devC.numel() * devC.element_size(),
                                                _stream(stream)))


def tl_pack_weights(codes, W, bits: int, stream=None) -> None:
    import torch

    N, K = codes.shape
    _raise_if(load().tl_pack_weights(_dev(codes, (torch.uint8,), "codes"), _dev(W, (torch.int32, torch.uint32), "W"),
                                     N, K, bits, _stream(stream)))


def tl_unpack_weights(W, codes, bits: int, stream=None) -> None:
    import torch

    N, K = codes.shape
    _raise_if(load().tl_unpack_weights(_dev(W, (torch.int32, torch.uint32), "W"), _dev(codes, (torch.uint8,), "codes"),
                                       N, K, bits, _stream(stream)))


def tl_requant_int4_to_int2(W4, s4, z4, W2, s2, z2, group: int, stream=None) -> None:
    import torch

    N = W4.shape[0]
    K = W4.shape[1] * 8
    i32 = (torch.int32, torch.uint32)
    _raise_if(load().tl_requant_int4_to_int2(_dev(W4, i32, "W4"), _dev(s4, (torch.float16,), "s4"),
                                             _dev(z4, (torch.float16,), "z4"), _dev(W2, i32, "W2"),
                                             _dev(s2, (torch.float16,), "s2"), _dev(z2, (torch.float16,), "z2"),
                                             N, K, group, _stream(stream)))


def tl_quant_gemm_swiglu(A, Wgu, scales, zeros, C, bits: int, group: int, stream=None, workspace=None) -> None:
    """The fused gate/up GEMM with the SwiGLU epilogue; with a workspace
    (uint8 CUDA tensor) through tl_quant_gemm_swiglu_ws."""
    import torch

    M, K = A.shape
    N2 = Wgu.shape[0]
    if tuple(C.shape) != (M, N2 // 2):
        raise ValueError("C must be [M, N2/2] = [%d, %d]" % (M, N2 // 2))
    args = (_dev(A, (torch.float16,), "A"), _dev(Wgu, (torch.int32, torch.uint32), "Wgu"),
            _dev(scales, (torch.float16,), "scales"), _dev(zeros, (torch.float16,), "zeros"),
            _dev(C, (torch.float16,), "C"), M, N2, K, bits, group)
    if workspace is None:
        _raise_if(load().tl_quant_gemm_swiglu(*args, _stream(stream)))
    else:
        _raise_if(load().tl_quant_gemm_swiglu_ws(*args, _dev(workspace, (torch.uint8,), "workspace"),
                                                 workspace.numel(), _stream(stream)))


def tl_dequant_fp16(W, scales, zeros, out, bits: int, group: int, stream=None) -> None:
    import torch

    N, K = out.shape
    if W.shape[0] != N or W.shape[1] * (32 // bits) != K:
        raise ValueError("W [%d, %d] does not hold [%d, %d] INT%d weights" % (W.shape[0], W.shape[1], N, K, bits))
    _raise_if(load().tl_dequant_fp16(_dev(W, (torch.int32, torch.uint32), "W"), _dev(scales, (torch.float16,), "scales"),
                                     _dev(zeros, (torch.float16,), "zeros"), _dev(out, (torch.float16,), "out"),
                                     N, K, bits, group, _stream(stream)))


def dequant_fp16(W, scales, zeros, bits: int, group: int, stream=None):
    """The FP16 body [N, K] of a packed weight (one rounding per weight)."""
    import torch

    out = torch.empty((W.shape[0], W.shape[1] * (32 // bits)), dtype=torch.float16, device=W.device)
    tl_dequant_fp16(W, scales, zeros, out, bits, group, stream)
    return out


def tl_interleave_rows(a, b, out, stream=None) -> None:
    """out[2i] = a[i], out[2i+1] = b[i] (row-major device tensors)."""
    for t, name in ((a, "a"), (b, "b"), (out, "out")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if a.shape != b.shape or a.dtype != b.dtype or out.dtype != a.dtype or out.shape[0] != 2 * a.shape[0] \
            or tuple(out.shape[1:]) != tuple(a.shape[1:]):
        raise ValueError("interleave_rows: a, b [rows, ...] and out [2 rows, ...] of one dtype")
    rows = a.shape[0]
    _raise_if(load().tl_interleave_rows(a.data_ptr(), b.data_ptr(), out.data_ptr(), rows,
                                        a.numel() * a.element_size() // rows, _stream(stream)))


def requant_descs(problems):
    """(W4, s4, z4, W2, s2, z2) tensor tuples -> a ctypes descriptor array."""
    import torch

    i32 = (torch.int32, torch.uint32)
    arr = (_RequantDesc * len(problems))()
    for i, (W4, s4, z4, W2, s2, z2) in enumerate(problems):
        arr[i] = _RequantDesc(_dev(W4, i32, "W4"), _dev(s4, (torch.float16,), "s4"), _dev(z4, (torch.float16,), "z4"),
                              _dev(W2, i32, "W2"), _dev(s2, (torch.float16,), "s2"), _dev(z2, (torch.float16,), "z2"),
                              W4.shape[0], W4.shape[1] * 8)
    return arr


def tl_requant_int4_to_int2_batched(descs, group: int, stream=None) -> None:
    if not isinstance(descs, ctypes.Array):
        descs = requant_descs(descs)
    _raise_if(load().tl_requant_int4_to_int2_batched(descs, len(descs), group, _stream(stream)))


def tl_loop_block_forward(x, block: "LoopBlock", L: int, stream=None) -> None:
    import torch

    M = x.shape[0]
    if M > block.max_rows:
        raise ValueError("x has %d rows, the block's scratch holds %d" % (M, block.max_rows))
    _raise_if(load().tl_loop_block_forward(_dev(x, (torch.float32,), "x"), ctypes.byref(block._c), L, M,
                                           _stream(stream)))


def _rows_for(block, M, chunk):
    rows = M if chunk <= 0 or chunk >= M else chunk
    if rows > block.max_rows:
        raise ValueError("%d rows per pass, the block's scratch holds %d" % (rows, block.max_rows))


def tl_loop_block_forward_chunked(x, block: "LoopBlock", L: int, chunk: int, stream=None) -> None:
    import torch

    _rows_for(block, x.shape[0], chunk)
    _raise_if(load().tl_loop_block_forward_chunked(_dev(x, (torch.float32,), "x"), ctypes.byref(block._c), L,
                                                   x.shape[0], chunk, _stream(stream)))


def tl_swiglu_block_forward_chunked(x, block: "SwiGLUBlock", L: int, chunk: int, stream=None) -> None:
    import torch

    _rows_for(block, x.shape[0], chunk)
    _raise_if(load().tl_swiglu_block_forward_chunked(_dev(x, (torch.float32,), "x"), ctypes.byref(block._c), L,
                                                     x.shape[0], chunk, _stream(stream)))


def tl_loop_block_forward_static_scratch(x, block: "LoopBlock", L: int, stream=None) -> None:
    """tl_loop_block_forward with the intermediates in the library's static
    device scratch (no caller buffers, no allocation); the block's own scratch
    tensors are not used."""
    import torch

    _raise_if(load().tl_loop_block_forward_static_scratch(_dev(x, (torch.float32,), "x"), ctypes.byref(block._c), L,
                                                          x.shape[0], _stream(stream)))


def tl_probe_read_bandwidth(buf, reps: int, sink, stream=None) -> None:
    """reps passes of L2-only 16-byte loads over buf (a CUDA tensor); sink is
    an int32 CUDA tensor of at least 2 * SMs * 512 elements."""
    _raise_if(load().tl_probe_read_bandwidth(buf.data_ptr(), buf.numel() * buf.element_size(), reps,
                                             sink.data_ptr(), _stream(stream)))


def tl_loop_block_l2_plan(block, L: int):
    """The block's L2 residency plan: (resident projection mask, weight
    bytes, budget bytes); bit i = projection i of (qkv, o, up / gate_up,
    down) streamed evict-last."""
    c = block._c
    if isinstance(c, _SwigluBlock):  # same plan over (qkv, o, gate_up, down)
        b = _Block()
        b.qkv, b.o, b.up, b.down, b.bits, b.group, b.D = c.qkv, c.o, c.gate_up, c.down, c.bits, c.group, c.D
        c = b
    mask, wb, bb = ctypes.c_int(), ctypes.c_size_t(), ctypes.c_size_t()
    _raise_if(load().tl_loop_block_l2_plan(ctypes.byref(c), L, ctypes.byref(mask), ctypes.byref(wb), ctypes.byref(bb)))
    return mask.value, wb.value, bb.value


def tl_check_status(stream=None) -> None:
    _raise_if(load().tl_check_status(_stream(stream)))


def tl_reset_status(stream=None) -> None:
    _raise_if(load().tl_reset_status(_stream(stream)))


def tl_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _raise_if(load().tl_selftest_wait_timeout(limit_us, _stream(stream)))


# ---------------------------------------------------------------------------
# conveniences that allocate their outputs with torch
# ---------------------------------------------------------------------------

def quant_gemm(A, W, scales, zeros, bits: int, group: int, stream=None):
    """C = A . dequant(W)^T, with the k-split workspace the kernel asks for
    (allocated here by torch)."""
    import torch

    C = torch.empty((A.shape[0], W.shape[0]), dtype=torch.float16, device=A.device)
    K = A.shape[1]
    ws = gemm_workspace(A.shape[0], W.shape[0], K, bits, group, A.device)
    tl_quant_gemm_ws(A, W, scales, zeros, C, bits, group, ws, stream)
    return C


def pack_weights(codes, bits: int, stream=None):
    import torch

    N, K = codes.shape
    W = torch.empty((N, K * bits // 32), dtype=torch.int32, device=codes.device)
    tl_pack_weights(codes, W, bits, stream)
    return W


def quant_gemm_swiglu(A, Wgu, scales, zeros, bits: int, group: int, stream=None):
    import torch

    C = torch.empty((A.shape[0], Wgu.shape[0] // 2), dtype=torch.float16, device=A.device)
    ws = gemm_workspace(A.shape[0], Wgu.shape[0], A.shape[1], bits, group, A.device)
    tl_quant_gemm_swiglu(A, Wgu, scales, zeros, C, bits, group, stream, ws)
    return C


def interleave_rows(a, b, stream=None):
    import torch

    out = torch.empty((2 * a.shape[0],) + tuple(a.shape[1:]), dtype=a.dtype, device=a.device)
    tl_interleave_rows(a, b, out, stream)
    return out


def requant_int4_to_int2(W4, s4, z4, group: int, in_place_scales: bool = False, stream=None):
    """INT4 weight -> (INT2 weight, scales, zeros), same group.  With
    in_place_scales the INT2 scales/zeros overwrite s4/z4."""
    import torch

    W2 = torch.empty((W4.shape[0], W4.shape[1] // 2), dtype=torch.int32, device=W4.device)
    s2, z2 = (s4, z4) if in_place_scales else (torch.empty_like(s4), torch.empty_like(z4))
    tl_requant_int4_to_int2(W4, s4, z4, W2, s2, z2, group, stream)
    return W2, s2, z2


def unpack_weights(W, K: int, bits: int, stream=None):
    import torch

    codes = torch.empty((W.shape[0], K), dtype=torch.uint8, device=W.device)
    tl_unpack_weights(W, codes, bits, stream)
    return codes


def _block_workspace(shapes, bits, group, max_rows, device):
    """One workspace for a block's GEMMs (they run in order): the largest any
    of them asks for at any row count up to max_rows (the planner's choice
    changes only at multiples of the 128-token tile)."""
    import torch

    ms = sorted({max_rows} | set(range(128, max_rows + 1, 128)) | ({17} if max_rows > 16 else set()))
    need = 0
    for M in ms:
        for (N, K) in shapes:
            need = max(need, tl_quant_gemm_workspace_size(M, N, K, bits, group))
    return torch.empty(need, dtype=torch.uint8, device=device) if need else None


def _sync(stream):
    import torch

    if stream is None:
        torch.cuda.current_stream().synchronize()
    elif isinstance(stream, int):
        torch.cuda.synchronize()
    else:
        stream.synchronize()


class _BlockBase:
    """Shared parts of the two loop blocks: projection descriptions, the
    FP16 scratch and the k-split workspace (all allocated here by torch)."""

    NAMES = ()
    STRUCT = None
    ACT = ""

    def _setup(self, proj, bits, group, max_rows, normalize, F_act):
        import torch

        self.proj = proj
        self.bits, self.group, self.max_rows, self.normalize = bits, group, max_rows, normalize
        cpw = 32 // bits
        self.dims = {k: (v[0].shape[0], v[0].shape[1] * cpw) for k, v in proj.items()}
        self.ldw = {k: 0 for k in proj}
        D = self.dims["o"][0]
        self.D, self.F = D, F_act
        dev = proj["o"][0].device
        self.h = torch.empty((max_rows, D), dtype=torch.float16, device=dev)
        self.qkv_out = torch.empty((max_rows, 3 * D), dtype=torch.float16, device=dev)
        self.o_out = torch.empty((max_rows, D), dtype=torch.float16, device=dev)
        self.act = torch.empty((max_rows, F_act), dtype=torch.float16, device=dev)
        self.workspace = _block_workspace(list(self.dims.values()), bits, group, max_rows, dev)
        self._bind()

    def _bind(self):
        import torch

        c = self.STRUCT()
        for name in self.NAMES:
            W, s, z = self.proj[name]
            N, K = self.dims[name]
            setattr(c, name, _QProj(_dev(W, (torch.int32, torch.uint32), name + ".W"),
                                    _dev(s, (torch.float16,), name + ".s"), _dev(z, (torch.float16,), name + ".z"),
                                    N, K, self.ldw[name]))
        c.bits, c.group, c.D = self.bits, self.group, self.D
        c.h, c.qkv_out, c.o_out = self.h.data_ptr(), self.qkv_out.data_ptr(), self.o_out.data_ptr()
        setattr(c, self.ACT, self.act.data_ptr())
        c.normalize = 1 if self.normalize else 0
        c.workspace = self.workspace.data_ptr() if self.workspace is not None else None
        c.workspace_bytes = self.workspace.numel() if self.workspace is not None else 0
        self._c = c

    def _to_int2(self, fn, in_place, stream):
        """The context-length tier switch through the C ABI ("beta-Informed
        Deployment Features", CTX-TIER, Phase 2 / 2b): one launch re-quantizes
        every INT4 weight, the library rewrites the block description to INT2.
        Out of place (default) the INT2 rows are compact new buffers and the
        INT4 words are released once the stream has passed the conversion;
        in place the INT2 rows overwrite the INT4 words at the INT4 row stride.
        Scales and zeros are converted in place either way.  One way; the
        group size is kept."""
        import torch

        if self.bits != 4:
            raise ValueError("to_int2 needs an INT4 block (bits=%d)" % self.bits)
        new = {}
        dst = None
        if not in_place:
            dst = (_QProj * 4)()
            for i, name in enumerate(self.NAMES):
                W4, s4, z4 = self.proj[name]
                N, K = self.dims[name]
                W2 = torch.empty((N, K // 16), dtype=torch.int32, device=W4.device)
                new[name] = (W2, s4, z4)
                dst[i] = _QProj(W2.data_ptr(), s4.data_ptr(), z4.data_ptr(), N, K, 0)
        _raise_if(fn(ctypes.byref(self._c), dst, _stream(stream)))
        _sync(stream)  # the INT4 words may go back to the allocator now
        for name in self.NAMES:
            self.ldw[name] = getattr(self._c, name).ldw
        if not in_place:
            self.proj = new
        self.bits = 2
        self._bind()
        return self


class LoopBlock(_BlockBase):
    """The shared-weight loop block: four packed projections plus FP16 scratch
    and the k-split workspace.

    ``proj`` maps "qkv", "o", "up", "down" to (W packed int32, scales, zeros)
    CUDA tensors; scratch for up to ``max_rows`` rows is allocated here."""

    NAMES = ("qkv", "o", "up", "down")
    STRUCT = _Block
    ACT = "up_out"

    def __init__(self, proj: dict, bits: int, group: int, max_rows: int, normalize: bool = True):
        self._setup(proj, bits, group, max_rows, normalize, proj["up"][0].shape[0])

    @property
    def up_out(self):
        return self.act

    def to_int2(self, stream=None, in_place: bool = False):
        """The tier switch (tl_loop_block_to_int2)."""
        return self._to_int2(load().tl_loop_block_to_int2, in_place, stream)

    def forward(self, x, L: int, stream=None, chunk: int = 0):
        """L iterations on x in place; chunk > 0 runs chunked prefill."""
        if chunk > 0:
            tl_loop_block_forward_chunked(x, self, L, chunk, stream)
        else:
            tl_loop_block_forward(x, self, L, stream)
        return x


class SwiGLUBlock(_BlockBase):
    """The five-weight SwiGLU loop block (attn_qkv, attn_out, mlp_gate,
    mlp_up, mlp_down).

    ``proj`` maps "qkv", "o", "gate", "up", "down" to (W packed int32,
    scales, zeros) CUDA tensors.  The gate and up weights are interleaved row
    by row into one [2F, ...] weight for the fused GEMM (tl_interleave_rows);
    scratch for up to ``max_rows`` rows is allocated here."""

    NAMES = ("qkv", "o", "gate_up", "down")
    STRUCT = _SwigluBlock
    ACT = "act_out"

    def __init__(self, proj: dict, bits: int, group: int, max_rows: int, normalize: bool = True, stream=None):
        gate, up = proj["gate"], proj["up"]
        gate_up = tuple(interleave_rows(g, u, stream) for g, u in zip(gate, up))
        fused = {"qkv": proj["qkv"], "o": proj["o"], "gate_up": gate_up, "down": proj["down"]}
        self._setup(fused, bits, group, max_rows, normalize, gate[0].shape[0])

    @property
    def act_out(self):
        return self.act

    def to_int2(self, stream=None, in_place: bool = False):
        """The tier switch for the five weights (tl_swiglu_block_to_int2; the
        fused gate/up weight re-quantizes row by row like the two it holds)."""
        return self._to_int2(load().tl_swiglu_block_to_int2, in_place, stream)

    def forward(self, x, L: int, stream=None, chunk: int = 0):
        """L iterations on x in place; chunk > 0 runs chunked prefill."""
        import torch

        M = x.shape[0]
        if chunk > 0:
            tl_swiglu_block_forward_chunked(x, self, L, chunk, stream)
            return x
        if M > self.max_rows:
            raise ValueError("x has %d rows, the block's scratch holds %d" % (M, self.max_rows))
        _raise_if(load().tl_swiglu_block_forward(_dev(x, (torch.float32,), "x"), ctypes.byref(self._c), L, M,
                                                 _stream(stream)))
        return x

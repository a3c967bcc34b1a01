"""CPU oracle for the weight-only quantized linear layer (test infrastructure).

This package is the plain, slow, obviously correct statement of what the GPU
library computes: unpack, dequantize exactly, accumulate in binary64 in plain
k order, round once to FP16.  It is test infrastructure: only the tests, the
package smoke check and the CPU-baseline leg of the benchmark use it.  The
product path never imports it, and it imports nothing from the product.

The arithmetic lives in ``tlq_oracle.c`` (plain C, compiled here with gcc);
this module only marshals numpy arrays.  Each function cites the documentation
passage it follows in the C file's header and in its own docstring.

Parity status of each function (what pins it, in ``tests/test_oracle.py``):
  half_to_double / double_to_half  exhaustive / randomized against numpy's
                                   IEEE binary16 conversion
  pack / unpack                    hand-written words, byte-layout restatement,
                                   round trip
  dequant                          exact rational arithmetic on every group
  dequant_half                     exact rational value rounded by an
                                   independent RNE search, closed forms
  quant_gemm                       exact rational sum rounded once (brute force),
                                   closed forms, torch binary64 matmul
  quant_gemm_points                equality with quant_gemm
  rms_norm_half                    closed forms (constant rows, scale invariance),
                                   exact rational values where eps matters
  loop_block                       brute force on tiny shapes, closed form
                                   (zero update), split-iteration invariant
  swiglu                           closed forms (g = 0, u = 0, large |g|),
                                   the identity silu(g) - silu(-g) = g,
                                   agreement with scipy's logistic function
  loop_block_swiglu                closed form (zero gate or zero up: no
                                   update), reduction to the bilinear block
                                   g * u when the gate output is large,
                                   split-iteration invariant
  requant_int4_to_int2             closed forms (a 4-level group, a constant
                                   group), per-weight error bound, and the
                                   page's test: error within 2x of direct
                                   binary32 -> INT2 rounding
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tlq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-5  # RMS-norm epsilon of the loop block


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA) and return the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-fopenmp", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_half_to_double.restype = ctypes.c_double
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_double_to_half.restype = ctypes.c_uint16
            lib.orc_double_to_half.argtypes = [ctypes.c_double]
            for name, args in {
                "orc_pack": [P, P, I, I, I],
                "orc_unpack": [P, P, I, I, I],
                "orc_dequant": [P, P, P, I, I, I, I, P],
                "orc_dequant_half": [P, P, P, I, I, I, I, P],
                "orc_quant_gemm": [P, I, P, P, P, P, I, I, I, I, I, I],
                "orc_quant_gemm_points": [P, I, P, P, P, I, I, I, I, I, P, P, I, P],
                "orc_rms_norm_half": [P, I, I, ctypes.c_double, P],
                "orc_loop_block": [P, I, I, I, P, P, P, P, I, I, I, I, ctypes.c_double],
                "orc_requant_int4_to_int2": [P, P, P, I, I, I, P, P, P],
                "orc_swiglu": [P, P, P, ctypes.c_size_t],
                "orc_loop_block_swiglu": [P, I, I, I, P, P, P, P, P, I, I, I, I, ctypes.c_double],
                "orc_set_threads": [I],
            }.items():
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _half_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (rc=%d)" % (what, rc))


def set_threads(n: int) -> int:
    """Host threads the GEMM's output rows are shared over (1 = single
    thread); 0 keeps the current count.  Returns the count in effect.  The
    results do not depend on it: every output is the same k-order sum."""
    return _load().orc_set_threads(int(n))


# ----------------------------------------------------------------------------
# FP16 conversions (IEEE-754 binary16, round to nearest even)
# ----------------------------------------------------------------------------

def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits) & 0xFFFF)


def double_to_half(x: float) -> int:
    return int(_load().orc_double_to_half(float(x)))


# ----------------------------------------------------------------------------
# Packing: "four INT2 codes are packed per byte", rows of K/2 (INT4) or K/4
# (INT2) bytes -- beta-Informed Deployment Features, CTX-TIER, "Details of the
# shipped kernel".  LSB-first within each 32-bit word (a reading of this library).
# ----------------------------------------------------------------------------

def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    out = np.empty((N, K * bits // 32), dtype=np.uint32)
    _check(_load().orc_pack(_ptr(codes), _ptr(out), N, K, bits), "pack")
    return out


def unpack(words: np.ndarray, K: int, bits: int) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    N = words.shape[0]
    assert words.shape[1] * 32 // bits == K
    out = np.empty((N, K), dtype=np.uint8)
    _check(_load().orc_unpack(_ptr(words), _ptr(out), N, K, bits), "unpack")
    return out


# ----------------------------------------------------------------------------
# Dequantization and the GEMM: "INT2 / INT4 packed data + FP16 scales + FP16
# zeros per quantized layer" -- Model, "VRAM cost", Weights.
# ----------------------------------------------------------------------------

def dequant(W: np.ndarray, scales, zeros, K: int, bits: int, group: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint32)
    s, z = _half_bits(scales), _half_bits(zeros)
    N = W.shape[0]
    out = np.empty((N, K), dtype=np.float64)
    _check(_load().orc_dequant(_ptr(W), _ptr(s), _ptr(z), N, K, bits, group, _ptr(out)), "dequant")
    return out


def dequant_half(W: np.ndarray, scales, zeros, K: int, bits: int, group: int) -> np.ndarray:
    """FP16 body of a packed weight: fp16_RNE((q - z) * s) per weight, +0 for
    exact zeros ("Model", "VRAM cost": the FP16 body cache)."""
    W = np.ascontiguousarray(W, dtype=np.uint32)
    s, z = _half_bits(scales), _half_bits(zeros)
    N = W.shape[0]
    out = np.empty((N, K), dtype=np.uint16)
    _check(_load().orc_dequant_half(_ptr(W), _ptr(s), _ptr(z), N, K, bits, group, _ptr(out)), "dequant_half")
    return out.view(np.float16)


def quant_gemm(A, W: np.ndarray, scales, zeros, bits: int, group: int, K: int | None = None) -> np.ndarray:
    """C = fp16(A . dequant(W)^T); A is FP16 [M][K]; returns FP16 [M][N]."""
    A = _half_bits(A)
    W = np.ascontiguousarray(W, dtype=np.uint32)
    s, z = _half_bits(scales), _half_bits(zeros)
    M, Ka = A.shape
    K = Ka if K is None else K
    N = W.shape[0]
    C = np.empty((M, N), dtype=np.uint16)
    _check(_load().orc_quant_gemm(_ptr(A), Ka, _ptr(W), _ptr(s), _ptr(z), _ptr(C), N,
                                  M, N, K, bits, group), "quant_gemm")
    return C.view(np.float16)


def quant_gemm_points(A, W, scales, zeros, bits: int, group: int, pm, pn) -> np.ndarray:
    """The GEMM definition evaluated only at outputs (pm[i], pn[i])."""
    A = _half_bits(A)
    W = np.ascontiguousarray(W, dtype=np.uint32)
    s, z = _half_bits(scales), _half_bits(zeros)
    pm = np.ascontiguousarray(pm, dtype=np.int32)
    pn = np.ascontiguousarray(pn, dtype=np.int32)
    M, K = A.shape
    N = W.shape[0]
    out = np.empty(pm.shape[0], dtype=np.uint16)
    _check(_load().orc_quant_gemm_points(_ptr(A), K, _ptr(W), _ptr(s), _ptr(z), M, N, K, bits,
                                         group, _ptr(pm), _ptr(pn), pm.shape[0], _ptr(out)),
           "quant_gemm_points")
    return out.view(np.float16)


# ----------------------------------------------------------------------------
# Loop block: FP32 residual, FP16 scratch -- Model, "VRAM cost", Runtime
# buffers; the block is reapplied in place with shared weights -- Warm-start
# mid-loop, internal flow, "Extend loop".
# ----------------------------------------------------------------------------

def rms_norm_half(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, D = x.shape
    h = np.empty((M, D), dtype=np.uint16)
    _check(_load().orc_rms_norm_half(_ptr(x), M, D, eps, _ptr(h)), "rms_norm_half")
    return h.view(np.float16)


class _Proj(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


def loop_block(x: np.ndarray, block: dict, bits: int, group: int, L: int, normalize: bool = True,
               eps: float = EPS) -> np.ndarray:
    """Apply the shared block L times to a copy of x (FP32 [M][D]) and return it.

    ``block`` maps "qkv", "o", "up", "down" to (W packed, scales, zeros)."""
    x = np.array(x, dtype=np.float32, order="C", copy=True)
    M, D = x.shape
    F = block["up"][0].shape[0]
    keep = []
    projs = []
    for name in ("qkv", "o", "up", "down"):
        W, s, z = block[name]
        W = np.ascontiguousarray(W, dtype=np.uint32)
        s, z = _half_bits(s), _half_bits(z)
        keep += [W, s, z]
        projs.append(_Proj(_ptr(W), _ptr(s), _ptr(z)))
    rc = _load().orc_loop_block(_ptr(x), M, D, F, *[ctypes.byref(p) for p in projs], bits, group,
                                L, 1 if normalize else 0, eps)
    _check(rc, "loop_block")
    return x


# ----------------------------------------------------------------------------
# SwiGLU feed-forward of the five-weight loop block: "Model", ffn_dim (the
# width of the gate and up projections); beta-Informed Deployment Features,
# CTX-TIER, Phase 2b (attn_qkv, attn_out, mlp_gate, mlp_up, mlp_down).
# ----------------------------------------------------------------------------

def swiglu(g, u) -> np.ndarray:
    """fp16(silu(g) * u) element-wise for FP16 arrays g, u (binary64 inside)."""
    g = _half_bits(g)
    u = _half_bits(u)
    assert g.shape == u.shape
    out = np.empty(g.shape, dtype=np.uint16)
    _check(_load().orc_swiglu(_ptr(g), _ptr(u), _ptr(out), g.size), "swiglu")
    return out.view(np.float16)


def loop_block_swiglu(x: np.ndarray, block: dict, bits: int, group: int, L: int, normalize: bool = True,
                      eps: float = EPS) -> np.ndarray:
    """The five-weight SwiGLU block L times on a copy of x (FP32 [M][D]).

    ``block`` maps "qkv", "o", "gate", "up", "down" to (W packed, scales,
    zeros)."""
    x = np.array(x, dtype=np.float32, order="C", copy=True)
    M, D = x.shape
    F = block["up"][0].shape[0]
    keep = []
    projs = []
    for name in ("qkv", "o", "gate", "up", "down"):
        W, s, z = block[name]
        W = np.ascontiguousarray(W, dtype=np.uint32)
        s, z = _half_bits(s), _half_bits(z)
        keep += [W, s, z]
        projs.append(_Proj(_ptr(W), _ptr(s), _ptr(z)))
    rc = _load().orc_loop_block_swiglu(_ptr(x), M, D, F, *[ctypes.byref(p) for p in projs], bits, group,
                                       L, 1 if normalize else 0, eps)
    _check(rc, "loop_block_swiglu")
    return x


# ----------------------------------------------------------------------------
# INT4 -> INT2 group re-quantization: beta-Informed Deployment Features,
# CTX-TIER, "Details of the shipped kernel" (per group: dequantize, scale =
# (max - min) / 3, zero = min, round to nearest, four codes per byte).
# ----------------------------------------------------------------------------

def requant_int4_to_int2(W4: np.ndarray, scales, zeros, K: int, group: int):
    """INT4 packed words [N][K/8] + FP16 scales/zeros [N][K/group] ->
    (INT2 words [N][K/16], FP16 scales, FP16 zeros), group unchanged; the
    binary32 steps are listed in tlq_oracle.c."""
    W4 = np.ascontiguousarray(W4, dtype=np.uint32)
    N = W4.shape[0]
    s4 = _half_bits(scales)
    z4 = _half_bits(zeros)
    W2 = np.zeros((N, K // 16), dtype=np.uint32)
    s2 = np.zeros((N, K // group), dtype=np.uint16)
    z2 = np.zeros((N, K // group), dtype=np.uint16)
    _check(_load().orc_requant_int4_to_int2(_ptr(W4), _ptr(s4), _ptr(z4), N, K, group, _ptr(W2), _ptr(s2),
                                            _ptr(z2)), "requant_int4_to_int2")
    return W2, s2.view(np.float16), z2.view(np.float16)

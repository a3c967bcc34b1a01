"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and rounds them to the storage types
(FP16 with numpy's round-to-nearest-even, codes as uint8).  It holds none of
the layer's arithmetic: no packing, no dequantization, no GEMM.

Value distributions follow the weight-only quantized workloads of the
TinyLoop documentation at D = 2048 ("Model", config example: 2048-dim,
8192 FFN):
  INT4, group 128: codes uniform 0..15, scales U[0.005, 0.02], zeros U[6, 9]
  INT2, group 64:  codes uniform 0..3,  scales U[0.02, 0.08],  zeros U[1, 2]
  activations N(0, 1) (times 0.5 for the prefill workload), FP16
  loop-block residual x0 N(0, 1), FP32
Draw order is fixed: activations, then per projection codes, scales, zeros.
"""
from __future__ import annotations

import numpy as np

# (N, K) of the four projections of the D = 2048 loop block
D_MODEL = 2048
FFN = 8192
SHAPES = {
    "qkv": (3 * D_MODEL, D_MODEL),
    "o": (D_MODEL, D_MODEL),
    "up": (FFN, D_MODEL),
    "down": (D_MODEL, FFN),
}
PROJ_ORDER = ("qkv", "o", "up", "down")

DIST = {
    4: dict(code_hi=15, s=(0.005, 0.02), z=(6.0, 9.0), group=128),
    2: dict(code_hi=3, s=(0.02, 0.08), z=(1.0, 2.0), group=64),
}


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def quant_weights(rng: np.random.Generator, N: int, K: int, bits: int, group: int | None = None):
    """codes uint8 [N][K], scales FP16 [N][K/group], zeros FP16 [N][K/group]."""
    d = DIST[bits]
    group = d["group"] if group is None else group
    assert K % group == 0
    G = K // group
    codes = rng.integers(0, d["code_hi"] + 1, size=(N, K), dtype=np.uint8)
    scales = rng.uniform(d["s"][0], d["s"][1], size=(N, G)).astype(np.float16)
    zeros = rng.uniform(d["z"][0], d["z"][1], size=(N, G)).astype(np.float16)
    return codes, scales, zeros


def activations(rng: np.random.Generator, M: int, K: int, scale: float = 1.0) -> np.ndarray:
    return (rng.standard_normal((M, K)) * scale).astype(np.float16)


def gemm_case(M: int, N: int, K: int, bits: int, group: int | None = None, seed: int = 0,
              a_scale: float = 1.0) -> dict:
    """One quant_gemm problem: A, codes, scales, zeros (all host numpy arrays)."""
    rng = rng_for(seed)
    A = activations(rng, M, K, a_scale)
    codes, scales, zeros = quant_weights(rng, N, K, bits, group)
    return dict(A=A, codes=codes, scales=scales, zeros=zeros, M=M, N=N, K=K, bits=bits,
                group=DIST[bits]["group"] if group is None else group)


def block_case(M: int, bits: int, group: int | None = None, seed: int = 0, D: int = D_MODEL,
               F: int = FFN) -> dict:
    """One loop-block problem: x0 and the four shared projections."""
    rng = rng_for(seed)
    x0 = rng.standard_normal((M, D)).astype(np.float32)
    shapes = {"qkv": (3 * D, D), "o": (D, D), "up": (F, D), "down": (D, F)}
    proj = {}
    for name in PROJ_ORDER:
        N, K = shapes[name]
        proj[name] = quant_weights(rng, N, K, bits, group)
    return dict(x0=x0, proj=proj, M=M, D=D, F=F, bits=bits,
                group=DIST[bits]["group"] if group is None else group)


def swiglu_block_case(M: int, bits: int, group: int | None = None, seed: int = 0, D: int = D_MODEL,
                      F: int = FFN) -> dict:
    """One five-weight SwiGLU loop-block problem: x0 and the shared
    projections qkv, o, gate, up, down (same value distributions)."""
    rng = rng_for(seed)
    x0 = rng.standard_normal((M, D)).astype(np.float32)
    shapes = {"qkv": (3 * D, D), "o": (D, D), "gate": (F, D), "up": (F, D), "down": (D, F)}
    proj = {}
    for name in ("qkv", "o", "gate", "up", "down"):
        N, K = shapes[name]
        proj[name] = quant_weights(rng, N, K, bits, group)
    return dict(x0=x0, proj=proj, M=M, D=D, F=F, bits=bits,
                group=DIST[bits]["group"] if group is None else group)

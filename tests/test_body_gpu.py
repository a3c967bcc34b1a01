"""GPU parity of tl_dequant_fp16 (the FP16 body cache) against the oracle:
every FP16 weight bit for bit, then a plain FP16 GEMM on the body (cuBLAS,
the comparison point) within the GEMM tolerance of the quantized layer."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def stress_weights(rng, N, K, bits, group):
    """Scales and zeros that stress the single rounding: signed, tiny and
    subnormal, huge, zero points tiny next to the codes."""
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    s = rng.choice([1.0, -1.0], (N, G)) * rng.choice([3e-7, 1e-4, 0.0123, 0.7, 300.0, 30000.0], (N, G))
    z = rng.choice([6e-8, 1e-5, 0.37, 7.3, -11.0, 2000.0], (N, G)) * rng.uniform(0.5, 1.5, (N, G))
    return codes, s.astype(np.float16), z.astype(np.float16)


def body_gpu(lib, codes, s, z, bits, group):
    W = lib.pack_weights(dev(codes), bits)
    out = lib.dequant_fp16(W, dev(s), dev(z), bits, group)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("bits,group,N,K", [(4, 32, 64, 512), (4, 128, 37, 1024), (4, 1024, 8, 2048),
                                            (2, 64, 64, 512), (2, 128, 19, 1024), (2, 2048, 3, 2048)])
@pytest.mark.parametrize("kind", ["workload", "stress"])
def test_body_bit_exact(lib, bits, group, N, K, kind):
    rng = np.random.default_rng(N + K + bits + group)
    if kind == "workload":
        codes, s, z = synth.quant_weights(rng, N, K, bits, group)
    else:
        codes, s, z = stress_weights(rng, N, K, bits, group)
    with np.errstate(over="ignore"):
        ref = oracle.dequant_half(oracle.pack(codes, bits), s, z, K, bits, group)
    got = body_gpu(lib, codes, s, z, bits, group)
    diff = np.count_nonzero(got.view(np.uint16) != ref.view(np.uint16))
    assert diff == 0, "%d of %d FP16 weights differ" % (diff, got.size)


@pytest.mark.parametrize("proj", synth.PROJ_ORDER)
def test_body_full_size(lib, proj):
    N, K = synth.SHAPES[proj]
    codes, s, z = synth.quant_weights(synth.rng_for(70 + len(proj)), N, K, 4, 128)
    ref = oracle.dequant_half(oracle.pack(codes, 4), s, z, K, 4, 128)
    got = body_gpu(lib, codes, s, z, 4, 128)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("M", [1, 16, 128])
def test_dense_gemm_on_body_matches_quant_gemm(lib, M):
    """The comparison point computes the same layer: a cuBLAS FP16 GEMM on the
    body (FP32 accumulation) against the oracle's quantized GEMM."""
    case = synth.gemm_case(M, 1024, 2048, 4, 128, seed=M)
    W = lib.pack_weights(dev(case["codes"]), 4)
    body = lib.dequant_fp16(W, dev(case["scales"]), dev(case["zeros"]), 4, 128)
    C = torch.matmul(dev(case["A"]), body.t())
    torch.cuda.synchronize()
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], 4), case["scales"], case["zeros"], 4, 128)
    assert_close(C.cpu().numpy(), ref, "dense body M%d" % M)

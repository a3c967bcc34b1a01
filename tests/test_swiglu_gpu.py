"""GPU parity of the SwiGLU path against the oracle, through the C ABI: the
row interleave (bit-exact), the fused gate/up GEMM with the SwiGLU epilogue
(decode and tensor-core kernels, every k split and token-tile setting), and
the five-weight loop block including its INT4 -> INT2 tier switch."""
import numpy as np
import pytest

import oracle
import synth
from devmem import flush_l2
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_words(W):
    return dev(np.ascontiguousarray(W).view(np.int32))


def gate_up_case(M, F, K, bits, group, seed):
    """A, and the gate and up weights (codes, scales, zeros) drawn like one projection each."""
    rng = synth.rng_for(seed)
    A = synth.activations(rng, M, K, 0.5 if M > 16 else 1.0)
    gate = synth.quant_weights(rng, F, K, bits, group)
    up = synth.quant_weights(rng, F, K, bits, group)
    return A, gate, up


def gpu_gate_up(lib, gate, up, bits):
    """Packed gate / up weights on the device, interleaved row by row on the device."""
    g = [lib.pack_weights(dev(gate[0]), bits), dev(gate[1]), dev(gate[2])]
    u = [lib.pack_weights(dev(up[0]), bits), dev(up[1]), dev(up[2])]
    return tuple(lib.interleave_rows(a, b) for a, b in zip(g, u))


def oracle_swiglu_gemm(A, gate, up, bits, group):
    g = oracle.quant_gemm(A, oracle.pack(gate[0], bits), gate[1], gate[2], bits, group)
    u = oracle.quant_gemm(A, oracle.pack(up[0], bits), up[1], up[2], bits, group)
    return oracle.swiglu(g, u)


# ---------------------------------------------------------------------------
# row interleave: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,shape", [(np.int32, (37, 64)), (np.float16, (200, 16)), (np.uint8, (5, 3)),
                                         (np.int32, (8192, 256))])
def test_interleave_rows_bit_exact(lib, dtype, shape):
    rng = np.random.default_rng(shape[0])
    a = rng.integers(0, 1 << 15, size=shape).astype(dtype)
    b = rng.integers(0, 1 << 15, size=shape).astype(dtype)
    out = lib.interleave_rows(dev(a), dev(b)).cpu().numpy()
    ref = np.empty((2 * shape[0],) + shape[1:], dtype)
    ref[0::2], ref[1::2] = a, b
    assert np.array_equal(out.view(np.uint8), ref.view(np.uint8))


# ---------------------------------------------------------------------------
# fused gate/up GEMM + SwiGLU epilogue
# ---------------------------------------------------------------------------

GEMM_CASES = [
    # bits, group, F, K
    (4, 128, 256, 1024),
    (4, 32, 200, 512),     # ragged 256-row tile (N2 = 400)
    (2, 64, 128, 1024),
    (2, 128, 264, 2048),   # ragged tile, INT2 with group 128 (re-quantized weights)
]


@pytest.mark.parametrize("bits,group,F,K", GEMM_CASES)
@pytest.mark.parametrize("M", [1, 5, 16, 40, 128, 300])
def test_swiglu_gemm_matches_oracle(lib, bits, group, F, K, M):
    A, gate, up = gate_up_case(M, F, K, bits, group, seed=M * 31 + F + K + bits)
    W, s, z = gpu_gate_up(lib, gate, up, bits)
    C = lib.quant_gemm_swiglu(dev(A), W, s, z, bits, group)
    torch.cuda.synchronize()
    lib.tl_check_status()
    assert_close(C.cpu().numpy(), oracle_swiglu_gemm(A, gate, up, bits, group),
                 "swiglu int%d g%d M%d F%d K%d" % (bits, group, M, F, K))


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("ks,nmt", [(2, 1), (4, 1), (8, 1), (1, 2), (2, 2)])
def test_swiglu_gemm_k_splits_and_token_tiles(lib, monkeypatch, bits, ks, nmt):
    """The split-K reduction (owners write the pairs) and two token tiles per
    CTA give the same outputs as the oracle."""
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", str(ks))
    monkeypatch.setenv("TLQ_PREFILL_NMT", str(nmt))
    group = 128 if bits == 4 else 64
    A, gate, up = gate_up_case(260, 192, 2048, bits, group, seed=ks * 10 + nmt)
    W, s, z = gpu_gate_up(lib, gate, up, bits)
    C = lib.quant_gemm_swiglu(dev(A), W, s, z, bits, group)
    torch.cuda.synchronize()
    lib.tl_check_status()
    assert_close(C.cpu().numpy(), oracle_swiglu_gemm(A, gate, up, bits, group), "ks%d nmt%d" % (ks, nmt))


@pytest.mark.parametrize("M", [1, 16, 128])
def test_swiglu_gemm_full_size_sampled(lib, M):
    """D = 2048, F = 8192 (the gate/up pair of the pages' block), INT4 group
    128: whole rows (all of them up to M = 16, 16 sampled at M = 128) against
    the oracle, with the per-row bound."""
    F, K, bits, group = synth.FFN, synth.D_MODEL, 4, 128
    A, gate, up = gate_up_case(M, F, K, bits, group, seed=900 + M)
    W, s, z = gpu_gate_up(lib, gate, up, bits)
    C = lib.quant_gemm_swiglu(dev(A), W, s, z, bits, group).cpu().numpy()
    rows = sample_rows(M, 16, np.random.default_rng(M))
    g = oracle.quant_gemm(A[rows], oracle.pack(gate[0], bits), gate[1], gate[2], bits, group)
    u = oracle.quant_gemm(A[rows], oracle.pack(up[0], bits), up[1], up[2], bits, group)
    assert_close(C[rows], oracle.swiglu(g, u), "full-size swiglu M%d" % M)


def test_swiglu_gemm_rejects_bad_shapes(lib):
    A = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    W = torch.zeros((24, 32), dtype=torch.int32, device="cuda")  # N2 = 24: not a multiple of 16
    s = torch.zeros((24, 2), dtype=torch.float16, device="cuda")
    C = torch.zeros((4, 12), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.TLQError):
        lib.tl_quant_gemm_swiglu(A, W, s, s, C, 4, 128)


# ---------------------------------------------------------------------------
# five-weight loop block
# ---------------------------------------------------------------------------

def make_block(lib, case, max_rows=None):
    bits = case["bits"]
    proj, host = {}, {}
    for name, (codes, s, z) in case["proj"].items():
        proj[name] = (lib.pack_weights(dev(codes), bits), dev(s), dev(z))
        host[name] = (oracle.pack(codes, bits), s, z)
    return lib.SwiGLUBlock(proj, bits, case["group"], max_rows or case["M"]), host


def run(lib, blk, x0, L):
    x = dev(x0.copy())
    blk.forward(x, L)
    torch.cuda.synchronize()
    lib.tl_check_status()
    return x.cpu().numpy()


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("M", [1, 5, 16, 40, 128])
@pytest.mark.parametrize("L", [1, 3])
def test_swiglu_block_small_matches_oracle(lib, bits, M, L):
    case = synth.swiglu_block_case(M, bits, seed=M * 7 + L, D=256, F=512)
    blk, host = make_block(lib, case)
    got = run(lib, blk, case["x0"], L)
    ref = oracle.loop_block_swiglu(case["x0"], host, bits, case["group"], L)
    assert_close(got, ref, "swiglu block int%d M%d L%d" % (bits, M, L))


@pytest.mark.parametrize("bits", [4, 2])
def test_swiglu_block_full_width_decode(lib, bits):
    """D = 2048, F = 8192 (32 MiB of INT4 weights, the pages' loop block), M = 1, L = 4.
    The L2 is flushed first: iteration 1 reads the weights from HBM, the later
    ones from L2."""
    case = synth.swiglu_block_case(1, bits, seed=5)
    blk, host = make_block(lib, case)
    flush_l2()
    got = run(lib, blk, case["x0"], 4)
    assert_close(got, oracle.loop_block_swiglu(case["x0"], host, bits, case["group"], 4), "int%d" % bits)


def test_swiglu_block_full_width_prefill(lib):
    """D = 2048, F = 8192, M = 128 (tensor-core path), L = 2, sampled rows."""
    case = synth.swiglu_block_case(128, 4, seed=6)
    blk, host = make_block(lib, case)
    got = run(lib, blk, case["x0"], 2)
    rows = [0, 63, 127]
    ref = oracle.loop_block_swiglu(case["x0"][rows], host, 4, case["group"], 2)
    assert_close(got[rows], ref, "swiglu block M128")


def test_swiglu_block_split_invariant_and_deterministic(lib):
    case = synth.swiglu_block_case(3, 4, seed=7, D=256, F=512)
    blk, _ = make_block(lib, case)
    full = run(lib, blk, case["x0"], 5)
    again = run(lib, blk, case["x0"], 5)
    rest = run(lib, blk, run(lib, blk, case["x0"], 2), 3)
    assert np.array_equal(full.view(np.uint32), again.view(np.uint32))
    assert np.array_equal(full.view(np.uint32), rest.view(np.uint32))


@pytest.mark.parametrize("in_place", [False, True])
def test_swiglu_block_tier_switch(lib, in_place):
    """SwiGLUBlock.to_int2 (tl_swiglu_block_to_int2, out of place or in place
    with the INT4 row stride kept): all five weights re-quantized in one launch (the
    fused gate/up weight row by row); the switched block equals an INT2
    block built from the oracle's re-quantized weights bit for bit, and one
    iteration matches the oracle's INT2 block."""
    case = synth.swiglu_block_case(16, 4, seed=8, D=512, F=1024)
    blk, host = make_block(lib, case, max_rows=16)
    blk.to_int2(in_place=in_place)
    assert blk.bits == 2
    host2, proj2 = {}, {}
    for name, (W4, s, z) in host.items():
        N, KW = W4.shape
        host2[name] = oracle.requant_int4_to_int2(W4, s, z, KW * 8, case["group"])
        proj2[name] = (dev_words(host2[name][0]), dev(host2[name][1]), dev(host2[name][2]))
    ref_blk = lib.SwiGLUBlock(proj2, 2, case["group"], 16)
    for M in (1, 16):
        x = case["x0"][:M]
        a, b = run(lib, blk, x, 2), run(lib, ref_blk, x, 2)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "M%d" % M
        got = run(lib, blk, x, 1)
        assert_close(got, oracle.loop_block_swiglu(x, host2, 2, case["group"], 1), "switched M%d" % M)

"""GPU parity of tl_requant_int4_to_int2 (the context-length tier switch's
weight conversion) against the oracle: codes, scales and zeros bit for bit,
then the INT2 GEMM and loop block fed by the converted weights."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def weights(rng, N, K, group, kind):
    """INT4 codes + FP16 scales/zeros of one distribution (all finite)."""
    G = K // group
    codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    if kind == "workload":
        s = rng.uniform(0.005, 0.02, (N, G))
        z = rng.uniform(6.0, 9.0, (N, G))
    elif kind == "signed":
        s = rng.uniform(-0.05, 0.05, (N, G))
        z = rng.uniform(-20.0, 20.0, (N, G))
    elif kind == "narrow":  # a few adjacent codes per row: cmin/cmax inside the range
        codes = (rng.integers(0, 3, size=(N, K)) + rng.integers(0, 13, size=(N, 1))).astype(np.uint8)
        s = rng.uniform(-1.0, 1.0, (N, G))
        z = rng.uniform(-3.0, 18.0, (N, G))
    elif kind == "degenerate":  # zero scales of both signs, integral zeros, constant groups
        s = rng.uniform(0.01, 0.1, (N, G))
        s[::3] = 0.0
        s[1::5] = -0.0
        z = rng.integers(0, 16, (N, G)).astype(np.float64)
        codes[::2] = rng.integers(0, 16, size=(1, 1), dtype=np.uint8)
    elif kind == "extreme":  # FP16 overflow of z2 and of s2, tiny scales
        s = rng.choice([1e-4, 3e-7, 2000.0, 50000.0], size=(N, G)) * rng.uniform(0.9, 1.1, (N, G))
        z = rng.choice([-60000.0, 0.5, 60000.0], size=(N, G))
    else:
        raise ValueError(kind)
    s, z = s.astype(np.float16), z.astype(np.float16)
    assert np.all(np.isfinite(s)) and np.all(np.isfinite(z))
    return codes, s, z


def run_gpu(lib, W4, s4, z4, group, in_place=False):
    W4d, s4d, z4d = dev(W4.view(np.int32)), dev(s4), dev(z4)
    W2, s2, z2 = lib.requant_int4_to_int2(W4d, s4d, z4d, group, in_place_scales=in_place)
    torch.cuda.synchronize()
    return W2.cpu().numpy().view(np.uint32), s2.cpu().numpy(), z2.cpu().numpy()


def assert_same(got, ref, what):
    W2, s2, z2 = got
    rW, rs, rz = ref
    assert np.array_equal(W2, rW), "%s: %d code words differ" % (what, np.count_nonzero(W2 != rW))
    assert np.array_equal(s2.view(np.uint16), rs.view(np.uint16)), what + ": scales differ"
    assert np.array_equal(z2.view(np.uint16), rz.view(np.uint16)), what + ": zeros differ"


# group -> chunks of 32 codes per group: 2, 4 (the workload), 6 (not a power
# of two), 16, 32 (a full warp), 128 (lanes loop over chunks)
SHAPES = [(64, 256, 128), (37, 512, 64), (24, 1024, 128), (16, 768, 192), (9, 2048, 512), (5, 2048, 1024),
          (3, 4096, 4096), (1, 128, 128)]


@pytest.mark.parametrize("N,K,group", SHAPES)
@pytest.mark.parametrize("kind", ["workload", "signed", "narrow", "degenerate", "extreme"])
def test_requant_bit_exact(lib, N, K, group, kind):
    rng = np.random.default_rng(N * 7919 + K + group + len(kind))
    codes, s4, z4 = weights(rng, N, K, group, kind)
    W4 = oracle.pack(codes, 4)
    with np.errstate(over="ignore"):
        ref = oracle.requant_int4_to_int2(W4, s4, z4, K, group)
    assert_same(run_gpu(lib, W4, s4, z4, group), ref, "%s N%d K%d g%d" % (kind, N, K, group))


def test_requant_scales_in_place(lib):
    rng = np.random.default_rng(5)
    N, K, group = 40, 1024, 128
    codes, s4, z4 = weights(rng, N, K, group, "signed")
    W4 = oracle.pack(codes, 4)
    ref = oracle.requant_int4_to_int2(W4, s4, z4, K, group)
    assert_same(run_gpu(lib, W4, s4, z4, group, in_place=True), ref, "in place")


@pytest.mark.parametrize("proj", synth.PROJ_ORDER)
def test_requant_full_size_loop_block_weights(lib, proj):
    """Each D=2048 loop-block projection on the INT4 workload distribution,
    every code, scale and zero against the oracle."""
    N, K = synth.SHAPES[proj]
    codes, s4, z4 = synth.quant_weights(synth.rng_for(31 + len(proj)), N, K, 4, 128)
    W4 = oracle.pack(codes, 4)
    ref = oracle.requant_int4_to_int2(W4, s4, z4, K, 128)
    assert_same(run_gpu(lib, W4, s4, z4, 128), ref, proj)


@pytest.mark.parametrize("group", [64, 128, 192, 2048])
def test_requant_batched_equals_oracle(lib, group):
    """Several weights of one group size in one launch (the grid strides over
    all of them): every output against the oracle; one weight converts its
    scales and zeros in place."""
    rng = np.random.default_rng(group)
    shapes = [(40, 2 * 3 * group), (8, 4 * group), (129, 2 * group), (1, group), (16, 6 * group)]
    host, probs = [], []
    for i, (N, K) in enumerate(shapes):
        codes, s4, z4 = weights(rng, N, K, group, ["workload", "signed", "narrow", "degenerate", "extreme"][i])
        W4 = oracle.pack(codes, 4)
        with np.errstate(over="ignore"):
            host.append(oracle.requant_int4_to_int2(W4, s4, z4, K, group))
        W4d, s4d, z4d = dev(W4.view(np.int32)), dev(s4), dev(z4)
        W2 = torch.empty((N, K // 16), dtype=torch.int32, device="cuda")
        if i == 2:
            probs.append((W4d, s4d, z4d, W2, s4d, z4d))
        else:
            probs.append((W4d, s4d, z4d, W2, torch.empty_like(s4d), torch.empty_like(z4d)))
    lib.tl_requant_int4_to_int2_batched(probs, group)
    torch.cuda.synchronize()
    for i, (p, ref) in enumerate(zip(probs, host)):
        got = (p[3].cpu().numpy().view(np.uint32), p[4].cpu().numpy(), p[5].cpu().numpy())
        assert_same(got, ref, "problem %d g%d" % (i, group))


def test_requant_deterministic(lib):
    codes, s4, z4 = synth.quant_weights(synth.rng_for(3), 512, 2048, 4, 128)
    W4 = oracle.pack(codes, 4)
    a = run_gpu(lib, W4, s4, z4, 128)
    b = run_gpu(lib, W4, s4, z4, 128)
    assert_same(a, b, "repeat")


@pytest.mark.parametrize("M", [1, 16, 256])
def test_requant_then_int2_gemm(lib, M):
    """The tier switch's data path: INT4 weight -> GPU re-quantization ->
    INT2 quant_gemm, against the oracle's re-quantization and GEMM."""
    N, K, group = 1024, 2048, 128
    rng = synth.rng_for(100 + M)
    A = synth.activations(rng, M, K)
    codes, s4, z4 = synth.quant_weights(rng, N, K, 4, group)
    W4 = oracle.pack(codes, 4)
    W2r, s2r, z2r = oracle.requant_int4_to_int2(W4, s4, z4, K, group)
    W2, s2, z2 = lib.requant_int4_to_int2(dev(W4.view(np.int32)), dev(s4), dev(z4), group)
    C = lib.quant_gemm(dev(A), W2, s2, z2, 2, group)
    torch.cuda.synchronize()
    lib.tl_check_status()
    ref = oracle.quant_gemm(A, W2r, s2r, z2r, 2, group)
    assert_close(C.cpu().numpy(), ref, "requant + int2 M%d" % M)


def test_requant_error_ratio_on_gpu(lib):
    """The page's acceptance test on the GPU's output: N=64, K=256, group 128
    Gaussian weights, INT4 rounding, re-quantization; error within 2x of direct
    binary32 -> INT2 rounding (the page measured 1.000)."""
    rng = np.random.default_rng(2026)
    N, K, group = 64, 256, 128
    G = K // group
    w = rng.standard_normal((N, K)).astype(np.float32)
    wg = w.reshape(N, G, group).astype(np.float64)
    lo, hi = wg.min(axis=2), wg.max(axis=2)
    s4 = ((hi - lo) / 15).astype(np.float16)
    z4 = (-lo / s4.astype(np.float64)).astype(np.float16)
    q4 = np.clip(np.rint(wg / s4.astype(np.float64)[..., None] + z4.astype(np.float64)[..., None]), 0, 15)
    W4 = oracle.pack(q4.reshape(N, K).astype(np.uint8), 4)
    W2, s2, z2 = run_gpu(lib, W4, s4, z4, group)
    err_rq = np.linalg.norm(oracle.dequant(W2, s2, z2, K, 2, group) - w.astype(np.float64))
    sc = (hi - lo) / 3
    q2d = np.clip(np.rint((wg - lo[..., None]) / sc[..., None]), 0, 3)
    err_direct = np.linalg.norm((lo[..., None] + q2d * sc[..., None]).reshape(N, K) - w.astype(np.float64))
    assert err_rq / err_direct <= 2.0


def test_loop_block_tier_switch(lib):
    """LoopBlock.to_int2: the INT4 block re-quantized in place of its scales,
    INT4 words released, later forwards on the INT2 kernels; against the
    oracle's re-quantization and loop block.  Full D=2048 width: M=1 (decode)
    and M=128 (tensor-core path, sampled rows) after the switch."""
    case = synth.block_case(128, 4, seed=77)
    proj, host2 = {}, {}
    for name, (codes, s, z) in case["proj"].items():
        W4 = oracle.pack(codes, 4)
        proj[name] = (dev(W4.view(np.int32)), dev(s), dev(z))
        N, K = codes.shape
        host2[name] = oracle.requant_int4_to_int2(W4, s, z, K, case["group"])
    blk = lib.LoopBlock(proj, 4, case["group"], 128)
    before = {name: proj[name][0].data_ptr() for name in proj}
    del proj
    blk.to_int2()
    assert blk.bits == 2
    for name in host2:
        assert blk.proj[name][0].data_ptr() != before[name]
        assert_same((blk.proj[name][0].cpu().numpy().view(np.uint32), blk.proj[name][1].cpu().numpy(),
                     blk.proj[name][2].cpu().numpy()), host2[name], name)
    # the switched block is the INT2 block of the oracle's weights, bit for bit
    ref_blk = lib.LoopBlock({name: tuple(dev(a.view(np.int32) if a.dtype == np.uint32 else a) for a in host2[name])
                             for name in host2}, 2, case["group"], 128)
    for M, rows in ((1, [0]), (128, [0, 77, 127])):
        for L in (1, 2):
            x = dev(case["x0"][:M].copy())
            y = x.clone()
            blk.forward(x, L)
            ref_blk.forward(y, L)
            torch.cuda.synchronize()
            lib.tl_check_status()
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), "M%d L%d" % (M, L)
        # one iteration against the oracle (C-6 holds per GEMM; longer chains of FP16-rounded
        # intermediates are covered by the loop-block tests)
        x = dev(case["x0"][:M].copy())
        blk.forward(x, 1)
        torch.cuda.synchronize()
        ref = oracle.loop_block(case["x0"][rows], host2, 2, case["group"], 1)
        assert_close(x.cpu().numpy()[rows], ref, "tier-switched block M%d" % M)
    with pytest.raises(ValueError):
        blk.to_int2()


def test_requant_argument_errors(lib):
    W4 = torch.zeros((8, 32), dtype=torch.int32, device="cuda")
    s = torch.zeros((8, 2), dtype=torch.float16, device="cuda")
    W2 = torch.zeros((8, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.TLQError):
        lib.tl_requant_int4_to_int2(W4, s, s.clone(), W2, s.clone(), s.clone(), 96)  # not a multiple of 64
    with pytest.raises(lib.TLQError):  # W2 inside W4 without being it (W2 == W4 is the in-place mode)
        lib.tl_requant_int4_to_int2(W4, s, s.clone(), W4.view(-1)[4:132].view(8, 16), s.clone(), s.clone(), 128)
    zs = s.clone()
    with pytest.raises(lib.TLQError):  # s2 overlapping z4 without being it
        lib.tl_requant_int4_to_int2(W4, s, zs, W2, zs, s.clone(), 128)


# ---------------------------------------------------------------------------
# in place ("Details of the shipped kernel", storage reuse): W2 == W4, the
# INT2 rows keep the INT4 row stride of K/8 words
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,group", [(64, 256, 128), (37, 512, 64), (16, 768, 192), (5, 2048, 1024),
                                       (3, 4096, 4096), (300, 8192, 128)])
@pytest.mark.parametrize("kind", ["workload", "signed", "degenerate"])
def test_requant_in_place_bit_exact(lib, N, K, group, kind):
    """Through a strided view: the first K/16 words of every INT4-stride row
    are the oracle's compact INT2 row bit for bit, the rest of the row is the
    INT4 words it held, and the scales/zeros (converted in place) match."""
    rng = np.random.default_rng(N + K + group + len(kind))
    codes, s4, z4 = weights(rng, N, K, group, kind)
    W4 = oracle.pack(codes, 4)
    with np.errstate(over="ignore"):
        rW, rs, rz = oracle.requant_int4_to_int2(W4, s4, z4, K, group)
    Wd, sd, zd = dev(W4.view(np.int32)), dev(s4), dev(z4)
    lib.tl_requant_int4_to_int2(Wd, sd, zd, Wd, sd, zd, group)
    torch.cuda.synchronize()
    got = Wd.cpu().numpy().view(np.uint32)
    assert np.array_equal(got[:, :K // 16], rW), "%s: %d words differ" % (kind, np.count_nonzero(got[:, :K // 16] != rW))
    assert np.array_equal(got[:, K // 16:], W4[:, K // 16:])
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), rs.view(np.uint16))
    assert np.array_equal(zd.cpu().numpy().view(np.uint16), rz.view(np.uint16))


@pytest.mark.parametrize("M", [1, 16, 256])
def test_int2_gemm_on_in_place_weights(lib, M):
    """The INT2 GEMM reads an in-place converted weight with its INT4 row
    stride (ldw = K/8): same bits as on a compact copy, and the oracle's GEMM
    on the oracle's re-quantization within the GEMM bar."""
    N, K, group = 1024, 2048, 128
    rng = synth.rng_for(300 + M)
    A = synth.activations(rng, M, K, 0.5 if M > 16 else 1.0)
    codes, s4, z4 = synth.quant_weights(rng, N, K, 4, group)
    W4 = oracle.pack(codes, 4)
    W2r, s2r, z2r = oracle.requant_int4_to_int2(W4, s4, z4, K, group)
    Wd, sd, zd = dev(W4.view(np.int32)), dev(s4), dev(z4)
    lib.tl_requant_int4_to_int2(Wd, sd, zd, Wd, sd, zd, group)
    Ad = dev(A)
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C2 = torch.empty_like(C)
    ws = lib.gemm_workspace(M, N, K, 2, group)
    compact = Wd[:, :K // 16].contiguous()
    lib.tl_quant_gemm_batched([(Ad, Wd, sd, zd, C, 2, group, ws, K // 8)])
    lib.tl_quant_gemm_batched([(Ad, compact, sd, zd, C2, 2, group, ws, 0)])
    torch.cuda.synchronize()
    lib.tl_check_status()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    assert_close(C.cpu().numpy(), oracle.quant_gemm(A, W2r, s2r, z2r, 2, group), "in-place int2 M%d" % M)


@pytest.mark.parametrize("in_place", [False, True])
def test_loop_block_tier_switch_through_c_abi(lib, in_place):
    """tl_loop_block_to_int2 (LoopBlock.to_int2): out of place the weights
    move to new compact buffers, in place they stay where they were with
    ldw = K/8; either way the switched block runs bit for bit like an INT2
    block built from the oracle's re-quantized weights."""
    case = synth.block_case(16, 4, seed=78, D=512, F=1024)
    proj, host2 = {}, {}
    for name, (codes, s, z) in case["proj"].items():
        W4 = oracle.pack(codes, 4)
        proj[name] = (dev(W4.view(np.int32)), dev(s), dev(z))
        N, K = codes.shape
        host2[name] = oracle.requant_int4_to_int2(W4, s, z, K, case["group"])
    blk = lib.LoopBlock(proj, 4, case["group"], 16)
    before = {name: proj[name][0].data_ptr() for name in proj}
    blk.to_int2(in_place=in_place)
    assert blk.bits == 2 and blk._c.bits == 2
    for name in host2:
        N, K = blk.dims[name]
        moved = blk.proj[name][0].data_ptr() != before[name]
        assert moved != in_place
        assert blk.ldw[name] == (K // 8 if in_place else 0) == getattr(blk._c, name).ldw
        words = blk.proj[name][0].cpu().numpy().view(np.uint32)[:, :K // 16]
        assert np.array_equal(words, host2[name][0]), name
    ref_blk = lib.LoopBlock({name: tuple(dev(a.view(np.int32) if a.dtype == np.uint32 else a) for a in host2[name])
                             for name in host2}, 2, case["group"], 16)
    for M in (1, 16):
        x = dev(case["x0"][:M].copy())
        y = x.clone()
        blk.forward(x, 3)
        ref_blk.forward(y, 3)
        torch.cuda.synchronize()
        lib.tl_check_status()
        assert torch.equal(x.view(torch.int32), y.view(torch.int32)), "M%d" % M

"""GPU parity of tl_pack_weights / tl_unpack_weights / tl_quant_gemm against
the CPU oracle, through the C ABI (Python binding = argument marshalling)."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_pack(lib, codes, bits):
    return lib.pack_weights(dev(codes), bits)


def run_case(lib, case):
    bits, group = case["bits"], case["group"]
    Wd = gpu_pack(lib, case["codes"], bits)
    C = lib.quant_gemm(dev(case["A"]), Wd, dev(case["scales"]), dev(case["zeros"]), bits, group)
    torch.cuda.synchronize()
    lib.tl_check_status()
    return Wd, C.cpu().numpy()


# ---------------------------------------------------------------------------
# packing: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("N,K", [(1, 64), (37, 256), (640, 2048), (3, 8192)])
def test_pack_unpack_bit_exact(lib, bits, N, K):
    rng = np.random.default_rng(N * 131 + K + bits)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)  # high bits must be dropped
    W = gpu_pack(lib, codes, bits)
    ref = oracle.pack(codes, bits)
    assert np.array_equal(W.cpu().numpy().view(np.uint32), ref)
    back = lib.unpack_weights(W, K, bits).cpu().numpy()
    assert np.array_equal(back, oracle.unpack(ref, K, bits))


# ---------------------------------------------------------------------------
# decode path (M <= 16): element-wise against the oracle on small shapes that
# still span several tiles, k-splits and a ragged row tile
# ---------------------------------------------------------------------------

DECODE_SHAPES = [
    # bits, group, N, K
    (4, 128, 256, 1024),
    (4, 128, 200, 2048),
    (4, 32, 96, 512),
    (4, 64, 136, 384),
    (4, 512, 64, 1024),
    (4, 4096, 64, 4096),   # one scale per row
    (2, 64, 256, 1024),
    (2, 128, 120, 2048),
    (2, 64, 72, 448),
    (2, 2048, 64, 2048),   # one scale per row
]


@pytest.mark.parametrize("bits,group,N,K", DECODE_SHAPES)
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_decode_matches_oracle(lib, bits, group, N, K, M):
    case = synth.gemm_case(M, N, K, bits, group, seed=M * 1000 + N + K)
    _, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "int%d g%d M%d N%d K%d" % (bits, group, M, N, K))


@pytest.mark.parametrize("bits,group,G_ok,G_bad", [(4, 32, 168, 176), (2, 64, 168, 176)])
def test_decode_largest_groups_per_row(lib, monkeypatch, bits, group, G_ok, G_bad):
    """The decode kernel stages a unit's scales and zeros in shared memory, so
    K/group has a ceiling (64-row units, two token tiles: 168 groups per row).
    At the ceiling the result matches the oracle; one step above it the call
    is refused on the host with TLQ_EUNSUPPORTED before anything is launched."""
    monkeypatch.setenv("TLQ_DECODE_ROWS", "64")
    M, N = 16, 128
    case = synth.gemm_case(M, N, group * G_ok, bits, group, seed=G_ok + bits)
    _, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "int%d g%d K%d" % (bits, group, group * G_ok))
    K = group * G_bad
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    W = torch.zeros((N, K * bits // 32), dtype=torch.int32, device="cuda")
    s = torch.ones((N, G_bad), dtype=torch.float16, device="cuda")
    z = torch.zeros((N, G_bad), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.TLQError) as e:
        lib.quant_gemm(A, W, s, z, bits, group)
    assert e.value.status == lib.TLQ_EUNSUPPORTED
    torch.cuda.synchronize()
    lib.tl_check_status()


@pytest.mark.parametrize("M", [2, 5, 7, 12, 15])
def test_decode_other_token_counts(lib, M):
    case = synth.gemm_case(M, 512, 2048, 4, 128, seed=M)
    _, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], 4), case["scales"], case["zeros"], 4, 128)
    assert_close(C, ref, "M%d" % M)


def test_decode_closed_form_zero(lib):
    """codes 8 with integer zero point 8: every output is 0 up to the FP32
    cancellation of the kernel's offset terms (sum_k a_k (base_k + q_k) minus
    its correction sums, |.| ~ 1024 * sum|a| * 2^-24 * s per set), far below
    the 1e-2 * |row| bound that random weights give (|C| ~ 3 here)."""
    M, N, K = 4, 256, 1024
    rng = synth.rng_for(3)
    A = synth.activations(rng, M, K)
    codes = np.full((N, K), 8, np.uint8)
    s = rng.uniform(0.005, 0.02, (N, K // 128)).astype(np.float16)
    z = np.full((N, K // 128), 8.0, np.float16)
    C = lib.quant_gemm(dev(A), gpu_pack(lib, codes, 4), dev(s), dev(z), 4, 128).cpu().numpy()
    assert np.max(np.abs(C.astype(np.float32))) < 1e-3


def test_decode_deterministic(lib):
    case = synth.gemm_case(16, 2048, 8192, 4, 128, seed=7)
    Wd = gpu_pack(lib, case["codes"], 4)
    A, s, z = dev(case["A"]), dev(case["scales"]), dev(case["zeros"])
    c1 = lib.quant_gemm(A, Wd, s, z, 4, 128)
    c2 = lib.quant_gemm(A, Wd, s, z, 4, 128)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("bits,group,N,K", [(4, 128, 200, 2048), (4, 32, 96, 512), (4, 64, 136, 384),
                                            (2, 64, 72, 448), (2, 128, 120, 2048), (4, 128, 64, 8192)])
@pytest.mark.parametrize("M", [1, 9, 16])
def test_decode_unit_heights_bitwise(lib, monkeypatch, bits, group, N, K, M):
    """Units of 16, 32 and 64 weight rows (TLQ_DECODE_ROWS) give the same
    bits, ragged last units included: a row's sums do not depend on the rows
    that share its unit.  The oracle agrees with all of them."""
    case = synth.gemm_case(M, N, K, bits, group, seed=M + N + K)
    outs = {}
    for rows in ("16", "32", "64"):
        monkeypatch.setenv("TLQ_DECODE_ROWS", rows)
        _, outs[rows] = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(outs["16"], ref, "16-row units int%d g%d M%d N%d K%d" % (bits, group, M, N, K))
    for rows in ("32", "64"):
        assert np.array_equal(outs[rows].view(np.uint16), outs["16"].view(np.uint16)), rows


@pytest.mark.parametrize("bits,group,N,K", [(4, 128, 200, 2048), (4, 256, 96, 1024), (4, 512, 64, 8192),
                                            (4, 128, 2048, 8192), (2, 64, 136, 2048), (2, 128, 72, 768),
                                            (2, 64, 2048, 8192)])
@pytest.mark.parametrize("M", [1, 9, 16])
def test_decode_fixed_forms_bitwise(lib, monkeypatch, bits, group, N, K, M):
    """INT4 launches whose groups are multiples of 128 codes run the decode
    kernel built for whole four-set spans only, INT2 launches with whole
    k-blocks (K a multiple of 256) the one without the ragged-k-block body;
    TLQ_DECODE_GENERIC=1 forces the general kernel.  All give the same bits,
    and the oracle agrees."""
    case = synth.gemm_case(M, N, K, bits, group, seed=3 * M + N + K)
    outs = {}
    for generic in ("1", "0"):
        monkeypatch.setenv("TLQ_DECODE_GENERIC", generic)
        _, outs[generic] = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(outs["0"], ref, "fixed-form kernel int%d g%d M%d N%d K%d" % (bits, group, M, N, K))
    assert np.array_equal(outs["0"].view(np.uint16), outs["1"].view(np.uint16))


@pytest.mark.parametrize("bits,group,M,N,K,ks", [(4, 128, 128, 512, 2048, 1), (4, 128, 40, 256, 4096, 4),
                                                 (4, 256, 300, 768, 4096, 2), (2, 64, 200, 512, 2048, 1),
                                                 (2, 128, 129, 256, 8192, 8), (4, 128, 2048, 2048, 2048, 1)])
def test_prefill_lean_form_bitwise(lib, monkeypatch, bits, group, M, N, K, ks):
    """Prefill launches with whole stages and row tiles, vector scales/zeros
    and a power-of-two group take the lean kernel form;
    TLQ_PREFILL_GENERIC=1 forces the general one.  Both give the same bits,
    with and without a k split, and the oracle agrees."""
    case = synth.gemm_case(M, N, K, bits, group, seed=M + N + K + ks, a_scale=0.5)
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", str(ks))
    Wd = gpu_pack(lib, case["codes"], bits)
    A, s, z = dev(case["A"]), dev(case["scales"]), dev(case["zeros"])
    wsb = lib.tl_quant_gemm_workspace_size(M, N, K, bits, group)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    outs = {}
    for generic in ("1", "0"):
        monkeypatch.setenv("TLQ_PREFILL_GENERIC", generic)
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        lib.tl_quant_gemm_ws(A, Wd, s, z, C, bits, group, ws)
        torch.cuda.synchronize()
        lib.tl_check_status()
        outs[generic] = C.cpu().numpy()
    assert np.array_equal(outs["0"].view(np.uint16), outs["1"].view(np.uint16))
    rows = sample_rows(M, 24, np.random.default_rng(K))
    ref = oracle.quant_gemm(case["A"][rows], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits,
                            group)
    assert_close(outs["0"][rows], ref, "lean prefill int%d g%d M%d N%d K%d ks%d" % (bits, group, M, N, K, ks))


def test_decode_batch_mixing_group_classes_bitwise(lib):
    """A batched INT4 decode call whose problems all have groups of 128 or 256
    takes the whole-span kernel; adding one problem with groups of 64 sends
    the whole batch to the general kernel.  Every problem's output is the same
    bits either way, and the oracle agrees."""
    specs = [(1, 256, 2048, 4, 128), (16, 192, 1024, 4, 256), (4, 320, 4096, 4, 128), (9, 160, 768, 4, 64)]
    probs = _problems(specs, seed=11)
    descs = lambda ps: [(p["A"], p["W"], p["s"], p["z"], p["C"], 4, p["case"]["group"]) for p in ps]
    lib.tl_quant_gemm_batched(descs(probs[:3]))
    torch.cuda.synchronize()
    whole = [p["C"].clone() for p in probs[:3]]
    for p in probs:
        p["C"].zero_()
    lib.tl_quant_gemm_batched(descs(probs))
    torch.cuda.synchronize()
    lib.tl_check_status()
    for i in range(3):
        assert torch.equal(whole[i].view(torch.int16), probs[i]["C"].view(torch.int16)), i
    for p in probs:
        c = p["case"]
        ref = oracle.quant_gemm(c["A"], oracle.pack(c["codes"], 4), c["scales"], c["zeros"], 4, c["group"])
        assert_close(p["C"].cpu().numpy(), ref, "batch g%d" % c["group"])


# ---------------------------------------------------------------------------
# full-size decode configurations (the four D = 2048 projections): every
# output against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("proj", list(synth.SHAPES))
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_full_size_sampled(lib, bits, proj, M):
    N, K = synth.SHAPES[proj]
    group = synth.DIST[bits]["group"]
    case = synth.gemm_case(M, N, K, bits, group, seed=0)
    Wd, C = run_case(lib, case)
    # every row (M <= 16) against the oracle, with the per-row bound
    ref = oracle.quant_gemm(case["A"], Wd.cpu().numpy().view(np.uint32), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "int%d %s M%d" % (bits, proj, M))


def test_gemv_config_full_oracle(lib):
    """M = 1, K = N = 2048, INT4 group 128: every output against the oracle."""
    case = synth.gemm_case(1, 2048, 2048, 4, 128, seed=0)
    _, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], 4), case["scales"], case["zeros"], 4, 128)
    assert_close(C, ref, "gemv")


# ---------------------------------------------------------------------------
# error paths and the bounded-wait self test
# ---------------------------------------------------------------------------

def test_gpu_argument_errors(lib):
    A = torch.zeros((1, 128), dtype=torch.float16, device="cuda")
    W = torch.zeros((8, 16), dtype=torch.int32, device="cuda")
    s = torch.zeros((8, 1), dtype=torch.float16, device="cuda")
    C = torch.zeros((1, 8), dtype=torch.float16, device="cuda")
    with pytest.raises(lib.TLQError, match="group"):
        lib.tl_quant_gemm(A, W, s, s, C, 4, 96)
    # a one-row slice at an 8-byte offset is "contiguous" for torch but not
    # 16-byte aligned: rejected before launch
    Aoff = torch.zeros((1, 136), dtype=torch.float16, device="cuda")[:, 4:132]
    assert Aoff.is_contiguous()
    with pytest.raises(lib.TLQError, match="aligned"):
        lib.tl_quant_gemm(Aoff, W, s, s, C, 4, 128)
    lib.tl_quant_gemm(Aoff.clone(), W, s, s, C, 4, 128)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C) == 0


def test_bounded_wait_reports_timeout(lib):
    lib.tl_reset_status()
    lib.tl_selftest_wait_timeout(2000)
    with pytest.raises(lib.TLQError) as ei:
        lib.tl_check_status()
    assert ei.value.status == lib.TLQ_ETIMEOUT
    lib.tl_reset_status()
    lib.tl_check_status()
    # the context is still usable
    case = synth.gemm_case(1, 64, 128, 4, 128, seed=1)
    run_case(lib, case)


# ---------------------------------------------------------------------------
# prefill path (M > 16, tcgen05): element-wise against the oracle on shapes
# with ragged token / row / k tails, every k-split, and full-size samples
# ---------------------------------------------------------------------------

PREFILL_SHAPES = [
    # bits, group, M, N, K
    (4, 128, 128, 256, 1024),
    (4, 128, 17, 264, 512),
    (4, 128, 200, 512, 2048),
    (4, 32, 96, 256, 96),      # K not a multiple of the 64-wide stage, two groups per stage
    (4, 64, 300, 520, 384),
    (4, 1024, 130, 256, 1024),  # one scale per row
    (2, 64, 128, 256, 1024),
    (2, 64, 33, 136, 448),
    (2, 128, 256, 512, 2048),
    (2, 512, 160, 256, 512),
]


@pytest.mark.parametrize("bits,group,M,N,K", PREFILL_SHAPES)
def test_prefill_matches_oracle(lib, bits, group, M, N, K):
    case = synth.gemm_case(M, N, K, bits, group, seed=M + N + K, a_scale=0.5)
    _, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "prefill int%d g%d M%d N%d K%d" % (bits, group, M, N, K))


@pytest.mark.parametrize("ks", ["1", "2", "4", "8"])
@pytest.mark.parametrize("bits", [4, 2])
def test_prefill_every_k_split(lib, monkeypatch, bits, ks):
    group = synth.DIST[bits]["group"]
    case = synth.gemm_case(150, 512, 2048, bits, group, seed=11, a_scale=0.5)
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", ks)
    Wd, C = run_case(lib, case)
    C2 = lib.quant_gemm(dev(case["A"]), Wd, dev(case["scales"]), dev(case["zeros"]), bits, group)
    assert torch.equal(torch.from_numpy(C).cuda().view(torch.int16), C2.view(torch.int16)), "not deterministic"
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "prefill ksplit %s int%d" % (ks, bits))


@pytest.mark.parametrize("ks", ["2", "4", "8"])
@pytest.mark.parametrize("bits", [4, 2])
def test_prefill_two_token_tiles_with_k_split(lib, monkeypatch, bits, ks):
    """Two token tiles per CTA and a cluster k split: the partial tiles are reduced once per token tile."""
    group = synth.DIST[bits]["group"]
    case = synth.gemm_case(300, 264, 2048, bits, group, seed=17, a_scale=0.5)
    monkeypatch.setenv("TLQ_PREFILL_NMT", "2")
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", ks)
    Wd, C = run_case(lib, case)
    C2 = lib.quant_gemm(dev(case["A"]), Wd, dev(case["scales"]), dev(case["zeros"]), bits, group)
    assert torch.equal(torch.from_numpy(C).cuda().view(torch.int16), C2.view(torch.int16)), "not deterministic"
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "prefill nmt 2 ksplit %s int%d" % (ks, bits))


@pytest.mark.parametrize("nmt", ["1", "2"])
@pytest.mark.parametrize("bits,group,M,N,K", [
    (4, 128, 129, 256, 512),   # second token tile holds one row
    (4, 128, 200, 520, 1024),  # ragged tokens and rows
    (4, 32, 300, 264, 96),     # ragged K, two groups per stage
    (4, 128, 512, 512, 2048),
    (2, 64, 257, 256, 448),
    (2, 128, 384, 512, 1024),
])
def test_prefill_token_tiles_per_cta(lib, monkeypatch, nmt, bits, group, M, N, K):
    """One and two 128-token tiles per CTA (forced) both match the oracle, and each other bit for bit when
    neither splits K (a k split changes the FP32 summation order)."""
    case = synth.gemm_case(M, N, K, bits, group, seed=3 * M + K, a_scale=0.5)
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", "1")
    monkeypatch.setenv("TLQ_PREFILL_NMT", nmt)
    Wd, C = run_case(lib, case)
    ref = oracle.quant_gemm(case["A"], oracle.pack(case["codes"], bits), case["scales"], case["zeros"], bits, group)
    assert_close(C, ref, "prefill nmt %s int%d M%d N%d K%d" % (nmt, bits, M, N, K))
    monkeypatch.setenv("TLQ_PREFILL_NMT", "2" if nmt == "1" else "1")
    C2 = lib.quant_gemm(dev(case["A"]), Wd, dev(case["scales"]), dev(case["zeros"]), bits, group)
    assert torch.equal(torch.from_numpy(C).cuda().view(torch.int16), C2.view(torch.int16)), \
        "one and two token tiles per CTA differ"


@pytest.mark.parametrize("proj", list(synth.SHAPES))
@pytest.mark.parametrize("M", [128, 512, 2048])
def test_prefill_full_size_sampled(lib, proj, M):
    N, K = synth.SHAPES[proj]
    case = synth.gemm_case(M, N, K, 4, 128, seed=0, a_scale=0.5)
    Wd, C = run_case(lib, case)
    # 16 whole rows (spread over every 128-token tile position) against the
    # oracle evaluated on those rows only, with the per-row bound
    rows = sample_rows(M, 16, np.random.default_rng(M * 7 + N))
    ref = oracle.quant_gemm(case["A"][rows], Wd.cpu().numpy().view(np.uint32), case["scales"], case["zeros"], 4, 128)
    assert_close(C[rows], ref, "prefill %s M%d" % (proj, M))
    # every row/column finite and the full output in the range the inputs allow
    assert np.all(np.isfinite(C.astype(np.float32)))


# ---------------------------------------------------------------------------
# the caller-owned k-split workspace
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("proj", ["o", "down"])
def test_prefill_workspace_is_optional(lib, proj):
    """M = 128 on a projection whose tiles leave SMs idle: the kernel asks for
    a k-split workspace.  Without one (tl_quant_gemm), with one too small for
    its first choice and with the size it asks for, every sampled row matches
    the oracle (the split changes only the FP32 summation order), a call with
    the full workspace repeats bit for bit, and nothing is drawn from the
    device's stream-ordered pool."""
    from devmem import default_pool_high_watermark

    N, K = synth.SHAPES[proj]
    M = 128
    case = synth.gemm_case(M, N, K, 4, 128, seed=17, a_scale=0.5)
    need = lib.tl_quant_gemm_workspace_size(M, N, K, 4, 128)
    assert need > 0
    Wd = gpu_pack(lib, case["codes"], 4)
    A, s, z = dev(case["A"]), dev(case["scales"]), dev(case["zeros"])
    rows = sample_rows(M, 16, np.random.default_rng(3))
    ref = oracle.quant_gemm(case["A"][rows], Wd.cpu().numpy().view(np.uint32), case["scales"], case["zeros"], 4, 128)
    outs = {}
    for label, nbytes in (("none", 0), ("small", need // 2 - 16), ("full", need)):
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
        torch.cuda.synchronize()
        default_pool_high_watermark(reset=True)
        if ws is None:
            lib.tl_quant_gemm(A, Wd, s, z, C, 4, 128)
        else:
            lib.tl_quant_gemm_ws(A, Wd, s, z, C, 4, 128, ws)
        torch.cuda.synchronize()
        assert default_pool_high_watermark() == 0, label
        lib.tl_check_status()
        outs[label] = C
        assert_close(C.cpu().numpy()[rows], ref, "%s workspace %s" % (proj, label))
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    lib.tl_quant_gemm_ws(A, Wd, s, z, C, 4, 128, torch.empty(need, dtype=torch.uint8, device="cuda"))
    assert torch.equal(C.view(torch.int16), outs["full"].view(torch.int16))


# ---------------------------------------------------------------------------
# batched launches: several independent problems, one decode launch per bit width
# ---------------------------------------------------------------------------

def _problems(specs, seed=0):
    out = []
    for i, (M, N, K, bits, group) in enumerate(specs):
        case = synth.gemm_case(M, N, K, bits, group, seed=seed + i, a_scale=0.5 if M > 16 else 1.0)
        W = torch.from_numpy(oracle.pack(case["codes"], bits).view(np.int32)).cuda()
        out.append(dict(case=case, A=dev(case["A"]), W=W, s=dev(case["scales"]), z=dev(case["zeros"]),
                        C=torch.empty((M, N), dtype=torch.float16, device="cuda")))
    return out


def test_batched_equals_separate_calls_bitwise(lib):
    specs = [(M, N, K, 4, 128) for M in (1, 4, 16) for (N, K) in synth.SHAPES.values()]
    probs = _problems(specs)
    lib.tl_quant_gemm_batched([(p["A"], p["W"], p["s"], p["z"], p["C"], 4, 128) for p in probs])
    torch.cuda.synchronize()
    lib.tl_check_status()
    for p, (M, N, K, bits, group) in zip(probs, specs):
        single = lib.quant_gemm(p["A"], p["W"], p["s"], p["z"], bits, group)
        assert torch.equal(single.view(torch.int16), p["C"].view(torch.int16)), (M, N, K)
    # and a sample against the oracle
    rng = np.random.default_rng(5)
    for p, (M, N, K, bits, group) in zip(probs, specs):
        rows = sample_rows(M, 4, rng)
        c = p["case"]
        ref = oracle.quant_gemm(c["A"][rows], p["W"].cpu().numpy().view(np.uint32), c["scales"], c["zeros"], bits,
                                group)
        assert_close(p["C"].cpu().numpy()[rows], ref, "batched M%d N%d K%d" % (M, N, K))


def test_batched_int2_decode_step_bitwise(lib):
    """The INT2 decode step (the four projections at M = 1, 4, 16, group 64)
    as one batched launch: the same bits as one call per problem, and a
    sample of rows against the oracle."""
    specs = [(M, N, K, 2, 64) for M in (1, 4, 16) for (N, K) in synth.SHAPES.values()]
    probs = _problems(specs, seed=70)
    lib.tl_quant_gemm_batched([(p["A"], p["W"], p["s"], p["z"], p["C"], 2, 64) for p in probs])
    torch.cuda.synchronize()
    lib.tl_check_status()
    for p, (M, N, K, bits, group) in zip(probs, specs):
        single = lib.quant_gemm(p["A"], p["W"], p["s"], p["z"], bits, group)
        assert torch.equal(single.view(torch.int16), p["C"].view(torch.int16)), (M, N, K)
    rng = np.random.default_rng(7)
    for p, (M, N, K, bits, group) in zip(probs, specs):
        rows = sample_rows(M, 4, rng)
        c = p["case"]
        ref = oracle.quant_gemm(c["A"][rows], p["W"].cpu().numpy().view(np.uint32), c["scales"], c["zeros"], bits,
                                group)
        assert_close(p["C"].cpu().numpy()[rows], ref, "batched int2 M%d N%d K%d" % (M, N, K))


def test_batched_prefill_side_streams_in_a_graph(lib):
    """The prefill problems of one batched call run side by side on side
    streams forked from the caller's stream.  A CUDA graph captured on that
    stream (after a call outside capture has set the side streams up) replays
    to the same bits as the direct call, with the side streams' work joined
    back before the stream completes; and the outputs agree with the oracle."""
    specs = [(128, 512, 1024, 4, 128), (200, 256, 2048, 4, 128), (256, 768, 512, 4, 128), (130, 1024, 1024, 4, 128),
             (5, 512, 1024, 4, 128)]
    probs = _problems(specs, seed=40)
    for p, (M, N, K, bits, group) in zip(probs, specs):  # each prefill problem its own k-split workspace
        p["ws"] = lib.gemm_workspace(M, N, K, bits, group)
    assert any(p["ws"] is not None for p in probs)
    descs = lib.gemm_descs([(p["A"], p["W"], p["s"], p["z"], p["C"], 4, 128, p["ws"]) for p in probs])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.tl_quant_gemm_batched(descs, s)
    torch.cuda.synchronize()
    lib.tl_check_status()
    direct = [p["C"].clone() for p in probs]
    for p in probs:
        p["C"].zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lib.tl_quant_gemm_batched(descs, s)
    for _ in range(2):
        g.replay()
        s.synchronize()
        lib.tl_check_status()
        for p, d in zip(probs, direct):
            assert torch.equal(p["C"].view(torch.int16), d.view(torch.int16))
    rng = np.random.default_rng(9)
    for p, (M, N, K, bits, group) in zip(probs, specs):
        rows = sample_rows(M, 8, rng)
        c = p["case"]
        ref = oracle.quant_gemm(c["A"][rows], p["W"].cpu().numpy().view(np.uint32), c["scales"], c["zeros"], bits,
                                group)
        assert_close(p["C"].cpu().numpy()[rows], ref, "side streams M%d N%d K%d" % (M, N, K))


@pytest.mark.parametrize("M,bits", [(128, 4), (512, 4), (2048, 4), (128, 2), (512, 2)])
def test_batched_prefill_step_full_size(lib, M, bits):
    """The four D = 2048 projections at M = 128 / 512 / 2048 (INT4) and 128 / 512
    (INT2) in one batched call, each
    with the workspace its own plan asks for: the launches run side by side
    with token tiles and k splits planned for the shared GPU (at M = 128 the
    DOWN projection alone keeps a k split).  16 whole rows per problem against
    the oracle; a second call gives the same bits."""
    group = synth.DIST[bits]["group"]
    specs = [(M, N, K, bits, group) for (N, K) in synth.SHAPES.values()]
    probs = _problems(specs, seed=50)
    for p, (M_, N, K, bits_, group_) in zip(probs, specs):
        p["ws"] = lib.gemm_workspace(M_, N, K, bits_, group_)
    descs = lib.gemm_descs([(p["A"], p["W"], p["s"], p["z"], p["C"], bits, group, p["ws"]) for p in probs])
    lib.tl_quant_gemm_batched(descs)
    torch.cuda.synchronize()
    lib.tl_check_status()
    first = [p["C"].clone() for p in probs]
    lib.tl_quant_gemm_batched(descs)
    torch.cuda.synchronize()
    for p, f in zip(probs, first):
        assert torch.equal(p["C"].view(torch.int16), f.view(torch.int16))
    rng = np.random.default_rng(M + bits)
    for p, (M_, N, K, bits_, group_) in zip(probs, specs):
        rows = sample_rows(M, 16, rng)
        c = p["case"]
        ref = oracle.quant_gemm(c["A"][rows], p["W"].cpu().numpy().view(np.uint32), c["scales"], c["zeros"], bits,
                                group)
        assert_close(p["C"].cpu().numpy()[rows], ref, "batched step int%d M%d N%d K%d" % (bits, M, N, K))


def test_batched_mixed_bits_and_paths(lib):
    specs = [(1, 256, 1024, 4, 128), (9, 136, 448, 2, 64), (40, 264, 512, 4, 128), (3, 512, 2048, 2, 128),
             (16, 64, 4096, 4, 4096), (130, 256, 1024, 2, 64)]
    probs = _problems(specs, seed=50)
    lib.tl_quant_gemm_batched([(p["A"], p["W"], p["s"], p["z"], p["C"], b, g)
                               for p, (_, _, _, b, g) in zip(probs, specs)])
    torch.cuda.synchronize()
    lib.tl_check_status()
    for p, (M, N, K, bits, group) in zip(probs, specs):
        c = p["case"]
        ref = oracle.quant_gemm(c["A"], oracle.pack(c["codes"], bits), c["scales"], c["zeros"], bits, group)
        assert_close(p["C"].cpu().numpy(), ref, "mixed M%d N%d K%d int%d" % (M, N, K, bits))


def test_batched_many_problems_and_errors(lib):
    specs = [(1 + (i % 16), 64 + 8 * i, 256 * (1 + i % 3), 4, 128) for i in range(20)]  # > 16 decode problems
    probs = _problems(specs, seed=70)
    lib.tl_quant_gemm_batched([(p["A"], p["W"], p["s"], p["z"], p["C"], 4, 128) for p in probs])
    torch.cuda.synchronize()
    for p, (M, N, K, bits, group) in zip(probs, specs):
        c = p["case"]
        ref = oracle.quant_gemm(c["A"], oracle.pack(c["codes"], bits), c["scales"], c["zeros"], bits, group)
        assert_close(p["C"].cpu().numpy(), ref, "many M%d N%d K%d" % (M, N, K))
    lib.tl_quant_gemm_batched([])  # no-op
    p0, p1 = probs[0], probs[1]
    with pytest.raises(lib.TLQError, match="overlap"):
        lib.tl_quant_gemm_batched([(p0["A"], p0["W"], p0["s"], p0["z"], p0["C"], 4, 128),
                                   (p1["A"], p1["W"], p1["s"], p1["z"], p0["C"], 4, 128)])


def test_batched_host_buffers_equal_device_call(lib):
    """tl_quant_gemm_batched_host (host activations in, host outputs out) gives
    the device call's outputs bit for bit, also when two calls alternate
    between two streams and two staging sets."""
    shapes = [(1, 256, 1024), (4, 512, 2048), (16, 256, 1024)]
    rng = np.random.default_rng(9)
    probs = []
    for (M, N, K) in shapes:
        case = synth.gemm_case(M, N, K, 4, 128, seed=M + N)
        probs.append((case, lib.pack_weights(dev(case["codes"]), 4), dev(case["scales"]), dev(case["zeros"])))
    na = sum(M * K for (M, N, K) in shapes)
    nc = sum(M * N for (M, N, K) in shapes)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    sets = []
    for b in range(2):
        dA = torch.empty(na, dtype=torch.float16, device="cuda")
        dC = torch.empty(nc, dtype=torch.float16, device="cuda")
        descs, oa, oc = [], 0, 0
        for (case, W, S, Z), (M, N, K) in zip(probs, shapes):
            descs.append((dA[oa:oa + M * K].view(M, K), W, S, Z, dC[oc:oc + M * N].view(M, N), 4, 128))
            oa += M * K
            oc += M * N
        sets.append((dA, dC, lib.gemm_descs(descs)))
    hostA = [torch.from_numpy(np.concatenate([(c["A"] * (1 + b)).astype(np.float16).ravel() for c, *_ in probs]))
             .pin_memory() for b in range(2)]
    hostC = [torch.empty(nc, dtype=torch.float16).pin_memory() for _ in range(2)]
    for it in range(4):
        b = it & 1
        dA, dC, d = sets[b]
        lib.tl_quant_gemm_batched_host(d, hostA[b], dA, hostC[b], dC, streams[b])
    torch.cuda.synchronize()
    for b in range(2):
        dA, dC, d = sets[b]
        dA.copy_(hostA[b].cuda())
        lib.tl_quant_gemm_batched(d)
        torch.cuda.synchronize()
        assert torch.equal(hostC[b].view(torch.int16), dC.cpu().view(torch.int16)), b

"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every entry point include/tlq.h declares, and rejects
bad arguments before launching anything."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tlq.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def clib():
    import weight_only_int4_quant_gb300 as tlq

    tlq.build()
    return tlq.load()


def test_header_declares_expected_entry_points():
    import weight_only_int4_quant_gb300 as tlq

    assert header_functions() == sorted(tlq.EXPORTED)


def test_library_exports_every_declared_symbol(clib):
    for name in header_functions():
        assert hasattr(clib, name), name
        assert ctypes.cast(getattr(clib, name), ctypes.c_void_p).value


def test_version(clib):
    import weight_only_int4_quant_gb300 as tlq

    assert "sm_103a" in tlq.tl_version()


def _gemm(clib, A=16, W=16, s=16, z=16, C=4096, M=1, N=8, K=128, bits=4, group=128):
    return clib.tl_quant_gemm(A, W, s, z, C, M, N, K, bits, group, None)


def test_gemm_rejects_bad_arguments_without_launching(clib):
    import weight_only_int4_quant_gb300 as tlq

    # null pointers
    assert _gemm(clib, A=None) == tlq.TLQ_EINVAL
    assert "null" in tlq.tl_last_error()
    assert _gemm(clib, C=None) == tlq.TLQ_EINVAL
    # bit width, shapes, groups
    assert _gemm(clib, bits=3) == tlq.TLQ_EINVAL and "bits" in tlq.tl_last_error()
    assert _gemm(clib, bits=8) == tlq.TLQ_EINVAL
    assert _gemm(clib, M=0) == tlq.TLQ_EINVAL and "M=" in tlq.tl_last_error()
    assert _gemm(clib, N=0) == tlq.TLQ_EINVAL
    assert _gemm(clib, K=0) == tlq.TLQ_EINVAL
    assert _gemm(clib, group=48) == tlq.TLQ_EINVAL and "group" in tlq.tl_last_error()
    assert _gemm(clib, bits=2, group=32) == tlq.TLQ_EINVAL  # INT2 groups are multiples of 64
    assert _gemm(clib, K=192, group=128) == tlq.TLQ_EINVAL and "multiple of group" in tlq.tl_last_error()
    assert _gemm(clib, N=12) == tlq.TLQ_EINVAL
    # alignment and aliasing
    assert _gemm(clib, A=18) == tlq.TLQ_EINVAL and "aligned" in tlq.tl_last_error()
    assert _gemm(clib, W=20) == tlq.TLQ_EINVAL
    assert _gemm(clib, A=4096, C=4096 + 64) == tlq.TLQ_EINVAL and "overlap" in tlq.tl_last_error()


def test_pack_and_block_reject_bad_arguments(clib):
    import weight_only_int4_quant_gb300 as tlq

    assert clib.tl_pack_weights(None, 16, 4, 64, 4, None) == tlq.TLQ_EINVAL
    assert clib.tl_pack_weights(16, 16, 4, 60, 4, None) == tlq.TLQ_EINVAL  # K % 8
    assert clib.tl_pack_weights(16, 16, 4, 64, 5, None) == tlq.TLQ_EINVAL
    assert clib.tl_unpack_weights(16, 16, 4, 72, 2, None) == tlq.TLQ_EINVAL  # K % 16
    assert clib.tl_loop_block_forward(None, None, 1, 1, None) == tlq.TLQ_EINVAL
    blk = tlq._Block()
    blk.D = 64
    assert clib.tl_loop_block_forward(16, ctypes.byref(blk), 1, 1, None) == tlq.TLQ_EINVAL
    assert clib.tl_loop_block_forward(16, ctypes.byref(blk), -1, 1, None) == tlq.TLQ_EINVAL
    assert clib.tl_selftest_wait_timeout(0, None) == tlq.TLQ_EINVAL


def test_requant_rejects_bad_arguments(clib):
    """Validation of tl_requant_int4_to_int2 happens before any launch; the
    addresses below are never dereferenced."""
    import weight_only_int4_quant_gb300 as tlq

    N, K, g = 8, 256, 128
    W4, s4, z4, W2, s2, z2 = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 6 << 20

    def rq(W4=W4, s4=s4, z4=z4, W2=W2, s2=s2, z2=z2, N=N, K=K, g=g):
        return clib.tl_requant_int4_to_int2(W4, s4, z4, W2, s2, z2, N, K, g, None)

    assert rq(W4=None) == tlq.TLQ_EINVAL and "null" in tlq.tl_last_error()
    assert rq(z2=None) == tlq.TLQ_EINVAL
    assert rq(N=0) == tlq.TLQ_EINVAL
    assert rq(g=32) == tlq.TLQ_EINVAL and "group" in tlq.tl_last_error()  # INT2 groups are multiples of 64
    assert rq(g=96) == tlq.TLQ_EINVAL
    assert rq(K=320) == tlq.TLQ_EINVAL  # K % group
    assert rq(W4=W4 + 8) == tlq.TLQ_EINVAL and "aligned" in tlq.tl_last_error()
    assert rq(s2=s2 + 1) == tlq.TLQ_EINVAL
    assert rq(W2=W4 + 64) == tlq.TLQ_EINVAL and "overlap" in tlq.tl_last_error()
    assert rq(s2=z4) == tlq.TLQ_EINVAL  # s2 on top of z4
    assert rq(s2=s4 + 2) == tlq.TLQ_EINVAL  # partial overlap with its own input
    assert rq(z2=s2 + 4) == tlq.TLQ_EINVAL  # outputs overlap each other

    # batched: count limits, a bad descriptor by index, overlaps across descriptors
    D = tlq._RequantDesc
    ok0 = D(W4, s4, z4, W2, s2, z2, N, K)
    arr = (D * 17)(*([ok0] * 17))
    assert clib.tl_requant_int4_to_int2_batched(arr, 17, g, None) == tlq.TLQ_EINVAL
    assert clib.tl_requant_int4_to_int2_batched(None, 2, g, None) == tlq.TLQ_EINVAL
    assert clib.tl_requant_int4_to_int2_batched(arr, 1, 100, None) == tlq.TLQ_EINVAL
    bad = (D * 2)(ok0, D(7 << 20, 8 << 20, 9 << 20, 10 << 20, 11 << 20, 12 << 20, N, 200))
    assert clib.tl_requant_int4_to_int2_batched(bad, 2, g, None) == tlq.TLQ_EINVAL
    assert "[1]" in tlq.tl_last_error()
    # problem 1 writes its W2 over problem 0's W4
    cross = (D * 2)(ok0, D(7 << 20, 8 << 20, 9 << 20, W4 + 256, 11 << 20, 12 << 20, N, K))
    assert clib.tl_requant_int4_to_int2_batched(cross, 2, g, None) == tlq.TLQ_EINVAL
    assert "overlap" in tlq.tl_last_error()
    # problem 1 converts its scales in place of problem 0's scales
    cross2 = (D * 2)(ok0, D(7 << 20, s4, 9 << 20, 10 << 20, s4, 12 << 20, N, K))
    assert clib.tl_requant_int4_to_int2_batched(cross2, 2, g, None) == tlq.TLQ_EINVAL


def test_swiglu_entry_points_reject_bad_arguments(clib):
    """Host-side validation of the SwiGLU GEMM, the row interleave and the
    SwiGLU block; nothing is launched (the addresses are never dereferenced)."""
    import weight_only_int4_quant_gb300 as tlq

    A, W, S, Z, C = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20
    ok = dict(A=A, W=W, S=S, Z=Z, C=C, M=4, N2=64, K=256, bits=4, group=128)

    def sw(**kw):
        a = dict(ok, **kw)
        return clib.tl_quant_gemm_swiglu(a["A"], a["W"], a["S"], a["Z"], a["C"], a["M"], a["N2"], a["K"],
                                         a["bits"], a["group"], None)

    assert sw(N2=24) == tlq.TLQ_EINVAL and "16" in tlq.tl_last_error()
    assert sw(A=None) == tlq.TLQ_EINVAL
    assert sw(bits=3) == tlq.TLQ_EINVAL
    assert sw(C=A + 64) == tlq.TLQ_EINVAL and "overlap" in tlq.tl_last_error()
    assert clib.tl_interleave_rows(None, W, C, 4, 64, None) == tlq.TLQ_EINVAL
    assert clib.tl_interleave_rows(A, W, C, 0, 64, None) == tlq.TLQ_EINVAL
    assert clib.tl_interleave_rows(A, W, A + 64, 4, 64, None) == tlq.TLQ_EINVAL  # out over a
    assert clib.tl_swiglu_block_forward(None, None, 1, 1, None) == tlq.TLQ_EINVAL
    blk = tlq._SwigluBlock()
    blk.D = 64
    assert clib.tl_swiglu_block_forward(16, ctypes.byref(blk), 1, 1, None) == tlq.TLQ_EINVAL
    blk.qkv.N, blk.qkv.K, blk.o.N, blk.o.K = 192, 64, 64, 64
    blk.gate_up.N, blk.gate_up.K, blk.down.N, blk.down.K = 120, 64, 64, 60  # 2F not a multiple of 16
    assert clib.tl_swiglu_block_forward(16, ctypes.byref(blk), 1, 1, None) == tlq.TLQ_EINVAL
    assert "gate_up" in tlq.tl_last_error()


def test_dequant_fp16_rejects_bad_arguments(clib):
    import weight_only_int4_quant_gb300 as tlq

    W, S, Z, O = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    assert clib.tl_dequant_fp16(None, S, Z, O, 8, 256, 4, 128, None) == tlq.TLQ_EINVAL
    assert clib.tl_dequant_fp16(W, S, Z, O, 8, 256, 3, 128, None) == tlq.TLQ_EINVAL
    assert clib.tl_dequant_fp16(W, S, Z, O, 8, 256, 2, 32, None) == tlq.TLQ_EINVAL
    assert clib.tl_dequant_fp16(W, S, Z, O, 8, 200, 4, 128, None) == tlq.TLQ_EINVAL
    assert clib.tl_dequant_fp16(W, S, Z, O + 8, 8, 256, 4, 128, None) == tlq.TLQ_EINVAL
    assert clib.tl_dequant_fp16(W, S, Z, W + 16, 8, 256, 4, 128, None) == tlq.TLQ_EINVAL
    assert "overlap" in tlq.tl_last_error()


def test_batched_host_rejects_bad_arguments_before_copying(clib):
    import weight_only_int4_quant_gb300 as tlq

    hA, dA, hC, dC = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    D = tlq._GemmDesc
    good = D(dA, 5 << 20, 6 << 20, 7 << 20, dC, 1, 64, 256, 4, 128, 0, None, 0)

    def call(descs, n=1, **kw):
        a = dict(hA=hA, dA=dA, ab=4096, hC=hC, dC=dC, cb=4096)
        a.update(kw)
        return clib.tl_quant_gemm_batched_host(descs, n, a["hA"], a["dA"], a["ab"], a["hC"], a["dC"], a["cb"], None)

    one = (D * 1)(good)
    assert call(one, hA=None) == tlq.TLQ_EINVAL
    assert call(one, dC=dA + 64) == tlq.TLQ_EINVAL and "overlap" in tlq.tl_last_error()
    assert call(one, ab=256) == tlq.TLQ_EINVAL and "inside devA" in tlq.tl_last_error()  # A needs 512 bytes
    bad_bits = (D * 1)(D(dA, 5 << 20, 6 << 20, 7 << 20, dC, 1, 64, 256, 3, 128, 0, None, 0))
    assert call(bad_bits) == tlq.TLQ_EINVAL and "bits" in tlq.tl_last_error()
    assert call(one, n=0) == tlq.TLQ_EINVAL


def test_workspace_and_stride_arguments_are_checked(clib):
    """The k-split workspace and the weight row stride are validated before
    anything is launched (the addresses are never dereferenced)."""
    import weight_only_int4_quant_gb300 as tlq

    A, W, S, Z, C, WS = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20, 8 << 20

    def g(ws=WS, nb=1 << 20, **kw):
        a = dict(A=A, W=W, S=S, Z=Z, C=C, M=128, N=64, K=256, bits=4, group=128)
        a.update(kw)
        return clib.tl_quant_gemm_ws(a["A"], a["W"], a["S"], a["Z"], a["C"], a["M"], a["N"], a["K"], a["bits"],
                                     a["group"], ws, nb, None)

    assert g(ws=WS + 8) == tlq.TLQ_EINVAL and "aligned" in tlq.tl_last_error()
    assert g(ws=None, nb=64) == tlq.TLQ_EINVAL and "null workspace" in tlq.tl_last_error()
    assert g(ws=C) == tlq.TLQ_EINVAL and "overlaps" in tlq.tl_last_error()
    assert g(ws=W - 64) == tlq.TLQ_EINVAL  # runs into the weights
    assert g(bits=3) == tlq.TLQ_EINVAL
    # the size query: no split for decode sizes or invalid shapes, a split for
    # a short-M tensor-core problem that would leave SMs idle
    assert clib.tl_quant_gemm_workspace_size(16, 2048, 2048, 4, 128) == 0
    assert clib.tl_quant_gemm_workspace_size(128, 2048, 2048, 3, 128) == 0
    D = tlq._GemmDesc
    good = D(A, W, S, Z, C, 1, 64, 256, 4, 128, 0, None, 0)
    for bad in (D(A, W, S, Z, C, 1, 64, 256, 4, 128, 30, None, 0),     # ldw below the row's 32 words
                D(A, W, S, Z, C, 1, 64, 256, 4, 128, 34, None, 0),     # not a multiple of 4
                D(A, W, S, Z, C, 1, 64, 256, 4, 128, 0, WS + 4, 64)):  # misaligned workspace
        assert clib.tl_quant_gemm_batched((D * 1)(bad), 1, None) == tlq.TLQ_EINVAL
    # two problems' workspaces may not overlap (they may run at the same time)
    two = (D * 2)(D(A, W, S, Z, C, 128, 64, 256, 4, 128, 0, WS, 4096),
                  D(A + 65536, W, S, Z, C + 65536, 128, 64, 256, 4, 128, 0, WS + 1024, 4096))
    assert clib.tl_quant_gemm_batched(two, 2, None) == tlq.TLQ_EINVAL and "workspace" in tlq.tl_last_error()
    assert clib.tl_quant_gemm_swiglu_ws(A, W, S, Z, C, 4, 64, 256, 4, 128, WS + 8, 64, None) == tlq.TLQ_EINVAL
    assert good.ldw == 0


def test_tier_switch_rejects_bad_blocks(clib):
    """tl_loop_block_to_int2 / tl_swiglu_block_to_int2 check everything before
    their launch and leave the block as it was on an error."""
    import weight_only_int4_quant_gb300 as tlq

    assert clib.tl_loop_block_to_int2(None, None, None) == tlq.TLQ_EINVAL
    assert clib.tl_swiglu_block_to_int2(None, None, None) == tlq.TLQ_EINVAL
    blk = tlq._Block()
    blk.bits, blk.group, blk.D = 2, 128, 64
    assert clib.tl_loop_block_to_int2(ctypes.byref(blk), None, None) == tlq.TLQ_EINVAL
    assert "INT4" in tlq.tl_last_error()
    base = 1 << 24
    for i, name in enumerate(("qkv", "o", "up", "down")):
        N, K = {"qkv": (192, 64), "o": (64, 64), "up": (128, 64), "down": (64, 128)}[name]
        setattr(blk, name, tlq._QProj(base + i * (1 << 20), base + i * (1 << 20) + (1 << 19),
                                      base + i * (1 << 20) + (3 << 18), N, K, 0))
    blk.bits, blk.group = 4, 32  # INT2 groups are multiples of 64
    assert clib.tl_loop_block_to_int2(ctypes.byref(blk), None, None) == tlq.TLQ_EINVAL
    assert blk.bits == 4 and blk.qkv.ldw == 0
    blk.group = 64
    dst = (tlq._QProj * 4)()
    for i in range(4):
        dst[i] = tlq._QProj(base + (8 + i) * (1 << 20), blk.qkv.s, blk.qkv.z, 1, 64, 0)  # wrong N
    assert clib.tl_loop_block_to_int2(ctypes.byref(blk), dst, None) == tlq.TLQ_EINVAL
    assert blk.bits == 4


def test_loop_block_l2_plan(clib):
    """The residency plan keeps the block's projections resident in
    iteration order while their running byte total fits the budget, and
    none when the block runs once; a block too large for the budget keeps
    only the prefix that fits.  Host-only: the query reads shapes, not
    device memory."""
    import weight_only_int4_quant_gb300 as tlq

    def plan(D, F, bits, group, L):
        blk = tlq._Block()
        for name, (N, K) in (("qkv", (3 * D, D)), ("o", (D, D)), ("up", (F, D)), ("down", (D, F))):
            setattr(blk, name, tlq._QProj(1 << 20, 2 << 20, 3 << 20, N, K, 0))
        blk.bits, blk.group, blk.D = bits, group, D
        m, wb, bb = ctypes.c_int(), ctypes.c_size_t(), ctypes.c_size_t()
        assert clib.tl_loop_block_l2_plan(ctypes.byref(blk), L, ctypes.byref(m), ctypes.byref(wb),
                                          ctypes.byref(bb)) == tlq.TLQ_OK
        sizes = [N * K * bits // 8 + 4 * N * (K // group) for (N, K) in ((3 * D, D), (D, D), (F, D), (D, F))]
        return m.value, wb.value, bb.value, sizes

    # the D = 2048 block: 26.7 MB (INT4 g128) / 15.7 MB (INT2 g64)
    for bits, group, total in ((4, 128, 26738688), (2, 64, 15728640)):
        m, wb, bb, sizes = plan(2048, 8192, bits, group, 8)
        assert wb == total == sum(sizes)
        expect = 0
        for i in range(4):
            if sum(sizes[:i + 1]) <= bb:
                expect |= 1 << i
            else:
                break
        assert m == expect
        assert plan(2048, 8192, bits, group, 1)[0] == 0  # one iteration: nothing to keep
    # a block four times wider: only a prefix fits (or none), never a gap
    m, wb, bb, sizes = plan(8192, 32768, 4, 128, 8)
    assert wb > bb and m in (0, 1, 3, 7)
    k = bin(m).count("1")
    assert sum(sizes[:k]) <= bb and (k == 4 or sum(sizes[:k + 1]) > bb)
    blk = tlq._Block()
    blk.bits = 3
    assert clib.tl_loop_block_l2_plan(ctypes.byref(blk), 2, ctypes.byref(ctypes.c_int()), None, None) == tlq.TLQ_EINVAL


def test_library_sources_allocate_nothing():
    """The library makes no device or host-pinned allocation anywhere: every
    buffer is the caller's (the allocation-free entry point's static array is
    a file-scope __device__ variable, not an allocation call)."""
    csrc = os.path.join(ROOT, "weight_only_int4_quant_gb300", "csrc")
    banned = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|cudaMemPool\w*|cudaHostAlloc|"
                        r"cudaMallocHost|cudaMallocManaged|cuMemCreate|cudaMallocAsync)\b")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        code = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", text, flags=re.S))  # calls, not comments
        hits = banned.findall(code)
        assert not hits, (name, hits)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import weight_only_int4_quant_gb300 as tlq

    monkeypatch.setattr(tlq, "_lib", None)
    monkeypatch.setattr(tlq, "_LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        tlq.load()


# GB300 as the prefill planners see it: 152 SMs; clusters of 1 / 2 / 4 / 8
# CTAs that fit at once (one CTA per SM) with one and with two token tiles
GB300 = (152, (152, 76, 36, 15), (152, 76, 36, 15))
PROJ = [(6144, 2048), (2048, 2048), (8192, 2048), (2048, 8192)]  # QKV, O, UP, DOWN (N, K)
UNLIMITED = 1 << 40


def test_prefill_plan_single_calls(clib, monkeypatch):
    """Plans of single calls on the GB300 description (host only: no CUDA
    call with a device description).  At M = 128 each projection alone asks
    for a k split (the weight tiles alone leave SMs idle); without a
    workspace it keeps K whole; M <= 16 is the decode kernel; the
    environment's forced choices win."""
    import weight_only_int4_quant_gb300 as tlq

    monkeypatch.delenv("TLQ_PREFILL_NMT", raising=False)
    monkeypatch.delenv("TLQ_PREFILL_KSPLIT", raising=False)
    for (N, K), want in zip(PROJ, [(1, 4), (1, 8), (1, 4), (1, 8)]):
        assert tlq.tl_prefill_plan([(128, N, K)], [UNLIMITED], GB300) == [want]
        assert tlq.tl_prefill_plan([(128, N, K)], [0], GB300) == [(1, 1)]
        assert tlq.tl_prefill_plan([(16, N, K)], [UNLIMITED], GB300) == [(0, 0)]
    # two token tiles per CTA only when M has two token tiles
    assert tlq.tl_prefill_plan([(2048, 8192, 2048)], [UNLIMITED], GB300) == [(2, 1)]
    assert all(p[0] == 1 for p in tlq.tl_prefill_plan([(128, N, K) for N, K in PROJ][:1], [UNLIMITED], GB300))
    monkeypatch.setenv("TLQ_PREFILL_KSPLIT", "2")
    assert tlq.tl_prefill_plan([(128, 2048, 8192)], [UNLIMITED], GB300) == [(1, 2)]
    with pytest.raises(tlq.TLQError):  # a forced split without its workspace
        tlq.tl_prefill_plan([(128, 2048, 8192)], [0], GB300)


def test_prefill_plan_joint(clib, monkeypatch):
    """Four projections side by side (a batched call): the joint plan is the
    combination measured fastest on GB300 at M = 128 (31.0 us against 46.1 us
    for the single-call plans; every combination swept), keeps splits of 8
    out, and uses far fewer CTAs than the single-call plans; at M = 512 and
    2048 every launch takes two token tiles per CTA and only DOWN splits K.
    Forcing a choice through the environment turns joint planning off."""
    import weight_only_int4_quant_gb300 as tlq

    monkeypatch.delenv("TLQ_PREFILL_NMT", raising=False)
    monkeypatch.delenv("TLQ_PREFILL_KSPLIT", raising=False)

    def ctas(M, plans):
        return sum(((N + 255) // 256) * ((M + 128 * nmt - 1) // (128 * nmt)) * ks
                   for (N, K), (nmt, ks) in zip(PROJ, plans))

    probs = [(128, N, K) for N, K in PROJ]
    joint = tlq.tl_prefill_plan(probs, [UNLIMITED] * 4, GB300)
    assert joint == [(1, 1), (1, 1), (1, 1), (1, 4)]
    solo = [tlq.tl_prefill_plan([p], [UNLIMITED], GB300)[0] for p in probs]
    assert ctas(128, joint) == 96 < ctas(128, solo) == 352
    assert tlq.tl_prefill_plan([(512, N, K) for N, K in PROJ], [UNLIMITED] * 4, GB300) == \
        [(2, 1), (2, 1), (2, 1), (2, 4)]
    assert tlq.tl_prefill_plan([(2048, N, K) for N, K in PROJ], [UNLIMITED] * 4, GB300) == \
        [(2, 1), (2, 1), (2, 1), (2, 2)]
    # each launch stays within its own workspace: none for QKV keeps it unsplit
    j = tlq.tl_prefill_plan(probs, [0, UNLIMITED, UNLIMITED, 0], GB300)
    assert j[0][1] == 1 and j[3][1] == 1
    # a decode-sized problem in the batch: no joint plan, each planned alone
    mixed = tlq.tl_prefill_plan([(1, 6144, 2048)] + probs[1:], [UNLIMITED] * 4, GB300)
    assert mixed == [(0, 0)] + solo[1:]
    monkeypatch.setenv("TLQ_PREFILL_NMT", "1")
    assert tlq.tl_prefill_plan(probs, [UNLIMITED] * 4, GB300) == solo


def test_prefill_plan_rejects_bad_arguments(clib):
    import weight_only_int4_quant_gb300 as tlq

    n = (ctypes.c_int * 1)(128)
    ws = (ctypes.c_size_t * 1)(0)
    out1, out2 = (ctypes.c_int * 1)(), (ctypes.c_int * 1)()
    dev = (ctypes.c_int * 9)(152, 152, 76, 36, 15, 152, 76, 36, 15)
    assert clib.tl_prefill_plan(n, n, n, ws, 0, dev, out1, out2) == tlq.TLQ_EINVAL
    assert clib.tl_prefill_plan(n, n, n, ws, 17, dev, out1, out2) == tlq.TLQ_EINVAL
    assert clib.tl_prefill_plan(n, None, n, ws, 1, dev, out1, out2) == tlq.TLQ_EINVAL
    zero = (ctypes.c_int * 1)(0)
    assert clib.tl_prefill_plan(n, zero, n, ws, 1, dev, out1, out2) == tlq.TLQ_EINVAL
    bad = (ctypes.c_int * 9)(152, 152, 76, 0, 15, 152, 76, 36, 15)
    assert clib.tl_prefill_plan(n, n, n, ws, 1, bad, out1, out2) == tlq.TLQ_EINVAL
    assert b"device[3]" in clib.tl_last_error()

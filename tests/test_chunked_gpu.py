"""GPU parity of chunked prefill (tl_loop_block_forward_chunked,
tl_swiglu_block_forward_chunked) against the oracle: every chunk size, ragged
last chunks, chunks on either side of the decode / tensor-core boundary, and
scratch sized for one chunk."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def make(lib, kind, case, max_rows):
    bits = case["bits"]
    proj, host = {}, {}
    for name, (codes, s, z) in case["proj"].items():
        proj[name] = (lib.pack_weights(dev(codes), bits), dev(s), dev(z))
        host[name] = (oracle.pack(codes, bits), s, z)
    cls = lib.LoopBlock if kind == "relu" else lib.SwiGLUBlock
    return cls(proj, bits, case["group"], max_rows), host


def ref_block(kind, x0, host, bits, group, L):
    f = oracle.loop_block if kind == "relu" else oracle.loop_block_swiglu
    return f(x0, host, bits, group, L)


def case_for(kind, M, bits, seed, D=256, F=512):
    if kind == "relu":
        return synth.block_case(M, bits, seed=seed, D=D, F=F)
    return synth.swiglu_block_case(M, bits, seed=seed, D=D, F=F)


@pytest.mark.parametrize("kind", ["relu", "swiglu"])
@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("chunk", [1, 7, 16, 17, 64, 128, 200])
def test_chunked_block_matches_oracle(lib, kind, bits, chunk):
    M, L = 300, 2
    case = case_for(kind, M, bits, seed=chunk + bits)
    blk, host = make(lib, kind, case, max_rows=min(chunk, M))  # scratch for one chunk only
    x = dev(case["x0"])
    blk.forward(x, L, chunk=chunk)
    torch.cuda.synchronize()
    lib.tl_check_status()
    ref = ref_block(kind, case["x0"], host, bits, case["group"], L)
    assert_close(x.cpu().numpy(), ref, "%s int%d chunk %d" % (kind, bits, chunk))


@pytest.mark.parametrize("kind", ["relu", "swiglu"])
def test_chunk_at_least_m_is_single_shot(lib, kind):
    case = case_for(kind, 40, 4, seed=3)
    blk, _ = make(lib, kind, case, max_rows=40)
    a, b = dev(case["x0"]), dev(case["x0"])
    blk.forward(a, 3)
    blk.forward(b, 3, chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_unchunked_call_needs_full_scratch(lib):
    case = case_for("swiglu", 64, 4, seed=4)
    blk, _ = make(lib, "swiglu", case, max_rows=16)
    with pytest.raises(ValueError):
        blk.forward(dev(case["x0"]), 1)
    with pytest.raises(ValueError):
        blk.forward(dev(case["x0"]), 1, chunk=32)
    blk.forward(dev(case["x0"]), 1, chunk=16)  # fits


def test_chunked_swiglu_full_width(lib):
    """D = 2048, F = 8192, a 512-token prompt in chunks of 128 (the
    tensor-core path per chunk), L = 2, sampled rows against the oracle."""
    case = synth.swiglu_block_case(512, 4, seed=5)
    blk, host = make(lib, "swiglu", case, max_rows=128)
    x = dev(case["x0"])
    blk.forward(x, 2, chunk=128)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 300, 511]
    ref = oracle.loop_block_swiglu(case["x0"][rows], host, 4, case["group"], 2)
    assert_close(x.cpu().numpy()[rows], ref, "chunked full width")

"""GPU parity of tl_loop_block_forward against the oracle's loop block."""
import numpy as np
import pytest

import oracle
import synth
from devmem import flush_l2
from parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def make_block(lib, case, normalize=True, max_rows=None):
    bits = case["bits"]
    proj = {}
    host = {}
    for name, (codes, s, z) in case["proj"].items():
        W = lib.pack_weights(torch.from_numpy(codes).cuda(), bits)
        proj[name] = (W, torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
        host[name] = (oracle.pack(codes, bits), s, z)
    blk = lib.LoopBlock(proj, bits, case["group"], max_rows or case["M"], normalize=normalize)
    return blk, host


def run_gpu(lib, blk, x0, L):
    x = torch.from_numpy(x0.copy()).cuda()
    blk.forward(x, L)
    torch.cuda.synchronize()
    lib.tl_check_status()
    return x.cpu().numpy()


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("M", [1, 5, 16, 40, 128])
@pytest.mark.parametrize("L", [1, 3])
def test_block_small_matches_oracle(lib, bits, M, L):
    case = synth.block_case(M, bits, seed=20 + M, D=256, F=512)
    blk, host = make_block(lib, case)
    got = run_gpu(lib, blk, case["x0"], L)
    ref = oracle.loop_block(case["x0"], host, bits, case["group"], L, normalize=True)
    assert_close(got, ref, "block int%d M%d L%d" % (bits, M, L))


@pytest.mark.parametrize("bits", [4, 2])
def test_block_two_token_tiles_per_cta(lib, monkeypatch, bits):
    """Prefill with two 128-token tiles per CTA (forced) in all three epilogues: store, ReLU, residual."""
    monkeypatch.setenv("TLQ_PREFILL_NMT", "2")
    case = synth.block_case(200, bits, seed=41, D=256, F=512)
    blk, host = make_block(lib, case)
    got = run_gpu(lib, blk, case["x0"], 2)
    ref = oracle.loop_block(case["x0"], host, bits, case["group"], 2, normalize=True)
    assert_close(got, ref, "block two token tiles int%d" % bits)


@pytest.mark.parametrize("bits", [4, 2])
def test_block_without_norm_one_iteration(lib, bits):
    case = synth.block_case(4, bits, seed=31, D=256, F=512)
    blk, host = make_block(lib, case, normalize=False)
    got = run_gpu(lib, blk, case["x0"], 1)
    ref = oracle.loop_block(case["x0"], host, bits, case["group"], 1, normalize=False)
    assert_close(got, ref, "block no-norm int%d" % bits)


@pytest.mark.parametrize("bits", [4, 2])
def test_block_full_width_decode(lib, bits):
    """D = 2048, FFN 8192, M = 1, L = 4 against the oracle.  The L2 is flushed
    first: iteration 1 reads the weights from HBM, the later ones from L2."""
    case = synth.block_case(1, bits, seed=0)
    blk, host = make_block(lib, case)
    flush_l2()
    got = run_gpu(lib, blk, case["x0"], 4)
    ref = oracle.loop_block(case["x0"], host, bits, case["group"], 4, normalize=True)
    assert_close(got, ref, "block D2048 int%d" % bits)


def test_block_split_invariant_bitwise(lib):
    """Running L1 then L - L1 iterations equals running L, bit for bit."""
    case = synth.block_case(3, 4, seed=40, D=256, F=512)
    blk, _ = make_block(lib, case)
    full = run_gpu(lib, blk, case["x0"], 6)
    mid = run_gpu(lib, blk, case["x0"], 2)
    rest = run_gpu(lib, blk, mid, 4)
    assert np.array_equal(full.view(np.uint32), rest.view(np.uint32))


def test_block_zero_iterations_is_noop(lib):
    case = synth.block_case(2, 4, seed=41, D=256, F=512)
    blk, _ = make_block(lib, case)
    got = run_gpu(lib, blk, case["x0"], 0)
    assert np.array_equal(got.view(np.uint32), case["x0"].view(np.uint32))


@pytest.mark.parametrize("bits", [4, 2])
def test_block_full_width_prefill(lib, bits):
    """D = 2048, FFN 8192, M = 128 (tensor-core path), L = 2, sampled rows."""
    case = synth.block_case(128, bits, seed=0)
    blk, host = make_block(lib, case)
    got = run_gpu(lib, blk, case["x0"], 2)
    rows = [0, 37, 127]
    ref = oracle.loop_block(case["x0"][rows], host, bits, case["group"], 2, normalize=True)
    assert_close(got[rows], ref, "block D2048 M128 int%d" % bits)

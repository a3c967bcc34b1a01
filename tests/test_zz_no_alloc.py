"""The allocation-free loop-block entry point.

Callers that cannot allocate device memory (a serving runtime with a fixed
memory budget, a plugin interface that only passes inputs and outputs) use
tl_loop_block_forward_static_scratch, whose intermediates live in a static
device array of the library.  Its results must match the caller-scratch entry
point within the parity tolerance, call after call.  This file is collected
last on purpose: the first call on a device also sets up the array address.
"""
import numpy as np
import pytest

import synth
from devmem import default_pool_high_watermark
from parity import assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _block(lib, case, rows):
    bits = case["bits"]
    proj = {}
    for name, (codes, s, z) in case["proj"].items():
        proj[name] = (lib.pack_weights(torch.from_numpy(codes).cuda(), bits), torch.from_numpy(s).cuda(),
                      torch.from_numpy(z).cuda())
    return lib.LoopBlock(proj, bits, case["group"], rows)


@pytest.mark.parametrize("bits,M,D,F,L", [(4, 1, 2048, 8192, 3), (2, 16, 256, 512, 4), (4, 64, 256, 512, 2)])
def test_static_scratch_matches_caller_scratch(lib, bits, M, D, F, L):
    case = synth.block_case(M, bits, seed=90 + M, D=D, F=F)
    blk = _block(lib, case, M)
    x_ref = torch.from_numpy(case["x0"].copy()).cuda()
    lib.tl_loop_block_forward(x_ref, blk, L)
    torch.cuda.synchronize()
    ref = x_ref.cpu().numpy()
    for call in range(2):  # two calls in a row share (and reuse) the static array
        x = torch.from_numpy(case["x0"].copy()).cuda()
        torch.cuda.synchronize()
        default_pool_high_watermark(reset=True)
        lib.tl_loop_block_forward_static_scratch(x, blk, L)
        torch.cuda.synchronize()
        # nothing came from the device's stream-ordered pool (the library's
        # sources hold no allocation call at all: tests/test_abi.py)
        assert default_pool_high_watermark() == 0
        lib.tl_check_status()
        assert_close(x.cpu().numpy(), ref, "static scratch call %d int%d M%d" % (call, bits, M))


def test_static_scratch_rejects_oversized_problem(lib):
    case = synth.block_case(1, 4, seed=99, D=256, F=512)
    blk = _block(lib, case, 1)
    blk._c.D = 2048
    blk._c.up.N = 8192
    x = torch.zeros((200, 2048), dtype=torch.float32, device="cuda")  # 200 rows need ~7.4 MB
    with pytest.raises(lib.TLQError, match="static scratch holds"):
        lib.tl_loop_block_forward_static_scratch(x, blk, 1)

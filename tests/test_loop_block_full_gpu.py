"""GPU parity of the loop blocks at the full looped-block workload: D = 2048,
FFN 8192, the ReLU block (four weights) and the five-weight SwiGLU block,
INT4 (group 128) and INT2 (group 64), L = 4, 8 and 16 iterations, at M = 1
(every element) and M = 128 (16 whole sampled rows; the tensor-core path).

Two checks per case:
  * iteration by iteration: the GPU's update of iteration l (x_{l+1} - x_l)
    against the oracle's update from the GPU's own x_l, at the GEMM bar;
  * the whole trajectory: x_L from x0 on the GPU against the oracle's x_L
    from x0, at the GEMM bar scaled by parity.trajectory_scale(L).
Rows of the block are independent (a per-row norm, row-wise GEMMs, a row-wise
residual), so the oracle runs only the sampled rows.  The GPU reaches x_l one
iteration per call; running L1 then L - L1 iterations equals L at once, bit
for bit ("Warm-start mid-loop", internal flow, "Extend loop": the block is
re-run in place on the residual), which the other block tests check.
"""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_close, sample_rows, trajectory_scale

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LS = (4, 8, 16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _blocks(lib, kind, case):
    bits = case["bits"]
    proj, host = {}, {}
    for name, (codes, s, z) in case["proj"].items():
        proj[name] = (lib.pack_weights(_dev(codes), bits), _dev(s), _dev(z))
        host[name] = (oracle.pack(codes, bits), s, z)
    cls = lib.LoopBlock if kind == "relu" else lib.SwiGLUBlock
    return cls(proj, bits, case["group"], case["M"]), host


@pytest.mark.parametrize("kind", ["relu", "swiglu"])
@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("M", [1, 128])
def test_loop_block_full_workload(lib, kind, bits, M):
    make = synth.block_case if kind == "relu" else synth.swiglu_block_case
    run = oracle.loop_block if kind == "relu" else oracle.loop_block_swiglu
    case = make(M, bits, seed=3)
    group = case["group"]
    blk, host = _blocks(lib, kind, case)
    rows = sample_rows(M, 16, np.random.default_rng(M + bits))

    # the GPU trajectory, one iteration per call
    x = _dev(case["x0"].copy())
    traj = [case["x0"][rows].astype(np.float64)]
    for _ in range(LS[-1]):
        blk.forward(x, 1)
        torch.cuda.synchronize()
        lib.tl_check_status()
        traj.append(x.cpu().numpy()[rows].astype(np.float64))
    assert np.all(np.isfinite(traj[-1]))

    # iteration by iteration, from the GPU's own inputs
    for l in range(LS[-1]):
        xl = traj[l].astype(np.float32)
        ref_update = run(xl, host, bits, group, 1).astype(np.float64) - traj[l]
        assert_close(traj[l + 1] - traj[l], ref_update, "%s int%d M%d iteration %d" % (kind, bits, M, l + 1))

    # whole trajectories from x0; fresh L-iteration calls give the same bits
    ref, done = case["x0"][rows], 0
    for L in LS:
        ref = run(ref, host, bits, group, L - done)
        done = L
        xL = _dev(case["x0"].copy())
        blk.forward(xL, L)
        torch.cuda.synchronize()
        got = xL.cpu().numpy()[rows]
        assert np.array_equal(got.view(np.uint32), traj[L].astype(np.float32).view(np.uint32)), L
        assert_close(got, ref, "%s int%d M%d L%d" % (kind, bits, M, L), scale=trajectory_scale(L))

"""Device-memory helpers for the GPU tests: the high watermark of the
device's default stream-ordered memory pool (what cudaMallocAsync draws
from), read through the CUDA runtime the library itself loaded, and an L2
flush."""
import ctypes

_POOL_USED_MEM_HIGH = 8  # cudaMemPoolAttrUsedMemHigh


def _cudart():
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    raise OSError("libcudart not found")


def default_pool_high_watermark(reset=False):
    """Bytes of the default pool that were in use at once since the last
    reset (reset=True sets the watermark back to zero first)."""
    import torch

    rt = _cudart()
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), torch.cuda.current_device()) == 0
    v = ctypes.c_uint64(0)
    if reset:
        assert rt.cudaMemPoolSetAttribute(pool, _POOL_USED_MEM_HIGH, ctypes.byref(v)) == 0
    assert rt.cudaMemPoolGetAttribute(pool, _POOL_USED_MEM_HIGH, ctypes.byref(v)) == 0
    return v.value


def flush_l2(nbytes=256 << 20):
    """Write a buffer twice the size of GB300's L2, so that whatever a kernel
    reads next comes from HBM unless that kernel's own earlier reads put it in
    L2."""
    import torch

    junk = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
    junk.fill_(1)
    torch.cuda.synchronize()
    del junk

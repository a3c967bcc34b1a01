// Measurement helper: the L2 read bandwidth that bounds the loop block, whose
// packed weights fit in L2 and are re-read every iteration.  Not part of the
// layer; the benchmark divides the loop block's effective bandwidth by it.
#include "common.cuh"

namespace tlq {
namespace {

constexpr int kProbeThreads = 512;

__device__ __forceinline__ uint4 ldg_cg_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Every thread reads 16-byte words of buf (L2 only, no L1) in a grid-stride
// loop, `reps` passes over the whole buffer, and folds them into one word so
// that no load can be dropped.
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4* __restrict__ buf, size_t n16, int reps,
                                                                    uint32_t* __restrict__ sink) {
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  uint32_t acc = 0;
  for (int r = 0; r < reps; ++r) {
    size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
#pragma unroll 4
    for (; i < n16; i += stride) {
      const uint4 v = ldg_cg_v4(buf + i);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  sink[(size_t)blockIdx.x * kProbeThreads + threadIdx.x] = acc;
}

}  // namespace
}  // namespace tlq

using namespace tlq;

extern "C" tlq_status tl_probe_read_bandwidth(const void* buf, size_t bytes, int reps, uint32_t* sink,
                                              void* stream) {
  clear_error();
  if (!buf || !sink) return set_error(TLQ_EINVAL, "tl_probe_read_bandwidth: null pointer");
  if (bytes < 16 || bytes % 16 || (reinterpret_cast<uintptr_t>(buf) & 15))
    return set_error(TLQ_EINVAL, "tl_probe_read_bandwidth: bytes=%zu (a positive multiple of 16, 16-byte aligned)",
                     bytes);
  if (reps < 1) return set_error(TLQ_EINVAL, "tl_probe_read_bandwidth: reps=%d (must be >= 1)", reps);
  const unsigned blocks = (unsigned)(2 * device_info().sms);
  read_probe_kernel<<<blocks, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), bytes / 16, reps, sink);
  return cuda_error(cudaGetLastError(), "tl_probe_read_bandwidth: launch");
}

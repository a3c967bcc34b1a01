// Weight packing / unpacking, the loop block's RMS pre-norm, and the bounded
// wait self-test kernel.
#include "common.cuh"

namespace tlq {

__device__ uint32_t g_status = 0;
__device__ uint32_t g_status_where = 0;

namespace {

// One thread per packed word.  Packing follows "beta-Informed Deployment
// Features", CTX-TIER, "Details of the shipped kernel": K/2 bytes per INT4 row,
// K/4 bytes per INT2 row; code j of a word at bits [bits*j, bits*j + bits).
template <int BITS>
__global__ void pack_kernel(const uint8_t* __restrict__ codes, uint32_t* __restrict__ W, int N, int K) {
  constexpr int CPW = 32 / BITS;
  const int wpr = K / CPW;
  const size_t total = (size_t)N * wpr;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t n = i / wpr, w = i - n * wpr;
    const uint8_t* src = codes + n * (size_t)K + w * CPW;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < CPW; ++j) word |= ((uint32_t)src[j] & ((1u << BITS) - 1u)) << (BITS * j);
    W[i] = word;
  }
}

template <int BITS>
__global__ void unpack_kernel(const uint32_t* __restrict__ W, uint8_t* __restrict__ codes, int N, int K) {
  constexpr int CPW = 32 / BITS;
  const int wpr = K / CPW;
  const size_t total = (size_t)N * wpr;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t n = i / wpr, w = i - n * wpr;
    const uint32_t word = W[i];
    uint8_t* dst = codes + n * (size_t)K + w * CPW;
#pragma unroll
    for (int j = 0; j < CPW; ++j) dst[j] = (uint8_t)((word >> (BITS * j)) & ((1u << BITS) - 1u));
  }
}

// h[m][:] = fp16( x[m][:] * (1 / sqrt(mean(x^2) + 1e-5)) ) or fp16(x) when
// normalize == 0.  One CTA per row; fixed-order reduction (deterministic).
// The residual is FP32 and the norm output FP16 ("Model", "VRAM cost",
// Runtime buffers: buf.main FP32, buf.norm FP16).
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float* __restrict__ x, __half* __restrict__ h,
                                                                int D, int normalize) {
  __shared__ float warp_sums[kNormThreads / 32];
  __shared__ float inv_s;
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();  // x is written by the preceding kernel
  const float* xr = x + (size_t)blockIdx.x * D;
  __half* hr = h + (size_t)blockIdx.x * D;
  float inv = 1.f;
  if (normalize) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < D; i += kNormThreads) ss = fmaf(xr[i], xr[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < kNormThreads / 32; ++w) t += warp_sums[w];
      inv_s = 1.0f / sqrtf(t / (float)D + 1e-5f);
    }
    __syncthreads();
    inv = inv_s;
  }
  for (int i = threadIdx.x; i < D; i += kNormThreads) hr[i] = __float2half_rn(normalize ? xr[i] * inv : xr[i]);
}

// Waits on an mbarrier that nothing ever arrives at, with a short limit: the
// wait must give up, record TLQ_ETIMEOUT and return.
__global__ void timeout_probe_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait_ns(&bar, 0, limit_ns, 0x900);
}

int grid_for(size_t work, int threads) {
  size_t b = (work + threads - 1) / threads;
  const size_t cap = (size_t)device_info().sms * 8;
  if (b > cap) b = cap;
  return (int)(b ? b : 1);
}

}  // namespace

tlq_status launch_pack(const uint8_t* codes, uint32_t* W, int N, int K, int bits, cudaStream_t stream) {
  const size_t words = (size_t)N * (K * bits / 32);
  const int th = 256;
  if (bits == 4)
    pack_kernel<4><<<grid_for(words, th), th, 0, stream>>>(codes, W, N, K);
  else
    pack_kernel<2><<<grid_for(words, th), th, 0, stream>>>(codes, W, N, K);
  return cuda_error(cudaGetLastError(), "pack: launch");
}

tlq_status launch_unpack(const uint32_t* W, uint8_t* codes, int N, int K, int bits, cudaStream_t stream) {
  const size_t words = (size_t)N * (K * bits / 32);
  const int th = 256;
  if (bits == 4)
    unpack_kernel<4><<<grid_for(words, th), th, 0, stream>>>(W, codes, N, K);
  else
    unpack_kernel<2><<<grid_for(words, th), th, 0, stream>>>(W, codes, N, K);
  return cuda_error(cudaGetLastError(), "unpack: launch");
}

tlq_status launch_rmsnorm(const float* x, __half* h, int M, int D, int normalize, cudaStream_t stream) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)M, 1, 1);
  lc.blockDim = dim3(kNormThreads, 1, 1);
  lc.stream = stream;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = &at;
  lc.numAttrs = pdl_enabled() ? 1 : 0;
  return cuda_error(cudaLaunchKernelEx(&lc, rmsnorm_kernel, x, h, D, normalize), "rmsnorm: launch");
}

tlq_status launch_timeout_probe(uint32_t limit_us, cudaStream_t stream) {
  timeout_probe_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull);
  return cuda_error(cudaGetLastError(), "timeout probe: launch");
}

}  // namespace tlq

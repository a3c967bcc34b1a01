// FP16 body of a quantized weight: every weight dequantized and rounded once
// to FP16, the dense copy kept by the FP16 body cache ("Model", section "VRAM
// cost": the opt-in FP16 body cache, about 3x the weight memory).  Used as a
// comparison point for the quantized GEMM: a dense FP16 GEMM on the body.
//
// body[n][k] = fp16_RNE((q - z) * s), +0 for an exact zero.  In binary32 the
// exact value is p + nzs with p = q * s and nzs = -(z * s), both exact (a
// 4-bit code or an 11-bit FP16 significand times an 11-bit one).  The sum is
// rounded once (hi) and TwoSum gives its exact error; when the error is not
// zero, hi is replaced by its odd neighbour on the error's side (round to
// odd), and rounding that to FP16 (13 fewer bits) gives the FP16 rounding of
// the exact value (double rounding through round-to-odd is innocuous when the
// wider format has at least two more bits; Boldo and Melquiond, "When double
// rounding is odd", 2005).
#include "common.cuh"

namespace tlq {

namespace {

constexpr int kBodyThreads = 256;

// Exactly (float)c for a code c < 2^23: the code in the significand of 2^23.
__device__ __forceinline__ float code_float(uint32_t c) { return __uint_as_float(0x4B000000u | c) - 8388608.0f; }

__device__ __forceinline__ __half body_half(float q, float s, float nzs) {
  const float p = __fmul_rn(q, s);  // exact
  const float hi = __fadd_rn(p, nzs);
  // TwoSum: hi + err == p + nzs exactly
  const float bb = __fsub_rn(hi, p);
  const float err = __fadd_rn(__fsub_rn(p, __fsub_rn(hi, bb)), __fsub_rn(nzs, bb));
  uint32_t b = __float_as_uint(hi);
  if (err != 0.0f && !(b & 1u)) b += ((__float_as_uint(err) ^ b) >> 31) ? 0xFFFFFFFFu : 1u;  // round to odd
  return __float2half_rn(__uint_as_float(b));  // an exact zero is hi = +0
}

// One thread per packed word: 32/BITS weights of one group.
template <int BITS>
__global__ void __launch_bounds__(kBodyThreads) body_kernel(const uint32_t* __restrict__ W, const __half* __restrict__ S,
                                                           const __half* __restrict__ Z, __half* __restrict__ out,
                                                           int N, int K, int group) {
  constexpr int CPW = 32 / BITS;
  const int wpr = K / CPW, G = K / group;
  const size_t total = (size_t)N * wpr;
  for (size_t i = (size_t)blockIdx.x * kBodyThreads + threadIdx.x; i < total; i += (size_t)gridDim.x * kBodyThreads) {
    const size_t n = i / wpr;
    const int w = (int)(i - n * wpr);
    const size_t gi = n * G + (size_t)(w * CPW) / group;
    const uint32_t x = __ldg(W + i);
    const float s = __half2float(S[gi]), z = __half2float(Z[gi]);
    const float nzs = -__fmul_rn(z, s);  // exact
    uint32_t h[CPW / 2];
#pragma unroll
    for (int j = 0; j < CPW / 2; ++j) {
      const __half a = body_half(code_float((x >> (BITS * 2 * j)) & ((1u << BITS) - 1u)), s, nzs);
      const __half b = body_half(code_float((x >> (BITS * (2 * j + 1))) & ((1u << BITS) - 1u)), s, nzs);
      h[j] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + n * (size_t)K + (size_t)w * CPW);
#pragma unroll
    for (int j = 0; j < CPW / 8; ++j) dst[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
  }
}

}  // namespace

tlq_status launch_body(const uint32_t* W, const uint16_t* s, const uint16_t* z, uint16_t* out, int N, int K, int bits,
                       int group, cudaStream_t stream) {
  const size_t words = (size_t)N * (K * bits / 32);
  size_t blocks = (words + kBodyThreads - 1) / kBodyThreads;
  const size_t cap = (size_t)device_info().sms * 8;
  if (blocks > cap) blocks = cap;
  const __half* S = reinterpret_cast<const __half*>(s);
  const __half* Z = reinterpret_cast<const __half*>(z);
  __half* O = reinterpret_cast<__half*>(out);
  if (bits == 4)
    body_kernel<4><<<(unsigned)blocks, kBodyThreads, 0, stream>>>(W, S, Z, O, N, K, group);
  else
    body_kernel<2><<<(unsigned)blocks, kBodyThreads, 0, stream>>>(W, S, Z, O, N, K, group);
  return cuda_error(cudaGetLastError(), "body: launch");
}

}  // namespace tlq

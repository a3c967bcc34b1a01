// INT4 -> INT2 group re-quantization: the weight conversion of the
// context-length tier switch ("beta-Informed Deployment Features", CTX-TIER,
// "Details of the shipped kernel").
//
// Per quantization group: dequantize w = (q4 - z4) * s4, take min and max,
// fit s2 = fp16((max - min) / 3) (1.0 when that is zero) and
// z2 = fp16(-min / s2) (the page's zero = min in this library's (q - z) * s
// form), and round every weight to q2 = clamp(rint(w / s2 + z2), 0, 3).
// Every floating-point step is binary32 with round-to-nearest-even, in that
// order, so the codes, s2 and z2 are bit-identical to a scalar evaluation.
//
// Two facts make the kernel a byte-SIMD stream instead of a per-weight divide:
//  * inside a group, w depends on the 4-bit code only, and c -> w(c) is
//    monotone (each rounded step is monotone; the direction is the sign of
//    s4).  So min/max of w over the group are w(cmin) and w(cmax), and
//  * q2(c) = f(w(c)) is monotone in c as well, so it is fixed by three integer
//    thresholds C_j = #{c in 0..15 : q2(c) < j}: q2 >= j iff c' >= C_j, with
//    c' = c (s4 > 0) or 15 - c (s4 < 0).  The 16 values q2(c) are evaluated
//    with the exact scalar formula, spread over the lanes of the group.
// The one exception to monotonicity is s4 = +-0: every w is a zero whose sign
// follows (c - z4), and the scalar min/max keep the group's first weight; the
// kernel then takes the first code of the group.
//
// Layout: the [N][K] codes are viewed as N*K/group consecutive groups (K is a
// multiple of group).  A group of `group` codes is T = group/32 chunks of 32
// codes (16 bytes of INT4 in, 8 bytes of INT2 out); P lanes (a power of two,
// P >= T up to 32) work on one group, lane l on chunks l, l+P, ...
#include "common.cuh"

namespace tlq {

namespace {

constexpr int kRqThreads = 256;

// w(c) = (c - z) * s, each step rounded (no contraction into an FMA).
__device__ __forceinline__ float rq_dequant(uint32_t c, float z, float s) {
  return __fmul_rn(__fsub_rn(static_cast<float>(c), z), s);
}

// q2 of one dequantized weight: clamp(rint(w / sh + zh), 0, 3).  t can be
// +-inf (zh overflows FP16 when the group's range is tiny next to its
// offset), never NaN; the clamp maps it like the scalar compare-and-assign.
__device__ __forceinline__ uint32_t rq_code(float w, float sh, float zh) {
  const float t = __fadd_rn(__fdiv_rn(w, sh), zh);
  const float r = fminf(fmaxf(rintf(t), 0.0f), 3.0f);
  return static_cast<uint32_t>(r);
}

// Byte-wise min / max accumulation of the 8 codes of one INT4 word.
__device__ __forceinline__ void rq_minmax(uint32_t x, uint32_t& mn, uint32_t& mx) {
  const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
  mn = __vminu4(mn, __vminu4(lo, hi));
  mx = __vmaxu4(mx, __vmaxu4(lo, hi));
}

// The 8 codes of one INT4 word -> 16 bits of INT2 codes (code j at bits 2j).
// b1..b3 hold (0x80 - C_j) in every byte: adding one to a byte of codes 0..15
// sets its bit 7 exactly when the code is >= C_j, with no carry out of the
// byte.  The three tests form a thermometer (C1 <= C2 <= C3), so q2's bit 1
// is test 2 and its bit 0 the parity of the three.
__device__ __forceinline__ uint32_t rq_pack8(uint32_t x, uint32_t flip, uint32_t b1, uint32_t b2, uint32_t b3) {
  const uint32_t lo = (x & 0x0F0F0F0Fu) ^ flip;          // codes 0, 2, 4, 6 (byte i = code 2i)
  const uint32_t hi = ((x >> 4) & 0x0F0F0F0Fu) ^ flip;   // codes 1, 3, 5, 7
  const uint32_t l1 = lo + b1, l2 = lo + b2, l3 = lo + b3;
  const uint32_t h1 = hi + b1, h2 = hi + b2, h3 = hi + b3;
  const uint32_t L0 = (l1 ^ l2 ^ l3) & 0x80808080u, L1 = l2 & 0x80808080u;
  const uint32_t H0 = (h1 ^ h2 ^ h3) & 0x80808080u, H1 = h2 & 0x80808080u;
  // byte i: bits 0..3 = q2(code 2i) | q2(code 2i+1) << 2
  uint32_t n = (L0 >> 7) | (L1 >> 6) | (H0 >> 5) | (H1 >> 4);
  n = (n | (n >> 4)) & 0x00FF00FFu;
  return (n | (n >> 8)) & 0x0000FFFFu;
}

// ONE: every lane holds at most one chunk (T <= 32), kept in registers
// between the two passes; otherwise lanes loop and re-read their chunks.
template <bool ONE>
__global__ void __launch_bounds__(kRqThreads) requant_kernel(const uint4* __restrict__ W4,
                                                             const uint16_t* s4, const uint16_t* z4,
                                                             uint2* __restrict__ W2, uint16_t* s2, uint16_t* z2,
                                                             long long ngroups, int T, int lg2P) {
  const int P = 1 << lg2P;
  const long long t = static_cast<long long>(blockIdx.x) * kRqThreads + threadIdx.x;
  const long long gi = t >> lg2P;
  if (gi >= ngroups) return;  // whole P-lane sets leave together (P divides 32)
  const int l = static_cast<int>(t & (P - 1));
  const int lane = threadIdx.x & 31;
  const int leader = lane & ~(P - 1);
  const unsigned mask = P == 32 ? 0xffffffffu : (((1u << P) - 1u) << leader);
  const uint4* src = W4 + gi * T;

  // Lane 0 of the set reads s4 / z4 (and later writes s2 / z2, which may
  // alias them); the others receive the values by shuffle.
  uint32_t sz = 0, first = 0;
  uint4 v = make_uint4(0, 0, 0, 0);
  uint32_t mn = 0x0F0F0F0Fu, mx = 0u;
  if (ONE) {
    if (l < T) {
      v = __ldg(src + l);
      rq_minmax(v.x, mn, mx);
      rq_minmax(v.y, mn, mx);
      rq_minmax(v.z, mn, mx);
      rq_minmax(v.w, mn, mx);
    }
  } else {
    for (int ch = l; ch < T; ch += P) {
      const uint4 u = __ldg(src + ch);
      if (ch == 0) v = u;
      rq_minmax(u.x, mn, mx);
      rq_minmax(u.y, mn, mx);
      rq_minmax(u.z, mn, mx);
      rq_minmax(u.w, mn, mx);
    }
  }
  if (l == 0) {
    sz = static_cast<uint32_t>(s4[gi]) | (static_cast<uint32_t>(z4[gi]) << 16);
    first = v.x & 15u;
  }
  // cmin in byte 0, 15 - cmax in byte 1: one byte-wise min reduction.
  uint32_t cmn = min(min(mn & 0xFFu, (mn >> 8) & 0xFFu), min((mn >> 16) & 0xFFu, mn >> 24));
  uint32_t cmx = max(max(mx & 0xFFu, (mx >> 8) & 0xFFu), max((mx >> 16) & 0xFFu, mx >> 24));
  uint32_t red = cmn | ((15u - cmx) << 8);
  for (int o = P >> 1; o > 0; o >>= 1) red = __vminu4(red, __shfl_xor_sync(mask, red, o));
  cmn = red & 0xFFu;
  cmx = 15u - ((red >> 8) & 0xFFu);
  sz = __shfl_sync(mask, sz, leader);
  first = __shfl_sync(mask, first, leader);

  const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(sz & 0xFFFFu)));
  const float z = __half2float(__ushort_as_half(static_cast<unsigned short>(sz >> 16)));
  float lo, hi;
  if (s == 0.0f) {
    lo = hi = rq_dequant(first, z, s);
  } else {
    const float a = rq_dequant(cmn, z, s), b = rq_dequant(cmx, z, s);
    lo = fminf(a, b);
    hi = fmaxf(a, b);
  }
  __half sb = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
  if (__half2float(sb) == 0.0f) sb = __float2half_rn(1.0f);
  const float sh = __half2float(sb);
  const __half zb = __float2half_rn(__fdiv_rn(-lo, sh));
  const float zh = __half2float(zb);

  // Threshold counts C_j = #{c : q2(c) < j}, one byte each, summed over lanes.
  uint32_t cnt = 0;
  for (uint32_t c = static_cast<uint32_t>(l); c < 16u; c += static_cast<uint32_t>(P)) {
    const uint32_t q = rq_code(rq_dequant(c, z, s), sh, zh);
    cnt += (q < 1u ? 1u : 0u) | (q < 2u ? 0x100u : 0u) | (q < 3u ? 0x10000u : 0u);
  }
  for (int o = P >> 1; o > 0; o >>= 1) cnt += __shfl_xor_sync(mask, cnt, o);
  const uint32_t b1 = (0x80u - (cnt & 0xFFu)) * 0x01010101u;
  const uint32_t b2 = (0x80u - ((cnt >> 8) & 0xFFu)) * 0x01010101u;
  const uint32_t b3 = (0x80u - ((cnt >> 16) & 0xFFu)) * 0x01010101u;
  const uint32_t flip = s < 0.0f ? 0x0F0F0F0Fu : 0u;

  uint2* dst = W2 + gi * T;
  if (ONE) {
    if (l < T)
      dst[l] = make_uint2(rq_pack8(v.x, flip, b1, b2, b3) | (rq_pack8(v.y, flip, b1, b2, b3) << 16),
                          rq_pack8(v.z, flip, b1, b2, b3) | (rq_pack8(v.w, flip, b1, b2, b3) << 16));
  } else {
    for (int ch = l; ch < T; ch += P) {
      const uint4 u = __ldg(src + ch);
      dst[ch] = make_uint2(rq_pack8(u.x, flip, b1, b2, b3) | (rq_pack8(u.y, flip, b1, b2, b3) << 16),
                           rq_pack8(u.z, flip, b1, b2, b3) | (rq_pack8(u.w, flip, b1, b2, b3) << 16));
    }
  }
  if (l == 0) {
    s2[gi] = __half_as_ushort(sb);
    z2[gi] = __half_as_ushort(zb);
  }
}

}  // namespace

tlq_status launch_requant(const uint32_t* W4, const uint16_t* s4, const uint16_t* z4, uint32_t* W2, uint16_t* s2,
                          uint16_t* z2, int N, int K, int group, cudaStream_t stream) {
  const long long ngroups = static_cast<long long>(N) * (K / group);
  const int T = group / 32;
  int lg2P = 0;
  while ((1 << lg2P) < T && lg2P < 5) ++lg2P;
  const long long threads = ngroups << lg2P;
  const long long blocks = (threads + kRqThreads - 1) / kRqThreads;
  if (blocks > 0x7fffffffLL) return set_error(TLQ_EINVAL, "tl_requant_int4_to_int2: N*K too large");
  const uint4* src = reinterpret_cast<const uint4*>(W4);
  uint2* dst = reinterpret_cast<uint2*>(W2);
  if (T <= 32)
    requant_kernel<true><<<static_cast<unsigned>(blocks), kRqThreads, 0, stream>>>(src, s4, z4, dst, s2, z2, ngroups,
                                                                                   T, lg2P);
  else
    requant_kernel<false><<<static_cast<unsigned>(blocks), kRqThreads, 0, stream>>>(src, s4, z4, dst, s2, z2, ngroups,
                                                                                    T, lg2P);
  return cuda_error(cudaGetLastError(), "requant: launch");
}

}  // namespace tlq

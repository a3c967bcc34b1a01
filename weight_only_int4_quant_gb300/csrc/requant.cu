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
// Inside a group w depends on the 4-bit code only, so the kernel evaluates the
// exact scalar formula for the 16 codes once per group and then maps codes
// with a table, not a divide per weight:
//  * c -> w(c) is monotone (each rounded step is monotone; the direction is
//    the sign of s4), so min/max of w over the group are w(cmin) and w(cmax)
//    of the smallest and largest code present;
//  * the table q2(c), c = 0..15, is held in four registers as byte pools of
//    two byte permutes (see rq_pack16), which translate four codes each.
// The one exception to monotonicity is s4 = +-0: every w is a zero whose sign
// follows (c - z4), and the scalar min/max keep the group's first weight; the
// kernel then takes the first code of the group.
//
// Layout: the [N][K] codes of a weight are N*K/group consecutive groups (K is
// a multiple of group); the groups of all weights of one launch are numbered
// one after the other.  One thread converts one group: T = group/32 chunks of
// 32 codes (16 bytes of INT4 in, 8 bytes of INT2 out each), so a group's
// per-group work (min/max reduction, two divides for s2 / z2, sixteen for the
// code map) is done once, without shuffles.  The grid is persistent (the
// resident CTAs of every SM, one launch for all weights): each thread strides
// over the groups and, for group sizes up to 128, loads its next group's
// words before it converts the current one.
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

// Byte-wise compare of two vectors of bytes 0..15: 0xFF where a >= b, else 0.
// (a | 0x80) - b keeps every byte in 0x71..0x8F (no borrow between bytes) and
// sets its bit 7 exactly when a >= b; a byte permute in sign mode widens it.
__device__ __forceinline__ uint32_t rq_ge_mask(uint32_t a, uint32_t b) {
  uint32_t m;
  // prmt selector nibbles 8..B: bytes 0..3 of the source, each replaced by
  // copies of its sign bit (PTX "prmt", default mode)
  asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"((a | 0x80808080u) - b));
  return m;
}

// Byte-wise min and max of two vectors of bytes 0..15.
__device__ __forceinline__ void rq_minmax2(uint32_t a, uint32_t b, uint32_t& mn, uint32_t& mx) {
  const uint32_t m = rq_ge_mask(a, b);
  mx = b ^ ((a ^ b) & m);
  mn = a ^ ((a ^ b) & m);
}
__device__ __forceinline__ uint32_t rq_min(uint32_t a, uint32_t b) { return a ^ ((a ^ b) & rq_ge_mask(a, b)); }
__device__ __forceinline__ uint32_t rq_max(uint32_t a, uint32_t b) { return b ^ ((a ^ b) & rq_ge_mask(a, b)); }

// Byte-wise min and max over the 32 codes of one chunk (4 INT4 words).
__device__ __forceinline__ void rq_chunk_minmax(const uint4& v, uint32_t& mn, uint32_t& mx) {
  uint32_t n0, x0, n1, x1, n2, x2, n3, x3;
  rq_minmax2(v.x & 0x0F0F0F0Fu, (v.x >> 4) & 0x0F0F0F0Fu, n0, x0);
  rq_minmax2(v.y & 0x0F0F0F0Fu, (v.y >> 4) & 0x0F0F0F0Fu, n1, x1);
  rq_minmax2(v.z & 0x0F0F0F0Fu, (v.z >> 4) & 0x0F0F0F0Fu, n2, x2);
  rq_minmax2(v.w & 0x0F0F0F0Fu, (v.w >> 4) & 0x0F0F0F0Fu, n3, x3);
  mn = rq_min(rq_min(n0, n1), rq_min(n2, n3));
  mx = rq_max(rq_max(x0, x1), rq_max(x2, x3));
}

// Byte permute (PTX prmt, default mode): byte i of the result is byte
// (sel_i & 7) of {lo, hi} (lo = bytes 0..3), or copies of that byte's bit 7
// when sel_i & 8.  sel_i is nibble i of `sel`, so the low 16 bits of an INT4
// word select with its first four codes.
__device__ __forceinline__ uint32_t rq_prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
  return r;
}

// Code table as byte pools.  For code c < 8: byte c of pool A holds bit 0 of
// q2(c) in bit 0, byte c of pool B bit 1 of q2(c) in bit 1.  For c >= 8 the
// selector nibble has bit 3 set, the permute copies bit 7 of byte c - 8, and
// that bit holds bit 0 (pool A) or bit 1 (pool B) of q2(c).  So for every
// code, (A & 1) | (B & 2) of its result byte is q2(c).
struct RqPools {
  uint32_t a0, a1, b0, b1;
};

// Four codes (the low 16 bits of sel) -> bytes q2(c_i), i = 0..3.
__device__ __forceinline__ uint32_t rq_lookup4(const RqPools& t, uint32_t sel) {
  return (rq_prmt(t.a0, t.a1, sel) & 0x01010101u) | (rq_prmt(t.b0, t.b1, sel) & 0x02020202u);
}

// Bytes q_0..q_3 (each 0..3) -> q_0 | q_1 << 2 | q_2 << 4 | q_3 << 6 in the
// top byte: the multiplier moves byte i (bit 8i) up by 24 - 6i; the other
// products land above bit 31 or sum to less than 2^24 below bit 24.
__device__ __forceinline__ uint32_t rq_compact4(uint32_t r) { return r * 0x01041040u; }

// Two INT4 words (16 codes) -> one INT2 word, code j at bits 2j.
__device__ __forceinline__ uint32_t rq_pack16(uint32_t x0, uint32_t x1, const RqPools& t) {
  const uint32_t m0 = rq_compact4(rq_lookup4(t, x0)), m1 = rq_compact4(rq_lookup4(t, x0 >> 16));
  const uint32_t m2 = rq_compact4(rq_lookup4(t, x1)), m3 = rq_compact4(rq_lookup4(t, x1 >> 16));
  return __byte_perm(__byte_perm(m0, m1, 0x0073), __byte_perm(m2, m3, 0x0073), 0x5410);
}

// One weight of a launch; gstart = number of groups of the weights before it.
struct RqProblem {
  const uint4* W4;
  const uint16_t* s4;
  const uint16_t* z4;
  uint2* W2;
  uint16_t* s2;
  uint16_t* z2;
  long long gstart;
};

struct RqLaunch {
  RqProblem p[kMaxRequantProblems];
  int count;
  long long ngroups;  // all weights
  int T;  // chunks of 32 codes per group
};

// The problem holding group g, at or after problem p (groups are visited in
// increasing order by each thread).
__device__ __forceinline__ int rq_advance(const RqLaunch& L, int p, long long g) {
#pragma unroll 1
  while (p + 1 < L.count && g >= L.p[p + 1].gstart) ++p;
  return p;
}

// A chunk of 32 codes from src: through the read-only path from global
// memory, or (GENERIC) a plain load through a generic address (the in-place
// kernel's shared-memory staging).
template <bool GENERIC>
__device__ __forceinline__ uint4 rq_load(const uint4* src) {
  if constexpr (GENERIC) return *src;
  else return __ldg(src);
}

// Converts one group held in v[0..TC) (TC > 0) or re-read from src (TC == 0,
// T chunks).  sz = s4 | z4 << 16.
template <int TC, bool GENERIC = false>
__device__ __forceinline__ void rq_group(const uint4* v, const uint4* __restrict__ src, int T, uint32_t sz,
                                         uint2* __restrict__ dst, uint16_t* s2, uint16_t* z2) {
  const int nch = TC > 0 ? TC : T;
  uint32_t mn = 0x0F0F0F0Fu, mx = 0u, first;
  if (TC > 0) {
#pragma unroll
    for (int i = 0; i < (TC > 0 ? TC : 1); ++i) {
      uint32_t a, b;
      rq_chunk_minmax(v[i], a, b);
      mn = rq_min(mn, a);
      mx = rq_max(mx, b);
    }
    first = v[0].x & 15u;
  } else {
    first = rq_load<GENERIC>(src).x & 15u;
#pragma unroll 1
    for (int i = 0; i < nch; ++i) {
      uint32_t a, b;
      rq_chunk_minmax(rq_load<GENERIC>(src + i), a, b);
      mn = rq_min(mn, a);
      mx = rq_max(mx, b);
    }
  }
  mn = rq_min(mn, mn >> 16);
  mn = rq_min(mn, mn >> 8);
  mx = rq_max(mx, mx >> 16);
  mx = rq_max(mx, mx >> 8);
  const uint32_t cmn = mn & 0xFFu, cmx = mx & 0xFFu;

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

  // The code table: q2(c) for c = 0..15 with the scalar formula.
  RqPools t = {0u, 0u, 0u, 0u};
#pragma unroll
  for (uint32_t c = 0; c < 16u; ++c) {
    const uint32_t q = rq_code(rq_dequant(c, z, s), sh, zh);
    const uint32_t sft = 8u * (c & 3u) + (c < 8u ? 0u : 7u);
    const uint32_t qa = (q & 1u) << sft, qb = (c < 8u ? (q & 2u) : (q >> 1)) << sft;
    if ((c & 7u) < 4u) {
      t.a0 |= qa;
      t.b0 |= qb;
    } else {
      t.a1 |= qa;
      t.b1 |= qb;
    }
  }

  if (TC > 0) {
#pragma unroll
    for (int i = 0; i < (TC > 0 ? TC : 1); ++i)
      dst[i] = make_uint2(rq_pack16(v[i].x, v[i].y, t), rq_pack16(v[i].z, v[i].w, t));
  } else {
#pragma unroll 1
    for (int i = 0; i < nch; ++i) {
      const uint4 u = rq_load<GENERIC>(src + i);
      dst[i] = make_uint2(rq_pack16(u.x, u.y, t), rq_pack16(u.z, u.w, t));
    }
  }
  *s2 = __half_as_ushort(sb);
  *z2 = __half_as_ushort(zb);
}

// TC = chunks per group known at compile time (2: group 64, 4: group 128),
// with the next group prefetched; 0 = any group size, chunks re-read.
template <int TC>
__global__ void __launch_bounds__(kRqThreads, 3) requant_kernel(const __grid_constant__ RqLaunch L) {
  const long long stride = static_cast<long long>(gridDim.x) * kRqThreads;
  long long g = static_cast<long long>(blockIdx.x) * kRqThreads + threadIdx.x;
  if (g >= L.ngroups) return;
  const int T = TC > 0 ? TC : L.T;
  int p = rq_advance(L, 0, g);
  constexpr int NV = TC > 0 ? TC : 1;
  uint4 vn[NV];
  uint32_t szn = 0;
  int pn = p;
  if (TC > 0) {
    const long long gl = g - L.p[p].gstart;
#pragma unroll
    for (int i = 0; i < NV; ++i) vn[i] = __ldg(L.p[p].W4 + gl * T + i);
    szn = static_cast<uint32_t>(L.p[p].s4[gl]) | (static_cast<uint32_t>(L.p[p].z4[gl]) << 16);
  }
#pragma unroll 1
  for (; g < L.ngroups; g += stride) {
    const RqProblem& pr = L.p[p];
    const long long gi = g - pr.gstart;
    uint4 v[NV];
    uint32_t sz;
    if (TC > 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = vn[i];
      sz = szn;
      const long long gn = g + stride;
      if (gn < L.ngroups) {  // the next group's words are in flight during this one
        pn = rq_advance(L, p, gn);
        const long long gl = gn - L.p[pn].gstart;
#pragma unroll
        for (int i = 0; i < NV; ++i) vn[i] = __ldg(L.p[pn].W4 + gl * T + i);
        szn = static_cast<uint32_t>(L.p[pn].s4[gl]) | (static_cast<uint32_t>(L.p[pn].z4[gl]) << 16);
      }
    } else {
      sz = static_cast<uint32_t>(pr.s4[gi]) | (static_cast<uint32_t>(pr.z4[gi]) << 16);
    }
    // s4 / z4 of this group were read above, before s2 / z2 (which may alias
    // them) are written.
    rq_group<TC>(v, pr.W4 + gi * T, T, sz, pr.W2 + gi * T, pr.s2 + gi, pr.z2 + gi);
    if (TC > 0) p = pn;
    else if (g + stride < L.ngroups) p = rq_advance(L, p, g + stride);
  }
}

// In place ("beta-Informed Deployment Features", CTX-TIER, "Details of the
// shipped kernel", storage reuse): W2 is W4 and the INT2 rows keep the INT4
// row stride (K/2 bytes), the second half of every row left as it was.  The
// INT2 bytes of group g land on bytes [g*group/4, (g+1)*group/4) of the row,
// which hold INT4 codes of groups below g only.  So one CTA per row converts
// the row's groups in chunks, in increasing order, staging each chunk's INT4
// words in shared memory before writing any of its INT2 words: every INT4
// byte is read before it can be overwritten.  The staging loads are plain
// L2 loads (the same kernel writes this memory).
constexpr int kIpThreads = 128;
constexpr int kIpStageBytes = 32768;

struct RqInPlaceLaunch {
  RqProblem p[kMaxRequantProblems];  // W2 and W4 address the same words
  long long rstart[kMaxRequantProblems];  // first row of each problem in the launch
  int G[kMaxRequantProblems];             // groups per row
  int count;
  int T;      // chunks of 32 codes per group
  int chunk;  // groups per staged pass
};

__global__ void __launch_bounds__(kIpThreads) requant_in_place_kernel(const __grid_constant__ RqInPlaceLaunch L) {
  extern __shared__ uint4 stage[];  // [chunk][T]
  const long long row = blockIdx.x;
  int p = 0;
#pragma unroll 1
  while (p + 1 < L.count && row >= L.rstart[p + 1]) ++p;
  const RqProblem& pr = L.p[p];
  const long long n = row - L.rstart[p];
  const int G = L.G[p], T = L.T;
  const uint4* src = pr.W4 + n * G * T;                       // the row's INT4 words, T chunks per group
  uint2* dst = pr.W2 + n * (long long)G * T * 2;              // the same row start (INT4 stride)
#pragma unroll 1
  for (int g0 = 0; g0 < G; g0 += L.chunk) {
    const int ng = min(L.chunk, G - g0);
    for (int i = threadIdx.x; i < ng * T; i += kIpThreads) stage[i] = __ldcg(src + (long long)g0 * T + i);
    __syncthreads();  // the chunk's INT4 words are staged before any of its INT2 words are written
    for (int j = threadIdx.x; j < ng; j += kIpThreads) {
      const long long gi = n * G + g0 + j;
      const uint32_t sz = static_cast<uint32_t>(pr.s4[gi]) | (static_cast<uint32_t>(pr.z4[gi]) << 16);
      rq_group<0, true>(nullptr, stage + j * T, T, sz, dst + (long long)(g0 + j) * T, pr.s2 + gi, pr.z2 + gi);
    }
    __syncthreads();  // the stage is read before the next chunk replaces it
  }
}

}  // namespace

tlq_status launch_requant_in_place(const RequantArgs* a, int count, int group, cudaStream_t stream) {
  RqInPlaceLaunch L = {};
  long long rows = 0;
  for (int i = 0; i < count; ++i) {
    L.p[i] = RqProblem{reinterpret_cast<const uint4*>(a[i].W4), a[i].s4, a[i].z4, reinterpret_cast<uint2*>(a[i].W2),
                       a[i].s2, a[i].z2, 0};
    L.rstart[i] = rows;
    L.G[i] = a[i].K / group;
    rows += a[i].N;
  }
  L.count = count;
  L.T = group / 32;
  L.chunk = kIpStageBytes / (L.T * 16);
  if (L.chunk < 1) L.chunk = 1;
  if (rows == 0) return TLQ_OK;
  if (rows > 0x7FFFFFFFll) return set_error(TLQ_EUNSUPPORTED, "requant in place: %lld rows in one launch", rows);
  if (L.T * 16 > 48 * 1024) return set_error(TLQ_EUNSUPPORTED, "requant in place: group %d is too large", group);
  int gmax = 1;
  for (int i = 0; i < count; ++i) gmax = L.G[i] > gmax ? L.G[i] : gmax;
  const size_t smem = (size_t)(L.chunk < gmax ? L.chunk : gmax) * L.T * 16;
  requant_in_place_kernel<<<(unsigned)rows, kIpThreads, smem, stream>>>(L);
  return cuda_error(cudaGetLastError(), "requant in place: launch");
}

tlq_status launch_requant(const RequantArgs* a, int count, int group, cudaStream_t stream) {
  RqLaunch L = {};
  long long g = 0;
  for (int i = 0; i < count; ++i) {
    L.p[i] = RqProblem{reinterpret_cast<const uint4*>(a[i].W4), a[i].s4, a[i].z4, reinterpret_cast<uint2*>(a[i].W2),
                       a[i].s2, a[i].z2, g};
    g += static_cast<long long>(a[i].N) * (a[i].K / group);
  }
  L.count = count;
  L.ngroups = g;
  L.T = group / 32;
  if (g == 0) return TLQ_OK;
  const int kind = L.T == 4 ? 2 : (L.T == 2 ? 1 : 0);
  // persistent: the resident CTAs of every SM, fewer when there is less work
  static int occ[3] = {0, 0, 0};
  int& o = occ[kind];
  if (o == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &o, kind == 2 ? requant_kernel<4> : (kind == 1 ? requant_kernel<2> : requant_kernel<0>), kRqThreads, 0);
    if (e != cudaSuccess || o < 1) o = 1;
  }
  const long long want = (g + kRqThreads - 1) / kRqThreads;
  const long long cap = static_cast<long long>(device_info().sms) * o;
  const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
  if (kind == 2)
    requant_kernel<4><<<blocks, kRqThreads, 0, stream>>>(L);
  else if (kind == 1)
    requant_kernel<2><<<blocks, kRqThreads, 0, stream>>>(L);
  else
    requant_kernel<0><<<blocks, kRqThreads, 0, stream>>>(L);
  return cuda_error(cudaGetLastError(), "requant: launch");
}

}  // namespace tlq

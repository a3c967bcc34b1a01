// Helpers shared by the tcgen05 kernels of libtlq (sm_103a): shared-memory
// matrix descriptors, TMEM allocation and access, MMA completion and the FP16
// dequantization of packed weight words.
#pragma once

#include "common.cuh"

namespace tlq {

// Half i (0..7) of a 16-byte vector, as the low 16 bits.
__device__ __forceinline__ uint32_t pick16(const uint4& v, int i) {
  const uint32_t w = (i & 4) ? ((i & 2) ? v.w : v.z) : ((i & 2) ? v.y : v.x);
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Shared-memory matrix descriptor: K-major, SWIZZLE_128B, 8-row atoms of
// 1024 bytes (stride byte offset 1024), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}


__device__ __forceinline__ uint32_t hadd2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The per-group constants of the dequantization: the zero point splits into
// an integer part zi = round(z) (clamped to +-1024) and the rest zf = z - zi
// (exact in FP16).  sub = (base + zi) for each code position's base (exact:
// integers of magnitude <= 2048), so the HSUB2 below yields the exact integer
// q - zi; nzf = -fp16(zf * s).  Then w = fp16((q - zi) * s - fp16(zf * s))
// with one FMA: one rounding of the exact (q - zi) * s plus the rounding of a
// bias of at most s / 2, instead of a bias of up to |z| * s.
struct GroupDq {
  uint32_t s2;     // (s, s)
  uint32_t nzf2;   // (-fp16(zf * s), same)
  uint32_t sub_a;  // INT4: (1024 + zi, 64 + zi); INT2: (1024 + zi, 256 + zi)
  uint32_t sub_b;  // INT2: (64 + zi, 16 + zi)
};

template <int BITS>
__device__ __forceinline__ GroupDq group_dq(uint32_t s_bits, uint32_t z_bits) {
  // zi = round(z) clamped to [-1024, 1024]: zf = z - zi is exact (|zf| <= 1/2
  // inside the clamp; beyond it z is an integer multiple of ulp(z) >= 1 and so
  // is z -+ 1024), and base + zi and q - zi stay integers of magnitude <= 2048
  const __half z = __ushort_as_half((unsigned short)z_bits);
  const __half lim = __ushort_as_half((unsigned short)0x6400u);  // 1024
  const __half zi = __hmax(__hneg(lim), __hmin(lim, hrint(z)));
  const __half zf = __hsub(z, zi);
  GroupDq g;
  g.s2 = (uint32_t)(s_bits & 0xFFFFu) * 0x00010001u;
  const uint32_t zf2 = (uint32_t)__half_as_ushort(zf) * 0x00010001u;
  g.nzf2 = hmul2u(zf2, g.s2) ^ 0x80008000u;
  const uint32_t zi2 = (uint32_t)__half_as_ushort(zi) * 0x00010001u;
  g.sub_a = hadd2u(BITS == 4 ? 0x54006400u : 0x5C006400u, zi2);
  g.sub_b = hadd2u(0x4C005400u, zi2);
  return g;
}

// FP16 weights of one packed word in k order: byte j of the word is copied
// into both halves (one PRMT), the codes it holds are masked into the
// mantissas of (base + q) halves (one LOP3 per pair), (base + zi) is removed
// exactly (one HSUB2) and one FMA applies scale and the fractional zero
// point (see GroupDq).  INT4: out[j] = (w_2j, w_2j+1); INT2: out[2j],
// out[2j+1] = (w_4j, w_4j+1), (w_4j+2, w_4j+3).
template <int BITS>
__device__ __forceinline__ void dequant_word(uint32_t w, const GroupDq& g, uint32_t (&out)[BITS == 4 ? 4 : 8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = prmt(w, 0u, (uint32_t)(j | (j << 8)));  // byte j in bytes 0 and 2
    if constexpr (BITS == 4) {
      const uint32_t h = and_or(x, 0x00F0000Fu, 0x54006400u);  // (1024 + q_2j, 64 + q_2j+1)
      out[j] = hfma2u(hsub2u(h, g.sub_a), g.s2, g.nzf2);
    } else {
      const uint32_t ha = and_or(x, 0x000C0003u, 0x5C006400u);  // (1024 + q_4j, 256 + q_4j+1)
      const uint32_t hb = and_or(x, 0x00C00030u, 0x4C005400u);  // (64 + q_4j+2, 16 + q_4j+3)
      out[2 * j] = hfma2u(hsub2u(ha, g.sub_a), g.s2, g.nzf2);
      out[2 * j + 1] = hfma2u(hsub2u(hb, g.sub_b), g.s2, g.nzf2);
    }
  }
}


}  // namespace tlq

// Decode path of quant_gemm (M <= 16 tokens): one pass over the packed
// weights, for one or several independent problems per launch.  The roofline
// is HBM bandwidth; on GB300 the kernel is held below it by its instruction
// stream (a copy that skips all weight and activation loads runs only 13 %
// faster).
//
// Layer: C[m][n] = fp16( sum_k A[m][k] * (q[n][k] - z[n][g]) * s[n][g] ).
// Source: "Model" (TinyLoop Python API), "VRAM cost", Weights (INT2 / INT4
// packed data + FP16 scales + FP16 zeros per quantized layer); "beta-Informed
// Deployment Features", CTX-TIER: the INT2 kernel's smaller footprint is what
// speeds decode up, so the kernel is built to stream weight bytes at HBM rate.
//
// Design (GB300):
//  * Persistent: one CTA per SM walks a list of work units (a 64-, 32- or
//    16-row tile of one problem, all of K).  The host deals units to CTAs
//    longest first (each to the least-loaded CTA), so a launch may hold up to
//    16 independent problems (a whole decode step) and the ~2-3 us fixed cost
//    of a launch is paid once.  Launches with few row tiles use shorter units
//    so that more SMs take part.
//  * Each of the 8 warps owns every 8th k-block (16 packed words per row) of a
//    unit and streams its packed weights through a private 2-stage TMA ring
//    (SWIZZLE_64B, so that the transposed word reads are bank-conflict free,
//    or unswizzled with the contiguous word mapping).  The rings run ahead
//    across unit boundaries.
//  * Scales and zeros of the unit two ahead are copied into a ring of shared
//    S / Z tiles with cp.async (no registers, no wait until the unit's
//    barrier); activations are read straight from global memory one k-block
//    ahead.
//  * A k-block is split into four "sets"; in a set, the four lanes that feed
//    one MMA row hold 4*32/bits codes of one quantization group.
//  * Codes become FP16 MMA operands with one LOP3 per pair: a code at mantissa
//    bit position p of a half with exponent e reads as 2^e + q exactly (the
//    "base" of that position: 1024, 256, 64, 16 or 4).  Over a span of codes
//    that share one (scale, zero) the MMA sums a * (base + q); two
//    row-independent correction sums (sum_k base_k a_k and sum_k a_k), which
//    one extra MMA per word computes for all rows at once, then remove the
//    base term and the zero point:
//        acc_span = sum_k a_k (base_k + q_k) - sum_k base_k a_k - z * sum_k a_k
//                 = sum_k a_k (q_k - z)
//        total   += s * acc_span          (FP32)
//  * Tokens are the MMA's N dimension (one or two 8-wide tiles), weight rows
//    its M dimension (m16n8k16, "swap AB").
//  * The eight warps' partial sums of a unit are added in a fixed order through
//    a double-buffered shared-memory tile (deterministic, no atomics).
//  * Programmatic dependent launch: weights, scales and zeros are fetched
//    before griddepcontrol.wait, activations and outputs only after it.
//  * The host keeps the launch descriptions (tensor maps, problem table, unit
//    lists) of recent calls, so repeated calls skip rebuilding them.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace tlq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSPW = 2;             // TMA stages per warp
constexpr int kWordsPerKBlock = 16; // per row: 64 bytes
constexpr int kStageRowBytes = kWordsPerKBlock * 4;
constexpr int kMaxProblems = kMaxDecodeProblems;

template <int BITS>
struct Fmt {
  static constexpr int CPW = 32 / BITS;               // codes per word
  static constexpr int KBLK = kWordsPerKBlock * CPW;  // codes per k-block
  static constexpr int SETC = 4 * CPW;                // codes per set
  static constexpr int MPS = CPW / 4;                 // MMAs per word (k16 each)
};

struct DecodeProblem {
  const __half* A;
  const __half* S;
  const __half* Z;
  __half* C;
  float* X;
  int lda, ldc, ldx;
  int M, N, K, G;
  int epi;
  int ntiles;           // row tiles
  int nkb;              // k-blocks
  int unit_begin;       // first global unit index
  uint64_t spg_magic;   // set index -> group index: (si * magic) >> 40
  int szvec;            // scale/zero rows copied in 16-byte pieces (K/group % 8 == 0, 16-byte aligned arrays)
  int spanq;            // sets per accumulation span inside a k-block (4, 2, 1) or 0 (generic)
};

// Per-CTA unit lists built on the host (longest-first greedy on estimated
// unit cost), up to kMaxPerCta units on each of up to kMaxListGrid CTAs, in
// fixed per-CTA slots so a CTA reads its whole list in parallel at start-up
// (no dependent parameter reads); larger launches deal units in snake order
// on the device instead.
constexpr int kMaxPerCta = 16;
constexpr int kMaxListGrid = 256;

struct DecodeLaunch {
  CUtensorMap wmap[kMaxProblems];
  DecodeProblem prob[kMaxProblems];
  int count;
  int total_units;
  int keep_mask;  // bit p: problem p's weights are streamed evict-last (kept in L2)
  int gmax;    // largest K/group
  int gpitch;  // row pitch of the scale/zero tiles in halves: gmax rounded up to 8, plus 8
  int nsz;     // scale/zero buffers (3 or 2, by shared memory)
  int listed;  // 1: CTA b runs cta_units[b][0 .. cta_count[b]) (problem | row tile << 4); 0: snake order
  uint8_t cta_count[kMaxListGrid];
  uint16_t cta_units[kMaxListGrid][kMaxPerCta];
};

// FP16 pairs (base + q) of one word: pairs[i] holds positions (i, i + CPW/2).
template <int BITS>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&p)[Fmt<BITS>::CPW / 2]) {
  if constexpr (BITS == 4) {
    const uint32_t w8 = w >> 8;
    p[0] = and_or(w, 0x000F000Fu, 0x64006400u);   // 1024 + q   codes 0, 4
    p[1] = and_or(w, 0x00F000F0u, 0x54005400u);   //   64 + q   codes 1, 5
    p[2] = and_or(w8, 0x000F000Fu, 0x64006400u);  // 1024 + q   codes 2, 6
    p[3] = and_or(w8, 0x00F000F0u, 0x54005400u);  //   64 + q   codes 3, 7
  } else {
    const uint32_t w10 = w >> 10;
    p[0] = and_or(w, 0x00030003u, 0x64006400u);    // 1024 + q  codes 0, 8
    p[1] = and_or(w, 0x000C000Cu, 0x5C005C00u);    //  256 + q  codes 1, 9
    p[2] = and_or(w, 0x00300030u, 0x54005400u);    //   64 + q  codes 2, 10
    p[3] = and_or(w, 0x00C000C0u, 0x4C004C00u);    //   16 + q  codes 3, 11
    p[4] = and_or(w, 0x03000300u, 0x44004400u);    //    4 + q  codes 4, 12
    p[5] = and_or(w10, 0x00030003u, 0x64006400u);  // 1024 + q  codes 5, 13
    p[6] = and_or(w10, 0x000C000Cu, 0x5C005C00u);  //  256 + q  codes 6, 14
    p[7] = and_or(w10, 0x00300030u, 0x54005400u);  //   64 + q  codes 7, 15
  }
}

// Correction operand of MMA e: rows 0-7 hold -base of the pair each k slot
// carries, rows 8-15 hold -1.  Returns {a0a1, a2a3, a4a5, a6a7}.
template <int BITS>
__device__ __forceinline__ uint4 correction_frag(int e) {
  const uint32_t m1 = 0xBC00BC00u;  // -1, -1
  if constexpr (BITS == 4) {
    return make_uint4(0xE400E400u, m1, 0xD400D400u, m1);  // -1024 | -64
  } else {
    // pair bases 1024, 256, 64, 16, 4, 1024, 256, 64 for pairs 0..7
    const uint32_t neg[8] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u,
                             0xC400C400u, 0xE400E400u, 0xDC00DC00u, 0xD400D400u};
    return make_uint4(neg[2 * e], m1, neg[2 * e + 1], m1);
  }
}

// The CTA's units, tabulated once in shared memory (problem index, first row
// and k-block count of each): from the host-built list when there is one,
// else dealt in snake order (round r takes global unit r*P + b when r is
// even, r*P + P-1-b when odd).
struct Sched {
  int p;
  int n0;
  int nkb;
  int pad;
};
constexpr int kMaxRounds = 256;  // units per CTA; the launcher caps total units at kMaxRounds * grid

__device__ __forceinline__ int problem_of(const DecodeLaunch& L, int unit) {
  int p = 0;
#pragma unroll 1
  for (int i = 1; i < L.count; ++i)
    if (unit >= L.prob[i].unit_begin) p = i;
  return p;
}

// Producer of one warp's TMA ring: items are (unit, k-block) in the order the
// warp consumes them, issued up to kSPW ahead.
struct Producer {
  int ri, kb, issued, warp, nrounds;
  __device__ __forceinline__ void skip(const Sched* tab) {  // to the next unit with a k-block for this warp
    while (ri < nrounds && kb >= tab[ri].nkb) {
      ++ri;
      kb = warp;
    }
  }
  __device__ __forceinline__ void init(const Sched* tab, int warp_, int nrounds_) {
    warp = warp_;
    nrounds = nrounds_;
    issued = 0;
    ri = 0;
    kb = warp;
    skip(tab);
  }
  template <int ROWS>
  __device__ __forceinline__ void issue(const DecodeLaunch& L, const Sched* tab, uint8_t* ring, uint64_t* full,
                                        uint64_t pol) {
    if (ri >= nrounds) return;
    constexpr int STAGE_BYTES = ROWS * kStageRowBytes;
    const int slot = warp * kSPW + (issued % kSPW);
    const Sched e = tab[ri];
    mbar_arrive_expect_tx(&full[slot], STAGE_BYTES);
    tma_load_2d_hint(&L.wmap[e.p], &full[slot], ring + slot * STAGE_BYTES, kb * kWordsPerKBlock, e.n0,
                     ((L.keep_mask >> e.p) & 1) ? policy_evict_last() : pol);
    ++issued;
    kb += kWarps;
    skip(tab);
  }
};

__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Scales and zeros of one unit in shared memory: an S tile [ROWS][gp] then a
// Z tile [ROWS][gp] of halves, gp = (K/group rounded up to 8) + 8, so rows
// are 16-byte aligned and the eight rows a warp reads at once fall in
// different banks.  Rows with K/group a multiple of 8 (and 16-byte aligned
// scale/zero arrays) are copied with cp.async 16-byte copies that need no
// registers and complete in the background; other shapes copy element by
// element.  Every thread commits one copy group per call, so the counts the
// waits rely on are uniform.  Rows past N copy row N - 1 (never used).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, unsigned short v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ float lds_half(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __half2float(__ushort_as_half(v));
}

template <int ROWS>
__device__ __forceinline__ void stage_unit_sz(const DecodeProblem& pr, int n0, int tid, uint32_t dst, int gp) {
  const int G = pr.G;
  if (pr.szvec) {
    const int cpr = G >> 3;  // 16-byte chunks per row
    const int per = ROWS * cpr;
    for (int i = tid; i < 2 * per; i += kThreads) {
      const int arr = i >= per;  // 0: S, 1: Z
      const int j = i - arr * per;
      const int row = j / cpr, ch = j - row * cpr;
      const int n = min(n0 + row, pr.N - 1);
      cp_async16(dst + (uint32_t)((arr * ROWS + row) * gp + ch * 8) * 2, (arr ? pr.Z : pr.S) + (size_t)n * G + ch * 8);
    }
  } else {
    const int per = ROWS * G;
    for (int i = tid; i < 2 * per; i += kThreads) {
      const int arr = i >= per;
      const int j = i - arr * per;
      const int row = j / G, gg = j - row * G;
      const int n = min(n0 + row, pr.N - 1);
      const __half* src = (arr ? pr.Z : pr.S) + (size_t)n * G + gg;
      sts16(dst + (uint32_t)((arr * ROWS + row) * gp + gg) * 2, __half_as_ushort(__ldg(src)));
    }
  }
  cp_async_commit();
}

// Per-unit values of the current problem, held in registers.
struct UnitRegs {
  const __half* ap[2];  // this lane's activation row (token 8t + g, clamped to token 0 past M) + word offset
  int qs;               // codes between this lane's words of consecutive sets
  int K, nkb, nkb_full, gp;  // gp: row pitch of the scale/zero tiles (halves)
  uint64_t magic;
  uint32_t szbase;           // S tile of this unit; the Z tile follows at + ROWS * gp halves
};

// INT4 with whole-k-block groups uses the contiguous word mapping: lane c of
// a row takes words 4c .. 4c+3 (one per set, one 16-byte shared load), else
// set q of lane c is word 4q + c.  The k order inside a span does not matter
// for a sum, only that the activations follow the same mapping.
template <int BITS, int SPANQ>
struct WordMap {
  static constexpr bool CONTIG = (BITS == 4 && SPANQ == 4);
};

__device__ __forceinline__ uint4 ldg_nc_v4(const __half* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldg_v4_pred(uint4& v, const __half* p, bool pred) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %5, 0;\n @p ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];\n}"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "l"(p), "r"((int)pred));
}

// Activations of the four sets of k-block kb for this lane: B-fragment raw
// data.  Tokens past M read token 0 (their sums are never stored); in the
// last, partial k-block the codes past K read zero (only the word-4q+c
// mapping has partial k-blocks: the contiguous one needs K % 128 == 0).
template <int BITS, int NTP>
__device__ __forceinline__ void load_acts(const UnitRegs& ur, int kb, uint4 (&ax)[4][NTP], uint4 (&ay)[4][NTP]) {
  using F = Fmt<BITS>;
  if (kb < ur.nkb_full) {
#pragma unroll
    for (int t = 0; t < NTP; ++t) {
      const __half* ap = ur.ap[t] + kb * F::KBLK;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ax[q][t] = ldg_nc_v4(ap + q * ur.qs);
        if constexpr (BITS == 2) ay[q][t] = ldg_nc_v4(ap + q * ur.qs + 8);
      }
    }
  } else {
#pragma unroll
    for (int t = 0; t < NTP; ++t) {
      const __half* ap = ur.ap[t] + kb * F::KBLK;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool ok = kb * F::KBLK + q * F::SETC < ur.K;
        ax[q][t] = make_uint4(0, 0, 0, 0);
        ldg_v4_pred(ax[q][t], ap + q * ur.qs, ok);
        if constexpr (BITS == 2) {
          ay[q][t] = make_uint4(0, 0, 0, 0);
          ldg_v4_pred(ay[q][t], ap + q * ur.qs + 8, ok);
        }
      }
    }
  }
}

// Packed FP32 pairs (sm_100 family): one instruction applies the same IEEE
// operation, rounded to nearest, to both halves, so the results are those of
// the scalar operations.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// One k-block (4 sets) of one warp: MMAs over the span(s), correction, and
// the scaled accumulation into tot.  SPANQ: sets per span (4, 2, 1), or 0 when
// the group size is not a multiple of the set width pattern (each set then
// computes its own group index).
template <int BITS, int RGW, int NTP, int SPANQ, bool FULL>
__device__ __forceinline__ void kblock(const UnitRegs& ur, int kb, uint32_t wq0, const uint32_t (&woff)[5], int g,
                                       const uint4 (&ax)[4][NTP], const uint4 (&ay)[4][NTP],
                                       float (&tot)[RGW][NTP][4]) {
  using F = Fmt<BITS>;
  constexpr bool partial = !FULL;
  int gbase = 0;
  if constexpr (SPANQ == 4) gbase = (int)(((uint64_t)(kb * 4) * ur.magic) >> 40);
  if constexpr (SPANQ == 2) gbase = 2 * kb;
  if constexpr (SPANQ == 1) gbase = 4 * kb;
  float acc[RGW][NTP][4];
  float corr[NTP][4];
  constexpr bool CONTIG = WordMap<BITS, SPANQ>::CONTIG;
  uint4 wv[CONTIG ? RGW : 1][2];  // contiguous mapping: this lane's 4 words of rows 16r+g and 16r+g+8
  if constexpr (CONTIG) {
#pragma unroll
    for (int r = 0; r < RGW; ++r) {
      wv[r][0] = lds128(wq0 + woff[4] + (uint32_t)(16 * r) * kStageRowBytes);
      wv[r][1] = lds128(wq0 + woff[4] + (uint32_t)(16 * r + 8) * kStageRowBytes);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (partial && kb * F::KBLK + q * F::SETC >= ur.K) break;
    constexpr int SQ = SPANQ == 0 ? 1 : SPANQ;
    const bool span_start = (q % SQ) == 0;
    const bool span_end = ((q % SQ) == SQ - 1) || (partial && kb * F::KBLK + (q + 1) * F::SETC >= ur.K);
    // ---- B fragments (activations) ----
    uint32_t bf[NTP][F::MPS][2];
#pragma unroll
    for (int t = 0; t < NTP; ++t) {
      const uint4 x = ax[q][t];
      if constexpr (BITS == 4) {
        // x = (a0,a1)(a2,a3)(a4,a5)(a6,a7); pairs (0,4)(1,5) | (2,6)(3,7)
        bf[t][0][0] = prmt(x.x, x.z, 0x5410);
        bf[t][0][1] = prmt(x.x, x.z, 0x7632);
        bf[t][1][0] = prmt(x.y, x.w, 0x5410);
        bf[t][1][1] = prmt(x.y, x.w, 0x7632);
      } else {
        // x = a0..a7, y = a8..a15; pairs (2e, 2e+8) and (2e+1, 2e+9)
        const uint4 y = ay[q][t];
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
        const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bf[t][e][0] = prmt(xs[e], ys[e], 0x5410);
          bf[t][e][1] = prmt(xs[e], ys[e], 0x7632);
        }
      }
    }
    // ---- correction sums over the span ----
#pragma unroll
    for (int t = 0; t < NTP; ++t) {
      if (span_start) {
#pragma unroll
        for (int u = 0; u < 4; ++u) corr[t][u] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < F::MPS; ++e) {
        const uint4 ka = correction_frag<BITS>(e);
        mma_16816(corr[t], ka.x, ka.y, ka.z, ka.w, bf[t][e][0], bf[t][e][1]);
      }
    }
    // ---- weight rows: sums of a * (base + q) over the span ----
    // All row groups are unpacked first; the MMAs then run k-slice-major, so
    // consecutive MMAs of one accumulator are RGW * NTP issues apart.
    const uint32_t wq = wq0 + woff[q];
    uint32_t pg[RGW][F::CPW / 2], ph[RGW][F::CPW / 2];
#pragma unroll
    for (int r = 0; r < RGW; ++r) {
      if constexpr (CONTIG) {
        unpack_word<BITS>(q == 0 ? wv[r][0].x : q == 1 ? wv[r][0].y : q == 2 ? wv[r][0].z : wv[r][0].w, pg[r]);
        unpack_word<BITS>(q == 0 ? wv[r][1].x : q == 1 ? wv[r][1].y : q == 2 ? wv[r][1].z : wv[r][1].w, ph[r]);
      } else {
        unpack_word<BITS>(lds32(wq + (uint32_t)(16 * r) * kStageRowBytes), pg[r]);
        unpack_word<BITS>(lds32(wq + (uint32_t)(16 * r + 8) * kStageRowBytes), ph[r]);
      }
    }
    if (span_start) {
#pragma unroll
      for (int r = 0; r < RGW; ++r)
#pragma unroll
        for (int t = 0; t < NTP; ++t)
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[r][t][u] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < F::MPS; ++e)
#pragma unroll
      for (int t = 0; t < NTP; ++t)
#pragma unroll
        for (int r = 0; r < RGW; ++r)
          mma_16816(acc[r][t], pg[r][2 * e], ph[r][2 * e], pg[r][2 * e + 1], ph[r][2 * e + 1], bf[t][e][0], bf[t][e][1]);
    // ---- span end: remove base and zero point, apply the scale ----
    if (span_end) {
      int gi;
      if constexpr (SPANQ == 0) gi = (int)(((uint64_t)(kb * 4 + q) * ur.magic) >> 40);
      else gi = gbase + q / SQ;
      const uint32_t sa = ur.szbase + (uint32_t)((g * ur.gp + gi) * 2);
      const uint32_t za = sa + (uint32_t)(16 * RGW * ur.gp * 2);
#pragma unroll
      for (int r = 0; r < RGW; ++r) {
        // (x, y) = (s, z) of rows 16r + g and 16r + g + 8
        const float2 fg = make_float2(lds_half(sa + (uint32_t)(16 * r * ur.gp) * 2),
                                      lds_half(za + (uint32_t)(16 * r * ur.gp) * 2));
        const float2 fh = make_float2(lds_half(sa + (uint32_t)((16 * r + 8) * ur.gp) * 2),
                                      lds_half(za + (uint32_t)((16 * r + 8) * ur.gp) * 2));
        // acc + corr0 + z * corr2 = sum a (q - z); then * s.  The two tokens
        // of a lane's pair share s and z, so they go through packed pairs
        // (the same bits as the scalar form below).  The INT2 two-tile body
        // keeps the scalar form: packed, it spilled registers (measured
        // slower); elsewhere packed pairs were 1 % (INT4) and 2.5 % (INT2
        // step) faster.
        if constexpr (BITS == 4 || NTP == 1) {
          const uint64_t SG = f2pack(fg.x, fg.x), ZG = f2pack(fg.y, fg.y);
          const uint64_t SH = f2pack(fh.x, fh.x), ZH = f2pack(fh.y, fh.y);
#pragma unroll
          for (int t = 0; t < NTP; ++t) {
            const uint64_t c01 = f2pack(corr[t][0], corr[t][1]), c23 = f2pack(corr[t][2], corr[t][3]);
            const uint64_t t01 = f2fma(SG, f2fma(ZG, c23, f2add(f2pack(acc[r][t][0], acc[r][t][1]), c01)),
                                       f2pack(tot[r][t][0], tot[r][t][1]));
            const uint64_t t23 = f2fma(SH, f2fma(ZH, c23, f2add(f2pack(acc[r][t][2], acc[r][t][3]), c01)),
                                       f2pack(tot[r][t][2], tot[r][t][3]));
            f2unpack(t01, tot[r][t][0], tot[r][t][1]);
            f2unpack(t23, tot[r][t][2], tot[r][t][3]);
          }
        } else {
#pragma unroll
          for (int t = 0; t < NTP; ++t) {
            tot[r][t][0] = fmaf(fg.x, fmaf(fg.y, corr[t][2], acc[r][t][0] + corr[t][0]), tot[r][t][0]);
            tot[r][t][1] = fmaf(fg.x, fmaf(fg.y, corr[t][3], acc[r][t][1] + corr[t][1]), tot[r][t][1]);
            tot[r][t][2] = fmaf(fh.x, fmaf(fh.y, corr[t][2], acc[r][t][2] + corr[t][0]), tot[r][t][2]);
            tot[r][t][3] = fmaf(fh.x, fmaf(fh.y, corr[t][3], acc[r][t][3] + corr[t][1]), tot[r][t][3]);
          }
        }
      }
    }
  }
}

// All k-blocks of one unit for this warp.  Activations run one k-block ahead
// in nx/ny (NT tiles): on entry they hold this warp's first k-block of the
// unit, on exit the first k-block of the next unit (nu), so no unit starts
// on an exposed global load.
template <int BITS, int RGW, int NTP, int SPANQ, int NT, bool ALLFULL>
__device__ __forceinline__ void run_unit(const DecodeLaunch& L, const Sched* tab, const UnitRegs& ur,
                                         const UnitRegs& nu, bool has_next, int warp, int lane,
                                         const uint32_t (&woff)[5], uint32_t ring_base, uint8_t* ring,
                                         uint64_t* full, uint64_t pol, Producer& prod, int& consumed, bool& ok,
                                         uint4 (&nx)[4][NT], uint4 (&ny)[4][NT], float (&tot)[RGW][NTP][4]) {
  constexpr int ROWS = 16 * RGW;
  constexpr int STAGE_BYTES = ROWS * kStageRowBytes;
  const int g = lane >> 2;
#pragma unroll
  for (int r = 0; r < RGW; ++r)
#pragma unroll
    for (int t = 0; t < NTP; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[r][t][i] = 0.f;
  for (int kb = warp; kb < ur.nkb; kb += kWarps) {
    uint4 ax[4][NTP], ay[4][NTP];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int t = 0; t < NTP; ++t) {
        ax[q][t] = nx[q][t];
        ay[q][t] = ny[q][t];
      }
    if (kb + kWarps < ur.nkb)
      load_acts<BITS, NT>(ur, kb + kWarps, nx, ny);
    else if (has_next && warp < nu.nkb)
      load_acts<BITS, NT>(nu, warp, nx, ny);
    const int slot = warp * kSPW + (consumed % kSPW);
    if (ok) ok = mbar_wait(&full[slot], (consumed / kSPW) & 1, 0x112);
    __syncwarp();  // the lanes leave the wait separately; the MMAs below are warp-collective
    if (ALLFULL || kb < ur.nkb_full)
      kblock<BITS, RGW, NTP, SPANQ, true>(ur, kb, ring_base + (uint32_t)slot * STAGE_BYTES, woff, g, ax, ay, tot);
    else
      kblock<BITS, RGW, NTP, SPANQ, false>(ur, kb, ring_base + (uint32_t)slot * STAGE_BYTES, woff, g, ax, ay, tot);
    ++consumed;
    // This slot is free again: refill it with the warp's next item.  Every
    // shared load of the slot has already delivered its value to an MMA of
    // this k-block, so no read can still be pending when the TMA overwrites it
    // (the release needs no proxy fence; measured 1 % faster on the decode step).
    __syncwarp();
    if (lane == 0) prod.template issue<ROWS>(L, tab, ring, full, pol);
  }
  if (warp >= ur.nkb && has_next && warp < nu.nkb) load_acts<BITS, NT>(nu, warp, nx, ny);
}

// SQ = 0: the group class (sets per span) is chosen per unit at run time;
// SQ = 4: every problem of the launch has four sets per span (INT4, groups of
// a multiple of 128 codes); SQ = 1: one set per span (INT2, groups of 64
// codes).  WHOLE: every problem's K is a whole number of
// k-blocks, so the body for a ragged last k-block is left out.  The arithmetic
// is the same in every form; leaving out the code that cannot run shrinks the
// loop the SMs fetch instructions for (measured on the decode steps: INT4
// 3028 -> 3176 GB/s with SQ = 4, INT2 1668 -> 1693 GB/s with WHOLE).
template <int BITS, int RGW, int NT, int SQ, bool WHOLE>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeLaunch L) {
  constexpr int ROWS = 16 * RGW;
  constexpr int STAGE_BYTES = ROWS * kStageRowBytes;
  constexpr int MT = 8 * NT;    // token slots
  constexpr int RP = ROWS + 4;  // reduction row pitch (conflict-free)
  using F = Fmt<BITS>;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;  // [warp][kSPW][STAGE_BYTES]
  const int gp = L.gpitch;
  const int szbytes = 4 * ROWS * gp;  // one unit's S and Z tiles
  const int nsz = L.nsz;              // scale/zero buffers: 3 (staged two units ahead) or 2 (one ahead)
  uint8_t* szb = ring + kWarps * kSPW * STAGE_BYTES;                          // [nsz][S, Z][ROWS][gp]
  float* red = reinterpret_cast<float*>(szb + nsz * szbytes);                 // [par][warp][MT][RP]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * kWarps * MT * RP);         // [warp][kSPW]
  Sched* tab = reinterpret_cast<Sched*>(full + kWarps * kSPW);                      // [kMaxRounds]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int P = gridDim.x;
  const int b = blockIdx.x;

  // the launch's tensor maps first: their descriptors are fetched while the rest starts
  if (warp == 0 && lane < L.count) tma_prefetch_desc(&L.wmap[lane]);
  if (tid == 0) {
    for (int i = 0; i < kWarps * kSPW; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  // this CTA's units.  Every thread walks the same rounds, so each parameter
  // read is a broadcast (per-thread rounds would make 256 divergent,
  // serialized constant-bank reads); one thread stores the table.
  int nrounds = 0;
  if (L.listed) {
    nrounds = L.cta_count[b];
    if (tid < kMaxPerCta) {
      const uint32_t w = L.cta_units[b][tid];  // problem | row tile << 4 (all entries read at once)
      if (tid < nrounds) {
        Sched e;
        e.p = (int)(w & 15u);
        e.n0 = (int)(w >> 4) * ROWS;
        e.nkb = L.prob[e.p].nkb;
        e.pad = 0;
        tab[tid] = e;
      }
    }
  } else {
#pragma unroll 1
    for (int r = 0; r < kMaxRounds; ++r) {
      const int u = r * P + ((r & 1) ? (P - 1 - b) : b);
      if (u >= L.total_units) break;
      if (tid == 0) {
        const int p = problem_of(L, u);
        Sched e;
        e.p = p;
        e.n0 = (u - L.prob[p].unit_begin) * ROWS;
        e.nkb = L.prob[p].nkb;
        e.pad = 0;
        tab[r] = e;
      }
      nrounds = r + 1;
    }
  }
  __syncthreads();  // barrier inits and the table are visible
  if (tid == 0) pdl_launch_dependents();

  const uint64_t pol = policy_evict_first();
  Producer prod;
  prod.init(tab, warp, nrounds);
  if (lane == 0)
    for (int i = 0; i < kSPW; ++i) prod.template issue<ROWS>(L, tab, ring, full, pol);
  const uint32_t szb_base = smem_u32(szb);
  // scales/zeros of the first nsz - 1 units (weights-side data: before the dependency wait)
  for (int i = 0; i < nsz - 1; ++i) {
    if (i < nrounds) stage_unit_sz<ROWS>(L.prob[tab[i].p], tab[i].n0, tid, szb_base + (uint32_t)(i * szbytes), gp);
    else cp_async_commit();
  }
  if (nsz == 3) cp_async_wait<1>();  // unit 0's copies (unit 1's may still be in flight)
  else cp_async_wait<0>();
  pdl_wait();  // activations (and the residual) may come from the preceding kernel

  // per-lane parts of the word addresses: [q] row g of set q -> word 4q + c in a
  // SWIZZLE_64B tile; [4] row g, words 4c .. 4c+3 in an unswizzled tile
  uint32_t woff[5];
#pragma unroll
  for (int q = 0; q < 4; ++q) woff[q] = (uint32_t)(g * kStageRowBytes + (((q ^ (g >> 1)) & 3) << 4) + (c << 2));
  woff[4] = (uint32_t)(g * kStageRowBytes + (c << 4));

  const uint32_t ring_base = smem_u32(ring);
  const uint32_t red_base = smem_u32(red);
  int consumed = 0;
  bool ok = true;
  __syncthreads();  // first unit's scales/zeros are in shared memory

  auto make_regs = [&](int s_, UnitRegs& ur) {
    const Sched e = tab[s_];
    const DecodeProblem& pr = L.prob[e.p];
    ur.K = pr.K;
    ur.nkb = e.nkb;
    ur.nkb_full = pr.K / F::KBLK;
    ur.gp = gp;
    ur.magic = pr.spg_magic;
    ur.szbase = szb_base + (uint32_t)((s_ % nsz) * szbytes);
    const bool contig = BITS == 4 && pr.spanq == 4;
    ur.qs = contig ? F::CPW : F::SETC;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int tok = 8 * t + g;
      ur.ap[t] = pr.A + (size_t)(tok < pr.M ? tok : 0) * pr.lda + c * (contig ? 4 * F::CPW : F::CPW);
    }
  };
  // activations of this warp's first k-block of the first unit
  uint4 nx[4][NT], ny[4][NT];
  UnitRegs ur, nu;
  if (nrounds > 0) {
    make_regs(0, ur);
    if (warp < ur.nkb) load_acts<BITS, NT>(ur, warp, nx, ny);
  }

  for (int s = 0; s < nrounds; ++s) {
    const int par = s & 1;
    const Sched e = tab[s];
    const DecodeProblem& pr = L.prob[e.p];
    const int n0 = e.n0;
    const int M = pr.M;
    const bool has_next = s + 1 < nrounds;
    // scales/zeros of unit s + nsz - 1 into the buffer unit s - 1 used (every
    // thread passed that unit's barrier, so no one reads it any more)
    {
      const int su = s + nsz - 1;
      if (su < nrounds)
        stage_unit_sz<ROWS>(L.prob[tab[su].p], tab[su].n0, tid, szb_base + (uint32_t)((su % nsz) * szbytes), gp);
      else
        cp_async_commit();
    }
    if (has_next) make_regs(s + 1, nu);
    const int spanq = pr.spanq;

    float tot[RGW][NT][4];
    bool done = false;
    if constexpr (NT == 2) {
      if (M > 8) {
        done = true;
        if constexpr (SQ == 1) {
          run_unit<BITS, RGW, 2, 1, NT, true>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot);
        } else if constexpr (SQ == 4) {
          run_unit<BITS, RGW, 2, 4, NT, true>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot);
        } else {
          switch (spanq) {
            case 4: run_unit<BITS, RGW, 2, 4, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot); break;
            case 2: run_unit<BITS, RGW, 2, 2, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot); break;
            case 1: run_unit<BITS, RGW, 2, 1, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot); break;
            default: run_unit<BITS, RGW, 2, 0, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, tot); break;
          }
        }
      }
    }
    if (!done) {
      float t1[RGW][1][4];
      if constexpr (SQ == 1) {
        run_unit<BITS, RGW, 1, 1, NT, true>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1);
      } else if constexpr (SQ == 4) {
        run_unit<BITS, RGW, 1, 4, NT, true>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1);
      } else {
        switch (spanq) {
          case 4: run_unit<BITS, RGW, 1, 4, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1); break;
          case 2: run_unit<BITS, RGW, 1, 2, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1); break;
          case 1: run_unit<BITS, RGW, 1, 1, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1); break;
          default: run_unit<BITS, RGW, 1, 0, NT, WHOLE>(L, tab, ur, nu, has_next, warp, lane, woff, ring_base, ring, full, pol, prod, consumed, ok, nx, ny, t1); break;
        }
      }
#pragma unroll
      for (int r = 0; r < RGW; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) tot[r][t][i] = t == 0 ? t1[r][0][i] : 0.f;
    }

    // ---- unit reduction: fixed-order sum of the eight warps' partials ----
    {
      const uint32_t myred = red_base + (uint32_t)((par * kWarps + warp) * MT * RP) * 4;
#pragma unroll
      for (int r = 0; r < RGW; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t == 1 && M <= 8) continue;
          const int ra = 16 * r + g, tk = 8 * t + 2 * c;
          sts_f32(myred + (uint32_t)(tk * RP + ra) * 4, tot[r][t][0]);
          sts_f32(myred + (uint32_t)((tk + 1) * RP + ra) * 4, tot[r][t][1]);
          sts_f32(myred + (uint32_t)(tk * RP + ra + 8) * 4, tot[r][t][2]);
          sts_f32(myred + (uint32_t)((tk + 1) * RP + ra + 8) * 4, tot[r][t][3]);
        }
    }
    // the next unit's scales/zeros have landed (only unit s + 2's group may
    // still be in flight); the barrier publishes them to every thread
    if (nsz == 3) cp_async_wait<1>();
    else cp_async_wait<0>();
    named_barrier(1, kThreads);
    {
      const float* rb = red + (size_t)par * kWarps * MT * RP;
      const int rows = min(ROWS, pr.N - n0);
      const int epi = pr.epi;
      // items of four consecutive rows of one token: eight 16-byte partial
      // loads, one 8-byte store (rows is a multiple of 8, ldc of 4)
      for (int i = tid; i < (ROWS / 4) * M; i += kThreads) {
        const int tk = i / (ROWS / 4), row = 4 * (i % (ROWS / 4));
        if (row >= rows) continue;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float4 x = *reinterpret_cast<const float4*>(rb + (w * MT + tk) * RP + row);
          v.x += x.x;
          v.y += x.y;
          v.z += x.z;
          v.w += x.w;
        }
        const int n = n0 + row;
        __half h[4] = {__float2half_rn(v.x), __float2half_rn(v.y), __float2half_rn(v.z), __float2half_rn(v.w)};
        if (epi == kEpiResidual) {
          float* xp = pr.X + (size_t)tk * pr.ldx + n;
#pragma unroll
          for (int j = 0; j < 4; ++j) xp[j] = xp[j] + __half2float(h[j]);
        } else if (epi == kEpiSwiglu) {  // rows (n, n+1), (n+2, n+3) are (gate, up) pairs
          const uint32_t o = (uint32_t)__half_as_ushort(swiglu_half(h[0], h[1])) |
                             ((uint32_t)__half_as_ushort(swiglu_half(h[2], h[3])) << 16);
          *reinterpret_cast<uint32_t*>(pr.C + (size_t)tk * pr.ldc + n / 2) = o;
        } else {
          if (epi == kEpiRelu) {
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = relu_half(h[j]);
          }
          uint2 o;
          o.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
          o.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
          *reinterpret_cast<uint2*>(pr.C + (size_t)tk * pr.ldc + n) = o;
        }
      }
    }
    if (has_next) ur = nu;
  }

  cp_async_wait<0>();  // (only empty groups can remain here)
  // error path only: copies still in flight land before the CTA exits
  if (!ok && lane == 0) {
    for (int j = consumed; j < prod.issued; ++j)
      if (!mbar_wait(&full[warp * kSPW + (j % kSPW)], (j / kSPW) & 1, 0x113)) break;
  }
}

uint64_t magic_div40(int d) { return (((uint64_t)1) << 40) / (uint64_t)d + 1; }

// Longest-processing-time-first assignment of the launch's units to `grid`
// CTAs: units in decreasing cost order, each to the CTA with the smallest
// load so far (ties: lowest index).  A unit's cost is its k-block count plus
// 8 for the unit's fixed work (barrier, reduction, epilogue: about as long
// as 8 k-blocks, measured), weighted by the token tiles it computes (two
// tiles cost about 1.7x one, measured).  Returns false when some CTA would
// hold more than kMaxRounds units.
bool build_unit_lists(DecodeLaunch& L, int grid) {
  const int units = L.total_units;
  if (grid > kMaxListGrid || units > grid * kMaxPerCta) return false;
  for (int j = 0; j < L.count; ++j)
    if (L.prob[j].ntiles > 4096) return false;  // an entry holds the row tile in 12 bits
  int pord[kMaxProblems];
  uint32_t cost[kMaxProblems];
  for (int j = 0; j < L.count; ++j) {
    pord[j] = j;
    cost[j] = (uint32_t)(L.prob[j].nkb + 8) * (L.prob[j].M > 8 ? 17u : 10u);
  }
  std::stable_sort(pord, pord + L.count, [&](int x, int y) { return cost[x] > cost[y]; });
  // binary min-heap of (load, cta)
  uint64_t heap[kMaxListGrid];
  for (int i = 0; i < grid; ++i) heap[i] = (uint64_t)i;  // load 0: already a heap
  uint8_t count_of[kMaxListGrid] = {};
  for (int j = 0; j < L.count; ++j) {
    const DecodeProblem& pr = L.prob[pord[j]];
    for (int t = 0; t < pr.ntiles; ++t) {
      const uint64_t top = heap[0];
      const int c = (int)(top & 0xFFFFu);
      if (count_of[c] >= kMaxPerCta) return false;
      L.cta_units[c][count_of[c]++] = (uint16_t)(pord[j] | (t << 4));  // costliest units first
      uint64_t v = top + ((uint64_t)cost[pord[j]] << 16);
      int i = 0;  // sift down
      for (;;) {
        const int l = 2 * i + 1, r = l + 1;
        int m = i;
        uint64_t mv = v;
        if (l < grid && heap[l] < mv) {
          m = l;
          mv = heap[l];
        }
        if (r < grid && heap[r] < mv) {
          m = r;
          mv = heap[r];
        }
        if (m == i) break;
        heap[i] = heap[m];
        i = m;
      }
      heap[i] = v;
    }
  }
  for (int c = 0; c < grid; ++c) L.cta_count[c] = count_of[c];
  return true;
}

bool same_args(const GemmArgs& x, const GemmArgs& y) {
  return x.A == y.A && x.lda == y.lda && x.W == y.W && x.S == y.S && x.Z == y.Z && x.C == y.C && x.ldc == y.ldc &&
         x.X == y.X && x.ldx == y.ldx && x.M == y.M && x.N == y.N && x.K == y.K && x.bits == y.bits &&
         x.group == y.group && x.epi == y.epi && x.l2_keep == y.l2_keep && x.ldw == y.ldw;
}

// The launch description of a call: tensor maps, problem table, unit lists,
// shared memory size and grid.
template <int BITS, int RGW, int NT>
tlq_status build_launch(const GemmArgs* a, int count, DecodeLaunch& L, size_t& smem_out, int& grid_out,
                        int& units_out) {
  using F = Fmt<BITS>;
  constexpr int ROWS = 16 * RGW;
  constexpr int MT = 8 * NT;
  memset(&L, 0, sizeof(L));
  // problems with more k-blocks per unit first (snake order then balances)
  int order[kMaxProblems];
  for (int i = 0; i < count; ++i) order[i] = i;
  std::stable_sort(order, order + count, [&](int x, int y) { return a[x].K > a[y].K; });
  int units = 0;
  int gmax = 1;
  for (int j = 0; j < count; ++j) {
    const GemmArgs& g = a[order[j]];
    DecodeProblem& pr = L.prob[j];
    pr.A = g.A;
    pr.S = g.S;
    pr.Z = g.Z;
    pr.C = g.C;
    pr.X = g.X;
    pr.lda = g.lda;
    pr.ldc = g.ldc;
    pr.ldx = g.ldx;
    pr.M = g.M;
    pr.N = g.N;
    pr.K = g.K;
    pr.G = g.K / g.group;
    pr.szvec = (pr.G % 8 == 0) && ((reinterpret_cast<uintptr_t>(g.S) | reinterpret_cast<uintptr_t>(g.Z)) % 16 == 0);
    pr.epi = g.epi;
    if (g.l2_keep) L.keep_mask |= 1 << j;
    pr.ntiles = (g.N + ROWS - 1) / ROWS;
    pr.nkb = (g.K + F::KBLK - 1) / F::KBLK;
    pr.unit_begin = units;
    {
      const int spg = g.group / F::SETC;  // sets per group
      pr.spanq = (spg % 4 == 0) ? 4 : (spg == 2 ? 2 : (spg == 1 ? 1 : 0));
      pr.spg_magic = magic_div40(pr.spanq == 4 ? spg : spg);
    }
    units += pr.ntiles;
    gmax = std::max(gmax, pr.G);
    const uint64_t wpr = (uint64_t)g.K / F::CPW;
    const bool contig = BITS == 4 && pr.spanq == 4;  // see WordMap
    const uint64_t ldw = g.ldw > 0 ? (uint64_t)g.ldw : wpr;  // row stride in words
    tlq_status st = encode_tiled_2d(&L.wmap[j], CU_TENSOR_MAP_DATA_TYPE_UINT32, g.W, wpr, (uint64_t)g.N, ldw * 4,
                                    kWordsPerKBlock, ROWS,
                                    contig ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (st != TLQ_OK) return st;
  }
  L.count = count;
  L.total_units = units;
  L.gmax = gmax;

  L.gpitch = (gmax + 7) / 8 * 8 + 8;
  const size_t fixed = 1024 + (size_t)kWarps * kSPW * ROWS * kStageRowBytes +
                       (size_t)2 * kWarps * MT * (ROWS + 4) * 4 + kWarps * kSPW * 8 + (size_t)kMaxRounds * sizeof(Sched);
  const size_t szbuf = (size_t)4 * ROWS * L.gpitch;
  L.nsz = fixed + 3 * szbuf <= (size_t)device_info().smem_optin ? 3 : 2;
  const size_t smem = fixed + (size_t)L.nsz * szbuf;
  if (smem > (size_t)device_info().smem_optin)
    return set_error(TLQ_EUNSUPPORTED, "decode: K/group = %d needs %zu bytes of shared memory (limit %d)", gmax,
                     smem, device_info().smem_optin);
  const int grid = std::max(1, std::min(units, device_info().sms));
  L.listed = build_unit_lists(L, grid) ? 1 : 0;
  if (units > kMaxRounds * grid)
    return set_error(TLQ_EUNSUPPORTED, "decode: %d row tiles exceed %d per launch", units, kMaxRounds * grid);
  smem_out = smem;
  grid_out = grid;
  units_out = units;
  return TLQ_OK;
}

// Launch descriptions of the last few calls per kernel, keyed by their full
// argument lists: a decode loop repeats the same calls, and rebuilding the
// description (12 tensor maps and the longest-first lists of a decode step)
// costs more host time than the launch itself.
constexpr int kLaunchCache = 8;

template <int BITS, int RGW, int NT, int SQ, bool WHOLE>
tlq_status launch_impl(const GemmArgs* a, int count, cudaStream_t stream) {
  constexpr int ROWS = 16 * RGW;
  static_assert(sizeof(DecodeLaunch) < 30000, "kernel parameter space");
  struct Entry {
    bool valid;
    int count;
    GemmArgs args[kMaxProblems];
    DecodeLaunch L;
    size_t smem;
    int grid, units;
  };
  static std::mutex mu;
  static Entry cache[kLaunchCache];
  static int next = 0;
  auto kern = decode_kernel<BITS, RGW, NT, SQ, WHOLE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_info().smem_optin);
  });
  if (attr_err != cudaSuccess) return cuda_error(attr_err, "decode: cudaFuncSetAttribute");

  std::lock_guard<std::mutex> lk(mu);
  Entry* hit = nullptr;
  for (Entry& e : cache) {
    if (!e.valid || e.count != count) continue;
    bool same = true;
    for (int i = 0; i < count && same; ++i) same = same_args(e.args[i], a[i]);
    if (same) {
      hit = &e;
      break;
    }
  }
  if (!hit) {
    Entry& e = cache[next];
    next = (next + 1) % kLaunchCache;
    e.valid = false;
    tlq_status st = build_launch<BITS, RGW, NT>(a, count, e.L, e.smem, e.grid, e.units);
    if (st != TLQ_OK) return st;
    e.count = count;
    for (int i = 0; i < count; ++i) e.args[i] = a[i];
    e.valid = true;
    hit = &e;
  }
  const DecodeLaunch& L = hit->L;
  const size_t smem = hit->smem;
  const int grid = hit->grid, units = hit->units;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = &attr;
  lc.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&lc, kern, L);
  if (e != cudaSuccess) return cuda_error(e, "decode: launch");
  if (log_enabled())
    fprintf(stderr, "[tlq] decode int%d: %d problem(s), %d units of %d rows, grid %d, smem %zu%s\n", BITS, count,
            units, ROWS, grid, smem,
            SQ == 4 ? ", whole k-blocks of 4-set spans" : SQ == 1 ? ", whole k-blocks of 1-set spans"
                                                         : WHOLE ? ", whole k-blocks" : "");
  return TLQ_OK;
}

// Rows per unit: 64, halved while the launch would have fewer row tiles than
// a third of the SMs, and once more when every problem has long rows (at
// least 32 k-blocks), since a long unit on few SMs then sets the time.
// Measured on the projection shapes at M = 1, 4, 16 (single launches): O
// (N = 2048, K = 2048) is fastest with 32-row units (2.64 against 3.26 us at
// M = 1), DOWN (N = 2048, K = 8192) with 16-row units (6.56 against 9.45 us);
// QKV, UP and the batched decode step keep 64.  Launches whose weights are
// kept in L2 (the loop block) also keep 64 (the next kernel's early start on
// the SMs they leave idle matters more), except the INT4 DOWN projection.
// The unit height does not change any result: every row's sums are formed
// the same way.  TLQ_DECODE_ROWS=16|32|64 forces it.
template <int BITS>
int decode_rgw(const GemmArgs* a, int count) {
  if (const char* e = getenv("TLQ_DECODE_ROWS")) {
    const int r = atoi(e);
    if (r == 16 || r == 32 || r == 64) return r / 16;
  }
  // launches whose weights stay in L2 (the loop block): 64-row units, except
  // a single INT4 problem with long rows (the block's DOWN projection), which
  // would leave most SMs idle: 16-row units (INT4 M = 1 blocks 8-10 % faster
  // per iteration, measured; INT2 unchanged, so it keeps 64)
  for (int i = 0; i < count; ++i)
    if (a[i].l2_keep) return (count == 1 && BITS == 4 && a[i].K >= 4096) ? 1 : 4;
  const int sms = device_info().sms;
  bool long_rows = true;
  for (int i = 0; i < count; ++i) long_rows &= (a[i].K + Fmt<BITS>::KBLK - 1) / Fmt<BITS>::KBLK >= 32;
  auto units = [&](int rgw) {
    int u = 0;
    for (int i = 0; i < count; ++i) u += (a[i].N + 16 * rgw - 1) / (16 * rgw);
    return u;
  };
  int rgw = 4;
  while (rgw > 1 && 3 * units(rgw) < sms) rgw /= 2;
  if (rgw > 1 && rgw < 4 && long_rows && units(rgw) < sms) rgw /= 2;
  return rgw;
}

// Kernel forms: INT4 launches whose groups are all multiples of 128 codes
// (four sets per span, which also makes every k-block whole) take the form
// with one k-block body per token-tile count; INT2 launches whose K are all
// whole k-blocks (256 codes) take the form without the ragged-k-block body,
// and with one k-block body per token-tile count when every group is 64 codes
// (one set per span).  Everything else takes the general form.
// TLQ_DECODE_GENERIC=1 forces the general form.
template <int BITS>
bool decode_fixed_form(const GemmArgs* a, int count) {
  if (const char* e = getenv("TLQ_DECODE_GENERIC"))
    if (atoi(e) != 0) return false;
  for (int i = 0; i < count; ++i) {
    if (a[i].K % Fmt<BITS>::KBLK != 0) return false;
    if (BITS == 4 && a[i].group % (4 * Fmt<BITS>::SETC) != 0) return false;
  }
  return true;
}

template <int BITS, int RGW, int NT>
tlq_status launch_sq(const GemmArgs* a, int count, cudaStream_t s) {
  bool one_set_spans = BITS == 2;
  for (int i = 0; i < count; ++i) one_set_spans &= a[i].group == Fmt<BITS>::SETC;
  if (decode_fixed_form<BITS>(a, count)) {
    if constexpr (BITS == 4) return launch_impl<BITS, RGW, NT, 4, true>(a, count, s);
    else if (one_set_spans) return launch_impl<BITS, RGW, NT, 1, true>(a, count, s);
    else return launch_impl<BITS, RGW, NT, 0, true>(a, count, s);
  }
  return launch_impl<BITS, RGW, NT, 0, false>(a, count, s);
}

// One launch per call: the two-token-tile kernel when any problem has M > 8
// (its problems with M <= 8 take the one-tile path inside it).  Splitting the
// call into a one-tile and a two-tile launch was measured slower for the INT4
// decode step: the second launch costs more than the leaner kernel saves.
template <int BITS>
tlq_status dispatch_bits(const GemmArgs* a, int count, cudaStream_t s) {
  bool two = false;
  for (int i = 0; i < count; ++i) two |= a[i].M > 8;
  switch (decode_rgw<BITS>(a, count)) {
    case 1: return two ? launch_sq<BITS, 1, 2>(a, count, s) : launch_sq<BITS, 1, 1>(a, count, s);
    case 2: return two ? launch_sq<BITS, 2, 2>(a, count, s) : launch_sq<BITS, 2, 1>(a, count, s);
    default: return two ? launch_sq<BITS, 4, 2>(a, count, s) : launch_sq<BITS, 4, 1>(a, count, s);
  }
}

}  // namespace

#ifndef TLQ_DECODE_INT2_UNIT
// The INT2 forms are compiled in decode_int2.cu (this file again, with
// TLQ_DECODE_INT2_UNIT defined), so that the two bit widths build in parallel.
tlq_status launch_decode_int2(const GemmArgs* a, int count, cudaStream_t stream);

tlq_status launch_decode(const GemmArgs* a, int count, cudaStream_t stream) {
  if (count < 1 || count > kMaxProblems)
    return set_error(TLQ_EINVAL, "decode: %d problems (1..%d per launch)", count, kMaxProblems);
  for (int i = 0; i < count; ++i) {
    if (a[i].M < 1 || a[i].M > 16) return set_error(TLQ_EINVAL, "decode: M=%d outside 1..16", a[i].M);
    if (a[i].bits != a[0].bits) return set_error(TLQ_EINVAL, "decode: mixed bit widths in one launch");
  }
  return a[0].bits == 4 ? dispatch_bits<4>(a, count, stream) : launch_decode_int2(a, count, stream);
}
#else
tlq_status launch_decode_int2(const GemmArgs* a, int count, cudaStream_t stream) {
  return dispatch_bits<2>(a, count, stream);
}
#endif

}  // namespace tlq

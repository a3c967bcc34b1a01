// Prefill path of quant_gemm (M > 16 tokens): a dense contraction on the
// 5th-generation tensor cores (tcgen05 + TMEM).
//
// Layer: C[m][n] = fp16( sum_k A[m][k] * (q[n][k] - z[n][g]) * s[n][g] ).
// Source: "Model" (TinyLoop Python API), "VRAM cost", Weights (packed INT2 /
// INT4 + FP16 scales + FP16 zeros per quantized layer); "Model", "Returns",
// item 2 (weights stay packed in GPU memory; dequantization happens in the
// GEMM, the FP16 body cache being the opt-in alternative).
//
// Tile: NMT x 128 tokens (UMMA M, NMT = 1 or 2) x 256 weight rows (UMMA N) x
// 64 k per stage, FP32 accumulators in TMEM (256 columns per 128 tokens).
// With NMT = 2 one dequantized weight tile feeds two token tiles, halving the
// dequantization work per MMA.  Warp roles (DQW = 16 dequantizing warps with
// one token tile, 8 with two):
//   warps 0 .. DQW-1  dequantize: the packed words of a stage (TMA ring) become
//              FP16 weights (q - z) * s (see GroupDq) in the UMMA K-major SWIZZLE_128B
//              layout of the B ring (two threads per weight row with one
//              token tile, one with two); after the main loop warps 0-7 drain
//              the accumulator (tcgen05.ld) in the epilogue.
//   warp DQW   TMA producer: lane 0 the activation tiles (SWIZZLE_128B),
//              lane 16 the packed weight tiles.
//   warp DQW+1 one elected thread issues tcgen05.mma (kind::f16, 4 x K=16 per
//              stage and token tile) and commits the stage release and
//              accumulator-ready barriers.
// Short-M problems split K over the CTAs of a thread-block cluster; partial
// tiles are reduced in a fixed rank order through an FP32 workspace in L2
// (deterministic, no atomics).  The workspace is the caller's: the library
// allocates nothing, and without a workspace large enough for a split the
// planner keeps K whole.  Every mbarrier wait is bounded.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace tlq {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 8;  // warps that own the TMEM accumulators in the epilogue (one row per thread)
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int kPrefetch = 3;          // scale/zero global-load distance (stages)
constexpr int W_STAGE_MAX = BN * BK * 4 / 8;  // packed bytes of one stage (INT4: 32 bytes per row)

// Ring depths, each with its own full/empty barriers: activations (SA, TMA),
// dequantized weights (SB, written by the dequantizing warps) and packed
// weights (SW, TMA).  Measured on GB300: with two token tiles a 2-deep B ring
// that frees shared memory for a 4-deep A ring is about 4% faster than 3/3;
// with one token tile 4/4/4 is best (6/2/6 was 5% slower).
template <int NMT>
struct PCfg {
  static constexpr int SA = 4;
  static constexpr int SB = NMT == 1 ? 4 : 2;
  static constexpr int SW = 4;
  static constexpr int RING = SA * NMT * A_STAGE + SB * B_STAGE;  // A and B rings (also the split-K slots)
  static constexpr int SMEM = 1024 + RING + SW * W_STAGE_MAX + 256;
  static constexpr uint32_t TMEM_COLS = 256u * NMT;
  // Dequantizing warps: one thread converts one weight row of a stage, so 8
  // warps write a stage.  With one token tile the MMAs of a stage are short
  // and the dequantization is the critical path: 16 warps, four per
  // scheduler, in two groups that take alternate stages (measured 3 % faster
  // per stage than two threads per row on every stage, and 2-4 % faster than
  // 8 warps).  With two token tiles the MMAs are the longer part: 8 warps.
  static constexpr int DQW = NMT == 1 ? 16 : 8;
  static constexpr int DQSTRIDE = DQW / 8;  // groups of 8 warps taking stages in turn
  static constexpr int DQARR = 8;           // warps that write one stage
  static constexpr int TMA_WARP = DQW, MMA_WARP = DQW + 1;
  static constexpr int THREADS = (DQW + 2) * 32;
};

static_assert(BN == kEpiWarps * 32, "one epilogue thread per weight row");
static_assert(PCfg<1>::SMEM <= 232448 && PCfg<2>::SMEM <= 232448, "shared memory");
static_assert((2 * PCfg<1>::SA + 2 * PCfg<1>::SB + 1 + 2 * PCfg<1>::SW) * 8 + 4 <= 256, "barriers fit");
static_assert((2 * PCfg<2>::SA + 2 * PCfg<2>::SB + 1 + 2 * PCfg<2>::SW) * 8 + 4 <= 256, "barriers fit");
static_assert(2 * BM * BN * 2 <= PCfg<2>::RING && BM * BN * 2 <= PCfg<1>::RING, "staged C tiles fit in the rings");

// Instruction descriptor, kind::f16: D = F32 (bits 4-5 = 1), A = B = F16,
// both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct PrefillParams {
  const uint32_t* W;
  const __half* S;
  const __half* Z;
  __half* C;
  int ldc;
  float* X;
  int ldx;
  int M, N, K, group;
  int kslice;  // k per cluster rank (multiple of BK)
  int ksplit;
  int l2_keep;  // stream the weights evict-last (kept in L2)
  int szvec;    // K/group % 8 == 0 and 16-byte aligned scale/zero arrays: 8 groups per 16-byte load
  int gshift;   // log2(group) when group is a power of two, else -1
  float* ws;    // k split: FP32 partial slices, NMT * ksplit^2 slices of BM x BN/ksplit per cluster
};

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accum)
      : "memory");
}

template <int EPI>
__device__ __forceinline__ void store_out(const PrefillParams& p, int m, int n, float v) {
  __half h = __float2half_rn(v);
  if constexpr (EPI == kEpiRelu) h = relu_half(h);
  if constexpr (EPI == kEpiResidual) {
    float* xp = p.X + (size_t)m * p.ldx + n;
    *xp = *xp + __half2float(h);
  } else {
    p.C[(size_t)m * p.ldc + n] = h;
  }
}

// LEAN: every stage is whole and every row of the tile exists (K a multiple
// of BK, N of BN), the scales and zeros take the 16-byte vector path and the
// group is a power of two, so the kernel leaves out the scalar scale/zero
// path and the body for ragged stages.  The arithmetic is the same; the
// dequantizing warps' loop is smaller (INT4 projection steps at M = 128 /
// 512 / 2048: 29.8 / 59.6 / 175.9 -> 27.1 / 58.3 / 173.2 us, measured).
template <int BITS, int EPI, int NMT, bool LEAN>
__global__ void __launch_bounds__(PCfg<NMT>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap wmap,
                   const __grid_constant__ CUtensorMap cmap, const PrefillParams p) {
  constexpr int SA = PCfg<NMT>::SA, SB = PCfg<NMT>::SB, SW = PCfg<NMT>::SW;
  constexpr uint32_t kTmemCols = PCfg<NMT>::TMEM_COLS;
  constexpr int CPW = 32 / BITS;
  constexpr int WPS = BK / CPW;                 // packed words per row per stage (8 or 4)
  constexpr int OUTW = BITS == 4 ? 4 : 8;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;                                // [SA][NMT][A_STAGE]
  constexpr int W_STAGE = BN * BK * BITS / 8;        // packed weights of one stage
  uint8_t* sb = smem + SA * NMT * A_STAGE;           // [SB][B_STAGE]
  uint8_t* sw = sb + SB * B_STAGE;                   // [SW][BN rows][BK * BITS / 8 bytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sw + SW * W_STAGE_MAX);
  uint64_t* full_a = bars;                // [SA] activation tile landed (TMA)
  uint64_t* empty_a = full_a + SA;        // [SA] the MMAs that read it completed
  uint64_t* full_b = empty_a + SA;        // [SB] dequantized weights written
  uint64_t* empty_b = full_b + SB;        // [SB] the MMAs that read them completed
  uint64_t* accum = empty_b + SB;
  uint64_t* wfull = accum + 1;            // [SW] packed tile landed (TMA)
  uint64_t* wempty = wfull + SW;          // [SW] the dequant warps read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wempty + SW);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM * NMT;
  const int rank = (int)blockIdx.z;  // == %cluster_ctarank (cluster dims (1, 1, ksplit))
  const int k0 = rank * p.kslice;
  const int klen = min(p.kslice, p.K - k0);
  const int nkb = (klen + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&full_a[i], 1);
      mbar_init(&empty_a[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&full_b[i], PCfg<NMT>::DQARR);
      mbar_init(&empty_b[i], 1);
    }
    mbar_init(accum, 1);
    for (int i = 0; i < SW; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], PCfg<NMT>::DQARR);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) pdl_launch_dependents();
  bool acc_ok = true;  // dequant warps: the accumulator is complete

  if (warp == PCfg<NMT>::TMA_WARP) {
    // ---------------- activations: TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&amap);
      pdl_wait();  // A may be written by the preceding kernel
      for (int kb = 0; kb < nkb; ++kb) {
        const int slot = kb % SA;
        if (!mbar_wait(&empty_a[slot], ((kb / SA) & 1) ^ 1, 0x201)) break;
        mbar_arrive_expect_tx(&full_a[slot], NMT * A_STAGE);
#pragma unroll
        for (int i = 0; i < NMT; ++i)
          tma_load_2d(&amap, &full_a[slot], sa + (slot * NMT + i) * A_STAGE, k0 + kb * BK, m0 + i * BM);
      }
      for (int kb = max(0, nkb - SA); kb < nkb; ++kb)
        if (!mbar_wait(&full_a[kb % SA], (kb / SA) & 1, 0x202)) break;
    } else if (lane == 16) {
      // ---------------- packed weights: TMA producer (no dependency wait: weights are inputs) ----------------
      tma_prefetch_desc(&wmap);
      for (int kb = 0; kb < nkb; ++kb) {
        const int ws = kb % SW;
        if (!mbar_wait(&wempty[ws], ((kb / SW) & 1) ^ 1, 0x208)) break;
        mbar_arrive_expect_tx(&wfull[ws], W_STAGE);
        if (p.l2_keep)
          tma_load_2d_hint(&wmap, &wfull[ws], sw + ws * W_STAGE, (k0 + kb * BK) * BITS / 32, n0, policy_evict_last());
        else
          tma_load_2d(&wmap, &wfull[ws], sw + ws * W_STAGE, (k0 + kb * BK) * BITS / 32, n0);
      }
      for (int kb = max(0, nkb - SW); kb < nkb; ++kb)
        if (!mbar_wait(&wfull[kb % SW], (kb / SW) & 1, 0x209)) break;
    }
    __syncwarp();
  } else if (warp == PCfg<NMT>::MMA_WARP) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int as = kb % SA, bs = kb % SB;
        ok = mbar_wait(&full_a[as], (kb / SA) & 1, 0x203) && mbar_wait(&full_b[bs], (kb / SB) & 1, 0x204);
        if (!ok) break;
        tc_fence_after();
        const uint32_t b0 = smem_u32(sb + bs * B_STAGE);
#pragma unroll
        for (int i = 0; i < NMT; ++i) {
          const uint32_t a0 = smem_u32(sa + (as * NMT + i) * A_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_f16(tmem + 256u * i, sw128_desc(a0 + kk * UMMA_K * 2), sw128_desc(b0 + kk * UMMA_K * 2),
                     (kb | kk) != 0);
        }
        umma_commit(&empty_a[as]);  // each commit tracks every MMA issued so far
        umma_commit(&empty_b[bs]);
      }
      umma_commit(accum);
    }
    __syncwarp();
  } else {
    // ---------------- dequantize weights into the B stages ----------------
    constexpr int STR = PCfg<NMT>::DQSTRIDE;
    const int r = (warp & 7) * 32 + lane;  // weight row inside the tile, 0..255
    const int sgrp = warp >> 3;            // this warp's group: stages sgrp, sgrp + STR, ...
    const int n = n0 + r;
    const bool row_ok = n < p.N;
    const int G = p.K / p.group;
    const __half* srow = p.S + (size_t)(row_ok ? n : 0) * G;
    const __half* zrow = p.Z + (size_t)(row_ok ? n : 0) * G;
    const bool two_groups = (BITS == 4) && (p.group < BK);  // INT4 with group 32

    // Scales/zeros.  Vector path (szvec): each thread holds its row's values
    // for a window of 8 groups in one 16-byte load per array, and the next
    // window in flight: one load pair per 8 groups instead of scattered 2-byte
    // loads every stage (those each touch 32 sectors per warp and crowd the
    // L1 that the dequantized tiles go through).  Otherwise: raw 16-bit bits,
    // kPrefetch stages ahead (the half2 broadcast happens at use, so no load
    // is waited on at issue).  The packed words come through the TMA ring.
    const bool szvec = LEAN || p.szvec != 0;
    uint4 sv = make_uint4(0, 0, 0, 0), zv = sv, svn = sv, zvn = sv;
    int win = 0;
    auto load_win = [&](int w, uint4& s4, uint4& z4) {
      if (row_ok && 8 * w < G) {
        s4 = __ldg(reinterpret_cast<const uint4*>(srow) + w);
        z4 = __ldg(reinterpret_cast<const uint4*>(zrow) + w);
      } else {
        s4 = make_uint4(0, 0, 0, 0);
        z4 = s4;
      }
    };
    if (szvec) {
      win = (k0 / p.group) >> 3;
      load_win(win, sv, zv);
      load_win(win + 1, svn, zvn);
    }
    unsigned short sring[kPrefetch][2], zring[kPrefetch][2];
    auto issue = [&](int kb, unsigned short (&sd)[2], unsigned short (&zd)[2]) {
      const int ks = k0 + kb * BK;
      const int g0 = ks / p.group;
      const int g1 = two_groups ? min(g0 + 1, G - 1) : g0;
      const unsigned short* sp = reinterpret_cast<const unsigned short*>(srow);
      const unsigned short* zp = reinterpret_cast<const unsigned short*>(zrow);
      sd[0] = row_ok ? __ldg(sp + g0) : (unsigned short)0;
      zd[0] = row_ok ? __ldg(zp + g0) : (unsigned short)0;
      sd[1] = row_ok ? __ldg(sp + g1) : (unsigned short)0;
      zd[1] = row_ok ? __ldg(zp + g1) : (unsigned short)0;
    };
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j)
      if (!szvec && sgrp + j * STR < nkb) issue(sgrp + j * STR, sring[j], zring[j]);

    // One stage: dequantize this thread's row of the packed tile into the B
    // ring (s_lo.. are raw FP16 bits of the scale / zero of the stage's first
    // and, for two groups per stage, second group).
    auto do_stage = [&](int kb, const GroupDq& g_lo, const GroupDq& g_hi) -> bool {
      // this stage's packed words: row r of the TMA tile (INT4: two 16-byte
      // chunks, swapped in rows with bit 2 set by SWIZZLE_32B; INT2: one)
      const int ws = kb % SW;
      if (!mbar_wait(&wfull[ws], (kb / SW) & 1, 0x207)) {
        return false;
      }
      uint32_t wv[WPS];  // this thread's words: the whole row of the stage
      {
        const uint32_t wr = smem_u32(sw + ws * W_STAGE) + (uint32_t)r * (BK * BITS / 8);
        if constexpr (BITS == 4) {
          const uint32_t sw32 = (uint32_t)((r >> 2) & 1) << 4;  // chunk of words 0..3
          const uint4 c0 = lds128(wr + sw32), c1 = lds128(wr + (sw32 ^ 16u));
          wv[0] = c0.x; wv[1] = c0.y; wv[2] = c0.z; wv[3] = c0.w;
          wv[4] = c1.x; wv[5] = c1.y; wv[6] = c1.z; wv[7] = c1.w;
        } else {
          const uint4 c = lds128(wr);
          wv[0] = c.x; wv[1] = c.y; wv[2] = c.z; wv[3] = c.w;
        }
      }
      const int slot = kb % SB;
      if (!mbar_wait(&empty_b[slot], ((kb / SB) & 1) ^ 1, 0x205)) {
        return false;
      }
      const uint32_t brow = smem_u32(sb + slot * B_STAGE) + (uint32_t)r * 128u;
      const int ks = k0 + kb * BK;
      if (LEAN || (row_ok && ks + BK <= p.K)) {  // full stage: no per-word checks
#pragma unroll
        for (int wj = 0; wj < WPS; ++wj) {
          const bool hi = two_groups && (wj >= WPS / 2);
          uint32_t o[OUTW];
          dequant_word<BITS>(wv[wj], hi ? g_hi : g_lo, o);
          if constexpr (BITS == 4) {
            sts128(brow + (((uint32_t)wj ^ (uint32_t)(r & 7)) << 4), o[0], o[1], o[2], o[3]);
          } else {
            sts128(brow + (((uint32_t)(2 * wj) ^ (uint32_t)(r & 7)) << 4), o[0], o[1], o[2], o[3]);
            sts128(brow + (((uint32_t)(2 * wj + 1) ^ (uint32_t)(r & 7)) << 4), o[4], o[5], o[6], o[7]);
          }
        }
      } else {
#pragma unroll
      for (int wj = 0; wj < WPS; ++wj) {
        const bool hi = two_groups && (wj >= WPS / 2);
        uint32_t o[OUTW];
        dequant_word<BITS>(wv[wj], hi ? g_hi : g_lo, o);
        const bool valid = row_ok && (ks + wj * CPW < p.K);
        if constexpr (BITS == 4) {
          const uint32_t c = (uint32_t)wj;
          const uint32_t addr = brow + ((c ^ (uint32_t)(r & 7)) << 4);
          if (valid) sts128(addr, o[0], o[1], o[2], o[3]);
          else sts128(addr, 0, 0, 0, 0);
        } else {
          const uint32_t c0 = (uint32_t)(2 * wj), c1 = c0 + 1;
          const uint32_t a0 = brow + ((c0 ^ (uint32_t)(r & 7)) << 4);
          const uint32_t a1 = brow + ((c1 ^ (uint32_t)(r & 7)) << 4);
          if (valid) {
            sts128(a0, o[0], o[1], o[2], o[3]);
            sts128(a1, o[4], o[5], o[6], o[7]);
          } else {
            sts128(a0, 0, 0, 0, 0);
            sts128(a1, 0, 0, 0, 0);
          }
        }
      }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full_b[slot]);
        mbar_arrive(&wempty[ws]);  // its words are consumed
      }
      return true;
    };

    bool ok = true;
    if (szvec) {
      // plain stage loop (no unrolled copies: the kernel's code stays small);
      // the group constants are formed once per group (a group of 128 codes
      // spans two stages), on a branch every thread takes together
      GroupDq g_lo = {}, g_hi = {};
      int gcur = -1;
      for (int kb = sgrp; kb < nkb && ok; kb += STR) {
        const int kpos = k0 + kb * BK;
        const int g0 = (LEAN || p.gshift >= 0) ? (kpos >> p.gshift) : kpos / p.group;
        if (g0 != gcur) {
          if ((g0 >> 3) > win) {  // a stage spans at most two groups: the window moves by one
            sv = svn;
            zv = zvn;
            ++win;
            load_win(win + 1, svn, zvn);
          }
          // with two groups per stage g0 is even, so g0 + 1 stays in the window
          g_lo = group_dq<BITS>(pick16(sv, g0 & 7), pick16(zv, g0 & 7));
          g_hi = two_groups ? group_dq<BITS>(pick16(sv, (g0 + 1) & 7), pick16(zv, (g0 + 1) & 7)) : g_lo;
          gcur = g0;
        }
        ok = do_stage(kb, g_lo, g_hi);
      }
    } else {
      for (int kb0 = sgrp; kb0 < nkb && ok; kb0 += kPrefetch * STR) {
#pragma unroll
        for (int j = 0; j < kPrefetch; ++j) {
          const int kb = kb0 + j * STR;
          if (kb < nkb && ok) {
            const GroupDq g_lo = group_dq<BITS>(sring[j][0], zring[j][0]);
            const GroupDq g_hi = two_groups ? group_dq<BITS>(sring[j][1], zring[j][1]) : g_lo;
            if (kb + kPrefetch * STR < nkb) issue(kb + kPrefetch * STR, sring[j], zring[j]);
            ok = do_stage(kb, g_lo, g_hi);
          }
        }
      }
    }

    // ---------------- epilogue: TMEM -> registers -> global ----------------
    acc_ok = mbar_wait(accum, 0, 0x206);
    __syncwarp();  // the warp-collective TMEM loads below need a converged warp
    tc_fence_after();
    if (warp < kEpiWarps) {  // the epilogue: one accumulator row per thread of warps 0..7
    const int q = warp & 3;        // TMEM lane quarter this warp may access
    const int half = warp >> 2;    // column half
    const int mrow = 32 * q + lane;
    if constexpr (EPI == kEpiStore || EPI == kEpiRelu) {
      if (p.ksplit == 1) {
        // Converted tiles go to shared memory (the rings are idle: every load
        // was consumed by a completed MMA) in the 128-byte-swizzled layout of
        // the C tensor map, 64 columns x 128 rows per box, and leave through
        // TMA tile stores, which drop rows past M and columns past N.
        uint8_t* so = smem;  // [NMT][4 column blocks][128 rows][128 bytes]
        if (acc_ok) {
#pragma unroll 1
          for (int ic = 0; ic < 4 * NMT; ++ic) {
            const int cc = ic & 3;
            const int mt = ic >> 2;
            const int col = half * 128 + cc * 32;
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * mt + col), v);
            uint32_t h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              __half lo = __float2half_rn(__uint_as_float(v[2 * i]));
              __half hi = __float2half_rn(__uint_as_float(v[2 * i + 1]));
              if constexpr (EPI == kEpiRelu) {
                lo = relu_half(lo);
                hi = relu_half(hi);
              }
              h[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
            }
            const uint32_t row = smem_u32(so + (mt * 4 + (col >> 6)) * (BM * 128)) + (uint32_t)mrow * 128u;
            const uint32_t c0 = (uint32_t)((col & 63) >> 3);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              sts128(row + (((c0 + j) ^ (uint32_t)(mrow & 7)) << 4), h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        named_barrier(1, kEpiWarps * 32);  // all eight epilogue warps, whatever their wait returned
        if (threadIdx.x == 0 && acc_ok) {
          pdl_wait();  // C may be read by the preceding kernel
          for (int mt = 0; mt < NMT; ++mt)
            for (int cb = 0; cb < 4; ++cb) {
              const int x = n0 + cb * 64, y = m0 + mt * BM;
              if (x < p.N && y < p.M) tma_store_2d(&cmap, so + (mt * 4 + cb) * (BM * 128), x, y);
            }
          bulk_commit_group();
          bulk_wait_all();
        }
      }
    } else if (acc_ok) {
      if (p.ksplit == 1) {
        pdl_wait();
#pragma unroll 1
        for (int ic = 0; ic < 4 * NMT; ++ic) {
          const int cc = ic & 3;
          const int mt = ic >> 2;  // token tile
          const int m = m0 + mt * BM + mrow;
          const int col = half * 128 + cc * 32;
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * mt + col), v);
          if (m < p.M) {
            if constexpr (EPI == kEpiResidual) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n0 + col + i < p.N) store_out<EPI>(p, m, n0 + col + i, __uint_as_float(v[i]));
            } else if constexpr (EPI == kEpiSwiglu) {
              // 32 rows = 16 (gate, up) pairs -> 16 outputs at column (n0 + col) / 2
#pragma unroll
              for (int c16 = 0; c16 < 2; ++c16) {
                const int nb = n0 + col + c16 * 16;
                if (nb < p.N) {  // N is a multiple of 16
                  uint32_t h[4];
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const int j = c16 * 16 + 4 * i;
                    const __half a0 = swiglu_half(__float2half_rn(__uint_as_float(v[j])),
                                                  __float2half_rn(__uint_as_float(v[j + 1])));
                    const __half a1 = swiglu_half(__float2half_rn(__uint_as_float(v[j + 2])),
                                                  __float2half_rn(__uint_as_float(v[j + 3])));
                    h[i] = (uint32_t)__half_as_ushort(a0) | ((uint32_t)__half_as_ushort(a1) << 16);
                  }
                  *reinterpret_cast<uint4*>(p.C + (size_t)m * p.ldc + nb / 2) = make_uint4(h[0], h[1], h[2], h[3]);
                }
              }
            }
          }
        }
      }
    }
    }  // epilogue warps
  }

  // ---------------- split-K: reduce partial tiles through L2 ----------------
  // Rank o owns columns [o * cpr, (o + 1) * cpr).  Every rank writes the
  // columns its peers own from TMEM into the launch's FP32 workspace: one
  // 128 x cpr slice per (token tile, owner, writer), stored as [cpr / 4][128
  // rows][4] so that a warp's 32 rows are one contiguous 512-byte store.  A
  // cluster barrier (release / acquire at cluster scope) publishes them, and
  // each owner adds, in rank order (fixed, so deterministic), its own columns
  // straight from TMEM and the peers' slices read from L2.
  // Measured: the same exchange pushed through distributed shared memory
  // (one bulk copy per peer between the ranks' shared memories) took 8-9 us
  // per launch, mostly waiting for the copies to land; per-thread remote
  // stores were slower still.
  if (p.ksplit > 1) {
    const int ks = p.ksplit;
    const int cpr = BN / ks;  // 32, 64 or 128: a 32-column TMEM block never straddles two owners
    const size_t slice = (size_t)BM * cpr;  // floats
    float* wsc = p.ws + (size_t)(blockIdx.x + gridDim.x * blockIdx.y) * NMT * ks * ks * slice;
    const int q = warp & 3, half = warp >> 2;
    const int mrow = 32 * q + lane;
    pdl_wait();  // the workspace and C may still be in use by the preceding kernel
    if (warp < kEpiWarps && acc_ok) {
#pragma unroll 1
      for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          const int col = half * 128 + cc * 32;
          const int owner = col / cpr;
          if (owner == rank) continue;  // added from TMEM by this CTA below
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * mt + col), v);
          float4* sl = reinterpret_cast<float4*>(wsc + ((size_t)(mt * ks + owner) * ks + rank) * slice);
          const int c40 = (col - owner * cpr) >> 2;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(sl + (size_t)(c40 + i) * BM + mrow,
                   make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                               __uint_as_float(v[4 * i + 3])));
        }
      }
    }
    cluster_sync();  // every rank's slices are in the workspace
    if (warp < kEpiWarps && acc_ok) {
#pragma unroll 1
      for (int mt = 0; mt < NMT; ++mt) {
        // this thread: row mrow, columns [half * cpr / 2, (half + 1) * cpr / 2) of the owned slice
        const int ncol = cpr / 2;
        const int cbeg = half * ncol;
#pragma unroll 1
        for (int cb = 0; cb < ncol; cb += 32) {
          const int w = ncol < 32 ? ncol : 32;   // 16 when cpr = 32
          const int tcol = rank * cpr + cbeg + cb;
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * mt + (tcol & ~31)), v);
          const bool upper = (tcol & 31) != 0;  // this thread's 16 columns are the upper half (w = 16)
          const int m = m0 + mt * BM + mrow;
#pragma unroll
          for (int c8 = 0; c8 < 32; c8 += 8) {
            if (c8 >= w) break;
            float own[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              own[i] = __uint_as_float(c8 < 16 ? (upper ? v[16 + c8 + i] : v[c8 + i]) : v[c8 + i]);
            float a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = 0.f;
            const int c4 = (cbeg + cb + c8) >> 2;  // column quad inside the owned slice
            for (int j = 0; j < ks; ++j) {
              if (j == rank) {
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] += own[i];
              } else {
                const float4* sl = reinterpret_cast<const float4*>(wsc + ((size_t)(mt * ks + rank) * ks + j) * slice);
                const float4 x0 = __ldcg(sl + (size_t)c4 * BM + mrow);
                const float4 x1 = __ldcg(sl + (size_t)(c4 + 1) * BM + mrow);
                a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
                a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
              }
            }
            const int n = n0 + rank * cpr + cbeg + cb + c8;
            if (m < p.M && n < p.N) {  // N is a multiple of 16 (SwiGLU) or 8: the group of 8 is whole
              if constexpr (EPI == kEpiSwiglu) {
                uint32_t hh[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  const __half x0 = swiglu_half(__float2half_rn(a[4 * i]), __float2half_rn(a[4 * i + 1]));
                  const __half x1 = swiglu_half(__float2half_rn(a[4 * i + 2]), __float2half_rn(a[4 * i + 3]));
                  hh[i] = (uint32_t)__half_as_ushort(x0) | ((uint32_t)__half_as_ushort(x1) << 16);
                }
                *reinterpret_cast<uint2*>(p.C + (size_t)m * p.ldc + n / 2) = make_uint2(hh[0], hh[1]);
              } else if constexpr (EPI == kEpiResidual) {
#pragma unroll
                for (int i = 0; i < 8; ++i) store_out<EPI>(p, m, n + i, a[i]);
              } else {
                uint32_t hh[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  __half lo = __float2half_rn(a[2 * i]), hi = __float2half_rn(a[2 * i + 1]);
                  if constexpr (EPI == kEpiRelu) {
                    lo = relu_half(lo);
                    hi = relu_half(hi);
                  }
                  hh[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
                }
                *reinterpret_cast<uint4*>(p.C + (size_t)m * p.ldc + n) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
              }
            }
          }
        }
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Whether a launch may take the lean kernel form (whole stages, whole row
// tiles; the caller adds the vector scale/zero path and a power-of-two
// group).  TLQ_PREFILL_GENERIC=1 forces the general form.
bool prefill_lean(const GemmArgs& a) {
  if (const char* e = getenv("TLQ_PREFILL_GENERIC"))
    if (atoi(e) != 0) return false;
  return a.K % BK == 0 && a.N % BN == 0;
}

// FP32 workspace of a launch with NMT token tiles per CTA and a k split of
// ks: every cluster's ks partial tiles (NMT * ks^2 slices of BM x BN/ks).
size_t split_ws_bytes(int M, int N, int nmt, int ks) {
  if (ks <= 1) return 0;
  const size_t ntile = (size_t)(N + BN - 1) / BN;
  const size_t mtile = (size_t)(M + BM * nmt - 1) / (BM * nmt);
  return ntile * mtile * (size_t)nmt * (size_t)ks * BM * BN * sizeof(float);
}

template <int BITS, int EPI, int NMT>
tlq_status launch_impl(const GemmArgs& a, int ks, cudaStream_t stream) {
  const int ntile = (a.N + BN - 1) / BN;
  const int mtile = (a.M + BM * NMT - 1) / (BM * NMT);
  const int nkb = (a.K + BK - 1) / BK;
  if (ks != 1 && ks != 2 && ks != 4 && ks != 8) return set_error(TLQ_EINVAL, "prefill: k split %d", ks);
  const int per = (nkb + ks - 1) / ks;
  const int ks_eff = (nkb + per - 1) / per;
  int ksplit = 1;
  while (ksplit < ks_eff) ksplit *= 2;  // cluster size must divide the 256 columns
  if (ksplit > ks_eff) {
    // fall back to the largest power of two whose slices are all non-empty
    ksplit = 1;
    while (ksplit * 2 <= ks_eff) ksplit *= 2;
  }
  const int per2 = (nkb + ksplit - 1) / ksplit;
  PrefillParams p;
  p.W = a.W;
  p.S = a.S;
  p.Z = a.Z;
  p.C = a.C;
  p.ldc = a.ldc;
  p.X = a.X;
  p.ldx = a.ldx;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.group = a.group;
  p.l2_keep = a.l2_keep;
  p.szvec = ((a.K / a.group) % 8 == 0 && (reinterpret_cast<uintptr_t>(a.S) & 15) == 0 &&
             (reinterpret_cast<uintptr_t>(a.Z) & 15) == 0) ? 1 : 0;
  p.gshift = -1;
  for (int sh = 5; sh < 31; ++sh)
    if ((1 << sh) == a.group) p.gshift = sh;
  p.kslice = per2 * BK;
  p.ksplit = (a.K + p.kslice - 1) / p.kslice;
  if (p.ksplit != ksplit) return set_error(TLQ_EINVAL, "prefill: inconsistent k split");

  CUtensorMap amap;
  tlq_status st = encode_tiled_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.A, (uint64_t)a.K, (uint64_t)a.M,
                                  (uint64_t)a.lda * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (st != TLQ_OK) return st;

  CUtensorMap wmap;
  const uint64_t wpr = (uint64_t)a.K * BITS / 32;  // words per row
  const uint64_t ldw = a.ldw > 0 ? (uint64_t)a.ldw : wpr;  // row stride in words
  st = encode_tiled_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, wpr, (uint64_t)a.N, ldw * 4, BK * BITS / 32, BN,
                       BITS == 4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (st != TLQ_OK) return st;

  // C as 64-column x 128-row SWIZZLE_128B boxes for the tile-store epilogue
  // (store / ReLU without a k split); unused otherwise
  CUtensorMap cmap = amap;
  if ((EPI == kEpiStore || EPI == kEpiRelu) && p.ksplit == 1) {
    st = encode_tiled_2d(&cmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.C, (uint64_t)a.N, (uint64_t)a.M,
                         (uint64_t)a.ldc * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (st != TLQ_OK) return st;
  }

  const size_t smem = (size_t)PCfg<NMT>::SMEM;
  const bool lean = prefill_lean(a) && p.szvec && p.gshift >= 0;
  auto kern = lean ? prefill_kernel<BITS, EPI, NMT, true> : prefill_kernel<BITS, EPI, NMT, false>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(prefill_kernel<BITS, EPI, NMT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(prefill_kernel<BITS, EPI, NMT, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (attr_err != cudaSuccess) return cuda_error(attr_err, "prefill: cudaFuncSetAttribute");

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)ntile, (unsigned)mtile, (unsigned)p.ksplit);
  lc.blockDim = dim3(PCfg<NMT>::THREADS, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (pdl_enabled()) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.ksplit > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = (unsigned)p.ksplit;
    ++na;
  }
  lc.attrs = attrs;
  lc.numAttrs = na;
  // k split: the partial slices go through the caller's FP32 workspace
  // (NMT * ksplit^2 slices of BM x BN/ksplit floats per cluster, i.e.
  // ksplit partial tiles); the planner only splits when it is large enough
  p.ws = nullptr;
  if (p.ksplit > 1) {
    const size_t wsb = split_ws_bytes(a.M, a.N, NMT, p.ksplit);
    if (!a.ws || a.ws_bytes < wsb)
      return set_error(TLQ_EINVAL, "prefill: a k split of %d needs a workspace of %zu bytes (%zu given)", p.ksplit,
                       wsb, a.ws ? a.ws_bytes : (size_t)0);
    p.ws = static_cast<float*>(a.ws);
  }
  cudaError_t e = cudaLaunchKernelEx(&lc, kern, amap, wmap, cmap, p);
  if (e != cudaSuccess) return cuda_error(e, "prefill: launch");
  if (log_enabled())
    fprintf(stderr,
            "[tlq] prefill int%d M=%d N=%d K=%d group=%d: %d token tile(s) per CTA, grid %dx%dx%d (kslice %d) "
            "smem=%zu%s\n",
            BITS, a.M, a.N, a.K, a.group, NMT, ntile, mtile, p.ksplit, p.kslice, smem, lean ? ", lean form" : "");
  return TLQ_OK;
}

// Clusters of `ks` CTAs of this kernel that fit on the GPU at once (one CTA
// per SM; a cluster needs ks free SMs of one GPC), from the occupancy API,
// cached per cluster size.
template <int BITS, int EPI, int NMT>
int max_clusters(int ks) {
  static std::mutex mu;
  static int cache[4] = {0, 0, 0, 0};
  const int idx = ks == 1 ? 0 : ks == 2 ? 1 : ks == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[idx] == 0) {
    int n = 0;
    if (ks == 1) {
      n = device_info().sms;
    } else {
      auto kern = prefill_kernel<BITS, EPI, NMT, false>;
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PCfg<NMT>::SMEM);
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3(1, 1, (unsigned)ks);
      lc.blockDim = dim3(PCfg<NMT>::THREADS, 1, 1);
      lc.dynamicSmemBytes = PCfg<NMT>::SMEM;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 1;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = (unsigned)ks;
      lc.attrs = &at;
      lc.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = device_info().sms / (2 * ks);  // conservative: half the SMs
      }
    }
    cache[idx] = n;
  }
  return cache[idx];
}

// Estimated time of a launch with NMT token tiles per CTA and a k split of
// ks: waves x (stages per slice x stage time + fixed cost).  The constants
// are measured on GB300 (sweeps of every projection shape at M = 256 ..
// 1024, graph-replayed): a 64-k stage takes about 0.70 us with one token
// tile and 0.77 us with two (SMs busy with other CTAs); the fixed cost
// (launch, first stage, epilogue) is about 1.6 / 3.5 us without a k split
// and 8.3 / 13.5 us with one (the partial tiles' exchange through L2).
double prefill_estimate_us(int nmt, int ks, int tiles, int nkb, int clusters) {
  const int waves = (tiles + clusters - 1) / clusters;
  const int stages = (nkb + ks - 1) / ks;
  const double stage_us = nmt == 1 ? 0.70 : 0.77;
  const double fixed_us = ks == 1 ? (nmt == 1 ? 1.6 : 3.5) : (nmt == 1 ? 8.3 : 13.5);
  return waves * (stages * stage_us + fixed_us);
}

// Token tiles per CTA (two share one dequantized weight tile) and k split:
// the candidate with the smallest estimate among NMT in {1, 2} (2 only when
// M has two token tiles) and ks in {1, 2, 4, 8} with slices of at least 4
// stages whose workspace fits in ws_bytes; ties keep the first (fewer tiles,
// smaller split).  TLQ_PREFILL_NMT=1|2 and TLQ_PREFILL_KSPLIT=1|2|4|8 force
// either choice.  Returns false when no candidate is left (a forced split
// without the workspace it needs).
struct PrefillPlan {
  int nmt, ks;
  double est_us;
};

int ks_index(int ks) { return ks == 1 ? 0 : ks == 2 ? 1 : ks == 4 ? 2 : 3; }

// The device as the planners see it: SMs, and the clusters of ks CTAs of the
// kernel with one or two token tiles that fit at once.  Queried once (the
// kernel's shared memory and threads depend on the token tiles only, so one
// bit width and epilogue stands for all).
const PlanDevice& plan_device() {
  static std::once_flag once;
  static PlanDevice d;
  std::call_once(once, [] {
    d.sms = device_info().sms;
    for (int i = 0; i < 4; ++i) {
      d.clusters[0][i] = max_clusters<4, kEpiStore, 1>(1 << i);
      d.clusters[1][i] = max_clusters<4, kEpiStore, 2>(1 << i);
    }
  });
  return d;
}

bool plan_solo(int M, int N, int K, size_t ws_bytes, const PlanDevice& dev, PrefillPlan& out) {
  int force_nmt = 0, force_ks = 0;
  if (const char* e = getenv("TLQ_PREFILL_NMT")) force_nmt = atoi(e);
  if (const char* e = getenv("TLQ_PREFILL_KSPLIT")) force_ks = atoi(e);
  if (force_nmt != 1 && force_nmt != 2) force_nmt = 0;
  const int ntile = (N + BN - 1) / BN;
  const int nkb = (K + BK - 1) / BK;
  out = PrefillPlan{1, 1, 1e30};
  for (int nmt = 1; nmt <= 2; ++nmt) {
    if (force_nmt && nmt != force_nmt) continue;
    if (nmt == 2 && M <= BM && !force_nmt) continue;
    const int tiles = ntile * ((M + BM * nmt - 1) / (BM * nmt));
    for (int ks = 1; ks <= 8; ks *= 2) {
      if (force_ks ? ks != force_ks : (ks > 1 && nkb / ks < 4)) continue;
      if (split_ws_bytes(M, N, nmt, ks) > ws_bytes) continue;
      const double t = prefill_estimate_us(nmt, ks, tiles, nkb, dev.clusters[nmt - 1][ks_index(ks)]);
      if (t < out.est_us) out = PrefillPlan{nmt, ks, t};
    }
  }
  return out.est_us < 1e29;
}

template <int BITS, int EPI>
bool plan_prefill(const GemmArgs& a, size_t ws_bytes, PrefillPlan& out) {
  return plan_solo(a.M, a.N, a.K, ws_bytes, plan_device(), out);
}

template <int BITS, int EPI>
tlq_status launch_pick(const GemmArgs& a, cudaStream_t s) {
  PrefillPlan pl;
  if (a.plan_nmt) {
    pl = PrefillPlan{a.plan_nmt, a.plan_ks, 0.0};  // a batch's joint plan (checked when it was made)
  } else if (!plan_prefill<BITS, EPI>(a, a.ws ? a.ws_bytes : 0, pl)) {
    return set_error(TLQ_EINVAL, "prefill: no k split allowed by TLQ_PREFILL_KSPLIT fits the workspace (%zu bytes)",
                     a.ws ? a.ws_bytes : (size_t)0);
  }
  if (log_enabled() && !a.plan_nmt) {
    const int c1 = plan_device().clusters[pl.nmt - 1][ks_index(pl.ks)];
    fprintf(stderr, "[tlq] prefill M=%d N=%d K=%d: %d token tile(s), k split %d (%d clusters fit), est %.1f us\n",
            a.M, a.N, a.K, pl.nmt, pl.ks, c1, pl.est_us);
  }
  return pl.nmt == 2 ? launch_impl<BITS, EPI, 2>(a, pl.ks, s) : launch_impl<BITS, EPI, 1>(a, pl.ks, s);
}

// Joint plan of problems that share the GPU.  Each problem's launch, planned
// alone, assumes it has every SM: at short M the four projections of a step
// then ask for 350-480 CTAs, most of them in k-split clusters, and together
// run 1.3-1.4x slower than the best joint choice (GB300, INT4, the D = 2048
// projections side by side, measured over every combination of token tiles
// per CTA and k split: M = 128 46.1 us planned alone, 31.0 us best; M = 512
// 85.2 and 61.2 us; M = 2048 173.2 us either way).  The estimate of a
// combination keeps each launch's own cost model (prefill_estimate_us) and
// combines the launches as
//     E = max(a, b) + 0.5 * min(a, b),
//     a = the longest launch alone (its waves x per-CTA time),
//     b = the CTA-time of all launches / SMs (the GPU's share of the work);
// the half weight on the smaller term stands for the imperfect packing of
// CTAs of different lengths (fitted to the measured combinations: within 7 %
// on average, and the best estimate is within 3 % of the best measured).
// Splits of 8 are left out: a cluster of 8 CTAs needs 8 free SMs of one GPC
// at once, which the other launches' CTAs rarely leave, and the estimate
// cannot see that (with splits of 8 allowed, its favourite at M = 128
// measured 37.9 us against the best 31.0).
constexpr int kJointMax = 4;
constexpr double kJointMix = 0.5;

struct JointCand {
  int nmt, ks;
  double t_cta;  // per-CTA time estimate (us)
  double waves;  // waves of this launch alone
  double ctas;
};

int joint_candidates(int M, int N, int K, size_t ws, const PlanDevice& dev, JointCand* out) {
  const int ntile = (N + BN - 1) / BN;
  const int nkb = (K + BK - 1) / BK;
  int n = 0;
  for (int nmt = 1; nmt <= 2; ++nmt) {
    if (nmt == 2 && M <= BM) continue;
    const int tiles = ntile * ((M + BM * nmt - 1) / (BM * nmt));
    for (int ks = 1; ks <= 4; ks *= 2) {
      if (ks > 1 && nkb / ks < 4) continue;
      if (split_ws_bytes(M, N, nmt, ks) > ws) continue;
      const int cl = dev.clusters[nmt - 1][ks_index(ks)];
      JointCand c;
      c.nmt = nmt;
      c.ks = ks;
      c.t_cta = prefill_estimate_us(nmt, ks, 1, nkb, 1);
      c.waves = (double)((tiles + cl - 1) / cl);
      c.ctas = (double)tiles * ks;
      out[n++] = c;
    }
  }
  return n;
}

}  // namespace

static bool plan_joint(const int* M, const int* N, const int* K, const size_t* ws, int n, const PlanDevice& dev, int* nmt,
                int* ks, double* est_us, double* each_us = nullptr) {
  if (n < 2 || n > kJointMax) return false;
  if (getenv("TLQ_PREFILL_NMT") || getenv("TLQ_PREFILL_KSPLIT")) return false;  // forced plans stay per launch
  const double sms = (double)dev.sms;
  JointCand cand[kJointMax][6];
  int nc[kJointMax];
  for (int i = 0; i < n; ++i) {
    if (M[i] <= 16) return false;
    nc[i] = joint_candidates(M[i], N[i], K[i], ws[i], dev, cand[i]);
    if (nc[i] == 0) return false;
  }
  // every combination (at most 6^4); ties keep fewer CTAs, then the earlier one
  int idx[kJointMax] = {0, 0, 0, 0};
  int best[kJointMax] = {0, 0, 0, 0};
  double best_e = 1e30, best_ctas = 1e30;
  for (;;) {
    double mx = 0.0, work = 0.0, ctas = 0.0;
    for (int i = 0; i < n; ++i) {
      const JointCand& c = cand[i][idx[i]];
      mx = std::max(mx, c.waves * c.t_cta);
      work += c.ctas * c.t_cta;
      ctas += c.ctas;
    }
    const double share = work / sms;
    const double e = std::max(mx, share) + kJointMix * std::min(mx, share);
    if (e < best_e * (1.0 - 1e-9) || (e <= best_e * (1.0 + 1e-9) && ctas < best_ctas)) {
      best_e = e;
      best_ctas = ctas;
      for (int i = 0; i < n; ++i) best[i] = idx[i];
    }
    int i = 0;
    while (i < n && ++idx[i] == nc[i]) idx[i++] = 0;
    if (i == n) break;
  }
  for (int i = 0; i < n; ++i) {
    nmt[i] = cand[i][best[i]].nmt;
    ks[i] = cand[i][best[i]].ks;
    if (each_us) each_us[i] = cand[i][best[i]].waves * cand[i][best[i]].t_cta;
  }
  if (est_us) *est_us = best_e;
  return true;
}

bool plan_prefill_joint(GemmArgs* a, int n, int* order) {
  if (n < 2 || n > kJointMax) return false;
  int M[kJointMax], N[kJointMax], K[kJointMax], nmt[kJointMax], ks[kJointMax];
  size_t ws[kJointMax];
  for (int i = 0; i < n; ++i) {
    M[i] = a[i].M;
    N[i] = a[i].N;
    K[i] = a[i].K;
    ws[i] = a[i].ws ? a[i].ws_bytes : 0;
  }
  double est = 0.0, each[kJointMax];
  if (!plan_joint(M, N, K, ws, n, plan_device(), nmt, ks, &est, each)) return false;
  // launch order: the longest launch first, so that its CTAs (clusters, when
  // it splits K) are placed before the shorter launches fill the SMs (GB300,
  // the four projections side by side, joint plans: 31.0 -> 29.9 us at
  // M = 128 and 62.7 -> 59.5 us at M = 512 with DOWN launched first)
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order, order + n, [&](int x, int y) { return each[x] > each[y]; });
  for (int i = 0; i < n; ++i) {
    a[i].plan_nmt = nmt[i];
    a[i].plan_ks = ks[i];
    if (log_enabled())
      fprintf(stderr, "[tlq] prefill (joint, %d side by side, est %.1f us) M=%d N=%d K=%d: %d token tile(s), k split %d\n",
              n, est, a[i].M, a[i].N, a[i].K, a[i].plan_nmt, a[i].plan_ks);
  }
  return true;
}

tlq_status prefill_plan(const int* M, const int* N, const int* K, const size_t* ws, int n, const PlanDevice* dev_in,
                        int* nmt, int* ks) {
  const PlanDevice& dev = dev_in ? *dev_in : plan_device();
  for (int i = 0; i < n; ++i) nmt[i] = ks[i] = 0;  // M <= 16: the decode kernel
  int np = 0;
  for (int i = 0; i < n; ++i) np += M[i] > 16;
  if (np == n && plan_joint(M, N, K, ws, n, dev, nmt, ks, nullptr)) return TLQ_OK;
  for (int i = 0; i < n; ++i) {
    if (M[i] <= 16) continue;
    PrefillPlan pl;
    if (!plan_solo(M[i], N[i], K[i], ws[i], dev, pl))
      return set_error(TLQ_EINVAL, "tl_prefill_plan[%d]: no k split allowed by TLQ_PREFILL_KSPLIT fits the workspace",
                       i);
    nmt[i] = pl.nmt;
    ks[i] = pl.ks;
  }
  return TLQ_OK;
}

namespace {

template <int BITS>
size_t workspace_bits(const GemmArgs& a) {
  PrefillPlan pl;
  const size_t unlimited = ~(size_t)0;
  bool ok;
  switch (a.epi) {
    case kEpiStore: ok = plan_prefill<BITS, kEpiStore>(a, unlimited, pl); break;
    case kEpiRelu: ok = plan_prefill<BITS, kEpiRelu>(a, unlimited, pl); break;
    case kEpiSwiglu: ok = plan_prefill<BITS, kEpiSwiglu>(a, unlimited, pl); break;
    default: ok = plan_prefill<BITS, kEpiResidual>(a, unlimited, pl); break;
  }
  return ok ? split_ws_bytes(a.M, a.N, pl.nmt, pl.ks) : 0;
}

template <int BITS>
tlq_status dispatch_epi(const GemmArgs& a, cudaStream_t s) {
  switch (a.epi) {
    case kEpiStore: return launch_pick<BITS, kEpiStore>(a, s);
    case kEpiRelu: return launch_pick<BITS, kEpiRelu>(a, s);
    case kEpiSwiglu: return launch_pick<BITS, kEpiSwiglu>(a, s);
    default: return launch_pick<BITS, kEpiResidual>(a, s);
  }
}

}  // namespace

size_t prefill_workspace_bytes(const GemmArgs& a) {
  if (a.M <= 16) return 0;
  return a.bits == 4 ? workspace_bits<4>(a) : workspace_bits<2>(a);
}

tlq_status launch_prefill(const GemmArgs& a, cudaStream_t stream) {
  if (a.lda % 8) return set_error(TLQ_EINVAL, "prefill: lda=%d must be a multiple of 8", a.lda);
  return a.bits == 4 ? dispatch_epi<4>(a, stream) : dispatch_epi<2>(a, stream);
}

}  // namespace tlq

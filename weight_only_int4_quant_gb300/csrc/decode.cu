// Decode path of quant_gemm (M <= 16 tokens): bandwidth-bound, one pass over
// the packed weights.
//
// Layer: C[m][n] = fp16( sum_k A[m][k] * (q[n][k] - z[n][g]) * s[n][g] ).
// Source: "Model" (TinyLoop Python API), "VRAM cost", Weights (INT2 / INT4
// packed data + FP16 scales + FP16 zeros per quantized layer); "beta-Informed
// Deployment Features", CTX-TIER: the INT2 kernel's smaller footprint is what
// speeds decode up, so the kernel is built to stream weight bytes at HBM rate.
//
// Design (GB300):
//  * A producer warp streams 64- or 32-row x 64-byte tiles of packed words into
//    a ring of shared-memory stages with TMA (SWIZZLE_64B, so that the
//    transposed word reads below are bank-conflict free).
//  * Four consumer warps each own whole k-blocks (16 words per row).  A k-block
//    is split into four "sets"; in a set, lane c of a row takes word c, so the
//    four lanes that feed one MMA row hold 4*32/bits consecutive codes that lie
//    in one quantization group.
//  * Codes become FP16 MMA operands with one LOP3 per pair: a code at mantissa
//    bit position p of a half with exponent e reads as 2^e + q exactly (the
//    "base" of that position: 1024, 256, 64, 16 or 4).  The MMA then sums
//    a * (base + q); the base term and the zero point are removed per set with
//    two row-independent correction sums (sum_k base_k a_k and sum_k a_k) that
//    one extra MMA per word computes for all rows at once:
//        acc_set = sum_k a_k (base_k + q_k) - sum_k base_k a_k - z * sum_k a_k
//                = sum_k a_k (q_k - z)
//        total  += s * acc_set           (FP32)
//  * Tokens are the MMA's N dimension (one or two 8-wide tiles), weight rows
//    its M dimension (m16n8k16, "swap AB").
//  * K is split across the four warps and, for short/wide shapes, across the
//    CTAs of a thread-block cluster; partial sums are reduced in a fixed order
//    through shared / distributed shared memory (no atomics: deterministic).
//  * Programmatic dependent launch: weights and scales are fetched before
//    griddepcontrol.wait, activations and the output only after it.
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace tlq {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 8;                 // multiple of kConsumerWarps
constexpr int kWordsPerKBlock = 16;        // per row, 64 bytes
constexpr int kStageRowBytes = kWordsPerKBlock * 4;

template <int BITS>
struct Fmt {
  static constexpr int CPW = 32 / BITS;            // codes per word
  static constexpr int KBLK = kWordsPerKBlock * CPW; // codes per k-block
  static constexpr int SETC = 4 * CPW;             // codes per set
  static constexpr int MPS = CPW / 4;              // MMAs per word (k16 each)
  // activation row stride (halves): stride*2 bytes == kActMod (mod 128) makes the
  // per-lane 16-byte activation loads conflict free.
  static constexpr int kActMod = BITS == 4 ? 64 : 16;
};

struct DecodeParams {
  const __half* A;
  int lda;
  const __half* S;
  const __half* Z;
  __half* C;
  int ldc;
  float* X;
  int ldx;
  int M, N, K, group;
  int kslice;      // codes per CTA (multiple of KBLK)
  int act_stride;  // halves
  int gsp;         // padded groups per row in the s/z tile
  int gs_count;    // groups touched by one K slice (<= gsp)
  int ksplit;      // CTAs per cluster along K
};

// Byte offset of word w of row r inside a SWIZZLE_64B stage (64-byte rows).
__device__ __forceinline__ uint32_t swz64(int r, int w) {
  return (uint32_t)(r * kStageRowBytes + ((((w >> 2) ^ (r >> 1)) & 3) << 4) + ((w & 3) << 2));
}

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

template <int BITS, int RGW, int NT, int EPI>
__global__ void __launch_bounds__(kThreads, NT == 2 ? 2 : 3)
    decode_kernel(const __grid_constant__ CUtensorMap wmap, const DecodeParams p) {
  using F = Fmt<BITS>;
  constexpr int ROWS = 16 * RGW;
  constexpr int STAGE_BYTES = ROWS * kStageRowBytes;
  constexpr int MT = 8 * NT;  // token slots

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  __half* act = reinterpret_cast<__half*>(smem + kStages * STAGE_BYTES);
  float2* sz = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(act) + (size_t)p.M * p.act_stride * 2);
  float* part = reinterpret_cast<float*>(sz + ROWS * p.gsp);          // [ROWS][MT]
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + ROWS * MT);     // full[S], empty[S]
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  float* red = reinterpret_cast<float*>(stages);  // reused after the main loop

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int row0 = blockIdx.x * ROWS;
  const int rank = (int)blockIdx.y;  // == %cluster_ctarank (cluster dims (1, ksplit, 1))
  const int kslice0 = rank * p.kslice;
  const int klen = min(p.kslice, p.K - kslice0);
  const int nkb = (klen + F::KBLK - 1) / F::KBLK;
  const int gs0 = kslice0 / p.group;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer: TMA weight tiles ----------------
    if (lane == 0) {
      tma_prefetch_desc(&wmap);
      const uint64_t pol = policy_evict_first();
      const int x0 = kslice0 / F::CPW;
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int slot = kb % kStages;
        ok = mbar_wait(&empty[slot], ((kb / kStages) & 1) ^ 1, 0x101);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[slot], STAGE_BYTES);
        tma_load_2d_hint(&wmap, &full[slot], stages + slot * STAGE_BYTES, x0 + kb * kWordsPerKBlock, row0, pol);
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int kb = max(0, nkb - kStages); kb < nkb; ++kb)
        if (!mbar_wait(&full[kb % kStages], (kb / kStages) & 1, 0x102)) break;
    }
    __syncwarp();
  } else {
    // ---------------- consumers ----------------
    // scales / zeros of this CTA's rows and K slice (independent of the previous kernel)
    const int G = p.K / p.group;
    for (int i = tid; i < ROWS * p.gs_count; i += kConsumerWarps * 32) {
      const int r = i / p.gs_count, j = i - r * p.gs_count;
      const int n = row0 + r;
      float2 v = make_float2(0.f, 0.f);
      if (n < p.N && gs0 + j < G) {
        const size_t o = (size_t)n * G + gs0 + j;
        v.x = __half2float(p.S[o]);
        v.y = __half2float(p.Z[o]);
      }
      sz[r * p.gsp + j] = v;
    }
    pdl_wait();  // activations may come from the preceding kernel
    // activations of this K slice, zero beyond K
    {
      const int chunks = p.kslice / 8;  // 16-byte chunks per token row
      for (int i = tid; i < p.M * chunks; i += kConsumerWarps * 32) {
        const int m = i / chunks, ch = i - m * chunks;
        const int k = kslice0 + ch * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k < p.K) v = *reinterpret_cast<const uint4*>(p.A + (size_t)m * p.lda + k);
        *reinterpret_cast<uint4*>(act + (size_t)m * p.act_stride + ch * 8) = v;
      }
    }
    named_barrier(1, kConsumerWarps * 32);

    const int g = lane >> 2;
    const int c = lane & 3;
    float tot[RGW][NT][4];
#pragma unroll
    for (int r = 0; r < RGW; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[r][t][i] = 0.f;

    const uint32_t act_base = smem_u32(act);
    const uint32_t sz_base = smem_u32(sz);
    for (int kb = warp; kb < nkb; kb += kConsumerWarps) {
      const int slot = kb % kStages;
      if (!mbar_wait(&full[slot], (kb / kStages) & 1, 0x103)) break;
      const uint32_t wbase = smem_u32(stages + slot * STAGE_BYTES);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int set_rel = kb * F::KBLK + q * F::SETC;
        if (set_rel >= klen) break;
        const int gl = (kslice0 + set_rel) / p.group - gs0;
        // ---- B fragments (activations) and the per-set correction sums ----
        uint32_t bf[NT][F::MPS][2];
        float corr[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int tok = 8 * t + g;
          uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
          if (tok < p.M) {
            const uint32_t a = act_base + (uint32_t)((tok * p.act_stride + set_rel + c * F::CPW) * 2);
            x = lds128(a);
            if constexpr (BITS == 2) y = lds128(a + 16);
          }
          if constexpr (BITS == 4) {
            // codes of the word: x = (a0,a1)(a2,a3)(a4,a5)(a6,a7); pairs (0,4)(1,5) | (2,6)(3,7)
            bf[t][0][0] = prmt(x.x, x.z, 0x5410);
            bf[t][0][1] = prmt(x.x, x.z, 0x7632);
            bf[t][1][0] = prmt(x.y, x.w, 0x5410);
            bf[t][1][1] = prmt(x.y, x.w, 0x7632);
          } else {
            // x = a0..a7, y = a8..a15; pairs (2e, 2e+8) and (2e+1, 2e+9)
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
            const uint32_t ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              bf[t][e][0] = prmt(xs[e], ys[e], 0x5410);
              bf[t][e][1] = prmt(xs[e], ys[e], 0x7632);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) corr[t][i] = 0.f;
#pragma unroll
          for (int e = 0; e < F::MPS; ++e) {
            const uint4 ka = correction_frag<BITS>(e);
            mma_16816(corr[t], ka.x, ka.y, ka.z, ka.w, bf[t][e][0], bf[t][e][1]);
          }
        }
        // ---- weight rows ----
#pragma unroll
        for (int r = 0; r < RGW; ++r) {
          const int rg = 16 * r + g;
          const uint32_t wg = lds32(wbase + swz64(rg, 4 * q + c));
          const uint32_t wh = lds32(wbase + swz64(rg + 8, 4 * q + c));
          const float2 szg = lds64f(sz_base + (uint32_t)((rg * p.gsp + gl) * 8));
          const float2 szh = lds64f(sz_base + (uint32_t)(((rg + 8) * p.gsp + gl) * 8));
          uint32_t pg[F::CPW / 2], ph[F::CPW / 2];
          unpack_word<BITS>(wg, pg);
          unpack_word<BITS>(wh, ph);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float acc[4];
            acc[0] = fmaf(szg.y, corr[t][2], corr[t][0]);
            acc[1] = fmaf(szg.y, corr[t][3], corr[t][1]);
            acc[2] = fmaf(szh.y, corr[t][2], corr[t][0]);
            acc[3] = fmaf(szh.y, corr[t][3], corr[t][1]);
#pragma unroll
            for (int e = 0; e < F::MPS; ++e)
              mma_16816(acc, pg[2 * e], ph[2 * e], pg[2 * e + 1], ph[2 * e + 1], bf[t][e][0], bf[t][e][1]);
            tot[r][t][0] = fmaf(szg.x, acc[0], tot[r][t][0]);
            tot[r][t][1] = fmaf(szg.x, acc[1], tot[r][t][1]);
            tot[r][t][2] = fmaf(szh.x, acc[2], tot[r][t][2]);
            tot[r][t][3] = fmaf(szh.x, acc[3], tot[r][t][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // all consumers done with the stage buffers -> reuse them for the reduction
    named_barrier(1, kConsumerWarps * 32);
    {
      float* my = red + warp * (ROWS * MT);
#pragma unroll
      for (int r = 0; r < RGW; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int ra = 16 * r + g, tk = 8 * t + 2 * c;
          my[ra * MT + tk] = tot[r][t][0];
          my[ra * MT + tk + 1] = tot[r][t][1];
          my[(ra + 8) * MT + tk] = tot[r][t][2];
          my[(ra + 8) * MT + tk + 1] = tot[r][t][3];
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    for (int i = tid; i < ROWS * MT; i += kConsumerWarps * 32) {
      float v = red[i];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) v += red[w * ROWS * MT + i];
      part[i] = v;
    }
  }

  // ---------------- cross-CTA (cluster) reduction and epilogue ----------------
  __syncwarp();
  if (p.ksplit > 1) cluster_sync();
  else __syncthreads();
  {
    // rank r finalizes rows [r * rpr, min(ROWS, (r + 1) * rpr)) of the tile
    const int rpr = (ROWS + p.ksplit - 1) / p.ksplit;
    const int rbeg = rank * rpr;
    const int rcnt = max(0, min(ROWS, rbeg + rpr) - rbeg);
    const int mt = p.M < MT ? p.M : MT;
    const uint32_t part_addr = smem_u32(part);
    for (int i = tid; i < rcnt * mt; i += kThreads) {
      const int tk = i / rcnt;
      const int r = rbeg + (i - tk * rcnt);
      const int n = row0 + r;
      float v;
      if (p.ksplit > 1) {
        v = 0.f;
        for (int j = 0; j < p.ksplit; ++j)
          v += ld_shared_cluster_f32(map_shared_rank(part_addr + (uint32_t)((r * MT + tk) * 4), (uint32_t)j));
      } else {
        v = part[r * MT + tk];
      }
      if (n < p.N) {
        __half h = __float2half_rn(v);
        if constexpr (EPI == kEpiRelu) h = relu_half(h);
        if constexpr (EPI == kEpiResidual) {
          float* xp = p.X + (size_t)tk * p.ldx + n;
          *xp = *xp + __half2float(h);
        } else {
          p.C[(size_t)tk * p.ldc + n] = h;
        }
      }
    }
  }
  __syncwarp();
  if (p.ksplit > 1) cluster_sync();  // keep shared memory alive until all ranks have read it
}

struct DecodeCfg {
  int rgw;     // row groups (16 rows) per warp: 4 or 2
  int ksplit;  // cluster size along K
  int kslice;  // codes per CTA
};

template <int BITS>
DecodeCfg choose_cfg(int M, int N, int K, int sms) {
  const int kblk = Fmt<BITS>::KBLK;
  const int nkb = (K + kblk - 1) / kblk;
  DecodeCfg best{4, 1, nkb * kblk};
  long best_score = -1;
  const char* env = getenv("TLQ_DECODE_CFG");  // "rgw,ksplit" (tuning sweeps)
  if (env) {
    int a = 0, b = 0;
    if (sscanf(env, "%d,%d", &a, &b) == 2 && (a == 2 || a == 4) && b >= 1 && b <= 8) {
      const int per = (nkb + b - 1) / b;
      return DecodeCfg{a, (nkb + per - 1) / per, per * kblk};
    }
  }
  for (int rgw : {4, 2}) {
    for (int ks : {1, 2, 4, 8}) {
      if (ks > nkb) continue;
      const int per = (nkb + ks - 1) / ks;
      const int ks_eff = (nkb + per - 1) / per;
      const long ctas = (long)((N + 16 * rgw - 1) / (16 * rgw)) * ks_eff;
      // score: enough CTAs to cover the GPU twice, all four warps busy, then
      // prefer fewer cluster ranks and wider row tiles
      long score = 0;
      score += (ctas >= 2L * sms) ? 4000 : (ctas * 4000) / (2L * sms);
      score += (per >= kConsumerWarps) ? 1000 : per * 250;
      score -= ks_eff * 10;
      score += rgw * 5;
      if ((long)M * (per * kblk + 64) * 2 > 96 * 1024) score -= 100000;  // activation tile too large
      if (score > best_score) {
        best_score = score;
        best = DecodeCfg{rgw, ks_eff, per * kblk};
      }
    }
  }
  return best;
}

template <int BITS, int RGW, int NT, int EPI>
tlq_status launch_impl(const GemmArgs& a, const DecodeCfg& cfg, cudaStream_t stream) {
  using F = Fmt<BITS>;
  constexpr int ROWS = 16 * RGW;
  constexpr int MT = 8 * NT;
  DecodeParams p;
  p.A = a.A;
  p.lda = a.lda;
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
  p.kslice = cfg.kslice;
  p.ksplit = cfg.ksplit;
  // activation row stride: >= kslice, stride*2 == kActMod (mod 128)
  {
    int s = cfg.kslice;
    while ((s * 2) % 128 != F::kActMod) s += 8;
    p.act_stride = s;
  }
  // groups touched by one slice: at most kslice/group + 1 (slices start on k-block bounds)
  const int gcount = (cfg.kslice + a.group - 1) / a.group + 1;
  p.gs_count = gcount;
  p.gsp = gcount | 1;

  CUtensorMap map;
  const uint64_t wpr = (uint64_t)a.K / F::CPW;
  tlq_status st = encode_tiled_2d(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, wpr, (uint64_t)a.N, wpr * 4,
                                  kWordsPerKBlock, ROWS, CU_TENSOR_MAP_SWIZZLE_64B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (st != TLQ_OK) return st;

  const size_t smem = 1024 + (size_t)kStages * ROWS * kStageRowBytes + (size_t)a.M * p.act_stride * 2 +
                      (size_t)ROWS * p.gsp * 8 + (size_t)ROWS * MT * 4 + 2 * kStages * 8;
  static_assert(kConsumerWarps * ROWS * MT * 4 <= kStages * ROWS * kStageRowBytes, "reduction buffer");
  if (smem > (size_t)device_info().smem_optin)
    return set_error(TLQ_EUNSUPPORTED, "decode: shared memory %zu exceeds the device limit", smem);

  auto kern = decode_kernel<BITS, RGW, NT, EPI>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    device_info().smem_optin);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess) return cuda_error(attr_err, "decode: cudaFuncSetAttribute");

  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)((a.N + ROWS - 1) / ROWS), (unsigned)cfg.ksplit, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cfg.ksplit > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = (unsigned)cfg.ksplit;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  lc.attrs = attrs;
  lc.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&lc, kern, map, p);
  if (e != cudaSuccess) return cuda_error(e, "decode: launch");
  if (log_enabled()) {
    fprintf(stderr, "[tlq] decode int%d M=%d N=%d K=%d group=%d: rows/CTA=%d ksplit=%d kslice=%d grid=%u smem=%zu\n",
            BITS, a.M, a.N, a.K, a.group, ROWS, cfg.ksplit, cfg.kslice, lc.gridDim.x * lc.gridDim.y, smem);
  }
  return TLQ_OK;
}

template <int BITS, int RGW, int NT>
tlq_status dispatch_epi(const GemmArgs& a, const DecodeCfg& cfg, cudaStream_t s) {
  switch (a.epi) {
    case kEpiStore: return launch_impl<BITS, RGW, NT, kEpiStore>(a, cfg, s);
    case kEpiRelu: return launch_impl<BITS, RGW, NT, kEpiRelu>(a, cfg, s);
    default: return launch_impl<BITS, RGW, NT, kEpiResidual>(a, cfg, s);
  }
}

template <int BITS>
tlq_status dispatch_bits(const GemmArgs& a, cudaStream_t s) {
  const DecodeCfg cfg = choose_cfg<BITS>(a.M, a.N, a.K, device_info().sms);
  const bool two = a.M > 8;
  if (cfg.rgw == 4) return two ? dispatch_epi<BITS, 4, 2>(a, cfg, s) : dispatch_epi<BITS, 4, 1>(a, cfg, s);
  return two ? dispatch_epi<BITS, 2, 2>(a, cfg, s) : dispatch_epi<BITS, 2, 1>(a, cfg, s);
}

}  // namespace

tlq_status launch_decode(const GemmArgs& a, cudaStream_t stream) {
  if (a.M < 1 || a.M > 16) return set_error(TLQ_EINVAL, "decode: M=%d outside 1..16", a.M);
  return a.bits == 4 ? dispatch_bits<4>(a, stream) : dispatch_bits<2>(a, stream);
}

}  // namespace tlq

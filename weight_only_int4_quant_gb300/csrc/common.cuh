// Shared device/host helpers of libtlq (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tlq.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libtlq is written for sm_103a (Blackwell) only"
#endif

namespace tlq {

// ---------------------------------------------------------------------------
// Device status word: kernels that give up on a bounded wait record it here.
// ---------------------------------------------------------------------------
enum : uint32_t { kStatusOk = 0, kStatusTimeout = 1 };
extern __device__ uint32_t g_status;
extern __device__ uint32_t g_status_where;  // site id of the first timeout

// 1 second of wall time per wait; far above any legitimate wait here.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_timeout(uint32_t where) {
  if (atomicCAS(&g_status, kStatusOk, kStatusTimeout) == kStatusOk) g_status_where = where;
}

// ---------------------------------------------------------------------------
// Shared-memory address helpers and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, records the timeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        record_timeout(where);
        return false;
      }
    }
  }
}

// Same with a caller-chosen limit (used by the timeout self-test).
__device__ __forceinline__ bool mbar_wait_ns(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                             uint32_t where) {
  uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_timeout(where);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Tile store shared -> global through a tensor map (bulk-group completion);
// elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every bulk store of this thread has completed (its global writes included)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Wait until the preceding grid (programmatic dependency) has completed and
// its memory is visible.  A no-op when launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid in the stream to start launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Register-level helpers
// ---------------------------------------------------------------------------
template <uint32_t kLut>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(kLut));
  return d;
}

// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  return lop3<(0xF0 & 0xCC) | 0xAA>(a, b, c);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Epilogue kinds shared by the GEMM kernels.  kEpiSwiglu: the weight rows are
// (gate, up) pairs, rows 2i and 2i+1; output column i (row stride ldc) is
// swiglu_half(fp16(acc[2i]), fp16(acc[2i+1])).
enum Epilogue : int { kEpiStore = 0, kEpiRelu = 1, kEpiResidual = 2, kEpiSwiglu = 3 };

__device__ __forceinline__ __half relu_half(__half v) {
  return (__half2float(v) > 0.f) ? v : __float2half_rn(0.f);
}

// fp16(silu(g) * u), silu(g) = g / (1 + exp(-g)), on the FP16 GEMM outputs
// ("Model", ffn_dim: the gate and up projections of SwiGLU).  FP32 with the
// hardware exponential and the approximate divide: silu's relative error is
// about 2^-20, far below FP16's 2^-11, and it keeps the decode kernel's
// register budget (an IEEE divide here spills).  For g below about -87 the
// divide returns 0 (silu's limit).
__device__ __forceinline__ __half swiglu_half(__half g, __half u) {
  const float gf = __half2float(g);
  return __float2half_rn(__fdividef(gf, 1.0f + __expf(-gf)) * __half2float(u));
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct GemmArgs {
  const __half* A;
  int lda;
  const uint32_t* W;
  const __half* S;
  const __half* Z;
  __half* C;
  int ldc;
  float* X;  // residual for kEpiResidual (row stride ldx)
  int ldx;
  int M, N, K, bits, group;
  int epi;
  int l2_keep = 0;       // 1: stream the weights with an L2 evict-last policy (reused soon, e.g. the loop block)
  int ldw = 0;           // packed-weight row stride in 32-bit words (0: compact rows of K*bits/32 words)
  void* ws = nullptr;    // caller-owned workspace for the prefill kernel's k split (nullptr: no k split)
  size_t ws_bytes = 0;
  int plan_nmt = 0;      // prefill: token tiles per CTA and k split chosen for a batch (0: the launch's own plan)
  int plan_ks = 0;
};

// Error reporting (thread-local message)
tlq_status set_error(tlq_status st, const char* fmt, ...);
// Clears the calling thread's message (every entry point starts with it).
void clear_error();
tlq_status cuda_error(cudaError_t e, const char* what);

// Tensor-map encoding through the driver entry point (no -lcuda needed).
tlq_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                           uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                           CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo);

struct DeviceInfo {
  int sms;
  int l2_bytes;
  int smem_optin;
};
const DeviceInfo& device_info();

bool log_enabled();
// Programmatic dependent launch between the library's kernels (default on;
// TLQ_PDL=0 turns it off).
bool pdl_enabled();

// Kernel launchers (each validates its own limits; the API validated shapes).
// launch_decode runs up to kMaxDecodeProblems independent M <= 16 problems of
// one bit width in a single persistent launch.
constexpr int kMaxDecodeProblems = 16;
tlq_status launch_decode(const GemmArgs* a, int count, cudaStream_t stream);
tlq_status launch_prefill(const GemmArgs& a, cudaStream_t stream);
// Workspace bytes the prefill kernel's planner would use for this problem with
// an unlimited workspace (0: it would not split K).
size_t prefill_workspace_bytes(const GemmArgs& a);
// Plans of n prefill problems that will run side by side (the batched call's
// side streams): sets every a[i].plan_nmt / plan_ks, and order[] to the
// order to launch them in (the longest first).  Returns false (and leaves
// the plans unset) when it does not plan jointly.
bool plan_prefill_joint(GemmArgs* a, int n, int* order);
// The device as the prefill planners see it: SMs, and for one and two token
// tiles per CTA the clusters of 1, 2, 4 and 8 CTAs that fit at once.
struct PlanDevice {
  int sms;
  int clusters[2][4];
};
// The plans of n problems (token tiles per CTA and k split; 0 and 0 for
// M <= 16, the decode kernel): joint when all n (2..4) run side by side as in
// a batched call, else each planned alone.  dev NULL: the current device.
tlq_status prefill_plan(const int* M, const int* N, const int* K, const size_t* ws, int n, const PlanDevice* dev,
                        int* nmt, int* ks);
tlq_status loop_block_forward_named(float* x, const tl_block* b, int L, int M, const char* who, void* stream);
tlq_status launch_pack(const uint8_t* codes, uint32_t* W, int N, int K, int bits, cudaStream_t stream);
tlq_status launch_unpack(const uint32_t* W, uint8_t* codes, int N, int K, int bits, cudaStream_t stream);
// INT4 -> INT2 re-quantization of up to kMaxRequantProblems weights sharing
// one group size, in one persistent launch.
constexpr int kMaxRequantProblems = 16;
struct RequantArgs {
  const uint32_t* W4;
  const uint16_t* s4;
  const uint16_t* z4;
  uint32_t* W2;  // == W4: in place (INT2 rows keep the INT4 row stride of K/8 words)
  uint16_t* s2;
  uint16_t* z2;
  int N, K;
};
tlq_status launch_requant(const RequantArgs* a, int count, int group, cudaStream_t stream);
// The in-place conversions of a batch (every problem has W2 == W4), one launch.
tlq_status launch_requant_in_place(const RequantArgs* a, int count, int group, cudaStream_t stream);
tlq_status launch_body(const uint32_t* W, const uint16_t* s, const uint16_t* z, uint16_t* out, int N, int K, int bits,
                       int group, cudaStream_t stream);
tlq_status launch_rmsnorm(const float* x, __half* h, int M, int D, int normalize, cudaStream_t stream);
tlq_status launch_timeout_probe(uint32_t limit_us, cudaStream_t stream);

}  // namespace tlq

// C ABI of libtlq: argument validation, dispatch and error reporting.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace tlq {

namespace {
thread_local char g_msg[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

tlq_status set_error(tlq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_msg[0] = 0; }

tlq_status cuda_error(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TLQ_OK;
  return set_error(TLQ_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool log_enabled() {
  static const bool on = [] {
    const char* v = getenv("TLQ_LOG");
    return v && v[0] && strcmp(v, "0") != 0;
  }();
  return on;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("TLQ_PDL");
    return !(v && strcmp(v, "0") == 0);
  }();
  return on;
}

const DeviceInfo& device_info() {
  static DeviceInfo info = [] {
    DeviceInfo d{148, 128 << 20, 227 * 1024};
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
      cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
      cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev);
      cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return d;
  }();
  return info;
}

tlq_status encode_tiled_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                           uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                           CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  static cudaError_t load_err = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    load_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (load_err == cudaSuccess && q != cudaDriverEntryPointSuccess) load_err = cudaErrorSymbolNotFound;
    fn = reinterpret_cast<EncodeFn>(p);
  });
  if (load_err != cudaSuccess || !fn) return cuda_error(load_err, "cuTensorMapEncodeTiled lookup");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(TLQ_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d): dims %llu x %llu, row %llu B, box %u x %u",
                     (int)r, (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)row_bytes,
                     box_inner, box_outer);
  return TLQ_OK;
}

// Shape rules shared by every GEMM entry point.
tlq_status check_gemm_shape(int M, int N, int K, int bits, int group, const char* who) {
  if (bits != 4 && bits != 2) return set_error(TLQ_EINVAL, "%s: bits=%d (must be 4 or 2)", who, bits);
  if (M < 1) return set_error(TLQ_EINVAL, "%s: M=%d (must be >= 1)", who, M);
  if (N < 1) return set_error(TLQ_EINVAL, "%s: N=%d (must be >= 1)", who, N);
  if (K < 1) return set_error(TLQ_EINVAL, "%s: K=%d (must be >= 1)", who, K);
  const int unit = bits == 4 ? 32 : 64;
  if (group < unit || group % unit)
    return set_error(TLQ_EINVAL, "%s: group=%d (must be a positive multiple of %d for INT%d)", who, group, unit, bits);
  if (K % group) return set_error(TLQ_EINVAL, "%s: K=%d is not a multiple of group=%d", who, K, group);
  return TLQ_OK;
}

tlq_status run_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.M <= 16) return launch_decode(&a, 1, stream);
  return launch_prefill(a, stream);
}

// Validation shared by tl_quant_gemm and tl_quant_gemm_batched.
tlq_status check_gemm_call(const uint16_t* A, const uint32_t* W, const uint16_t* S, const uint16_t* Z,
                           const uint16_t* C, int M, int N, int K, int bits, int group, const char* who) {
  if (!A || !W || !S || !Z || !C)
    return set_error(TLQ_EINVAL, "%s: null pointer (A=%p W=%p scales=%p zeros=%p C=%p)", who, (const void*)A,
                     (const void*)W, (const void*)S, (const void*)Z, (const void*)C);
  tlq_status st = check_gemm_shape(M, N, K, bits, group, who);
  if (st != TLQ_OK) return st;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C))
    return set_error(TLQ_EINVAL, "%s: A, Wpacked and C must be 16-byte aligned", who);
  if (N % 8) return set_error(TLQ_EINVAL, "%s: N=%d must be a multiple of 8", who, N);
  return TLQ_OK;
}

// Row stride of a packed weight in words: 0 (compact) or at least the row's
// words, a multiple of 4 (16-byte rows for the tensor maps).
tlq_status check_ldw(int ldw, int K, int bits, const char* who) {
  const int wpr = K / (32 / bits);
  if (ldw != 0 && (ldw < wpr || ldw % 4))
    return set_error(TLQ_EINVAL, "%s: ldw=%d (0, or >= K*bits/32 = %d and a multiple of 4)", who, ldw, wpr);
  return TLQ_OK;
}

tlq_status check_workspace(const void* ws, size_t bytes, const char* who) {
  if (ws && !aligned16(ws)) return set_error(TLQ_EINVAL, "%s: workspace must be 16-byte aligned", who);
  if (!ws && bytes) return set_error(TLQ_EINVAL, "%s: null workspace with %zu bytes", who, bytes);
  return TLQ_OK;
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const char* a0 = static_cast<const char*>(a);
  const char* b0 = static_cast<const char*>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

GemmArgs plain_args(const uint16_t* A, const uint32_t* W, const uint16_t* S, const uint16_t* Z, uint16_t* C, int M,
                    int N, int K, int bits, int group, int ldw = 0, void* ws = nullptr, size_t ws_bytes = 0) {
  GemmArgs a;
  a.A = reinterpret_cast<const __half*>(A);
  a.lda = K;
  a.W = W;
  a.S = reinterpret_cast<const __half*>(S);
  a.Z = reinterpret_cast<const __half*>(Z);
  a.C = reinterpret_cast<__half*>(C);
  a.ldc = N;
  a.X = nullptr;
  a.ldx = 0;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bits = bits;
  a.group = group;
  a.epi = kEpiStore;
  a.ldw = ldw;
  a.ws = ws;
  a.ws_bytes = ws ? ws_bytes : 0;
  return a;
}

// Bytes of the packed weight (rows of ldw words, the last row only its own).
size_t weight_bytes(int N, int K, int bits, int ldw) {
  const size_t wpr = (size_t)K / (32 / bits);
  return ((size_t)(N - 1) * (ldw ? (size_t)ldw : wpr) + wpr) * 4;
}

}  // namespace tlq

using namespace tlq;

extern "C" {

const char* tl_last_error(void) { return g_msg; }

const char* tl_version(void) { return "tlq 0.1 sm_103a"; }

tlq_status tl_quant_gemm(const uint16_t* A, const uint32_t* Wpacked, const uint16_t* scales, const uint16_t* zeros,
                         uint16_t* C, int M, int N, int K, int bits, int group, void* stream) {
  g_msg[0] = 0;
  tlq_status st = check_gemm_call(A, Wpacked, scales, zeros, C, M, N, K, bits, group, "tl_quant_gemm");
  if (st != TLQ_OK) return st;
  if (overlaps(A, (size_t)M * K * 2, C, (size_t)M * N * 2))
    return set_error(TLQ_EINVAL, "tl_quant_gemm: A and C overlap");
  return run_gemm(plain_args(A, Wpacked, scales, zeros, C, M, N, K, bits, group), static_cast<cudaStream_t>(stream));
}

size_t tl_quant_gemm_workspace_size(int M, int N, int K, int bits, int group) {
  g_msg[0] = 0;
  if (M <= 16 || check_gemm_shape(M, N, K, bits, group, "tl_quant_gemm_workspace_size") != TLQ_OK) return 0;
  GemmArgs a = plain_args(nullptr, nullptr, nullptr, nullptr, nullptr, M, N, K, bits, group);
  return prefill_workspace_bytes(a);
}

tlq_status tl_prefill_plan(const int* M, const int* N, const int* K, const size_t* ws_bytes, int count,
                           const int* device, int* nmt_out, int* ks_out) {
  g_msg[0] = 0;
  if (count < 1 || count > 16) return set_error(TLQ_EINVAL, "tl_prefill_plan: count=%d (1..16)", count);
  if (!M || !N || !K || !ws_bytes || !nmt_out || !ks_out) return set_error(TLQ_EINVAL, "tl_prefill_plan: null array");
  for (int i = 0; i < count; ++i)
    if (M[i] < 1 || N[i] < 1 || K[i] < 1)
      return set_error(TLQ_EINVAL, "tl_prefill_plan[%d]: M=%d N=%d K=%d (must be >= 1)", i, M[i], N[i], K[i]);
  PlanDevice d;
  if (device) {
    for (int i = 0; i < 9; ++i)
      if (device[i] < 1) return set_error(TLQ_EINVAL, "tl_prefill_plan: device[%d]=%d (must be >= 1)", i, device[i]);
    d.sms = device[0];
    for (int i = 0; i < 4; ++i) {
      d.clusters[0][i] = device[1 + i];
      d.clusters[1][i] = device[5 + i];
    }
  }
  return prefill_plan(M, N, K, ws_bytes, count, device ? &d : nullptr, nmt_out, ks_out);
}

tlq_status tl_quant_gemm_ws(const uint16_t* A, const uint32_t* Wpacked, const uint16_t* scales,
                            const uint16_t* zeros, uint16_t* C, int M, int N, int K, int bits, int group,
                            void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  const char* who = "tl_quant_gemm_ws";
  tlq_status st = check_gemm_call(A, Wpacked, scales, zeros, C, M, N, K, bits, group, who);
  if (st != TLQ_OK) return st;
  if ((st = check_workspace(workspace, workspace_bytes, who)) != TLQ_OK) return st;
  if (overlaps(A, (size_t)M * K * 2, C, (size_t)M * N * 2)) return set_error(TLQ_EINVAL, "%s: A and C overlap", who);
  if (workspace && (overlaps(workspace, workspace_bytes, A, (size_t)M * K * 2) ||
                    overlaps(workspace, workspace_bytes, C, (size_t)M * N * 2) ||
                    overlaps(workspace, workspace_bytes, Wpacked, weight_bytes(N, K, bits, 0))))
    return set_error(TLQ_EINVAL, "%s: the workspace overlaps A, C or the weights", who);
  return run_gemm(plain_args(A, Wpacked, scales, zeros, C, M, N, K, bits, group, 0, workspace, workspace_bytes),
                  static_cast<cudaStream_t>(stream));
}

namespace {
tlq_status check_batched(const tl_gemm_desc* d, int count);
}  // namespace

tlq_status tl_quant_gemm_batched_host(const tl_gemm_desc* d, int count, const void* hostA, void* devA, size_t a_bytes,
                                      void* hostC, const void* devC, size_t c_bytes, void* stream_) {
  g_msg[0] = 0;
  const char* who = "tl_quant_gemm_batched_host";
  if (!hostA || !devA || !hostC || !devC) return set_error(TLQ_EINVAL, "%s: null buffer", who);
  if (!d || count < 1) return set_error(TLQ_EINVAL, "%s: null descriptors or count %d", who, count);
  if (overlaps(devA, a_bytes, devC, c_bytes)) return set_error(TLQ_EINVAL, "%s: devA and devC overlap", who);
  // every problem reads inside devA and writes inside devC (rows of lda = K / ldc = N)
  const char* a0 = static_cast<const char*>(devA);
  const char* c0 = static_cast<const char*>(devC);
  for (int i = 0; i < count; ++i) {
    const char* ap = reinterpret_cast<const char*>(d[i].A);
    const char* cp = reinterpret_cast<const char*>(d[i].C);
    const size_t ab = (size_t)d[i].M * d[i].K * 2, cb = (size_t)d[i].M * d[i].N * 2;
    if (!ap || !cp || ap < a0 || ap + ab > a0 + a_bytes || cp < c0 || cp + cb > c0 + c_bytes)
      return set_error(TLQ_EINVAL, "%s[%d]: A must lie inside devA and C inside devC", who, i);
  }
  tlq_status vst = check_batched(d, count);  // everything is validated before the first copy
  if (vst != TLQ_OK) return vst;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemcpyAsync(devA, hostA, a_bytes, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_error(e, "tl_quant_gemm_batched_host: copy to the device");
  tlq_status st = tl_quant_gemm_batched(d, count, stream_);
  if (st != TLQ_OK) return st;
  e = cudaMemcpyAsync(hostC, devC, c_bytes, cudaMemcpyDeviceToHost, stream);
  return cuda_error(e, "tl_quant_gemm_batched_host: copy to the host");
}

namespace {
tlq_status swiglu_gemm(const uint16_t* A, const uint32_t* Wgu, const uint16_t* scales, const uint16_t* zeros,
                       uint16_t* C, int M, int N2, int K, int bits, int group, void* ws, size_t ws_bytes, void* stream,
                       const char* who) {
  tlq_status st = check_gemm_call(A, Wgu, scales, zeros, C, M, N2, K, bits, group, who);
  if (st != TLQ_OK) return st;
  if ((st = check_workspace(ws, ws_bytes, who)) != TLQ_OK) return st;
  if (N2 % 16) return set_error(TLQ_EINVAL, "%s: N2=%d must be a multiple of 16", who, N2);
  if (overlaps(A, (size_t)M * K * 2, C, (size_t)M * (N2 / 2) * 2)) return set_error(TLQ_EINVAL, "%s: A and C overlap", who);
  if (ws && (overlaps(ws, ws_bytes, A, (size_t)M * K * 2) || overlaps(ws, ws_bytes, C, (size_t)M * (N2 / 2) * 2) ||
             overlaps(ws, ws_bytes, Wgu, weight_bytes(N2, K, bits, 0))))
    return set_error(TLQ_EINVAL, "%s: the workspace overlaps A, C or the weights", who);
  GemmArgs a = plain_args(A, Wgu, scales, zeros, C, M, N2, K, bits, group, 0, ws, ws_bytes);
  a.ldc = N2 / 2;
  a.epi = kEpiSwiglu;
  return run_gemm(a, static_cast<cudaStream_t>(stream));
}
}  // namespace

tlq_status tl_quant_gemm_swiglu(const uint16_t* A, const uint32_t* Wgu, const uint16_t* scales, const uint16_t* zeros,
                                uint16_t* C, int M, int N2, int K, int bits, int group, void* stream) {
  g_msg[0] = 0;
  return swiglu_gemm(A, Wgu, scales, zeros, C, M, N2, K, bits, group, nullptr, 0, stream, "tl_quant_gemm_swiglu");
}

tlq_status tl_quant_gemm_swiglu_ws(const uint16_t* A, const uint32_t* Wgu, const uint16_t* scales,
                                   const uint16_t* zeros, uint16_t* C, int M, int N2, int K, int bits, int group,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  return swiglu_gemm(A, Wgu, scales, zeros, C, M, N2, K, bits, group, workspace, workspace_bytes, stream,
                     "tl_quant_gemm_swiglu_ws");
}

tlq_status tl_dequant_fp16(const uint32_t* Wpacked, const uint16_t* scales, const uint16_t* zeros, uint16_t* out, int N,
                           int K, int bits, int group, void* stream) {
  g_msg[0] = 0;
  if (!Wpacked || !scales || !zeros || !out) return set_error(TLQ_EINVAL, "tl_dequant_fp16: null pointer");
  tlq_status st = check_gemm_shape(1, N, K, bits, group, "tl_dequant_fp16");
  if (st != TLQ_OK) return st;
  if (!aligned16(Wpacked) || !aligned16(out))
    return set_error(TLQ_EINVAL, "tl_dequant_fp16: Wpacked and out must be 16-byte aligned");
  const size_t ob = (size_t)N * K * 2, wb = (size_t)N * K * bits / 8, gb = (size_t)N * (K / group) * 2;
  if (overlaps(out, ob, Wpacked, wb) || overlaps(out, ob, scales, gb) || overlaps(out, ob, zeros, gb))
    return set_error(TLQ_EINVAL, "tl_dequant_fp16: out overlaps an input");
  return launch_body(Wpacked, scales, zeros, out, N, K, bits, group, static_cast<cudaStream_t>(stream));
}

tlq_status tl_interleave_rows(const void* a, const void* b, void* out, int rows, size_t row_bytes, void* stream) {
  g_msg[0] = 0;
  if (!a || !b || !out) return set_error(TLQ_EINVAL, "tl_interleave_rows: null pointer");
  if (rows < 1 || row_bytes < 1)
    return set_error(TLQ_EINVAL, "tl_interleave_rows: rows=%d row_bytes=%zu must be >= 1", rows, row_bytes);
  const size_t n = (size_t)rows * row_bytes;
  if (overlaps(out, 2 * n, a, n) || overlaps(out, 2 * n, b, n))
    return set_error(TLQ_EINVAL, "tl_interleave_rows: out overlaps an input");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpy2DAsync(out, 2 * row_bytes, a, row_bytes, row_bytes, (size_t)rows, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(static_cast<char*>(out) + row_bytes, 2 * row_bytes, b, row_bytes, row_bytes, (size_t)rows,
                          cudaMemcpyDeviceToDevice, s);
  return cuda_error(e, "tl_interleave_rows: copy");
}

namespace {
// Validation of a batched call (shapes, pointers, aliasing); nothing launched.
tlq_status check_batched(const tl_gemm_desc* d, int count) {
  if (!d || count < 0) return set_error(TLQ_EINVAL, "tl_quant_gemm_batched: null descriptors or count %d", count);
  char who[64];
  for (int i = 0; i < count; ++i) {
    snprintf(who, sizeof(who), "tl_quant_gemm_batched[%d]", i);
    tlq_status st = check_gemm_call(d[i].A, d[i].Wpacked, d[i].scales, d[i].zeros, d[i].C, d[i].M, d[i].N, d[i].K,
                                    d[i].bits, d[i].group, who);
    if (st != TLQ_OK) return st;
    if ((st = check_ldw(d[i].ldw, d[i].K, d[i].bits, who)) != TLQ_OK) return st;
    if ((st = check_workspace(d[i].workspace, d[i].workspace_bytes, who)) != TLQ_OK) return st;
  }
  for (int i = 0; i < count; ++i)
    for (int j = 0; j < count; ++j) {
      if (overlaps(d[j].A, (size_t)d[j].M * d[j].K * 2, d[i].C, (size_t)d[i].M * d[i].N * 2))
        return set_error(TLQ_EINVAL, "tl_quant_gemm_batched: C of problem %d overlaps A of problem %d", i, j);
      if (i < j && overlaps(d[i].C, (size_t)d[i].M * d[i].N * 2, d[j].C, (size_t)d[j].M * d[j].N * 2))
        return set_error(TLQ_EINVAL, "tl_quant_gemm_batched: outputs of problems %d and %d overlap", i, j);
      const void* w = d[i].workspace;
      const size_t wb = d[i].workspace_bytes;
      if (!w) continue;
      if (overlaps(w, wb, d[j].A, (size_t)d[j].M * d[j].K * 2) || overlaps(w, wb, d[j].C, (size_t)d[j].M * d[j].N * 2) ||
          overlaps(w, wb, d[j].Wpacked, weight_bytes(d[j].N, d[j].K, d[j].bits, d[j].ldw)) ||
          (i < j && d[j].workspace && overlaps(w, wb, d[j].workspace, d[j].workspace_bytes)))
        return set_error(TLQ_EINVAL, "tl_quant_gemm_batched: the workspace of problem %d overlaps a buffer of problem %d",
                         i, j);
    }
  return TLQ_OK;
}
}  // namespace

namespace {
// Side streams for the independent prefill problems of one batched call: per
// (device, caller stream) three non-blocking streams, with events that fork
// them from the caller's stream and join them back.  The problems then run
// side by side (each launch alone fills only part of the GPU at short M);
// the event record / wait pairs also carry the fork and join into a graph
// capture of the caller's stream.  Sets are created outside stream capture
// (a capture with no set for its stream launches the problems in order).
constexpr int kSideStreams = 3;
constexpr int kSideSets = 16;
struct SideSet {
  int dev;
  cudaStream_t caller;
  cudaStream_t s[kSideStreams];
  cudaEvent_t fork, join[kSideStreams];
};
std::mutex g_side_mu;
SideSet g_side[kSideSets];
int g_nside = 0;

SideSet* side_streams(cudaStream_t caller) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_side_mu);
  for (int i = 0; i < g_nside; ++i)
    if (g_side[i].dev == dev && g_side[i].caller == caller) return &g_side[i];
  if (g_nside == kSideSets) return nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
  SideSet& e = g_side[g_nside];
  e.dev = dev;
  e.caller = caller;
  int made = 0;
  bool ok = cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming) == cudaSuccess;
  for (; ok && made < kSideStreams; ++made) {
    if (cudaStreamCreateWithFlags(&e.s[made], cudaStreamNonBlocking) != cudaSuccess) {
      ok = false;
      break;
    }
    if (cudaEventCreateWithFlags(&e.join[made], cudaEventDisableTiming) != cudaSuccess) {
      cudaStreamDestroy(e.s[made]);
      ok = false;
      break;
    }
  }
  if (!ok) {
    for (int k = 0; k < made; ++k) {
      cudaStreamDestroy(e.s[k]);
      cudaEventDestroy(e.join[k]);
    }
    cudaGetLastError();
    return nullptr;
  }
  ++g_nside;
  return &e;
}
}  // namespace

tlq_status tl_quant_gemm_batched(const tl_gemm_desc* d, int count, void* stream_) {
  g_msg[0] = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  tlq_status vst = check_batched(d, count);
  if (vst != TLQ_OK) return vst;
  // decode-sized problems share launches (one per bit width, up to 16 problems each)
  for (int bits : {4, 2}) {
    GemmArgs batch[kMaxDecodeProblems];
    int n = 0;
    for (int i = 0; i < count; ++i) {
      if (d[i].M > 16 || d[i].bits != bits) continue;
      batch[n++] = plain_args(d[i].A, d[i].Wpacked, d[i].scales, d[i].zeros, d[i].C, d[i].M, d[i].N, d[i].K,
                              d[i].bits, d[i].group, d[i].ldw);
      if (n == kMaxDecodeProblems) {
        tlq_status st = launch_decode(batch, n, stream);
        if (st != TLQ_OK) return st;
        n = 0;
      }
    }
    if (n) {
      tlq_status st = launch_decode(batch, n, stream);
      if (st != TLQ_OK) return st;
    }
  }
  // the other problems: one prefill launch each, several at a time on side streams
  int np = 0;
  for (int i = 0; i < count; ++i) np += d[i].M > 16;
  SideSet* ss = np > 1 ? side_streams(stream) : nullptr;
  const int used = ss ? std::min(np - 1, kSideStreams) : 0;
  if (ss) {
    cudaError_t e = cudaEventRecord(ss->fork, stream);
    for (int k = 0; k < used && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(ss->s[k], ss->fork, 0);
    if (e != cudaSuccess) return cuda_error(e, "tl_quant_gemm_batched: fork");
  }
  // up to four problems all run at once (one per stream): their token tiles
  // and k splits are chosen together for the shared GPU
  GemmArgs joint[kSideStreams + 1];
  int order[kSideStreams + 1];
  bool together = ss && np >= 2 && np <= kSideStreams + 1;
  if (together) {
    for (int i = 0, j = 0; i < count; ++i)
      if (d[i].M > 16)
        joint[j++] = plain_args(d[i].A, d[i].Wpacked, d[i].scales, d[i].zeros, d[i].C, d[i].M, d[i].N, d[i].K,
                                d[i].bits, d[i].group, d[i].ldw, d[i].workspace, d[i].workspace_bytes);
    together = plan_prefill_joint(joint, np, order);
  }
  tlq_status st = TLQ_OK;
  if (together) {  // the jointly planned launches, the longest first
    for (int j = 0; j < np && st == TLQ_OK; ++j)
      st = launch_prefill(joint[order[j]], j % (used + 1) ? ss->s[j % (used + 1) - 1] : stream);
  } else {
    for (int i = 0, j = 0; i < count && st == TLQ_OK; ++i) {
      if (d[i].M <= 16) continue;
      const int lane = used ? j % (used + 1) : 0;  // 0: the caller's stream
      st = launch_prefill(plain_args(d[i].A, d[i].Wpacked, d[i].scales, d[i].zeros, d[i].C, d[i].M, d[i].N, d[i].K,
                                     d[i].bits, d[i].group, d[i].ldw, d[i].workspace, d[i].workspace_bytes),
                          lane ? ss->s[lane - 1] : stream);
      ++j;
    }
  }
  for (int k = 0; k < used; ++k) {  // join even after a failed launch
    cudaError_t e = cudaEventRecord(ss->join[k], ss->s[k]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ss->join[k], 0);
    if (e != cudaSuccess && st == TLQ_OK) st = cuda_error(e, "tl_quant_gemm_batched: join");
  }
  return st;
}

tlq_status tl_pack_weights(const uint8_t* codes, uint32_t* Wpacked, int N, int K, int bits, void* stream) {
  g_msg[0] = 0;
  if (!codes || !Wpacked) return set_error(TLQ_EINVAL, "tl_pack_weights: null pointer");
  if (bits != 4 && bits != 2) return set_error(TLQ_EINVAL, "tl_pack_weights: bits=%d (must be 4 or 2)", bits);
  if (N < 1 || K < 1) return set_error(TLQ_EINVAL, "tl_pack_weights: N=%d K=%d must be >= 1", N, K);
  if (K % (32 / bits)) return set_error(TLQ_EINVAL, "tl_pack_weights: K=%d not a multiple of %d", K, 32 / bits);
  return launch_pack(codes, Wpacked, N, K, bits, static_cast<cudaStream_t>(stream));
}

tlq_status tl_unpack_weights(const uint32_t* Wpacked, uint8_t* codes, int N, int K, int bits, void* stream) {
  g_msg[0] = 0;
  if (!codes || !Wpacked) return set_error(TLQ_EINVAL, "tl_unpack_weights: null pointer");
  if (bits != 4 && bits != 2) return set_error(TLQ_EINVAL, "tl_unpack_weights: bits=%d (must be 4 or 2)", bits);
  if (N < 1 || K < 1) return set_error(TLQ_EINVAL, "tl_unpack_weights: N=%d K=%d must be >= 1", N, K);
  if (K % (32 / bits)) return set_error(TLQ_EINVAL, "tl_unpack_weights: K=%d not a multiple of %d", K, 32 / bits);
  return launch_unpack(Wpacked, codes, N, K, bits, static_cast<cudaStream_t>(stream));
}

namespace {
// Validation of one re-quantization problem against itself.
tlq_status check_requant(const tl_requant_desc& d, int group, const char* who, int idx) {
  if (!d.W4 || !d.s4 || !d.z4 || !d.W2 || !d.s2 || !d.z2) return set_error(TLQ_EINVAL, "%s[%d]: null pointer", who, idx);
  if (d.N < 1 || d.K < 1) return set_error(TLQ_EINVAL, "%s[%d]: N=%d K=%d must be >= 1", who, idx, d.N, d.K);
  if (d.K % group) return set_error(TLQ_EINVAL, "%s[%d]: group=%d does not divide K=%d", who, idx, group, d.K);
  if (!aligned16(d.W4) || !aligned16(d.W2))
    return set_error(TLQ_EINVAL, "%s[%d]: W4 and W2 must be 16-byte aligned", who, idx);
  if ((reinterpret_cast<uintptr_t>(d.s4) | reinterpret_cast<uintptr_t>(d.z4) | reinterpret_cast<uintptr_t>(d.s2) |
       reinterpret_cast<uintptr_t>(d.z2)) & 1u)
    return set_error(TLQ_EINVAL, "%s[%d]: scales/zeros must be 2-byte aligned", who, idx);
  return TLQ_OK;
}

struct RqRegion {
  const void* p;
  size_t n;
  int prob;
  int kind;  // 0 W4, 1 s4, 2 z4, 3 W2, 4 s2, 5 z2
};

// Outputs (W2, s2, z2) may overlap nothing, except that s2 / z2 may be
// exactly the s4 / z4 of the same problem.  Inputs may overlap each other.
tlq_status check_requant_overlaps(const tl_requant_desc* d, int count, int group, const char* who) {
  RqRegion r[6 * kMaxRequantProblems];
  int n = 0;
  for (int i = 0; i < count; ++i) {
    // in place (W2 == W4): the INT2 rows keep the INT4 stride, so W2 spans W4
    const size_t b4 = (size_t)d[i].N * d[i].K / 2;
    const size_t b2 = d[i].W2 == d[i].W4 ? b4 : (size_t)d[i].N * d[i].K / 4;
    const size_t bg = (size_t)d[i].N * (d[i].K / group) * 2;
    r[n++] = {d[i].W4, b4, i, 0};
    r[n++] = {d[i].s4, bg, i, 1};
    r[n++] = {d[i].z4, bg, i, 2};
    r[n++] = {d[i].W2, b2, i, 3};
    r[n++] = {d[i].s2, bg, i, 4};
    r[n++] = {d[i].z2, bg, i, 5};
  }
  for (int a = 0; a < n; ++a) {
    if (r[a].kind < 3) continue;  // every pair with at least one output
    for (int b = 0; b < n; ++b) {
      if (b == a || (r[b].kind >= 3 && b < a)) continue;
      if (!overlaps(r[a].p, r[a].n, r[b].p, r[b].n)) continue;
      const bool same_prob = r[a].prob == r[b].prob;
      if (same_prob && r[a].p == r[b].p && r[a].n == r[b].n && r[a].kind - r[b].kind == 3)
        continue;  // W2 == W4, s2 == s4 or z2 == z4: converted in place
      static const char* names[6] = {"W4", "s4", "z4", "W2", "s2", "z2"};
      return set_error(TLQ_EINVAL, "%s: %s of problem %d overlaps %s of problem %d", who, names[r[a].kind], r[a].prob,
                       names[r[b].kind], r[b].prob);
    }
  }
  return TLQ_OK;
}

tlq_status requant(const tl_requant_desc* d, int count, int group, void* stream, const char* who) {
  if (count < 0 || count > kMaxRequantProblems)
    return set_error(TLQ_EINVAL, "%s: count=%d (0..%d)", who, count, kMaxRequantProblems);
  if (count > 0 && !d) return set_error(TLQ_EINVAL, "%s: null descriptor array", who);
  if (group < 64 || group % 64)
    return set_error(TLQ_EINVAL, "%s: group=%d must be a multiple of 64 (the INT2 kernels' rule)", who, group);
  for (int i = 0; i < count; ++i) {
    tlq_status st = check_requant(d[i], group, who, i);
    if (st != TLQ_OK) return st;
  }
  tlq_status st = check_requant_overlaps(d, count, group, who);
  if (st != TLQ_OK) return st;
  if (count == 0) return TLQ_OK;
  RequantArgs out[kMaxRequantProblems], inpl[kMaxRequantProblems];
  int no = 0, ni = 0;
  for (int i = 0; i < count; ++i) {
    const RequantArgs a{d[i].W4, d[i].s4, d[i].z4, d[i].W2, d[i].s2, d[i].z2, d[i].N, d[i].K};
    if (d[i].W2 == d[i].W4) inpl[ni++] = a;
    else out[no++] = a;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (no) {
    st = launch_requant(out, no, group, s);
    if (st != TLQ_OK) return st;
  }
  return ni ? launch_requant_in_place(inpl, ni, group, s) : TLQ_OK;
}
}  // namespace

tlq_status tl_requant_int4_to_int2(const uint32_t* W4, const uint16_t* s4, const uint16_t* z4, uint32_t* W2,
                                   uint16_t* s2, uint16_t* z2, int N, int K, int group, void* stream) {
  g_msg[0] = 0;
  const tl_requant_desc d = {W4, s4, z4, W2, s2, z2, N, K};
  return requant(&d, 1, group, stream, "tl_requant_int4_to_int2");
}

tlq_status tl_requant_int4_to_int2_batched(const tl_requant_desc* descs, int count, int group, void* stream) {
  g_msg[0] = 0;
  return requant(descs, count, group, stream, "tl_requant_int4_to_int2_batched");
}

namespace {
// One loop block for the driver: the ReLU block (ff = up, [F x D]) or the
// SwiGLU block (ff = interleaved gate/up, [2F x D]).
struct BlockSpec {
  const tl_qproj* proj[4];  // qkv, o, ff, down
  int bits, group, D, F;
  bool swiglu;
  uint16_t *h, *qkv_out, *o_out, *act_out;
  int normalize;
  const char* who;
  void* ws;  // the caller's k-split workspace, shared by the block's GEMMs (they run in order)
  size_t ws_bytes;
};

// The loop block's L2 residency plan: bytes of packed weights and scales /
// zeros per projection, a budget of half the L2 (GB300 measured: re-reads of
// up to ~80 MB of the 126 MB L2 run at full L2 bandwidth; the other half
// leaves room for activations and other streams), and the projections kept
// resident: the longest run from the first, in iteration order, that fits.
struct L2Plan {
  int mask;  // bit i: projection i (qkv, o, ff, down) streamed evict-last
  size_t weight_bytes, budget_bytes;
};

L2Plan plan_l2(const tl_qproj* const* proj, int bits, int group, int L) {
  L2Plan pl{0, 0, (size_t)device_info().l2_bytes / 2};
  const int cpw = 32 / bits;
  size_t cum = 0;
  bool fits = true;
  for (int i = 0; i < 4; ++i) {
    const size_t bytes =
        (size_t)proj[i]->N * (proj[i]->K / cpw) * 4 + (size_t)proj[i]->N * (proj[i]->K / group) * 4;
    pl.weight_bytes += bytes;
    cum += bytes;
    fits = fits && cum <= pl.budget_bytes;
    if (fits && L > 1) pl.mask |= 1 << i;
  }
  return pl;
}

tlq_status block_forward(float* x, const BlockSpec& b, int L, int M, cudaStream_t stream) {
  const char* who = b.who;
  if (L < 0) return set_error(TLQ_EINVAL, "%s: L=%d (must be >= 0)", who, L);
  if (M < 1) return set_error(TLQ_EINVAL, "%s: M=%d (must be >= 1)", who, M);
  const int D = b.D, F = b.F;
  if (D < 1 || D % 8) return set_error(TLQ_EINVAL, "%s: D=%d must be a positive multiple of 8", who, D);
  const char* ffname = b.swiglu ? "gate_up" : "up";
  if (b.proj[0]->N != 3 * D || b.proj[0]->K != D) return set_error(TLQ_EINVAL, "%s: qkv must be [3D x D]", who);
  if (b.proj[1]->N != D || b.proj[1]->K != D) return set_error(TLQ_EINVAL, "%s: o must be [D x D]", who);
  if (b.proj[2]->K != D || F < 1) return set_error(TLQ_EINVAL, "%s: %s must have K = D", who, ffname);
  if (b.swiglu && (b.proj[2]->N % 16))
    return set_error(TLQ_EINVAL, "%s: gate_up N=%d must be 2F with F a multiple of 8", who, b.proj[2]->N);
  if (b.proj[3]->N != D || b.proj[3]->K != F) return set_error(TLQ_EINVAL, "%s: down must be [D x F]", who);
  if (!b.h || !b.qkv_out || !b.o_out || !b.act_out) return set_error(TLQ_EINVAL, "%s: null scratch buffer", who);
  const char* names[4] = {"qkv", "o", ffname, "down"};
  for (int i = 0; i < 4; ++i) {
    const tl_qproj* p = b.proj[i];
    if (!p->W || !p->s || !p->z) return set_error(TLQ_EINVAL, "%s: %s has a null pointer", who, names[i]);
    if (!aligned16(p->W)) return set_error(TLQ_EINVAL, "%s: %s weights not 16-byte aligned", who, names[i]);
    tlq_status st = check_gemm_shape(M, p->N, p->K, b.bits, b.group, names[i]);
    if (st != TLQ_OK) return st;
    if (p->N % 8) return set_error(TLQ_EINVAL, "%s: %s N=%d must be a multiple of 8", who, names[i], p->N);
    if ((st = check_ldw(p->ldw, p->K, b.bits, names[i])) != TLQ_OK) return st;
  }
  {
    tlq_status st = check_workspace(b.ws, b.ws_bytes, who);
    if (st != TLQ_OK) return st;
  }
  if (!aligned16(b.h) || !aligned16(b.qkv_out) || !aligned16(b.o_out) || !aligned16(b.act_out))
    return set_error(TLQ_EINVAL, "%s: scratch buffers must be 16-byte aligned", who);

  // The block's weights are re-read every iteration ("Model", "Returns",
  // item 4: auto tile sizing reports loop-block vs L2 residency): the plan
  // keeps the projections resident with an L2 evict-last policy in iteration
  // order while they fit the L2 budget, and streams the rest evict-first so
  // they do not push the resident ones out.
  const L2Plan plan = plan_l2(b.proj, b.bits, b.group, L);
  static std::once_flag logged;
  if (log_enabled()) {
    std::call_once(logged, [&] {
      static const char* nm[4] = {"qkv", "o", "ff", "down"};
      char kept[64] = "", streamed[64] = "";
      for (int i = 0; i < 4; ++i) {
        char* dst = ((plan.mask >> i) & 1) ? kept : streamed;
        strncat(dst, nm[i], sizeof(kept) - strlen(dst) - 2);
        strncat(dst, " ", sizeof(kept) - strlen(dst) - 1);
      }
      fprintf(stderr,
              "[tlq] loop block: INT%d group %d, packed weights + scales/zeros %.1f MB, L2 %.1f MB, budget %.1f MB: "
              "resident (evict-last) [ %s], streamed [ %s]\n",
              b.bits, b.group, plan.weight_bytes / 1e6, device_info().l2_bytes / 1e6, plan.budget_bytes / 1e6, kept,
              streamed);
    });
  }

  auto gemm = [&](const tl_qproj* p, const uint16_t* A, int lda, uint16_t* C, int ldc, int epi) {
    GemmArgs a;
    a.bits = b.bits;
    a.group = b.group;
    a.M = M;
    a.l2_keep = (plan.mask >> (p == b.proj[0] ? 0 : p == b.proj[1] ? 1 : p == b.proj[2] ? 2 : 3)) & 1;
    a.ldw = p->ldw;
    a.ws = b.ws;
    a.ws_bytes = b.ws ? b.ws_bytes : 0;
    a.A = reinterpret_cast<const __half*>(A);
    a.lda = lda;
    a.W = p->W;
    a.S = reinterpret_cast<const __half*>(p->s);
    a.Z = reinterpret_cast<const __half*>(p->z);
    a.C = reinterpret_cast<__half*>(C);
    a.ldc = ldc;
    a.X = epi == kEpiResidual ? x : nullptr;
    a.ldx = epi == kEpiResidual ? D : 0;
    a.N = p->N;
    a.K = p->K;
    a.epi = epi;
    return run_gemm(a, stream);
  };
  for (int l = 0; l < L; ++l) {
    tlq_status st = launch_rmsnorm(x, reinterpret_cast<__half*>(b.h), M, D, b.normalize, stream);
    if (st != TLQ_OK) return st;
    if ((st = gemm(b.proj[0], b.h, D, b.qkv_out, 3 * D, kEpiStore)) != TLQ_OK) return st;  // QKV
    if ((st = gemm(b.proj[1], b.qkv_out, 3 * D, b.o_out, D, kEpiStore)) != TLQ_OK) return st;  // O on qkv[:, :D]
    // UP + ReLU, or the fused gate/up GEMM + SwiGLU
    if ((st = gemm(b.proj[2], b.o_out, D, b.act_out, F, b.swiglu ? kEpiSwiglu : kEpiRelu)) != TLQ_OK) return st;
    if ((st = gemm(b.proj[3], b.act_out, F, nullptr, 0, kEpiResidual)) != TLQ_OK) return st;  // DOWN + FP32 residual
  }
  return TLQ_OK;
}
}  // namespace

tlq_status tl_loop_block_l2_plan(const tl_block* b, int L, int* resident_mask, size_t* weight_bytes,
                                 size_t* budget_bytes) {
  g_msg[0] = 0;
  if (!b || !resident_mask) return set_error(TLQ_EINVAL, "tl_loop_block_l2_plan: null pointer");
  if (b->bits != 4 && b->bits != 2) return set_error(TLQ_EINVAL, "tl_loop_block_l2_plan: bits=%d", b->bits);
  if (b->group < 32 || b->group % 32) return set_error(TLQ_EINVAL, "tl_loop_block_l2_plan: group=%d", b->group);
  const tl_qproj* proj[4] = {&b->qkv, &b->o, &b->up, &b->down};
  const L2Plan pl = plan_l2(proj, b->bits, b->group, L);
  *resident_mask = pl.mask;
  if (weight_bytes) *weight_bytes = pl.weight_bytes;
  if (budget_bytes) *budget_bytes = pl.budget_bytes;
  return TLQ_OK;
}

tlq_status tl_loop_block_forward(float* x, const tl_block* b, int L, int M, void* stream) {
  g_msg[0] = 0;
  if (!x || !b) return set_error(TLQ_EINVAL, "tl_loop_block_forward: null x or block");
  const BlockSpec s = {{&b->qkv, &b->o, &b->up, &b->down}, b->bits, b->group, b->D, b->up.N, false,
                       b->h, b->qkv_out, b->o_out, b->up_out, b->normalize, "tl_loop_block_forward",
                       b->workspace, b->workspace_bytes};
  return block_forward(x, s, L, M, static_cast<cudaStream_t>(stream));
}


namespace {
// Chunk-first prefill: rows [r0, r0 + chunk) run through all L iterations,
// then the next chunk, with scratch for `chunk` rows only.
tlq_status block_forward_chunked(float* x, const BlockSpec& s, int L, int M, int chunk, cudaStream_t stream) {
  if (M < 1) return set_error(TLQ_EINVAL, "%s: M=%d (must be >= 1)", s.who, M);
  if (chunk <= 0 || chunk > M) chunk = M;
  for (int r0 = 0; r0 < M; r0 += chunk) {
    const int rows = M - r0 < chunk ? M - r0 : chunk;
    tlq_status st = block_forward(x + (size_t)r0 * s.D, s, L, rows, stream);
    if (st != TLQ_OK) return st;
  }
  return TLQ_OK;
}
}  // namespace

tlq_status tl_loop_block_forward_chunked(float* x, const tl_block* b, int L, int M, int chunk, void* stream) {
  g_msg[0] = 0;
  if (!x || !b) return set_error(TLQ_EINVAL, "tl_loop_block_forward_chunked: null x or block");
  const BlockSpec s = {{&b->qkv, &b->o, &b->up, &b->down}, b->bits, b->group, b->D, b->up.N, false,
                       b->h, b->qkv_out, b->o_out, b->up_out, b->normalize, "tl_loop_block_forward_chunked",
                       b->workspace, b->workspace_bytes};
  return block_forward_chunked(x, s, L, M, chunk, static_cast<cudaStream_t>(stream));
}

tlq_status tl_swiglu_block_forward_chunked(float* x, const tl_swiglu_block* b, int L, int M, int chunk, void* stream) {
  g_msg[0] = 0;
  if (!x || !b) return set_error(TLQ_EINVAL, "tl_swiglu_block_forward_chunked: null x or block");
  const BlockSpec s = {{&b->qkv, &b->o, &b->gate_up, &b->down}, b->bits, b->group, b->D, b->gate_up.N / 2, true,
                       b->h, b->qkv_out, b->o_out, b->act_out, b->normalize, "tl_swiglu_block_forward_chunked",
                       b->workspace, b->workspace_bytes};
  return block_forward_chunked(x, s, L, M, chunk, static_cast<cudaStream_t>(stream));
}

tlq_status tl_swiglu_block_forward(float* x, const tl_swiglu_block* b, int L, int M, void* stream) {
  g_msg[0] = 0;
  if (!x || !b) return set_error(TLQ_EINVAL, "tl_swiglu_block_forward: null x or block");
  const BlockSpec s = {{&b->qkv, &b->o, &b->gate_up, &b->down}, b->bits, b->group, b->D, b->gate_up.N / 2, true,
                       b->h, b->qkv_out, b->o_out, b->act_out, b->normalize, "tl_swiglu_block_forward",
                       b->workspace, b->workspace_bytes};
  return block_forward(x, s, L, M, static_cast<cudaStream_t>(stream));
}

namespace {
// The context-length tier switch of a loop block: every INT4 projection
// re-quantized to INT2 (out of place into dst[i], or in place when dst is
// NULL or dst[i].W is the INT4 weight itself), then the block's description
// rewritten so later forwards take the INT2 kernels.
tlq_status block_to_int2(tl_qproj* const* proj, int* bits, int group, const tl_qproj* dst, const char* who,
                         void* stream) {
  if (*bits != 4) return set_error(TLQ_EINVAL, "%s: the block holds INT%d weights (INT4 needed)", who, *bits);
  tl_requant_desc d[4];
  tl_qproj next[4];
  for (int i = 0; i < 4; ++i) {
    const tl_qproj& p = *proj[i];
    if (p.ldw != 0 && p.ldw != p.K / 8)
      return set_error(TLQ_EINVAL, "%s: projection %d: INT4 weights with ldw=%d (compact rows needed)", who, i, p.ldw);
    const tl_qproj* o = dst ? &dst[i] : nullptr;
    if (o && (o->N != p.N || o->K != p.K))
      return set_error(TLQ_EINVAL, "%s: projection %d: destination is [%d x %d], the weight [%d x %d]", who, i, o->N,
                       o->K, p.N, p.K);
    uint32_t* W2 = const_cast<uint32_t*>(o ? o->W : p.W);
    uint16_t* s2 = const_cast<uint16_t*>(o ? o->s : p.s);
    uint16_t* z2 = const_cast<uint16_t*>(o ? o->z : p.z);
    d[i] = tl_requant_desc{p.W, p.s, p.z, W2, s2, z2, p.N, p.K};
    next[i] = tl_qproj{W2, s2, z2, p.N, p.K, W2 == p.W ? p.K / 8 : 0};
  }
  tlq_status st = requant(d, 4, group, stream, who);  // validates everything before any launch
  if (st != TLQ_OK) return st;
  for (int i = 0; i < 4; ++i) *proj[i] = next[i];
  *bits = 2;
  return TLQ_OK;
}
}  // namespace

tlq_status tl_loop_block_to_int2(tl_block* block, const tl_qproj* dst, void* stream) {
  g_msg[0] = 0;
  if (!block) return set_error(TLQ_EINVAL, "tl_loop_block_to_int2: null block");
  tl_qproj* proj[4] = {&block->qkv, &block->o, &block->up, &block->down};
  return block_to_int2(proj, &block->bits, block->group, dst, "tl_loop_block_to_int2", stream);
}

tlq_status tl_swiglu_block_to_int2(tl_swiglu_block* block, const tl_qproj* dst, void* stream) {
  g_msg[0] = 0;
  if (!block) return set_error(TLQ_EINVAL, "tl_swiglu_block_to_int2: null block");
  tl_qproj* proj[4] = {&block->qkv, &block->o, &block->gate_up, &block->down};
  return block_to_int2(proj, &block->bits, block->group, dst, "tl_swiglu_block_to_int2", stream);
}

tlq_status tl_check_status(void* stream) {
  g_msg[0] = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "tl_check_status: stream synchronize");
  uint32_t st = 0, where = 0;
  e = cudaMemcpyFromSymbol(&st, g_status, sizeof(st));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&where, g_status_where, sizeof(where));
  if (e != cudaSuccess) return cuda_error(e, "tl_check_status: read status");
  if (st == kStatusTimeout)
    return set_error(TLQ_ETIMEOUT, "a device-side wait gave up (site 0x%x); results of that launch are invalid", where);
  return TLQ_OK;
}

tlq_status tl_reset_status(void* stream) {
  g_msg[0] = 0;
  const uint32_t z = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyToSymbolAsync(g_status, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(g_status_where, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_error(e, "tl_reset_status");
}

tlq_status tl_selftest_wait_timeout(unsigned limit_us, void* stream) {
  g_msg[0] = 0;
  if (limit_us < 1 || limit_us > 1000000)
    return set_error(TLQ_EINVAL, "tl_selftest_wait_timeout: limit_us=%u outside 1..1000000", limit_us);
  return launch_timeout_probe(limit_us, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
namespace tlq {
// The ReLU loop block under a caller-chosen name (the allocation-free entry
// point reports its own name in messages).
tlq_status loop_block_forward_named(float* x, const tl_block* b, int L, int M, const char* who, void* stream) {
  if (!x || !b) return set_error(TLQ_EINVAL, "%s: null x or block", who);
  const BlockSpec s = {{&b->qkv, &b->o, &b->up, &b->down}, b->bits, b->group, b->D, b->up.N, false,
                       b->h, b->qkv_out, b->o_out, b->up_out, b->normalize, who, b->workspace, b->workspace_bytes};
  return block_forward(x, s, L, M, static_cast<cudaStream_t>(stream));
}
}  // namespace tlq

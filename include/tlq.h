/*
 * tlq.h -- C ABI of the GB300 (sm_103a) weight-only quantized linear layer.
 *
 * One shared library (libtlq.so) implements the hot path of the TinyLoop
 * looped-transformer runtime: the quantized linear layer quant_gemm (routed
 * to the INT4 or INT2 kernels) and the shared-weight loop block that reapplies
 * one set of projections L times.
 *
 * Data types in this header are plain C: FP16 values are passed as their
 * IEEE-754 binary16 bit patterns (uint16_t), FP32 as float.  Every pointer
 * argument is a DEVICE pointer (cudaMalloc / torch CUDA tensor memory)
 * unless the comment says otherwise; `stream` is a cudaStream_t passed as
 * void* (NULL = the legacy default stream).
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller owns every input, output, scratch and workspace
 *    buffer; the library allocates no device memory in any call.  A GEMM
 *    with M > 16 whose tiles would leave SMs idle splits K over a
 *    thread-block cluster and exchanges partial tiles through an FP32
 *    workspace that the caller passes (tl_quant_gemm_ws, the workspace fields
 *    of tl_gemm_desc, tl_block and tl_swiglu_block); the size it wants comes
 *    from tl_quant_gemm_workspace_size.  With no workspace, or one too small,
 *    the kernel keeps K whole (same arithmetic per output, possibly slower).
 *    tl_loop_block_forward_static_scratch also needs no caller scratch: it
 *    uses a static array the library owns.  Host state: the library keeps
 *    the launch descriptions (tensor maps, work lists) of recent calls, keyed
 *    by their full argument lists, and for tl_quant_gemm_batched up to three
 *    side streams per caller stream; it keeps no device state between calls.
 *  - Ordering: calls are asynchronous and ordered on `stream`.  Apart from
 *    tl_loop_block_forward_static_scratch the library holds no shared
 *    scratch, so calls on different streams with disjoint buffers may run
 *    concurrently; one model instance is meant to drive one
 *    stream ("Model", section "Thread safety": a single CUDA stream for all
 *    forward-pass work).
 *  - Errors: arguments are checked on the host before anything is launched.
 *    A rejected call returns TLQ_EINVAL (bad argument) or TLQ_EUNSUPPORTED
 *    (valid but not implemented, e.g. a group size the kernels do not take)
 *    and launches nothing; a failed launch returns TLQ_ECUDA.  The message of
 *    the last failure on the calling thread names the failing argument or
 *    step ("Model", section "Raises": errors name the failure point).
 *  - Device waits are bounded: a kernel that gives up on a wait records
 *    TLQ_ETIMEOUT in a device status word and returns; tl_check_status()
 *    reports it.
 *  - Determinism: identical inputs give bit-identical outputs on every call
 *    (no floating-point atomics, fixed reduction order) -- "Model", section
 *    "Determinism".
 *  - Environment (read by the library; none is needed): TLQ_LOG=1 prints each
 *    launch's configuration to stderr; TLQ_PDL=0 turns programmatic dependent
 *    launch off; TLQ_PREFILL_NMT=1|2, TLQ_PREFILL_KSPLIT=1|2|4|8 and
 *    TLQ_DECODE_ROWS=16|32|64 force the kernels' tiling choices (for tests
 *    and measurements; the results of the decode kernel do not depend on
 *    TLQ_DECODE_ROWS); TLQ_DECODE_GENERIC=1 and TLQ_PREFILL_GENERIC=1 force
 *    the kernels' general forms instead of the forms built for whole blocks
 *    (the same results, bit for bit).
 */
#ifndef TLQ_H_
#define TLQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TLQ_OK = 0,
  TLQ_EINVAL = 1,       /* an argument is invalid; nothing was launched      */
  TLQ_EUNSUPPORTED = 2, /* valid request this build does not implement       */
  TLQ_ECUDA = 3,        /* a CUDA runtime/driver call failed                 */
  TLQ_ETIMEOUT = 4      /* a device-side wait hit its limit (see status)     */
} tlq_status;

/* Message of the last failure on the calling thread ("" if none).  The
 * string is owned by the library and valid until the next call on the same
 * thread. */
const char* tl_last_error(void);

/* Library version string, e.g. "tlq 0.1 sm_103a". */
const char* tl_version(void);

/*
 * tl_quant_gemm -- the quantized linear layer (quant_gemm).
 *
 *   C[m][n] = fp16( sum_k A[m][k] * w[n][k] ),  w[n][k] = (q[n][k] - z[n][g]) * s[n][g],
 *   g = k / group, accumulated in FP32 on the GPU.
 *
 * Source: "Model" (TinyLoop Python API), "VRAM cost", Weights -- each
 * quantized layer holds INT2 / INT4 packed data, FP16 scales and FP16 zeros;
 * "beta-Informed Deployment Features", CTX-TIER, "What Phase 2 ships" -- the
 * dispatcher routes on the weight's bit width (INT4 kernel or int2_gemm).
 *
 *   A       FP16 [M][K], row-major, row stride K elements, 16-byte aligned.
 *   Wpacked uint32 [N][K*bits/32], the format tl_pack_weights writes: row n
 *           is K-contiguous, code j of a word at bits [bits*j, bits*j+bits).
 *           16-byte aligned.
 *   scales  FP16 [N][K/group], row-major.
 *   zeros   FP16 [N][K/group], row-major (zero points, need not be integral).
 *   C       FP16 [M][N], row-major, row stride N; must not overlap A.
 *   M >= 1; N >= 1 and a multiple of 8; K >= 1 with K % group == 0.
 *   bits    4 or 2.
 *   group   a multiple of 32 (bits = 4) or 64 (bits = 2), dividing K;
 *           group = K (one scale per row) is allowed.
 *   M <= 16 runs the bandwidth-bound decode kernel, larger M the tensor-core
 *   (tcgen05) prefill kernel, here without a k split (no workspace; see
 *   tl_quant_gemm_ws).
 * Returns TLQ_OK, TLQ_EINVAL (null pointer, misalignment, bad shape/bits/
 * group), or TLQ_ECUDA.
 */
tlq_status tl_quant_gemm(const uint16_t* A, const uint32_t* Wpacked, const uint16_t* scales,
                         const uint16_t* zeros, uint16_t* C, int M, int N, int K, int bits,
                         int group, void* stream);

/*
 * tl_quant_gemm_workspace_size -- bytes of FP32 workspace with which the
 * tensor-core kernel would split K for this problem (its planner's choice
 * with no limit on the workspace); 0 when it would not split (always for
 * M <= 16) or for an invalid shape.  Honors TLQ_PREFILL_NMT / _KSPLIT.
 * A library choice (launch shape), not an operation of the pages.
 */
size_t tl_quant_gemm_workspace_size(int M, int N, int K, int bits, int group);

/*
 * tl_prefill_plan -- the launch plan the library would use for `count`
 * problems: per problem the token tiles per CTA of the tensor-core kernel
 * (1 or 2) and its k split (1, 2, 4 or 8), or 0 and 0 when M <= 16 (the
 * decode kernel).  count = 1 plans a single call (tl_quant_gemm_ws with the
 * given workspace); count = 2..4 with every M > 16 gives the joint plan of a
 * batched call whose launches run side by side; otherwise each problem is
 * planned alone.
 *   M, N, K, ws_bytes  HOST arrays of `count` entries (ws_bytes: the bytes of
 *                      workspace each problem is given, 0 = none).
 *   device             NULL: the current device.  Else a HOST int[9]: the SM
 *                      count, then how many clusters of 1, 2, 4 and 8 CTAs
 *                      fit at once with one token tile per CTA, then the same
 *                      with two.  With a device description no CUDA call is
 *                      made (the planners are host code).
 *   nmt_out, ks_out    HOST arrays of `count` entries, written.
 * TLQ_PREFILL_NMT / TLQ_PREFILL_KSPLIT force the choice as they do for the
 * launches.  A library choice (launch shape), not an operation of the pages.
 * Returns TLQ_OK or TLQ_EINVAL (count outside 1..16, null arrays, a size
 * below 1, a device entry below 1, or a forced split without the workspace
 * it needs).
 */
tlq_status tl_prefill_plan(const int* M, const int* N, const int* K, const size_t* ws_bytes, int count,
                           const int* device, int* nmt_out, int* ks_out);

/*
 * tl_quant_gemm_ws -- tl_quant_gemm with a caller-owned workspace for the
 * tensor-core kernel's k split (same operation, layouts and errors).
 *   workspace        device buffer, 16-byte aligned, or NULL; must not
 *                    overlap A, C or the weights.  Its contents on entry do
 *                    not matter; on return they are undefined.  Calls whose
 *                    executions overlap on the GPU need separate workspaces.
 *   workspace_bytes  its size.  The kernel splits K only with a split whose
 *                    workspace fits (the largest it wants is
 *                    tl_quant_gemm_workspace_size); results of each output do
 *                    not depend on it beyond FP32 summation order.
 */
tlq_status tl_quant_gemm_ws(const uint16_t* A, const uint32_t* Wpacked, const uint16_t* scales,
                            const uint16_t* zeros, uint16_t* C, int M, int N, int K, int bits, int group,
                            void* workspace, size_t workspace_bytes, void* stream);

/* One problem of tl_quant_gemm_batched: the arguments of one
 * tl_quant_gemm_ws call (device pointers, same layouts and rules), plus the
 * packed weight's row stride.
 *   ldw        row stride of Wpacked in 32-bit words; 0 = compact rows of
 *              K*bits/32 words; else >= K*bits/32 and a multiple of 4 (an
 *              INT2 weight converted in place keeps the INT4 stride K/8).
 *   workspace  this problem's own k-split workspace (NULL / 0: none); the
 *              problems of one call may run at the same time, so their
 *              workspaces must not overlap. */
typedef struct {
  const uint16_t* A;
  const uint32_t* Wpacked;
  const uint16_t* scales;
  const uint16_t* zeros;
  uint16_t* C;
  int M, N, K, bits, group;
  int ldw;
  void* workspace;
  size_t workspace_bytes;
} tl_gemm_desc;

/*
 * tl_quant_gemm_batched -- several independent quant_gemm problems in as few
 * launches as possible: every problem with M <= 16 of one bit width goes into
 * one persistent decode launch (up to 16 problems per launch), each larger
 * problem gets its own tensor-core launch.  Those launches run side by side
 * on up to three library-owned streams per caller stream, forked from
 * `stream` and joined back with events (so the call's work still completes in
 * `stream` order, and a graph capture of `stream` records the fork and join).
 * When two to four such launches run at once, their token tiles per CTA and
 * k splits are planned together for the shared GPU (within the workspace
 * each descriptor gives); otherwise each is planned as a single call would
 * plan it.  Results equal `count` separate tl_quant_gemm_ws calls within the
 * layer's tolerance, and M <= 16 problems bit for bit (a tensor-core
 * problem's k split, and so its FP32 summation order, may differ from the
 * one a single call picks); repeated calls give the same bits.  Same source passages as tl_quant_gemm; batching is a
 * launch-overhead measure of this library (the layers of one decode step that
 * do not depend on each other, or several requests at once).
 *   descs  HOST array of `count` descriptors (count >= 0; 0 is a no-op).
 *   No C may overlap any A or another C.  Every descriptor is validated
 *   before anything is launched (TLQ_EINVAL names the offending index).
 */
tlq_status tl_quant_gemm_batched(const tl_gemm_desc* descs, int count, void* stream);

/*
 * tl_quant_gemm_batched_host -- tl_quant_gemm_batched on HOST activations and
 * outputs: one host -> device copy of the step's activations, the batched
 * GEMMs, one device -> host copy of the outputs, in that order on `stream`.
 * Same source passages as tl_quant_gemm.
 *   hostA   a_bytes of activations (pinned host memory for asynchronous
 *           copies; pageable memory works but the copy blocks the caller).
 *   devA    device staging of a_bytes; every descriptor's A lies inside it.
 *   hostC   c_bytes of outputs (pinned host memory); written when the stream
 *           reaches the copy.
 *   devC    device staging of c_bytes; every descriptor's C lies inside it.
 *   Calls on two streams with two staging sets overlap one call's copies with
 *   the other's GEMMs.  Returns the errors of tl_quant_gemm_batched, TLQ_EINVAL
 *   for null or misplaced buffers, TLQ_ECUDA for a failed copy.
 */
tlq_status tl_quant_gemm_batched_host(const tl_gemm_desc* descs, int count, const void* hostA, void* devA,
                                      size_t a_bytes, void* hostC, const void* devC, size_t c_bytes, void* stream);

/*
 * tl_pack_weights -- pack quantization codes into the kernels' weight format.
 *
 * Source: "beta-Informed Deployment Features", CTX-TIER, "Details of the
 * shipped kernel": an INT4 row takes K/2 bytes, an INT2 row K/4 bytes, four
 * INT2 codes per byte.  The bit order is this library's reading (LSB first).
 *
 *   codes   uint8 [N][K] device array, one code per byte; only the low `bits`
 *           bits of each byte are stored.
 *   Wpacked uint32 [N][K*bits/32] output.
 *   K % (32/bits) == 0.  Bit-exact; deterministic.
 */
tlq_status tl_pack_weights(const uint8_t* codes, uint32_t* Wpacked, int N, int K, int bits,
                           void* stream);

/* Inverse of tl_pack_weights: codes[n][k] = code k of row n (0 .. 2^bits-1). */
tlq_status tl_unpack_weights(const uint32_t* Wpacked, uint8_t* codes, int N, int K, int bits,
                             void* stream);

/*
 * tl_requant_int4_to_int2 -- re-quantize an INT4 weight to INT2, the weight
 * conversion of the context-length tier switch after which quant_gemm routes
 * the layer to the INT2 kernel.
 *
 * Source: "beta-Informed Deployment Features", CTX-TIER, "Details of the
 * shipped kernel" (Phase 2 / 2b): per quantization group the INT4 weights are
 * dequantized, an asymmetric INT2 grid with scale = (max - min) / 3 and
 * zero = min is fitted, and each weight is rounded to the nearest of its four
 * levels; the group size is kept; the INT2 rows are compact so the INT4
 * buffer can be released afterwards.
 *
 * In this library's (q - z) * s form, per group of row n (binary32, rounded
 * to nearest even after every step, in this order):
 *   w  = (q4 - z4) * s4;  lo, hi = min, max of w over the group
 *   s2 = fp16((hi - lo) / 3), or 1.0 when that is zero;  z2 = fp16(-lo / s2)
 *   q2 = clamp(rint(w / s2 + z2), 0, 3)
 * so (q2 - z2) * s2 is the INT2 GEMM's weight.  Codes, s2 and z2 are
 * bit-exact and deterministic.
 *
 *   W4      uint32 [N][K/8] INT4 weight in the tl_pack_weights format;
 *           16-byte aligned; read only.
 *   s4, z4  FP16 [N][K/group] scales / zeros of W4; finite values.
 *   W2      uint32 [N][K/16] output, compact INT2 rows; 16-byte aligned; must
 *           not overlap any other argument -- or exactly W4: converted in
 *           place ("Details of the shipped kernel", storage reuse), the INT2
 *           rows keeping the INT4 row stride of K/8 words with the second
 *           half of every row left untouched; GEMMs then read it with
 *           ldw = K/8 (tl_qproj, tl_gemm_desc).
 *   s2, z2  FP16 [N][K/group] output scales / zeros.  Each may be exactly its
 *           input (s2 == s4, z2 == z4: converted in place) or overlap nothing.
 *   N >= 1; K >= 1; group a multiple of 64 dividing K (the INT2 kernel's
 *   rule); the INT2 weight keeps the INT4 weight's group.
 *   The caller owns every buffer; W4 may be freed once the stream has passed
 *   an out-of-place call.  Returns TLQ_OK, TLQ_EINVAL (null, misaligned, overlapping or
 *   bad shape) or TLQ_ECUDA.
 */
tlq_status tl_requant_int4_to_int2(const uint32_t* W4, const uint16_t* s4, const uint16_t* z4, uint32_t* W2,
                                   uint16_t* s2, uint16_t* z2, int N, int K, int group, void* stream);

/* One weight of tl_requant_int4_to_int2_batched (device pointers, the same
 * layouts and rules as tl_requant_int4_to_int2). */
typedef struct {
  const uint32_t* W4;
  const uint16_t* s4;
  const uint16_t* z4;
  uint32_t* W2;
  uint16_t* s2;
  uint16_t* z2;
  int N, K;
} tl_requant_desc;

/*
 * tl_requant_int4_to_int2_batched -- up to 16 weights of one group size
 * re-quantized in a single launch (the tier switch converts all projections
 * of the loop block at once).  Results equal `count` separate
 * tl_requant_int4_to_int2 calls.
 *   descs  HOST array of `count` descriptors (0 <= count <= 16; 0 is a no-op).
 *   No output (W2, s2, z2) may overlap any other buffer of any descriptor,
 *   except s2 == s4 / z2 == z4 of the same descriptor.  Everything is
 *   validated before the launch (TLQ_EINVAL names the offending index).
 */
tlq_status tl_requant_int4_to_int2_batched(const tl_requant_desc* descs, int count, int group, void* stream);

/*
 * tl_quant_gemm_swiglu -- the SwiGLU feed-forward's gate and up projections as
 * one GEMM with the gate*up product in its epilogue.
 *
 *   C[m][i] = fp16( silu(g) * u ),  g = fp16(acc[m][2i]),  u = fp16(acc[m][2i+1]),
 *   silu(g) = g / (1 + exp(-g)),  acc = A . dequant(Wgu)^T in FP32.
 *
 * Source: "Model", ffn_dim -- "For SwiGLU this is the width of the gate and up
 * projections"; the loop block's mlp_gate / mlp_up weights ("beta-Informed
 * Deployment Features", CTX-TIER, Phase 2b).  g and u are rounded to FP16 like
 * any GEMM output of the block; the product is formed in FP32 (the pages fix
 * neither).
 *   Wgu     packed weights [N2][K] whose rows alternate gate and up: row 2i is
 *           gate row i, row 2i+1 up row i (tl_interleave_rows builds it from
 *           the two packed weights; scales and zeros are interleaved the same
 *           way).  N2 = 2F, a multiple of 16.
 *   C       FP16 [M][N2/2], row stride N2/2; must not overlap A.
 *   Other arguments and errors as tl_quant_gemm.
 */
tlq_status tl_quant_gemm_swiglu(const uint16_t* A, const uint32_t* Wgu, const uint16_t* scales,
                                const uint16_t* zeros, uint16_t* C, int M, int N2, int K, int bits, int group,
                                void* stream);

/* tl_quant_gemm_swiglu with a caller-owned k-split workspace (the rules of
 * tl_quant_gemm_ws; its size from tl_quant_gemm_workspace_size(M, N2, K, ...)). */
tlq_status tl_quant_gemm_swiglu_ws(const uint16_t* A, const uint32_t* Wgu, const uint16_t* scales,
                                   const uint16_t* zeros, uint16_t* C, int M, int N2, int K, int bits, int group,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * tl_dequant_fp16 -- the FP16 body of a quantized weight: out[n][k] =
 * fp16_RNE((q - z) * s), each weight rounded once from its exact value, +0
 * for an exact zero.  Bit-exact and deterministic.
 *
 * Source: "Model", section "VRAM cost": the opt-in FP16 body cache (a dense
 * FP16 copy of the loop-block weights, about 3x their quantized memory).
 * This library offers it as a comparison point for the quantized GEMM: a
 * plain FP16 GEMM on the body.
 *   Wpacked, scales, zeros  as tl_quant_gemm (16-byte aligned Wpacked).
 *   out     FP16 [N][K], row-major, 16-byte aligned, caller-owned; must not
 *           overlap the inputs.
 *   bits, group, N, K: the rules of tl_quant_gemm (N need not be a multiple
 *   of 8).  Returns TLQ_OK, TLQ_EINVAL or TLQ_ECUDA.
 */
tlq_status tl_dequant_fp16(const uint32_t* Wpacked, const uint16_t* scales, const uint16_t* zeros, uint16_t* out,
                           int N, int K, int bits, int group, void* stream);

/*
 * tl_interleave_rows -- out row 2i = row i of a, out row 2i+1 = row i of b
 * (device buffers of `rows` rows of `row_bytes` bytes; out holds 2*rows).
 * Lays out the gate and up weights (packed words, scales, zeros) for
 * tl_quant_gemm_swiglu.  out must not overlap a or b.  Asynchronous on
 * `stream`.  Returns TLQ_OK, TLQ_EINVAL or TLQ_ECUDA.
 */
tlq_status tl_interleave_rows(const void* a, const void* b, void* out, int rows, size_t row_bytes, void* stream);

/* One quantized projection of the loop block: weights [N][K] in the packed
 * format, FP16 scales/zeros [N][K/group]; ldw is the weight's row stride in
 * 32-bit words (0 = compact rows of K*bits/32 words; else >= that and a
 * multiple of 4, e.g. K/8 for an INT2 weight converted in place). */
typedef struct {
  const uint32_t* W;
  const uint16_t* s;
  const uint16_t* z;
  int N;
  int K;
  int ldw;
} tl_qproj;

/*
 * The shared-weight loop block (one weight set reused every iteration).
 *   qkv  : N = 3*D, K = D        o    : N = D, K = D
 *   up   : N = F,   K = D        down : N = D, K = F
 * Scratch buffers are caller-owned device FP16 arrays with at least M rows:
 *   h [M][D], qkv_out [M][3D], o_out [M][D], up_out [M][F].
 * normalize = 1 applies the per-row RMS pre-norm h = fp16(x / sqrt(mean x^2 +
 * 1e-5)) before the QKV projection (the block's LayerNorm position, "Model",
 * "VRAM cost", with buf.norm as its FP16 output); 0 feeds fp16(x) directly.
 * workspace / workspace_bytes: the caller's k-split workspace for the block's
 * GEMMs with M > 16 (they run one after another and share it; NULL / 0 = no
 * k split); the largest tl_quant_gemm_workspace_size of the four GEMMs at M
 * rows is what they can use.  Must not overlap any other buffer.
 */
typedef struct {
  tl_qproj qkv, o, up, down;
  int bits;
  int group;
  int D;
  uint16_t* h;
  uint16_t* qkv_out;
  uint16_t* o_out;
  uint16_t* up_out;
  int normalize;
  void* workspace;
  size_t workspace_bytes;
} tl_block;

/*
 * The five-weight SwiGLU loop block (attn_qkv, attn_out, mlp_gate, mlp_up,
 * mlp_down -- "beta-Informed Deployment Features", CTX-TIER, Phase 2b;
 * "Model", ffn_dim):
 *   h = norm(x); qkv = Q(h); o = Q(qkv[:, :D]);
 *   a = fp16(silu(Q_gate(o)) * Q_up(o)); x += float(Q_down(a))
 * with every GEMM output rounded to FP16 and the residual add in FP32.
 *   qkv     : N = 3*D, K = D          o    : N = D, K = D
 *   gate_up : N = 2*F, K = D, rows interleaved (see tl_quant_gemm_swiglu)
 *   down    : N = D, K = F
 * Scratch (caller-owned device FP16, at least M rows): h [M][D],
 * qkv_out [M][3D], o_out [M][D], act_out [M][F].  normalize and workspace as
 * tl_block.
 */
typedef struct {
  tl_qproj qkv, o, gate_up, down;
  int bits;
  int group;
  int D;
  uint16_t* h;
  uint16_t* qkv_out;
  uint16_t* o_out;
  uint16_t* act_out;
  int normalize;
  void* workspace;
  size_t workspace_bytes;
} tl_swiglu_block;

/*
 * tl_loop_block_forward -- apply the shared block L times to the FP32
 * residual stream x[M][D] in place:
 *
 *   for l in 0..L-1:
 *     h   = fp16(rmsnorm(x))            (or fp16(x) when normalize = 0)
 *     qkv = quant_gemm(h, qkv)          [M][3D]
 *     o   = quant_gemm(qkv[:, :D], o)   [M][D]   (row stride 3D)
 *     u   = relu(quant_gemm(o, up))     [M][F]   relu(v) = v > 0 ? v : +0
 *     x  += float(quant_gemm(u, down))  FP32 add of the FP16 result
 *
 * Source: "Model", "VRAM cost", Runtime buffers (buf.main is the FP32
 * residual, the scratch buffers are FP16); "Warm-start mid-loop", internal
 * flow, "Extend loop" (the block is re-run in place on the residual, so
 * running L1 then L - L1 iterations equals running L, bit for bit).
 *   x      FP32 [M][D] device array, updated in place.
 *   block  HOST pointer to a tl_block describing device buffers.
 *   L >= 0 (L = 0 is a no-op); M >= 1.
 * L2 residency (see tl_loop_block_l2_plan): the projections the plan keeps
 * resident are streamed with an evict-last policy, the others evict-first.
 * With TLQ_LOG=1 in the environment the first call prints the plan.
 */
tlq_status tl_loop_block_forward(float* x, const tl_block* block, int L, int M, void* stream);

/*
 * tl_loop_block_l2_plan -- the loop block's L2 residency plan ("Model",
 * "Returns", item 4: auto tile sizing reports loop-block vs L2 cache
 * residency).  The block's weights (packed words plus FP16 scales and zeros)
 * are re-read every iteration; the plan keeps projections resident, in
 * iteration order (qkv, o, up, down), while their running total fits a
 * budget of half the device's L2, and only when L > 1.
 *   block          HOST pointer; only the projections' N and K, bits and
 *                  group are read (no device memory is touched).
 *   resident_mask  out: bit i set when projection i is kept resident.
 *   weight_bytes, budget_bytes  out (may be NULL): the block's weight bytes
 *                  and the budget.
 * The SwiGLU block uses the same plan over (qkv, o, gate_up, down).
 * Returns TLQ_OK or TLQ_EINVAL.
 */
tlq_status tl_loop_block_l2_plan(const tl_block* block, int L, int* resident_mask, size_t* weight_bytes,
                                 size_t* budget_bytes);

/*
 * tl_swiglu_block_forward -- the five-weight SwiGLU loop block applied L times
 * to the FP32 residual x [M][D] in place (same rules, errors and L2 policy as
 * tl_loop_block_forward; the gate/up GEMM runs with the SwiGLU epilogue, so a
 * block iteration is five launches like the ReLU block).
 */
tlq_status tl_swiglu_block_forward(float* x, const tl_swiglu_block* block, int L, int M, void* stream);

/*
 * tl_loop_block_forward_chunked / tl_swiglu_block_forward_chunked -- chunked
 * prefill: the M rows of x are split into chunks of `chunk` rows and each
 * chunk runs through all L iterations before the next one starts, so the
 * scratch buffers need only min(chunk, M) rows.
 *
 * Source: "Model", section "Chunked prefill": prompts longer than
 * prefill_chunk are split into chunks that each run through all blocks and
 * loop iterations in turn; the buffer VRAM shrinks with the chunk while the
 * launch count grows with the number of chunks.  The block's rows are
 * independent (no attention on this path), so every chunk is the block on a
 * row slice; results match single-shot within the GEMM tolerance (the kernel
 * choice and summation order depend on the row count: M <= 16 takes the
 * decode kernel).
 *   chunk <= 0 or chunk >= M: single shot.  Other arguments and errors as the
 *   unchunked calls; scratch rows must cover min(chunk, M).
 */
tlq_status tl_loop_block_forward_chunked(float* x, const tl_block* block, int L, int M, int chunk, void* stream);
tlq_status tl_swiglu_block_forward_chunked(float* x, const tl_swiglu_block* block, int L, int M, int chunk,
                                           void* stream);

/*
 * tl_loop_block_to_int2 / tl_swiglu_block_to_int2 -- the context-length tier
 * switch of a loop block: its four weights (the SwiGLU block's fused gate/up
 * weight re-quantizes row by row like the two it holds) are re-quantized
 * INT4 -> INT2 as tl_requant_int4_to_int2 does, and the HOST block
 * description is rewritten (bits = 2, each projection's W / s / z / ldw) so
 * later forwards run the INT2 kernels.
 *
 * Source: "beta-Informed Deployment Features", CTX-TIER, "What Phase 2
 * ships", item 2 (apply_tier_to_model: the loop block's weights re-quantized,
 * the bit width flipped so the dispatcher routes to int2_gemm) and Phase 2b
 * (compact INT2 buffers, the INT4 ones released).
 *   block  HOST pointer; an INT4 block (bits = 4, compact INT4 rows, a group
 *          that is a multiple of 64).
 *   dst    HOST array of four destinations (qkv, o, up or gate_up, down), each
 *          with the weight's N and K: W compact INT2 rows (K/16 words) or the
 *          INT4 weight itself (in place, ldw = K/8 afterwards); s / z new
 *          arrays or the INT4 ones (converted in place).  NULL: everything in
 *          place (no new memory at all).
 *   Every check happens before the launch; on an error the block is left as
 *   it was.  Out of place, the INT4 buffers may be freed once `stream` has
 *   passed the call.  Returns TLQ_OK, TLQ_EINVAL or TLQ_ECUDA.
 */
tlq_status tl_loop_block_to_int2(tl_block* block, const tl_qproj* dst, void* stream);
tlq_status tl_swiglu_block_to_int2(tl_swiglu_block* block, const tl_qproj* dst, void* stream);

/*
 * tl_loop_block_forward_static_scratch -- tl_loop_block_forward for callers
 * that cannot allocate device memory or provide scratch buffers (a serving
 * runtime that forbids allocation after start-up, a plugin interface that only
 * passes a layer its inputs and outputs).  There is no counterpart on the
 * pages: it is a packaging choice of this library.
 *
 * Identical arithmetic to tl_loop_block_forward; block->h, qkv_out, o_out,
 * up_out and workspace are ignored (may be NULL): the GEMMs run without a k
 * split.  The four FP16 intermediates live in one
 * 4 MiB static device array inside the library, which every GPU that loads
 * the library holds until the process exits.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *   Size limit: 2*M*(5*D + F) bytes (each buffer rounded up to 256 bytes)
 *   must fit in 4 MiB -- e.g. M <= 113 at D = 2048, F = 8192 -- otherwise
 *   TLQ_EINVAL with a message that names the sizes, and nothing is launched.
 *   First call on a device: looks up the array's device address (once per
 *   device, with that device current) and keeps it for the life of the
 *   process; make that first call before any stream capture.  A device reset
 *   (cudaDeviceReset) invalidates the kept address: after one, this entry
 *   point must not be called again in the same process.
 *   All calls on a device share the one array, which keeps whatever the last
 *   call left in it; every intermediate is fully written before it is read,
 *   so nothing needs clearing.  Calls whose executions overlap on the GPU
 *   (other streams, other threads) race on the array: serialize them.
 */
tlq_status tl_loop_block_forward_static_scratch(float* x, const tl_block* block, int L, int M, void* stream);

/*
 * tl_probe_read_bandwidth -- a measurement helper, no operation of the pages:
 * `reps` passes of 16-byte L2-only loads (ld.global.cg) over buf, folded into
 * one word per thread of sink (2 x SMs x 512 words, caller-owned).  With buf
 * small enough to stay in L2 it measures the L2 read bandwidth that bounds
 * the loop block (its packed weights fit in L2 and are re-read every
 * iteration); the benchmark times it with CUDA events.
 *   buf    device buffer, 16-byte aligned; bytes a positive multiple of 16.
 * Returns TLQ_OK, TLQ_EINVAL or TLQ_ECUDA.
 */
tlq_status tl_probe_read_bandwidth(const void* buf, size_t bytes, int reps, uint32_t* sink, void* stream);

/*
 * Synchronize `stream` and report the device status word: TLQ_OK, or
 * TLQ_ETIMEOUT if a kernel gave up on a bounded wait since the last
 * tl_reset_status().  Also returns TLQ_ECUDA on an asynchronous CUDA error.
 */
tlq_status tl_check_status(void* stream);

/* Clear the device status word of the current device; synchronizes `stream`. */
tlq_status tl_reset_status(void* stream);

/*
 * Self-test of the bounded device waits (no counterpart on the pages; it
 * backs the library's own failure-detection contract).  Launches a one-thread
 * kernel that waits on a shared-memory barrier nothing ever arrives at; the
 * wait gives up after limit_us microseconds (1 .. 1,000,000), records
 * TLQ_ETIMEOUT in the status word and the kernel returns normally, leaving the
 * context usable.  Read the result with tl_check_status().
 */
tlq_status tl_selftest_wait_timeout(unsigned limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TLQ_H_ */

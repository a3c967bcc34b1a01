/*
 * Reference oracle for the weight-only quantized linear layer (quant_gemm) and
 * the shared-weight loop block of the TinyLoop runtime.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU library computes.  Only the test-suite, the
 * package smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or constant generator with the CUDA library
 * and includes nothing from it.
 *
 * Sources (TinyLoop documentation):
 *  - "Model" (Python API), section "VRAM cost", item Weights: each quantized
 *    layer is INT2 / INT4 packed data plus FP16 scales plus FP16 zeros; item
 *    Runtime buffers: the residual stream buf.main is FP32, the scratch
 *    buffers (norm, scratch1, attn_down) are FP16.
 *  - "beta-Informed Deployment Features", section CTX-TIER, "Details of the
 *    shipped kernel": group-wise asymmetric quantization (groups of typically
 *    128 weights), an INT4 row occupies K/2 bytes and an INT2 row K/4 bytes,
 *    four INT2 codes share one byte.
 *  - "Warm-start mid-loop", section on the internal flow (Extend loop): the
 *    shared block is applied in place on the residual, iteration after
 *    iteration, with the same weights.
 *
 * Readings where the pages are silent (each one is a choice of this library):
 *  - Bit order: code j of a 32-bit word sits at bits [b*j, b*j + b) (LSB
 *    first); word w of row n holds k = w*(32/b) ... w*(32/b) + 32/b - 1.
 *  - Dequantization: w = (q - z) * s with z and s FP16 per (row, group);
 *    scales and zeros are two row-major [N][K/group] arrays.
 *  - C[m][n] = fp16_RNE( sum_k A[m][k] * w[n][k] ): accumulate in binary64 in
 *    plain k order, round once.
 *  - Loop block: h = fp16(x / sqrt(mean(x^2) + eps)) (or fp16(x) without the
 *    norm); qkv = Q(h); o = Q(qkv[:, :D]); u = relu(Q(o)); x += float(Q(u)),
 *    every GEMM output rounded to FP16, the residual add done in FP32.
 *    relu(v) = v if v > 0 else +0.
 *  - SwiGLU loop block (five weights: qkv, o, gate, up, down): as above up
 *    to o, then g = Q_gate(o), u = Q_up(o) (FP16 GEMM outputs) and
 *    a = fp16_RNE(silu(g) * u) with silu(g) = g / (1 + exp(-g)) evaluated in
 *    binary64 on the FP16 values; x += float(Q_down(a)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> binary64, written from the format definition. */
/* ------------------------------------------------------------------ */

double orc_half_to_double(uint16_t h) {
  int neg = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return neg ? -v : v;
}

/* Round a binary64 value to binary16, round-to-nearest, ties to even. */
uint16_t orc_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* 65504 + ulp/2: ties go to the even neighbour, inf */
  int e2;
  frexp(a, &e2);       /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;      /* a in [2^E, 2^(E+1)) */
  int qexp = (E < -14) ? -24 : E - 10; /* weight of the last kept bit */
  double scaled = ldexp(a, -qexp);     /* exact: a power-of-two scaling */
  double fl = floor(scaled);
  double frac = scaled - fl;           /* exact */
  uint32_t r = (uint32_t)fl;
  if (frac > 0.5 || (frac == 0.5 && (r & 1u))) r += 1u;
  if (E < -14) {
    /* subnormal range: r in [0, 1024]; r == 1024 is the smallest normal */
    return (uint16_t)(sign | r);
  }
  if (r == 2048u) { /* carried into the next binade */
    r = 1024u;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint32_t)((E + 15) << 10) | (r - 1024u));
}

/* ------------------------------------------------------------------ */
/* Packing                                                              */
/* ------------------------------------------------------------------ */

/* codes [N][K] (one code per byte, only the low `bits` bits are kept) ->
 * words [N][K*bits/32].  Returns 0, or -1 for an unsupported shape. */
int orc_pack(const uint8_t* codes, uint32_t* words, int N, int K, int bits) {
  if (bits != 2 && bits != 4) return -1;
  int cpw = 32 / bits;
  if (N < 0 || K < 0 || K % cpw) return -1;
  int wpr = K / cpw;
  uint32_t mask = (1u << bits) - 1u;
  for (int n = 0; n < N; ++n) {
    for (int w = 0; w < wpr; ++w) {
      uint32_t word = 0;
      for (int j = 0; j < cpw; ++j) {
        uint32_t q = (uint32_t)codes[(size_t)n * K + (size_t)w * cpw + j] & mask;
        word |= q << (bits * j);
      }
      words[(size_t)n * wpr + w] = word;
    }
  }
  return 0;
}

int orc_unpack(const uint32_t* words, uint8_t* codes, int N, int K, int bits) {
  if (bits != 2 && bits != 4) return -1;
  int cpw = 32 / bits;
  if (N < 0 || K < 0 || K % cpw) return -1;
  int wpr = K / cpw;
  uint32_t mask = (1u << bits) - 1u;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      uint32_t word = words[(size_t)n * wpr + k / cpw];
      codes[(size_t)n * K + k] = (uint8_t)((word >> (bits * (k % cpw))) & mask);
    }
  return 0;
}

static int check_shape(int N, int K, int bits, int group) {
  if (bits != 2 && bits != 4) return -1;
  if (N < 0 || K <= 0 || group <= 0) return -1;
  if (K % group) return -1;
  if (K % (32 / bits)) return -1;
  return 0;
}

/* One code of a packed row. */
static uint32_t code_at(const uint32_t* row_words, int k, int bits) {
  int cpw = 32 / bits;
  return (row_words[k / cpw] >> (bits * (k % cpw))) & ((1u << bits) - 1u);
}

/* w[n][k] = (q - z[n][k/group]) * s[n][k/group], in binary64.  The value is
 * exact: q - z needs at most 12 significant bits and the product at most 23. */
int orc_dequant(const uint32_t* W, const uint16_t* scales, const uint16_t* zeros,
                int N, int K, int bits, int group, double* w) {
  if (check_shape(N, K, bits, group)) return -1;
  int wpr = K * bits / 32;
  int G = K / group;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      double q = (double)code_at(W + (size_t)n * wpr, k, bits);
      double s = orc_half_to_double(scales[(size_t)n * G + k / group]);
      double z = orc_half_to_double(zeros[(size_t)n * G + k / group]);
      w[(size_t)n * K + k] = (q - z) * s;
    }
  return 0;
}

/* The FP16 "body" of a quantized weight: each weight dequantized exactly
 * and rounded once to FP16 (RNE); an exact zero is stored as +0.  This is the
 * dense copy the runtime's dequant-to-FP16 cache keeps ("Model", section
 * "VRAM cost", the FP16 body cache option), here as a comparison point for
 * the quantized GEMM. */
int orc_dequant_half(const uint32_t* W, const uint16_t* scales, const uint16_t* zeros,
                     int N, int K, int bits, int group, uint16_t* out) {
  if (check_shape(N, K, bits, group)) return -1;
  int wpr = K * bits / 32;
  int G = K / group;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      double q = (double)code_at(W + (size_t)n * wpr, k, bits);
      double sc = orc_half_to_double(scales[(size_t)n * G + k / group]);
      double z = orc_half_to_double(zeros[(size_t)n * G + k / group]);
      double w = (q - z) * sc; /* exact in binary64 */
      out[(size_t)n * K + k] = w == 0.0 ? (uint16_t)0 : orc_double_to_half(w);
    }
  return 0;
}

/* ------------------------------------------------------------------ */
/* The quantized GEMM                                                   */
/* ------------------------------------------------------------------ */

/* C[m][n] (row stride ldc) = fp16( sum_k A[m][k] (row stride lda) * w[n][k] ).
 * Binary64 accumulation in plain k order, one final rounding.  Output rows n
 * are independent, so they are shared out over the host's threads (OpenMP);
 * each output is still the same plain k-order sum whatever the thread count. */
int orc_quant_gemm(const uint16_t* A, int lda, const uint32_t* W, const uint16_t* scales,
                   const uint16_t* zeros, uint16_t* C, int ldc, int M, int N, int K,
                   int bits, int group) {
  if (check_shape(N, K, bits, group) || M < 0 || lda < K || ldc < N) return -1;
  double* arow = (double*)malloc(sizeof(double) * (size_t)K * (M > 0 ? M : 1));
  if (!arow) return -2;
  for (int m = 0; m < M; ++m)
    for (int k = 0; k < K; ++k) arow[(size_t)m * K + k] = orc_half_to_double(A[(size_t)m * lda + k]);
  int wpr = K * bits / 32;
  int G = K / group;
  int bad = 0;
#pragma omp parallel reduction(| : bad)
  {
    double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
    if (!wrow) bad = 1;
#pragma omp for schedule(static)
    for (int n = 0; n < N; ++n) {
      if (!wrow) continue;
      for (int k = 0; k < K; ++k) {
        double q = (double)code_at(W + (size_t)n * wpr, k, bits);
        double s = orc_half_to_double(scales[(size_t)n * G + k / group]);
        double z = orc_half_to_double(zeros[(size_t)n * G + k / group]);
        wrow[k] = (q - z) * s;
      }
      for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        const double* a = arow + (size_t)m * K;
        for (int k = 0; k < K; ++k) acc += a[k] * wrow[k];
        C[(size_t)m * ldc + n] = orc_double_to_half(acc);
      }
    }
    free(wrow);
  }
  free(arow);
  return bad ? -2 : 0;
}

/* Thread count of the OpenMP loops above (1 = the plain single-thread
 * oracle); returns the count now in effect. */
int orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* The same definition evaluated at P chosen output positions (pm[i], pn[i]);
 * used to check full-size results on a sample of outputs. */
int orc_quant_gemm_points(const uint16_t* A, int lda, const uint32_t* W, const uint16_t* scales,
                          const uint16_t* zeros, int M, int N, int K, int bits, int group,
                          const int* pm, const int* pn, int P, uint16_t* out) {
  if (check_shape(N, K, bits, group) || M < 0 || lda < K) return -1;
  int wpr = K * bits / 32;
  int G = K / group;
  for (int i = 0; i < P; ++i) {
    int m = pm[i], n = pn[i];
    if (m < 0 || m >= M || n < 0 || n >= N) return -1;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
      double q = (double)code_at(W + (size_t)n * wpr, k, bits);
      double s = orc_half_to_double(scales[(size_t)n * G + k / group]);
      double z = orc_half_to_double(zeros[(size_t)n * G + k / group]);
      acc += orc_half_to_double(A[(size_t)m * lda + k]) * ((q - z) * s);
    }
    out[i] = orc_double_to_half(acc);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Loop block                                                           */
/* ------------------------------------------------------------------ */

/* h[m][:] = fp16( x[m][:] / sqrt(mean_k x[m][k]^2 + eps) ), binary64 inside. */
int orc_rms_norm_half(const float* x, int M, int D, double eps, uint16_t* h) {
  if (M < 0 || D <= 0) return -1;
  for (int m = 0; m < M; ++m) {
    const float* r = x + (size_t)m * D;
    double ss = 0.0;
    for (int k = 0; k < D; ++k) ss += (double)r[k] * (double)r[k];
    double inv = 1.0 / sqrt(ss / (double)D + eps);
    for (int k = 0; k < D; ++k) h[(size_t)m * D + k] = orc_double_to_half((double)r[k] * inv);
  }
  return 0;
}

typedef struct {
  const uint32_t* W;
  const uint16_t* scales;
  const uint16_t* zeros;
} orc_proj;

/* x[M][D] (FP32, updated in place) <- L applications of the shared block
 * {qkv: [3D x D], o: [D x D], up: [F x D], down: [D x F]}. */
int orc_loop_block(float* x, int M, int D, int F, const orc_proj* qkv, const orc_proj* o,
                   const orc_proj* up, const orc_proj* down, int bits, int group, int L,
                   int normalize, double eps) {
  if (M < 0 || D <= 0 || F <= 0 || L < 0) return -1;
  if (check_shape(3 * D, D, bits, group) || check_shape(D, F, bits, group)) return -1;
  size_t nh = (size_t)M * D, nq = (size_t)M * 3 * D, nu = (size_t)M * F;
  uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  uint16_t* q = (uint16_t*)malloc(sizeof(uint16_t) * (nq ? nq : 1));
  uint16_t* ob = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * (nu ? nu : 1));
  uint16_t* d = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  int rc = 0;
  if (!h || !q || !ob || !u || !d) rc = -2;
  for (int l = 0; l < L && rc == 0; ++l) {
    if (normalize) {
      orc_rms_norm_half(x, M, D, eps, h);
    } else {
      for (size_t i = 0; i < nh; ++i) h[i] = orc_double_to_half((double)x[i]);
    }
    rc |= orc_quant_gemm(h, D, qkv->W, qkv->scales, qkv->zeros, q, 3 * D, M, 3 * D, D, bits, group);
    rc |= orc_quant_gemm(q, 3 * D, o->W, o->scales, o->zeros, ob, D, M, D, D, bits, group);
    rc |= orc_quant_gemm(ob, D, up->W, up->scales, up->zeros, u, F, M, F, D, bits, group);
    for (size_t i = 0; i < nu; ++i) {
      double v = orc_half_to_double(u[i]);
      if (!(v > 0.0)) u[i] = 0; /* relu, +0 */
    }
    rc |= orc_quant_gemm(u, F, down->W, down->scales, down->zeros, d, D, M, D, F, bits, group);
    for (size_t i = 0; i < nh; ++i) {
      float dv = (float)orc_half_to_double(d[i]); /* exact: FP16 fits FP32 */
      x[i] = x[i] + dv;                           /* FP32 addition, one rounding */
    }
  }
  free(h);
  free(q);
  free(ob);
  free(u);
  free(d);
  return rc;
}

/* ------------------------------------------------------------------ */
/* SwiGLU: the gated feed-forward of the five-weight loop block         */
/* ------------------------------------------------------------------ */

/* "Model", ffn_dim: "For SwiGLU this is the width of the gate and up
 * projections"; the five loop-block weights attn_qkv, attn_out, mlp_gate,
 * mlp_up, mlp_down ("beta-Informed Deployment Features", CTX-TIER, Phase 2b).
 * out[i] = fp16_RNE( g * u / (1 + exp(-g)) ) in binary64, g and u FP16. */
int orc_swiglu(const uint16_t* g, const uint16_t* u, uint16_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    const double gv = orc_half_to_double(g[i]);
    const double uv = orc_half_to_double(u[i]);
    const double silu = gv / (1.0 + exp(-gv));
    out[i] = orc_double_to_half(silu * uv);
  }
  return 0;
}

/* x[M][D] (FP32, updated in place) <- L applications of the SwiGLU block
 * {qkv: [3D x D], o: [D x D], gate: [F x D], up: [F x D], down: [D x F]}. */
int orc_loop_block_swiglu(float* x, int M, int D, int F, const orc_proj* qkv, const orc_proj* o,
                          const orc_proj* gate, const orc_proj* up, const orc_proj* down, int bits,
                          int group, int L, int normalize, double eps) {
  if (M < 0 || D <= 0 || F <= 0 || L < 0) return -1;
  if (check_shape(3 * D, D, bits, group) || check_shape(F, D, bits, group) || check_shape(D, F, bits, group))
    return -1;
  size_t nh = (size_t)M * D, nq = (size_t)M * 3 * D, nu = (size_t)M * F;
  uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  uint16_t* q = (uint16_t*)malloc(sizeof(uint16_t) * (nq ? nq : 1));
  uint16_t* ob = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  uint16_t* gb = (uint16_t*)malloc(sizeof(uint16_t) * (nu ? nu : 1));
  uint16_t* ub = (uint16_t*)malloc(sizeof(uint16_t) * (nu ? nu : 1));
  uint16_t* ab = (uint16_t*)malloc(sizeof(uint16_t) * (nu ? nu : 1));
  uint16_t* d = (uint16_t*)malloc(sizeof(uint16_t) * (nh ? nh : 1));
  int rc = 0;
  if (!h || !q || !ob || !gb || !ub || !ab || !d) rc = -2;
  for (int l = 0; l < L && rc == 0; ++l) {
    if (normalize) {
      orc_rms_norm_half(x, M, D, eps, h);
    } else {
      for (size_t i = 0; i < nh; ++i) h[i] = orc_double_to_half((double)x[i]);
    }
    rc |= orc_quant_gemm(h, D, qkv->W, qkv->scales, qkv->zeros, q, 3 * D, M, 3 * D, D, bits, group);
    rc |= orc_quant_gemm(q, 3 * D, o->W, o->scales, o->zeros, ob, D, M, D, D, bits, group);
    rc |= orc_quant_gemm(ob, D, gate->W, gate->scales, gate->zeros, gb, F, M, F, D, bits, group);
    rc |= orc_quant_gemm(ob, D, up->W, up->scales, up->zeros, ub, F, M, F, D, bits, group);
    rc |= orc_swiglu(gb, ub, ab, nu);
    rc |= orc_quant_gemm(ab, F, down->W, down->scales, down->zeros, d, D, M, D, F, bits, group);
    for (size_t i = 0; i < nh; ++i) {
      float dv = (float)orc_half_to_double(d[i]);
      x[i] = x[i] + dv;
    }
  }
  free(h);
  free(q);
  free(ob);
  free(gb);
  free(ub);
  free(ab);
  free(d);
  return rc;
}

/* ------------------------------------------------------------------ */
/* INT4 -> INT2 group re-quantization                                  */
/* ------------------------------------------------------------------ */

/* "beta-Informed Deployment Features", CTX-TIER, "Details of the shipped
 * kernel": every quantization group of the INT4 weight is dequantized, a new
 * asymmetric INT2 grid with scale = (max - min) / 3 and zero = min is fitted,
 * and each weight is rounded to the nearest of the grid's four levels; the
 * group size stays that of the INT4 weight and the INT2 rows are compact
 * (K/4 bytes, out of place, as in the page's Phase 2b).
 *
 * Readings of this library, all in binary32 and in this order (the GPU takes
 * every integer decision in the same precision):
 *   w      = (q4 - z4) * s4                  exact (see orc_dequant)
 *   lo, hi = min and max of w over the group
 *   s2     = fp16_RNE((hi - lo) / 3); 1.0 when that is zero
 *   z2     = fp16_RNE(-lo / s2)              zero = min in this library's
 *                                            (q - z) * s form
 *   q2     = clamp(rint(w / s2 + z2), 0, 3)  round to nearest, ties to even
 * so that (q2 - z2) * s2 is exactly what the INT2 GEMM reads. */
int orc_requant_int4_to_int2(const uint32_t* W4, const uint16_t* s4, const uint16_t* z4, int N, int K,
                             int group, uint32_t* W2, uint16_t* s2, uint16_t* z2) {
  if (check_shape(N, K, 4, group) || check_shape(N, K, 2, group) || group % 16) return -1;
  const int wpr4 = K / 8, wpr2 = K / 16, G = K / group;
  float* w = (float*)malloc(sizeof(float) * (size_t)group);
  if (!w) return -2;
  memset(W2, 0, sizeof(uint32_t) * (size_t)N * wpr2);
  for (int n = 0; n < N; ++n) {
    for (int g = 0; g < G; ++g) {
      const size_t gi = (size_t)n * G + g;
      const float s = (float)orc_half_to_double(s4[gi]); /* exact: binary16 fits binary32 */
      const float z = (float)orc_half_to_double(z4[gi]);
      float lo = INFINITY, hi = -INFINITY;
      for (int j = 0; j < group; ++j) {
        const int k = g * group + j;
        const float q = (float)code_at(W4 + (size_t)n * wpr4, k, 4);
        const float v = (q - z) * s;
        w[j] = v;
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      uint16_t sb = orc_double_to_half((double)((hi - lo) / 3.0f));
      if (orc_half_to_double(sb) == 0.0) sb = orc_double_to_half(1.0);
      const float sh = (float)orc_half_to_double(sb);
      const uint16_t zb = orc_double_to_half((double)(-lo / sh));
      const float zh = (float)orc_half_to_double(zb);
      for (int j = 0; j < group; ++j) {
        const int k = g * group + j;
        float t = w[j] / sh;
        t = t + zh;
        float r = rintf(t);
        if (r < 0.0f) r = 0.0f;
        if (r > 3.0f) r = 3.0f;
        W2[(size_t)n * wpr2 + k / 16] |= (uint32_t)r << (2 * (k % 16));
      }
      s2[gi] = sb;
      z2[gi] = zb;
    }
  }
  free(w);
  return 0;
}

/*
 * CPU oracle for one batch-1 autoregressive decode step of a dense (or top-k MoE)
 * decoder-only transformer.  TEST INFRASTRUCTURE ONLY: the product path never
 * links, loads or calls this file; only tests, the smoke check and the timed CPU
 * baseline of the benchmark do.  It shares no code with the CUDA engine.
 *
 * What it computes follows the pages on single-request decode:
 *  - [H] hakusoku.com, "標準GPUによるリアルタイムLLM推論：リクエストあたり3,000トークン/秒":
 *      section "GPU推論の速度制限要因：メモリ帯域幅" (at batch 1 the step is matrix-vector
 *      products over every active weight, plus the KV cache), section
 *      "Kog Inference Engineの特徴とイノベーション" (the step's stages: MatMul,
 *      attention, normalization, routing, sampling).
 *  - [A] aether-echoes.com, "標準 GPU で LLM 推論 3000 tokens/s/req", section "どう出したか":
 *      no quantization, no speculative decoding, no pruning, no KV-cache compression —
 *      so the step is the exact transformer step, with the KV cache kept in full.
 * Where the pages leave a step open, the readings taken are: pre-norm decoder with
 * RMSNorm (eps inside the root, gain after), rotate-half RoPE applied before caching,
 * grouped-query attention over positions 0..p with query head h reading KV head
 * floor(h*hkv/hq), SwiGLU FFN, softmax top-k routing renormalised over the chosen
 * experts, per-output-channel e4m3 expert scales applied after the dot product,
 * greedy argmax (lowest index on ties) or inverse-CDF temperature sampling.
 * Every activation is fp32; the only rounding to a narrow type is the KV store.
 *
 * Two modes:
 *  ORC_PLAIN  the textbook step: sequential fp32 sums, libm expf.  This is the
 *             definition the logits tolerances are taken against.
 *  ORC_EXACT  the same step under the engine's stated arithmetic contract (fixed
 *             summation trees and block structure, an exp of our own), so that KV
 *             rows, logits and tokens can be compared bit for bit.  The contract:
 *    dot(w,x,K,VW): 32 partial sums; vector v (VW consecutive elements) goes to
 *        partial v mod 32 in ascending v, its elements fused-multiply-added in
 *        ascending order; the partials are then folded pairwise (i, i+16), (i, i+8),
 *        (i, i+4), (i, i+2), (i, i+1).  The step uses VW = 8 for every operand type.
 *    rmsnorm: ss = dot(x,x,d,8); r = 1/sqrtf(ss/d + eps); xn_i = (x_i*r)*g_i.
 *    rope:    a' = fma(a, c, -(b*s)); b' = fma(b, c, a*s); cos/sin tables from
 *             double pow/cos/sin rounded to fp32.
 *    exp_c:   Cody-Waite reduction by a two-part ln 2, degree-7 Taylor polynomial
 *             (Horner, fma), scaling by 2^n; 0 below -87, +inf from 88 up.
 *    attention: blocks of 32 positions; per block m = max, e = exp_c(s-m),
 *             l = sequential sum, o = sequential fma chain; blocks merged in
 *             ascending order with w_b = exp_c(m_b - M): L = fma(w_b, l_b, L),
 *             O = fma(w_b, o_b, O), out = O / L.
 *    silu(g)*u = (g / (1 + exp_c(-g))) * u.
 *    nvfp4 layer matrices (4-bit e2m1 codes, one e4m3 scale per 16 consecutive elements of a row,
 *             one fp32 scale per row): per 8-element vector v the codes' products with x are
 *             fused-multiply-added into t_v (from 0, elements ascending), then
 *             partial[v mod 32] = fma(blockscale(v), t_v, partial); fold as dot; times the row
 *             scale.  (PLAIN: rowscale * sequential sum of (blockscale * code) * x.)
 *    router softmax: sequential sum over experts; top-k ties to the lower index;
 *             gates = P / (sequential sum of the chosen P in choice order);
 *             expert outputs combined by an fma chain in choice order.
 *    sampling: e_i = exp_c((l_i - M) / T); per 256-entry vocabulary block
 *             S_b = dot(e_block, 1, n, 8); Z = sequential sum of S_b; tau = u*Z;
 *             the first block whose running prefix exceeds tau, then the first
 *             index in it whose running sum (from the block's prefix) exceeds tau.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp -std=c11 -ffp-contract=off (no fast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F32 = 3, ORC_NVFP4 = 4 };
enum { ORC_PLAIN = 0, ORC_EXACT = 1 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ECTX = -3, ORC_ENOMEM = -4 };

typedef struct {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab, max_ctx;
  float rms_eps, rope_theta;
  int32_t tied_embeddings;
  int32_t weight_dtype, kv_dtype;
  int32_t n_experts, top_k, d_expert;
  int32_t router_dtype, expert_dtype;
  int32_t embed_dtype;  /* embedding, LM head, norm gains when weight_dtype is e4m3 or nvfp4 */
} orc_config;

typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm;
  const void *w_gate, *w_up, *w_down;
  const void *router;
  const void *e_gate, *e_up, *e_down;
  const float *e_gate_scale, *e_up_scale, *e_down_scale;
  /* per-output-channel scales of the layer matrices when weight_dtype is e4m3 or nvfp4 (else NULL) */
  const float *wq_scale, *wk_scale, *wv_scale, *wo_scale, *w_gate_scale, *w_up_scale, *w_down_scale;
  /* nvfp4 only: e4m3 scale codes of each 16-element block, [rows][K/16] (else NULL); the matrices
   * then hold two e2m1 codes per byte, element 2i in the low nibble */
  const uint8_t *wq_bscale, *wk_bscale, *wv_bscale, *wo_bscale, *w_gate_bscale, *w_up_bscale, *w_down_bscale;
} orc_layer;

typedef struct {
  const void *tok_emb, *lm_head, *final_norm;
  const orc_layer* layers;
} orc_weights;

/* ------------------------------------------------------------------ storage types */

static float F16_TABLE[65536];
static float E4M3_TABLE[256];
static float E2M1_TABLE[16];
static int tables_ready = 0;

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static float f16_value(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  float v;
  if (e == 0) v = ldexpf((float)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexpf((float)(1024 + m), e - 25);
  return s ? -v : v;
}

/* OCP 8-bit floating point, E4M3 ("fn"): bias 7, subnormals, no infinities,
 * exponent 15 with fraction 7 is NaN. */
static float e4m3_value(uint8_t q) {
  int s = (q >> 7) & 1, e = (q >> 3) & 15, m = q & 7;
  float v;
  if (e == 0) v = ldexpf((float)m, -9);
  else if (e == 15 && m == 7) v = NAN;
  else v = ldexpf((float)(8 + m), e - 10);
  return s ? -v : v;
}

/* 4-bit floating point E2M1 (the element type of NVFP4): sign bit 3, exponent bits 2..1 (bias 1),
 * one fraction bit; exponent 0 is subnormal (0 or 0.5); no infinities or NaN. */
static float e2m1_value(uint8_t q) {
  int s = (q >> 3) & 1, e = (q >> 1) & 3, m = q & 1;
  float v = e == 0 ? 0.5f * (float)m : ldexpf((float)(2 + m), e - 2);
  return s ? -v : v;
}

void orc_init(void) {
  if (tables_ready) return;
  for (int i = 0; i < 65536; ++i) F16_TABLE[i] = f16_value((uint16_t)i);
  for (int i = 0; i < 256; ++i) E4M3_TABLE[i] = e4m3_value((uint8_t)i);
  for (int i = 0; i < 16; ++i) E2M1_TABLE[i] = e2m1_value((uint8_t)i);
  tables_ready = 1;
}

const float* orc_e4m3_table(void) { orc_init(); return E4M3_TABLE; }
const float* orc_e2m1_table(void) { orc_init(); return E2M1_TABLE; }

static inline float bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static inline float load_elem(const void* base, size_t i, int dt) {
  switch (dt) {
    case ORC_F16: return F16_TABLE[((const uint16_t*)base)[i]];
    case ORC_BF16: return bf16_value(((const uint16_t*)base)[i]);
    case ORC_E4M3: return E4M3_TABLE[((const uint8_t*)base)[i]];
    default: return ((const float*)base)[i];
  }
}

static inline size_t elem_size(int dt) { return dt == ORC_E4M3 ? 1 : (dt == ORC_F32 ? 4 : 2); }

static void widen_row(const void* base, size_t row, int K, int dt, float* out) {
  const size_t off = row * (size_t)K;
  for (int i = 0; i < K; ++i) out[i] = load_elem(base, off + i, dt);
}

/* fp32 -> binary16, round to nearest even, written from the value (frexp/ldexp). */
uint16_t orc_round_f16(float f) {
  if (isnan(f)) return 0x7E00;
  uint16_t sign = signbit(f) ? 0x8000 : 0;
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  if (isinf(f)) return (uint16_t)(sign | 0x7C00);
  if (a < ldexp(1.0, -14)) {                         /* subnormal: multiples of 2^-24 */
    double q = nearbyint(a * ldexp(1.0, 24));
    return (uint16_t)(sign | (uint16_t)q);           /* q == 1024 is the smallest normal */
  }
  int e;
  double fr = frexp(a, &e);                          /* a = fr * 2^e, fr in [0.5, 1) */
  double q = nearbyint(fr * 2048.0);                 /* 11 significant bits */
  if (q == 2048.0) { q = 1024.0; e += 1; }
  int be = e - 1 + 15;                               /* biased exponent of 1.f * 2^(e-1) */
  if (be >= 31) return (uint16_t)(sign | 0x7C00);
  return (uint16_t)(sign | (uint16_t)(be << 10) | (uint16_t)((int)q - 1024));
}

/* fp32 -> bfloat16, round to nearest even (8 significant bits, fp32 exponent range). */
uint16_t orc_round_bf16(float f) {
  if (isnan(f)) return 0x7FC0;
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  if (isinf(f)) return (uint16_t)(sign | 0x7F80);
  int e;
  double fr = frexp(a, &e);
  double q;
  if (e - 1 < -126) {                                /* fp32 subnormal range: spacing 2^-133 */
    q = nearbyint(a * ldexp(1.0, 133));
    return (uint16_t)(sign | (uint16_t)q);
  }
  q = nearbyint(fr * 256.0);
  if (q == 256.0) { q = 128.0; e += 1; }
  int be = e - 1 + 127;
  if (be >= 255) return (uint16_t)(sign | 0x7F80);
  return (uint16_t)(sign | (uint16_t)(be << 7) | (uint16_t)((int)q - 128));
}

static inline uint16_t round_kv(float f, int dt) { return dt == ORC_BF16 ? orc_round_bf16(f) : orc_round_f16(f); }
static inline float kv_value(uint16_t b, int dt) { return dt == ORC_BF16 ? bf16_value(b) : F16_TABLE[b]; }

/* ------------------------------------------------------------------ arithmetic */

/* exp of the contract: Cody & Waite argument reduction (Cody, W. J. & Waite, W.,
 * "Software Manual for the Elementary Functions", 1980) with ln 2 split into a
 * 15-bit head (so n*LN2_HI is exact for |n| < 256) and a tail; Taylor series of
 * e^r to degree 7 (coefficients 1/k! rounded to fp32) by Horner's rule with fma;
 * the result scaled by 2^n with one fp32 multiply. */
float orc_exp_c(float x) {
  const float LOG2E = 1.44269502162933349609375f; /* fp32(1/ln 2) */
  const float LN2_HI = 0.693145751953125f;        /* ln 2 to 15 bits */
  const float LN2_LO = 1.428606765330187e-06f;    /* fp32(ln 2 - LN2_HI) */
  if (isnan(x)) return x;
  if (x <= -87.0f) return 0.0f;
  if (x >= 88.0f) return INFINITY;
  float n = nearbyintf(x * LOG2E);
  float r = fmaf(-n, LN2_HI, x);
  r = fmaf(-n, LN2_LO, r);
  float p = 1.98412701138295233249664306640625e-4f; /* 1/7! */
  p = fmaf(p, r, 1.38888892251998186111450195312e-3f); /* 1/6! */
  p = fmaf(p, r, 8.33333376795053482055664062500e-3f); /* 1/5! */
  p = fmaf(p, r, 4.16666679084300994873046875000e-2f); /* 1/4! */
  p = fmaf(p, r, 1.66666671633720397949218750000e-1f); /* 1/3! */
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  uint32_t bits = (uint32_t)((int)n + 127) << 23;
  float scale;
  memcpy(&scale, &bits, 4);
  return p * scale;
}

/* Contract dot product (see file header). */
float orc_dot_exact(const float* w, const float* x, int K, int VW) {
  float a[32];
  for (int l = 0; l < 32; ++l) a[l] = 0.0f;
  const int nv = K / VW;
  for (int base = 0; base < nv; base += 32) {
    for (int e = 0; e < VW; ++e) {
      for (int l = 0; l < 32; ++l) {
        const int v = base + l;
        if (v < nv) a[l] = fmaf(w[v * VW + e], x[v * VW + e], a[l]);
      }
    }
  }
  for (int off = 16; off >= 1; off >>= 1)
    for (int i = 0; i < off; ++i) a[i] = a[i] + a[i + off];
  return a[0];
}

/* Textbook dot product: one running fp32 sum in index order. */
float orc_dot_plain(const float* w, const float* x, int K) {
  float s = 0.0f;
  for (int i = 0; i < K; ++i) s = s + w[i] * x[i];
  return s;
}

static inline float dotm(const float* w, const float* x, int K, int VW, int mode) {
  return mode == ORC_EXACT ? orc_dot_exact(w, x, K, VW) : orc_dot_plain(w, x, K);
}

static inline float expm(float x, int mode) { return mode == ORC_EXACT ? orc_exp_c(x) : expf(x); }

/* One nvfp4 row (codes: K/2 bytes, bscale: K/16 e4m3 codes) dotted with x, before the row scale. */
static float dot_nvfp4(const uint8_t* codes, const uint8_t* bscale, const float* x, int K, int mode) {
  if (mode == ORC_EXACT) {
    float a[32];
    for (int l = 0; l < 32; ++l) a[l] = 0.0f;
    const int nv = K / 8;
    for (int v = 0; v < nv; ++v) {
      float t = 0.0f;
      for (int e = 0; e < 8; ++e) {
        const int j = v * 8 + e;
        const uint8_t q = (codes[j >> 1] >> ((j & 1) * 4)) & 15;
        t = fmaf(E2M1_TABLE[q], x[j], t);
      }
      a[v % 32] = fmaf(E4M3_TABLE[bscale[v >> 1]], t, a[v % 32]);
    }
    for (int off = 16; off >= 1; off >>= 1)
      for (int i = 0; i < off; ++i) a[i] = a[i] + a[i + off];
    return a[0];
  }
  float s = 0.0f;
  for (int j = 0; j < K; ++j) {
    const uint8_t q = (codes[j >> 1] >> ((j & 1) * 4)) & 15;
    s = s + (E4M3_TABLE[bscale[j >> 4]] * E2M1_TABLE[q]) * x[j];
  }
  return s;
}

/* Exported for the pins: dot_nvfp4 of one row. */
float orc_dot_nvfp4(const uint8_t* codes, const uint8_t* bscale, const float* x, int K, int mode) {
  orc_init();
  return dot_nvfp4(codes, bscale, x, K, mode);
}

/* y[r] = scale[r] * (W[r,:] . x) for r < rows (scale NULL -> 1, applied after the dot); nvfp4
 * matrices (dt ORC_NVFP4) also take their block scales. */
static int gemv(const void* Wt, int dt, int rows, int K, const float* x, const float* scale, const uint8_t* bscale,
                float* y, int mode) {
  const int VW = 8;
  if (dt == ORC_NVFP4) {
    if (!bscale || !scale || K % 16) return ORC_EINVAL;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r)
      y[r] = scale[r] * dot_nvfp4((const uint8_t*)Wt + (size_t)r * (K / 2), bscale + (size_t)r * (K / 16), x, K, mode);
    return ORC_OK;
  }
  int fail = 0;
#pragma omp parallel reduction(| : fail)
  {
    float* buf = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
    for (int r = 0; r < rows; ++r) {
      if (!buf) { fail = 1; continue; }
      widen_row(Wt, (size_t)r, K, dt, buf);
      float v = dotm(buf, x, K, VW, mode);
      y[r] = scale ? scale[r] * v : v;
    }
    free(buf);
  }
  return fail ? ORC_ENOMEM : ORC_OK;
}

/* Exported for the pins: gemv of one matrix. */
int orc_gemv(const void* Wt, int dt, int rows, int K, const float* x, const float* scale, const uint8_t* bscale,
             float* y, int mode) {
  orc_init();
  return gemv(Wt, dt, rows, K, x, scale, bscale, y, mode);
}

/* RMSNorm: xn_i = x_i * (mean(x^2) + eps)^(-1/2) * g_i. */
void orc_rmsnorm(const float* x, const void* g, int gdt, int d, float eps, int mode, float* out) {
  float ss = mode == ORC_EXACT ? orc_dot_exact(x, x, d, 8) : orc_dot_plain(x, x, d);
  float mean = ss / (float)d;
  float r = 1.0f / sqrtf(mean + eps);
  for (int i = 0; i < d; ++i) out[i] = (x[i] * r) * load_elem(g, (size_t)i, gdt);
}

/* RoPE (rotate-half pairs (i, i + hd/2)), inv_freq_i = theta^(-2i/hd), angle = p * inv_freq_i,
 * all in double, cos and sin rounded to fp32. */
void orc_rope_row(float theta, int hd, int pos, float* cs, float* sn) {
  for (int i = 0; i < hd / 2; ++i) {
    double ex = (double)(2 * i) / (double)hd;
    double inv = pow((double)theta, -ex);
    double ang = (double)pos * inv;
    cs[i] = (float)cos(ang);
    sn[i] = (float)sin(ang);
  }
}

static void rope_apply(float* y, int hd, const float* cs, const float* sn, int mode) {
  const int h2 = hd / 2;
  for (int i = 0; i < h2; ++i) {
    float a = y[i], b = y[i + h2], c = cs[i], s = sn[i];
    if (mode == ORC_EXACT) {
      y[i] = fmaf(a, c, -(b * s));
      y[i + h2] = fmaf(b, c, a * s);
    } else {
      y[i] = a * c - b * s;
      y[i + h2] = b * c + a * s;
    }
  }
}

/* RoPE of one head vector y[hd] at position pos (exported for the oracle's own checks). */
void orc_rope(float* y, int hd, int pos, float theta, int mode) {
  float cs[512], sn[512];
  orc_rope_row(theta, hd, pos, cs, sn);
  rope_apply(y, hd, cs, sn, mode);
}

/* Attention of one query head over cached positions 0..n-1 (K, V rows of hd stored
 * values at stride hd).  Exact mode follows the 32-position block contract. */
void orc_attention_head(const float* q, const void* Kc, const void* Vc, int kvdt, int n, int hd, float scale,
                        int mode, float* out) {
  float* s = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  float* kf = (float*)malloc(sizeof(float) * (size_t)hd);
  const uint16_t* K = (const uint16_t*)Kc;
  const uint16_t* V = (const uint16_t*)Vc;
  for (int j = 0; j < n; ++j) {
    for (int d = 0; d < hd; ++d) kf[d] = kv_value(K[(size_t)j * hd + d], kvdt);
    s[j] = dotm(kf, q, hd, 8, mode) * scale;
  }
  if (mode == ORC_EXACT) {
    const int B = 32, nb = (n + B - 1) / B;
    float* m = (float*)malloc(sizeof(float) * (size_t)nb);
    float* l = (float*)malloc(sizeof(float) * (size_t)nb);
    float* o = (float*)malloc(sizeof(float) * (size_t)nb * hd);
    for (int b = 0; b < nb; ++b) {
      const int j0 = b * B, j1 = (j0 + B < n) ? j0 + B : n;
      float mb = s[j0];
      for (int j = j0 + 1; j < j1; ++j) mb = s[j] > mb ? s[j] : mb;
      float lb = 0.0f;
      float* ob = o + (size_t)b * hd;
      for (int d = 0; d < hd; ++d) ob[d] = 0.0f;
      for (int j = j0; j < j1; ++j) {
        float e = orc_exp_c(s[j] - mb);
        lb = lb + e;
        for (int d = 0; d < hd; ++d) ob[d] = fmaf(e, kv_value(V[(size_t)j * hd + d], kvdt), ob[d]);
      }
      m[b] = mb;
      l[b] = lb;
    }
    float M = m[0];
    for (int b = 1; b < nb; ++b) M = m[b] > M ? m[b] : M;
    float L = 0.0f;
    for (int d = 0; d < hd; ++d) out[d] = 0.0f;
    for (int b = 0; b < nb; ++b) {
      float w = orc_exp_c(m[b] - M);
      L = fmaf(w, l[b], L);
      for (int d = 0; d < hd; ++d) out[d] = fmaf(w, o[(size_t)b * hd + d], out[d]);
    }
    for (int d = 0; d < hd; ++d) out[d] = out[d] / L;
    free(m); free(l); free(o);
  } else {
    float M = s[0];
    for (int j = 1; j < n; ++j) M = s[j] > M ? s[j] : M;
    float Z = 0.0f;
    for (int j = 0; j < n; ++j) { s[j] = expf(s[j] - M); Z = Z + s[j]; }
    for (int d = 0; d < hd; ++d) out[d] = 0.0f;
    for (int j = 0; j < n; ++j) {
      float a = s[j] / Z;
      for (int d = 0; d < hd; ++d) out[d] = out[d] + a * kv_value(V[(size_t)j * hd + d], kvdt);
    }
  }
  free(s); free(kf);
}

static inline float silu_mul(float g, float u, int mode) {
  float t = expm(-g, mode);
  float den = 1.0f + t;
  return (g / den) * u;
}

/* Softmax over E router logits, top-k (ties to the lower index), gates renormalised
 * over the chosen experts.  sel/gate receive k entries in choice order; P (optional) E probs. */
void orc_route(const float* r, int E, int k, int mode, int32_t* sel, float* gate, float* P_out) {
  float P[1024];
  float M = r[0];
  for (int e = 1; e < E; ++e) M = r[e] > M ? r[e] : M;
  float Z = 0.0f;
  for (int e = 0; e < E; ++e) { P[e] = expm(r[e] - M, mode); Z = Z + P[e]; }
  for (int e = 0; e < E; ++e) P[e] = P[e] / Z;
  unsigned char used[1024];
  memset(used, 0, sizeof(used));
  float Zs = 0.0f;
  for (int i = 0; i < k; ++i) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!used[e] && (best < 0 || P[e] > P[best])) best = e;
    used[best] = 1;
    sel[i] = best;
    Zs = Zs + P[best];
  }
  for (int i = 0; i < k; ++i) gate[i] = P[sel[i]] / Zs;
  if (P_out) memcpy(P_out, P, sizeof(float) * (size_t)E);
}

/* Greedy: first index of the maximum logit. */
int32_t orc_argmax(const float* l, int V) {
  int32_t best = 0;
  for (int i = 1; i < V; ++i) if (l[i] > l[best]) best = i;
  return best;
}

/* Temperature sampling by inverse CDF with one uniform u in [0, 1). */
int32_t orc_sample(const float* l, int V, float T, float u, int mode) {
  float M = l[0];
  for (int i = 1; i < V; ++i) M = l[i] > M ? l[i] : M;
  float* e = (float*)malloc(sizeof(float) * (size_t)V);
  int32_t tok = -1, last_pos = 0;
  for (int i = 0; i < V; ++i) {
    e[i] = expm((l[i] - M) / T, mode);
    if (e[i] > 0.0f) last_pos = i;
  }
  if (mode == ORC_EXACT) {
    const int B = 256, nb = (V + B - 1) / B;
    float* S = (float*)malloc(sizeof(float) * (size_t)nb);
    float ones[256];
    for (int i = 0; i < B; ++i) ones[i] = 1.0f;
    for (int b = 0; b < nb; ++b) {
      const int i0 = b * B, n = (i0 + B <= V) ? B : V - i0;
      S[b] = orc_dot_exact(e + i0, ones, n, 8);
    }
    float Z = 0.0f;
    for (int b = 0; b < nb; ++b) Z = Z + S[b];
    const float tau = u * Z;
    float P = 0.0f;
    int bstar = -1;
    for (int b = 0; b < nb; ++b) {
      float Pn = P + S[b];
      if (Pn > tau) { bstar = b; break; }
      P = Pn;
    }
    if (bstar < 0) {
      tok = last_pos;
    } else {
      const int i0 = bstar * B, i1 = (i0 + B <= V) ? i0 + B : V;
      float run = P;
      int lastb = i0;
      for (int i = i0; i < i1; ++i) {
        if (e[i] > 0.0f) lastb = i;
        run = run + e[i];
        if (run > tau) { tok = i; break; }
      }
      if (tok < 0) tok = lastb;
    }
    free(S);
  } else {
    float Z = 0.0f;
    for (int i = 0; i < V; ++i) Z = Z + e[i];
    const float tau = u * Z;
    float run = 0.0f;
    for (int i = 0; i < V; ++i) {
      run = run + e[i];
      if (run > tau) { tok = i; break; }
    }
    if (tok < 0) tok = last_pos;
  }
  free(e);
  return tok;
}

/* ------------------------------------------------------------------ one decode step */

/* One decode step: the token `token` at position `pos` (its K/V row written to the
 * cache before attention), returning the V logits and the next token.
 *   kc, vc        host KV cache, [n_layers][n_kv_heads][max_ctx][head_dim] of the KV dtype
 *   temperature   0 -> greedy argmax, else inverse-CDF sampling with uniform u
 *   force         optional [n_layers][top_k] expert ids to use instead of the router's choice
 *   sel_out/gate_out  optional [n_layers][top_k]: the router's own choice and gates
 *   trace         optional [n_layers + 1][d_model]: the residual entering each layer and the
 *                 final residual
 */
int orc_step(const orc_config* c, const orc_weights* W, void* kc, void* vc, int32_t pos, int32_t token,
             int32_t mode, float temperature, float u, const int32_t* force, float* logits, int32_t* next,
             int32_t* sel_out, float* gate_out, float* trace) {
  orc_init();
  if (!c || !W || !kc || !vc || !logits) return ORC_EINVAL;
  const int L = c->n_layers, d = c->d_model, hq = c->n_heads, hkv = c->n_kv_heads, hd = c->head_dim;
  const int V = c->vocab, wdt = c->weight_dtype, kvdt = c->kv_dtype;
  /* with e4m3 or nvfp4 layer matrices the embedding, LM head and norm gains keep a 16-bit type */
  const int edt = (wdt == ORC_E4M3 || wdt == ORC_NVFP4) ? c->embed_dtype : wdt;
  if (pos < 0 || pos >= c->max_ctx) return ORC_ECTX;
  if (token < 0 || token >= V) return ORC_EINVAL;
  const int moe = c->n_experts > 0;
  const int ff = moe ? c->d_expert : c->d_ff;
  const int wide = (ff > d ? ff : d) > hq * hd ? (ff > d ? ff : d) : hq * hd;
  float* x = (float*)calloc((size_t)d, sizeof(float));
  float* xn = (float*)calloc((size_t)d, sizeof(float));
  float* q = (float*)calloc((size_t)hq * hd, sizeof(float));
  float* k = (float*)calloc((size_t)hkv * hd, sizeof(float));
  float* v = (float*)calloc((size_t)hkv * hd, sizeof(float));
  float* att = (float*)calloc((size_t)hq * hd, sizeof(float));
  float* y = (float*)calloc((size_t)wide, sizeof(float));
  float* g = (float*)calloc((size_t)ff, sizeof(float));
  float* uu = (float*)calloc((size_t)ff, sizeof(float));
  float* acc = (float*)calloc((size_t)d, sizeof(float));
  float* cs = (float*)calloc((size_t)hd, sizeof(float));
  float* sn = (float*)calloc((size_t)hd, sizeof(float));
  float* r = (float*)calloc((size_t)(moe ? c->n_experts : 1), sizeof(float));
  int rc = ORC_OK;
  if (!x || !xn || !q || !k || !v || !att || !y || !g || !uu || !acc || !cs || !sn || !r) { rc = ORC_ENOMEM; goto done; }

  widen_row(W->tok_emb, (size_t)token, d, edt, x);   /* embedding: exact widening */
  orc_rope_row(c->rope_theta, hd, pos, cs, sn);
  const float scale = (float)(1.0 / sqrt((double)hd));

  for (int l = 0; l < L; ++l) {
    const orc_layer* lw = &W->layers[l];
    if (trace) memcpy(trace + (size_t)l * d, x, sizeof(float) * (size_t)d);
    /* attention block */
    orc_rmsnorm(x, lw->attn_norm, edt, d, c->rms_eps, mode, xn);
    if ((rc = gemv(lw->wq, wdt, hq * hd, d, xn, lw->wq_scale, lw->wq_bscale, q, mode))) goto done;
    if ((rc = gemv(lw->wk, wdt, hkv * hd, d, xn, lw->wk_scale, lw->wk_bscale, k, mode))) goto done;
    if ((rc = gemv(lw->wv, wdt, hkv * hd, d, xn, lw->wv_scale, lw->wv_bscale, v, mode))) goto done;
    for (int h = 0; h < hq; ++h) rope_apply(q + (size_t)h * hd, hd, cs, sn, mode);
    for (int h = 0; h < hkv; ++h) rope_apply(k + (size_t)h * hd, hd, cs, sn, mode);
    for (int h = 0; h < hkv; ++h) {
      const size_t row = (((size_t)l * hkv + h) * (size_t)c->max_ctx + (size_t)pos) * hd;
      for (int i = 0; i < hd; ++i) {
        ((uint16_t*)kc)[row + i] = round_kv(k[(size_t)h * hd + i], kvdt);
        ((uint16_t*)vc)[row + i] = round_kv(v[(size_t)h * hd + i], kvdt);
      }
    }
#pragma omp parallel for schedule(static)
    for (int h = 0; h < hq; ++h) {
      const int grp = (int)(((long long)h * hkv) / hq);
      const size_t base = ((size_t)l * hkv + grp) * (size_t)c->max_ctx * hd;
      orc_attention_head(q + (size_t)h * hd, (const uint16_t*)kc + base, (const uint16_t*)vc + base, kvdt, pos + 1,
                         hd, scale, mode, att + (size_t)h * hd);
    }
    if ((rc = gemv(lw->wo, wdt, d, hq * hd, att, lw->wo_scale, lw->wo_bscale, y, mode))) goto done;
    for (int i = 0; i < d; ++i) x[i] = x[i] + y[i];
    /* feed-forward block */
    orc_rmsnorm(x, lw->ffn_norm, edt, d, c->rms_eps, mode, xn);
    if (!moe) {
      if ((rc = gemv(lw->w_gate, wdt, ff, d, xn, lw->w_gate_scale, lw->w_gate_bscale, g, mode))) goto done;
      if ((rc = gemv(lw->w_up, wdt, ff, d, xn, lw->w_up_scale, lw->w_up_bscale, uu, mode))) goto done;
      for (int i = 0; i < ff; ++i) g[i] = silu_mul(g[i], uu[i], mode);
      if ((rc = gemv(lw->w_down, wdt, d, ff, g, lw->w_down_scale, lw->w_down_bscale, y, mode))) goto done;
      for (int i = 0; i < d; ++i) x[i] = x[i] + y[i];
    } else {
      const int E = c->n_experts, K = c->top_k;
      int32_t sel[64];
      float gate[64];
      if ((rc = gemv(lw->router, c->router_dtype, E, d, xn, NULL, NULL, r, mode))) goto done;
      orc_route(r, E, K, mode, sel, gate, NULL);
      if (sel_out) memcpy(sel_out + (size_t)l * K, sel, sizeof(int32_t) * (size_t)K);
      if (gate_out) memcpy(gate_out + (size_t)l * K, gate, sizeof(float) * (size_t)K);
      if (force) {
        /* forced experts keep the router's gate of that expert, renormalised over the forced set */
        float P[1024];
        int32_t s2[64];
        float g2[64];
        orc_route(r, E, E, mode, s2, g2, P);
        float Zs = 0.0f;
        for (int i = 0; i < K; ++i) { sel[i] = force[(size_t)l * K + i]; Zs = Zs + P[sel[i]]; }
        for (int i = 0; i < K; ++i) gate[i] = P[sel[i]] / Zs;
      }
      const int fe = c->d_expert;
      const size_t gu_sz = (size_t)fe * d, dn_sz = (size_t)d * fe;
      for (int i = 0; i < d; ++i) acc[i] = 0.0f;
      for (int s = 0; s < K; ++s) {
        const int e = sel[s];
        const uint8_t* Qg = (const uint8_t*)lw->e_gate + (size_t)e * gu_sz;
        const uint8_t* Qu = (const uint8_t*)lw->e_up + (size_t)e * gu_sz;
        const uint8_t* Qd = (const uint8_t*)lw->e_down + (size_t)e * dn_sz;
        if ((rc = gemv(Qg, c->expert_dtype, fe, d, xn, lw->e_gate_scale + (size_t)e * fe, NULL, g, mode))) goto done;
        if ((rc = gemv(Qu, c->expert_dtype, fe, d, xn, lw->e_up_scale + (size_t)e * fe, NULL, uu, mode))) goto done;
        for (int i = 0; i < fe; ++i) g[i] = silu_mul(g[i], uu[i], mode);
        if ((rc = gemv(Qd, c->expert_dtype, d, fe, g, lw->e_down_scale + (size_t)e * d, NULL, y, mode))) goto done;
        if (mode == ORC_EXACT)
          for (int i = 0; i < d; ++i) acc[i] = fmaf(gate[s], y[i], acc[i]);
        else
          for (int i = 0; i < d; ++i) acc[i] = acc[i] + gate[s] * y[i];
      }
      for (int i = 0; i < d; ++i) x[i] = x[i] + acc[i];
    }
  }
  if (trace) memcpy(trace + (size_t)L * d, x, sizeof(float) * (size_t)d);
  orc_rmsnorm(x, W->final_norm, edt, d, c->rms_eps, mode, xn);
  {
    const void* head = c->tied_embeddings ? W->tok_emb : W->lm_head;
    if ((rc = gemv(head, edt, V, d, xn, NULL, NULL, logits, mode))) goto done;
  }
  if (next) *next = temperature > 0.0f ? orc_sample(logits, V, temperature, u, mode) : orc_argmax(logits, V);
done:
  free(x); free(xn); free(q); free(k); free(v); free(att); free(y); free(g); free(uu); free(acc);
  free(cs); free(sn); free(r);
  return rc;
}

/*
 * oracle.c — plain, slow, single-threaded CPU oracle of the verify-step hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library. It shares no code, header, table or constant
 * generator with the CUDA library, and it includes nothing from it.
 *
 * Built with -ffp-contract=off: every floating-point operation below is the one written.
 * fp64 everywhere, except where the workload fixes fp32 (the block-score definition).
 *
 * What each function follows (pages about the DeepSeek V4.1 Flash Q4 fork with a native
 * multi-token drafter, "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP"):
 *   orc_router        paragraph "Decode" (the 384-expert router); sigmoid scores, top-k
 *                     by (score desc, index asc), weights renormalised over the k chosen.
 *   orc_moe_forward   paragraphs "Decode" and "DSpark" (shared expert gate+up+SwiGLU,
 *                     routed experts on Q4 weights, BF16 rounding inside the producer):
 *                     dequantise, then fp64 matmul; bf16 rounding of h and of y only.
 *   orc_select        paragraph "Decode at depth": score admitted blocks only,
 *                     compact the admitted index per row, take the top 512 by
 *                     (score desc, index asc); canonical fp32 score order.
 *   orc_q8_project    paragraph "DSpark" (paired Q8 projections shared by the verify
 *                     rows): dequantise, then fp64 products; one bf16 rounding.
 *   orc_verify_greedy / orc_verify_sample
 *                     paragraph "DSpark" (a 6-row verify per decode step; identical
 *                     output under greedy decode; exact speculative sampling at
 *                     temperature > 0): accepted drafts, then one target token.
 *   orc_sparse_attention
 *                     paragraph "Decode at depth" (attention reads the 512 blocks the
 *                     selection picks): softmax attention of each query head over the
 *                     tokens of the row's selected blocks, fp64, one bf16 rounding.
 * Readings where the pages are silent are stated beside the code that takes them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- number formats ---- */

/* bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 31;
  int fr = h & 1023;
  double v;
  if (ex == 0)
    v = ldexp((double)fr, -24);                 /* zero / subnormal: fr * 2^-24 */
  else if (ex == 31)
    v = fr ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + fr), ex - 25);    /* (1 + fr/1024) * 2^(ex-15)    */
  return sign ? -v : v;
}

/* Round a double to the nearest bf16 (8 significant bits, exponent range of binary32),
 * ties to even; overflow gives infinity. Rounds once, straight from the double. */
uint16_t orc_bf16_rne(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1)                  */
  int qexp = e - 8;             /* quantum of an 8-significant-bit value       */
  if (qexp < -133) qexp = -133; /* below 2^-126 the quantum is the subnormal 2^-133 */
  double r = nearbyint(ldexp(a, -qexp)); /* default rounding mode: nearest, ties even */
  double val = ldexp(r, qexp);
  const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (val > bf16_max) return (uint16_t)(sign | 0x7F80);
  float f = (float)val;         /* exact: val has at most 8 significant bits   */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

/* ------------------------------------------------------------------- Q4 weights ----- */

/* Value k of row `row` of a Q4 matrix with K columns (format: blocks of 32 along K,
 * 16 bytes per block, byte j = value 2j in the low nibble | value 2j+1 in the high
 * nibble, nibble = q + 8; one fp16 scale per block). Returns scale * q in fp64. */
double orc_q4_value(const uint8_t* qs, const uint16_t* sc, int64_t K, int64_t row, int64_t k) {
  uint8_t byte = qs[row * (K / 2) + k / 2];
  int nib = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
  int q = nib - 8;
  double s = orc_f16_to_f64(sc[row * (K / 32) + k / 32]);
  return s * (double)q;
}

/* ------------------------------------------------------------------- Q8 weights ----- */

/* Paragraph "DSpark": the verify rows share one weight stream through paired Q8
 * projections. Reading: blocks of 32 signed 8-bit values (two's complement) along K with
 * one fp16 scale per block, value = scale * q; planar, qs int8 [rows][K] and sc fp16
 * [rows][K/32]. Returns value k of row `row` in fp64. */
double orc_q8_value(const int8_t* qs, const uint16_t* sc, int64_t K, int64_t row, int64_t k) {
  double s = orc_f16_to_f64(sc[row * (K / 32) + k / 32]);
  return s * (double)qs[row * K + k];
}

/* The R verify rows through one Q8 projection: y[r][i] = sum_k W[i][k] * x[r][k] in fp64
 * (x bf16 [R][K], W the dequantised [rows][K]), and, when ybf is non-NULL, y rounded once
 * to bf16 (round to nearest, ties to even). */
void orc_q8_project(const int8_t* qs, const uint16_t* sc, int64_t rows, int64_t K,
                    const uint16_t* x, int32_t R, double* y, uint16_t* ybf) {
  double* xr = (double*)malloc(sizeof(double) * (size_t)K);
  for (int32_t r = 0; r < R; ++r) {
    for (int64_t k = 0; k < K; ++k) xr[k] = orc_bf16_to_f64(x[(int64_t)r * K + k]);
    for (int64_t i = 0; i < rows; ++i) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += orc_q8_value(qs, sc, K, i, k) * xr[k];
      y[(int64_t)r * rows + i] = acc;
      if (ybf) ybf[(int64_t)r * rows + i] = orc_bf16_rne(acc);
    }
  }
  free(xr);
}

/* y[i] = sum_k W[i][k] * x[k] for the dequantised Q4 matrix W [rows][K], fp64.
 * If a is non-NULL, a[i] = sum_k |W[i][k] * x[k]| (the scale of the terms, used to bound
 * the rounding error of a lower-precision evaluation of the same sum). */
static void q4_matvec_abs(const uint8_t* qs, const uint16_t* sc, int64_t rows, int64_t K,
                          const double* x, double* y, double* a) {
  for (int64_t i = 0; i < rows; ++i) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double t = orc_q4_value(qs, sc, K, i, k) * x[k];
      acc += t;
      aacc += fabs(t);
    }
    y[i] = acc;
    if (a) a[i] = aacc;
  }
}

static void q4_matvec(const uint8_t* qs, const uint16_t* sc, int64_t rows, int64_t K,
                      const double* x, double* y) {
  q4_matvec_abs(qs, sc, rows, K, x, y, NULL);
}

/* ----------------------------------------------------------------------- router ----- */

typedef struct { double s; int32_t e; } scored_expert;

/* Larger score first; equal scores: lower expert id first. */
static int cmp_scored_expert(const void* a, const void* b) {
  const scored_expert* p = (const scored_expert*)a;
  const scored_expert* q = (const scored_expert*)b;
  if (p->s > q->s) return -1;
  if (p->s < q->s) return 1;
  return (p->e > q->e) - (p->e < q->e);
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Router of one layer for R rows: z = x . Wr^T (fp64), s = sigmoid(z); the k experts
 * with the largest s (ties: lower id) in rank order; w_j = s_j / (sum of the k chosen s).
 * No bias, grouping or scaling factor (reading: plain sigmoid top-k, renormalised).
 *   x [R][H] bf16, wr [E][H] bf16 -> idx [R][k], w [R][k], s [R][E] (s may be NULL). */
void orc_router(const uint16_t* x, int32_t R, int32_t H, const uint16_t* wr, int32_t E,
                int32_t k, int32_t* idx, double* w, double* s_out) {
  scored_expert* se = (scored_expert*)malloc(sizeof(scored_expert) * (size_t)E);
  for (int32_t r = 0; r < R; ++r) {
    for (int32_t e = 0; e < E; ++e) {
      double z = 0.0;
      for (int32_t i = 0; i < H; ++i)
        z += orc_bf16_to_f64(x[(int64_t)r * H + i]) * orc_bf16_to_f64(wr[(int64_t)e * H + i]);
      se[e].s = sigmoid(z);
      se[e].e = e;
      if (s_out) s_out[(int64_t)r * E + e] = se[e].s;
    }
    qsort(se, (size_t)E, sizeof(scored_expert), cmp_scored_expert);
    double sum = 0.0;
    for (int32_t j = 0; j < k; ++j) sum += se[j].s;
    for (int32_t j = 0; j < k; ++j) {
      idx[(int64_t)r * k + j] = se[j].e;
      w[(int64_t)r * k + j] = se[j].s / sum;
    }
  }
  free(se);
}

/* ----------------------------------------------------------------------- MoE layer -- */

/* The oracle's own description of a layer (independent of the library's struct).
 * Routed arrays are expert-major stacks; the shared expert is separate. */
typedef struct {
  int32_t H, E, I, k;
  const uint16_t* router_w;                 /* bf16 [E][H]          */
  const uint8_t* gate_qs; const uint16_t* gate_sc;   /* [E][I][H]   */
  const uint8_t* up_qs;   const uint16_t* up_sc;     /* [E][I][H]   */
  const uint8_t* down_qs; const uint16_t* down_sc;   /* [E][H][I]   */
  const uint8_t* sg_qs;   const uint16_t* sg_sc;     /* shared [I][H] */
  const uint8_t* su_qs;   const uint16_t* su_sc;     /* shared [I][H] */
  const uint8_t* sd_qs;   const uint16_t* sd_sc;     /* shared [H][I] */
} orc_moe_layer;

/* One expert on one row: h = bf16(silu(Wg x) * (Wu x)), o = Wd h (fp64).
 * aux (may be NULL): per intermediate element i, {g, u, sum|Wg x terms|, sum|Wu x terms|}. */
static void expert_forward(const uint8_t* gq, const uint16_t* gs, const uint8_t* uq,
                           const uint16_t* us, const uint8_t* dq, const uint16_t* ds,
                           int32_t H, int32_t I, const double* x, double* o,
                           double* g, double* u, double* h, double* ag, double* au,
                           double* aux) {
  q4_matvec_abs(gq, gs, I, H, x, g, ag);
  q4_matvec_abs(uq, us, I, H, x, u, au);
  for (int32_t i = 0; i < I; ++i) {
    double silu = g[i] / (1.0 + exp(-g[i]));   /* silu(g) = g * sigmoid(g) */
    h[i] = orc_bf16_to_f64(orc_bf16_rne(silu * u[i]));  /* rounding point 1 */
    if (aux) {
      aux[4 * i + 0] = g[i];
      aux[4 * i + 1] = u[i];
      aux[4 * i + 2] = ag[i];
      aux[4 * i + 3] = au[i];
    }
  }
  q4_matvec(dq, ds, H, I, h, o);
}

/* Whole MoE layer for R rows (each row independently; R only batches the calls).
 *   y [R][H] bf16; idx [R][k]; w [R][k]; s [R][E] (may be NULL).
 * If idx_in is non-NULL, its experts (rank order) are used instead of the oracle's own
 * top-k, with weights renormalised from the oracle's scores of those experts; this is
 * how a permitted near-tie swap on the GPU side is re-checked.
 * h_out (may be NULL) receives the rounded h as bf16 [R][1+k][I], slot 0 = shared. */
void orc_moe_forward(const orc_moe_layer* L, const uint16_t* x, int32_t R,
                     const int32_t* idx_in, uint16_t* y, int32_t* idx, double* w,
                     double* s, uint16_t* h_out, double* aux) {
  const int32_t H = L->H, E = L->E, I = L->I, k = L->k;
  double* s_all = (double*)malloc(sizeof(double) * (size_t)R * E);
  orc_router(x, R, H, L->router_w, E, k, idx, w, s_all);
  if (idx_in) {
    for (int32_t r = 0; r < R; ++r) {
      double sum = 0.0;
      for (int32_t j = 0; j < k; ++j) sum += s_all[(int64_t)r * E + idx_in[(int64_t)r * k + j]];
      for (int32_t j = 0; j < k; ++j) {
        int32_t e = idx_in[(int64_t)r * k + j];
        idx[(int64_t)r * k + j] = e;
        w[(int64_t)r * k + j] = s_all[(int64_t)r * E + e] / sum;
      }
    }
  }
  if (s) memcpy(s, s_all, sizeof(double) * (size_t)R * E);

  double* xr = (double*)malloc(sizeof(double) * (size_t)H);
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* ag = (double*)malloc(sizeof(double) * (size_t)I);
  double* au = (double*)malloc(sizeof(double) * (size_t)I);
  const int64_t gu_stride = (int64_t)I * H / 2, gu_sstride = (int64_t)I * H / 32;
  const int64_t d_stride = (int64_t)H * I / 2, d_sstride = (int64_t)H * I / 32;

  for (int32_t r = 0; r < R; ++r) {
    for (int32_t i = 0; i < H; ++i) xr[i] = orc_bf16_to_f64(x[(int64_t)r * H + i]);
    /* shared expert, weight 1 */
    expert_forward(L->sg_qs, L->sg_sc, L->su_qs, L->su_sc, L->sd_qs, L->sd_sc, H, I, xr,
                   acc, g, u, h, ag, au, aux ? aux + ((int64_t)r * (1 + k)) * I * 4 : NULL);
    if (h_out)
      for (int32_t i = 0; i < I; ++i)
        h_out[((int64_t)r * (1 + k) + 0) * I + i] = orc_bf16_rne(h[i]);
    /* routed experts in rank order, weight w_j; no residual, no routed scaling */
    for (int32_t j = 0; j < k; ++j) {
      int64_t e = idx[(int64_t)r * k + j];
      expert_forward(L->gate_qs + e * gu_stride, L->gate_sc + e * gu_sstride,
                     L->up_qs + e * gu_stride, L->up_sc + e * gu_sstride,
                     L->down_qs + e * d_stride, L->down_sc + e * d_sstride, H, I, xr, o,
                     g, u, h, ag, au,
                     aux ? aux + ((int64_t)r * (1 + k) + 1 + j) * I * 4 : NULL);
      if (h_out)
        for (int32_t i = 0; i < I; ++i)
          h_out[((int64_t)r * (1 + k) + 1 + j) * I + i] = orc_bf16_rne(h[i]);
      double wj = w[(int64_t)r * k + j];
      for (int32_t i = 0; i < H; ++i) acc[i] += wj * o[i];
    }
    for (int32_t i = 0; i < H; ++i) y[(int64_t)r * H + i] = orc_bf16_rne(acc[i]); /* point 2 */
  }
  free(xr); free(acc); free(o); free(g); free(u); free(h); free(ag); free(au); free(s_all);
}

/* Down projection and combine from given activations (the second half of the layer):
 *   y[r] = bf16( Wd_shared h[r][0] + sum_j w[r][j] Wd_{idx[r][j]} h[r][1+j] ),  fp64.
 * h_in: bf16 [R][1+k][I]. Used to compare a device's y with the oracle applied to the
 * device's own h, which separates the two bf16 rounding points. */
void orc_moe_down_combine(const orc_moe_layer* L, int32_t R, const int32_t* idx, const double* w,
                          const uint16_t* h_in, uint16_t* y, double* yaux) {
  const int32_t H = L->H, I = L->I, k = L->k;
  const int64_t d_stride = (int64_t)H * I / 2, d_sstride = (int64_t)H * I / 32;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  double* ao = (double*)malloc(sizeof(double) * (size_t)H);
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  double* aacc = (double*)malloc(sizeof(double) * (size_t)H);
  for (int32_t r = 0; r < R; ++r) {
    for (int32_t i = 0; i < I; ++i) h[i] = orc_bf16_to_f64(h_in[((int64_t)r * (1 + k)) * I + i]);
    q4_matvec_abs(L->sd_qs, L->sd_sc, H, I, h, acc, aacc);
    for (int32_t j = 0; j < k; ++j) {
      int64_t e = idx[(int64_t)r * k + j];
      for (int32_t i = 0; i < I; ++i)
        h[i] = orc_bf16_to_f64(h_in[((int64_t)r * (1 + k) + 1 + j) * I + i]);
      q4_matvec_abs(L->down_qs + e * d_stride, L->down_sc + e * d_sstride, H, I, h, o, ao);
      double wj = w[(int64_t)r * k + j];
      for (int32_t i = 0; i < H; ++i) {
        acc[i] += wj * o[i];
        aacc[i] += fabs(wj) * ao[i];
      }
    }
    for (int32_t i = 0; i < H; ++i) {
      y[(int64_t)r * H + i] = orc_bf16_rne(acc[i]);
      if (yaux) {
        yaux[((int64_t)r * H + i) * 2 + 0] = acc[i];   /* y before rounding */
        yaux[((int64_t)r * H + i) * 2 + 1] = aacc[i];  /* scale of its terms */
      }
    }
  }
  free(h); free(o); free(ao); free(acc); free(aacc);
}

/* Elementwise orc_bf16_rne over n doubles. */
void orc_bf16_rne_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------ block select ---- */

/* Canonical fp32 score of one block for one row (reading of the score formula
 * s = sum_h w_h * relu(q_h . k_b) with a fixed rounding order):
 *   d_h = 0.0f; for i ascending: d_h = fmaf(q_h[i], k[i], d_h)
 *   s = +0.0f;  for h ascending: s = fmaf(w_h, d_h > 0 ? d_h : +0.0f, s)
 * q [Hh][D] bf16, key [D] bf16, w [Hh] fp32. */
float orc_block_score(const uint16_t* q, const uint16_t* key, const float* w, int32_t Hh,
                      int32_t D) {
  float s = 0.0f;
  for (int32_t hh = 0; hh < Hh; ++hh) {
    float d = 0.0f;
    for (int32_t i = 0; i < D; ++i)
      d = fmaf((float)orc_bf16_to_f64(q[(int64_t)hh * D + i]), (float)orc_bf16_to_f64(key[i]), d);
    float rl = d > 0.0f ? d : 0.0f;
    s = fmaf(w[hh], rl, s);
  }
  return s;
}

typedef struct { float s; int32_t b; } scored_block;

/* Larger score first (-0.0 == +0.0 by float comparison); equal: lower block first. */
static int cmp_scored_block(const void* a, const void* b) {
  const scored_block* p = (const scored_block*)a;
  const scored_block* q = (const scored_block*)b;
  if (p->s > q->s) return -1;
  if (p->s < q->s) return 1;
  return (p->b > q->b) - (p->b < q->b);
}

static int cmp_int32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Block selection for layers [l0, l1) of L and all R rows.
 *   keys [L][N][D] bf16 (layer stride key_stride elements); q [L][R][Hh][D] bf16;
 *   hw [L][R][Hh] fp32; mask [L][R][ceil(N/32)]; limit [L][R].
 * Outputs (full [L][R] arrays; only layers l0..l1-1 written):
 *   sel [L][R][topk] ascending, -1 padded; nsel [L][R]; cidx [L][R][N] admitted blocks
 *   ascending; ccount [L][R]; cscore [L][R][N] canonical scores aligned with cidx
 *   (cidx, ccount and cscore may be NULL). */
void orc_select(int32_t L, int32_t R, int32_t Hh, int32_t D, int32_t N, int32_t topk,
                const uint16_t* keys, int64_t key_stride, const uint16_t* q, const float* hw,
                const uint32_t* mask, const int32_t* limit, int32_t l0, int32_t l1,
                int32_t* sel, int32_t* nsel, int32_t* cidx, int32_t* ccount, float* cscore) {
  (void)L;
  const int64_t W = (N + 31) / 32;
  scored_block* list = (scored_block*)malloc(sizeof(scored_block) * (size_t)(N > 0 ? N : 1));
  for (int32_t l = l0; l < l1; ++l) {
    for (int32_t r = 0; r < R; ++r) {
      const int64_t lr = (int64_t)l * R + r;
      const uint16_t* qr = q + lr * Hh * D;
      const float* wr = hw + lr * Hh;
      const uint32_t* mr = mask + lr * W;
      int32_t lim = limit[lr];
      int32_t cnt = 0;
      for (int32_t b = 0; b < lim && b < N; ++b) {
        if (!((mr[b / 32] >> (b % 32)) & 1u)) continue;   /* not admitted: not scored */
        float sc = orc_block_score(qr, keys + (int64_t)l * key_stride + (int64_t)b * D, wr, Hh, D);
        if (cidx) cidx[lr * N + cnt] = b;
        if (cscore) cscore[lr * N + cnt] = sc;
        list[cnt].s = sc;
        list[cnt].b = b;
        ++cnt;
      }
      if (ccount) ccount[lr] = cnt;
      qsort(list, (size_t)cnt, sizeof(scored_block), cmp_scored_block);
      int32_t m = cnt < topk ? cnt : topk;
      int32_t* out = sel + lr * topk;
      for (int32_t j = 0; j < m; ++j) out[j] = list[j].b;
      qsort(out, (size_t)m, sizeof(int32_t), cmp_int32);
      for (int32_t j = m; j < topk; ++j) out[j] = -1;
      nsel[lr] = m;
    }
  }
  free(list);
}

/* ------------------------------------------------------- speculative bookkeeping ---- */

/* Tokens committed by one verify step of R rows (1 + R-1 drafts), given the R-1 draft
 * acceptance outcomes in draft order (1 = accepted): 1 + the number of leading
 * acceptances. Reading of "weight bytes per committed token" with a Bernoulli
 * stand-in for the drafter. */
int32_t orc_committed_tokens(const uint8_t* accepted, int32_t R) {
  int32_t c = 1;
  for (int32_t j = 0; j < R - 1; ++j) {
    if (!accepted[j]) break;
    ++c;
  }
  return c;
}

/* ------------------------------------------------------------ verify acceptance ---- */

/* Paragraph "DSpark": a decode step verifies R rows (the last committed token and R - 1
 * drafted tokens) in one pass; under greedy decode the output is the same as without
 * drafts, and at temperature > 0 the drafts are accepted by exact speculative sampling.
 * Readings: row r's target logits (fp32 [R][V]) predict the token after row r's input;
 * draft token j (draft[j], j = 0..R-2) is the input of row j + 1, so it is checked against
 * row j's prediction. Both functions write the emitted tokens to out (at most R) and
 * return how many: the accepted drafts, then one token from the target (the correction at
 * the first rejection, or the bonus token after the last row). */

/* Greedy: a draft is accepted iff it equals the argmax of its row (ties to the lower id). */
int32_t orc_verify_greedy(const float* logits, int32_t R, int32_t V, const int32_t* draft,
                          int32_t* out) {
  int32_t n = 0;
  for (int32_t r = 0; r < R; ++r) {
    const float* z = logits + (int64_t)r * V;
    int32_t best = 0;
    for (int32_t v = 1; v < V; ++v)
      if (z[v] > z[best]) best = v;
    out[n++] = best;
    if (r == R - 1 || draft[r] != best) break;
  }
  return n;
}

/* The smallest x with u * sum(w) < w[0] + ... + w[x] (sums in index order, fp64); when
 * rounding leaves none, the last x with w[x] > 0. u in [0, 1). */
static int32_t sample_weights(const double* w, int32_t V, double u) {
  double total = 0.0;
  int32_t last = 0;
  for (int32_t v = 0; v < V; ++v) {
    total += w[v];
    if (w[v] > 0.0) last = v;
  }
  const double target = u * total;
  double acc = 0.0;
  for (int32_t v = 0; v < V; ++v) {
    acc += w[v];
    if (target < acc) return v;
  }
  return last;
}

/* p = softmax(z / T) in fp64: exp(z / T - max z / T) over the row, divided by their sum in
 * index order. */
static void softmax_t(const float* z, int32_t V, double T, double* p) {
  double m = (double)z[0] / T;
  for (int32_t v = 1; v < V; ++v)
    if ((double)z[v] / T > m) m = (double)z[v] / T;
  double s = 0.0;
  for (int32_t v = 0; v < V; ++v) {
    p[v] = exp((double)z[v] / T - m);
    s += p[v];
  }
  for (int32_t v = 0; v < V; ++v) p[v] /= s;
}

/* Exact speculative sampling at temperature T > 0. The drafter's proposal distributions
 * qd (fp64 [R-1][V], rows summing to 1) and the uniforms in [0, 1) are inputs. Row r's
 * draft d = draft[r] is accepted iff u_acc[r] * qd_r[d] < p_r[d] (probability
 * min(1, p_r[d] / qd_r[d])); at the first rejection the correction is drawn from the
 * residual max(p_r - qd_r, 0) with u_res[r] (from p_r if rounding leaves the residual
 * empty); after R - 1 acceptances the bonus token is drawn from p_{R-1} with u_res[R-1].
 * Returns -1 (nothing written) when T is not a finite positive number. */
int32_t orc_verify_sample(const float* logits, int32_t R, int32_t V, double T, const double* qd,
                          const int32_t* draft, const double* u_acc, const double* u_res,
                          int32_t* out) {
  if (!(T > 0.0) || !isfinite(T)) return -1;   /* softmax(z / T) needs a finite T > 0 */
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* res = (double*)malloc(sizeof(double) * (size_t)V);
  int32_t n = 0;
  for (int32_t r = 0; r < R; ++r) {
    softmax_t(logits + (int64_t)r * V, V, T, p);
    if (r == R - 1) {
      out[n++] = sample_weights(p, V, u_res[r]);
      break;
    }
    const double* q = qd + (int64_t)r * V;
    const int32_t d = draft[r];
    if (u_acc[r] * q[d] < p[d]) {
      out[n++] = d;
      continue;
    }
    double rs = 0.0;
    for (int32_t v = 0; v < V; ++v) {
      res[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;
      rs += res[v];
    }
    out[n++] = sample_weights(rs > 0.0 ? res : p, V, u_res[r]);
    break;
  }
  free(p);
  free(res);
  return n;
}

/* ---------------------------------------------------------- sparse attention ---- */

/* Attention of R query rows over the tokens of their selected blocks (one layer).
 * Reading (the pages stop at the selection): blocks of `bs` consecutive tokens; row r reads
 * the tokens bs*b .. bs*b + bs - 1 of every selected block b (sel[r][j] >= 0, j < K); all
 * Hq query heads of a row share one key and one value per token (D values each). For
 * row r and head h, with the tokens t in ascending order:
 *   s_t = (q_{r,h} . k_t) / sqrt(D),  p = softmax(s),  o_{r,h} = sum_t p_t v_t,
 * in fp64 from the bf16 inputs, then o rounded once to bf16 (round to nearest even). A row
 * with no selected block gets o = 0. q bf16 [R][Hq][D], k and v bf16 [T][D], sel int32
 * [R][K] (ascending, -1 padded), o64 fp64 [R][Hq][D] and obf bf16 [R][Hq][D] (either may
 * be NULL). Returns -1 when a selected block lies outside [0, T / bs), else 0. */
int32_t orc_sparse_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             int64_t T, int32_t D, int32_t R, int32_t Hq, const int32_t* sel,
                             int32_t K, int32_t bs, double* o64, uint16_t* obf) {
  const int64_t nblk = T / bs;
  for (int32_t r = 0; r < R; ++r)
    for (int32_t j = 0; j < K; ++j) {
      const int32_t b = sel[(int64_t)r * K + j];
      if (b >= nblk) return -1;
    }
  double* s = (double*)malloc(sizeof(double) * (size_t)K * (size_t)bs + 1);
  double* acc = (double*)malloc(sizeof(double) * (size_t)D);
  const double scale = 1.0 / sqrt((double)D);
  for (int32_t r = 0; r < R; ++r) {
    const int32_t* sr = sel + (int64_t)r * K;
    for (int32_t h = 0; h < Hq; ++h) {
      const uint16_t* qh = q + ((int64_t)r * Hq + h) * D;
      /* scores of the selected tokens in token order, and their maximum */
      int64_t n = 0;
      double m = -INFINITY;
      for (int32_t j = 0; j < K; ++j) {
        const int32_t b = sr[j];
        if (b < 0) continue;
        for (int32_t e = 0; e < bs; ++e) {
          const uint16_t* kt = k + ((int64_t)b * bs + e) * D;
          double dot = 0.0;
          for (int32_t i = 0; i < D; ++i) dot += orc_bf16_to_f64(qh[i]) * orc_bf16_to_f64(kt[i]);
          s[n] = dot * scale;
          if (s[n] > m) m = s[n];
          ++n;
        }
      }
      for (int32_t i = 0; i < D; ++i) acc[i] = 0.0;
      double den = 0.0;
      n = 0;
      for (int32_t j = 0; j < K; ++j) {
        const int32_t b = sr[j];
        if (b < 0) continue;
        for (int32_t e = 0; e < bs; ++e) {
          const double w = exp(s[n++] - m);
          const uint16_t* vt = v + ((int64_t)b * bs + e) * D;
          den += w;
          for (int32_t i = 0; i < D; ++i) acc[i] += w * orc_bf16_to_f64(vt[i]);
        }
      }
      for (int32_t i = 0; i < D; ++i) {
        const double o = n > 0 ? acc[i] / den : 0.0;
        const int64_t at = ((int64_t)r * Hq + h) * D + i;
        if (o64) o64[at] = o;
        if (obf) obf[at] = orc_bf16_rne(o);
      }
    }
  }
  free(s);
  free(acc);
  return 0;
}

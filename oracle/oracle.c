/*
 * ORACLE - test infrastructure only.
 *
 * A plain, slow, element-by-element CPU statement of the per-parameter update
 * that the packed-state optimizer performs. Only the tests, the smoke check and
 * the bench's CPU-baseline leg may load this file's library. It shares no code,
 * header or constant with the CUDA library.
 *
 * What it follows:
 *   - "Training 70B Models on Consumer Hardware (If You're Willing to Wait)",
 *     section "The Math": Adam written as an additive delta on the stored
 *     weight, first moment m, second moment v, bias corrections 1 - beta^t with
 *     one global step t, and eps added to the square root of the corrected
 *     second moment.
 *   - same page, section "The Assumption Everyone Makes": the SGD form
 *     W_new = W_old - lr * g rewritten as W += (-lr * g).
 *   - "MegaTrain" summary page, section on the memory bottleneck of the usual
 *     training setup: bf16 weight, bf16 gradient, fp32 m and v (12 B/param);
 *     the Cloudera full-training memory article (weights / gradients /
 *     optimizer states line items) and the "Transformer Training 09 - Memory"
 *     deck (16 B/param): an fp32 master copy of the weight, and plain fp32
 *     Adam with fp32 weight and gradient.
 *   - Decoupled weight decay (AdamW): not on the pages; the reading used is
 *     w' = w * (1 - lr * wd) - lr * u, applied to the weight before the Adam
 *     step, uniformly to every element.
 *
 * Precision: the pages keep the moments and the master copy in fp32, so every
 * arithmetic step below is one IEEE fp32 operation, rounded to nearest, in the
 * order written. Build without contraction (-ffp-contract=off) and without
 * fast-math. The step scalars (1 - beta1, 1 - beta2, 1 - beta1^t, 1 - beta2^t,
 * 1 - lr * wd) are formed in double and rounded once to fp32.
 *
 * bf16 conversions are written here from the format's definition: widening is
 * exact (the 16 bits become the top half of an fp32 word); narrowing rounds to
 * nearest, ties to even, and keeps NaN a quiet NaN.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  int64_t step;
} orc_hparams;

typedef struct {
  float beta1, beta2;
  float one_minus_beta1, one_minus_beta2;
  float bias_correction1, bias_correction2; /* 1 - beta^t */
  float eps, lr;
  float decay; /* 1 - lr * wd */
} orc_scalars;

/* ---- bf16 <-> fp32 ---------------------------------------------------- */

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep sign and top payload, force quiet */
    return (uint16_t)((u >> 16) | 0x0040u);
  /* Add just under half of the dropped part's range, plus the kept lsb, so
     that exact halves go to the even neighbour; a carry out of the mantissa
     moves the exponent (and past the largest finite value gives infinity). */
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

void orc_bf16_from_f32_array(int64_t n, const float* in, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

void orc_f32_from_bf16_array(int64_t n, const uint16_t* in, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}

/* ---- step scalars ----------------------------------------------------- */

/* Returns 0, or -1 if the hyperparameters are outside the method's domain. */
int orc_make_scalars(const orc_hparams* hp, orc_scalars* s) {
  if (!hp || !s) return -1;
  if (hp->step < 1) return -1;
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f)) return -1;
  if (!(hp->beta2 >= 0.0f && hp->beta2 < 1.0f)) return -1;
  if (!isfinite(hp->lr) || !isfinite(hp->eps) || !isfinite(hp->weight_decay)) return -1;
  double b1 = hp->beta1, b2 = hp->beta2, t = (double)hp->step;
  s->beta1 = hp->beta1;
  s->beta2 = hp->beta2;
  s->one_minus_beta1 = (float)(1.0 - b1);
  s->one_minus_beta2 = (float)(1.0 - b2);
  s->bias_correction1 = (float)(1.0 - pow(b1, t));
  s->bias_correction2 = (float)(1.0 - pow(b2, t));
  s->eps = hp->eps;
  s->lr = hp->lr;
  s->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
  return 0;
}

/* ---- one element ------------------------------------------------------ */

/* Adam moments, bias correction and the decoupled-decay additive step for one
   parameter. w is the fp32 value being updated; m and v are updated in place.
   Returns the new w. */
static float adamw_one(float g, float w, float* m, float* v, const orc_scalars* s) {
  /* first and second moments */
  float m_new = s->beta1 * (*m) + s->one_minus_beta1 * g;
  float g_sq = g * g;
  float v_new = s->beta2 * (*v) + s->one_minus_beta2 * g_sq;
  *m = m_new;
  *v = v_new;
  /* bias-corrected moments */
  float m_hat = m_new / s->bias_correction1;
  float v_hat = v_new / s->bias_correction2;
  /* normalised step, eps outside the root */
  float denom = sqrtf(v_hat) + s->eps;
  float u = m_hat / denom;
  /* decoupled decay of the pre-step weight, then the additive delta */
  float w_decayed = w * s->decay;
  float step = s->lr * u;
  return w_decayed - step;
}

/* ---- the three layouts ------------------------------------------------ */

/* 12 B/param: bf16 G (in), bf16 W (in/out), fp32 m, v (in/out). */
void orc_adamw_l12(int64_t n, const uint16_t* G, uint16_t* W, float* m, float* v,
                   const orc_scalars* s) {
  for (int64_t i = 0; i < n; ++i) {
    float g = orc_bf16_to_f32(G[i]);
    float w = orc_bf16_to_f32(W[i]);
    float w_new = adamw_one(g, w, &m[i], &v[i], s);
    W[i] = orc_f32_to_bf16(w_new);
  }
}

/* 16 B/param mixed: bf16 G (in), fp32 master (in/out), fp32 m, v (in/out),
   bf16 W (out) = master rounded to nearest even. */
void orc_adamw_l16m(int64_t n, const uint16_t* G, float* master, float* m, float* v, uint16_t* W,
                    const orc_scalars* s) {
  for (int64_t i = 0; i < n; ++i) {
    float g = orc_bf16_to_f32(G[i]);
    float w_new = adamw_one(g, master[i], &m[i], &v[i], s);
    master[i] = w_new;
    W[i] = orc_f32_to_bf16(w_new);
  }
}

/* 16 B/param fp32: fp32 G (in), fp32 W, m, v (in/out). */
void orc_adamw_l16f(int64_t n, const float* G, float* W, float* m, float* v, const orc_scalars* s) {
  for (int64_t i = 0; i < n; ++i) W[i] = adamw_one(G[i], W[i], &m[i], &v[i], s);
}

/* ---- SGD as an additive delta: W += (-lr * g) --------------------------- */

static float sgd_one(float g, float w, float lr) {
  float delta = -(lr * g);
  return w + delta;
}

void orc_sgd_l12(int64_t n, const uint16_t* G, uint16_t* W, float lr) {
  for (int64_t i = 0; i < n; ++i)
    W[i] = orc_f32_to_bf16(sgd_one(orc_bf16_to_f32(G[i]), orc_bf16_to_f32(W[i]), lr));
}

void orc_sgd_l16m(int64_t n, const uint16_t* G, float* master, uint16_t* W, float lr) {
  for (int64_t i = 0; i < n; ++i) {
    float w_new = sgd_one(orc_bf16_to_f32(G[i]), master[i], lr);
    master[i] = w_new;
    W[i] = orc_f32_to_bf16(w_new);
  }
}

void orc_sgd_l16f(int64_t n, const float* G, float* W, float lr) {
  for (int64_t i = 0; i < n; ++i) W[i] = sgd_one(G[i], W[i], lr);
}

/* ---- gradient magnitude for progressive layer locking -------------------- */

/* Sum of g^2 over a block's gradient, in double, element by element in order
   ("Training 70B Models on Consumer Hardware", section "Progressive Layer
   Locking": a layer is locked when its gradient magnitude falls below a
   threshold; the squared L2 norm is the plain reading of that magnitude). */
double orc_grad_sq_bf16(int64_t n, const uint16_t* G) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double g = (double)orc_bf16_to_f32(G[i]);
    s += g * g;
  }
  return s;
}

double orc_grad_sq_f32(int64_t n, const float* G) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double g = (double)G[i];
    s += g * g;
  }
  return s;
}

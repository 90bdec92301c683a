/* Oracle: plain FP64 CPU restatement of one decode token of the hybrid
 * Gated-DeltaNet / GQA-attention / MoE transformer.  TEST INFRASTRUCTURE ONLY:
 * see oracle.h for who may use it, its precision rules and its pins.
 *
 * Sources (the pages this is written from):
 *  [Strata]  "Beating llama.cpp from Scratch on Consumer AMD: Building Strata,
 *            a Native Rust + HIP Local AI Engine"
 *  [14h]     "Fourteen hours to 100 tokens per second"
 *  [Flash]   "Flash-Next on Strix Halo"
 * Where the pages name a step without giving its formula, the plainest reading
 * is taken; each such reading is marked "reading:" below.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- formats */

double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* bf16 code of x: x is first rounded to FP32 (the kernels' precision), then
 * to bf16 with round-to-nearest-even.  [Strata] "The Beast": the KV cache is
 * bf16. */
uint16_t orc_to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf/nan: truncate */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* IEEE binary16 -> double, from the format's definition. */
double orc_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1024.0 + m, e - 25);
  return sign ? -v : v;
}

/* 4-bit block value.  [Flash] "Correctness fixes": the q4_0 layout keeps a
 * split-nibble +8 offset for a 32-wide K block; reading: byte b of a block
 * holds element b (low nibble) and element b+16 (high nibble), each stored as
 * value+8, with one fp16 scale per block: w = scale * (nibble - 8). */
double orc_q4_value(const orc_mat* m, int64_t r, int64_t c) {
  int64_t blk = c / 32, e = c % 32;
  uint8_t byte = m->qs[r * (m->cols / 2) + blk * 16 + (e % 16)];
  int nib = e < 16 ? (byte & 0xF) : (byte >> 4);
  double s = orc_fp16_to_double(m->scales[r * (m->cols / 32) + blk]);
  return s * (double)(nib - 8);
}

void orc_mat_row(const orc_mat* m, int64_t r, double* out) {
  if (m->fmt == 0) {
    const uint16_t* row = m->bf16 + r * m->cols;
    for (int64_t c = 0; c < m->cols; ++c) out[c] = orc_bf16_to_double(row[c]);
  } else {
    for (int64_t c = 0; c < m->cols; ++c) out[c] = orc_q4_value(m, r, c);
  }
}

/* rows [r0, r0+n) of m as a matrix of its own */
static orc_mat orc_mat_rows(const orc_mat* m, int64_t r0, int64_t n) {
  orc_mat s = *m;
  s.rows = n;
  if (m->fmt == 0) {
    s.bf16 = m->bf16 + r0 * m->cols;
  } else {
    s.qs = m->qs + r0 * (m->cols / 2);
    s.scales = m->scales + r0 * (m->cols / 32);
  }
  return s;
}

/* ------------------------------------------------------------ primitives */

/* y = W x, one plain dot product per row.  [Strata] "Act 0", pass 3: decode
 * at M = 1 is a matrix-vector product. */
void orc_gemv(const orc_mat* m, const double* x, double* y) {
#pragma omp parallel
  {
    double* row = (double*)malloc(sizeof(double) * (size_t)m->cols);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < m->rows; ++r) {
      orc_mat_row(m, r, row);
      double acc = 0.0;
      for (int64_t c = 0; c < m->cols; ++c) acc += row[c] * x[c];
      y[r] = acc;
    }
    free(row);
  }
}

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g.  [Strata] "Act 6" lists norms
 * among the decode ops; reading: pre-norm RMSNorm with eps inside the root. */
void orc_rmsnorm(const double* x, const float* g, int32_t n, double eps, double* y) {
  double ss = 0.0;
  for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int32_t i = 0; i < n; ++i) y[i] = x[i] * inv * (double)g[i];
}

/* reading: q and k of a DeltaNet head are L2-normalised, eps inside the root */
void orc_l2norm(double* v, int32_t n, double eps) {
  double ss = 0.0;
  for (int32_t i = 0; i < n; ++i) ss += v[i] * v[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int32_t i = 0; i < n; ++i) v[i] *= inv;
}

double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
double orc_silu(double x) { return x / (1.0 + exp(-x)); }

/* RoPE at absolute position pos.  [Strata] "Act 1" (RoPE position
 * embeddings applied per token); reading: rotate-half pairs (i, i + hd/2) over
 * the full head, angle pos * theta^(-2i/hd). */
void orc_rope(double* v, int32_t hd, int32_t pos, double theta) {
  int32_t half = hd / 2;
  for (int32_t i = 0; i < half; ++i) {
    double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)hd);
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* Causal depthwise conv of width k over the DeltaNet input channels, decode
 * form.  [Strata] "The Beast": the state updates via a 1D convolution and a
 * gated delta rule; "Act 1": causal Conv1D.  reading: out = silu(sum_j
 * w[c][j] * u_{t-(k-1)+j}), tap k-1 on the current input, zeros before t = 0,
 * no bias.  state holds the previous k-1 inputs, oldest first, and is shifted
 * by one. */
void orc_conv_step(const double* u, double* state, const uint16_t* w, int32_t channels, int32_t k, double* out) {
  for (int32_t c = 0; c < channels; ++c) {
    double acc = 0.0;
    for (int32_t j = 0; j < k - 1; ++j) acc += orc_bf16_to_double(w[(int64_t)c * k + j]) * state[(int64_t)j * channels + c];
    acc += orc_bf16_to_double(w[(int64_t)c * k + (k - 1)]) * u[c];
    out[c] = orc_silu(acc);
  }
  for (int32_t j = 0; j + 1 < k - 1; ++j)
    memcpy(state + (int64_t)j * channels, state + (int64_t)(j + 1) * channels, sizeof(double) * (size_t)channels);
  if (k > 1) memcpy(state + (int64_t)(k - 2) * channels, u, sizeof(double) * (size_t)channels);
}

/* One gated delta-rule step of one head, in its plain matrix form:
 *   S <- alpha * S (I - beta k k^T) + beta v k^T,   o = S q
 * with S in R^{dv x dk}, row i (value index) contiguous over the key index.
 * [Strata] "The Beast": fixed-size FP32 state updated in place by a gated
 * delta update rule.  The (I - beta k k^T) matrix is formed explicitly. */
void orc_gdn_step(float* S, int32_t dk, int32_t dv, const double* q, const double* k, const double* v,
                  double alpha, double beta, double* o) {
  double* M = (double*)malloc(sizeof(double) * (size_t)dk * (size_t)dk);
  double* Sn = (double*)malloc(sizeof(double) * (size_t)dk);
  for (int32_t a = 0; a < dk; ++a)
    for (int32_t b = 0; b < dk; ++b) M[(int64_t)a * dk + b] = (a == b ? 1.0 : 0.0) - beta * k[a] * k[b];
  for (int32_t i = 0; i < dv; ++i) {
    float* Si = S + (int64_t)i * dk;
    for (int32_t j = 0; j < dk; ++j) {
      double acc = 0.0;
      for (int32_t m = 0; m < dk; ++m) acc += (double)Si[m] * M[(int64_t)m * dk + j];
      Sn[j] = alpha * acc + beta * v[i] * k[j];
    }
    double oi = 0.0;
    for (int32_t j = 0; j < dk; ++j) {
      Si[j] = (float)Sn[j];
      oi += (double)Si[j] * q[j];
    }
    o[i] = oi;
  }
  free(Sn);
  free(M);
}

/* int8 quantisation of one cached vector x[0..n) with one FP32 scale:
 * "hanzo-engine: A Portable Single-Binary LLM Inference Engine...", section
 * "System Architecture" (an int8 KV cache with one f32 scale per cached
 * vector) and "Results" ("int8 KV").  The pages name only the format; the
 * rule is the plainest symmetric one: with a = max_i |x_i| (x taken in FP32,
 * where the decisions are made), scale = a / 127 and q_i = round-half-even(x_i
 * * (127 / a)) in FP32, clamped to [-127, 127]; a = 0 gives codes 0 and scale
 * 0.  The stored value of element i is q_i * scale. */
void orc_quant_i8(const double* x, int32_t n, int8_t* q, float* scale) {
  float amax = 0.0f;
  for (int32_t i = 0; i < n; ++i) {
    float f = fabsf((float)x[i]);
    if (f > amax) amax = f;
  }
  if (amax == 0.0f) {
    for (int32_t i = 0; i < n; ++i) q[i] = 0;
    *scale = 0.0f;
    return;
  }
  volatile float inv = 127.0f / amax; /* FP32 division, as the kernel's */
  for (int32_t i = 0; i < n; ++i) {
    volatile float prod = (float)x[i] * inv; /* one FP32 rounding of the product */
    float r = rintf(prod);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
  *scale = amax / 127.0f;
}

/* Attention of orc_attention over an int8 cache: K and V values are the
 * stored codes times their vector's scale. */
void orc_attention_i8(const double* q, const int8_t* Kq, const float* Ks, const int8_t* Vq, const float* Vs,
                      int32_t nq, int32_t nkv, int32_t hd, int32_t cap, int32_t npos, double* o) {
  int32_t group = nq / nkv;
  double scale = 1.0 / sqrt((double)hd);
  double* s = (double*)malloc(sizeof(double) * (size_t)(npos > 0 ? npos : 1));
  for (int32_t j = 0; j < nq; ++j) {
    int32_t g = j / group;
    double mx = -INFINITY;
    for (int32_t p = 0; p < npos; ++p) {
      const int8_t* kr = Kq + ((int64_t)g * cap + p) * hd;
      double ks = (double)Ks[(int64_t)g * cap + p];
      double acc = 0.0;
      for (int32_t d = 0; d < hd; ++d) acc += q[(int64_t)j * hd + d] * ((double)kr[d] * ks);
      s[p] = acc * scale;
      if (s[p] > mx) mx = s[p];
    }
    double den = 0.0;
    for (int32_t p = 0; p < npos; ++p) {
      s[p] = exp(s[p] - mx);
      den += s[p];
    }
    for (int32_t d = 0; d < hd; ++d) {
      double acc = 0.0;
      for (int32_t p = 0; p < npos; ++p)
        acc += s[p] * ((double)Vq[((int64_t)g * cap + p) * hd + d] * (double)Vs[(int64_t)g * cap + p]);
      o[(int64_t)j * hd + d] = npos > 0 ? acc / den : 0.0;
    }
  }
  free(s);
}

/* Single-pass softmax attention of nq query heads over positions [0, npos) of
 * a bf16 cache [nkv][cap][hd]; query head j reads kv head j / (nq / nkv).
 * [Strata] "The Beast" (GQA layers, bf16 KV cache [kv_heads, seq_len, dim]);
 * reading: scores scaled by 1/sqrt(hd), contiguous GQA grouping. */
void orc_attention(const double* q, const uint16_t* K, const uint16_t* V, int32_t nq, int32_t nkv, int32_t hd,
                   int32_t cap, int32_t npos, double* o) {
  int32_t group = nq / nkv;
  double scale = 1.0 / sqrt((double)hd);
  double* s = (double*)malloc(sizeof(double) * (size_t)(npos > 0 ? npos : 1));
  for (int32_t j = 0; j < nq; ++j) {
    int32_t g = j / group;
    const uint16_t* Kg = K + (int64_t)g * cap * hd;
    const uint16_t* Vg = V + (int64_t)g * cap * hd;
    double mx = -INFINITY;
    for (int32_t p = 0; p < npos; ++p) {
      double acc = 0.0;
      for (int32_t d = 0; d < hd; ++d) acc += q[(int64_t)j * hd + d] * orc_bf16_to_double(Kg[(int64_t)p * hd + d]);
      s[p] = acc * scale;
      if (s[p] > mx) mx = s[p];
    }
    double den = 0.0;
    for (int32_t p = 0; p < npos; ++p) {
      s[p] = exp(s[p] - mx);
      den += s[p];
    }
    for (int32_t d = 0; d < hd; ++d) {
      double acc = 0.0;
      for (int32_t p = 0; p < npos; ++p) acc += s[p] * orc_bf16_to_double(Vg[(int64_t)p * hd + d]);
      o[(int64_t)j * hd + d] = npos > 0 ? acc / den : 0.0;
    }
  }
  free(s);
}

/* The same attention computed as nsplit partial sums over contiguous position
 * chunks, then merged with their log-sum-exp weights:
 *   m = max_s m_s,  o = sum_s e^{m_s - m} o_s / sum_s e^{m_s - m} l_s.
 * [Strata] "Act 4" (per-split partial sums over the KV length) and "What
 * Broke" section 1 (partial sums combined across separate workgroups).  Used
 * only to pin that the split form equals the single pass. */
void orc_attention_split(const double* q, const uint16_t* K, const uint16_t* V, int32_t nq, int32_t nkv,
                         int32_t hd, int32_t cap, int32_t npos, int32_t nsplit, double* o) {
  int32_t group = nq / nkv;
  double scale = 1.0 / sqrt((double)hd);
  double* ms = (double*)malloc(sizeof(double) * (size_t)nsplit);
  double* ls = (double*)malloc(sizeof(double) * (size_t)nsplit);
  double* os = (double*)malloc(sizeof(double) * (size_t)nsplit * (size_t)hd);
  for (int32_t j = 0; j < nq; ++j) {
    int32_t g = j / group;
    const uint16_t* Kg = K + (int64_t)g * cap * hd;
    const uint16_t* Vg = V + (int64_t)g * cap * hd;
    for (int32_t sp = 0; sp < nsplit; ++sp) {
      int32_t p0 = (int32_t)((int64_t)sp * npos / nsplit), p1 = (int32_t)((int64_t)(sp + 1) * npos / nsplit);
      double m = -INFINITY, l = 0.0;
      for (int32_t d = 0; d < hd; ++d) os[(int64_t)sp * hd + d] = 0.0;
      for (int32_t p = p0; p < p1; ++p) {
        double acc = 0.0;
        for (int32_t d = 0; d < hd; ++d) acc += q[(int64_t)j * hd + d] * orc_bf16_to_double(Kg[(int64_t)p * hd + d]);
        if (acc * scale > m) m = acc * scale;
      }
      for (int32_t p = p0; p < p1; ++p) {
        double acc = 0.0;
        for (int32_t d = 0; d < hd; ++d) acc += q[(int64_t)j * hd + d] * orc_bf16_to_double(Kg[(int64_t)p * hd + d]);
        double e = exp(acc * scale - m);
        l += e;
        for (int32_t d = 0; d < hd; ++d) os[(int64_t)sp * hd + d] += e * orc_bf16_to_double(Vg[(int64_t)p * hd + d]);
      }
      ms[sp] = m;
      ls[sp] = l;
    }
    double mx = -INFINITY;
    for (int32_t sp = 0; sp < nsplit; ++sp)
      if (ms[sp] > mx) mx = ms[sp];
    double den = 0.0;
    for (int32_t sp = 0; sp < nsplit; ++sp)
      if (ls[sp] > 0.0) den += exp(ms[sp] - mx) * ls[sp];
    for (int32_t d = 0; d < hd; ++d) {
      double acc = 0.0;
      for (int32_t sp = 0; sp < nsplit; ++sp)
        if (ls[sp] > 0.0) acc += exp(ms[sp] - mx) * os[(int64_t)sp * hd + d];
      o[(int64_t)j * hd + d] = den > 0.0 ? acc / den : 0.0;
    }
  }
  free(os);
  free(ls);
  free(ms);
}

/* Greedy pick: index of the largest value (compared as FP32), lowest index on
 * ties.  [Strata] "Act 0", pass 3: on-device argmax returns one token id. */
int32_t orc_argmax(const double* v, int64_t n) {
  int64_t best = 0;
  float bv = (float)v[0];
  for (int64_t i = 1; i < n; ++i) {
    float f = (float)v[i];
    if (f > bv) {
      bv = f;
      best = i;
    }
  }
  return (int32_t)best;
}

/* Top-k by repeated selection of the largest remaining value (compared as
 * FP32), lowest index on ties; ids come out in descending order.
 * [14h] "Starting point" (8 of 256 experts per token) and "The trace that
 * changed everything" (F32 router, top-k routing). */
void orc_topk(const double* r, int32_t n, int32_t k, int32_t* ids) {
  unsigned char* taken = (unsigned char*)calloc((size_t)n, 1);
  for (int32_t t = 0; t < k; ++t) {
    int32_t best = -1;
    float bv = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
      if (taken[i]) continue;
      float f = (float)r[i];
      if (best < 0 || f > bv) {
        bv = f;
        best = i;
      }
    }
    ids[t] = best;
    taken[best] = 1;
  }
  free(taken);
}

void orc_softmax(const double* x, int32_t n, double* p) {
  double mx = -INFINITY;
  for (int32_t i = 0; i < n; ++i)
    if (x[i] > mx) mx = x[i];
  double den = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    p[i] = exp(x[i] - mx);
    den += p[i];
  }
  for (int32_t i = 0; i < n; ++i) p[i] /= den;
}

/* ------------------------------------------------------------ the model */

static int32_t count_layers(const orc_config* cfg, int attn) {
  int32_t n = 0;
  for (int32_t l = 0; l < cfg->n_layers; ++l) n += (cfg->is_attn[l] ? 1 : 0) == attn;
  return n;
}

static int32_t conv_channels(const orc_config* cfg) { return 2 * cfg->gdn_heads * cfg->gdn_dk + cfg->gdn_heads * cfg->gdn_dv; }

int orc_cache_create(const orc_config* cfg, int32_t capacity, orc_cache* out) {
  memset(out, 0, sizeof(*out));
  out->capacity = capacity;
  int64_t ng = count_layers(cfg, 0), na = count_layers(cfg, 1);
  int64_t st = ng * cfg->gdn_heads * (int64_t)cfg->gdn_dv * cfg->gdn_dk;
  int64_t cs = ng * (int64_t)(cfg->conv_k - 1) * conv_channels(cfg);
  int64_t kv = na * (int64_t)cfg->attn_kv_heads * capacity * cfg->head_dim;
  out->gdn_state = (float*)calloc((size_t)(st > 0 ? st : 1), sizeof(float));
  out->conv_state = (double*)calloc((size_t)(cs > 0 ? cs : 1), sizeof(double));
  out->k_cache = (uint16_t*)calloc((size_t)(kv > 0 ? kv : 1), sizeof(uint16_t));
  out->v_cache = (uint16_t*)calloc((size_t)(kv > 0 ? kv : 1), sizeof(uint16_t));
  if (cfg->kv_format == 1) {
    int64_t ns = na * (int64_t)cfg->attn_kv_heads * capacity;
    out->k_q = (int8_t*)calloc((size_t)(kv > 0 ? kv : 1), 1);
    out->v_q = (int8_t*)calloc((size_t)(kv > 0 ? kv : 1), 1);
    out->k_s = (float*)calloc((size_t)(ns > 0 ? ns : 1), sizeof(float));
    out->v_s = (float*)calloc((size_t)(ns > 0 ? ns : 1), sizeof(float));
    if (!out->k_q || !out->v_q || !out->k_s || !out->v_s) {
      orc_cache_destroy(out);
      return -1;
    }
  }
  if (!out->gdn_state || !out->conv_state || !out->k_cache || !out->v_cache) {
    orc_cache_destroy(out);
    return -1;
  }
  return 0;
}

void orc_cache_destroy(orc_cache* c) {
  free(c->gdn_state);
  free(c->conv_state);
  free(c->k_cache);
  free(c->v_cache);
  free(c->k_q);
  free(c->v_q);
  free(c->k_s);
  free(c->v_s);
  memset(c, 0, sizeof(*c));
}

void orc_cache_reset(const orc_config* cfg, orc_cache* c) {
  int64_t ng = count_layers(cfg, 0), na = count_layers(cfg, 1);
  memset(c->gdn_state, 0, sizeof(float) * (size_t)(ng * cfg->gdn_heads * (int64_t)cfg->gdn_dv * cfg->gdn_dk));
  memset(c->conv_state, 0, sizeof(double) * (size_t)(ng * (int64_t)(cfg->conv_k - 1) * conv_channels(cfg)));
  memset(c->k_cache, 0, sizeof(uint16_t) * (size_t)(na * (int64_t)cfg->attn_kv_heads * c->capacity * cfg->head_dim));
  memset(c->v_cache, 0, sizeof(uint16_t) * (size_t)(na * (int64_t)cfg->attn_kv_heads * c->capacity * cfg->head_dim));
  if (c->k_q) {
    size_t nkv = (size_t)(na * (int64_t)cfg->attn_kv_heads * c->capacity);
    memset(c->k_q, 0, nkv * (size_t)cfg->head_dim);
    memset(c->v_q, 0, nkv * (size_t)cfg->head_dim);
    memset(c->k_s, 0, nkv * sizeof(float));
    memset(c->v_s, 0, nkv * sizeof(float));
  }
  c->len = 0;
}

/* x += W_d (silu(W_g xn) * (W_u xn)): a SwiGLU FFN.  [Strata] "Act 6"
 * (hidden x intermediate projection sizes); [14h] "Eight levers that worked"
 * (silu(gate) * x in the gated kernel). */
static void swiglu_ffn(const orc_mat* wg, const orc_mat* wu, const orc_mat* wd, const double* xn, double scale,
                       double* acc_out) {
  int64_t F = wg->rows, H = wd->rows;
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  orc_gemv(wg, xn, g);
  orc_gemv(wu, xn, u);
  for (int64_t i = 0; i < F; ++i) g[i] = orc_silu(g[i]) * u[i];
  orc_gemv(wd, g, y);
  for (int64_t i = 0; i < H; ++i) acc_out[i] += scale * y[i];
  free(y);
  free(u);
  free(g);
}

int orc_forward_token(const orc_config* cfg, const orc_weights* w, orc_cache* c, int32_t token, double* logits,
                      double* hidden, int32_t* router_ids, double* router_logits) {
  if (c->len >= c->capacity) return -1;
  const int32_t H = cfg->hidden, pos = c->len;
  const int32_t nh = cfg->gdn_heads, dk = cfg->gdn_dk, dv = cfg->gdn_dv, CC = conv_channels(cfg);
  const int32_t nq = cfg->attn_q_heads, nkv = cfg->attn_kv_heads, hd = cfg->head_dim;
  int64_t maxrows = H;
  if (2 * (int64_t)CC > maxrows) maxrows = 2 * (int64_t)CC;
  if ((int64_t)(nq + 2 * nkv) * hd > maxrows) maxrows = (int64_t)(nq + 2 * nkv) * hd;
  if (cfg->n_experts + 1 > maxrows) maxrows = cfg->n_experts + 1;
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* xn = (double*)malloc(sizeof(double) * (size_t)H);
  double* y = (double*)malloc(sizeof(double) * (size_t)maxrows);
  double* cv = (double*)malloc(sizeof(double) * (size_t)maxrows);
  double* o = (double*)malloc(sizeof(double) * (size_t)maxrows);
  double* d = (double*)malloc(sizeof(double) * (size_t)H);

  /* embedding row, bf16 widened */
  for (int32_t i = 0; i < H; ++i) x[i] = orc_bf16_to_double(w->embed[(int64_t)token * H + i]);

  int32_t gi = 0, ai = 0;
  for (int32_t l = 0; l < cfg->n_layers; ++l) {
    const orc_layer* L = &w->layers[l];
    orc_rmsnorm(x, L->norm1, H, cfg->rms_eps, xn);
    orc_gemv(&L->w_in, xn, y);
    if (cfg->is_attn[l]) {
      /* GQA layer: q|k|v, RoPE at pos, append bf16 K/V at row pos, attend
       * over positions 0..pos. */
      double* q = y;
      double* k = y + (int64_t)nq * hd;
      double* v = y + (int64_t)(nq + nkv) * hd;
      for (int32_t j = 0; j < nq; ++j) orc_rope(q + (int64_t)j * hd, hd, pos, cfg->rope_theta);
      for (int32_t g = 0; g < nkv; ++g) orc_rope(k + (int64_t)g * hd, hd, pos, cfg->rope_theta);
      if (cfg->kv_format == 1) {
        /* int8 cache: each new k and v vector quantised with its own scale */
        int8_t* Kq = c->k_q + (int64_t)ai * nkv * c->capacity * hd;
        int8_t* Vq = c->v_q + (int64_t)ai * nkv * c->capacity * hd;
        float* Ks = c->k_s + (int64_t)ai * nkv * c->capacity;
        float* Vs = c->v_s + (int64_t)ai * nkv * c->capacity;
        for (int32_t g = 0; g < nkv; ++g) {
          int64_t row = (int64_t)g * c->capacity + pos;
          orc_quant_i8(k + (int64_t)g * hd, hd, Kq + row * hd, Ks + row);
          orc_quant_i8(v + (int64_t)g * hd, hd, Vq + row * hd, Vs + row);
        }
        orc_attention_i8(q, Kq, Ks, Vq, Vs, nq, nkv, hd, c->capacity, pos + 1, o);
      } else {
        uint16_t* Kc = c->k_cache + (int64_t)ai * nkv * c->capacity * hd;
        uint16_t* Vc = c->v_cache + (int64_t)ai * nkv * c->capacity * hd;
        for (int32_t g = 0; g < nkv; ++g)
          for (int32_t e = 0; e < hd; ++e) {
            Kc[((int64_t)g * c->capacity + pos) * hd + e] = orc_to_bf16(k[(int64_t)g * hd + e]);
            Vc[((int64_t)g * c->capacity + pos) * hd + e] = orc_to_bf16(v[(int64_t)g * hd + e]);
          }
        orc_attention(q, Kc, Vc, nq, nkv, hd, c->capacity, pos + 1, o);
      }
      ++ai;
    } else {
      /* Gated DeltaNet layer: conv over q|k|v, per-head gates, delta rule. */
      double* cst = c->conv_state + (int64_t)gi * (cfg->conv_k - 1) * CC;
      orc_conv_step(y, cst, L->conv_w, CC, cfg->conv_k, cv);
      const double* a = y + CC;
      const double* b = y + CC + nh;
#pragma omp parallel for schedule(static)
      for (int32_t h = 0; h < nh; ++h) {
        double* qh = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kh = (double*)malloc(sizeof(double) * (size_t)dk);
        memcpy(qh, cv + (int64_t)h * dk, sizeof(double) * (size_t)dk);
        memcpy(kh, cv + (int64_t)nh * dk + (int64_t)h * dk, sizeof(double) * (size_t)dk);
        const double* vh = cv + 2 * (int64_t)nh * dk + (int64_t)h * dv;
        orc_l2norm(qh, dk, 1e-6);
        orc_l2norm(kh, dk, 1e-6);
        for (int32_t j = 0; j < dk; ++j) qh[j] /= sqrt((double)dk);
        float* S = c->gdn_state + ((int64_t)gi * nh + h) * (int64_t)dv * dk;
        orc_gdn_step(S, dk, dv, qh, kh, vh, orc_sigmoid(a[h]), orc_sigmoid(b[h]), o + (int64_t)h * dv);
        free(kh);
        free(qh);
      }
      ++gi;
    }
    orc_gemv(&L->w_o, o, d);
    for (int32_t i = 0; i < H; ++i) x[i] += d[i];

    orc_rmsnorm(x, L->norm2, H, cfg->rms_eps, xn);
    if (cfg->ffn > 0) {
      swiglu_ffn(&L->w_gate, &L->w_up, &L->w_down, xn, 1.0, x);
    } else {
      /* MoE: router logits over E experts plus the shared expert's gate row;
       * top-k by logit, softmax over the selected logits; the shared expert is
       * weighted by the sigmoid of its row ([14h] "The router with 257
       * rows"). */
      const int32_t E = cfg->n_experts, K = cfg->top_k, Fe = cfg->expert_ffn;
      double* r = y;
      orc_gemv(&L->router, xn, r);
      int32_t ids[64];
      double sel[64], wts[64];
      orc_topk(r, E, K, ids);
      for (int32_t t = 0; t < K; ++t) sel[t] = r[ids[t]];
      orc_softmax(sel, K, wts);
      if (router_ids) memcpy(router_ids + (int64_t)l * K, ids, sizeof(int32_t) * (size_t)K);
      if (router_logits) memcpy(router_logits + (int64_t)l * (E + 1), r, sizeof(double) * (size_t)(E + 1));
      double gs = orc_sigmoid(r[E]);
      memset(d, 0, sizeof(double) * (size_t)H);
      for (int32_t t = 0; t < K; ++t) {
        orc_mat g = orc_mat_rows(&L->exp_gate, (int64_t)ids[t] * Fe, Fe);
        orc_mat u = orc_mat_rows(&L->exp_up, (int64_t)ids[t] * Fe, Fe);
        orc_mat dn = orc_mat_rows(&L->exp_down, (int64_t)ids[t] * H, H);
        swiglu_ffn(&g, &u, &dn, xn, wts[t], d);
      }
      swiglu_ffn(&L->sh_gate, &L->sh_up, &L->sh_down, xn, gs, d);
      for (int32_t i = 0; i < H; ++i) x[i] += d[i];
    }
    if (hidden) memcpy(hidden + (int64_t)l * H, x, sizeof(double) * (size_t)H);
  }
  orc_rmsnorm(x, w->final_norm, H, cfg->rms_eps, xn);
  orc_gemv(&w->lm_head, xn, logits);
  c->len += 1;
  free(d);
  free(o);
  free(cv);
  free(y);
  free(xn);
  free(x);
  return 0;
}

int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

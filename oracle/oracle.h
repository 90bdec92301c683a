/* Oracle: a plain, slow, FP64 CPU restatement of one decode token of a hybrid
 * Gated-DeltaNet / GQA-attention / MoE transformer.
 *
 * TEST INFRASTRUCTURE ONLY.  It exists to check the CUDA library against, and
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no source with the CUDA library and includes
 * none of its headers.
 *
 * Precision: every intermediate is double.  Only the storage formats that the
 * pages fix are applied, at the points where they apply them:
 *   - weights are bf16 (or 4-bit blocks) widened exactly to double;
 *   - the attention KV cache is stored as bf16 ("Beating llama.cpp from Scratch
 *     on Consumer AMD", section "The Beast: Qwen 3.5 Hybrid Architecture");
 *   - the Gated DeltaNet recurrent state is stored as FP32 (same section).
 * Where a float decides an integer (the bf16 code of a cached K/V element, the
 * greedy argmax, the router's top-k), the decision is taken on the value
 * rounded to FP32, the precision of the CUDA kernels.
 *
 * Parity pins: every function below is pinned by tests under tests/ against
 * closed forms, invariants, special cases or brute force.  The whole-model
 * composition (orc_forward_token) has no worked example on the pages; it is
 * pinned by a closed form in vectors at the first two positions of a fresh
 * sequence, and beyond them by its component pins.
 */
#ifndef HYBRID_ORACLE_H
#define HYBRID_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A weight matrix [rows][cols], bf16 or 4-bit blocks of 32 along cols. */
typedef struct {
  int32_t fmt;            /* 0: bf16; 1: 4-bit blocks of 32 */
  int64_t rows;
  int64_t cols;
  const uint16_t* bf16;   /* fmt 0: [rows][cols] bf16 bits */
  const uint8_t* qs;      /* fmt 1: [rows][cols/2] packed nibbles */
  const uint16_t* scales; /* fmt 1: [rows][cols/32] fp16 bits */
} orc_mat;

typedef struct {
  int32_t n_layers, hidden, vocab, ffn; /* ffn == 0: MoE FFN */
  int32_t gdn_heads, gdn_dk, gdn_dv, conv_k;
  int32_t attn_q_heads, attn_kv_heads, head_dim;
  int32_t n_experts, top_k, expert_ffn, shared_ffn;
  double rms_eps, rope_theta;
  const uint8_t* is_attn; /* [n_layers]: 1 = GQA attention layer, 0 = Gated DeltaNet */
  int32_t kv_format;      /* 0: bf16 KV cache; 1: int8 codes with one FP32 scale per cached vector */
} orc_config;

typedef struct {
  const float* norm1;     /* [H] */
  orc_mat w_in;           /* GDN: q|k|v|a|b rows; attention: q|k|v rows */
  const uint16_t* conv_w; /* GDN only: bf16 [2*nh*dk + nh*dv][conv_k] */
  orc_mat w_o;
  const float* norm2;     /* [H] */
  orc_mat w_gate, w_up, w_down;           /* dense FFN */
  orc_mat router;                         /* MoE: [E+1][H] */
  orc_mat exp_gate, exp_up;               /* MoE: [E*Fe][H] */
  orc_mat exp_down;                       /* MoE: [E*H][Fe] */
  orc_mat sh_gate, sh_up, sh_down;        /* MoE shared expert */
} orc_layer;

typedef struct {
  const uint16_t* embed;  /* bf16 [V][H] */
  const float* final_norm;
  orc_mat lm_head;        /* [V][H] */
  const orc_layer* layers;
} orc_weights;

/* Per-sequence cache, owned by the oracle (orc_cache_create / destroy). */
typedef struct {
  int32_t len, capacity;
  float* gdn_state;    /* per GDN layer: [nh][dv][dk] FP32 */
  double* conv_state;  /* per GDN layer: [conv_k-1][channels], oldest first */
  uint16_t* k_cache;   /* per attention layer: [nkv][capacity][hd] bf16 (kv_format 0) */
  uint16_t* v_cache;
  int8_t* k_q;         /* kv_format 1, per attention layer: codes [nkv][capacity][hd] */
  int8_t* v_q;
  float* k_s;          /* kv_format 1, per attention layer: scales [nkv][capacity] */
  float* v_s;
} orc_cache;

/* --- scalar formats ------------------------------------------------------ */
double orc_bf16_to_double(uint16_t b);
uint16_t orc_to_bf16(double x);           /* x rounded to FP32, then bf16 RNE */
double orc_fp16_to_double(uint16_t h);
double orc_q4_value(const orc_mat* m, int64_t r, int64_t c);

/* --- building blocks ----------------------------------------------------- */
void orc_mat_row(const orc_mat* m, int64_t r, double* out);
void orc_gemv(const orc_mat* m, const double* x, double* y);
void orc_rmsnorm(const double* x, const float* g, int32_t n, double eps, double* y);
void orc_l2norm(double* v, int32_t n, double eps);
double orc_sigmoid(double x);
double orc_silu(double x);
void orc_rope(double* v, int32_t hd, int32_t pos, double theta);
void orc_conv_step(const double* u, double* state, const uint16_t* w, int32_t channels, int32_t k, double* out);
void orc_gdn_step(float* S, int32_t dk, int32_t dv, const double* q, const double* k, const double* v,
                  double alpha, double beta, double* o);
void orc_attention(const double* q, const uint16_t* K, const uint16_t* V, int32_t nq, int32_t nkv, int32_t hd,
                   int32_t cap, int32_t npos, double* o);
void orc_attention_split(const double* q, const uint16_t* K, const uint16_t* V, int32_t nq, int32_t nkv,
                         int32_t hd, int32_t cap, int32_t npos, int32_t nsplit, double* o);
void orc_quant_i8(const double* x, int32_t n, int8_t* q, float* scale);
void orc_attention_i8(const double* q, const int8_t* Kq, const float* Ks, const int8_t* Vq, const float* Vs,
                      int32_t nq, int32_t nkv, int32_t hd, int32_t cap, int32_t npos, double* o);
int32_t orc_argmax(const double* v, int64_t n);
void orc_topk(const double* r, int32_t n, int32_t k, int32_t* ids);
void orc_softmax(const double* x, int32_t n, double* p);

/* --- whole model ---------------------------------------------------------- */
int orc_cache_create(const orc_config* cfg, int32_t capacity, orc_cache* out);
void orc_cache_destroy(orc_cache* c);
void orc_cache_reset(const orc_config* cfg, orc_cache* c);

/* One token at position cache->len; on return cache->len has grown by one.
 * logits: [V] (required).  hidden: [n_layers][H] residual after each layer
 * (nullable).  router_ids: [n_layers][top_k], router_logits: [n_layers][E+1]
 * (nullable; MoE layers only).  Returns 0, or -1 when the cache is full. */
int orc_forward_token(const orc_config* cfg, const orc_weights* w, orc_cache* c, int32_t token, double* logits,
                      double* hidden, int32_t* router_ids, double* router_logits);

/* Number of OpenMP threads the oracle uses (1 when built without OpenMP). */
int orc_threads(void);
void orc_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif

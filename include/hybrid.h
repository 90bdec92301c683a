/* hybrid.h -- C ABI of the GB300 (sm_103a) decode library for hybrid
 * Gated-DeltaNet / GQA-attention / MoE transformers.
 *
 * The library runs the single-token decode step (batch 1) of such a model on
 * one GPU: fused RMSNorm + bf16 GEMV chains, an in-place Gated DeltaNet state
 * update, split-KV GQA attention with a log-sum-exp combine, a fused router
 * top-k with expert-gathered GEMV, and a greedy argmax, all captured into one
 * CUDA graph per decode step.
 *
 * Sources (pages this interface follows):
 *   [Strata] "Beating llama.cpp from Scratch on Consumer AMD: Building Strata,
 *            a Native Rust + HIP Local AI Engine"
 *   [14h]    "Fourteen hours to 100 tokens per second"
 *   [Flash]  "Flash-Next on Strix Halo"
 *
 * Conventions for every call:
 *   - Pointers named *_dev are CUDA device pointers; *_host are host pointers.
 *     Weights are borrowed (caller-owned device memory that must outlive the
 *     model); caches and scratch are owned by the library; output buffers are
 *     caller-owned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are stream-ordered and do not synchronise unless stated.
 *   - Every call returns HY_OK (0) or an HY_ERR_* code; a text description of
 *     the last error of the calling thread is available from hy_last_error().
 *     No call aborts the process.
 *   - All matrices are row-major; bf16 values are IEEE bfloat16 bit patterns
 *     (uint16).  Every weight pointer must be 16-byte aligned and every row
 *     length (in bytes) a multiple of 16.
 */
#ifndef HYBRID_H
#define HYBRID_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
#define HY_OK 0
#define HY_ERR_ARG 1          /* invalid argument (null pointer, bad shape, misalignment) */
#define HY_ERR_CAPACITY 2     /* a sequence would grow past its cache capacity; nothing was launched */
#define HY_ERR_CUDA 3         /* a CUDA runtime call failed */
#define HY_ERR_DEVICE_GUARD 4 /* a device-side guard fired (see hy_check_device) */
#define HY_ERR_UNSUPPORTED 5  /* a shape or option the library does not handle */
#define HY_ERR_NOMEM 6        /* device allocation failed */

/* Device guard bits reported by hy_check_device(). */
#define HY_GUARD_WAIT_TIMEOUT 1u  /* a bounded in-kernel wait gave up */
#define HY_GUARD_BAD_INDEX 2u     /* a token or expert id was out of range */
#define HY_GUARD_BAD_POSITION 4u  /* a position was outside the cache capacity */

/* Model flags. */
#define HY_FLAG_DEBUG 1u    /* keep per-layer hidden states and router results of the last step */
#define HY_FLAG_NO_GRAPH 2u /* launch kernels one by one instead of replaying a CUDA graph */
#define HY_FLAG_NO_PDL 4u   /* no programmatic dependent launch between kernels */
#define HY_FLAG_TOKEN_PREFILL 16u /* run prompts token by token through the decode step (no chunked prefill) */
/* Other flag bits are refused (HY_ERR_ARG). */

/* Model shape.  [Strata] "The Beast: Qwen 3.5 Hybrid Architecture": Gated
 * DeltaNet layers with a fixed FP32 state plus full GQA layers with a bf16 KV
 * cache; [14h] "Starting point": MoE FFN with 256 experts, top-8 plus one
 * shared expert. */
typedef struct {
  int32_t n_layers;        /* <= 64 */
  int32_t hidden;          /* H */
  int32_t vocab;           /* V */
  int32_t ffn;             /* dense SwiGLU width F; 0 selects the MoE FFN */
  int32_t gdn_heads;       /* Gated DeltaNet heads nh */
  int32_t gdn_dk;          /* key dim (64, 128 or 256) */
  int32_t gdn_dv;          /* value dim */
  int32_t conv_k;          /* causal conv width (4) */
  int32_t attn_q_heads;    /* nq */
  int32_t attn_kv_heads;   /* nkv (nq % nkv == 0, nq / nkv <= 8) */
  int32_t head_dim;        /* 64, 128 or 256 */
  uint64_t attn_layer_mask;/* bit l set: layer l is GQA attention, else Gated DeltaNet */
  int32_t n_experts;       /* E (MoE), 1..511 (HY_ERR_UNSUPPORTED above) */
  int32_t top_k;           /* k (MoE, <= 16) */
  int32_t expert_ffn;      /* Fe (MoE) */
  int32_t shared_ffn;      /* Fs (MoE shared expert) */
  float rms_eps;           /* RMSNorm epsilon */
  float rope_theta;        /* RoPE base */
  int32_t weight_format;   /* 0 = bf16; 1 = 4-bit blocks of 32 for the linear weights (see hy_tensor) */
  int32_t attn_splits;     /* split-KV chunks per kv head; 0 = chosen from the SM count */
  uint32_t flags;          /* HY_FLAG_* */
  int32_t kv_format;       /* 0 = bf16 KV cache; 1 = int8 codes with one FP32 scale per cached k or v vector */
} hy_config;

/* One linear weight [rows][cols]: bf16 in `w` (`scales` unused), or with
 * weight_format 1 packed 4-bit blocks of 32 along cols in `w` ([rows][cols/2]
 * bytes; byte i of a block holds element i in its low nibble and element
 * i + 16 in its high nibble, each stored as value + 8) and one fp16 scale per
 * block in `scales` ([rows][cols/32]): w = scale * (nibble - 8) ([Flash]
 * "Correctness fixes").  The router, the conv taps and the embedding stay
 * bf16 in 4-bit models. */
typedef struct {
  const void* w;
  const void* scales;
} hy_tensor;

/* Weights of one layer (device pointers).  Layouts:
 *   norm1, norm2 : float [H]                    RMSNorm gains
 *   w_in  GDN    : [2*nh*dk + nh*dv + 2*nh][H]  rows q | k | v | a | b
 *         attn   : [(nq + 2*nkv)*hd][H]         rows q | k | v
 *   conv_w (GDN) : bf16 [2*nh*dk + nh*dv][conv_k]  taps, the last on the current input
 *   w_o    GDN   : [H][nh*dv];  attn: [H][nq*hd]
 *   dense FFN    : w_gate, w_up [F][H], w_down [H][F]
 *   MoE FFN      : router bf16 [E + 1][H] (row E gates the shared expert),
 *                  exp_gate, exp_up [E][Fe][H], exp_down [E][H][Fe],
 *                  sh_gate, sh_up [Fs][H], sh_down [H][Fs] */
typedef struct {
  const float* norm1;
  hy_tensor w_in;
  const void* conv_w;
  hy_tensor w_o;
  const float* norm2;
  hy_tensor w_gate, w_up, w_down;
  const void* router;
  hy_tensor exp_gate, exp_up, exp_down;
  hy_tensor sh_gate, sh_up, sh_down;
} hy_layer_weights;

typedef struct {
  const void* embed;             /* bf16 [V][H] */
  const float* final_norm;       /* float [H] */
  hy_tensor lm_head;             /* [V][H] */
  const hy_layer_weights* layers;/* host array [n_layers]; copied by hy_model_create */
} hy_weights;

typedef struct hy_model hy_model;
typedef struct hy_cache hy_cache;

/* Text of the calling thread's last error ("" if none). */
const char* hy_last_error(void);

/* Validate the config and weight pointers and record them (borrowed) for
 * the current CUDA device.  No graph is captured yet.  [Strata] "Why Safe
 * Rust with HIP?": raw device pointers confined behind one narrow interface. */
int hy_model_create(const hy_config* cfg, const hy_weights* weights, hy_model** out);
void hy_model_free(hy_model* m);

/* Allocate, for up to max_seqs sequences, the per-sequence KV cache (bf16
 * [nkv][capacity][hd] per attention layer), the Gated DeltaNet state (FP32
 * [nh][dv][dk] per GDN layer), the conv state and the decode scratch, all
 * zeroed, all owned by the library.  capacity_host[s] is the most tokens
 * sequence s may hold ([Strata] "What Broke" section 2: a pre-allocated cache
 * with a hard bound).  Synchronises the device. */
int hy_cache_alloc(hy_model* m, int32_t max_seqs, const int32_t* capacity_host, hy_cache** out);
void hy_cache_free(hy_cache* c);

/* hy_cache_alloc with a paged KV cache ("hanzo-engine: A Portable Single-Binary
 * LLM Inference Engine...", section "System Architecture": paged KV cache and
 * continuous batching).  Instead of a slab of capacity_host[s] positions per
 * sequence, K and V live in one pool of pool_pages pages of page_tokens
 * positions (a positive multiple of 128), each holding every attention
 * layer's K and V of page_tokens consecutive positions of one sequence.  A
 * sequence takes pages as it grows (hy_prefill, hy_decode_step and
 * hy_seq_fill_synthetic take them, on `stream`, before they launch anything;
 * HY_ERR_CAPACITY, with nothing launched and no page taken, when the pool is
 * short) and gives them back on hy_seq_reset, so sequences of any mix of
 * lengths share the pool and may join or leave a batch between steps.
 * capacity_host[s] still bounds each sequence's length.  Recurrent state and
 * scratch are as for hy_cache_alloc.  bf16 K/V only (HY_ERR_UNSUPPORTED with
 * kv_format 1). */
int hy_cache_alloc_paged(hy_model* m, int32_t max_seqs, const int32_t* capacity_host, int32_t page_tokens,
                         int32_t pool_pages, hy_cache** out);
/* Pages left in the pool of a paged cache, or -1 for a cache without pages. */
int32_t hy_cache_free_pages(const hy_cache* c);

/* Forget sequence `seq`: length 0, recurrent and conv state zeroed
 * (stream-ordered). */
int hy_seq_reset(hy_cache* c, int32_t seq, void* stream);

/* Tokens held by sequence `seq`, or -1 for a bad handle.  A sequence is
 * exhausted when hy_seq_len == its capacity ([Strata] "What Broke" section 2,
 * context_exhausted()). */
int32_t hy_seq_len(const hy_cache* c, int32_t seq);
int32_t hy_seq_capacity(const hy_cache* c, int32_t seq);

/* Give sequence `seq` `len` positions of synthetic cache contents (KV rows
 * [0, len) of every attention layer filled with seeded bf16 values in
 * [-1, 1), the DeltaNet states with seeded values in [-0.01, 0.01), the conv
 * rings zeroed), as if a prompt of that length had been run.  A decode step's
 * cost depends on the lengths only, so benchmarks of long or ragged contexts
 * use this instead of a token-by-token prefill; outputs after it are not
 * those of any prompt.  HY_ERR_CAPACITY if len exceeds the capacity.
 * Stream-ordered.
 *
 * The values, exactly (all integers mod 2^64; mix64 is the SplitMix64 output
 * function; GOLDEN = 0x9E3779B97F4A7C15): value i of the stream with key k is
 *   z = mix64(k + (i + 1) * GOLDEN),
 *   v = (float)(z >> 40) * 2^-23 - 1, times the float scale (FP32 arithmetic).
 * K (w = 0) and V (w = 1) of attention layer a (0-based among the attention
 * layers), kv head g: key seed * 1000003 + (2 a + w) * 64 + g, scale 1, element
 * (row r, column j) is value r * head_dim + j rounded to bf16 (nearest even).
 * The DeltaNet states of all DeltaNet layers, in the order
 * [layer][head][dv][dk]: one stream with key seed * 1000003 + 977, scale 0.01.
 * A host copy of the same values lets a CPU reference start from this state. */
int hy_seq_fill_synthetic(hy_cache* c, int32_t seq, int32_t len, uint64_t seed, void* stream);

/* Distinct routed experts the batched MoE steps (hy_decode_step with several
 * sequences, or 4-bit weights) read since the last call, summed over layers
 * and steps: each layer reads the union of its tokens' picks once.  Resets
 * the count.  Batch-1 bf16 steps read top_k per layer and do not count.
 * Synchronises `stream`.  [14h] "Eight levers that worked" (expert-gathered
 * GEMVs read only the selected experts). */
int hy_experts_read(hy_cache* c, void* stream, uint64_t* total_out);

/* Kernels the last recorded decode step launches (one per operation); 0
 * before any step. */
int32_t hy_step_kernels(const hy_cache* c);

/* Split-KV chunks per kv head that a batch-1 decode step of sequence `seq`
 * uses: hy_config.attn_splits when set, else one CTA per SM across the kv
 * heads, or, for a cache of 16384 positions or more with up to 4 query heads
 * per kv head, 64 splits run as two CTAs per SM.  0 for a bad sequence index
 * or a model without attention layers.  (A step of several sequences with
 * the automatic count shares the step's splits among them in proportion to
 * their lengths, worked out on the device at every step.) */
int32_t hy_step_splits(const hy_cache* c, int32_t seq);

/* Run the n prompt tokens tokens_dev[0..n) of sequence `seq` through the
 * model at positions len .. len+n-1, filling its caches.  logits_dev
 * (nullable) receives the FP32 logits [V] of the last token.
 * HY_ERR_CAPACITY (nothing launched) if len + n > capacity.  bf16 models
 * (dense and MoE) with the bf16 cache run the prompt in chunks of up to 2048
 * tokens (HY_PREFILL_CHUNK in the environment overrides) through tensor-core
 * GEMMs (tcgen05, the activations as bf16 hi + lo parts, FP32 accumulation;
 * the MoE experts as grouped GEMMs over the chunk's picks) and prompt
 * kernels of the mixers, with buffers the library allocates at the first
 * such call; the caches it leaves equal those of a token-by-token prefill
 * within rounding.  4-bit models, int8-cache models and models created with
 * HY_FLAG_TOKEN_PREFILL run the prompt one position at a time through the
 * decode step.  [Strata] "Act 1" (batched chunk kernels: one launch per layer
 * for all prompt tokens). */
int hy_prefill(hy_model* m, hy_cache* c, int32_t seq, const int32_t* tokens_dev, int32_t n, float* logits_dev,
               void* stream);

/* One greedy decode step for the distinct sequences seqs_host[0..nseq)
 * (1 <= nseq <= 8): consumes tokens_dev[i] at position len(seqs[i]), writes
 * the FP32 logits [nseq][V] to logits_dev (nullable) and the argmax token id
 * (lowest index on ties) to ids_dev[i], then len += 1 for each.  With
 * nseq > 1 (and always for 4-bit models) every weight is read once for all
 * the sequences: the projections run as batched tensor-core GEMVs, the MoE
 * FFN over the union of the experts the tokens selected ([Strata] "Act 5":
 * batched decode rows).  The first call for a given (sequence list,
 * logits_dev, ids_dev) captures a CUDA graph; later calls replay it: one
 * graph launch per step ([Strata] "Act 0", pass 3).  HY_ERR_CAPACITY
 * (nothing launched) if a sequence is full; HY_ERR_UNSUPPORTED (nothing
 * launched) if a batched MoE step would hold more than 64 routed picks
 * (nseq x top_k > 64). */
int hy_decode_step(hy_model* m, hy_cache* c, const int32_t* seqs_host, int32_t nseq, const int32_t* tokens_dev,
                   float* logits_dev, int32_t* ids_dev, void* stream);

/* hy_decode_step with host buffers: copies tokens_host to the device, runs
 * the step, copies ids (and logits when logits_host is not NULL) back, and
 * synchronises `stream` before returning. */
int hy_decode_step_host(hy_model* m, hy_cache* c, const int32_t* seqs_host, int32_t nseq, const int32_t* tokens_host,
                        float* logits_host, int32_t* ids_host, void* stream);

/* Synchronise `stream` and read (then clear) the device guard word of the
 * cache; *bits_out receives HY_GUARD_* bits.  Returns HY_ERR_DEVICE_GUARD
 * when any bit was set. */
int hy_check_device(hy_cache* c, void* stream, uint32_t* bits_out);

/* With HY_FLAG_DEBUG: copy the residual stream after layer `layer` of the
 * last step (FP32 [H]) into dst_dev. */
int hy_debug_hidden(hy_cache* c, int32_t layer, float* dst_dev, void* stream);
/* With HY_FLAG_DEBUG, MoE layers: the last step's router logits (FP32
 * [E + 1]) and selected experts (int32 [top_k], in selection order). */
int hy_debug_router(hy_cache* c, int32_t layer, float* logits_dev, int32_t* ids_dev, void* stream);

/* ------------------------------------------------------------- single ops
 * The kernels of the decode step, callable on their own (used by tests and
 * measurements).  All device pointers, stream-ordered.  Their kernels report
 * device-side refusals (a position at or past the cache capacity, a bounded
 * wait that gave up) in a guard word, not in the return code, which only
 * covers what the host checks before launching: read it with
 * hy_op_check_device. */

/* Synchronise `stream`, then read and clear the guard words of the single-op
 * calls on the current device (every hy_op_* call, and the allocation-free
 * attention, whose word each of its calls clears first, so that it reports
 * that call's refusals only).  *bits_out (nullable) receives the HY_GUARD_*
 * bits.  Returns HY_ERR_DEVICE_GUARD when any bit was set.  Allocates
 * nothing. */
int hy_op_check_device(void* stream, uint32_t* bits_out);

/* y = W * xhat, xhat = x (norm_g == NULL) or RMSNorm(x) * norm_g with eps:
 * W bf16 [rows][cols], x, y FP32.  accumulate != 0: y += W * xhat.
 * [Strata] "Act 0", pass 3 (vectorised GEMV for M = 1 decode). */
int hy_op_gemv(const void* W_dev, int32_t rows, int32_t cols, const float* x_dev, const float* norm_g_dev, float eps,
               float* y_dev, int32_t accumulate, void* stream);

/* h = silu(Wg * xhat) * (Wu * xhat), Wg, Wu bf16 [rows][cols].  [14h] "Eight
 * levers that worked" (silu(gate) * x in the gated kernel). */
int hy_op_gemv_swiglu(const void* Wg_dev, const void* Wu_dev, int32_t rows, int32_t cols, const float* x_dev,
                      const float* norm_g_dev, float eps, float* h_dev, void* stream);

/* Batched GEMV over `batch` (1..8) token vectors through one weight stream:
 * y[b] = W * xhat[b] (accumulate != 0: y[b] += ...), or with w_up non-null
 * y[b] = silu(W * xhat[b]) * (W_up * xhat[b]).  xhat[b] = x[b], or its
 * RMSNorm times norm_g.  x_dev [batch][ldx], y_dev [batch][ldy] FP32.
 * weight_format 0: bf16 W.w [rows][cols], cols % 64 == 0; 1: 4-bit blocks of
 * 32 along cols, W.w packed nibbles [rows][cols/2] (byte i of a block holds
 * elements i and i+16 as value+8), W.scales fp16 [rows][cols/32],
 * cols % 256 == 0.  Weight pointers 16-byte aligned.  The products run on the
 * tensor cores with xhat rounded to the MMA operand type (bf16 hi + lo parts
 * for bf16 weights, FP16 for 4-bit weights); 4-bit weights are dequantised
 * exactly.  HY_ERR_UNSUPPORTED (nothing launched) for other cols, or when the
 * batch's vectors do not fit the kernel's shared memory (bf16 cols above
 * 5824, or 4672 with w_up; 4-bit cols above 11264, or 8704 with w_up).  [Strata] "Act 5" (batched decode rows),
 * [Flash] "Correctness fixes" (the 4-bit block layout). */
int hy_op_gemv_batch(const hy_tensor* w, const hy_tensor* w_up, int32_t weight_format, int32_t rows, int32_t cols,
                     int32_t batch, const float* x_dev, int32_t ldx, const float* norm_g_dev, float eps, float* y_dev,
                     int32_t ldy, int32_t accumulate, void* stream);

/* Prompt GEMM on the tensor cores: for the M token rows of x (FP32
 * [M][ldx], K columns used), xhat = x or its RMSNorm times norm_g (eps), and
 * y[m][n] = sum_k xhat[m][k] W[n][k] (accumulate != 0: y += ...), W bf16
 * [N][K], y FP32 [M][ldy].  xhat reaches the tensor cores as two bf16 parts
 * hi + lo (relative error ~2^-16) written to workspace_dev
 * (hy_op_gemm_workspace(M, K) bytes, caller-owned, no zeroing needed); the
 * products accumulate in FP32 in tensor memory.  K % 8 == 0.  [Strata]
 * "Act 1" (the prompt through batched kernels, one launch per layer). */
size_t hy_op_gemm_workspace(int32_t M, int32_t K);
int hy_op_gemm(const void* W_dev, int32_t N, int32_t K, int32_t M, const float* x_dev, int32_t ldx,
               const float* norm_g_dev, float eps, float* y_dev, int32_t ldy, int32_t accumulate, void* workspace_dev,
               void* stream);
/* The gate/up pair of the same: h = silu(xhat Wg^T) * (xhat Wu^T), returned
 * as its bf16 hi and lo parts (h ~ hi + lo, relative error ~2^-16) in
 * h_hi_dev, h_lo_dev [M][ldh] (the form the down projection's GEMM takes).
 * [14h] "Eight levers that worked" (silu(gate) * up fused into the GEMM). */
int hy_op_gemm_swiglu(const void* Wg_dev, const void* Wu_dev, int32_t N, int32_t K, int32_t M, const float* x_dev,
                      int32_t ldx, const float* norm_g_dev, float eps, uint16_t* h_hi_dev, uint16_t* h_lo_dev,
                      int32_t ldh, void* workspace_dev, void* stream);

/* MoE FFN of one token in two kernels ([14h] "Eight levers that worked":
 * router top-k fused into the expert-gathered GEMV; "The router with 257
 * rows": the shared expert's sigmoid gate as the router's extra row).
 * hy_op_moe_gateup: from the router logits [n_experts + 1] (the last is the
 * shared expert's gate), every CTA picks the top_k experts (largest logit,
 * lowest index on ties), then h[s * Fe + r] = silu(g) * u of the picked
 * experts' gate / up rows (slots 0..top_k-1, in selection order) and of the
 * shared expert (slot top_k), with xhat = x or RMSNorm(x) * norm_g.  ids_dev
 * [top_k] receives the picks, w_dev [top_k + 1] the softmax over the picked
 * logits and sigmoid of the shared gate.  Expert tensors bf16: exp_gate /
 * exp_up [n_experts][Fe][hidden], sh_gate / sh_up [Fe][hidden]; h FP32
 * [(top_k + 1) * Fe].
 * hy_op_moe_down: y[H] += sum_s w[s] * Wd_s h_s over the picked experts'
 * down matrices (exp_down [n_experts][hidden][Fe]) and the shared expert's
 * (sh_down [hidden][Fe]).  top_k <= 16, n_experts <= 511. */
int hy_op_moe_gateup(const void* exp_gate_dev, const void* exp_up_dev, const void* sh_gate_dev, const void* sh_up_dev,
                     int32_t n_experts, int32_t top_k, int32_t expert_ffn, int32_t hidden,
                     const float* router_logits_dev, const float* x_dev, const float* norm_g_dev, float eps,
                     float* h_dev, int32_t* ids_dev, float* w_dev, void* stream);
int hy_op_moe_down(const void* exp_down_dev, const void* sh_down_dev, int32_t n_experts, int32_t top_k,
                   int32_t expert_ffn, int32_t hidden, const int32_t* ids_dev, const float* w_dev, const float* h_dev,
                   float* y_dev, void* stream);

/* Greedy head: logits = W * xhat (logits_dev nullable), *id_dev = argmax
 * (lowest index on ties).  workspace_dev: hy_op_argmax_workspace() bytes,
 * zeroed before its first use and left zeroed after each call.
 * [Strata] "Act 0", pass 3 (on-device argmax, a 4-byte result). */
size_t hy_op_argmax_workspace(void);
int hy_op_gemv_argmax(const void* W_dev, int32_t rows, int32_t cols, const float* x_dev, const float* norm_g_dev,
                      float eps, float* logits_dev, int32_t* id_dev, void* workspace_dev, void* stream);

/* One Gated DeltaNet decode step of one layer at position *pos_dev:
 * y_dev = projection output [2*nh*dk + nh*dv + 2*nh] (q|k|v|a|b), conv_w
 * bf16 [channels][conv_k], conv_state FP32 ring [conv_k][channels] (slot
 * t % conv_k holds the input of position t), S FP32 [nh][dv][dk] updated in
 * place, o_dev FP32 [nh*dv].  [Strata] "The Beast". */
int hy_op_gdn_step(const float* y_dev, const void* conv_w_dev, float* conv_state_dev, float* S_dev, float* o_dev,
                   int32_t nh, int32_t dk, int32_t dv, int32_t conv_k, const int32_t* pos_dev, void* stream);

/* (cos, sin) of position * theta^(-2i/hd) for positions [0, cap), i < hd/2:
 * table_dev float2 [cap][hd/2] (computed in double, rounded once). */
int hy_op_rope_table(float* table_dev, int32_t cap, int32_t hd, float theta, void* stream);

/* GQA decode attention of one layer at position T = *len_dev: y_dev =
 * projection output [(nq + 2*nkv)*hd] (q|k|v, before RoPE); rotates q and
 * the new k with rope_table_dev, appends bf16 k, v at row T of K_dev, V_dev
 * (bf16 [nkv][cap][hd]), attends over rows [0, T], writes o_dev FP32
 * [nq*hd].  nsplit chunks per kv head (0 = automatic).  workspace_dev:
 * hy_op_attention_workspace() bytes, zeroed before its first use and then
 * passed unmodified to later calls (its counters carry a generation number
 * from call to call).  [Strata] "Act 4" and "What Broke" section 1. */
size_t hy_op_attention_workspace(int32_t nq, int32_t nkv, int32_t hd, int32_t nsplit);
int hy_op_attention(const float* y_dev, void* K_dev, void* V_dev, int32_t cap, int32_t nq, int32_t nkv, int32_t hd,
                    const int32_t* len_dev, const float* rope_table_dev, int32_t nsplit, float* o_dev,
                    void* workspace_dev, void* stream);

/* hy_op_attention over an int8 cache ("hanzo-engine: A Portable Single-Binary
 * LLM Inference Engine...", sections "System Architecture" and "Results":
 * int8 KV, one f32 scale per cached vector).  Kq_dev, Vq_dev: int8 codes
 * [nkv][cap][hd]; Ks_dev, Vs_dev: FP32 scales [nkv][cap4], cap4 = cap rounded
 * up to a multiple of 4 (all four 16-byte aligned).  A cached value is code *
 * scale.  The new k (after RoPE) and v vectors at row T = *len_dev are
 * quantised on the device: a = max |x| (FP32), scale = a / 127, code =
 * round-half-even(x * (127 / a)) clamped to [-127, 127] (a = 0: codes 0,
 * scale 0); they are attended to as stored.  Other arguments as for
 * hy_op_attention (same workspace size). */
int hy_op_attention_i8(const float* y_dev, void* Kq_dev, float* Ks_dev, void* Vq_dev, float* Vs_dev, int32_t cap,
                       int32_t nq, int32_t nkv, int32_t hd, const int32_t* len_dev, const float* rope_table_dev,
                       int32_t nsplit, float* o_dev, void* workspace_dev, void* stream);

/* hy_op_attention without a caller-provided workspace, for callers that
 * cannot allocate device memory: a host framework that owns the whole memory
 * budget through its own pool, a latency path where an allocation and the
 * synchronisation it implies are not allowed, or a plug-in whose host forbids
 * allocations outside its allocator.  The pages have no counterpart of this
 * call; it exists only for such callers.
 *
 * Same arguments, layout and results as hy_op_attention (nsplit <= 0 selects
 * the automatic split count); the scratch (guard
 * word, per-kv-head tickets, per-split partials) lives instead in one fixed
 * device array of HY_NOALLOC_SCRATCH_BYTES that every GPU loading this
 * library holds until the process exits.  The call makes no allocation: it
 * clears the guard word and the tickets on `stream`, then launches.  A
 * position at or past `cap` is refused on the device: the kernel returns
 * without touching o_dev or the cache and sets HY_GUARD_BAD_POSITION, which
 * hy_op_check_device reports until the next call clears it.
 *   - Returns HY_ERR_UNSUPPORTED, launching nothing, when the scratch this
 *     shape needs (hy_op_attention_workspace(nq, nkv, hd, nsplit) bytes, with
 *     nsplit = 0 resolved as hy_op_attention resolves it) exceeds
 *     HY_NOALLOC_SCRATCH_BYTES.
 *   - The first call on a device (the current one) sets up that device: it
 *     looks up the array's device address and the kernels' shared-memory
 *     limits.  Make that first call before any stream capture begins.
 *   - Every call on a device uses the same array, which keeps what the last
 *     call left: calls that can overlap on the GPU (other streams, other host
 *     threads without ordering between them) race and corrupt each other's
 *     results.  Order them on one stream or otherwise serialise them. */
#define HY_NOALLOC_SCRATCH_BYTES (1u << 20)
int hy_op_attention_noalloc(const float* y_dev, void* K_dev, void* V_dev, int32_t cap, int32_t nq, int32_t nkv,
                            int32_t hd, const int32_t* len_dev, const float* rope_table_dev, int32_t nsplit,
                            float* o_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif

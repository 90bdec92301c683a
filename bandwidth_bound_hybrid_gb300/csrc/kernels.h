// Internal launch interface of the decode-step kernels (host side).  Not part
// of the public C ABI (include/hybrid.h); used by engine.cu and capi.cu.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace hy {

// ---------------------------------------------------------------- GDN
namespace gdn {
constexpr int kRowsPerCta = 16;
constexpr int kThreads = 128;
constexpr int kMaxB = 8;
struct Params {
  const float* y;          // projection output: q|k|v|a|b  (conv_channels + 2*nh)
  const uint16_t* conv_w;  // bf16 [channels][conv_k]
  float* conv_state;       // ring of conv_k slots [conv_k][channels]; slot t % conv_k holds input t
  float* S;                // [nh][dv][dk]
  const int* pos;          // position t of the token
  float* o;                // [nh*dv]
  int nh, dk, dv, conv_k;
  unsigned* guard;
  // batch (nb > 0): token z = blockIdx.z uses y + z*ld_y, o + z*ld_o and its
  // own sequence's state, conv ring and position
  int nb, ld_y, ld_o;
  float* S_b[kMaxB];
  float* conv_b[kMaxB];
  const int* pos_b[kMaxB];
};
cudaError_t launch(const Params& p, cudaStream_t st, bool pdl);
}  // namespace gdn

// ---------------------------------------------------------------- GEMV
namespace gemv {

enum Src : int { kSrcDense = 0, kSrcExpertRows = 1, kSrcExpertSegs = 2 };
enum In : int { kInX = 0, kInEmbed = 1, kInMoeZ = 2 };
enum Epi : int { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiArgmax = 3 };

#ifndef HY_GEMV_WARPS
#define HY_GEMV_WARPS 12
#endif
constexpr int kConsumerWarps = HY_GEMV_WARPS;  // compute warps; one more warp issues the copies
constexpr int kThreads = (kConsumerWarps + 1) * 32;
#ifndef HY_GEMV_MAXREG
#define HY_GEMV_MAXREG 112
#endif
// Register cap: 13 warps of 112 leave each SM sub-partition room for a warp of
// a small kernel (the DeltaNet step) launched early by programmatic dependent
// launch, so that it runs beside the GEMV instead of after it.
constexpr int kMaxRegs = HY_GEMV_MAXREG;
constexpr int kMaxStages = 8;
#ifndef HY_GEMV_STAGE_KB
#define HY_GEMV_STAGE_KB 60
#endif
#ifndef HY_GEMV_INFLIGHT_KB
#define HY_GEMV_INFLIGHT_KB 180
#endif
constexpr int kStageTarget = HY_GEMV_STAGE_KB * 1024;  // preferred bytes per pipeline stage
constexpr int kStageCap = HY_GEMV_STAGE_KB * 1024;     // largest preferred minimum tile
constexpr int kInFlight = HY_GEMV_INFLIGHT_KB * 1024;  // bytes kept in flight per CTA in shared memory
constexpr int kPrefetchAhead = 0;           // bytes the L2 prefetch cursor runs ahead of the ring
constexpr int kMaxSmem = 220 * 1024;        // dynamic; leaves room for static shared data
constexpr int kCtasPerSm = 1;
constexpr int kPreStages = 0;               // tiles issued before the input vector is requested
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 512;  // routed experts a router can select from

// Rows of a matrix that CTA b of an ncta-CTA GEMV owns, prefetched into L2 by
// CTA b of the kernel before it: [b*rows/ncta, (b+1)*rows/ncta), at most
// `bytes` from the start of that range.
struct PfSpan {
  const uint8_t* base;
  int rows, row_bytes, ncta, bytes;
};
constexpr int kMaxPfSpans = 3;

struct Params {
  // ---- weights (bf16 rows of C columns)
  const uint8_t* W[2];          // kSrcDense: matrix bases (W[1]: up matrix of a gate/up pair)
  const uint8_t* exp_base[2];   // MoE: routed-expert tensor bases ([E][rows][cols])
  const uint8_t* sh_base[2];    // MoE: shared-expert matrices
  long long exp_stride;         // bytes from one routed expert to the next
  const int* moe_ids;           // [top_k] selected experts
  const float* moe_w;           // [top_k + 1] routing weights; last = shared-expert gate
  int top_k, n_experts;
  int slot_rows;                // kSrcExpertRows: rows per routed expert slot
  int sh_rows;                  // kSrcExpertRows: rows of the shared slot
  int seg_cols;                 // kSrcExpertSegs: columns per expert segment
  int R, C, npair;
  // ---- input
  const float* x;               // kInX: [C]; kInMoeZ: expert activations [(top_k+1)*seg_cols]
  const uint16_t* embed;        // kInEmbed: bf16 [vocab][C]
  const int* tok;               // kInEmbed: token id
  int vocab;
  float* x_out;                 // kInEmbed: residual stream to initialise (CTA 0 writes it)
  const float* norm_g;          // RMSNorm gain; null = no norm
  float eps;
  // ---- output
  float* y;                     // store / residual target / SwiGLU output / logits (nullable for argmax)
  float* part_val;              // argmax partials [ncta]
  int* part_idx;
  unsigned* counter;            // last-CTA ticket (zero between launches)
  int* ids_out;                 // argmax result
  int* len_inc;                 // incremented once after the argmax (nullable)
  const float* router_logits;   // route_here: the router's stored logits [n_experts + 1]
  int* out_ids;                 // route_here: selected experts [top_k] (CTA 0 writes them)
  float* out_w;                 // route_here: routing weights [top_k + 1]
  int* dbg_ids;                 // route_here debug copies (nullable)
  float* dbg_logits;
  int route_here;               // kSrcExpertRows: every CTA picks the experts itself from router_logits (the
                                //   router kernel only stored them); CTA 0 writes out_ids / out_w (and dbg_ids)
  // ---- prefetch
  PfSpan nx[kMaxPfSpans];       // what the next kernels read first (weights known when the step is recorded)
  int n_nx;
  // ---- plan
  int ncta, tile_rows, nchunk, chunk_vecs, stage_bytes, nstages, rows_cta_max, xs_floats, gs_floats;
  int pre_stages;               // tiles issued before griddepcontrol.wait (ahead of the input vector)
  int pf_ahead;                 // L2 prefetch cursor distance in bytes (0 = off)
  unsigned* guard;
};

struct Plan {
  int ncta, tile_rows, nchunk, chunk_vecs, vpl, stage_bytes, nstages, rows_cta_max, xs_floats, gs_floats, smem;
  int pre_stages, pf_ahead;
  bool full;  // every lane's vectors lie inside its column chunk
  bool ok;
};

// Launch plan of an R x C GEMV (npair matrices sharing the input; `norm`: the
// input is RMS-normalised with a gain vector) on nsm SMs.
Plan plan(int R, int C, int npair, int nsm, bool norm);
cudaError_t init();
cudaError_t launch(const Params& p, const Plan& pl, int src, int in, int epi, cudaStream_t st, bool pdl);

}  // namespace gemv


// ---------------------------------------------------------------- attention
namespace attn {
constexpr int kThreads = 288;  // 8 compute warps + 1 copy warp
constexpr int kRing = 6;       // ring stages, one K or V tile each
struct Params {
  const float* y;          // projection output: q|k|v
  uint16_t* K;             // bf16 [nkv][cap][hd]; with kv8: int8 codes [nkv][cap][hd] (bytes)
  uint16_t* V;
  int kv8;                 // int8 cache: one FP32 scale per cached vector in Ks / Vs [nkv][cap_s]
  float* Ks;
  float* Vs;
  int cap_s;               // scale row stride (a multiple of 4)
  // paged cache (pages != null): row r of kv head g is at K + pages[r / page_tokens] * page_elems
  // + (g * page_tokens + r % page_tokens) * hd; K, V point at this layer's K or V block of page 0
  const int* pages;
  int page_tokens;
  long long page_elems;
  const int* len;          // position of the new token (= cached rows)
  const float2* rope;      // [>= cap][hd/2] (cos, sin) of position * theta^(-2i/hd)
  int cap, nq, nkv, hd, nsplit;
  float scale;
  float* part;             // [nkv][nsplit][G][hd + 2]
  unsigned* counter;       // [nkv]: arrivals in bits 0-15 (zero between launches), a generation above
  int mergers;            // set by launch(): the last `mergers` CTAs of a kv head merge its partials
  float* o;                // [nq*hd]
  unsigned* guard;
  // batch (nb > 0): token z = blockIdx.z uses y + z*ld_y, o + z*ld_o,
  // part + z*ld_part, counter + z*nkv and its own sequence's cache
  int nb, ld_y, ld_o;
  // batch spread (spread > 0, nb > 0): the grid is nkv x spread; its rows are
  // the batch's splits, each token taking a share in proportion to its cache
  // length, worked out on the device from len_b (nsplit is then per token);
  // ld_part must hold spread - nb + 1 splits
  int spread;
  long long ld_part;
  uint16_t* K_b[8];
  uint16_t* V_b[8];
  float* Ks_b[8];
  float* Vs_b[8];
  const int* pages_b[8];
  const int* len_b[8];
  int cap_b[8];
  int cap_s_b[8];
};
size_t part_floats(int nq, int nkv, int hd, int nsplit);
int auto_splits(int nkv, int nsm);   // the single ops' automatic count
int step_splits(int nkv, int nsm);   // the decode step's
int long_context_splits(int nq, int nkv, int nsm);  // for caches of kLongContext positions or more
constexpr int kLongContext = 16384;
cudaError_t init();
cudaError_t launch(const Params& p, cudaStream_t st, bool pdl);
cudaError_t rope_table(float2* tab, int cap, int hd, double theta, cudaStream_t st);
}  // namespace attn

// ---------------------------------------------------------------- batched GEMV
// Up to kMaxB token vectors through one weight stream (tensor-core MMA), bf16
// or 4-bit block weights.
namespace bgemv {
constexpr int kWarps = 8;
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kMaxB = 8;
constexpr int kTileRows = 16;
constexpr int kMaxStages = 8;
constexpr int kInFlight = 160 * 1024;
constexpr int kMaxSmem = 220 * 1024;
enum Fmt : int { kFmtBf16 = 0, kFmtQ4 = 1 };
enum Src : int { kSrcDense = 0, kSrcUnionRows = 1, kSrcUnionDown = 2 };
enum In : int { kInX = 0, kInEmbed = 1 };
enum Epi : int { kEpiStore = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiArgmax = 3 };
constexpr int kMaxUnion = 64;  // distinct routed experts of one step (top_k * batch at most)
struct Params {
  int fmt, src, in, epi;
  // ---- MoE over the union of the experts the batch selected (src != kSrcDense)
  //   kSrcUnionRows: virtual rows u * slot_rows + r, u < n_union: routed expert
  //     union_ids[u]; u == n_union: the shared expert (R = (n_union + 1) * slot_rows)
  //   kSrcUnionDown: units (u, a row block of R); the input of unit u is
  //     x + b * ldx + u * C; outputs go to part_out[(b * (top_k + 1) + slot) * R + row]
  //     for the tokens b whose slot slot_of[u * kMaxB + b] >= 0
  const uint8_t* exp_base[2];
  const uint16_t* exp_scale[2];
  long long exp_stride, exp_sstride;  // bytes from one routed expert to the next (weights, scales)
  const uint8_t* sh_base[2];
  const uint16_t* sh_scale[2];
  const int* union_ids;
  const int* n_union;
  const int* slot_of;
  int slot_rows, top_k;
  float* part_out;
  const uint8_t* W[2];      // bf16 [R][C] or packed nibbles [R][C/2] (W[1]: up matrix of a gate/up pair)
  const uint16_t* S[2];     // 4-bit: fp16 scales [R][C/32]
  int R, C, B;
  int ldw;                  // kSrcDense: elements from one weight row to the next (0: C); C columns are used
  const float* x;           // kInX: [B][ldx]
  int ldx;
  const uint16_t* embed;    // kInEmbed: bf16 [vocab][C]
  const int* tok;           // kInEmbed: [B]
  int vocab;
  float* x_out;             // kInEmbed: residual streams to initialise [B][ldx_out] (CTA 0)
  int ldx_out;
  const float* norm_g;      // per-token RMSNorm gain (null: none)
  float eps;
  float* y;                 // [B][ldy]: store / residual / SwiGLU / logits (nullable for argmax)
  int ldy;
  float* part_val;          // argmax partials [ncta][kMaxB]
  int* part_idx;
  unsigned* counter;        // argmax ticket (zero between launches)
  int* ids_out;             // [B]
  int* len_inc[kMaxB];      // per token, incremented after the argmax (nullable)
  int n_exp;                // union sources: routed experts in the expert tensors
  // ---- kSrcUnionRows with route_here: every CTA routes the batch itself from
  // the stored router logits r_logits [B][r_ld] before its copy lane requests
  // expert rows (top_k of the r_E logits per token, FP32 compare, lowest index
  // on ties; softmax over the picks; shared gate sigmoid(logit r_E)); CTA 0
  // publishes r_ids [B][top_k] (nullable), r_w [B][top_k + 1], and the union
  // of the picks (ascending) with its slot map in union_ids / n_union / slot_of
  int* r_ids;
  float* r_w;
  int r_E;
  int route_here;
  const float* r_logits;
  int r_ld;
  unsigned long long* union_count;  // routing publishers add the union size (routed experts read) here (nullable)
  int ncta, nstages;        // from the plan
  int gw, ks;               // row groups of 16 x strip lanes of the 8 compute warps (gw * ks = 8)
  unsigned* guard;
};
struct Plan {
  int ncta, nstages, smem, gw, ks;
  bool ok;
};
// R: rows to spread over the SMs (for a union source, the rows of the
// expected union); row_mult: a multiple of the row block that blocks must
// divide (the rows of one expert of a union source), 0 for a dense matrix.
// C must be a multiple of 256 (4-bit) or 64 (bf16).
Plan plan(int R, int C, int fmt, int epi, int nsm, int row_mult = 0);
cudaError_t init();
cudaError_t launch(const Params& p, const Plan& pl, cudaStream_t st, bool pdl);

// y[b][row] += sum_{k <= top_k} w[b][k] * part[(b * (top_k + 1) + k) * R + row]
cudaError_t moe_reduce(float* y, int ldy, const float* part, const float* w, int R, int B, int top_k, cudaStream_t st,
                       bool pdl);
}  // namespace bgemv

// ---------------------------------------------------------------- prompt GEMM
// Y[m][n] = sum_k A[m][k] W[n][k] on the tensor cores (tcgen05), with the
// FP32 activations as two bf16 parts A_hi + A_lo (gemm.cu).
namespace gemm {
enum Epi : int { kEpiStore = 0, kEpiResid = 1, kEpiSwigluSplit = 2 };
struct Params {
  int M, N, K, epi;
  float* y;             // store / residual: FP32 [M][ldy]
  int ldy;
  uint16_t* h_hi;       // SwiGLU: silu(A Wg^T) * (A Wu^T) as bf16 hi / lo parts [M][ldh]
  uint16_t* h_lo;
  int ldh;
  unsigned* guard;
  // grouped (tiles != null): row tile i of the grid is tiles[3i .. 3i+2] = {first A row, rows (<= 128),
  // group g}; its W rows are g * w_group_rows + n (W holds n_groups * w_group_rows rows); output rows are
  // A's; tiles i >= *ntiles do nothing.  M = rows of A (and of the output).
  const int* tiles;
  const int* ntiles;
  int max_tiles, w_group_rows, n_groups;
};
cudaError_t init();
bool supported(int M, int N, int K);
// a_hi, a_lo: bf16 [M][lda]; w0 (and the up matrix w1 for SwiGLU): bf16 [N][ldw].
cudaError_t launch(const Params& p, const uint16_t* a_hi, const uint16_t* a_lo, int lda, const uint16_t* w0,
                   const uint16_t* w1, int ldw, cudaStream_t st);
// rows of x -> RMSNorm with gain g (or none when g is null) -> bf16 hi / lo parts.
cudaError_t norm_split(const float* x, int ld_x, const float* g, float eps, int rows, int cols, uint16_t* hi,
                       uint16_t* lo, int ld_out, cudaStream_t st);
}  // namespace gemm

// ---------------------------------------------------------------- prompt MoE
// The MoE FFN of a chunk of n prompt tokens (moe_prefill.cu), around the
// router GEMM, the grouped expert GEMMs and the shared expert's GEMMs.
namespace moepf {
constexpr int kTileRows = 128;  // rows of a grouped GEMM tile
// Routing of every token: logits [n][ldl] (E routed + the shared gate at E) ->
// ids [n][K] (top K, descending, lowest index on ties) and weights [n][K+1]
// (softmax over the picks; last: sigmoid of the shared gate).
cudaError_t route(const float* logits, int ldl, int n, int E, int K, int* ids, float* w, cudaStream_t st);
// Tokens grouped by expert, in token order (deterministic): pos_of[t*K+k] is
// the gathered row of pick (t, k), tok_of[row] its token; tiles / ntiles: the
// grouped GEMM's row tiles {first row, rows, expert} (at most
// max_tiles(n, E, K)).  One CTA.
int max_tiles(int n, int E, int K);
cudaError_t bucket(const int* ids, int n, int E, int K, int* pos_of, int* tok_of, int* tiles, int* ntiles,
                   unsigned* guard, cudaStream_t st);
// Gathered activations: rows [n*K] of hi / lo (ld) = rows tok_of[r] of src_hi / src_lo.
cudaError_t gather(const uint16_t* src_hi, const uint16_t* src_lo, int ld, int cols, const int* tok_of, int rows,
                   uint16_t* dst_hi, uint16_t* dst_lo, cudaStream_t st);
// x[t] += sum_k w[t][k] Ye[pos_of[t*K+k]] + w[t][K] Ysh[t], in that order.
cudaError_t combine(float* x, int H, int n, int K, const float* w, const int* pos_of, const float* Ye,
                    const float* Ysh, cudaStream_t st);
}  // namespace moepf

// ---------------------------------------------------------------- prompt mixers
// The chunk of n prompt tokens at positions t0 .. t0+n-1 of one sequence
// (prefill.cu).  Mixer outputs are written as bf16 hi / lo parts [n][ldo], the
// A operand of the output projection's GEMM.
namespace prefill {
struct GdnArgs {
  const float* Y;          // projection rows q|k|v|a|b of the chunk [n][ldy]
  int ldy;
  const uint16_t* conv_w;  // bf16 [channels][conv_k]
  float* ring;             // conv ring [conv_k][channels] (inputs of the positions before t0; updated)
  float* S;                // state [nh][dv][dk], updated in place
  float* Qn;               // scratch: normalised, scaled q [n][nh][dk]
  float* Kn;               // scratch: normalised k [n][nh][dk]
  float* V;                // scratch: conv outputs of v [n][nh][dv]
  float* AB;               // scratch: alpha, beta [n][nh][2]
  uint16_t* O_hi;
  uint16_t* O_lo;
  int ldo;
  int n, t0, nh, dk, dv, conv_k;
};
struct AttnArgs {
  const float* Y;          // projection rows q|k|v of the chunk [n][ldy]
  int ldy;
  uint16_t* K;             // bf16 cache [nkv][cap][hd]; rows t0 .. t0+n-1 are written
  uint16_t* V;
  int cap;
  const float2* rope;      // (cos, sin) [>= t0 + n][hd/2]
  float* Qr;               // scratch: rotated, scaled queries [n][nq][hd]
  const int* pages;        // paged cache (as attn::Params), else null
  int page_tokens;
  long long page_elems;
  uint16_t* O_hi;
  uint16_t* O_lo;
  int ldo;
  int n, t0, nq, nkv, hd;
  float scale;
};
cudaError_t init();
cudaError_t embed_rows(const uint16_t* embed, const int* tok, int n, int H, int vocab, float* X, unsigned* guard,
                       cudaStream_t st);
cudaError_t gdn(const GdnArgs& a, cudaStream_t st);
cudaError_t attention(const AttnArgs& a, cudaStream_t st);
cudaError_t set_len(int* len, int value, cudaStream_t st);
}  // namespace prefill

// Guard word of the allocation-free attention call on the current device
// (null before its first call there); read by hy_op_check_device.
unsigned* noalloc_guard();

// Record `msg` as the calling thread's last error (hy_last_error) and return
// `code`; for C-ABI entry points defined outside engine.cu.
int set_error(int code, const char* msg);

// Launch with the programmatic-stream-serialization attribute when pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

}  // namespace hy

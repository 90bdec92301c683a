// The decode-step engine behind include/hybrid.h: model and cache objects,
// the per-step kernel plan, CUDA-graph capture and replay, and the C ABI.
//
// One decode step is ~5 kernels per layer plus the head, all launched with
// programmatic dependent launch so each kernel's weight stream starts while
// its predecessor drains, and captured once into a CUDA graph that is
// replayed per token with its positions read from device memory ("Beating
// llama.cpp from Scratch on Consumer AMD", Act 0 pass 3: the whole decode
// iteration captured once and replayed; argmax on the device, a 4-byte id
// back).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/hybrid.h"
#include "common.cuh"
#include "kernels.h"

using namespace hy;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define HY_CK(call)                                                                         \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) return fail(HY_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

std::mutex g_init_mu;
std::map<int, bool> g_inited;
std::map<int, unsigned*> g_op_guard;

int ensure_init(int dev) {
  std::lock_guard<std::mutex> lk(g_init_mu);
  if (g_inited[dev]) return HY_OK;
  HY_CK(gemv::init());
  HY_CK(attn::init());
  HY_CK(bgemv::init());
  HY_CK(gemm::init());
  HY_CK(prefill::init());
  g_inited[dev] = true;
  return HY_OK;
}

int current_device(int* dev, int* nsm) {
  HY_CK(cudaGetDevice(dev));
  HY_CK(cudaDeviceGetAttribute(nsm, cudaDevAttrMultiProcessorCount, *dev));
  return HY_OK;
}

// Seeded values for synthetic caches: a 64-bit mix of (seed, index) mapped
// to [-scale, scale).
__device__ __forceinline__ float synth_value(uint64_t seed, uint64_t i, float scale) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return ((float)(uint32_t)(z >> 40) * (1.0f / 8388608.0f) - 1.0f) * scale;
}

// Rows [first_row, first_row + rows) of a seeded bf16 stream (value index
// row * row_len + column) into dst (row stride `stride`).
__global__ void k_fill_bf16(uint16_t* dst, long long rows, int row_len, long long stride, uint64_t seed,
                            long long first_row = 0) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < rows * row_len;
       e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / row_len, k = e % row_len;
    dst[r * stride + k] = f32_to_bf16_rne(synth_value(seed, (uint64_t)(e + first_row * row_len), 1.0f));
  }
}

// int8 cache rows: the same seeded values as k_fill_bf16 (in FP32), each row
// quantised with its own scale (amax / 127, codes round-half-even of
// x * (127 / amax)).  One warp per row.
__global__ void k_fill_i8(int8_t* dst, float* scales, long long rows, int row_len, uint64_t seed) {
  const int lane = threadIdx.x & 31;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    float a = 0.f;
    for (int k = lane; k < row_len; k += 32) a = fmaxf(a, fabsf(synth_value(seed, (uint64_t)(r * row_len + k), 1.0f)));
    a = warp_max(a);
    const float inv = a > 0.f ? 127.0f / a : 0.f;
    for (int k = lane; k < row_len; k += 32) {
      float q = rintf(__fmul_rn(synth_value(seed, (uint64_t)(r * row_len + k), 1.0f), inv));
      q = fminf(fmaxf(q, -127.f), 127.f);
      dst[r * row_len + k] = (int8_t)(int)q;
    }
    if (lane == 0) scales[r] = a / 127.0f;
  }
}

__global__ void k_fill_f32(float* dst, long long n, uint64_t seed, float scale) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x)
    dst[e] = synth_value(seed, (uint64_t)e, scale);
}

__global__ void k_copy_f32(const float* __restrict__ src, float* __restrict__ dst, int n) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

}  // namespace

int hy::set_error(int code, const char* msg) { return fail(code, "%s", msg); }

// ====================================================================== model

struct hy_model {
  hy_config cfg;
  std::vector<hy_layer_weights> layers;
  hy_weights w;
  int device = 0, nsm = 0;
  int n_gdn = 0, n_attn = 0;
  std::vector<int> sub;      // index of a layer among layers of its kind
  std::vector<bool> is_attn;
  int CC = 0, gdn_rows = 0, attn_rows = 0;
  int y_len = 0, o_len = 0, h_len = 0;
  int splits = 1;
  bool moe = false, pdl = true, graphs = true, debug = false;
  bool q4 = false;          // 4-bit linear weights: every step runs the batched path
  bool splits_auto = true;  // split-KV count chosen from the SM count (the batched step then scales it down)
  int splits_long = 0;      // splits of a single sequence whose cache holds attn::kLongContext positions or more
  int batch_spread = -1;    // batched attention: -1 = the step's splits shared over the batch by length, 0 = off,
                            //   > 0 = that many splits shared (HY_ATTN_BATCH_SPREAD)
  bool chunk_prefill = false;  // prompts run as chunks through the tensor-core GEMMs (else token by token)
};

struct hy_cache {
  hy_model* m = nullptr;
  int max_seqs = 0;
  std::vector<int> cap, len;
  std::vector<uint8_t*> mem;
  std::vector<size_t> off_kv;
  size_t off_conv = 0;
  int* d_len = nullptr;
  // scratch
  float *x = nullptr, *y = nullptr, *o = nullptr, *h = nullptr, *part = nullptr, *am_val = nullptr;
  float *rlog = nullptr, *moe_w = nullptr, *logits_buf = nullptr;
  int *am_idx = nullptr, *tok = nullptr, *ids = nullptr, *moe_ids = nullptr;
  unsigned *cnt_attn = nullptr, *cnt_am = nullptr, *guard = nullptr;
  float2* rope = nullptr;
  float *dbg_hidden = nullptr, *dbg_rlog = nullptr;
  int* dbg_rids = nullptr;
  std::vector<void*> allocs;
  cudaStream_t cap_stream = nullptr;
  // batched steps (several sequences, or 4-bit weights): per-token scratch
  float *bx = nullptr, *by = nullptr, *bo = nullptr, *bh = nullptr, *brlog = nullptr, *bw = nullptr;
  float *bpart = nullptr, *bapart = nullptr, *bam_val = nullptr;
  int *btok = nullptr, *bids = nullptr, *bunion = nullptr, *bnu = nullptr, *bslot = nullptr, *bam_idx = nullptr;
  int* brids = nullptr;
  unsigned *bcnt_attn = nullptr, *bcnt_am = nullptr;
  unsigned long long* experts_read = nullptr;  // distinct routed experts the batched steps read (hy_experts_read)
  int bh_len = 0;
  size_t bapart_len = 0;
  struct BGraph {
    std::vector<int> seqs;
    float* logits;
    int* ids;
    cudaGraphExec_t exec;
  };
  std::vector<BGraph> bgraphs;
  int last_kernels = 0;          // kernels of the last recorded step
  // chunked prompt (prefill) buffers, allocated at the first chunked prefill for pf_rows tokens
  int pf_rows = 0, pf_ka = 0;
  float *pf_x = nullptr, *pf_y = nullptr, *pf_qn = nullptr, *pf_kn = nullptr, *pf_v = nullptr, *pf_ab = nullptr;
  float* pf_qr = nullptr;
  uint16_t *pf_ahi = nullptr, *pf_alo = nullptr, *pf_hhi = nullptr, *pf_hlo = nullptr;
  // MoE models: router logits, routing, the picks grouped by expert, their gathered activations, expert
  // outputs, and the shared expert's
  float *pf_rlog = nullptr, *pf_rw = nullptr, *pf_ye = nullptr, *pf_ysh = nullptr;
  int *pf_ids = nullptr, *pf_pos = nullptr, *pf_tok = nullptr, *pf_tiles = nullptr, *pf_ntiles = nullptr;
  uint16_t *pf_ghi = nullptr, *pf_glo = nullptr, *pf_ehi = nullptr, *pf_elo = nullptr, *pf_shi = nullptr,
           *pf_slo = nullptr;
  struct Graph {
    int seq;
    float* logits;
    int* ids;
    cudaGraphExec_t exec;
  };
  std::vector<Graph> graphs;
  // paged KV cache (page_tokens > 0): pages of page_tokens positions (every
  // attention layer's K and V of one sequence) drawn from one pool on demand
  int page_tokens = 0, max_pages = 0;
  long long page_elems = 0;
  uint16_t* pool = nullptr;
  int* d_pages = nullptr;  // [max_seqs][max_pages]: the page of each block of page_tokens positions
  std::vector<int> free_pages;
  std::vector<std::vector<int>> seq_pages;
};

namespace {

float* gdn_state(hy_cache* c, int seq, int gi) {
  const hy_model* m = c->m;
  return reinterpret_cast<float*>(c->mem[seq]) + (size_t)gi * m->cfg.gdn_heads * m->cfg.gdn_dv * m->cfg.gdn_dk;
}
float* conv_state(hy_cache* c, int seq, int gi) {
  const hy_model* m = c->m;
  return reinterpret_cast<float*>(c->mem[seq] + c->off_conv) + (size_t)gi * m->cfg.conv_k * m->CC;
}
// Scale row stride of an int8 cache (a multiple of 4, so that every kv
// head's scales start 16-byte aligned).
int cap_scales(int cap) { return (cap + 3) & ~3; }

// K (which = 0) or V rows of attention layer ai: bf16 [nkv][cap][hd], or with
// the int8 cache the codes [nkv][cap][hd] (bytes, returned as uint16_t*).
uint16_t* kv_cache(hy_cache* c, int seq, int ai, int which) {
  const hy_model* m = c->m;
  if (c->page_tokens)  // this layer's K or V block in page 0 of the pool; kv rows then go through the page table
    return c->pool + ((size_t)ai * 2 + which) * m->cfg.attn_kv_heads * c->page_tokens * m->cfg.head_dim;
  const size_t per = (size_t)m->cfg.attn_kv_heads * c->cap[seq] * m->cfg.head_dim;
  const size_t esz = m->cfg.kv_format == 1 ? 1 : 2;
  return reinterpret_cast<uint16_t*>(c->mem[seq] + c->off_kv[seq] + ((size_t)ai * 2 + which) * per * esz);
}

const int* seq_page_table(hy_cache* c, int seq) {
  return c->page_tokens ? c->d_pages + (size_t)seq * c->max_pages : nullptr;
}

// int8 cache: the FP32 scales [nkv][cap_scales(cap)] of K (which = 0) or V of
// attention layer ai, after every layer's codes.
float* kv_scales(hy_cache* c, int seq, int ai, int which) {
  const hy_model* m = c->m;
  if (m->cfg.kv_format != 1) return nullptr;
  const size_t codes = (size_t)m->n_attn * 2 * m->cfg.attn_kv_heads * c->cap[seq] * m->cfg.head_dim;
  const size_t base = c->off_kv[seq] + ((codes + 255) & ~(size_t)255);
  const size_t per = (size_t)m->cfg.attn_kv_heads * cap_scales(c->cap[seq]);
  return reinterpret_cast<float*>(c->mem[seq] + base) + ((size_t)ai * 2 + which) * per;
}

// One kernel of the decode step, recorded before any is launched so that each
// GEMV can be told what the kernels after it read first.
struct StepOp {
  enum Kind { kGemv, kGdn, kAttn, kCopy } kind;
  gemv::Params g;
  int src, in, epi;
  const char* what;
  gdn::Params d;
  attn::Params a;
  const float* csrc;
  float* cdst;
  int cn;
};

// Bytes of each of the next GEMV's CTA row ranges that the CTAs of the GEMV
// before it prefetch into L2 once their own rows are in flight.
// L2 prefetch of the next kernel's first bytes per CTA (measured on the dense
// 4B step: 0 KB 650.6, 32 KB 661.9, 64 KB 674.4, 96 KB 664.7, 128 KB 665.0
// tokens/s; MoE unchanged).
int next_prefetch_bytes() {
  const char* v = getenv("HY_GEMV_NEXT_KB");
  return (v && *v) ? atoi(v) * 1024 : 64 * 1024;
}

// Prefetch spans of GEMV op i: the first rows of the next dense-source GEMV
// (wrapping to the start of the step: the graph replays it per token) and the
// recurrent state of a Gated DeltaNet kernel that directly follows.
void plan_prefetch(std::vector<StepOp>& ops, size_t i, int nsm) {
  gemv::Params& g = ops[i].g;
  g.n_nx = 0;
  const int nb = next_prefetch_bytes();
  if (nb <= 0) return;
  const int my_ncta = gemv::plan(g.R, g.C, ops[i].epi == gemv::kEpiSwiglu ? 2 : 1, nsm, g.norm_g != nullptr).ncta;
  if (i + 1 < ops.size() && ops[i + 1].kind == StepOp::kGdn) {
    const gdn::Params& d = ops[i + 1].d;
    g.nx[g.n_nx++] = gemv::PfSpan{(const uint8_t*)d.S, d.nh * d.dv, d.dk * 4, my_ncta, 1 << 30};
  }
  for (size_t k = 1; k <= ops.size(); ++k) {
    const StepOp& o = ops[(i + k) % ops.size()];
    if (o.kind != StepOp::kGemv) continue;
    if (o.src != gemv::kSrcDense) break;  // expert rows are known only after the router
    const int npair = o.epi == gemv::kEpiSwiglu ? 2 : 1;
    const gemv::Plan pl = gemv::plan(o.g.R, o.g.C, npair, nsm, o.g.norm_g != nullptr);
    for (int j = 0; j < npair && g.n_nx < gemv::kMaxPfSpans; ++j)
      g.nx[g.n_nx++] = gemv::PfSpan{o.g.W[j], o.g.R, o.g.C * 2, pl.ncta, nb};
    break;
  }
}

int launch_ops(hy_model* m, std::vector<StepOp>& ops, cudaStream_t st) {
  const bool pdl = m->pdl;
  for (size_t i = 0; i < ops.size(); ++i) {
    StepOp& o = ops[i];
    cudaError_t e = cudaSuccess;
    if (o.kind == StepOp::kGemv) {
      plan_prefetch(ops, i, m->nsm);
      const int npair = (o.epi == gemv::kEpiSwiglu) ? 2 : 1;
      const gemv::Plan pl = gemv::plan(o.g.R, o.g.C, npair, m->nsm, o.g.norm_g != nullptr);
      if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for %s (%d x %d)", o.what, o.g.R, o.g.C);
      e = gemv::launch(o.g, pl, o.src, o.in, o.epi, st, pdl);
    } else if (o.kind == StepOp::kGdn) {
      e = gdn::launch(o.d, st, pdl);
    } else if (o.kind == StepOp::kAttn) {
      e = attn::launch(o.a, st, pdl);
    } else {
      e = launch_k(k_copy_f32, dim3((o.cn + 255) / 256), dim3(256), 0, st, pdl, o.csrc, o.cdst, o.cn);
    }
    if (e != cudaSuccess) return fail(HY_ERR_CUDA, "%s launch: %s", o.kind == StepOp::kGemv ? o.what : "kernel",
                                      cudaGetErrorString(e));
  }
  return HY_OK;
}

// The operations of one decode step for sequence `seq`, in order.  The MoE
// router GEMV only stores its logits; the expert gate/up kernel's CTAs pick
// the experts themselves.
int collect_ops(hy_cache* c, int seq, float* logits, int* ids, std::vector<StepOp>& ops) {
  hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  const int H = cf.hidden;
  int* pos = c->d_len + seq;
  ops.clear();
  ops.reserve(8 * cf.n_layers + 2);

  auto gemv_base = [&]() {
    gemv::Params p;
    memset(&p, 0, sizeof(p));
    p.guard = c->guard;
    p.eps = cf.rms_eps;
    return p;
  };
  auto run = [&](gemv::Params& p, int src, int in, int epi, const char* what) -> int {
    StepOp o;
    memset(&o, 0, sizeof(o));
    o.kind = StepOp::kGemv;
    o.g = p;
    o.src = src;
    o.in = in;
    o.epi = epi;
    o.what = what;
    ops.push_back(o);
    return HY_OK;
  };

  for (int l = 0; l < cf.n_layers; ++l) {
    const hy_layer_weights& L = m->layers[l];
    const bool attn_l = m->is_attn[l];
    int rc;
    {  // RMSNorm + input projection (layer 0 also gathers the embedding row)
      gemv::Params p = gemv_base();
      p.W[0] = (const uint8_t*)L.w_in.w;
      p.R = attn_l ? m->attn_rows : m->gdn_rows;
      p.C = H;
      p.x = c->x;
      p.norm_g = L.norm1;
      p.y = c->y;
      int in = gemv::kInX;
      if (l == 0) {
        in = gemv::kInEmbed;
        p.embed = (const uint16_t*)m->w.embed;
        p.tok = c->tok;
        p.vocab = cf.vocab;
        p.x_out = c->x;
      }
      if ((rc = run(p, gemv::kSrcDense, in, gemv::kEpiStore, "in-proj")) != HY_OK) return rc;
    }
    if (attn_l) {
      attn::Params a;
      memset(&a, 0, sizeof(a));
      a.y = c->y;
      a.K = kv_cache(c, seq, m->sub[l], 0);
      a.V = kv_cache(c, seq, m->sub[l], 1);
      a.kv8 = cf.kv_format == 1;
      a.Ks = kv_scales(c, seq, m->sub[l], 0);
      a.Vs = kv_scales(c, seq, m->sub[l], 1);
      a.cap_s = cap_scales(c->cap[seq]);
      a.pages = seq_page_table(c, seq);
      a.page_tokens = c->page_tokens;
      a.page_elems = c->page_elems;
      a.len = pos;
      a.rope = c->rope;
      a.cap = c->cap[seq];
      a.nq = cf.attn_q_heads;
      a.nkv = cf.attn_kv_heads;
      a.hd = cf.head_dim;
      a.nsplit = c->cap[seq] >= attn::kLongContext ? m->splits_long : m->splits;
      a.scale = 1.0f / sqrtf((float)cf.head_dim);
      a.part = c->part;
      a.counter = c->cnt_attn;
      a.o = c->o;
      a.guard = c->guard;
      StepOp o;
      memset(&o, 0, sizeof(o));
      o.kind = StepOp::kAttn;
      o.a = a;
      ops.push_back(o);
    } else {
      gdn::Params g;
      memset(&g, 0, sizeof(g));
      g.y = c->y;
      g.conv_w = (const uint16_t*)L.conv_w;
      g.conv_state = conv_state(c, seq, m->sub[l]);
      g.S = gdn_state(c, seq, m->sub[l]);
      g.o = c->o;
      g.nh = cf.gdn_heads;
      g.dk = cf.gdn_dk;
      g.dv = cf.gdn_dv;
      g.conv_k = cf.conv_k;
      g.pos = pos;
      g.guard = c->guard;
      StepOp o;
      memset(&o, 0, sizeof(o));
      o.kind = StepOp::kGdn;
      o.d = g;
      ops.push_back(o);
    }
    {  // output projection + residual
      gemv::Params p = gemv_base();
      p.W[0] = (const uint8_t*)L.w_o.w;
      p.R = H;
      p.C = attn_l ? cf.attn_q_heads * cf.head_dim : cf.gdn_heads * cf.gdn_dv;
      p.x = c->o;
      p.y = c->x;
      if ((rc = run(p, gemv::kSrcDense, gemv::kInX, gemv::kEpiResid, "out-proj")) != HY_OK) return rc;
    }
    if (!m->moe) {
      gemv::Params p = gemv_base();
      p.W[0] = (const uint8_t*)L.w_gate.w;
      p.W[1] = (const uint8_t*)L.w_up.w;
      p.R = cf.ffn;
      p.C = H;
      p.x = c->x;
      p.norm_g = L.norm2;
      p.y = c->h;
      if ((rc = run(p, gemv::kSrcDense, gemv::kInX, gemv::kEpiSwiglu, "gate/up")) != HY_OK) return rc;
      gemv::Params d = gemv_base();
      d.W[0] = (const uint8_t*)L.w_down.w;
      d.R = H;
      d.C = cf.ffn;
      d.x = c->h;
      d.y = c->x;
      if ((rc = run(d, gemv::kSrcDense, gemv::kInX, gemv::kEpiResid, "down")) != HY_OK) return rc;
    } else {
      const int E = cf.n_experts, K = cf.top_k, Fe = cf.expert_ffn;
      gemv::Params r = gemv_base();
      r.W[0] = (const uint8_t*)L.router;
      r.R = E + 1;
      r.C = H;
      r.x = c->x;
      r.norm_g = L.norm2;
      r.y = c->rlog;
      if ((rc = run(r, gemv::kSrcDense, gemv::kInX, gemv::kEpiStore, "router")) != HY_OK) return rc;
      gemv::Params gu = gemv_base();
      gu.exp_base[0] = (const uint8_t*)L.exp_gate.w;
      gu.exp_base[1] = (const uint8_t*)L.exp_up.w;
      gu.sh_base[0] = (const uint8_t*)L.sh_gate.w;
      gu.sh_base[1] = (const uint8_t*)L.sh_up.w;
      gu.exp_stride = (long long)Fe * H * 2;
      gu.moe_ids = c->moe_ids;
      gu.top_k = K;
      gu.n_experts = E;
      gu.slot_rows = Fe;
      gu.sh_rows = cf.shared_ffn;
      gu.R = K * Fe + cf.shared_ffn;
      gu.C = H;
      gu.x = c->x;
      gu.norm_g = L.norm2;
      gu.y = c->h;
      gu.route_here = 1;
      gu.router_logits = c->rlog;
      gu.out_ids = c->moe_ids;
      gu.out_w = c->moe_w;
      if (m->debug) {
        gu.dbg_ids = c->dbg_rids + (size_t)l * K;
        gu.dbg_logits = c->dbg_rlog + (size_t)l * (E + 1);
      }
      if ((rc = run(gu, gemv::kSrcExpertRows, gemv::kInX, gemv::kEpiSwiglu, "expert gate/up")) != HY_OK) return rc;
      gemv::Params dn = gemv_base();
      dn.exp_base[0] = (const uint8_t*)L.exp_down.w;
      dn.sh_base[0] = (const uint8_t*)L.sh_down.w;
      dn.exp_stride = (long long)H * Fe * 2;
      dn.moe_ids = c->moe_ids;
      dn.moe_w = c->moe_w;
      dn.top_k = K;
      dn.n_experts = E;
      dn.seg_cols = Fe;
      dn.R = H;
      dn.C = (K + 1) * Fe;
      dn.x = c->h;
      dn.y = c->x;
      if ((rc = run(dn, gemv::kSrcExpertSegs, gemv::kInMoeZ, gemv::kEpiResid, "expert down")) != HY_OK) return rc;
    }
    if (m->debug) {
      StepOp o;
      memset(&o, 0, sizeof(o));
      o.kind = StepOp::kCopy;
      o.csrc = c->x;
      o.cdst = c->dbg_hidden + (size_t)l * H;
      o.cn = H;
      ops.push_back(o);
    }
  }
  {  // final RMSNorm + LM head + argmax; the last CTA advances the position
    gemv::Params p = gemv_base();
    p.W[0] = (const uint8_t*)m->w.lm_head.w;
    p.R = cf.vocab;
    p.C = H;
    p.x = c->x;
    p.norm_g = m->w.final_norm;
    p.y = logits;
    p.part_val = c->am_val;
    p.part_idx = c->am_idx;
    p.counter = c->cnt_am;
    p.ids_out = ids;
    p.len_inc = pos;
    int rc = run(p, gemv::kSrcDense, gemv::kInX, gemv::kEpiArgmax, "lm-head");
    if (rc != HY_OK) return rc;
  }
  return HY_OK;
}

// Issue one decode step for sequence `seq` on `st`, one kernel per operation.
int record_step(hy_cache* c, int seq, float* logits, int* ids, cudaStream_t st) {
  hy_model* m = c->m;
  std::vector<StepOp> ops;
  int rc = collect_ops(c, seq, logits, ids, ops);
  if (rc != HY_OK) return rc;
  c->last_kernels = (int)ops.size();
  return launch_ops(m, ops, st);
}

// ---------------------------------------------------------------- batched step
// Issue one decode step for the sequences `seqs` (their token ids already in
// c->btok): every weight is read once for all of them.
int record_batch(hy_cache* c, const std::vector<int>& seqs, float* logits, int* ids, cudaStream_t st) {
  hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  const int H = cf.hidden, B = (int)seqs.size(), fmt = m->q4 ? 1 : 0;
  const bool pdl = m->pdl;
  int kernels = 0;
  auto ck = [&](cudaError_t e, const char* what) -> int {
    if (e != cudaSuccess) return fail(HY_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    ++kernels;
    return HY_OK;
  };
  auto bparams = [&](int wfmt, int src, int in, int epi) {
    bgemv::Params p;
    memset(&p, 0, sizeof(p));
    p.fmt = wfmt;
    p.src = src;
    p.in = in;
    p.epi = epi;
    p.B = B;
    p.eps = cf.rms_eps;
    p.guard = c->guard;
    return p;
  };
  auto set_w = [](bgemv::Params& p, int j, const hy_tensor& t) {
    p.W[j] = (const uint8_t*)t.w;
    p.S[j] = (const uint16_t*)t.scales;
  };
  // A dense batched GEMV.  A bf16 matrix whose token vectors do not fit the
  // kernel's shared memory, with no RMSNorm on its input (the dense down
  // projection), runs as column slices of at most 3072 that accumulate into
  // the output in order; other matrices too wide for it run per token
  // through the single-token kernel (same epilogue).
  auto dense = [&](bgemv::Params p, const char* what) -> int {
    const bgemv::Plan pl = bgemv::plan(p.R, p.C, p.fmt, p.epi, m->nsm);
    if (pl.ok) return ck(bgemv::launch(p, pl, st, pdl), what);
    if (p.fmt != bgemv::kFmtBf16) return fail(HY_ERR_UNSUPPORTED, "no batched plan for %s (%d x %d)", what, p.R, p.C);
    if (!p.norm_g && p.in == bgemv::kInX && (p.epi == bgemv::kEpiStore || p.epi == bgemv::kEpiResid) && p.C % 64 == 0) {
      constexpr int kSlice = 3072;
      bool slices_ok = true;
      for (int c0 = 0; c0 < p.C && slices_ok; c0 += kSlice) {
        const int cc = std::min(kSlice, p.C - c0);
        slices_ok = bgemv::plan(p.R, cc, p.fmt, bgemv::kEpiResid, m->nsm).ok;
      }
      if (slices_ok) {
        for (int c0 = 0; c0 < p.C; c0 += kSlice) {
          bgemv::Params q = p;
          q.C = std::min(kSlice, p.C - c0);
          q.ldw = p.C;
          q.W[0] = p.W[0] + (size_t)c0 * 2;
          q.x = p.x + c0;
          if (c0 > 0) q.epi = bgemv::kEpiResid;  // later slices add to what the first one stored
          const bgemv::Plan pq = bgemv::plan(q.R, q.C, q.fmt, q.epi, m->nsm);
          int rc = ck(bgemv::launch(q, pq, st, pdl), what);
          if (rc != HY_OK) return rc;
        }
        return HY_OK;
      }
    }
    for (int b = 0; b < B; ++b) {
      gemv::Params g;
      memset(&g, 0, sizeof(g));
      g.guard = c->guard;
      g.eps = cf.rms_eps;
      g.W[0] = p.W[0];
      g.W[1] = p.W[1];
      g.R = p.R;
      g.C = p.C;
      g.norm_g = p.norm_g;
      int in = gemv::kInX, epi = gemv::kEpiStore;
      if (p.in == bgemv::kInEmbed) {
        in = gemv::kInEmbed;
        g.embed = p.embed;
        g.tok = p.tok + b;
        g.vocab = p.vocab;
        g.x_out = p.x_out + (size_t)b * p.ldx_out;
      } else {
        g.x = p.x + (size_t)b * p.ldx;
      }
      if (p.epi == bgemv::kEpiResid) epi = gemv::kEpiResid;
      if (p.epi == bgemv::kEpiSwiglu) epi = gemv::kEpiSwiglu;
      if (p.epi == bgemv::kEpiArgmax) {
        epi = gemv::kEpiArgmax;
        g.y = p.y ? p.y + (size_t)b * p.ldy : nullptr;
        g.part_val = c->am_val;
        g.part_idx = c->am_idx;
        g.counter = c->cnt_am;
        g.ids_out = p.ids_out + b;
        g.len_inc = p.len_inc[b];
      } else {
        g.y = p.y + (size_t)b * p.ldy;
      }
      const gemv::Plan gp = gemv::plan(g.R, g.C, epi == gemv::kEpiSwiglu ? 2 : 1, m->nsm, g.norm_g != nullptr);
      if (!gp.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for %s (%d x %d)", what, g.R, g.C);
      int rc = ck(gemv::launch(g, gp, gemv::kSrcDense, in, epi, st, pdl), what);
      if (rc != HY_OK) return rc;
    }
    return HY_OK;
  };

  for (int l = 0; l < cf.n_layers; ++l) {
    const hy_layer_weights& L = m->layers[l];
    const bool attn_l = m->is_attn[l];
    int rc;
    {  // RMSNorm + input projection (layer 0 gathers the embedding rows)
      bgemv::Params p = bparams(fmt, bgemv::kSrcDense, l == 0 ? bgemv::kInEmbed : bgemv::kInX, bgemv::kEpiStore);
      set_w(p, 0, L.w_in);
      p.R = attn_l ? m->attn_rows : m->gdn_rows;
      p.C = H;
      p.x = c->bx;
      p.ldx = H;
      p.embed = (const uint16_t*)m->w.embed;
      p.tok = c->btok;
      p.vocab = cf.vocab;
      p.x_out = c->bx;
      p.ldx_out = H;
      p.norm_g = L.norm1;
      p.y = c->by;
      p.ldy = m->y_len;
      if ((rc = dense(p, "in-proj")) != HY_OK) return rc;
    }
    if (attn_l) {
      attn::Params a;
      memset(&a, 0, sizeof(a));
      a.y = c->by;
      a.rope = c->rope;
      a.nq = cf.attn_q_heads;
      a.nkv = cf.attn_kv_heads;
      a.hd = cf.head_dim;
      // the step's splits (one CTA per SM over the kv heads) shared among the
      // batch's sequences in proportion to their lengths, on the device
      // (ragged contexts: every CTA streams about the same rows); with the
      // spread off, each sequence takes the same count (the largest power of
      // two <= 2 SMs / (kv heads x batch))
      a.nsplit = m->splits;
      if (m->splits_auto && m->batch_spread != 0) {
        a.spread = std::max(m->batch_spread > 0 ? m->batch_spread : m->splits, B);
        a.spread = std::min(a.spread, std::max(m->splits, m->splits_long) + B - 1);  // scratch: ld_part splits
      } else if (m->splits_auto) {
        int sb = 1;
        while (2 * sb <= std::max(1, 2 * m->nsm / (cf.attn_kv_heads * B))) sb *= 2;
        a.nsplit = std::min(m->splits, sb);
      }
      a.scale = 1.0f / sqrtf((float)cf.head_dim);
      a.part = c->bapart;
      a.counter = c->bcnt_attn;
      a.o = c->bo;
      a.guard = c->guard;
      a.nb = B;
      a.ld_y = m->y_len;
      a.ld_o = m->o_len;
      a.ld_part = (long long)c->bapart_len;
      for (int b = 0; b < B; ++b) {
        a.K_b[b] = kv_cache(c, seqs[b], m->sub[l], 0);
        a.V_b[b] = kv_cache(c, seqs[b], m->sub[l], 1);
        a.Ks_b[b] = kv_scales(c, seqs[b], m->sub[l], 0);
        a.Vs_b[b] = kv_scales(c, seqs[b], m->sub[l], 1);
        a.cap_s_b[b] = cap_scales(c->cap[seqs[b]]);
        a.pages_b[b] = seq_page_table(c, seqs[b]);
        a.len_b[b] = c->d_len + seqs[b];
        a.cap_b[b] = c->cap[seqs[b]];
      }
      a.K = a.K_b[0];
      a.V = a.V_b[0];
      a.kv8 = cf.kv_format == 1;
      a.Ks = a.Ks_b[0];
      a.Vs = a.Vs_b[0];
      a.cap_s = a.cap_s_b[0];
      a.pages = a.pages_b[0];
      a.page_tokens = c->page_tokens;
      a.page_elems = c->page_elems;
      a.len = a.len_b[0];
      a.cap = a.cap_b[0];
      if ((rc = ck(attn::launch(a, st, pdl), "attention")) != HY_OK) return rc;
    } else {
      gdn::Params g;
      memset(&g, 0, sizeof(g));
      g.y = c->by;
      g.conv_w = (const uint16_t*)L.conv_w;
      g.o = c->bo;
      g.nh = cf.gdn_heads;
      g.dk = cf.gdn_dk;
      g.dv = cf.gdn_dv;
      g.conv_k = cf.conv_k;
      g.guard = c->guard;
      g.nb = B;
      g.ld_y = m->y_len;
      g.ld_o = m->o_len;
      for (int b = 0; b < B; ++b) {
        g.S_b[b] = gdn_state(c, seqs[b], m->sub[l]);
        g.conv_b[b] = conv_state(c, seqs[b], m->sub[l]);
        g.pos_b[b] = c->d_len + seqs[b];
      }
      g.S = g.S_b[0];
      g.conv_state = g.conv_b[0];
      g.pos = g.pos_b[0];
      if ((rc = ck(gdn::launch(g, st, pdl), "DeltaNet")) != HY_OK) return rc;
    }
    {  // output projection + residual
      bgemv::Params p = bparams(fmt, bgemv::kSrcDense, bgemv::kInX, bgemv::kEpiResid);
      set_w(p, 0, L.w_o);
      p.R = H;
      p.C = attn_l ? cf.attn_q_heads * cf.head_dim : cf.gdn_heads * cf.gdn_dv;
      p.x = c->bo;
      p.ldx = m->o_len;
      p.y = c->bx;
      p.ldy = H;
      if ((rc = dense(p, "out-proj")) != HY_OK) return rc;
    }
    if (!m->moe) {
      bgemv::Params p = bparams(fmt, bgemv::kSrcDense, bgemv::kInX, bgemv::kEpiSwiglu);
      set_w(p, 0, L.w_gate);
      set_w(p, 1, L.w_up);
      p.R = cf.ffn;
      p.C = H;
      p.x = c->bx;
      p.ldx = H;
      p.norm_g = L.norm2;
      p.y = c->bh;
      p.ldy = c->bh_len;
      if ((rc = dense(p, "gate/up")) != HY_OK) return rc;
      bgemv::Params d = bparams(fmt, bgemv::kSrcDense, bgemv::kInX, bgemv::kEpiResid);
      set_w(d, 0, L.w_down);
      d.R = H;
      d.C = cf.ffn;
      d.x = c->bh;
      d.ldx = c->bh_len;
      d.y = c->bx;
      d.ldy = H;
      if ((rc = dense(d, "down")) != HY_OK) return rc;
    } else {
      const int E = cf.n_experts, K = cf.top_k, Fe = cf.expert_ffn;
      {  // router logits of every token (the router stays bf16); the expert gate/up kernel routes
        bgemv::Params r = bparams(bgemv::kFmtBf16, bgemv::kSrcDense, bgemv::kInX, bgemv::kEpiStore);
        r.W[0] = (const uint8_t*)L.router;
        r.R = E + 1;
        r.C = H;
        r.x = c->bx;
        r.ldx = H;
        r.norm_g = L.norm2;
        r.y = c->brlog;
        r.ldy = E + 1;
        const bgemv::Plan pl = bgemv::plan(r.R, r.C, r.fmt, r.epi, m->nsm);
        if (!pl.ok || E > 511 || B * K > bgemv::kMaxUnion)
          return fail(HY_ERR_UNSUPPORTED, "no batched router for %d experts at hidden %d", E, H);
        if ((rc = ck(bgemv::launch(r, pl, st, pdl), "router")) != HY_OK) return rc;
      }
      // rows the union kernels spread over the SMs: the expected union of B
      // tokens' top-K picks under uniform routing, plus the shared expert
      const double pk = 1.0 - std::pow(1.0 - (double)K / E, (double)B);
      const int u_exp = std::min(std::min(E, B * K), (int)std::ceil(E * pk)) + 1;
      const long long ew = fmt ? (long long)Fe * H / 2 : (long long)Fe * H * 2;  // bytes of one expert matrix
      const long long es = fmt ? (long long)Fe * H / 16 : 0;                     // bytes of its scales
      {  // gate/up + SwiGLU over the union of selected experts and the shared expert
        bgemv::Params p = bparams(fmt, bgemv::kSrcUnionRows, bgemv::kInX, bgemv::kEpiSwiglu);
        p.exp_base[0] = (const uint8_t*)L.exp_gate.w;
        p.exp_base[1] = (const uint8_t*)L.exp_up.w;
        p.exp_scale[0] = (const uint16_t*)L.exp_gate.scales;
        p.exp_scale[1] = (const uint16_t*)L.exp_up.scales;
        p.exp_stride = ew;
        p.exp_sstride = es;
        p.sh_base[0] = (const uint8_t*)L.sh_gate.w;
        p.sh_base[1] = (const uint8_t*)L.sh_up.w;
        p.sh_scale[0] = (const uint16_t*)L.sh_gate.scales;
        p.sh_scale[1] = (const uint16_t*)L.sh_up.scales;
        p.union_ids = c->bunion;
        p.n_union = c->bnu;
        p.slot_of = c->bslot;
        p.slot_rows = Fe;
        p.top_k = K;
        p.R = (bgemv::kMaxUnion + 1) * Fe;
        p.C = H;
        p.x = c->bx;
        p.ldx = H;
        p.norm_g = L.norm2;
        p.y = c->bh;
        p.ldy = c->bh_len;
        p.n_exp = E;
        p.route_here = 1;  // every CTA routes the batch from the stored logits; CTA 0 publishes
        p.r_logits = c->brlog;
        p.r_ld = E + 1;
        p.r_ids = c->brids;
        p.r_w = c->bw;
        p.r_E = E;
        p.union_count = c->experts_read;
        const bgemv::Plan pl = bgemv::plan(u_exp * Fe, p.C, p.fmt, p.epi, m->nsm, Fe);
        if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no batched plan for the expert gate/up (%d x %d)", Fe, H);
        if ((rc = ck(bgemv::launch(p, pl, st, pdl), "expert gate/up")) != HY_OK) return rc;
      }
      {  // down projections of the union, per (expert, token) slot
        bgemv::Params p = bparams(fmt, bgemv::kSrcUnionDown, bgemv::kInX, bgemv::kEpiStore);
        p.exp_base[0] = (const uint8_t*)L.exp_down.w;
        p.exp_scale[0] = (const uint16_t*)L.exp_down.scales;
        p.exp_stride = ew;
        p.exp_sstride = es;
        p.sh_base[0] = (const uint8_t*)L.sh_down.w;
        p.sh_scale[0] = (const uint16_t*)L.sh_down.scales;
        p.union_ids = c->bunion;
        p.n_union = c->bnu;
        p.slot_of = c->bslot;
        p.slot_rows = Fe;
        p.top_k = K;
        p.R = H;
        p.C = Fe;
        p.x = c->bh;
        p.ldx = c->bh_len;
        p.part_out = c->bpart;
        p.n_exp = E;
        const bgemv::Plan pl = bgemv::plan(u_exp * H, p.C, p.fmt, p.epi, m->nsm, H);
        if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no batched plan for the expert down");
        if ((rc = ck(bgemv::launch(p, pl, st, pdl), "expert down")) != HY_OK) return rc;
        if ((rc = ck(bgemv::moe_reduce(c->bx, H, c->bpart, c->bw, H, B, K, st, pdl), "expert sum")) != HY_OK) return rc;
      }
      if (m->debug) {  // the first token's router results
        HY_CK(cudaMemcpyAsync(c->dbg_rlog + (size_t)l * (E + 1), c->brlog, sizeof(float) * (E + 1),
                              cudaMemcpyDeviceToDevice, st));
        HY_CK(cudaMemcpyAsync(c->dbg_rids + (size_t)l * K, c->brids, sizeof(int) * K, cudaMemcpyDeviceToDevice, st));
      }
    }
    if (m->debug)  // the residual stream of every token after this layer
      HY_CK(cudaMemcpyAsync(c->dbg_hidden + (size_t)l * H, c->bx, sizeof(float) * H, cudaMemcpyDeviceToDevice, st));
  }
  {  // final RMSNorm + LM head + argmax per token; each sequence's position advances
    bgemv::Params p = bparams(fmt, bgemv::kSrcDense, bgemv::kInX, bgemv::kEpiArgmax);
    set_w(p, 0, m->w.lm_head);
    p.R = cf.vocab;
    p.C = H;
    p.x = c->bx;
    p.ldx = H;
    p.norm_g = m->w.final_norm;
    p.y = logits;
    p.ldy = cf.vocab;
    p.part_val = c->bam_val;
    p.part_idx = c->bam_idx;
    p.counter = c->bcnt_am;
    p.ids_out = ids;
    for (int b = 0; b < B; ++b) p.len_inc[b] = c->d_len + seqs[b];
    int rc = dense(p, "lm-head");
    if (rc != HY_OK) return rc;
  }
  c->last_kernels = kernels;
  return HY_OK;
}

int run_batch(hy_cache* c, const std::vector<int>& seqs, float* logits, int* ids, cudaStream_t st) {
  if (!c->m->graphs) return record_batch(c, seqs, logits, ids, st);
  cudaGraphExec_t exec = nullptr;
  for (auto& g : c->bgraphs)
    if (g.seqs == seqs && g.logits == logits && g.ids == ids) exec = g.exec;
  if (!exec) {
    if (c->bgraphs.size() >= 16) {
      cudaGraphExecDestroy(c->bgraphs.front().exec);
      c->bgraphs.erase(c->bgraphs.begin());
    }
    HY_CK(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    int rc = record_batch(c, seqs, logits, ids, c->cap_stream);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
    if (rc != HY_OK) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (e != cudaSuccess) return fail(HY_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(HY_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    c->bgraphs.push_back({seqs, logits, ids, exec});
  }
  HY_CK(cudaGraphLaunch(exec, st));
  return HY_OK;
}

int get_graph(hy_cache* c, int seq, float* logits, int* ids, cudaGraphExec_t* out) {
  for (auto& g : c->graphs)
    if (g.seq == seq && g.logits == logits && g.ids == ids) {
      *out = g.exec;
      return HY_OK;
    }
  if (c->graphs.size() >= 16) {
    cudaGraphExecDestroy(c->graphs.front().exec);
    c->graphs.erase(c->graphs.begin());
  }
  HY_CK(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
  int rc = record_step(c, seq, logits, ids, c->cap_stream);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
  if (rc != HY_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
  c->graphs.push_back({seq, logits, ids, exec});
  *out = exec;
  return HY_OK;
}

// one step of sequence `seq` whose token id is already in c->tok
int run_step(hy_cache* c, int seq, float* logits, int* ids, cudaStream_t st) {
  if (!c->m->graphs) return record_step(c, seq, logits, ids, st);
  cudaGraphExec_t exec;
  int rc = get_graph(c, seq, logits, ids, &exec);
  if (rc != HY_OK) return rc;
  HY_CK(cudaGraphLaunch(exec, st));
  return HY_OK;
}

int check_model_cfg(const hy_config* c) {
  const uint32_t known = HY_FLAG_DEBUG | HY_FLAG_NO_GRAPH | HY_FLAG_NO_PDL | HY_FLAG_TOKEN_PREFILL;
  if (c->flags & ~known) return fail(HY_ERR_ARG, "unknown flag bits 0x%x", c->flags & ~known);
  if (c->n_layers < 1 || c->n_layers > 64) return fail(HY_ERR_ARG, "n_layers must be in 1..64");
  if (c->hidden <= 0 || c->hidden % 8 || c->vocab <= 0) return fail(HY_ERR_ARG, "hidden must be a positive multiple of 8");
  if (c->weight_format != 0 && c->weight_format != 1) return fail(HY_ERR_ARG, "weight_format must be 0 or 1");
  if (c->weight_format == 1) {
    // 4-bit rows: 32-element blocks whose scale rows stay 16-byte aligned
    const int odim = std::max(c->gdn_heads * c->gdn_dv, c->attn_q_heads * c->head_dim);
    if (c->hidden % 256 || odim % 256 || (c->ffn > 0 && c->ffn % 256) || (c->ffn == 0 && c->expert_ffn % 256))
      return fail(HY_ERR_UNSUPPORTED, "4-bit weights need hidden, head outputs and FFN widths divisible by 256");
  }
  const uint64_t mask = c->n_layers == 64 ? c->attn_layer_mask : (c->attn_layer_mask & ((1ull << c->n_layers) - 1));
  const bool any_attn = mask != 0, any_gdn = (uint64_t)__builtin_popcountll(mask) < (uint64_t)c->n_layers;
  if (any_gdn) {
    if (c->gdn_heads <= 0 || (c->gdn_dk != 64 && c->gdn_dk != 128 && c->gdn_dk != 256) || c->gdn_dv <= 0 ||
        c->gdn_dv % 8)
      return fail(HY_ERR_UNSUPPORTED, "GDN shape: dk must be 64/128/256, dv a multiple of 8");
    if (c->conv_k < 1 || c->conv_k > 8) return fail(HY_ERR_ARG, "conv_k must be in 1..8");
  }
  if (any_attn) {
    if (c->attn_kv_heads <= 0 || c->attn_q_heads % c->attn_kv_heads || c->attn_q_heads / c->attn_kv_heads > 8)
      return fail(HY_ERR_UNSUPPORTED, "attention: nq must be a multiple of nkv with nq/nkv <= 8");
    const int G = c->attn_q_heads / c->attn_kv_heads;
    if ((c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) || (G != 1 && G != 2 && G != 4 && G != 8))
      return fail(HY_ERR_UNSUPPORTED, "attention: head_dim must be 64/128/256 and nq/nkv in {1,2,4,8}");
  }
  if (c->kv_format != 0 && c->kv_format != 1) return fail(HY_ERR_ARG, "kv_format must be 0 or 1");
  if (c->ffn < 0) return fail(HY_ERR_ARG, "ffn < 0");
  if (c->ffn == 0) {
    if (c->n_experts <= 0 || c->top_k <= 0 || c->top_k > 16 || c->top_k > c->n_experts || c->expert_ffn <= 0 ||
        c->expert_ffn % 8)
      return fail(HY_ERR_ARG, "MoE shape");
    if (c->n_experts > 511) return fail(HY_ERR_UNSUPPORTED, "MoE: at most 511 routed experts");
    if (c->shared_ffn != c->expert_ffn) return fail(HY_ERR_UNSUPPORTED, "MoE: shared_ffn must equal expert_ffn");
  } else if (c->ffn % 8) {
    return fail(HY_ERR_ARG, "ffn must be a multiple of 8");
  }
  return HY_OK;
}

void free_cache_mem(hy_cache* c) {
  for (auto& g : c->graphs) cudaGraphExecDestroy(g.exec);
  c->graphs.clear();
  for (auto& g : c->bgraphs) cudaGraphExecDestroy(g.exec);
  c->bgraphs.clear();
  for (void* p : c->allocs) cudaFree(p);
  c->allocs.clear();
  for (uint8_t* p : c->mem) cudaFree(p);
  c->mem.clear();
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  c->cap_stream = nullptr;
}

template <typename T>
int dalloc(hy_cache* c, T** p, size_t count) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, count * sizeof(T) > 0 ? count * sizeof(T) : 16);
  if (e != cudaSuccess) return fail(HY_ERR_NOMEM, "cudaMalloc of %zu bytes: %s", count * sizeof(T), cudaGetErrorString(e));
  c->allocs.push_back(q);
  *p = reinterpret_cast<T*>(q);
  e = cudaMemset(q, 0, count * sizeof(T) > 0 ? count * sizeof(T) : 16);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  return HY_OK;
}

int valid_seq(const hy_cache* c, int seq) { return c && seq >= 0 && seq < c->max_seqs; }

}  // namespace

// ---------------------------------------------------------------- page pool
// Pages so that each (sequence, length) of `need` holds `length` positions:
// taken from the pool and entered in the device page table on `st` before
// any launch that reads them.  HY_ERR_CAPACITY, with nothing taken, when the
// pool is short.
int ensure_pages(hy_cache* c, const std::vector<std::pair<int, int>>& need, cudaStream_t st) {
  if (!c->page_tokens) return HY_OK;
  const int P = c->page_tokens;
  size_t want = 0;
  for (const auto& sl : need) {
    const size_t np = (size_t)(sl.second + P - 1) / P;
    if (np > c->seq_pages[sl.first].size()) want += np - c->seq_pages[sl.first].size();
  }
  if (want > c->free_pages.size())
    return fail(HY_ERR_CAPACITY, "page pool: %zu more pages needed, %zu free", want, c->free_pages.size());
  for (const auto& sl : need) {
    auto& pages = c->seq_pages[sl.first];
    while ((long long)pages.size() * P < sl.second) {
      const int pg = c->free_pages.back();
      c->free_pages.pop_back();
      cudaError_t e = prefill::set_len(c->d_pages + (size_t)sl.first * c->max_pages + pages.size(), pg, st);
      if (e != cudaSuccess) return fail(HY_ERR_CUDA, "page table update: %s", cudaGetErrorString(e));
      pages.push_back(pg);
    }
  }
  return HY_OK;
}

// ---------------------------------------------------------------- chunked prompt
// Prompt tokens per chunk (the GEMMs' M); HY_PREFILL_CHUNK overrides.
int prefill_chunk_rows() {
  const char* v = getenv("HY_PREFILL_CHUNK");
  const int r = (v && *v) ? atoi(v) : 2048;
  return r > 0 ? r : 2048;
}

// Buffers of a chunk of `rows` prompt tokens (grown when a longer chunk comes).
int prefill_buffers(hy_cache* c, int rows) {
  if (c->pf_rows >= rows) return HY_OK;
  hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  const int H = cf.hidden;
  const int ka = std::max(H, std::max(m->o_len, 8));
  for (void* p : {(void*)c->pf_x, (void*)c->pf_y, (void*)c->pf_qn, (void*)c->pf_kn, (void*)c->pf_v, (void*)c->pf_ab,
                  (void*)c->pf_qr, (void*)c->pf_ahi, (void*)c->pf_alo, (void*)c->pf_hhi, (void*)c->pf_hlo,
                  (void*)c->pf_rlog, (void*)c->pf_rw, (void*)c->pf_ye, (void*)c->pf_ysh, (void*)c->pf_ids,
                  (void*)c->pf_pos, (void*)c->pf_tok, (void*)c->pf_tiles, (void*)c->pf_ntiles, (void*)c->pf_ghi,
                  (void*)c->pf_glo, (void*)c->pf_ehi, (void*)c->pf_elo, (void*)c->pf_shi, (void*)c->pf_slo})
    if (p) {
      c->allocs.erase(std::remove(c->allocs.begin(), c->allocs.end(), p), c->allocs.end());
      cudaFree(p);
    }
  c->pf_x = c->pf_y = c->pf_qn = c->pf_kn = c->pf_v = c->pf_ab = c->pf_qr = nullptr;
  c->pf_ahi = c->pf_alo = c->pf_hhi = c->pf_hlo = nullptr;
  c->pf_rlog = c->pf_rw = c->pf_ye = c->pf_ysh = nullptr;
  c->pf_ids = c->pf_pos = c->pf_tok = c->pf_tiles = c->pf_ntiles = nullptr;
  c->pf_ghi = c->pf_glo = c->pf_ehi = c->pf_elo = c->pf_shi = c->pf_slo = nullptr;
  c->pf_rows = 0;
  const size_t R = (size_t)rows;
  const size_t gq = m->n_gdn ? R * cf.gdn_heads * cf.gdn_dk : 1;
  int rc;
  if ((rc = dalloc(c, &c->pf_x, R * H)) || (rc = dalloc(c, &c->pf_y, R * m->y_len)) ||
      (rc = dalloc(c, &c->pf_ahi, R * ka)) || (rc = dalloc(c, &c->pf_alo, R * ka)) ||
      (rc = dalloc(c, &c->pf_hhi, R * std::max(cf.ffn, 8))) || (rc = dalloc(c, &c->pf_hlo, R * std::max(cf.ffn, 8))) ||
      (rc = dalloc(c, &c->pf_qn, gq)) || (rc = dalloc(c, &c->pf_kn, gq)) ||
      (rc = dalloc(c, &c->pf_v, m->n_gdn ? R * cf.gdn_heads * cf.gdn_dv : 1)) ||
      (rc = dalloc(c, &c->pf_ab, m->n_gdn ? R * cf.gdn_heads * 2 : 1)) ||
      (rc = dalloc(c, &c->pf_qr, m->n_attn ? R * cf.attn_q_heads * cf.head_dim : 1)))
    return rc;
  if (m->moe) {
    const size_t E = cf.n_experts, K = cf.top_k, Fe = cf.expert_ffn, Fs = cf.shared_ffn, P = R * K;
    if ((rc = dalloc(c, &c->pf_rlog, R * (E + 1))) || (rc = dalloc(c, &c->pf_rw, R * (K + 1))) ||
        (rc = dalloc(c, &c->pf_ye, P * H)) || (rc = dalloc(c, &c->pf_ysh, R * H)) || (rc = dalloc(c, &c->pf_ids, P)) ||
        (rc = dalloc(c, &c->pf_pos, P)) || (rc = dalloc(c, &c->pf_tok, P)) ||
        (rc = dalloc(c, &c->pf_tiles, (size_t)3 * moepf::max_tiles(rows, (int)E, (int)K))) ||
        (rc = dalloc(c, &c->pf_ntiles, 1)) || (rc = dalloc(c, &c->pf_ghi, P * H)) ||
        (rc = dalloc(c, &c->pf_glo, P * H)) || (rc = dalloc(c, &c->pf_ehi, P * Fe)) ||
        (rc = dalloc(c, &c->pf_elo, P * Fe)) || (rc = dalloc(c, &c->pf_shi, R * Fs)) ||
        (rc = dalloc(c, &c->pf_slo, R * Fs)))
      return rc;
  }
  c->pf_rows = rows;
  c->pf_ka = ka;
  return HY_OK;
}

// The MoE FFN of a chunk of n tokens whose normalised activations are in
// pf_ahi / pf_alo: router GEMM, routing, picks grouped by expert, the grouped
// expert GEMMs (gate/up with SwiGLU, then down), the shared expert's GEMMs,
// and the weighted sum into the residual pf_x.
cudaError_t moe_chunk(hy_cache* c, const hy_layer_weights& L, int n, cudaStream_t st) {
  hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  const int H = cf.hidden, ka = c->pf_ka, E = cf.n_experts, K = cf.top_k, Fe = cf.expert_ffn,
            Fs = cf.shared_ffn, P = n * K;
  auto base = [&](int M, int N, int Kd, int epi) {
    gemm::Params g;
    memset(&g, 0, sizeof(g));
    g.M = M;
    g.N = N;
    g.K = Kd;
    g.epi = epi;
    g.guard = c->guard;
    return g;
  };
  gemm::Params g = base(n, E + 1, H, gemm::kEpiStore);  // router logits [n][E + 1]
  g.y = c->pf_rlog;
  g.ldy = E + 1;
  cudaError_t e = gemm::launch(g, c->pf_ahi, c->pf_alo, ka, (const uint16_t*)L.router, nullptr, H, st);
  if (e == cudaSuccess) e = moepf::route(c->pf_rlog, E + 1, n, E, K, c->pf_ids, c->pf_rw, st);
  if (e == cudaSuccess)
    e = moepf::bucket(c->pf_ids, n, E, K, c->pf_pos, c->pf_tok, c->pf_tiles, c->pf_ntiles, c->guard, st);
  if (e == cudaSuccess) e = moepf::gather(c->pf_ahi, c->pf_alo, ka, H, c->pf_tok, P, c->pf_ghi, c->pf_glo, st);
  const int mt = moepf::max_tiles(n, E, K);
  if (e == cudaSuccess) {  // grouped gate/up + SwiGLU: [P][Fe] hi / lo
    g = base(P, Fe, H, gemm::kEpiSwigluSplit);
    g.h_hi = c->pf_ehi;
    g.h_lo = c->pf_elo;
    g.ldh = Fe;
    g.tiles = c->pf_tiles;
    g.ntiles = c->pf_ntiles;
    g.max_tiles = mt;
    g.w_group_rows = Fe;
    g.n_groups = E;
    e = gemm::launch(g, c->pf_ghi, c->pf_glo, H, (const uint16_t*)L.exp_gate.w, (const uint16_t*)L.exp_up.w, H, st);
  }
  if (e == cudaSuccess) {  // grouped down: [P][H] FP32
    g = base(P, H, Fe, gemm::kEpiStore);
    g.y = c->pf_ye;
    g.ldy = H;
    g.tiles = c->pf_tiles;
    g.ntiles = c->pf_ntiles;
    g.max_tiles = mt;
    g.w_group_rows = H;
    g.n_groups = E;
    e = gemm::launch(g, c->pf_ehi, c->pf_elo, Fe, (const uint16_t*)L.exp_down.w, nullptr, Fe, st);
  }
  if (e == cudaSuccess) {  // shared expert gate/up + SwiGLU
    g = base(n, Fs, H, gemm::kEpiSwigluSplit);
    g.h_hi = c->pf_shi;
    g.h_lo = c->pf_slo;
    g.ldh = Fs;
    e = gemm::launch(g, c->pf_ahi, c->pf_alo, ka, (const uint16_t*)L.sh_gate.w, (const uint16_t*)L.sh_up.w, H, st);
  }
  if (e == cudaSuccess) {  // shared expert down: [n][H] FP32
    g = base(n, H, Fs, gemm::kEpiStore);
    g.y = c->pf_ysh;
    g.ldy = H;
    e = gemm::launch(g, c->pf_shi, c->pf_slo, Fs, (const uint16_t*)L.sh_down.w, nullptr, Fs, st);
  }
  if (e == cudaSuccess) e = moepf::combine(c->pf_x, H, n, K, c->pf_rw, c->pf_pos, c->pf_ye, c->pf_ysh, st);
  return e;
}

// One chunk of n prompt tokens of sequence `seq` at positions t0 .. t0+n-1
// through every layer; `last`: also the final norm, the LM head and argmax of
// its last token (logits nullable, id to c->ids) and the debug copies.
int prefill_chunk(hy_cache* c, int seq, const int* tok, int n, int t0, bool last, float* logits, cudaStream_t st) {
  hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  const int H = cf.hidden, ka = c->pf_ka;
  cudaError_t e = prefill::embed_rows((const uint16_t*)m->w.embed, tok, n, H, cf.vocab, c->pf_x, c->guard, st);
  auto gemm_run = [&](int N, int K, int epi, const uint16_t* ahi, const uint16_t* alo, int lda, const void* w0,
                      const void* w1, float* y, int ldy) {
    gemm::Params g;
    memset(&g, 0, sizeof(g));
    g.M = n;
    g.N = N;
    g.K = K;
    g.epi = epi;
    g.y = y;
    g.ldy = ldy;
    g.h_hi = c->pf_hhi;
    g.h_lo = c->pf_hlo;
    g.ldh = cf.ffn;
    g.guard = c->guard;
    return gemm::launch(g, ahi, alo, lda, (const uint16_t*)w0, (const uint16_t*)w1, K, st);
  };
  for (int l = 0; l < cf.n_layers && e == cudaSuccess; ++l) {
    const hy_layer_weights& L = m->layers[l];
    const bool attn_l = m->is_attn[l];
    const int rows = attn_l ? m->attn_rows : m->gdn_rows;
    const int od = attn_l ? cf.attn_q_heads * cf.head_dim : cf.gdn_heads * cf.gdn_dv;
    e = gemm::norm_split(c->pf_x, H, L.norm1, cf.rms_eps, n, H, c->pf_ahi, c->pf_alo, ka, st);
    if (e == cudaSuccess)
      e = gemm_run(rows, H, gemm::kEpiStore, c->pf_ahi, c->pf_alo, ka, L.w_in.w, nullptr, c->pf_y, m->y_len);
    if (e == cudaSuccess && attn_l) {
      prefill::AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.Y = c->pf_y;
      a.ldy = m->y_len;
      a.K = kv_cache(c, seq, m->sub[l], 0);
      a.V = kv_cache(c, seq, m->sub[l], 1);
      a.cap = c->cap[seq];
      a.rope = c->rope;
      a.Qr = c->pf_qr;
      a.pages = seq_page_table(c, seq);
      a.page_tokens = c->page_tokens;
      a.page_elems = c->page_elems;
      a.O_hi = c->pf_ahi;
      a.O_lo = c->pf_alo;
      a.ldo = ka;
      a.n = n;
      a.t0 = t0;
      a.nq = cf.attn_q_heads;
      a.nkv = cf.attn_kv_heads;
      a.hd = cf.head_dim;
      a.scale = 1.0f / sqrtf((float)cf.head_dim);
      e = prefill::attention(a, st);
    } else if (e == cudaSuccess) {
      prefill::GdnArgs g;
      memset(&g, 0, sizeof(g));
      g.Y = c->pf_y;
      g.ldy = m->y_len;
      g.conv_w = (const uint16_t*)L.conv_w;
      g.ring = conv_state(c, seq, m->sub[l]);
      g.S = gdn_state(c, seq, m->sub[l]);
      g.Qn = c->pf_qn;
      g.Kn = c->pf_kn;
      g.V = c->pf_v;
      g.AB = c->pf_ab;
      g.O_hi = c->pf_ahi;
      g.O_lo = c->pf_alo;
      g.ldo = ka;
      g.n = n;
      g.t0 = t0;
      g.nh = cf.gdn_heads;
      g.dk = cf.gdn_dk;
      g.dv = cf.gdn_dv;
      g.conv_k = cf.conv_k;
      e = prefill::gdn(g, st);
    }
    if (e == cudaSuccess) e = gemm_run(H, od, gemm::kEpiResid, c->pf_ahi, c->pf_alo, ka, L.w_o.w, nullptr, c->pf_x, H);
    if (e == cudaSuccess) e = gemm::norm_split(c->pf_x, H, L.norm2, cf.rms_eps, n, H, c->pf_ahi, c->pf_alo, ka, st);
    if (e == cudaSuccess && m->moe) {
      e = moe_chunk(c, L, n, st);
    } else if (e == cudaSuccess) {
      e = gemm_run(cf.ffn, H, gemm::kEpiSwigluSplit, c->pf_ahi, c->pf_alo, ka, L.w_gate.w, L.w_up.w, nullptr, 0);
      if (e == cudaSuccess)
        e = gemm_run(H, cf.ffn, gemm::kEpiResid, c->pf_hhi, c->pf_hlo, cf.ffn, L.w_down.w, nullptr, c->pf_x, H);
    }
    if (e == cudaSuccess && last && m->debug && m->moe) {  // the last token's routing, as a decode step records it
      const int K = cf.top_k, E = cf.n_experts;
      e = cudaMemcpyAsync(c->dbg_rids + (size_t)l * K, c->pf_ids + (size_t)(n - 1) * K, sizeof(int) * K,
                          cudaMemcpyDeviceToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(c->dbg_rlog + (size_t)l * (E + 1), c->pf_rlog + (size_t)(n - 1) * (E + 1),
                            sizeof(float) * (E + 1), cudaMemcpyDeviceToDevice, st);
    }
    if (e == cudaSuccess && last && m->debug)
      e = cudaMemcpyAsync(c->dbg_hidden + (size_t)l * H, c->pf_x + (size_t)(n - 1) * H, sizeof(float) * H,
                          cudaMemcpyDeviceToDevice, st);
  }
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "prompt chunk launch: %s", cudaGetErrorString(e));
  if (!last) return HY_OK;
  gemv::Params p;  // final RMSNorm + LM head + argmax of the last token
  memset(&p, 0, sizeof(p));
  p.guard = c->guard;
  p.eps = cf.rms_eps;
  p.W[0] = (const uint8_t*)m->w.lm_head.w;
  p.R = cf.vocab;
  p.C = H;
  p.x = c->pf_x + (size_t)(n - 1) * H;
  p.norm_g = m->w.final_norm;
  p.y = logits;
  p.part_val = c->am_val;
  p.part_idx = c->am_idx;
  p.counter = c->cnt_am;
  p.ids_out = c->ids;
  const gemv::Plan pl = gemv::plan(p.R, p.C, 1, m->nsm, true);
  if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for the LM head");
  e = gemv::launch(p, pl, gemv::kSrcDense, gemv::kInX, gemv::kEpiArgmax, st, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "LM head launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

// ====================================================================== C ABI

extern "C" {

const char* hy_last_error(void) { return g_err.c_str(); }

int hy_model_create(const hy_config* cfg, const hy_weights* w, hy_model** out) {
  if (!cfg || !w || !out) return fail(HY_ERR_ARG, "null argument");
  *out = nullptr;
  int rc = check_model_cfg(cfg);
  if (rc != HY_OK) return rc;
  if (!w->layers) return fail(HY_ERR_ARG, "weights.layers is null");
  const hy_config& c = *cfg;
  const int H = c.hidden;
  auto need = [&](const void* p, const char* name, int l) -> int {
    if (!aligned16(p)) return fail(HY_ERR_ARG, "weight %s of layer %d is null or not 16-byte aligned", name, l);
    return HY_OK;
  };
  if ((rc = need(w->embed, "embed", -1)) || (rc = need(w->final_norm, "final_norm", -1)) ||
      (rc = need(w->lm_head.w, "lm_head", -1)))
    return rc;
  const bool q4 = c.weight_format == 1;
  auto need_t = [&](const hy_tensor& t, const char* name, int l) -> int {
    int r = need(t.w, name, l);
    if (r == HY_OK && q4 && !aligned16(t.scales))
      r = fail(HY_ERR_ARG, "4-bit weight %s of layer %d has no 16-byte aligned scales", name, l);
    return r;
  };
  if ((rc = need_t(w->lm_head, "lm_head", -1))) return rc;
  auto* m = new hy_model();
  m->cfg = c;
  m->w = *w;
  m->layers.assign(w->layers, w->layers + c.n_layers);
  m->w.layers = nullptr;
  m->is_attn.resize(c.n_layers);
  m->sub.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    m->is_attn[l] = (c.attn_layer_mask >> l) & 1ull;
    m->sub[l] = m->is_attn[l] ? m->n_attn++ : m->n_gdn++;
    const hy_layer_weights& L = m->layers[l];
    if ((rc = need(L.norm1, "norm1", l)) || (rc = need_t(L.w_in, "w_in", l)) || (rc = need_t(L.w_o, "w_o", l)) ||
        (rc = need(L.norm2, "norm2", l)))
      break;
    if (!m->is_attn[l] && !L.conv_w) { rc = fail(HY_ERR_ARG, "conv_w of layer %d is null", l); break; }
    if (c.ffn > 0) {
      if ((rc = need_t(L.w_gate, "w_gate", l)) || (rc = need_t(L.w_up, "w_up", l)) ||
          (rc = need_t(L.w_down, "w_down", l)))
        break;
    } else {
      if ((rc = need(L.router, "router", l)) || (rc = need_t(L.exp_gate, "exp_gate", l)) ||
          (rc = need_t(L.exp_up, "exp_up", l)) || (rc = need_t(L.exp_down, "exp_down", l)) ||
          (rc = need_t(L.sh_gate, "sh_gate", l)) || (rc = need_t(L.sh_up, "sh_up", l)) ||
          (rc = need_t(L.sh_down, "sh_down", l)))
        break;
    }
  }
  if (rc != HY_OK) {
    delete m;
    return rc;
  }
  if ((rc = current_device(&m->device, &m->nsm)) != HY_OK || (rc = ensure_init(m->device)) != HY_OK) {
    delete m;
    return rc;
  }
  m->CC = 2 * c.gdn_heads * c.gdn_dk + c.gdn_heads * c.gdn_dv;
  m->gdn_rows = m->CC + 2 * c.gdn_heads;
  m->attn_rows = (c.attn_q_heads + 2 * c.attn_kv_heads) * c.head_dim;
  m->moe = c.ffn == 0;
  int y = H;
  if (m->n_gdn) y = std::max(y, m->gdn_rows);
  if (m->n_attn) y = std::max(y, m->attn_rows);
  m->y_len = y;
  m->o_len = std::max(m->n_gdn ? c.gdn_heads * c.gdn_dv : 0, m->n_attn ? c.attn_q_heads * c.head_dim : 0);
  m->h_len = m->moe ? (c.top_k + 1) * c.expert_ffn : c.ffn;
  m->splits = c.attn_splits > 0 ? c.attn_splits : attn::step_splits(c.attn_kv_heads, m->nsm);
  m->splits_auto = c.attn_splits <= 0;
  m->splits_long = m->splits_auto ? attn::long_context_splits(c.attn_q_heads, c.attn_kv_heads, m->nsm) : m->splits;
  if (const char* v = getenv("HY_ATTN_BATCH_SPREAD")) {
    if (*v) m->batch_spread = std::max(atoi(v), 0);
  }
  m->pdl = !(c.flags & HY_FLAG_NO_PDL);
  m->graphs = !(c.flags & HY_FLAG_NO_GRAPH);
  m->debug = (c.flags & HY_FLAG_DEBUG) != 0;
  m->q4 = c.weight_format == 1;
  {  // the chunked prompt path: bf16 models whose GEMM widths suit the tensor copies
    const int od = std::max(m->n_gdn ? c.gdn_heads * c.gdn_dv : 8, m->n_attn ? c.attn_q_heads * c.head_dim : 8);
    const bool ffn_ok = m->moe ? (c.expert_ffn % 8 == 0 && c.shared_ffn % 8 == 0 && c.shared_ffn > 0 &&
                                  c.n_experts <= 512 && c.top_k <= 16)
                               : c.ffn % 8 == 0;
    m->chunk_prefill = !m->q4 && c.kv_format == 0 && !(c.flags & HY_FLAG_TOKEN_PREFILL) && H % 8 == 0 && ffn_ok &&
                       od % 8 == 0;
  }
  *out = m;
  g_err.clear();
  return HY_OK;
}

void hy_model_free(hy_model* m) { delete m; }

static int cache_alloc(hy_model* m, int32_t max_seqs, const int32_t* capacity_host, int32_t page_tokens,
                       int32_t pool_pages, hy_cache** out) {
  if (!m || !out || max_seqs <= 0 || !capacity_host) return fail(HY_ERR_ARG, "bad argument");
  *out = nullptr;
  const hy_config& cf = m->cfg;
  const bool paged = page_tokens > 0;
  if (paged && (page_tokens % 128 || pool_pages <= 0))
    return fail(HY_ERR_ARG, "page_tokens must be a positive multiple of 128 and pool_pages positive");
  if (paged && cf.kv_format != 0) return fail(HY_ERR_UNSUPPORTED, "paged caches hold bf16 K/V only");
  auto* c = new hy_cache();
  c->m = m;
  c->max_seqs = max_seqs;
  c->cap.assign(capacity_host, capacity_host + max_seqs);
  c->len.assign(max_seqs, 0);
  int rc = HY_OK;
  int max_cap = 1;
  for (int s = 0; s < max_seqs; ++s) {
    if (c->cap[s] <= 0) { delete c; return fail(HY_ERR_ARG, "capacity of sequence %d must be positive", s); }
    max_cap = std::max(max_cap, c->cap[s]);
  }
  const size_t state_b = (size_t)m->n_gdn * cf.gdn_heads * cf.gdn_dv * cf.gdn_dk * 4;
  const size_t conv_b = (size_t)m->n_gdn * std::max(cf.conv_k, 1) * m->CC * 4;
  c->off_conv = (state_b + 255) & ~(size_t)255;
  const size_t off_kv = (c->off_conv + conv_b + 255) & ~(size_t)255;
  for (int s = 0; s < max_seqs; ++s) {
    size_t kv_b = paged ? 0 : (size_t)m->n_attn * 2 * cf.attn_kv_heads * c->cap[s] * cf.head_dim * 2;
    if (cf.kv_format == 1) {  // int8 codes, then the per-vector scales
      const size_t codes = (size_t)m->n_attn * 2 * cf.attn_kv_heads * c->cap[s] * cf.head_dim;
      kv_b = ((codes + 255) & ~(size_t)255) + (size_t)m->n_attn * 2 * cf.attn_kv_heads * cap_scales(c->cap[s]) * 4;
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, off_kv + kv_b + 256);
    if (e != cudaSuccess) {
      free_cache_mem(c);
      delete c;
      return fail(HY_ERR_NOMEM, "cache of sequence %d (%zu bytes): %s", s, off_kv + kv_b, cudaGetErrorString(e));
    }
    c->mem.push_back((uint8_t*)p);
    c->off_kv.push_back(off_kv);
    if ((e = cudaMemset(p, 0, off_kv)) != cudaSuccess) {
      free_cache_mem(c);
      delete c;
      return fail(HY_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
    }
  }
  const int G = cf.attn_kv_heads > 0 ? cf.attn_q_heads / cf.attn_kv_heads : 1;
  const size_t part = m->n_attn ? attn::part_floats(cf.attn_q_heads, cf.attn_kv_heads, cf.head_dim,
                                                   std::max(m->splits, m->splits_long)) : 1;
  (void)G;
  if ((rc = dalloc(c, &c->d_len, max_seqs)) || (rc = dalloc(c, &c->x, cf.hidden)) ||
      (rc = dalloc(c, &c->y, m->y_len)) || (rc = dalloc(c, &c->o, std::max(m->o_len, 1))) ||
      (rc = dalloc(c, &c->h, std::max(m->h_len, 1))) || (rc = dalloc(c, &c->part, part)) ||
      (rc = dalloc(c, &c->am_val, 1024)) || (rc = dalloc(c, &c->am_idx, 1024)) ||
      (rc = dalloc(c, &c->rlog, std::max(cf.n_experts + 1, 1))) || (rc = dalloc(c, &c->moe_w, gemv::kMaxTopK + 4)) ||
      (rc = dalloc(c, &c->moe_ids, 16)) || (rc = dalloc(c, &c->tok, max_seqs)) || (rc = dalloc(c, &c->ids, max_seqs)) ||
      (rc = dalloc(c, &c->cnt_attn, std::max(cf.attn_kv_heads, 1))) || (rc = dalloc(c, &c->cnt_am, 1)) ||
      (rc = dalloc(c, &c->guard, 1)) ||
      (rc = dalloc(c, &c->logits_buf, (size_t)cf.vocab * bgemv::kMaxB))) {
    free_cache_mem(c);
    delete c;
    return rc;
  }
  {  // batched-step scratch
    const int B = bgemv::kMaxB, K = std::max(cf.top_k, 1), E1 = std::max(cf.n_experts + 1, 1);
    c->bh_len = m->moe ? (bgemv::kMaxUnion + 1) * cf.expert_ffn : std::max(cf.ffn, 1);
    c->bapart_len = part;
    if ((rc = dalloc(c, &c->bx, (size_t)B * cf.hidden)) || (rc = dalloc(c, &c->by, (size_t)B * m->y_len)) ||
        (rc = dalloc(c, &c->bo, (size_t)B * std::max(m->o_len, 1))) || (rc = dalloc(c, &c->bh, (size_t)B * c->bh_len)) ||
        (rc = dalloc(c, &c->brlog, (size_t)B * E1)) || (rc = dalloc(c, &c->bw, (size_t)B * (K + 1))) ||
        (rc = dalloc(c, &c->bpart, m->moe ? (size_t)B * (K + 1) * cf.hidden : 1)) ||
        (rc = dalloc(c, &c->bapart, (size_t)B * part)) || (rc = dalloc(c, &c->bam_val, (size_t)1024 * B)) ||
        (rc = dalloc(c, &c->bam_idx, (size_t)1024 * B)) || (rc = dalloc(c, &c->btok, B)) ||
        (rc = dalloc(c, &c->bids, B)) || (rc = dalloc(c, &c->bunion, bgemv::kMaxUnion)) ||
        (rc = dalloc(c, &c->bnu, 1)) || (rc = dalloc(c, &c->bslot, (size_t)(bgemv::kMaxUnion + 1) * B)) ||
        (rc = dalloc(c, &c->brids, (size_t)B * K)) ||
        (rc = dalloc(c, &c->bcnt_attn, (size_t)B * std::max(cf.attn_kv_heads, 1))) || (rc = dalloc(c, &c->bcnt_am, 1)) ||
        (rc = dalloc(c, &c->experts_read, 1))) {
      free_cache_mem(c);
      delete c;
      return rc;
    }
  }
  if (paged) {  // the page pool and the page tables
    c->page_tokens = page_tokens;
    c->max_pages = (max_cap + page_tokens - 1) / page_tokens;
    c->page_elems = (long long)std::max(m->n_attn, 1) * 2 * cf.attn_kv_heads * page_tokens * cf.head_dim;
    if ((rc = dalloc(c, &c->pool, (size_t)pool_pages * c->page_elems)) ||
        (rc = dalloc(c, &c->d_pages, (size_t)max_seqs * c->max_pages))) {
      free_cache_mem(c);
      delete c;
      return rc;
    }
    for (int pg = pool_pages - 1; pg >= 0; --pg) c->free_pages.push_back(pg);
    c->seq_pages.assign(max_seqs, {});
  }
  if (m->n_attn) {
    if ((rc = dalloc(c, &c->rope, (size_t)max_cap * (cf.head_dim / 2)))) {
      free_cache_mem(c);
      delete c;
      return rc;
    }
    cudaError_t e = attn::rope_table(c->rope, max_cap, cf.head_dim, (double)cf.rope_theta, 0);
    if (e != cudaSuccess) {
      free_cache_mem(c);
      delete c;
      return fail(HY_ERR_CUDA, "rope table: %s", cudaGetErrorString(e));
    }
  }
  if (m->debug) {
    if ((rc = dalloc(c, &c->dbg_hidden, (size_t)cf.n_layers * cf.hidden)) ||
        (rc = dalloc(c, &c->dbg_rlog, (size_t)cf.n_layers * std::max(cf.n_experts + 1, 1))) ||
        (rc = dalloc(c, &c->dbg_rids, (size_t)cf.n_layers * std::max(cf.top_k, 1)))) {
      free_cache_mem(c);
      delete c;
      return rc;
    }
  }
  cudaError_t e = cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_cache_mem(c);
    delete c;
    return fail(HY_ERR_CUDA, "cache setup: %s", cudaGetErrorString(e));
  }
  *out = c;
  g_err.clear();
  return HY_OK;
}

int hy_cache_alloc(hy_model* m, int32_t max_seqs, const int32_t* capacity_host, hy_cache** out) {
  return cache_alloc(m, max_seqs, capacity_host, 0, 0, out);
}

int hy_cache_alloc_paged(hy_model* m, int32_t max_seqs, const int32_t* capacity_host, int32_t page_tokens,
                         int32_t pool_pages, hy_cache** out) {
  if (page_tokens <= 0) return fail(HY_ERR_ARG, "page_tokens must be a positive multiple of 128");
  return cache_alloc(m, max_seqs, capacity_host, page_tokens, pool_pages, out);
}

int32_t hy_cache_free_pages(const hy_cache* c) {
  return (c && c->page_tokens) ? (int32_t)c->free_pages.size() : -1;
}

void hy_cache_free(hy_cache* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  free_cache_mem(c);
  delete c;
}

int hy_seq_reset(hy_cache* c, int32_t seq, void* stream) {
  if (!valid_seq(c, seq)) return fail(HY_ERR_ARG, "bad sequence handle %d", seq);
  cudaStream_t st = (cudaStream_t)stream;
  HY_CK(cudaMemsetAsync(c->mem[seq], 0, c->off_kv[seq], st));
  HY_CK(cudaMemsetAsync(c->d_len + seq, 0, sizeof(int), st));
  c->len[seq] = 0;
  if (c->page_tokens) {  // the sequence's pages go back to the pool
    for (int pg : c->seq_pages[seq]) c->free_pages.push_back(pg);
    c->seq_pages[seq].clear();
  }
  return HY_OK;
}

int32_t hy_seq_len(const hy_cache* c, int32_t seq) { return valid_seq(c, seq) ? c->len[seq] : -1; }
int32_t hy_seq_capacity(const hy_cache* c, int32_t seq) { return valid_seq(c, seq) ? c->cap[seq] : -1; }
int32_t hy_step_kernels(const hy_cache* c) { return c ? c->last_kernels : 0; }
int32_t hy_step_splits(const hy_cache* c, int32_t seq) {
  if (!c || seq < 0 || seq >= (int32_t)c->cap.size() || !c->m->n_attn) return 0;
  return c->cap[seq] >= attn::kLongContext ? c->m->splits_long : c->m->splits;
}

int hy_experts_read(hy_cache* c, void* stream, uint64_t* total_out) {
  if (!c || !total_out) return fail(HY_ERR_ARG, "null argument");
  cudaStream_t st = (cudaStream_t)stream;
  unsigned long long v = 0;
  if (c->experts_read) {
    HY_CK(cudaMemcpyAsync(&v, c->experts_read, sizeof(v), cudaMemcpyDeviceToHost, st));
    HY_CK(cudaMemsetAsync(c->experts_read, 0, sizeof(v), st));
    HY_CK(cudaStreamSynchronize(st));
  }
  *total_out = (uint64_t)v;
  return HY_OK;
}

int hy_seq_fill_synthetic(hy_cache* c, int32_t seq, int32_t len, uint64_t seed, void* stream) {
  if (!valid_seq(c, seq) || len < 0) return fail(HY_ERR_ARG, "bad argument");
  if (len > c->cap[seq]) return fail(HY_ERR_CAPACITY, "sequence %d: length %d exceeds capacity %d", seq, len, c->cap[seq]);
  const hy_model* m = c->m;
  const hy_config& cf = m->cfg;
  cudaStream_t st = (cudaStream_t)stream;
  {
    int rc = ensure_pages(c, {{seq, len}}, st);
    if (rc != HY_OK) return rc;
  }
  for (int a = 0; a < m->n_attn; ++a)
    for (int w = 0; w < 2; ++w)
      for (int g = 0; g < cf.attn_kv_heads && len > 0; ++g) {
        const uint64_t key = seed * 1000003ull + (uint64_t)((a * 2 + w) * 64 + g);
        if (cf.kv_format == 1) {
          int8_t* base = reinterpret_cast<int8_t*>(kv_cache(c, seq, a, w)) + (size_t)g * c->cap[seq] * cf.head_dim;
          float* sc = kv_scales(c, seq, a, w) + (size_t)g * cap_scales(c->cap[seq]);
          k_fill_i8<<<1024, 256, 0, st>>>(base, sc, len, cf.head_dim, key);
        } else if (c->page_tokens) {  // block by block through the sequence's pages
          const int P = c->page_tokens;
          for (int j = 0; j * P < len; ++j) {
            uint16_t* base = kv_cache(c, seq, a, w) + (size_t)c->seq_pages[seq][j] * c->page_elems +
                             (size_t)g * P * cf.head_dim;
            k_fill_bf16<<<256, 256, 0, st>>>(base, std::min(P, len - j * P), cf.head_dim, cf.head_dim, key,
                                             (long long)j * P);
          }
        } else {
          uint16_t* base = kv_cache(c, seq, a, w) + (size_t)g * c->cap[seq] * cf.head_dim;
          k_fill_bf16<<<1024, 256, 0, st>>>(base, len, cf.head_dim, cf.head_dim, key);
        }
      }
  if (m->n_gdn) {
    const long long n = (long long)m->n_gdn * cf.gdn_heads * cf.gdn_dv * cf.gdn_dk;
    k_fill_f32<<<1024, 256, 0, st>>>(gdn_state(c, seq, 0), n, seed * 1000003ull + 977ull, 0.01f);
    HY_CK(cudaMemsetAsync(conv_state(c, seq, 0), 0, sizeof(float) * (size_t)m->n_gdn * cf.conv_k * m->CC, st));
  }
  HY_CK(cudaGetLastError());
  HY_CK(cudaMemcpyAsync(c->d_len + seq, &len, sizeof(int), cudaMemcpyHostToDevice, st));
  HY_CK(cudaStreamSynchronize(st));  // &len is a host stack value
  c->len[seq] = len;
  return HY_OK;
}

int hy_prefill(hy_model* m, hy_cache* c, int32_t seq, const int32_t* tokens_dev, int32_t n, float* logits_dev,
               void* stream) {
  if (!m || !c || c->m != m || !valid_seq(c, seq) || (n > 0 && !tokens_dev) || n < 0)
    return fail(HY_ERR_ARG, "bad argument");
  if ((long long)c->len[seq] + n > c->cap[seq])
    return fail(HY_ERR_CAPACITY, "sequence %d: %d + %d tokens exceed capacity %d", seq, c->len[seq], n, c->cap[seq]);
  cudaStream_t st = (cudaStream_t)stream;
  {
    int rc = ensure_pages(c, {{seq, c->len[seq] + n}}, st);
    if (rc != HY_OK) return rc;
  }
  if (m->chunk_prefill && n > 0) {
    const int P = std::min(n, prefill_chunk_rows());
    int rc = prefill_buffers(c, P);
    if (rc != HY_OK) return rc;
    const int t_start = c->len[seq];
    for (int i0 = 0; i0 < n; i0 += P) {
      const int cn = std::min(P, n - i0);
      rc = prefill_chunk(c, seq, tokens_dev + i0, cn, t_start + i0, i0 + cn == n, logits_dev, st);
      if (rc != HY_OK) return rc;
    }
    cudaError_t e = prefill::set_len(c->d_len + seq, t_start + n, st);
    if (e != cudaSuccess) return fail(HY_ERR_CUDA, "position update: %s", cudaGetErrorString(e));
    c->len[seq] = t_start + n;
    return HY_OK;
  }
  const std::vector<int> one{seq};
  for (int i = 0; i < n; ++i) {
    float* lg = (i == n - 1) ? logits_dev : nullptr;
    int rc;
    if (m->q4) {  // 4-bit weights: the batched path, with one sequence
      HY_CK(cudaMemcpyAsync(c->btok, tokens_dev + i, sizeof(int), cudaMemcpyDeviceToDevice, st));
      rc = run_batch(c, one, lg, c->bids, st);
    } else {
      HY_CK(cudaMemcpyAsync(c->tok, tokens_dev + i, sizeof(int), cudaMemcpyDeviceToDevice, st));
      rc = run_step(c, seq, lg, c->ids, st);
    }
    if (rc != HY_OK) return rc;
    c->len[seq] += 1;
  }
  return HY_OK;
}

namespace {
// Checks of a decode step's sequence list (distinct, valid, not full).
int check_seqs(hy_cache* c, const int32_t* seqs_host, int32_t nseq, std::vector<int>& seqs) {
  if (nseq < 1 || nseq > bgemv::kMaxB) return fail(HY_ERR_ARG, "nseq must be in 1..%d", bgemv::kMaxB);
  const hy_model* m = c->m;
  // the batched MoE step keeps the union of the tokens' picks in kMaxUnion
  // slots; refuse here, before any launch, rather than part-way through a step
  if (m->moe && (nseq > 1 || m->q4) && nseq * m->cfg.top_k > bgemv::kMaxUnion)
    return fail(HY_ERR_UNSUPPORTED, "a batched MoE step holds at most %d routed picks: %d sequences x top_k %d",
                bgemv::kMaxUnion, nseq, m->cfg.top_k);
  seqs.assign(seqs_host, seqs_host + nseq);
  for (int i = 0; i < nseq; ++i) {
    if (!valid_seq(c, seqs[i])) return fail(HY_ERR_ARG, "bad sequence handle %d", seqs[i]);
    for (int j = 0; j < i; ++j)
      if (seqs[j] == seqs[i]) return fail(HY_ERR_ARG, "sequence %d appears twice in one step", seqs[i]);
    if (c->len[seqs[i]] >= c->cap[seqs[i]])
      return fail(HY_ERR_CAPACITY, "sequence %d is at its capacity %d", seqs[i], c->cap[seqs[i]]);
  }
  return HY_OK;
}
}  // namespace

int hy_decode_step(hy_model* m, hy_cache* c, const int32_t* seqs_host, int32_t nseq, const int32_t* tokens_dev,
                   float* logits_dev, int32_t* ids_dev, void* stream) {
  if (!m || !c || c->m != m || !seqs_host || !tokens_dev || !ids_dev) return fail(HY_ERR_ARG, "null argument");
  std::vector<int> seqs;
  int rc = check_seqs(c, seqs_host, nseq, seqs);
  if (rc != HY_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  {
    std::vector<std::pair<int, int>> need;
    for (int s_ : seqs) need.push_back({s_, c->len[s_] + 1});
    if ((rc = ensure_pages(c, need, st)) != HY_OK) return rc;
  }
  if (nseq == 1 && !m->q4) {
    HY_CK(cudaMemcpyAsync(c->tok, tokens_dev, sizeof(int), cudaMemcpyDeviceToDevice, st));
    rc = run_step(c, seqs[0], logits_dev, ids_dev, st);
  } else {
    HY_CK(cudaMemcpyAsync(c->btok, tokens_dev, sizeof(int) * nseq, cudaMemcpyDeviceToDevice, st));
    rc = run_batch(c, seqs, logits_dev, ids_dev, st);
  }
  if (rc != HY_OK) return rc;
  for (int s : seqs) c->len[s] += 1;
  return HY_OK;
}

int hy_decode_step_host(hy_model* m, hy_cache* c, const int32_t* seqs_host, int32_t nseq, const int32_t* tokens_host,
                        float* logits_host, int32_t* ids_host, void* stream) {
  if (!m || !c || c->m != m || !seqs_host || !tokens_host || !ids_host) return fail(HY_ERR_ARG, "null argument");
  std::vector<int> seqs;
  int rc = check_seqs(c, seqs_host, nseq, seqs);
  if (rc != HY_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  {
    std::vector<std::pair<int, int>> need;
    for (int s_ : seqs) need.push_back({s_, c->len[s_] + 1});
    if ((rc = ensure_pages(c, need, st)) != HY_OK) return rc;
  }
  float* lg = logits_host ? c->logits_buf : nullptr;
  int* ids = nullptr;
  if (nseq == 1 && !m->q4) {
    HY_CK(cudaMemcpyAsync(c->tok, tokens_host, sizeof(int), cudaMemcpyHostToDevice, st));
    ids = c->ids;
    rc = run_step(c, seqs[0], lg, ids, st);
  } else {
    HY_CK(cudaMemcpyAsync(c->btok, tokens_host, sizeof(int) * nseq, cudaMemcpyHostToDevice, st));
    ids = c->bids;
    rc = run_batch(c, seqs, lg, ids, st);
  }
  if (rc != HY_OK) return rc;
  for (int s : seqs) c->len[s] += 1;
  HY_CK(cudaMemcpyAsync(ids_host, ids, sizeof(int) * nseq, cudaMemcpyDeviceToHost, st));
  if (logits_host)
    HY_CK(cudaMemcpyAsync(logits_host, c->logits_buf, sizeof(float) * (size_t)m->cfg.vocab * nseq,
                          cudaMemcpyDeviceToHost, st));
  HY_CK(cudaStreamSynchronize(st));
  return HY_OK;
}

int hy_check_device(hy_cache* c, void* stream, uint32_t* bits_out) {
  if (!c) return fail(HY_ERR_ARG, "null cache");
  cudaStream_t st = (cudaStream_t)stream;
  unsigned bits = 0;
  HY_CK(cudaMemcpyAsync(&bits, c->guard, sizeof(unsigned), cudaMemcpyDeviceToHost, st));
  HY_CK(cudaStreamSynchronize(st));
  if (bits_out) *bits_out = bits;
  if (bits) {
    HY_CK(cudaMemsetAsync(c->guard, 0, sizeof(unsigned), st));
    HY_CK(cudaStreamSynchronize(st));
    return fail(HY_ERR_DEVICE_GUARD, "device guard bits 0x%x", bits);
  }
  return HY_OK;
}

int hy_debug_hidden(hy_cache* c, int32_t layer, float* dst_dev, void* stream) {
  if (!c || !dst_dev || layer < 0 || layer >= c->m->cfg.n_layers) return fail(HY_ERR_ARG, "bad argument");
  if (!c->m->debug) return fail(HY_ERR_ARG, "model was created without HY_FLAG_DEBUG");
  HY_CK(cudaMemcpyAsync(dst_dev, c->dbg_hidden + (size_t)layer * c->m->cfg.hidden, sizeof(float) * c->m->cfg.hidden,
                        cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
  return HY_OK;
}

int hy_debug_router(hy_cache* c, int32_t layer, float* logits_dev, int32_t* ids_dev, void* stream) {
  if (!c || layer < 0 || layer >= c->m->cfg.n_layers) return fail(HY_ERR_ARG, "bad argument");
  if (!c->m->debug || !c->m->moe) return fail(HY_ERR_ARG, "needs a MoE model created with HY_FLAG_DEBUG");
  const hy_config& cf = c->m->cfg;
  cudaStream_t st = (cudaStream_t)stream;
  if (logits_dev)
    HY_CK(cudaMemcpyAsync(logits_dev, c->dbg_rlog + (size_t)layer * (cf.n_experts + 1),
                          sizeof(float) * (cf.n_experts + 1), cudaMemcpyDeviceToDevice, st));
  if (ids_dev)
    HY_CK(cudaMemcpyAsync(ids_dev, c->dbg_rids + (size_t)layer * cf.top_k, sizeof(int) * cf.top_k,
                          cudaMemcpyDeviceToDevice, st));
  return HY_OK;
}

// ---------------------------------------------------------------- single ops

static int op_guard(unsigned** g) {
  int dev = 0, nsm = 0;
  int rc = current_device(&dev, &nsm);
  if (rc != HY_OK) return rc;
  if ((rc = ensure_init(dev)) != HY_OK) return rc;
  std::lock_guard<std::mutex> lk(g_init_mu);
  auto it = g_op_guard.find(dev);
  if (it == g_op_guard.end()) {
    unsigned* p = nullptr;
    HY_CK(cudaMalloc(&p, sizeof(unsigned)));
    HY_CK(cudaMemset(p, 0, sizeof(unsigned)));
    it = g_op_guard.emplace(dev, p).first;
  }
  *g = it->second;
  return HY_OK;
}

static int op_nsm() {
  int dev = 0, nsm = 0;
  if (current_device(&dev, &nsm) != HY_OK) return 0;
  return nsm;
}

static int op_gemv_run(gemv::Params& p, int in, int epi, void* stream) {
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  p.guard = guard;
  const gemv::Plan pl = gemv::plan(p.R, p.C, epi == gemv::kEpiSwiglu ? 2 : 1, op_nsm(), p.norm_g != nullptr);
  if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for %d x %d", p.R, p.C);
  cudaError_t e = gemv::launch(p, pl, gemv::kSrcDense, in, epi, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "GEMV launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

int hy_op_gemv(const void* W_dev, int32_t rows, int32_t cols, const float* x_dev, const float* norm_g_dev, float eps,
               float* y_dev, int32_t accumulate, void* stream) {
  if (!aligned16(W_dev) || !aligned16(x_dev) || !y_dev || rows <= 0 || cols <= 0 || cols % 8)
    return fail(HY_ERR_ARG, "bad GEMV arguments");
  gemv::Params p;
  memset(&p, 0, sizeof(p));
  p.W[0] = (const uint8_t*)W_dev;
  p.R = rows;
  p.C = cols;
  p.x = x_dev;
  p.norm_g = norm_g_dev;
  p.eps = eps;
  p.y = y_dev;
  return op_gemv_run(p, gemv::kInX, accumulate ? gemv::kEpiResid : gemv::kEpiStore, stream);
}

int hy_op_gemv_swiglu(const void* Wg_dev, const void* Wu_dev, int32_t rows, int32_t cols, const float* x_dev,
                      const float* norm_g_dev, float eps, float* h_dev, void* stream) {
  if (!aligned16(Wg_dev) || !aligned16(Wu_dev) || !aligned16(x_dev) || !h_dev || rows <= 0 || cols <= 0 || cols % 8)
    return fail(HY_ERR_ARG, "bad GEMV arguments");
  gemv::Params p;
  memset(&p, 0, sizeof(p));
  p.W[0] = (const uint8_t*)Wg_dev;
  p.W[1] = (const uint8_t*)Wu_dev;
  p.R = rows;
  p.C = cols;
  p.x = x_dev;
  p.norm_g = norm_g_dev;
  p.eps = eps;
  p.y = h_dev;
  return op_gemv_run(p, gemv::kInX, gemv::kEpiSwiglu, stream);
}

int hy_op_gemv_batch(const hy_tensor* w, const hy_tensor* w_up, int32_t weight_format, int32_t rows, int32_t cols,
                     int32_t batch, const float* x_dev, int32_t ldx, const float* norm_g_dev, float eps, float* y_dev,
                     int32_t ldy, int32_t accumulate, void* stream) {
  if (!w || !aligned16(w->w) || !x_dev || !y_dev || rows <= 0 || cols <= 0 || batch < 1 ||
      batch > bgemv::kMaxB || ldx < cols || ldy < rows || (weight_format != 0 && weight_format != 1))
    return fail(HY_ERR_ARG, "bad batched GEMV arguments");
  if (weight_format == 1 && !aligned16(w->scales)) return fail(HY_ERR_ARG, "4-bit weights need scales");
  if (w_up && (!aligned16(w_up->w) || (weight_format == 1 && !aligned16(w_up->scales))))
    return fail(HY_ERR_ARG, "bad up matrix");
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  bgemv::Params p;
  memset(&p, 0, sizeof(p));
  p.fmt = weight_format;
  p.in = bgemv::kInX;
  p.epi = w_up ? bgemv::kEpiSwiglu : (accumulate ? bgemv::kEpiResid : bgemv::kEpiStore);
  p.W[0] = (const uint8_t*)w->w;
  p.S[0] = (const uint16_t*)w->scales;
  if (w_up) {
    p.W[1] = (const uint8_t*)w_up->w;
    p.S[1] = (const uint16_t*)w_up->scales;
  }
  p.R = rows;
  p.C = cols;
  p.B = batch;
  p.x = x_dev;
  p.ldx = ldx;
  p.norm_g = norm_g_dev;
  p.eps = eps;
  p.y = y_dev;
  p.ldy = ldy;
  p.guard = guard;
  const bgemv::Plan pl = bgemv::plan(rows, cols, weight_format, p.epi, op_nsm());
  if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no batched GEMV plan for %d x %d (format %d)", rows, cols, weight_format);
  cudaError_t e = bgemv::launch(p, pl, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "batched GEMV launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

int hy_op_check_device(void* stream, uint32_t* bits_out) {
  cudaStream_t st = (cudaStream_t)stream;
  unsigned* words[2] = {nullptr, hy::noalloc_guard()};
  {
    int dev = 0;
    HY_CK(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_init_mu);
    auto it = g_op_guard.find(dev);  // never created here: this call allocates nothing
    if (it != g_op_guard.end()) words[0] = it->second;
  }
  unsigned got[2] = {0u, 0u};
  for (int i = 0; i < 2; ++i)
    if (words[i]) HY_CK(cudaMemcpyAsync(&got[i], words[i], sizeof(unsigned), cudaMemcpyDeviceToHost, st));
  HY_CK(cudaStreamSynchronize(st));
  const unsigned bits = got[0] | got[1];
  if (bits_out) *bits_out = bits;
  if (!bits) return HY_OK;
  for (int i = 0; i < 2; ++i)
    if (got[i]) HY_CK(cudaMemsetAsync(words[i], 0, sizeof(unsigned), st));
  HY_CK(cudaStreamSynchronize(st));
  return fail(HY_ERR_DEVICE_GUARD, "device guard bits 0x%x", bits);
}

namespace {
size_t split_part_bytes(int32_t M, int32_t K) { return ((size_t)M * K * 2 + 255) / 256 * 256; }

// The activations of a prompt GEMM op: RMSNorm (optional) and the bf16 hi / lo
// split into the workspace, then the GEMM.
int op_gemm_run(gemm::Params& p, const void* W0, const void* W1, const float* x_dev, int32_t ldx,
                const float* norm_g_dev, float eps, void* workspace_dev, void* stream) {
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  p.guard = guard;
  cudaStream_t st = (cudaStream_t)stream;
  uint16_t* hi = (uint16_t*)workspace_dev;
  uint16_t* lo = (uint16_t*)((uint8_t*)workspace_dev + split_part_bytes(p.M, p.K));
  cudaError_t e = gemm::norm_split(x_dev, ldx, norm_g_dev, eps, p.M, p.K, hi, lo, p.K, st);
  if (e == cudaSuccess) e = gemm::launch(p, hi, lo, p.K, (const uint16_t*)W0, (const uint16_t*)W1, p.K, st);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "prompt GEMM launch: %s", cudaGetErrorString(e));
  return HY_OK;
}
}  // namespace

size_t hy_op_gemm_workspace(int32_t M, int32_t K) {
  if (M <= 0 || K <= 0) return 0;
  return 2 * split_part_bytes(M, K);
}

int hy_op_gemm(const void* W_dev, int32_t N, int32_t K, int32_t M, const float* x_dev, int32_t ldx,
               const float* norm_g_dev, float eps, float* y_dev, int32_t ldy, int32_t accumulate, void* workspace_dev,
               void* stream) {
  if (!aligned16(W_dev) || !x_dev || !y_dev || !aligned16(workspace_dev) || N <= 0 || M <= 0 || K <= 0 || K % 8 ||
      ldx < K || ldy < N)
    return fail(HY_ERR_ARG, "bad prompt GEMM arguments");
  gemm::Params p;
  memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.epi = accumulate ? gemm::kEpiResid : gemm::kEpiStore;
  p.y = y_dev;
  p.ldy = ldy;
  return op_gemm_run(p, W_dev, nullptr, x_dev, ldx, norm_g_dev, eps, workspace_dev, stream);
}

int hy_op_gemm_swiglu(const void* Wg_dev, const void* Wu_dev, int32_t N, int32_t K, int32_t M, const float* x_dev,
                      int32_t ldx, const float* norm_g_dev, float eps, uint16_t* h_hi_dev, uint16_t* h_lo_dev,
                      int32_t ldh, void* workspace_dev, void* stream) {
  if (!aligned16(Wg_dev) || !aligned16(Wu_dev) || !x_dev || !h_hi_dev || !h_lo_dev || !aligned16(workspace_dev) ||
      N <= 0 || M <= 0 || K <= 0 || K % 8 || ldx < K || ldh < N)
    return fail(HY_ERR_ARG, "bad prompt GEMM arguments");
  gemm::Params p;
  memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.epi = gemm::kEpiSwigluSplit;
  p.h_hi = h_hi_dev;
  p.h_lo = h_lo_dev;
  p.ldh = ldh;
  return op_gemm_run(p, Wg_dev, Wu_dev, x_dev, ldx, norm_g_dev, eps, workspace_dev, stream);
}

int hy_op_moe_gateup(const void* exp_gate_dev, const void* exp_up_dev, const void* sh_gate_dev, const void* sh_up_dev,
                     int32_t n_experts, int32_t top_k, int32_t expert_ffn, int32_t hidden,
                     const float* router_logits_dev, const float* x_dev, const float* norm_g_dev, float eps,
                     float* h_dev, int32_t* ids_dev, float* w_dev, void* stream) {
  if (!aligned16(exp_gate_dev) || !aligned16(exp_up_dev) || !aligned16(sh_gate_dev) || !aligned16(sh_up_dev) ||
      !router_logits_dev || !aligned16(x_dev) || !h_dev || !ids_dev || !w_dev || n_experts < 1 || top_k < 1 ||
      top_k > gemv::kMaxTopK || top_k > n_experts || expert_ffn <= 0 || hidden <= 0 || hidden % 8)
    return fail(HY_ERR_ARG, "bad MoE gate/up arguments");
  if (n_experts > gemv::kMaxExperts - 1) return fail(HY_ERR_UNSUPPORTED, "at most %d routed experts", gemv::kMaxExperts - 1);
  gemv::Params p;
  memset(&p, 0, sizeof(p));
  p.exp_base[0] = (const uint8_t*)exp_gate_dev;
  p.exp_base[1] = (const uint8_t*)exp_up_dev;
  p.sh_base[0] = (const uint8_t*)sh_gate_dev;
  p.sh_base[1] = (const uint8_t*)sh_up_dev;
  p.exp_stride = (long long)expert_ffn * hidden * 2;
  p.moe_ids = ids_dev;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.slot_rows = expert_ffn;
  p.sh_rows = expert_ffn;
  p.R = (top_k + 1) * expert_ffn;
  p.C = hidden;
  p.x = x_dev;
  p.norm_g = norm_g_dev;
  p.eps = eps;
  p.y = h_dev;
  p.route_here = 1;
  p.router_logits = router_logits_dev;
  p.out_ids = ids_dev;
  p.out_w = w_dev;
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  p.guard = guard;
  const gemv::Plan pl = gemv::plan(p.R, p.C, 2, op_nsm(), norm_g_dev != nullptr);
  if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for the expert gate/up (%d x %d)", p.R, p.C);
  cudaError_t e = gemv::launch(p, pl, gemv::kSrcExpertRows, gemv::kInX, gemv::kEpiSwiglu, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "expert gate/up launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

int hy_op_moe_down(const void* exp_down_dev, const void* sh_down_dev, int32_t n_experts, int32_t top_k,
                   int32_t expert_ffn, int32_t hidden, const int32_t* ids_dev, const float* w_dev, const float* h_dev,
                   float* y_dev, void* stream) {
  if (!aligned16(exp_down_dev) || !aligned16(sh_down_dev) || !ids_dev || !aligned16(w_dev) || !aligned16(h_dev) ||
      !y_dev || n_experts < 1 || top_k < 1 || top_k > gemv::kMaxTopK || expert_ffn <= 0 || expert_ffn % 8 ||
      hidden <= 0)
    return fail(HY_ERR_ARG, "bad MoE down arguments");
  gemv::Params p;
  memset(&p, 0, sizeof(p));
  p.exp_base[0] = (const uint8_t*)exp_down_dev;
  p.sh_base[0] = (const uint8_t*)sh_down_dev;
  p.exp_stride = (long long)hidden * expert_ffn * 2;
  p.moe_ids = ids_dev;
  p.moe_w = w_dev;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.seg_cols = expert_ffn;
  p.R = hidden;
  p.C = (top_k + 1) * expert_ffn;
  p.x = h_dev;
  p.y = y_dev;
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  p.guard = guard;
  const gemv::Plan pl = gemv::plan(p.R, p.C, 1, op_nsm(), false);
  if (!pl.ok) return fail(HY_ERR_UNSUPPORTED, "no GEMV plan for the expert down (%d x %d)", p.R, p.C);
  cudaError_t e = gemv::launch(p, pl, gemv::kSrcExpertSegs, gemv::kInMoeZ, gemv::kEpiResid, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "expert down launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

size_t hy_op_argmax_workspace(void) { return 256 + 1024 * 8; }

int hy_op_gemv_argmax(const void* W_dev, int32_t rows, int32_t cols, const float* x_dev, const float* norm_g_dev,
                      float eps, float* logits_dev, int32_t* id_dev, void* workspace_dev, void* stream) {
  if (!aligned16(W_dev) || !aligned16(x_dev) || !id_dev || !aligned16(workspace_dev) || rows <= 0 || cols <= 0 ||
      cols % 8)
    return fail(HY_ERR_ARG, "bad GEMV arguments");
  uint8_t* ws = (uint8_t*)workspace_dev;
  gemv::Params p;
  memset(&p, 0, sizeof(p));
  p.W[0] = (const uint8_t*)W_dev;
  p.R = rows;
  p.C = cols;
  p.x = x_dev;
  p.norm_g = norm_g_dev;
  p.eps = eps;
  p.y = logits_dev;
  p.counter = (unsigned*)ws;
  p.part_val = (float*)(ws + 256);
  p.part_idx = (int*)(ws + 256 + 1024 * 4);
  p.ids_out = id_dev;
  return op_gemv_run(p, gemv::kInX, gemv::kEpiArgmax, stream);
}

int hy_op_gdn_step(const float* y_dev, const void* conv_w_dev, float* conv_state_dev, float* S_dev, float* o_dev,
                   int32_t nh, int32_t dk, int32_t dv, int32_t conv_k, const int32_t* pos_dev, void* stream) {
  if (!y_dev || !conv_w_dev || !conv_state_dev || !aligned16(S_dev) || !o_dev || !pos_dev || nh <= 0 || dv <= 0)
    return fail(HY_ERR_ARG, "bad GDN arguments");
  if (dk != 64 && dk != 128 && dk != 256) return fail(HY_ERR_UNSUPPORTED, "dk must be 64, 128 or 256");
  if (conv_k < 1 || conv_k > 8) return fail(HY_ERR_ARG, "conv_k must be in 1..8");
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  gdn::Params g;
  memset(&g, 0, sizeof(g));
  g.y = y_dev;
  g.conv_w = (const uint16_t*)conv_w_dev;
  g.conv_state = conv_state_dev;
  g.S = S_dev;
  g.o = o_dev;
  g.nh = nh;
  g.dk = dk;
  g.dv = dv;
  g.conv_k = conv_k;
  g.pos = pos_dev;
  g.guard = guard;
  cudaError_t e = gdn::launch(g, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "GDN launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

int hy_op_rope_table(float* table_dev, int32_t cap, int32_t hd, float theta, void* stream) {
  if (!table_dev || cap <= 0 || hd <= 0 || hd % 2) return fail(HY_ERR_ARG, "bad RoPE table arguments");
  cudaError_t e = attn::rope_table((float2*)table_dev, cap, hd, (double)theta, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "RoPE table: %s", cudaGetErrorString(e));
  return HY_OK;
}

int hy_op_attention_i8(const float* y_dev, void* Kq_dev, float* Ks_dev, void* Vq_dev, float* Vs_dev, int32_t cap,
                       int32_t nq, int32_t nkv, int32_t hd, const int32_t* len_dev, const float* rope_table_dev,
                       int32_t nsplit, float* o_dev, void* workspace_dev, void* stream) {
  if (!y_dev || !aligned16(Kq_dev) || !aligned16(Vq_dev) || !aligned16(Ks_dev) || !aligned16(Vs_dev) || !len_dev ||
      !rope_table_dev || !o_dev || !aligned16(workspace_dev) || cap <= 0 || nkv <= 0 || nq <= 0 || nq % nkv)
    return fail(HY_ERR_ARG, "bad attention arguments");
  if ((hd != 64 && hd != 128 && hd != 256) || nq / nkv > 8 || ((nq / nkv) & (nq / nkv - 1)))
    return fail(HY_ERR_UNSUPPORTED, "attention: head_dim 64/128/256 and nq/nkv in {1,2,4,8}");
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  if (nsplit <= 0) nsplit = attn::auto_splits(nkv, op_nsm());
  uint8_t* ws = (uint8_t*)workspace_dev;
  attn::Params a;
  memset(&a, 0, sizeof(a));
  a.y = y_dev;
  a.K = (uint16_t*)Kq_dev;
  a.V = (uint16_t*)Vq_dev;
  a.kv8 = 1;
  a.Ks = Ks_dev;
  a.Vs = Vs_dev;
  a.cap_s = cap_scales(cap);
  a.len = len_dev;
  a.rope = (const float2*)rope_table_dev;
  a.cap = cap;
  a.nq = nq;
  a.nkv = nkv;
  a.hd = hd;
  a.nsplit = nsplit;
  a.scale = 1.0f / sqrtf((float)hd);
  a.counter = (unsigned*)ws;
  a.part = (float*)(ws + 256 + ((size_t)nkv * 4 + 255) / 256 * 256);
  a.o = o_dev;
  a.guard = guard;
  cudaError_t e = attn::launch(a, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

size_t hy_op_attention_workspace(int32_t nq, int32_t nkv, int32_t hd, int32_t nsplit) {
  if (nkv <= 0 || nq <= 0) return 0;
  if (nsplit <= 0) nsplit = attn::auto_splits(nkv, op_nsm());
  return 256 + ((size_t)nkv * 4 + 255) / 256 * 256 + attn::part_floats(nq, nkv, hd, nsplit) * 4;
}

int hy_op_attention(const float* y_dev, void* K_dev, void* V_dev, int32_t cap, int32_t nq, int32_t nkv, int32_t hd,
                    const int32_t* len_dev, const float* rope_table_dev, int32_t nsplit, float* o_dev,
                    void* workspace_dev, void* stream) {
  if (!y_dev || !aligned16(K_dev) || !aligned16(V_dev) || !len_dev || !rope_table_dev || !o_dev ||
      !aligned16(workspace_dev) || cap <= 0 || nkv <= 0 || nq <= 0 || nq % nkv)
    return fail(HY_ERR_ARG, "bad attention arguments");
  if ((hd != 64 && hd != 128 && hd != 256) || nq / nkv > 8 || ((nq / nkv) & (nq / nkv - 1)))
    return fail(HY_ERR_UNSUPPORTED, "attention: head_dim 64/128/256 and nq/nkv in {1,2,4,8}");
  unsigned* guard = nullptr;
  int rc = op_guard(&guard);
  if (rc != HY_OK) return rc;
  if (nsplit <= 0) nsplit = attn::auto_splits(nkv, op_nsm());
  uint8_t* ws = (uint8_t*)workspace_dev;
  attn::Params a;
  memset(&a, 0, sizeof(a));
  a.y = y_dev;
  a.K = (uint16_t*)K_dev;
  a.V = (uint16_t*)V_dev;
  a.len = len_dev;
  a.rope = (const float2*)rope_table_dev;
  a.cap = cap;
  a.nq = nq;
  a.nkv = nkv;
  a.hd = hd;
  a.nsplit = nsplit;
  a.scale = 1.0f / sqrtf((float)hd);
  a.counter = (unsigned*)ws;
  a.part = (float*)(ws + 256 + ((size_t)nkv * 4 + 255) / 256 * 256);
  a.o = o_dev;
  a.guard = guard;
  cudaError_t e = attn::launch(a, (cudaStream_t)stream, false);
  if (e != cudaSuccess) return fail(HY_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

}  // extern "C"

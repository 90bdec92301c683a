// GQA decode attention on sm_103a: RoPE + bf16 KV append + split-KV partial
// softmax + log-sum-exp combine, one launch.
//
// Prior art: "Beating llama.cpp from Scratch on Consumer AMD", Act 4 (a
// decode attention whose KV scan is split into partial sums over segments of
// the cache and reduced in shared memory) and "What Broke" section 1 (that
// design was capped at 14,080 tokens by its per-block shared-memory need;
// going further needs partial sums combined across separate workgroups).
// Here each split is its own CTA with no length-dependent shared memory:
//   grid (kv_heads, splits); CTA (g, s) owns positions [s L / S, (s+1) L / S)
//   of kv head g (L = T + 1 keys), streams its K and V rows HBM -> shared
//   memory as separate tiles with bulk copies (one copy warp, a 6-stage ring,
//   started before griddepcontrol.wait since earlier positions were written
//   by earlier steps), and serves all G = nq / nkv query heads of the group
//   from one read of each K/V row.
//   Per chunk of up to 512 positions: scores of all its K tiles (8 bf16 per
//   lane, head sums reduce-scattered across the lanes of a row), one online
//   softmax pass per head, then P V over its V tiles with each thread owning
//   two output dims; warps release tiles one by one, so a chunk costs three
//   block barriers whatever its tile count.  The CTA holding position T
//   rotates and rounds the new k/v to bf16, appends them to the cache and
//   attends to them from shared memory as the chunk's last row.
//   Partials (m, l, o) go to a scratch buffer and are merged
//     m = max_s m_s,  o = sum_s e^{m_s - m} o_s / sum_s e^{m_s - m} l_s
//   by the last few CTAs of a kv head to finish, each a slice of the outputs
//   (a ticket counter: earlier CTAs exit at once, the last ones wait for the
//   very last, bounded, then merge together).
// A batch of tokens (each its own sequence and cache) runs in one launch:
// grid (kv_heads, splits, tokens), or (kv_heads, spread) with the spread's
// rows shared among the tokens in proportion to their cache lengths, so that
// ragged contexts give every CTA about the same number of rows.
#include "attn_kernel.cuh"

namespace hy {
namespace attn {
namespace {

template <int HD, int G>
void* kern(bool kv8) {
  return kv8 ? (void*)k_attn<HD, G, true, false> : (void*)k_attn<HD, G, false, false>;
}

void* pick(int hd, int G, size_t* smem, bool kv8) {
#define HY_ATTN_CASE(H_, G_)            \
  if (hd == H_ && G == G_) {            \
    *smem = Smem<H_, G_>::total;        \
    return kern<H_, G_>(kv8);           \
  }
  HY_ATTN_CASE(64, 1) HY_ATTN_CASE(64, 2) HY_ATTN_CASE(64, 4) HY_ATTN_CASE(64, 8)
  HY_ATTN_CASE(128, 1) HY_ATTN_CASE(128, 2) HY_ATTN_CASE(128, 4) HY_ATTN_CASE(128, 8)
  HY_ATTN_CASE(256, 1) HY_ATTN_CASE(256, 2) HY_ATTN_CASE(256, 4) HY_ATTN_CASE(256, 8)
#undef HY_ATTN_CASE
  return nullptr;
}

__global__ void k_rope_table(float2* tab, int cap, int hd, double theta) {
  const int half = hd / 2;
  const long long n = (long long)cap * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / half), i = (int)(e % half);
    const double ang = (double)t * pow(theta, -2.0 * (double)i / (double)hd);
    double s, c;
    sincos(ang, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

}  // namespace

size_t part_floats(int nq, int nkv, int hd, int nsplit) {
  return (size_t)nkv * nsplit * (nq / nkv) * (hd + 2);
}

int auto_splits(int nkv, int nsm) {
  int s = (2 * nsm) / (nkv > 0 ? nkv : 1);
  if (s < 1) s = 1;
  if (s > 32) s = 32;
  return s;
}

// The decode step's splits: one CTA per SM over all kv heads, at least the
// automatic count (measured in the step: dense 4B 38 splits 685.3 tokens/s
// against 683.8 with 32; MoE 35B-A3B 76 splits 578.3 against 573.5).
int step_splits(int nkv, int nsm) {
  const int s1 = auto_splits(nkv, nsm);
  int s = nsm / (nkv > 0 ? nkv : 1);
  if (s > 96) s = 96;
  return s > s1 ? s : s1;
}

// Long contexts (a cache of kLongContext positions or more): with up to 4
// query heads per kv head, 64 splits run as CTA pairs (measured on the dense
// 4B shape at context 32k: 641 tokens/s against 629 with 32 splits; at 4k,
// 32 splits stay ahead, 686 against 685).
int long_context_splits(int nq, int nkv, int nsm) {
  const int G = nkv > 0 ? nq / nkv : 1;
  const int s1 = step_splits(nkv, nsm);
  if (G > 4) return s1;
  int s = (2 * nsm) / (nkv > 0 ? nkv : 1);
  if (s > 64) s = 64;
  return s > s1 ? s : s1;
}

cudaError_t init() {
  const int hds[] = {64, 128, 256};
  const int gs[] = {1, 2, 4, 8};
  for (int h : hds)
    for (int gg : gs)
      for (int kv8 = 0; kv8 < 2; ++kv8) {
        size_t smem = 0;
        void* k = pick(h, gg, &smem, kv8 != 0);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
      }
  return init_pair();
}

cudaError_t launch(const Params& p, cudaStream_t st, bool pdl) {
  if (p.nkv <= 0 || p.nq % p.nkv != 0 || p.nsplit < 1) return cudaErrorInvalidValue;
  if (p.kv8 && (p.cap_s % 4 || p.cap_s < p.cap)) return cudaErrorInvalidValue;
  if (p.pages && (p.kv8 || p.page_tokens <= 0 || p.page_tokens % 128)) return cudaErrorInvalidValue;
  if (p.nb < 0 || p.nb > 8 || p.nsplit > 0xFFFF) return cudaErrorInvalidValue;
  if (p.spread < 0 || (p.spread > 0 && (p.nb < 1 || p.spread < p.nb || p.spread > 0xFFFF)))
    return cudaErrorInvalidValue;
  // Mergers per kv head: enough that each merges about 16 partial values
  // per thread; while they wait, at most (mergers - 1) CTAs per head and
  // token hold an SM, which must leave at least one SM for the CTAs they wait
  // for (every SM holds at least one CTA).
  static int nsm_of[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (nsm_of[dev] == 0) {
    int n = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    nsm_of[dev] = n;
  }
  // more CTAs than SMs: the CTA-pair variant where it exists
  // grid rows: splits of one token (z over the batch), or of the whole batch (spread)
  const int rows = p.spread > 0 ? p.spread : p.nsplit, zs = (p.nb > 0 && p.spread == 0) ? p.nb : 1;
  const long long grid = (long long)p.nkv * rows * zs;
  size_t smem = 0;
  void* k = grid > nsm_of[dev] ? pick_pair(p.hd, p.nq / p.nkv, &smem, p.kv8 != 0) : nullptr;
  if (!k) k = pick(p.hd, p.nq / p.nkv, &smem, p.kv8 != 0);
  if (!k) return cudaErrorInvalidValue;
  Params q = p;
  // partial o values of one kv head (spread: of a token's average share; the
  // kernel caps the mergers at each token's own split count)
  const long long per = p.spread > 0 ? (p.spread + p.nb - 1) / p.nb : p.nsplit;
  const long long values = (long long)p.nq * p.hd * per / p.nkv;
  long long K = (values + 16 * kCT - 1) / (16 * kCT);
  const long long groups = (long long)p.nkv * (p.nb > 0 ? p.nb : 1);
  const long long kmax = (nsm_of[dev] - 1) / groups + 1;
  if (K > kmax) K = kmax;
  if (K > per) K = per;
  q.mergers = K < 1 ? 1 : (int)K;
  return launch_k(reinterpret_cast<void (*)(Params)>(k), dim3(p.nkv, rows, zs), dim3(kThreads),
                  smem, st, pdl, q);
}

cudaError_t rope_table(float2* tab, int cap, int hd, double theta, cudaStream_t st) {
  if (cap <= 0) return cudaSuccess;
  const long long n = (long long)cap * (hd / 2);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  k_rope_table<<<blocks, 256, 0, st>>>(tab, cap, hd, theta);
  return cudaGetLastError();
}

}  // namespace attn
}  // namespace hy

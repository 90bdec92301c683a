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
#include "attn_dev.cuh"
#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace attn {
namespace {

template <int HD, int G>
struct Smem {
  static constexpr size_t stages = (size_t)kRing * Tile<HD>::kBytes;
  static constexpr size_t work = Work<HD, G>::total;
  static constexpr size_t bars = 2 * kRing * 8;
  static constexpr size_t total = stages + ((work + 15) & ~(size_t)15) + bars + 64;
};

template <int HD, int G, bool KV8>
__global__ void __launch_bounds__(kThreads, 1) k_attn(const Params p0) {
  Params p = p0;
  if (p0.nb > 0) {  // token blockIdx.z of a batch: its sequence's cache and scratch
    const int z = blockIdx.z;
    p.y = p0.y + (long long)z * p0.ld_y;
    p.o = p0.o + (long long)z * p0.ld_o;
    p.part = p0.part + (long long)z * p0.ld_part;
    p.counter = p0.counter + z * p0.nkv;
    p.K = p0.K_b[z];
    p.V = p0.V_b[z];
    p.Ks = p0.Ks_b[z];
    p.Vs = p0.Vs_b[z];
    p.len = p0.len_b[z];
    p.cap = p0.cap_b[z];
    p.cap_s = p0.cap_s_b[z];
    p.pages = p0.pages_b[z];
  }
  using S_ = Smem<HD, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  WorkPtrs<HD, G> w;
  w.carve(smem + S_::stages);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S_::stages + ((S_::work + 15) & ~(size_t)15));
  uint64_t* empty = full + kRing;

  const int g = blockIdx.x, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = *p.len;  // written only by the previous step's last kernel
  if (T < 0 || T >= p.cap) {  // the host checks capacity first; never touch memory past it
    if (threadIdx.x == 0) set_guard(p.guard, kGuardBadPosition);
    return;
  }
  const Item it = item_of<HD>(p, T, sp);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);  // one arrival per compute warp
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kCWarps) {
    pdl_launch_dependents();  // the CTA's trigger needs every thread (or its exit)
    if (lane == 0) {
      // issue order = consumption order: per chunk its K tiles, then its V tiles
      const uint64_t pol = l2_evict_first_policy();
      constexpr int CH = Tile<HD>::CH;
      int q = 0;
      bool ok = true;
      for (int t0 = 0; ok && t0 < it.ntiles; t0 += CH) {
        const int t1 = (t0 + CH < it.ntiles) ? t0 + CH : it.ntiles;
        for (int kv = 0; ok && kv < 2; ++kv)
          for (int t = t0; t < t1; ++t, ++q) {
            const int s = q % kRing;
            if (q >= kRing && !mbar_wait(&empty[s], ((q / kRing) - 1) & 1)) {
              set_guard(p.guard, kGuardWaitTimeout);
              ok = false;
              break;
            }
            issue_tile<HD, KV8>(p, g, it, t, kv, stages + s * Tile<HD>::kBytes, &full[s], pol);
          }
      }
      for (int u = (q > kRing ? q - kRing : 0); u < q; ++u)
        if (!mbar_wait(&full[u % kRing], (u / kRing) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  // Per chunk: scores of its K tiles (each warp releases a tile as it is
  // done), one softmax pass, then P V over its V tiles.  The new row (held in
  // shared memory) is the last row of the last chunk.
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  Acc<HD, G> A;
  begin_item<HD, G, KV8>(p, g, T, it, w, A, ctid);
  constexpr int TP = Tile<HD>::TP, CH = Tile<HD>::CH;
  const int nchunks = it.ntiles > 0 ? (it.ntiles + CH - 1) / CH : 1;
  int q = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int t0 = c * CH, t1 = (t0 + CH < it.ntiles) ? t0 + CH : it.ntiles;
    const bool last = (c == nchunks - 1);
    int rows_c = 0;
    for (int t = t0; t < t1; ++t, ++q) {
      const int s = q % kRing;
      if (!mbar_wait(&full[s], (q / kRing) & 1)) {
        if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
        return;
      }
      const uint8_t* st = stages + s * Tile<HD>::kBytes;
      const int rows = tile_rows<HD>(it, t);
      const float* ks = KV8 ? reinterpret_cast<const float*>(st + scale_off<HD>()) + ((it.p0 + t * TP) & 3) : nullptr;
      tile_scores<HD, G, KV8>(reinterpret_cast<const uint16_t*>(st), rows, rows_c, w, A, ctid, ks);
      rows_c += rows;
      __syncwarp();
      if ((ctid & 31) == 0) mbar_arrive(&empty[s]);
    }
    const bool with_new = last && it.has_new;
    if (with_new) tile_scores<HD, G, KV8>(w.kn, 1, rows_c, w, A, ctid, w.kvs);
    named_barrier(1, kCT);
    chunk_softmax<HD, G>(rows_c + (with_new ? 1 : 0), w, A, ctid);
    int rb = 0;
    for (int t = t0; t < t1; ++t, ++q) {
      const int s = q % kRing;
      if (!mbar_wait(&full[s], (q / kRing) & 1)) {
        if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
        return;
      }
      const uint8_t* st = stages + s * Tile<HD>::kBytes;
      const int rows = tile_rows<HD>(it, t);
      const float* vs = KV8 ? reinterpret_cast<const float*>(st + scale_off<HD>()) + ((it.p0 + t * TP) & 3) : nullptr;
      tile_pv<HD, G, KV8>(reinterpret_cast<const uint16_t*>(st), rows, rb, w, A, ctid, vs);
      rb += rows;
      __syncwarp();
      if ((ctid & 31) == 0) mbar_arrive(&empty[s]);
    }
    if (with_new) tile_pv<HD, G, KV8>(w.vn, 1, rows_c, w, A, ctid, w.kvs + 1);
    if (!last) named_barrier(1, kCT);  // the next chunk's scores overwrite w.sc
  }
  end_item<HD, G>(p, g, sp, w, A, ctid);
}

template <int HD, int G>
void* kern(bool kv8) {
  return kv8 ? (void*)k_attn<HD, G, true> : (void*)k_attn<HD, G, false>;
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
  return cudaSuccess;
}

cudaError_t launch(const Params& p, cudaStream_t st, bool pdl) {
  if (p.nkv <= 0 || p.nq % p.nkv != 0 || p.nsplit < 1) return cudaErrorInvalidValue;
  size_t smem = 0;
  void* k = pick(p.hd, p.nq / p.nkv, &smem, p.kv8 != 0);
  if (!k) return cudaErrorInvalidValue;
  if (p.kv8 && (p.cap_s % 4 || p.cap_s < p.cap)) return cudaErrorInvalidValue;
  if (p.pages && (p.kv8 || p.page_tokens <= 0 || p.page_tokens % 128)) return cudaErrorInvalidValue;
  if (p.nb < 0 || p.nb > 8 || p.nsplit > 0xFFFF) return cudaErrorInvalidValue;
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
  Params q = p;
  const long long values = (long long)p.nq * p.hd * p.nsplit / p.nkv;  // partial o values of one kv head
  long long K = (values + 16 * kCT - 1) / (16 * kCT);
  const long long groups = (long long)p.nkv * (p.nb > 0 ? p.nb : 1);
  const long long kmax = (nsm_of[dev] - 1) / groups + 1;
  if (K > kmax) K = kmax;
  if (K > p.nsplit) K = p.nsplit;
  q.mergers = K < 1 ? 1 : (int)K;
  return launch_k(reinterpret_cast<void (*)(Params)>(k), dim3(p.nkv, p.nsplit, p.nb > 0 ? p.nb : 1), dim3(kThreads),
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

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
//   of kv head g (L = T + 1 keys), streams its K/V rows HBM -> shared memory
//   with bulk copies (one copy warp, 3 stages, started before
//   griddepcontrol.wait since earlier positions were written by earlier
//   steps), and serves all G = nq / nkv query heads of the group from one
//   read of each K/V row.
//   Per tile: scores (8 bf16 per lane, reduced across the lanes of a row with
//   shuffles) -> online softmax per head -> P V with each thread owning two
//   output dims.  The CTA holding position T rotates and rounds the new k/v
//   to bf16, appends them to the cache and attends to them from shared memory.
//   Partials (m, l, o) go to a scratch buffer; the last CTA of a kv head to
//   finish (atomic ticket, nobody waits) merges them:
//     m = max_s m_s,  o = sum_s e^{m_s - m} o_s / sum_s e^{m_s - m} l_s.
#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace attn {
namespace {

constexpr int kCWarps = 8;
constexpr int kCThreads = kCWarps * 32;

template <int HD>
struct Tile {
  static constexpr int TP = HD >= 256 ? 32 : (HD >= 128 ? 64 : 128);  // positions per tile
  static constexpr int kBytesKV = TP * HD * 2;                          // one of K or V
  static constexpr int kStageBytes = 2 * kBytesKV;
};

template <int HD, int G>
struct Smem {
  static constexpr int NP = HD / 2;              // dim pairs
  static constexpr int NG = kCThreads / NP;      // position groups in P V
  static constexpr size_t stages = (size_t)kStages * Tile<HD>::kStageBytes;
  static constexpr size_t q = (size_t)G * HD * 4;
  static constexpr size_t sc = (size_t)G * Tile<HD>::TP * 4;
  static constexpr size_t ored = (size_t)NG * G * HD * 4;
  static constexpr size_t kvnew = 2 * HD * 2;
  static constexpr size_t bars = 2 * kStages * 8;
  static constexpr size_t total = stages + q + sc + ored + kvnew + bars + 64;
};

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 1) k_attn(const Params p) {
  using T_ = Tile<HD>;
  using S_ = Smem<HD, G>;
  constexpr int TP = T_::TP;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* q_s = reinterpret_cast<float*>(smem + S_::stages);
  float* sc = q_s + G * HD;
  float* ored = sc + G * TP;
  uint16_t* kn_s = reinterpret_cast<uint16_t*>(ored + S_::NG * G * HD);
  uint16_t* vn_s = kn_s + HD;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ((S_::stages + S_::q + S_::sc + S_::ored + S_::kvnew + 7) & ~(size_t)7));
  uint64_t* empty = full + kStages;
  __shared__ float s_m[G], s_l[G], s_corr[G];
  __shared__ int s_last;

  const int g = blockIdx.x, sp = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = *p.len;  // written only by the previous step's last kernel
  if (T < 0 || T >= p.cap) {  // the host checks capacity first; never touch memory past it
    if (threadIdx.x == 0) set_guard(p.guard, kGuardBadPosition);
    return;
  }
  const long long L = (long long)T + 1;
  const int p0 = (int)((long long)sp * L / p.nsplit), p1 = (int)((long long)(sp + 1) * L / p.nsplit);
  const int pc1 = p1 < T ? p1 : T;  // cached rows [p0, pc1)
  const int ncached = pc1 > p0 ? pc1 - p0 : 0;
  const int ntiles = (ncached + TP - 1) / TP;
  const bool has_new = (T >= p0 && T < p1);
  const uint16_t* Kg = p.K + (long long)g * p.cap * HD;
  const uint16_t* Vg = p.V + (long long)g * p.cap * HD;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  if (threadIdx.x < G) {
    s_m[threadIdx.x] = -INFINITY;
    s_l[threadIdx.x] = 0.f;
  }
  __syncthreads();

  // ------------------------------------------------------------ copy warp
  if (warp == kCWarps) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages, k = t / kStages;
        if (t >= kStages && !mbar_wait(&empty[s], (k - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        const int r0 = p0 + t * TP;
        const int rows = (pc1 - r0) < TP ? (pc1 - r0) : TP;
        const uint32_t bytes = (uint32_t)rows * HD * 2;
        uint8_t* dst = stages + s * T_::kStageBytes;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        bulk_g2s(dst, Kg + (long long)r0 * HD, bytes, &full[s], pol);
        bulk_g2s(dst + T_::kBytesKV, Vg + (long long)r0 * HD, bytes, &full[s], pol);
        ++issued;
      }
      const int first = issued > kStages ? issued - kStages : 0;
      for (int u = first; u < issued; ++u)
        if (!mbar_wait(&full[u % kStages], (u / kStages) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const float2* rope = p.rope + (long long)T * (HD / 2);
  // rotated, scaled queries of the G heads of this kv group
  for (int e = ctid; e < G * (HD / 2); e += kCThreads) {
    const int j = e / (HD / 2), i = e % (HD / 2);
    const float* qh = p.y + (long long)(g * G + j) * HD;
    const float2 cs = rope[i];
    const float a = qh[i], b = qh[i + HD / 2];
    q_s[j * HD + i] = (a * cs.x - b * cs.y) * p.scale;
    q_s[j * HD + i + HD / 2] = (b * cs.x + a * cs.y) * p.scale;
  }
  if (has_new) {
    const float* kh = p.y + (long long)(p.nq + g) * HD;
    const float* vh = p.y + (long long)(p.nq + p.nkv + g) * HD;
    uint16_t* Kw = p.K + ((long long)g * p.cap + T) * HD;
    uint16_t* Vw = p.V + ((long long)g * p.cap + T) * HD;
    for (int i = ctid; i < HD / 2; i += kCThreads) {
      const float2 cs = rope[i];
      const float a = kh[i], b = kh[i + HD / 2];
      const uint16_t k0 = f32_to_bf16_rne(a * cs.x - b * cs.y), k1 = f32_to_bf16_rne(b * cs.x + a * cs.y);
      kn_s[i] = k0;
      kn_s[i + HD / 2] = k1;
      Kw[i] = k0;
      Kw[i + HD / 2] = k1;
    }
    for (int i = ctid; i < HD; i += kCThreads) {
      const uint16_t v = f32_to_bf16_rne(vh[i]);
      vn_s[i] = v;
      Vw[i] = v;
    }
  }
  named_barrier(1, kCThreads);

  // per-lane query slice: 8 dims per lane, LPR lanes per K row
  constexpr int LPR = HD / 8, RPW = 32 / LPR;
  const int sub = lane / LPR, li = lane % LPR;
  float qr[G][8];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) qr[j][e] = q_s[j * HD + li * 8 + e];
  // P V ownership: two dims per thread, positions strided by NG
  const int pg = ctid / S_::NP, dp = ctid % S_::NP;
  float acc[G][2];
#pragma unroll
  for (int j = 0; j < G; ++j) acc[j][0] = acc[j][1] = 0.f;

  auto process = [&](const uint16_t* tk, const uint16_t* tv, int rows) {
    // scores
    for (int base = warp * RPW; base < rows; base += kCWarps * RPW) {
      const int row = base + sub;
      float d[G];
#pragma unroll
      for (int j = 0; j < G; ++j) d[j] = 0.f;
      if (row < rows) {
        const uint4 kv = *reinterpret_cast<const uint4*>(tk + row * HD + li * 8);
#pragma unroll
        for (int j = 0; j < G; ++j) d[j] = dot8(kv, qr[j]);
      }
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < G; ++j) d[j] += __shfl_xor_sync(0xffffffffu, d[j], o);
      if (li == 0 && row < rows)
#pragma unroll
        for (int j = 0; j < G; ++j) sc[j * TP + row] = d[j];
    }
    named_barrier(1, kCThreads);
    // online softmax, one warp per head
    if (warp < G) {
      const int j = warp;
      float mx = -INFINITY;
      for (int r = lane; r < rows; r += 32) mx = fmaxf(mx, sc[j * TP + r]);
      mx = warp_max(mx);
      const float m_old = s_m[j];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int r = lane; r < rows; r += 32) {
        const float e = __expf(sc[j * TP + r] - m_new);
        sc[j * TP + r] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        const float corr = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
        s_corr[j] = corr;
        s_l[j] = s_l[j] * corr + sum;
        s_m[j] = m_new;
      }
    }
    named_barrier(1, kCThreads);
    // P V
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float c = s_corr[j];
      acc[j][0] *= c;
      acc[j][1] *= c;
    }
    const uint32_t* tv32 = reinterpret_cast<const uint32_t*>(tv);
    for (int r = pg; r < rows; r += S_::NG) {
      const uint32_t v2 = tv32[r * S_::NP + dp];
      const float vx = bf16_lo(v2), vy = bf16_hi(v2);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float pj = sc[j * TP + r];
        acc[j][0] = fmaf(pj, vx, acc[j][0]);
        acc[j][1] = fmaf(pj, vy, acc[j][1]);
      }
    }
    named_barrier(1, kCThreads);
  };

  bool abort = false;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kStages, k = t / kStages;
    if (!mbar_wait(&full[s], k & 1)) {
      if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
      abort = true;
      break;
    }
    const int r0 = p0 + t * TP;
    const int rows = (pc1 - r0) < TP ? (pc1 - r0) : TP;
    const uint8_t* st = stages + s * T_::kStageBytes;
    process(reinterpret_cast<const uint16_t*>(st), reinterpret_cast<const uint16_t*>(st + T_::kBytesKV), rows);
    if (ctid == 0) mbar_arrive(&empty[s]);
  }
  if (abort) return;
  if (has_new) process(kn_s, vn_s, 1);

  // ------------------------------------------------------------ partials
#pragma unroll
  for (int j = 0; j < G; ++j) {
    ored[(pg * G + j) * HD + 2 * dp] = acc[j][0];
    ored[(pg * G + j) * HD + 2 * dp + 1] = acc[j][1];
  }
  named_barrier(1, kCThreads);
  float* part = p.part + ((long long)g * p.nsplit + sp) * G * (HD + 2);
  for (int e = ctid; e < G * HD; e += kCThreads) {
    const int j = e / HD, d = e % HD;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < S_::NG; ++q) v += ored[(q * G + j) * HD + d];
    part[j * (HD + 2) + d] = v;
  }
  if (ctid < G) {
    part[ctid * (HD + 2) + HD] = s_m[ctid];
    part[ctid * (HD + 2) + HD + 1] = s_l[ctid];
  }
  named_barrier(1, kCThreads);
  if (ctid == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(p.counter + g, 1u);
    s_last = (ticket == (unsigned)(p.nsplit - 1));
  }
  named_barrier(1, kCThreads);
  if (!s_last) return;
  __threadfence();
  // ------------------------------------------------------------ combine (last CTA of kv head g)
  // Split weights first (one load per (split, head), all in flight together),
  // then each thread merges its (head, dim) outputs with batches of
  // independent loads, so the merge costs a few L2 round trips.
  const float* pg0 = p.part + (long long)g * p.nsplit * G * (HD + 2);
  float* s_w = reinterpret_cast<float*>(stages);              // [nsplit][G] weights e^{m_s - M}
  float* s_den = s_w + p.nsplit * G;                           // [G]
  for (int e = ctid; e < p.nsplit * G; e += kCThreads) {
    const float* ps = pg0 + (long long)e * (HD + 2);
    s_w[e] = __ldcg(ps + HD);                                  // m_s, replaced by its weight below
    ored[e] = __ldcg(ps + HD + 1);                             // l_s
  }
  named_barrier(1, kCThreads);
  if (ctid < G) {
    const int j = ctid;
    float M = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, s_w[s * G + j]);
    float den = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
      const float l = ored[s * G + j];
      const float w = (l > 0.f) ? __expf(s_w[s * G + j] - M) : 0.f;
      s_w[s * G + j] = w;
      den = fmaf(w, l, den);
    }
    s_den[j] = den;
  }
  named_barrier(1, kCThreads);
  for (int e = ctid; e < G * HD; e += kCThreads) {
    const int j = e / HD, d = e % HD;
    float num = 0.f;
    for (int s0 = 0; s0 < p.nsplit; s0 += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = (s0 + u < p.nsplit) ? __ldcg(pg0 + ((long long)(s0 + u) * G + j) * (HD + 2) + d) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (s0 + u < p.nsplit) num = fmaf(s_w[(s0 + u) * G + j], v[u], num);
    }
    p.o[(long long)(g * G + j) * HD + d] = num / s_den[j];
  }
  if (ctid == 0) p.counter[g] = 0u;
}

template <int HD, int G>
void* kern() {
  return (void*)k_attn<HD, G>;
}

void* pick(int hd, int G, size_t* smem) {
#define HY_ATTN_CASE(H_, G_)            \
  if (hd == H_ && G == G_) {            \
    *smem = Smem<H_, G_>::total;        \
    return kern<H_, G_>();              \
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
    for (int gg : gs) {
      size_t smem = 0;
      void* k = pick(h, gg, &smem);
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t launch(const Params& p, cudaStream_t st, bool pdl) {
  if (p.nkv <= 0 || p.nq % p.nkv != 0 || p.nsplit < 1) return cudaErrorInvalidValue;
  size_t smem = 0;
  void* k = pick(p.hd, p.nq / p.nkv, &smem);
  if (!k) return cudaErrorInvalidValue;
  return launch_k(reinterpret_cast<void (*)(Params)>(k), dim3(p.nkv, p.nsplit), dim3(kThreads), smem, st, pdl, p);
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

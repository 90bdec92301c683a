// Device building blocks of split-KV GQA decode attention (kernel in attn.cu).
//
// One work item (g, s) = kv head g, split s: positions [s L / S, (s+1) L / S)
// of the L = T + 1 keys.  Its cached K/V rows arrive as shared-memory tiles
// (copied by the TMA engine); the new row T (rotated, rounded to bf16 and
// appended to the cache by the item that holds it) is attended from shared
// memory.  The item leaves (m, l, o) partials for its G query heads, merged
// with log-sum-exp weights by the last few items of kv head g to finish, each
// a slice of the outputs
// ("Beating llama.cpp from Scratch on Consumer AMD", Act 4 and "What Broke"
// section 1: partial sums over segments of the KV cache, combined across
// separate workgroups).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace attn {

constexpr int kCWarps = 8;
constexpr int kCT = kCWarps * 32;

// A tile is TP cached rows of K or of V (one ring stage); a chunk is CH
// tiles (CP positions) whose scores are all formed before one softmax pass.
template <int HD>
struct Tile {
  static constexpr int TP = HD >= 256 ? 32 : (HD >= 128 ? 64 : 128);  // positions per tile
  static constexpr int kBytes = TP * HD * 2;                            // one K or V tile
  static constexpr int CP = 512;                                        // positions per chunk
  static constexpr int CH = CP / TP;                                    // tiles per chunk
};

// Shared memory a work item uses besides its tiles (floats unless noted).
template <int HD, int G>
struct Work {
  static constexpr int NP = HD / 2;          // dim pairs
  static constexpr int NG = kCT / NP;        // position groups in P V
  static constexpr int TP = Tile<HD>::TP;
  static constexpr size_t q = (size_t)G * HD * 4;
  static constexpr size_t sc = (size_t)G * Tile<HD>::CP * 4;  // chunk scores / probabilities [row][G]
  static constexpr size_t ored = (size_t)NG * G * HD * 4;
  static constexpr size_t kvnew = 2 * HD * 2;
  static constexpr size_t small = 3 * G * 4 + 16 + 64;  // m, l, corr, last; int8 cache: the new row's scales, amax
  static constexpr size_t total = q + sc + ored + kvnew + small;
};

template <int HD, int G>
struct WorkPtrs {
  float* q_s;
  float* sc;
  float* ored;
  uint16_t* kn;
  uint16_t* vn;
  float* m;
  float* l;
  float* corr;
  int* last;
  float* kvs;  // int8 cache: the new row's k and v scales [2], then amax scratch [8]
  __device__ __forceinline__ void carve(uint8_t* base) {
    using W = Work<HD, G>;
    q_s = reinterpret_cast<float*>(base);
    sc = reinterpret_cast<float*>(base + W::q);
    ored = reinterpret_cast<float*>(base + W::q + W::sc);
    kn = reinterpret_cast<uint16_t*>(base + W::q + W::sc + W::ored);
    vn = kn + HD;
    m = reinterpret_cast<float*>(base + W::q + W::sc + W::ored + W::kvnew);
    l = m + G;
    corr = l + G;
    last = reinterpret_cast<int*>(corr + G);
    kvs = reinterpret_cast<float*>(last + 4);
  }
};

struct Item {
  int p0, p1, pc1, ntiles;
  bool has_new;
};

// Element offset of cached row r of kv head g: contiguous [nkv][cap][HD], or
// through the sequence's page table.
template <int HD>
__device__ __forceinline__ long long kv_row(const Params& p, int g, int r) {
  if (p.pages)
    return (long long)p.pages[r / p.page_tokens] * p.page_elems + ((long long)g * p.page_tokens + r % p.page_tokens) * HD;
  return ((long long)g * p.cap + r) * HD;
}

// Batch spread: grid row y of nkv x spread.  Token b of the batch owns n_b
// consecutive rows, n_b = 1 + floor((spread - nb) L_b / sum L) plus one for
// the tokens with the largest remainders (ties to the lower index) until the
// rows are used up, L_b = cached rows + 1 (clamped to [1, cap_b]), so that every
// CTA streams about the same number of cached rows whatever the mix of
// lengths.  Every CTA works out the same shares from the same lengths.
// Returns the token of row y, its split within the token (*sp) and the
// token's split count (*ns).
__device__ __forceinline__ int spread_row(const Params& p, int y, int* sp, int* ns) {
  const int nb = p.nb;
  long long Lb[8], tot = 0;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    long long L = 0;
    if (b < nb) {
      L = (long long)*p.len_b[b] + 1;
      L = L < 1 ? 1 : (L > p.cap_b[b] ? p.cap_b[b] : L);
      if (L < 1) L = 1;
    }
    Lb[b] = L;
    tot += L;
  }
  const long long rest = p.spread - nb;
  int n[8];
  long long rem[8];
  int left = (int)rest;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const long long q = rest * Lb[b];
    n[b] = b < nb ? 1 + (int)(q / tot) : 0;
    rem[b] = b < nb ? q % tot : -1;
    left -= b < nb ? n[b] - 1 : 0;
  }
  int first = 0, z = nb - 1;
  *sp = 0;
  *ns = 1;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    if (b < nb) {
      int rank = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) rank += (rem[c] > rem[b] || (rem[c] == rem[b] && c < b)) ? 1 : 0;
      const int nbb = n[b] + (rank < left ? 1 : 0);
      if (y >= first && y < first + nbb) {
        z = b;
        *sp = y - first;
        *ns = nbb;
      }
      first += nbb;
    }
  }
  return z;
}

template <int HD>
__device__ __forceinline__ Item item_of(const Params& p, int T, int sp) {
  Item it;
  const long long L = (long long)T + 1;
  it.p0 = (int)((long long)sp * L / p.nsplit);
  it.p1 = (int)((long long)(sp + 1) * L / p.nsplit);
  if (p.pages) {  // paged cache: split boundaries on tile multiples, so that no tile straddles a page
    constexpr int TP = Tile<HD>::TP;
    it.p0 &= ~(TP - 1);
    it.p1 = (sp == p.nsplit - 1) ? (int)L : (it.p1 & ~(TP - 1));
  }
  it.pc1 = it.p1 < T ? it.p1 : T;  // cached rows [p0, pc1)
  const int nc = it.pc1 > it.p0 ? it.pc1 - it.p0 : 0;
  it.ntiles = (nc + Tile<HD>::TP - 1) / Tile<HD>::TP;
  it.has_new = (T >= it.p0 && T < it.p1);
  return it;
}

// Copy lane: the K (kv = 0) or V (kv = 1) rows of tile t of the item into
// dst.  int8 cache: the code rows at 0, then the rows' scales from the
// 16-byte boundary at or before the tile's first row (so that the copy starts
// aligned) at scale_off(); row r's scale is float (r0 & 3) + r there.
template <int HD>
__device__ __forceinline__ int scale_off() {
  return Tile<HD>::TP * HD;
}
template <int HD, bool KV8>
__device__ __forceinline__ void issue_tile(const Params& p, int g, const Item& it, int t, int kv, uint8_t* dst,
                                           uint64_t* bar, uint64_t pol) {
  constexpr int TP = Tile<HD>::TP;
  const int r0 = it.p0 + t * TP;
  const int rows = (it.pc1 - r0) < TP ? (it.pc1 - r0) : TP;
  if (KV8) {
    const uint32_t bytes = (uint32_t)rows * HD;
    const int ra = r0 & ~3, n4 = ((r0 + rows + 3) & ~3) - ra;
    mbar_arrive_expect_tx(bar, bytes + n4 * 4);
    const uint8_t* C8 = reinterpret_cast<const uint8_t*>(kv ? p.V : p.K);
    const float* S = kv ? p.Vs : p.Ks;
    bulk_g2s(dst, C8 + ((long long)g * p.cap + r0) * HD, bytes, bar, pol);
    bulk_g2s(dst + scale_off<HD>(), S + (long long)g * p.cap_s + ra, n4 * 4, bar, pol);
    return;
  }
  const uint32_t bytes = (uint32_t)rows * HD * 2;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(dst, (kv ? p.V : p.K) + kv_row<HD>(p, g, r0), bytes, bar, pol);
}

// Eight int8 codes (one 8-byte word) as floats.
__device__ __forceinline__ void i8x8(uint2 u, float* f) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[i] = (float)(int)(int8_t)(u.x >> (8 * i));
    f[4 + i] = (float)(int)(int8_t)(u.y >> (8 * i));
  }
}

// int8 quantisation of a vector held by the compute threads (the same rule as
// the oracle's: amax in FP32, codes round-half-even of x * (127 / amax),
// scale amax / 127).  Every compute thread calls it; `red` >= 8 floats.
__device__ __forceinline__ float block_amax(float local, float* red, int ctid) {
  local = warp_max(local);
  if ((ctid & 31) == 0) red[ctid >> 5] = local;
  named_barrier(1, kCT);
  float a = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kCWarps; ++w2) a = fmaxf(a, red[w2]);
  named_barrier(1, kCT);
  return a;
}
__device__ __forceinline__ int8_t quant_code(float x, float inv) {
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (int8_t)(int)r;
}

template <int HD>
__device__ __forceinline__ int tile_rows(const Item& it, int t) {
  const int r0 = it.p0 + t * Tile<HD>::TP;
  return (it.pc1 - r0) < Tile<HD>::TP ? (it.pc1 - r0) : Tile<HD>::TP;
}

// Per-thread state of a work item.
template <int HD, int G>
struct Acc {
  float qr[G][8];   // query slice: 8 dims per lane
  float acc[G][2];  // P V: two output dims per thread
};

// Compute threads: rotated, scaled queries; the new row (rotated k and v in
// bf16, also appended to the cache) when the item holds position T.
template <int HD, int G, bool KV8 = false>
__device__ __forceinline__ void begin_item(const Params& p, int g, int T, const Item& it, const WorkPtrs<HD, G>& w,
                                           Acc<HD, G>& A, int ctid) {
  const int lane = ctid & 31;
  const float2* rope = p.rope + (long long)T * (HD / 2);
  static_assert(kCT >= HD, "one new-row element per thread");
  // the new row's k and v inputs are loaded with the queries (one round trip)
  float nk0 = 0.f, nk1 = 0.f, nv = 0.f;
  if (it.has_new) {
    const float* kh = p.y + (long long)(p.nq + g) * HD;
    const float* vh = p.y + (long long)(p.nq + p.nkv + g) * HD;
    if (ctid < HD / 2) {
      nk0 = kh[ctid];
      nk1 = kh[ctid + HD / 2];
    }
    if (ctid < HD) nv = vh[ctid];
  }
  // all query pairs of this thread are loaded before any is stored
  constexpr int NQ = (G * (HD / 2) + kCT - 1) / kCT;
  float qa[NQ], qb[NQ];
  float2 qc[NQ];
#pragma unroll
  for (int u = 0; u < NQ; ++u) {
    const int e = ctid + u * kCT;
    if (e < G * (HD / 2)) {
      const int j = e / (HD / 2), i = e % (HD / 2);
      const float* qh = p.y + (long long)(g * G + j) * HD;
      qc[u] = rope[i];
      qa[u] = qh[i];
      qb[u] = qh[i + HD / 2];
    }
  }
#pragma unroll
  for (int u = 0; u < NQ; ++u) {
    const int e = ctid + u * kCT;
    if (e < G * (HD / 2)) {
      const int j = e / (HD / 2), i = e % (HD / 2);
      w.q_s[j * HD + i] = (qa[u] * qc[u].x - qb[u] * qc[u].y) * p.scale;
      w.q_s[j * HD + i + HD / 2] = (qb[u] * qc[u].x + qa[u] * qc[u].y) * p.scale;
    }
  }
  if (KV8 && it.has_new) {
    // int8 cache: the new k and v vectors quantised with their own scales
    int8_t* K8 = reinterpret_cast<int8_t*>(p.K) + ((long long)g * p.cap + T) * HD;
    int8_t* V8 = reinterpret_cast<int8_t*>(p.V) + ((long long)g * p.cap + T) * HD;
    int8_t* kn8 = reinterpret_cast<int8_t*>(w.kn);
    int8_t* vn8 = reinterpret_cast<int8_t*>(w.vn);
    float k0 = 0.f, k1 = 0.f, v0 = 0.f;
    if (ctid < HD / 2) {
      const float2 cs = rope[ctid];
      k0 = nk0 * cs.x - nk1 * cs.y;
      k1 = nk1 * cs.x + nk0 * cs.y;
    }
    if (ctid < HD) v0 = nv;
    const float ka = block_amax(fmaxf(fabsf(k0), fabsf(k1)), w.kvs + 2, ctid);
    const float va = block_amax(fabsf(v0), w.kvs + 2, ctid);
    const float kinv = ka > 0.f ? 127.0f / ka : 0.f, vinv = va > 0.f ? 127.0f / va : 0.f;
    if (ctid < HD / 2) {
      const int8_t c0 = quant_code(k0, kinv), c1 = quant_code(k1, kinv);
      kn8[ctid] = c0;
      kn8[ctid + HD / 2] = c1;
      K8[ctid] = c0;
      K8[ctid + HD / 2] = c1;
    }
    if (ctid < HD) {
      const int8_t c = quant_code(v0, vinv);
      vn8[ctid] = c;
      V8[ctid] = c;
    }
    if (ctid == 0) {
      w.kvs[0] = ka / 127.0f;
      w.kvs[1] = va / 127.0f;
      p.Ks[(long long)g * p.cap_s + T] = ka / 127.0f;
      p.Vs[(long long)g * p.cap_s + T] = va / 127.0f;
    }
  }
  if (!KV8 && it.has_new) {  // kCT >= HD: one k pair and one v element per thread at most
    uint16_t* Kw = p.K + kv_row<HD>(p, g, T);
    uint16_t* Vw = p.V + kv_row<HD>(p, g, T);
    if (ctid < HD / 2) {
      const float2 cs = rope[ctid];
      const uint16_t k0 = f32_to_bf16_rne(nk0 * cs.x - nk1 * cs.y), k1 = f32_to_bf16_rne(nk1 * cs.x + nk0 * cs.y);
      w.kn[ctid] = k0;
      w.kn[ctid + HD / 2] = k1;
      Kw[ctid] = k0;
      Kw[ctid + HD / 2] = k1;
    }
    if (ctid < HD) {
      const uint16_t v = f32_to_bf16_rne(nv);
      w.vn[ctid] = v;
      Vw[ctid] = v;
    }
  }
  if (ctid < G) {
    w.m[ctid] = -INFINITY;
    w.l[ctid] = 0.f;
  }
  named_barrier(1, kCT);
  constexpr int LPR = HD / 8;
  const int li = lane % LPR;
#pragma unroll
  for (int j = 0; j < G; ++j) {
#pragma unroll
    for (int e = 0; e < 8; ++e) A.qr[j][e] = w.q_s[j * HD + li * 8 + e];
    A.acc[j][0] = A.acc[j][1] = 0.f;
  }
}

// Reduce-scatter of C per-head partial sums over the lanes of a row: at
// each halving of the lane distance O a lane keeps half of its heads (the
// upper half if bit O of its lane index is set) and adds its partner's sums
// of them; once one head is left the remaining levels are a plain all-reduce.
// On return v[0] is the full sum of head li / (lanes per row / heads).
template <int C, int O>
__device__ __forceinline__ void head_scatter(float* v, int li) {
  if constexpr (O > 0) {
    if constexpr (C > 1) {
      const bool up = (li & O) != 0;
#pragma unroll
      for (int i = 0; i < C / 2; ++i) {
        const float send = up ? v[i] : v[i + C / 2];
        const float keep = up ? v[i + C / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      head_scatter<C / 2, O / 2>(v, li);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      head_scatter<1, O / 2>(v, li);
    }
  }
}

// Scores of one K tile (rows rows, chunk rows row_base ..): a row is read by
// HD / 8 lanes (8 dims each, one 16-byte shared load), every warp takes its
// rows of all passes at once (independent loads and shuffles in flight), and
// the head sums are reduce-scattered.  Written to w.sc row-major [row][G].
// int8 cache: ks[row] is the row's scale.
template <int HD, int G, bool KV8 = false>
__device__ __forceinline__ void tile_scores(const uint16_t* tk, int rows, int row_base, const WorkPtrs<HD, G>& w,
                                            const Acc<HD, G>& A, int ctid, const float* ks = nullptr) {
  constexpr int TP = Tile<HD>::TP;
  constexpr int LPR = HD / 8, RPW = 32 / LPR, RSTEP = kCWarps * RPW;
  constexpr int NPASS = (TP + RSTEP - 1) / RSTEP;
  constexpr int GL = LPR / G;  // lanes left per head after the scatter
  static_assert(G <= LPR, "heads per group above lanes per row");
  const int warp = ctid >> 5, lane = ctid & 31;
  const int sub = lane / LPR, li = lane % LPR;
  float d[NPASS][G];
#pragma unroll
  for (int ps = 0; ps < NPASS; ++ps) {
    const int row = ps * RSTEP + warp * RPW + sub;
#pragma unroll
    for (int j = 0; j < G; ++j) d[ps][j] = 0.f;
    if (row < rows) {
      if (KV8) {
        const uint2 k8 = *reinterpret_cast<const uint2*>(reinterpret_cast<const int8_t*>(tk) + row * HD + li * 8);
        float kf[8];
        i8x8(k8, kf);
        const float sk = ks[row];
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(kf[e], A.qr[j][e], a);
          d[ps][j] = a * sk;
        }
      } else {
        const uint4 kv = *reinterpret_cast<const uint4*>(tk + row * HD + li * 8);
#pragma unroll
        for (int j = 0; j < G; ++j) d[ps][j] = dot8(kv, A.qr[j]);
      }
    }
  }
#pragma unroll
  for (int ps = 0; ps < NPASS; ++ps) {
    head_scatter<G, LPR / 2>(d[ps], li);
    const int row = ps * RSTEP + warp * RPW + sub;
    if (li % GL == 0 && row < rows) w.sc[(row_base + row) * G + li / GL] = d[ps][0];
  }
}

// Online softmax over the chunk's rows (one warp per head; every compute
// thread calls it after the chunk's scores are in w.sc): new running max,
// probabilities in place, running sum; then every thread rescales its
// accumulators by e^{m_old - m_new}.
template <int HD, int G>
__device__ __forceinline__ void chunk_softmax(int rows, const WorkPtrs<HD, G>& w, Acc<HD, G>& A, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  if (warp < G) {
    const int j = warp;
    float mx = -INFINITY;
    for (int r = lane; r < rows; r += 32) mx = fmaxf(mx, w.sc[r * G + j]);
    mx = warp_max(mx);
    const float m_old = w.m[j];
    const float m_new = fmaxf(m_old, mx);
    float sum = 0.f;
    for (int r = lane; r < rows; r += 32) {
      const float e = __expf(w.sc[r * G + j] - m_new);
      w.sc[r * G + j] = e;
      sum += e;
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      const float corr = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
      w.corr[j] = corr;
      w.l[j] = w.l[j] * corr + sum;
      w.m[j] = m_new;
    }
  }
  named_barrier(1, kCT);
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const float c = w.corr[j];
    A.acc[j][0] *= c;
    A.acc[j][1] *= c;
  }
}

// P V of one V tile (rows rows, chunk rows row_base ..): each thread owns two
// output dims and a position group; a row's G probabilities are vector loads.
// int8 cache: vs[row] is the row's scale.
template <int HD, int G, bool KV8 = false>
__device__ __forceinline__ void tile_pv(const uint16_t* tv, int rows, int row_base, const WorkPtrs<HD, G>& w,
                                        Acc<HD, G>& A, int ctid, const float* vs = nullptr) {
  using W = Work<HD, G>;
  const int pg = ctid / W::NP, dp = ctid % W::NP;
  const uint32_t* tv32 = reinterpret_cast<const uint32_t*>(tv);
  const uint16_t* tv16 = reinterpret_cast<const uint16_t*>(tv);  // int8 cache: two codes
#pragma unroll 4
  for (int r = pg; r < rows; r += W::NG) {
    float vx, vy;
    if (KV8) {
      const uint16_t c2 = tv16[r * W::NP + dp];
      const float sv = vs[r];
      vx = (float)(int)(int8_t)(c2 & 0xFF) * sv;
      vy = (float)(int)(int8_t)(c2 >> 8) * sv;
    } else {
      const uint32_t v2 = tv32[r * W::NP + dp];
      vx = bf16_lo(v2);
      vy = bf16_hi(v2);
    }
    const float* pr = w.sc + (row_base + r) * G;
    float pj[G];
    if constexpr (G % 4 == 0) {
#pragma unroll
      for (int j = 0; j < G; j += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(pr + j);
        pj[j] = q4.x;
        pj[j + 1] = q4.y;
        pj[j + 2] = q4.z;
        pj[j + 3] = q4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < G; ++j) pj[j] = pr[j];
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      A.acc[j][0] = fmaf(pj[j], vx, A.acc[j][0]);
      A.acc[j][1] = fmaf(pj[j], vy, A.acc[j][1]);
    }
  }
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* a) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// Merge of the partials of kv head g by the last p.mergers items to finish.
// The head's counter holds arrivals in its low 16 bits and a generation
// above them.  Every item arrives once its partials are written; items that
// arrive before the last p.mergers exit at once (their SMs go to the next
// kernel).  Each of the last p.mergers waits for the generation to step: the
// very last one clears the count and steps it, which releases the others.
// Merger r then merges slice r of the G * HD outputs,
//   M = max_s m_s,  o = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s,
// up to 32 splits at a time (lane u holds m, l of split u and its weight).  At most p.mergers - 1 items of a head wait at a time and the
// launch keeps that below the SM count over all heads and tokens, so the
// items they wait for always find an SM.
template <int HD, int G>
__device__ __forceinline__ void merge(const Params& p, int g, const WorkPtrs<HD, G>& w, int ctid) {
  unsigned* ctr = p.counter + g;
  const int K = p.mergers;
  if (ctid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(ctr, 1u);
    const int ticket = (int)(old & 0xFFFFu);
    int role = ticket - (p.nsplit - K);
    if (role >= 0) {
      if (ticket == p.nsplit - 1) {
        atomicAdd(ctr, 0x10000u - (unsigned)p.nsplit);
      } else {
        uint64_t t0 = 0;
        for (uint32_t i = 0; (ld_acquire_gpu(ctr) >> 16) == (old >> 16); ++i) {
          if ((i & 255u) == 255u) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
              t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
              set_guard(p.guard, kGuardWaitTimeout);
              role = -1;
              break;
            }
          }
        }
      }
    }
    *w.last = role;
  }
  named_barrier(1, kCT);
  const int role = *w.last;
  if (role < 0) return;
  // merger `role` takes its share of the G * HD / 32 groups of 32 outputs
  // (one head each, since 32 divides HD); a group's outputs are one warp's
  // lanes, so that each load of a split's o values is 128 contiguous bytes,
  // and when groups are few several warps share a group's splits
  constexpr int NGR = G * HD / 32;
  const int gpm = (NGR + K - 1) / K;
  const int ga = role * gpm, gb = (ga + gpm < NGR) ? ga + gpm : NGR;
  if (ga >= gb) return;
  const int ng = gb - ga;
  const int wpg = ng >= kCWarps ? 1 : kCWarps / ng;  // warps per group
  const int gstep = kCWarps / wpg;                    // groups per round
  const int spw = (p.nsplit + wpg - 1) / wpg;         // splits per warp
  const int warp = ctid >> 5, lane = ctid & 31;
  const int wg = warp / wpg, wsp = warp % wpg;
  const float* pg0 = p.part + (long long)g * p.nsplit * G * (HD + 2);
  float* s_num = w.ored;  // [kCWarps][32], then M and den per warp
  float* s_M = s_num + kCWarps * 32;
  float* s_den = s_M + kCWarps;
  const int rounds = (ng + gstep - 1) / gstep;
  for (int rd = 0; rd < rounds; ++rd) {
    const int gi = ga + rd * gstep + wg;
    const bool vg = (wg < gstep) && gi < gb;  // warp-uniform
    const int e = (vg ? gi : ga) * 32 + lane;
    const int j = e / HD, d = e % HD;
    float M = -INFINITY, den = 0.f, num = 0.f;
    if (vg) {
      const int sa = wsp * spw, se = (sa + spw < p.nsplit) ? sa + spw : p.nsplit;
      for (int s0 = sa; s0 < se; s0 += 32) {
        const int ns = (se - s0 < 32) ? se - s0 : 32;
        float mi = -INFINITY, lv = 0.f;
        if (lane < ns) {
          const float* ps = pg0 + ((long long)(s0 + lane) * G + j) * (HD + 2);
          mi = __ldcg(ps + HD);
          lv = __ldcg(ps + HD + 1);
        }
        float ov[32];
#pragma unroll
        for (int u = 0; u < 32; ++u)
          ov[u] = (u < ns) ? __ldcg(pg0 + ((long long)(s0 + u) * G + j) * (HD + 2) + d) : 0.f;
        const float bm = warp_max(lv > 0.f ? mi : -INFINITY);
        if (bm > -INFINITY) {
          const float nm = fmaxf(M, bm);
          const float c = (M == -INFINITY) ? 0.f : __expf(M - nm);
          const float wt = (lv > 0.f) ? __expf(mi - nm) : 0.f;  // lane u: weight of split s0 + u
          den = den * c + warp_sum(wt * lv);
          num *= c;
#pragma unroll
          for (int u = 0; u < 32; ++u) num = fmaf(__shfl_sync(0xffffffffu, wt, u), ov[u], num);
          M = nm;
        }
      }
    }
    if (wpg > 1) {
      // the wpg warps of a group combine through shared memory
      s_num[warp * 32 + lane] = num;
      if (lane == 0) {
        s_M[warp] = M;
        s_den[warp] = den;
      }
      named_barrier(1, kCT);
      if (vg && wsp == 0) {
        for (int q = 1; q < wpg; ++q) {
          const float Mq = s_M[warp + q];
          const float nm = fmaxf(M, Mq);
          if (nm == -INFINITY) continue;
          const float c0 = (M == -INFINITY) ? 0.f : __expf(M - nm);
          const float c1 = (Mq == -INFINITY) ? 0.f : __expf(Mq - nm);
          den = den * c0 + s_den[warp + q] * c1;
          num = num * c0 + s_num[(warp + q) * 32 + lane] * c1;
          M = nm;
        }
        p.o[(long long)g * G * HD + e] = num / den;
      }
      named_barrier(1, kCT);
    } else if (vg) {
      p.o[(long long)g * G * HD + e] = num / den;
    }
  }
}

// Partials of the item (o reduced over the position groups, then m and l),
// then the merge.
template <int HD, int G>
__device__ __forceinline__ void end_item(const Params& p, int g, int sp, const WorkPtrs<HD, G>& w, Acc<HD, G>& A,
                                         int ctid) {
  using W = Work<HD, G>;
  const int pg = ctid / W::NP, dp = ctid % W::NP;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    w.ored[(pg * G + j) * HD + 2 * dp] = A.acc[j][0];
    w.ored[(pg * G + j) * HD + 2 * dp + 1] = A.acc[j][1];
  }
  named_barrier(1, kCT);
  float* part = p.part + ((long long)g * p.nsplit + sp) * G * (HD + 2);
  for (int e = ctid; e < G * HD; e += kCT) {
    const int j = e / HD, d = e % HD;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < W::NG; ++q) v += w.ored[(q * G + j) * HD + d];
    part[j * (HD + 2) + d] = v;
  }
  if (ctid < G) {
    part[ctid * (HD + 2) + HD] = w.m[ctid];
    part[ctid * (HD + 2) + HD + 1] = w.l[ctid];
  }
  named_barrier(1, kCT);
  merge<HD, G>(p, g, w, ctid);
}

}  // namespace attn
}  // namespace hy

// Prompt (prefill) kernels of the mixers and the glue around the prompt GEMMs
// on sm_103a: the whole chunk of n prompt tokens (positions t0 .. t0+n-1) of
// one sequence per launch instead of one launch per token ("Beating llama.cpp
// from Scratch on Consumer AMD", Act 1: batched chunk kernels, one launch per
// layer for all prompt tokens).
//
//   k_embed_rows   X[i] = embedding row of token i (FP32)
//   k_gdn_prep     per (token, head): causal conv over the projection rows
//                  (earlier positions from the conv ring), SiLU, L2 norms of
//                  q and k (q scaled by dk^-1/2), the gates alpha and beta --
//                  every token at once, since none depends on the state
//   k_gdn_scan     per (head, 16 state rows): the rows stay in registers
//                  for the whole chunk and take the gated delta rule token
//                  after token (the decode step's arithmetic, in the same
//                  order), writing each output as bf16 hi + lo parts for the
//                  output projection's GEMM; the rows are stored once at the end
//   k_gdn_ring     the conv ring gets the inputs of the chunk's last positions
//   k_attn_prep    per token: RoPE of the queries (scaled by hd^-1/2) and of
//                  the keys, bf16 keys and values appended at their positions
//   k_attn_causal  per (kv head, block of query tokens): causal softmax
//                  attention over the cached rows, all G query heads of the
//                  group sharing each K/V tile; online softmax per query
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace prefill {
namespace {

__device__ __forceinline__ void split_bf16(float v, uint16_t* hi, uint16_t* lo) {
  const uint16_t a = f32_to_bf16_rne(v);
  *hi = a;
  *lo = f32_to_bf16_rne(v - bf16_to_f32(a));
}

__global__ void k_embed_rows(const uint16_t* __restrict__ embed, const int* __restrict__ tok, int n, int H, int vocab,
                             float* __restrict__ X, unsigned* guard) {
  const int i = blockIdx.x;
  if (i >= n) return;
  int t = tok[i];
  if (t < 0 || t >= vocab) {  // never read outside the embedding table
    if (threadIdx.x == 0) set_guard(guard, kGuardBadIndex);
    t = 0;
  }
  const uint16_t* e = embed + (long long)t * H;
  for (int j = threadIdx.x; j < H; j += blockDim.x) X[(long long)i * H + j] = bf16_to_f32(e[j]);
}

// ------------------------------------------------------------------ Gated DeltaNet
constexpr int kPrepThreads = 128;

__global__ void __launch_bounds__(kPrepThreads) k_gdn_prep(GdnArgs a) {
  const int i = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int nh = a.nh, dk = a.dk, dv = a.dv, K = a.conv_k;
  const int CC = 2 * nh * dk + nh * dv;
  const int t = a.t0 + i;
  extern __shared__ float sh[];  // q[dk] k[dk] red[2][4]
  float* sq = sh;
  float* sk = sh + dk;
  float* red = sh + 2 * dk;
  const float* yi = a.Y + (long long)i * a.ldy;
  for (int c = tid; c < 2 * dk + dv; c += kPrepThreads) {
    int ch;
    if (c < dk) ch = h * dk + c;
    else if (c < 2 * dk) ch = nh * dk + h * dk + (c - dk);
    else ch = 2 * nh * dk + h * dv + (c - 2 * dk);
    // the taps on the K-1 earlier inputs, oldest first, then the new input
    float acc = 0.f;
    for (int j = 0; j < K - 1; ++j) {
      const int p = t - (K - 1) + j;
      float u = 0.f;
      if (p >= a.t0) u = a.Y[(long long)(p - a.t0) * a.ldy + ch];
      else if (p >= 0) u = a.ring[(long long)(p % K) * CC + ch];
      acc = fmaf(bf16_to_f32(a.conv_w[(long long)ch * K + j]), u, acc);
    }
    acc = fmaf(bf16_to_f32(a.conv_w[(long long)ch * K + K - 1]), yi[ch], acc);
    const float cv = siluf_(acc);
    if (c < dk) sq[c] = cv;
    else if (c < 2 * dk) sk[c - dk] = cv;
    else a.V[((long long)i * nh + h) * dv + (c - 2 * dk)] = cv;
  }
  __syncthreads();
  float tq = 0.f, tk = 0.f;
  for (int j = tid; j < dk; j += kPrepThreads) {
    tq += sq[j] * sq[j];
    tk += sk[j] * sk[j];
  }
  tq = warp_sum(tq);
  tk = warp_sum(tk);
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) {
    red[warp] = tq;
    red[4 + warp] = tk;
  }
  __syncthreads();
  tq = red[0] + red[1] + red[2] + red[3];
  tk = red[4] + red[5] + red[6] + red[7];
  const float qs = 1.0f / (sqrtf(tq + 1e-6f) * sqrtf((float)dk));
  const float ks = 1.0f / sqrtf(tk + 1e-6f);
  float* Qo = a.Qn + ((long long)i * nh + h) * dk;
  float* Ko = a.Kn + ((long long)i * nh + h) * dk;
  for (int j = tid; j < dk; j += kPrepThreads) {
    Qo[j] = sq[j] * qs;
    Ko[j] = sk[j] * ks;
  }
  if (tid == 0) {
    a.AB[((long long)i * nh + h) * 2] = sigmoidf_(yi[CC + h]);
    a.AB[((long long)i * nh + h) * 2 + 1] = sigmoidf_(yi[CC + nh + h]);
  }
}

constexpr int kScanRows = 16, kScanThreads = 512, kScanRPW = kScanRows / (kScanThreads / 32);
constexpr int kScanTB = 32;  // tokens whose inputs are staged in shared memory at a time

// Floats of one staged token: k [dk], q [dk], the CTA's v rows [16], alpha and
// beta, padding to 16 bytes.
__host__ __device__ constexpr int scan_tok_floats(int dk) { return 2 * dk + kScanRows + 4; }
size_t scan_smem(int dk) { return (size_t)2 * kScanTB * scan_tok_floats(dk) * sizeof(float); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The recurrence over the chunk's tokens for one head and 16 state rows: the
// rows stay in registers for the whole chunk; the inputs of blocks of 32
// tokens (k, q, the v rows, the gates) are staged in shared memory by the
// whole CTA with asynchronous copies, the next block's while the current one
// runs, so that a token's step waits on no global load.
template <int EPL>
__global__ void __launch_bounds__(kScanThreads) k_gdn_scan(GdnArgs a) {
  extern __shared__ __align__(16) float stage[];
  const int h = blockIdx.x, rc = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int dk = EPL * 32;
  constexpr int TF = scan_tok_floats(dk);
  const int nh = a.nh, dv = a.dv;
  float S[kScanRPW][EPL];
  float* ptr[kScanRPW];
  int row[kScanRPW];
  uint16_t* ohi[kScanRPW];  // the row's output at token 0; token i at + i * ldo
  uint16_t* olo[kScanRPW];
#pragma unroll
  for (int r = 0; r < kScanRPW; ++r) {
    row[r] = rc * kScanRows + warp * kScanRPW + r;
    ptr[r] = a.S + ((long long)h * dv + (row[r] < dv ? row[r] : 0)) * dk + lane * EPL;
    ohi[r] = a.O_hi + h * dv + row[r];
    olo[r] = a.O_lo + h * dv + row[r];
#pragma unroll
    for (int e = 0; e < EPL; ++e) S[r][e] = ptr[r][e];
  }
  // block b's inputs into buffer b & 1: per token dk/4 + dk/4 + 4 16-byte pieces and the gates (8 bytes)
  auto issue = [&](int b) {
    float* buf = stage + (b & 1) * kScanTB * TF;
    const int i0 = b * kScanTB, nt = (a.n - i0 < kScanTB) ? a.n - i0 : kScanTB;
    constexpr int per = dk / 2 + kScanRows / 4 + 1;
    for (int c = tid; c < nt * per; c += kScanThreads) {
      const int j = c / per, q = c % per;
      const long long i = i0 + j;
      float* d = buf + j * TF;
      if (q < dk / 4) {
        cp_async16(d + 4 * q, a.Kn + (i * nh + h) * dk + 4 * q);
      } else if (q < dk / 2) {
        const int u = q - dk / 4;
        cp_async16(d + dk + 4 * u, a.Qn + (i * nh + h) * dk + 4 * u);
      } else if (q < dk / 2 + kScanRows / 4) {
        const int u = q - dk / 2;
        if (rc * kScanRows + 4 * u + 3 < dv) cp_async16(d + 2 * dk + 4 * u, a.V + (i * nh + h) * dv + rc * kScanRows + 4 * u);
      } else {
        cp_async8(d + 2 * dk + kScanRows, a.AB + (i * nh + h) * 2);
      }
    }
    cp_async_commit();
  };
  const int nb = (a.n + kScanTB - 1) / kScanTB;
  if (nb > 0) issue(0);
  for (int b = 0; b < nb; ++b) {
    if (b + 1 < nb) {
      issue(b + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* buf = stage + (b & 1) * kScanTB * TF;
    const int i0 = b * kScanTB, nt = (a.n - i0 < kScanTB) ? a.n - i0 : kScanTB;
    for (int j = 0; j < nt; ++j) {
      const float* tk = buf + j * TF;
      float kq[EPL], qq[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        kq[e] = tk[lane * EPL + e];
        qq[e] = tk[dk + lane * EPL + e];
      }
      const float al = tk[2 * dk + kScanRows], be = tk[2 * dk + kScanRows + 1];
      // the decode step's arithmetic: u_i = S_i . k and S_i . q reduce together,
      // o_i = alpha (S_i . q) + d_i (k . q), then the row update
      float kqd = 0.f, u[kScanRPW], sq[kScanRPW];
#pragma unroll
      for (int e = 0; e < EPL; ++e) kqd = fmaf(kq[e], qq[e], kqd);
#pragma unroll
      for (int r = 0; r < kScanRPW; ++r) {
        u[r] = 0.f;
        sq[r] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          u[r] = fmaf(S[r][e], kq[e], u[r]);
          sq[r] = fmaf(S[r][e], qq[e], sq[r]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        kqd += __shfl_xor_sync(0xffffffffu, kqd, o);
#pragma unroll
        for (int r = 0; r < kScanRPW; ++r) {
          u[r] += __shfl_xor_sync(0xffffffffu, u[r], o);
          sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], o);
        }
      }
#pragma unroll
      for (int r = 0; r < kScanRPW; ++r) {
        const float vr = row[r] < dv ? tk[2 * dk + warp * kScanRPW + r] : 0.f;
        const float d = be * (vr - al * u[r]);
        const float o = fmaf(al, sq[r], d * kqd);
#pragma unroll
        for (int e = 0; e < EPL; ++e) S[r][e] = fmaf(al, S[r][e], d * kq[e]);
        if (lane == 0 && row[r] < dv) {
          split_bf16(o, ohi[r], olo[r]);
          ohi[r] += a.ldo;
          olo[r] += a.ldo;
        }
      }
    }
    __syncthreads();  // buffer b & 1 is refilled with block b + 2 next
  }
#pragma unroll
  for (int r = 0; r < kScanRPW; ++r)
    if (row[r] < dv)
#pragma unroll
      for (int e = 0; e < EPL; ++e) ptr[r][e] = S[r][e];
}

// Ring slot p % K gets the input of position p for the chunk's last K positions.
__global__ void k_gdn_ring(GdnArgs a) {
  const int CC = 2 * a.nh * a.dk + a.nh * a.dv, K = a.conv_k;
  const int p0 = a.n > K ? a.t0 + a.n - K : a.t0;
  const long long total = (long long)(a.t0 + a.n - p0) * CC;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int p = p0 + (int)(e / CC), ch = (int)(e % CC);
    a.ring[(long long)(p % K) * CC + ch] = a.Y[(long long)(p - a.t0) * a.ldy + ch];
  }
}

// ------------------------------------------------------------------ attention
// Element offset of cached row r of kv head g (contiguous, or through the page table).
__device__ __forceinline__ long long kv_off(const AttnArgs& a, int g, int r) {
  if (a.pages)
    return (long long)a.pages[r / a.page_tokens] * a.page_elems + ((long long)g * a.page_tokens + r % a.page_tokens) * a.hd;
  return ((long long)g * a.cap + r) * a.hd;
}

__global__ void k_attn_prep(AttnArgs a) {
  const int i = blockIdx.x;
  const int t = a.t0 + i;
  const int hd = a.hd, half = hd / 2;
  const float2* rope = a.rope + (long long)t * half;
  const float* yi = a.Y + (long long)i * a.ldy;
  for (int e = threadIdx.x; e < a.nq * half; e += blockDim.x) {
    const int j = e / half, d = e % half;
    const float2 cs = rope[d];
    const float x0 = yi[j * hd + d], x1 = yi[j * hd + d + half];
    float* q = a.Qr + ((long long)i * a.nq + j) * hd;
    q[d] = (x0 * cs.x - x1 * cs.y) * a.scale;
    q[d + half] = (x1 * cs.x + x0 * cs.y) * a.scale;
  }
  for (int e = threadIdx.x; e < a.nkv * half; e += blockDim.x) {
    const int g = e / half, d = e % half;
    const float2 cs = rope[d];
    const float x0 = yi[(a.nq + g) * hd + d], x1 = yi[(a.nq + g) * hd + d + half];
    uint16_t* kr = a.K + kv_off(a, g, t);
    kr[d] = f32_to_bf16_rne(x0 * cs.x - x1 * cs.y);
    kr[d + half] = f32_to_bf16_rne(x1 * cs.x + x0 * cs.y);
  }
  for (int e = threadIdx.x; e < a.nkv * hd; e += blockDim.x) {
    const int g = e / hd, d = e % hd;
    a.V[kv_off(a, g, t) + d] = f32_to_bf16_rne(yi[(a.nq + a.nkv + g) * hd + d]);
  }
}

// Causal attention of a block of query tokens over the cached rows [0, t]
// of their kv head.  64 query vectors per CTA (64 / G tokens x G heads);
// 256 threads; a thread owns 4 query vectors (qgroup = tid / 16) and, for the
// scores, 4 keys of the tile (kgroup = tid % 16, keys kgroup + 16 m), for
// P V, hd / 16 output dims (dims kgroup * hd / 16 ...).
constexpr int kQV = 64, kTK = 64, kCausalThreads = 256;

template <int HD>
struct CausalSmem {
  static constexpr int kRow = HD * 2 + 16;  // padded bf16 row (bytes): the 16 key rows of a warp spread over the banks
  static constexpr size_t q = (size_t)kQV * HD * 4;
  static constexpr size_t kv = (size_t)kTK * kRow;
  static constexpr size_t p = (size_t)kQV * (kTK + 1) * 4;
  static constexpr size_t total = q + 2 * kv + p;
};

template <int HD>
__global__ void __launch_bounds__(kCausalThreads) k_attn_causal(AttnArgs a) {
  using SM = CausalSmem<HD>;
  constexpr int DPT = HD / 16;  // output dims per thread
  extern __shared__ __align__(16) uint8_t smem[];
  float* Qs = reinterpret_cast<float*>(smem);
  uint8_t* Ks = smem + SM::q;
  uint8_t* Vs = Ks + SM::kv;
  float* Ps = reinterpret_cast<float*>(Vs + SM::kv);
  const int G = a.nq / a.nkv;
  const int QT = kQV / G;  // query tokens of the CTA
  const int g = blockIdx.x, i0 = blockIdx.y * QT;
  const int tid = threadIdx.x, qg = tid >> 4, kg = tid & 15;
  const int nvalid = min(QT, a.n - i0);
  // query vector v = token (v / G) x head g*G + v % G
  for (int e = tid; e < kQV * HD; e += kCausalThreads) {
    const int v = e / HD, d = e % HD;
    const int tok = v / G, j = v % G;
    Qs[e] = (tok < nvalid) ? a.Qr[((long long)(i0 + tok) * a.nq + g * G + j) * HD + d] : 0.f;
  }
  float m[4], l[4], acc[4][DPT];
  int qpos[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
    const int v = qg * 4 + r;
    qpos[r] = (v / G < nvalid) ? a.t0 + i0 + v / G : -1;  // -1: padding query, every key masked
#pragma unroll
    for (int d = 0; d < DPT; ++d) acc[r][d] = 0.f;
  }
  const int last = a.t0 + i0 + nvalid - 1;  // last key position any query of the CTA sees
  const int ntiles = last / kTK + 1;

  for (int tt = 0; tt < ntiles; ++tt) {
    const int p0 = tt * kTK;
    __syncthreads();  // the previous tile's K, V and P are no longer read
    for (int e = tid; e < kTK * (HD / 8); e += kCausalThreads) {
      const int r = e / (HD / 8), c = e % (HD / 8);
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (p0 + r <= last) {
        const long long off = kv_off(a, g, p0 + r);
        kv = *reinterpret_cast<const uint4*>(a.K + off + c * 8);
        vv = *reinterpret_cast<const uint4*>(a.V + off + c * 8);
      }
      *reinterpret_cast<uint4*>(Ks + r * SM::kRow + c * 16) = kv;
      *reinterpret_cast<uint4*>(Vs + r * SM::kRow + c * 16) = vv;
    }
    __syncthreads();
    // scores of 4 query vectors x 4 keys
    float s[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
    for (int d = 0; d < HD; d += 4) {
      float4 q4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) q4[r] = *reinterpret_cast<const float4*>(Qs + (qg * 4 + r) * HD + d);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint2 kb = *reinterpret_cast<const uint2*>(Ks + (kg + 16 * c) * SM::kRow + d * 2);
        const float k0 = bf16_lo(kb.x), k1 = bf16_hi(kb.x), k2 = bf16_lo(kb.y), k3 = bf16_hi(kb.y);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          s[r][c] = fmaf(q4[r].x, k0, s[r][c]);
          s[r][c] = fmaf(q4[r].y, k1, s[r][c]);
          s[r][c] = fmaf(q4[r].z, k2, s[r][c]);
          s[r][c] = fmaf(q4[r].w, k3, s[r][c]);
        }
      }
    }
    // online softmax per query vector over this tile (the 16 threads of a
    // qgroup hold its 64 scores)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kp = p0 + kg + 16 * c;
        if (kp > qpos[r]) s[r][c] = -INFINITY;
        mx = fmaxf(mx, s[r][c]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m[r], mx);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float e = (mn == -INFINITY) ? 0.f : __expf(s[r][c] - mn);
        Ps[(qg * 4 + r) * (kTK + 1) + kg + 16 * c] = e;
        sum += e;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const float corr = (m[r] == -INFINITY) ? 0.f : __expf(m[r] - mn);
      l[r] = l[r] * corr + sum;
      m[r] = mn;
#pragma unroll
      for (int d = 0; d < DPT; ++d) acc[r][d] *= corr;
    }
    __syncthreads();
    // P V: this thread's 4 query vectors x DPT dims
    const int nk = min(kTK, last - p0 + 1);
    for (int k = 0; k < nk; ++k) {
      float pv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) pv[r] = Ps[(qg * 4 + r) * (kTK + 1) + k];
      const uint16_t* vrow = reinterpret_cast<const uint16_t*>(Vs + k * SM::kRow) + kg * DPT;
#pragma unroll
      for (int d = 0; d < DPT; d += 4) {  // 4 bf16 (8 bytes) at a time: DPT is a multiple of 4
        const uint2 vb = *reinterpret_cast<const uint2*>(vrow + d);
        const float vf[4] = {bf16_lo(vb.x), bf16_hi(vb.x), bf16_lo(vb.y), bf16_hi(vb.y)};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[r][d + e] = fmaf(pv[r], vf[e], acc[r][d + e]);
      }
    }
  }
  // outputs as bf16 hi + lo parts: O[token][head * HD + dim]
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int v = qg * 4 + r;
    const int tok = v / G, j = v % G;
    if (tok >= nvalid) continue;
    const float inv = 1.0f / l[r];
    const long long off = (long long)(i0 + tok) * a.ldo + (g * G + j) * HD + kg * DPT;
#pragma unroll
    for (int d = 0; d < DPT; ++d) split_bf16(acc[r][d] * inv, a.O_hi + off + d, a.O_lo + off + d);
  }
}

__global__ void k_set_len(int* len, int value) { *len = value; }

template <int HD>
cudaError_t launch_causal(const AttnArgs& a, cudaStream_t st) {
  const int G = a.nq / a.nkv;
  const int QT = kQV / G;
  const dim3 grid(a.nkv, (a.n + QT - 1) / QT);
  return launch_k(k_attn_causal<HD>, grid, dim3(kCausalThreads), CausalSmem<HD>::total, st, false, a);
}

}  // namespace

cudaError_t init() {
  cudaError_t e = cudaFuncSetAttribute(k_attn_causal<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)CausalSmem<64>::total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_causal<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)CausalSmem<128>::total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_attn_causal<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)CausalSmem<256>::total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_gdn_scan<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_gdn_scan<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem(128));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_gdn_scan<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem(256));
  return e;
}

cudaError_t embed_rows(const uint16_t* embed, const int* tok, int n, int H, int vocab, float* X, unsigned* guard,
                       cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_embed_rows<<<n, 256, 0, st>>>(embed, tok, n, H, vocab, X, guard);
  return cudaGetLastError();
}

cudaError_t gdn(const GdnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  if (a.dk % 32 || a.conv_k < 1 || a.conv_k > 8) return cudaErrorInvalidValue;
  k_gdn_prep<<<dim3(a.n, a.nh), kPrepThreads, (2 * a.dk + 8) * sizeof(float), st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid(a.nh, (a.dv + kScanRows - 1) / kScanRows);
  if (a.dv % 4) return cudaErrorInvalidValue;
  const size_t sm = scan_smem(a.dk);
  switch (a.dk / 32) {
    case 2: k_gdn_scan<2><<<grid, kScanThreads, sm, st>>>(a); break;
    case 4: k_gdn_scan<4><<<grid, kScanThreads, sm, st>>>(a); break;
    case 8: k_gdn_scan<8><<<grid, kScanThreads, sm, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_gdn_ring<<<256, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t attention(const AttnArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  const int G = a.nkv > 0 ? a.nq / a.nkv : 0;
  if (a.nkv <= 0 || a.nq % a.nkv || (G != 1 && G != 2 && G != 4 && G != 8)) return cudaErrorInvalidValue;
  k_attn_prep<<<a.n, 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (a.hd) {
    case 64: return launch_causal<64>(a, st);
    case 128: return launch_causal<128>(a, st);
    case 256: return launch_causal<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t set_len(int* len, int value, cudaStream_t st) {
  k_set_len<<<1, 1, 0, st>>>(len, value);
  return cudaGetLastError();
}

}  // namespace prefill
}  // namespace hy

// Gated DeltaNet decode step, in place, on sm_103a.
//
// Per head h: causal depthwise conv (width conv_k) + SiLU over the q|k|v
// projection channels, L2-normalised q and k (q also scaled by dk^-1/2),
// alpha = sigmoid(a_h), beta = sigmoid(b_h), then the gated delta rule on the
// FP32 state S in R^{dv x dk} ("Beating llama.cpp from Scratch on Consumer
// AMD", "The Beast": fixed-size FP32 state updated in place by a 1D
// convolution and a gated delta update rule):
//     S <- alpha S (I - beta k k^T) + beta v k^T,   o = S q.
// The kernel uses the equivalent rank-1 form per value row i:
//     u_i = S_i . k,   S_i <- alpha S_i + beta (v_i - alpha u_i) k,   o_i = S_i . q.
// Row i is read and written in place by one warp: the read row is the write
// row, so no gather or copy of the state is needed ("Fourteen hours to 100
// tokens per second", "Eight levers that worked": zero-copy state).
//
// Grid: (heads, dv / 16); a CTA owns 16 value rows of one head (4 warps x 4
// rows).  The state rows are loaded before griddepcontrol.wait: no earlier
// kernel of the same step writes them, so their HBM latency overlaps the
// projection GEMV's tail.  The conv state is a ring of conv_k slots indexed
// by position: step t reads the slots of t-conv_k+1 .. t-1 and writes slot
// t mod conv_k, which no CTA of step t reads, so CTAs sharing a head's q/k
// channels never race.
#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace gdn {
namespace {

constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kRowsPerCta / kWarps;
constexpr int kMaxK = 8;

template <int EPL>  // state elements per lane: dk / 32
__global__ void __launch_bounds__(kThreads) k_gdn(const Params p) {
  __shared__ float s_q[EPL * 32], s_k[EPL * 32], s_v[kRowsPerCta];
  __shared__ float s_red[2][kWarps];
  const int h = blockIdx.x, rc = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dk = EPL * 32, nh = p.nh, dv = p.dv, K = p.conv_k;
  const int CC = 2 * nh * dk + nh * dv;

  // ---- state rows (pre-wait)
  float Sr[kRowsPerWarp][EPL];
  float* rowp[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = rc * kRowsPerCta + warp * kRowsPerWarp + r;
    rowp[r] = p.S + ((long long)h * dv + (i < dv ? i : 0)) * dk + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 4) {
      if (EPL >= 4) {
        const float4 v = *reinterpret_cast<const float4*>(rowp[r] + e);
        Sr[r][e] = v.x; Sr[r][e + 1] = v.y; Sr[r][e + 2] = v.z; Sr[r][e + 3] = v.w;
      }
    }
    if (EPL < 4) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) Sr[r][e] = rowp[r][e];
    }
  }

  pdl_wait();
  pdl_launch_dependents();

  const int t = *p.pos;
  // ---- conv + SiLU over this CTA's channels: q and k of head h (2*dk), v rows of this CTA
  const int nqk = 2 * dk;
  for (int c = threadIdx.x; c < nqk + kRowsPerCta; c += kThreads) {
    int ch;
    if (c < nqk) {
      ch = (c < dk) ? h * dk + c : nh * dk + h * dk + (c - dk);
    } else {
      const int i = rc * kRowsPerCta + (c - nqk);
      if (i >= dv) continue;
      ch = 2 * nh * dk + h * dv + i;
    }
    const float u = p.y[ch];
    float acc = 0.f;
    for (int j = 0; j < K - 1; ++j) {
      const int slot = (t - (K - 1) + j) % K;
      const int sl = slot < 0 ? slot + K : slot;
      acc = fmaf(bf16_to_f32(p.conv_w[(long long)ch * K + j]), p.conv_state[(long long)sl * CC + ch], acc);
    }
    acc = fmaf(bf16_to_f32(p.conv_w[(long long)ch * K + (K - 1)]), u, acc);
    const float cv = siluf_(acc);
    if (c < dk) s_q[c] = cv;
    else if (c < nqk) s_k[c - dk] = cv;
    else s_v[c - nqk] = cv;
    // ring write of the new input: q/k channels by the CTA of row chunk 0 only
    if (c >= nqk || rc == 0) p.conv_state[(long long)(t % K) * CC + ch] = u;
  }
  __syncthreads();

  // ---- L2 norms of q and k
  float sq = 0.f, sk = 0.f;
  for (int j = threadIdx.x; j < dk; j += kThreads) {
    sq += s_q[j] * s_q[j];
    sk += s_k[j] * s_k[j];
  }
  sq = warp_sum(sq);
  sk = warp_sum(sk);
  if (lane == 0) { s_red[0][warp] = sq; s_red[1][warp] = sk; }
  __syncthreads();
  float tq = 0.f, tk = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) { tq += s_red[0][w]; tk += s_red[1][w]; }
  const float qs = 1.0f / (sqrtf(tq + 1e-6f) * sqrtf((float)dk));
  const float ks = 1.0f / sqrtf(tk + 1e-6f);
  float kq[EPL], qq[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    kq[e] = s_k[lane * EPL + e] * ks;
    qq[e] = s_q[lane * EPL + e] * qs;
  }
  const float alpha = sigmoidf_(p.y[CC + h]);
  const float beta = sigmoidf_(p.y[CC + nh + h]);

  // ---- delta rule, one warp per row, in place
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int li = warp * kRowsPerWarp + r;
    const int i = rc * kRowsPerCta + li;
    if (i >= dv) continue;
    float u = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) u = fmaf(Sr[r][e], kq[e], u);
    u = warp_sum(u);
    const float d = beta * (s_v[li] - alpha * u);
    float o = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      Sr[r][e] = fmaf(alpha, Sr[r][e], d * kq[e]);
      o = fmaf(Sr[r][e], qq[e], o);
    }
    if (EPL >= 4) {
#pragma unroll
      for (int e = 0; e < EPL; e += 4)
        *reinterpret_cast<float4*>(rowp[r] + e) = make_float4(Sr[r][e], Sr[r][e + 1], Sr[r][e + 2], Sr[r][e + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) rowp[r][e] = Sr[r][e];
    }
    o = warp_sum(o);
    if (lane == 0) p.o[h * dv + i] = o;
  }
}

}  // namespace

cudaError_t launch(const Params& p, cudaStream_t st, bool pdl) {
  if (p.dk % 32 != 0 || p.conv_k < 1 || p.conv_k > kMaxK) return cudaErrorInvalidValue;
  const dim3 grid(p.nh, (p.dv + kRowsPerCta - 1) / kRowsPerCta);
  switch (p.dk / 32) {
    case 2: return launch_k(k_gdn<2>, grid, dim3(kThreads), 0, st, pdl, p);
    case 4: return launch_k(k_gdn<4>, grid, dim3(kThreads), 0, st, pdl, p);
    case 8: return launch_k(k_gdn<8>, grid, dim3(kThreads), 0, st, pdl, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
}  // namespace hy

// Device building block of the Gated DeltaNet decode step (kernel in gdn.cu).
//
// One work item = 16 value rows of one head h (row chunk rc):
//   causal depthwise conv (width conv_k) + SiLU over q_h, k_h and this item's
//   v rows; q, k L2-normalised (q also scaled by dk^-1/2); alpha =
//   sigmoid(a_h), beta = sigmoid(b_h); then per value row i, in place
//       u_i = S_i . k,   S_i <- alpha S_i + beta (v_i - alpha u_i) k,   o_i = S_i . q
// which is S <- alpha S (I - beta k k^T) + beta v k^T, o = S q written per row;
// o_i of the updated row is formed as alpha (S_i . q) + d_i (k . q) with
// d_i = beta (v_i - alpha u_i), so that u_i and S_i . q reduce in one pass
// ("Beating llama.cpp from Scratch on Consumer AMD", "The Beast": a fixed FP32
// state updated in place by a 1D convolution and a gated delta rule).  The
// read row is the write row ("Fourteen hours to 100 tokens per second",
// "Eight levers that worked": zero-copy state).  The conv state is a ring of
// conv_k slots: step t reads the slots of t-conv_k+1 .. t-1 and writes slot
// t mod conv_k, which no item of step t reads, so items sharing a head's q/k
// channels never race.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace gdn {

// Shared scratch of one item.
template <int EPL>
struct ItemShared {
  float q[EPL * 32];
  float k[EPL * 32];
  float v[kRowsPerCta];
  float red[2][16];
};

// NW warps (NW * 32 threads, tid 0..) process the item; `sync` synchronises
// exactly those threads.  S rows are loaded by load_rows (it may run before
// the projection output is ready) and consumed by run_item.
template <int EPL, int NW>
struct Rows {
  static constexpr int RPW = kRowsPerCta / NW;
  float S[RPW][EPL];
  float* ptr[RPW];
};

// The part of this thread's conv outputs that does not depend on the
// projection output: the taps applied to the conv_k - 1 previous inputs from
// the ring, and the tap of the new input.  Computed before
// griddepcontrol.wait (no kernel of the current step writes the ring or the
// position before this one).
constexpr int kMaxConvK = 8;
template <int EPL, int NW>
struct ConvRegs {
  static constexpr int NCH = (2 * EPL * 32 + kRowsPerCta + NW * 32 - 1) / (NW * 32);  // channels per thread
  float part[NCH];  // sum over the previous inputs
  float last[NCH];  // tap of the new input
  int ch[NCH];      // -1: no channel
  int t;
};

template <int EPL, int NW>
__device__ __forceinline__ void load_conv(const Params& p, int h, int rc, ConvRegs<EPL, NW>& V, int tid) {
  constexpr int NCH = ConvRegs<EPL, NW>::NCH;
  constexpr int NT = NW * 32;
  constexpr int dk = EPL * 32;
  const int nh = p.nh, dv = p.dv, K = p.conv_k;
  const int CC = 2 * nh * dk + nh * dv;
  const int t = *p.pos;
  V.t = t;
#pragma unroll
  for (int q = 0; q < NCH; ++q) {
    const int c = tid + q * NT;
    int ch = -1;
    if (c < 2 * dk) {
      ch = (c < dk) ? h * dk + c : nh * dk + h * dk + (c - dk);
    } else if (c < 2 * dk + kRowsPerCta) {
      const int i = rc * kRowsPerCta + (c - 2 * dk);
      if (i < dv) ch = 2 * nh * dk + h * dv + i;
    }
    V.ch[q] = ch;
    float acc = 0.f, last = 0.f;
    if (ch >= 0) {
      for (int j = 0; j < K - 1; ++j) {
        const int slot = (t - (K - 1) + j) % K;
        acc = fmaf(bf16_to_f32(p.conv_w[(long long)ch * K + j]),
                   p.conv_state[(long long)(slot < 0 ? slot + K : slot) * CC + ch], acc);
      }
      last = bf16_to_f32(p.conv_w[(long long)ch * K + K - 1]);
    }
    V.part[q] = acc;
    V.last[q] = last;
  }
}

template <int EPL, int NW>
__device__ __forceinline__ void load_rows(const Params& p, int h, int rc, Rows<EPL, NW>& R, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int dk = EPL * 32;
#pragma unroll
  for (int r = 0; r < Rows<EPL, NW>::RPW; ++r) {
    const int i = rc * kRowsPerCta + warp * Rows<EPL, NW>::RPW + r;
    R.ptr[r] = p.S + ((long long)h * p.dv + (i < p.dv ? i : 0)) * dk + lane * EPL;
    if (EPL >= 4) {
#pragma unroll
      for (int e = 0; e < EPL; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(R.ptr[r] + e);
        R.S[r][e] = v.x;
        R.S[r][e + 1] = v.y;
        R.S[r][e + 2] = v.z;
        R.S[r][e + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) R.S[r][e] = R.ptr[r][e];
    }
  }
}

template <int EPL, int NW, typename Sync>
__device__ __forceinline__ void run_item(const Params& p, int h, int rc, Rows<EPL, NW>& R,
                                         const ConvRegs<EPL, NW>& V, ItemShared<EPL>& sh, int tid, Sync sync) {
  constexpr int kChanPerThread = ConvRegs<EPL, NW>::NCH;
  constexpr int NT = NW * 32;
  constexpr int RPW = Rows<EPL, NW>::RPW;
  constexpr int dk = EPL * 32;
  const int warp = tid >> 5, lane = tid & 31;
  const int nh = p.nh, dv = p.dv, K = p.conv_k;
  const int CC = 2 * nh * dk + nh * dv;
  const int t = V.t;
  // conv + SiLU over this item's channels (q and k of head h, its v rows):
  // only the new input comes from the projection output
  const int nqk = 2 * dk;
  // the gate inputs go out with the conv inputs: one round trip for all
  const float a_in = p.y[CC + h], b_in = p.y[CC + nh + h];
  float u[kChanPerThread];
#pragma unroll
  for (int q = 0; q < kChanPerThread; ++q) u[q] = V.ch[q] >= 0 ? p.y[V.ch[q]] : 0.f;
#pragma unroll
  for (int q = 0; q < kChanPerThread; ++q) {
    const int ch = V.ch[q];
    if (ch < 0) continue;
    const int c = tid + q * NT;
    const float acc = fmaf(V.last[q], u[q], V.part[q]);
    const float cv = siluf_(acc);
    if (c < dk) sh.q[c] = cv;
    else if (c < nqk) sh.k[c - dk] = cv;
    else sh.v[c - nqk] = cv;
    // ring write of the new input: q/k channels by row chunk 0 only
    if (c >= nqk || rc == 0) p.conv_state[(long long)(t % K) * CC + ch] = u[q];
  }
  sync();
  float sq = 0.f, sk = 0.f;
  for (int j = tid; j < dk; j += NT) {
    sq += sh.q[j] * sh.q[j];
    sk += sh.k[j] * sh.k[j];
  }
  sq = warp_sum(sq);
  sk = warp_sum(sk);
  if (lane == 0) {
    sh.red[0][warp] = sq;
    sh.red[1][warp] = sk;
  }
  sync();
  float tq = 0.f, tk = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    tq += sh.red[0][w];
    tk += sh.red[1][w];
  }
  const float qs = 1.0f / (sqrtf(tq + 1e-6f) * sqrtf((float)dk));
  const float ks = 1.0f / sqrtf(tk + 1e-6f);
  float kq[EPL], qq[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    kq[e] = sh.k[lane * EPL + e] * ks;
    qq[e] = sh.q[lane * EPL + e] * qs;
  }
  const float alpha = sigmoidf_(a_in);
  const float beta = sigmoidf_(b_in);
  // o_i = S_i' . q = alpha (S_i . q) + d_i (k . q): both dots of a row reduce
  // together, before its update
  float kqd = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) kqd = fmaf(kq[e], qq[e], kqd);
  float ur[RPW], qr[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    ur[r] = 0.f;
    qr[r] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      ur[r] = fmaf(R.S[r][e], kq[e], ur[r]);
      qr[r] = fmaf(R.S[r][e], qq[e], qr[r]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kqd += __shfl_xor_sync(0xffffffffu, kqd, o);
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      ur[r] += __shfl_xor_sync(0xffffffffu, ur[r], o);
      qr[r] += __shfl_xor_sync(0xffffffffu, qr[r], o);
    }
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int li = warp * RPW + r;
    const int i = rc * kRowsPerCta + li;
    if (i >= dv) continue;
    const float d = beta * (sh.v[li] - alpha * ur[r]);
    const float o = fmaf(alpha, qr[r], d * kqd);
#pragma unroll
    for (int e = 0; e < EPL; ++e) R.S[r][e] = fmaf(alpha, R.S[r][e], d * kq[e]);
    if (EPL >= 4) {
#pragma unroll
      for (int e = 0; e < EPL; e += 4)
        *reinterpret_cast<float4*>(R.ptr[r] + e) = make_float4(R.S[r][e], R.S[r][e + 1], R.S[r][e + 2], R.S[r][e + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) R.ptr[r][e] = R.S[r][e];
    }
    if (lane == 0) p.o[h * dv + i] = o;
  }
  sync();  // the item's shared scratch may be reused after this
}

}  // namespace gdn
}  // namespace hy

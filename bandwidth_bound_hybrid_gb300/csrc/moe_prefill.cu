// The MoE FFN of a prompt chunk on sm_103a, around tensor-core GEMMs (the
// router, the experts as one grouped GEMM per projection, the shared expert):
//   route    one warp per token: top K of the E routed logits (warp_topk:
//            descending, lowest index on ties), softmax over the picks and
//            the sigmoid of the shared expert's gate, as in the decode step;
//   bucket   one CTA: the picks grouped by expert in token order (counts,
//            offsets, then per expert a ballot scan over the tokens), the
//            gathered row of every pick and the grouped GEMM's row tiles;
//   gather   the normalised activations (bf16 hi / lo parts) of every pick
//            into its gathered row;
//   combine  x[t] += sum_k w[t][k] y_e[row of (t, k)] + w[t][K] y_shared[t].
// ("Fourteen hours to 100 tokens per second", "Eight levers that worked":
// only the selected experts' weights are read, and here each of them once for
// all the chunk's tokens that picked it.)
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace moepf {
namespace {

constexpr int kMaxE = 512;   // routed experts
constexpr int kMaxK = 16;    // picks per token
constexpr int kRouteWarps = 8;

__global__ void __launch_bounds__(kRouteWarps * 32) k_route(const float* logits, int ldl, int n, int E, int K,
                                                             int* ids, float* w) {
  __shared__ int s_sel[kRouteWarps][kMaxK];
  __shared__ float s_selv[kRouteWarps][kMaxK];
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + wi;
  if (t >= n) return;  // the whole warp
  const float* row = logits + (long long)t * ldl;
  auto logit = [&](int e) { return row[e]; };
  if (E <= 128)
    warp_topk<4>(logit, E, K, s_sel[wi], s_selv[wi], lane);
  else if (E <= 256)
    warp_topk<8>(logit, E, K, s_sel[wi], s_selv[wi], lane);
  else
    warp_topk<kMaxE / 32>(logit, E, K, s_sel[wi], s_selv[wi], lane);
  if (lane == 0) {
    const float m = s_selv[wi][0];
    float den = 0.f;
    for (int q = 0; q < K; ++q) den += __expf(s_selv[wi][q] - m);
    for (int q = 0; q < K; ++q) {
      ids[(long long)t * K + q] = s_sel[wi][q];
      w[(long long)t * (K + 1) + q] = __expf(s_selv[wi][q] - m) / den;
    }
    w[(long long)t * (K + 1) + K] = sigmoidf_(row[E]);
  }
}

__device__ __forceinline__ int valid_id(int e, int E, unsigned* guard) {
  if (e < 0 || e >= E) {  // never index past the expert tensors
    set_guard(guard, kGuardBadIndex);
    return 0;
  }
  return e;
}

__global__ void __launch_bounds__(1024) k_bucket(const int* ids, int n, int E, int K, int* pos_of, int* tok_of,
                                                 int* tiles, int* ntiles, unsigned* guard) {
  __shared__ int cnt[kMaxE];
  __shared__ int off[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  for (int i = tid; i < n * K; i += blockDim.x) {  // every row and pick names a valid row even if an id was bad
    tok_of[i] = 0;
    pos_of[i] = 0;
  }
  __syncthreads();
  for (int i = tid; i < n * K; i += blockDim.x) atomicAdd(&cnt[valid_id(ids[i], E, guard)], 1);
  __syncthreads();
  if (warp == 0) {  // exclusive prefix sum of the counts
    int run = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int v = (c0 + lane < E) ? cnt[c0 + lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (c0 + lane < E) off[c0 + lane] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  // expert e's picks take rows off[e] .. in token order
  for (int e = warp; e < E; e += nw) {
    int run = off[e];
    for (int t0 = 0; t0 < n; t0 += 32) {
      const int t = t0 + lane;
      int hit = -1;
      if (t < n)
        for (int k = 0; k < K; ++k)
          if (valid_id(ids[(long long)t * K + k], E, nullptr) == e) hit = k;
      const unsigned b = __ballot_sync(0xffffffffu, hit >= 0);
      if (hit >= 0) {
        const int pos = run + __popc(b & ((1u << lane) - 1u));
        tok_of[pos] = t;
        pos_of[(long long)t * K + hit] = pos;
      }
      run += __popc(b);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int nt = 0;
    for (int e = 0; e < E; ++e)
      for (int r = 0; r < cnt[e]; r += kTileRows) {
        tiles[3 * nt] = off[e] + r;
        tiles[3 * nt + 1] = (cnt[e] - r < kTileRows) ? cnt[e] - r : kTileRows;
        tiles[3 * nt + 2] = e;
        ++nt;
      }
    *ntiles = nt;
  }
}

__global__ void k_gather(const uint16_t* __restrict__ shi, const uint16_t* __restrict__ slo, int ld, int cols,
                         const int* __restrict__ tok_of, int rows, uint16_t* __restrict__ dhi,
                         uint16_t* __restrict__ dlo) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (r >= rows) return;
  const long long t = tok_of[r];
  const uint4* a = reinterpret_cast<const uint4*>(shi + t * ld);
  const uint4* b = reinterpret_cast<const uint4*>(slo + t * ld);
  uint4* c = reinterpret_cast<uint4*>(dhi + (long long)r * cols);
  uint4* d = reinterpret_cast<uint4*>(dlo + (long long)r * cols);
  for (int v = lane; v < cols / 8; v += 32) {
    c[v] = a[v];
    d[v] = b[v];
  }
}

__global__ void k_combine(float* __restrict__ x, int H, int n, int K, const float* __restrict__ w,
                          const int* __restrict__ pos_of, const float* __restrict__ Ye,
                          const float* __restrict__ Ysh) {
  const long long total = (long long)n * H;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / H;
    const int c = (int)(i % H);
    const float* wt = w + t * (K + 1);
    float acc = 0.f;
    for (int k = 0; k < K; ++k) acc = fmaf(wt[k], Ye[(long long)pos_of[t * K + k] * H + c], acc);
    acc = fmaf(wt[K], Ysh[t * H + c], acc);
    x[i] += acc;
  }
}

}  // namespace

int max_tiles(int n, int E, int K) {
  const int picks = n * K;
  return (picks + kTileRows - 1) / kTileRows + (E < picks ? E : picks) + 1;
}

cudaError_t route(const float* logits, int ldl, int n, int E, int K, int* ids, float* w, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (E < 1 || E > kMaxE || K < 1 || K > kMaxK || K > E || ldl < E + 1) return cudaErrorInvalidValue;
  k_route<<<(n + kRouteWarps - 1) / kRouteWarps, kRouteWarps * 32, 0, st>>>(logits, ldl, n, E, K, ids, w);
  return cudaGetLastError();
}

cudaError_t bucket(const int* ids, int n, int E, int K, int* pos_of, int* tok_of, int* tiles, int* ntiles,
                   unsigned* guard, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (E < 1 || E > kMaxE || K < 1 || K > kMaxK) return cudaErrorInvalidValue;
  k_bucket<<<1, 1024, 0, st>>>(ids, n, E, K, pos_of, tok_of, tiles, ntiles, guard);
  return cudaGetLastError();
}

cudaError_t gather(const uint16_t* src_hi, const uint16_t* src_lo, int ld, int cols, const int* tok_of, int rows,
                   uint16_t* dst_hi, uint16_t* dst_lo, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 8 || ld % 8) return cudaErrorInvalidValue;
  k_gather<<<(rows * 32 + 255) / 256, 256, 0, st>>>(src_hi, src_lo, ld, cols, tok_of, rows, dst_hi, dst_lo);
  return cudaGetLastError();
}

cudaError_t combine(float* x, int H, int n, int K, const float* w, const int* pos_of, const float* Ye,
                    const float* Ysh, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long total = (long long)n * H;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 152LL * 16);
  k_combine<<<blocks, 256, 0, st>>>(x, H, n, K, w, pos_of, Ye, Ysh);
  return cudaGetLastError();
}

}  // namespace moepf
}  // namespace hy

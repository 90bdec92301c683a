// The MoE FFN of a prompt chunk on sm_103a, around tensor-core GEMMs (the
// router, the experts as one grouped GEMM per projection, the shared expert):
//   route    one warp per token: top K of the E routed logits (warp_topk:
//            descending, lowest index on ties), softmax over the picks and
//            the sigmoid of the shared expert's gate, as in the decode step;
//   bucket   one CTA: the picks grouped by expert in token order (a stable
//            counting sort: per-warp counts over contiguous token ranges,
//            prefix sums, placement), the gathered row of every pick and the
//            grouped GEMM's row tiles;
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

constexpr int kBucketWarps = 16;

// A stable counting sort of the picks by expert: warp w owns tokens
// [w n / 16, (w + 1) n / 16); (1) each warp counts its picks per expert (lane k
// takes slot k of a token; a token's picks are distinct experts, so the lanes
// never touch the same counter at once); (2) per expert, the prefix over the
// experts before it and over the warps before w gives warp w's first row;
// (3) each warp walks its tokens in order again and hands out rows.
__global__ void __launch_bounds__(kBucketWarps * 32) k_bucket(const int* ids, int n, int E, int K, int* pos_of,
                                                               int* tok_of, int* tiles, int* ntiles,
                                                               unsigned* guard) {
  __shared__ int hist[kBucketWarps][kMaxE];  // counts, then next free row
  __shared__ int tot[kMaxE];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kBucketWarps * kMaxE; i += blockDim.x) (&hist[0][0])[i] = 0;
  for (int i = tid; i < n * K; i += blockDim.x) {  // every row and pick names a valid row even if an id was bad
    tok_of[i] = 0;
    pos_of[i] = 0;
  }
  __syncthreads();
  const int t0 = (int)((long long)warp * n / kBucketWarps), t1 = (int)((long long)(warp + 1) * n / kBucketWarps);
  for (int t = t0; t < t1; ++t) {
    if (lane < K) ++hist[warp][valid_id(ids[(long long)t * K + lane], E, guard)];
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {  // per expert: warp offsets, total
    int run = 0;
    for (int w = 0; w < kBucketWarps; ++w) {
      const int c = hist[w][e];
      hist[w][e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over the experts, added to every warp's offsets
    int run = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      const int v = (e < E) ? tot[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (e < E) {
        const int base = run + incl - v;
        for (int w = 0; w < kBucketWarps; ++w) hist[w][e] += base;
        tot[e] = base;  // expert e's first row
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_total = run;
  }
  __syncthreads();
  for (int t = t0; t < t1; ++t) {
    if (lane < K) {
      const int e = valid_id(ids[(long long)t * K + lane], E, nullptr);
      const int pos = hist[warp][e]++;
      tok_of[pos] = t;
      pos_of[(long long)t * K + lane] = pos;
    }
    __syncwarp();
  }
  __syncthreads();
  if (tid == 0) {
    int nt = 0;
    for (int e = 0; e < E; ++e) {
      const int cnt = (e + 1 < E ? tot[e + 1] : s_total) - tot[e];
      for (int r = 0; r < cnt; r += kTileRows) {
        tiles[3 * nt] = tot[e] + r;
        tiles[3 * nt + 1] = (cnt - r < kTileRows) ? cnt - r : kTileRows;
        tiles[3 * nt + 2] = e;
        ++nt;
      }
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
  k_bucket<<<1, kBucketWarps * 32, 0, st>>>(ids, n, E, K, pos_of, tok_of, tiles, ntiles, guard);
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

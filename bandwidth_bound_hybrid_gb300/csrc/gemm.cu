// Tensor-core GEMM for the prompt (prefill) on sm_103a:
//     Y[m][n] = sum_k A[m][k] W[n][k]      (m: tokens, n: output rows)
// where the FP32 activations reach the tensor cores as two bf16 parts
// A = A_hi + A_lo (relative representation error ~2^-16) and W is the bf16
// weight matrix, so Y = A_hi W^T + A_lo W^T accumulates in FP32.
//
// Prefill is the one place of the step where the work is a dense contraction
// ("Beating llama.cpp from Scratch on Consumer AMD", Act 1: the prompt runs
// through batched kernels, one launch per layer for all its tokens).  Design:
//   * one CTA per 128-token x 256-row output tile (a SwiGLU pair: 128 rows of
//     the gate and of the up matrix), 192 threads: warps 0-3 epilogue (TMEM
//     lanes 0-127 = the tile's tokens), warp 4 copies, warp 5 issues MMAs;
//   * the copy lane stages 64-wide K slices of A_hi, A_lo and W with 2D
//     tensor copies (TMA, 128-byte swizzle) into a 3-stage ring (64 KB each);
//   * one thread issues tcgen05.mma (M = 128, N = 256 or 2 x 128, K = 16) into
//     an FP32 accumulator of 256 TMEM columns and releases each ring stage
//     with tcgen05.commit;
//   * the epilogue reads the accumulator with tcgen05.ld and stores it, adds it
//     to a residual, or applies SwiGLU and splits the result into the bf16
//     hi/lo parts the next GEMM consumes;
//   * grouped form (the MoE experts of a prompt chunk): each row tile comes
//     from a device-side table {first row of the gathered activations, rows,
//     expert}, and the expert selects the block of weight rows it reads.
// Rows past M or N and K past the end arrive as zeros from the tensor copies.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"

namespace hy {
namespace gemm {
namespace {

constexpr int BM = 128, BK = 64, kStages = 3;
constexpr int kThreads = 192;
constexpr int kTileA = BM * BK * 2;               // 16 KB
constexpr int kTileB = 256 * BK * 2;              // 32 KB
constexpr int kStageBytes = 2 * kTileA + kTileB;  // 64 KB
constexpr int kSmem = kStages * kStageBytes + 1024 + 128;
constexpr uint32_t kTmemCols = 256;

struct Maps {
  CUtensorMap a_hi, a_lo, b0, b1;
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// bf16 matrix [rows][cols] (row stride ld elements) as a 2D map with a
// {64, box_rows} box and the 128-byte swizzle.
bool encode(CUtensorMap* m, const void* base, long long rows, int cols, int ld, int box_rows) {
  if (!base || rows <= 0 || cols <= 0 || (reinterpret_cast<uintptr_t>(base) & 15) || (ld * 2) % 16) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t str[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, str, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  hi = f32_to_bf16_rne(v);
  lo = f32_to_bf16_rne(v - bf16_to_f32(hi));
}

__global__ void __launch_bounds__(kThreads, 1) k_gemm(const __grid_constant__ Params p, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool pair = p.epi == kEpiSwigluSplit;
  const int BN = pair ? 128 : 256;
  const int n0 = blockIdx.x * BN;
  int m0 = blockIdx.y * BM, mrows = p.M - m0, wr0 = n0;  // first A row, valid rows, first W row
  if (p.tiles) {  // grouped: the tile table (written by an earlier kernel of the stream)
    const int i = blockIdx.y;
    if (i >= *p.ntiles) return;
    m0 = p.tiles[3 * i];
    mrows = p.tiles[3 * i + 1];
    const int g = p.tiles[3 * i + 2];
    if (g < 0 || g >= p.n_groups || m0 < 0 || mrows < 1 || mrows > BM || m0 + mrows > p.M) {
      if (threadIdx.x == 0) set_guard(p.guard, kGuardBadIndex);
      return;
    }
    wr0 = g * p.w_group_rows + n0;
  }
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      int t = 0;
      for (; t < nk; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !mbar_wait(&empty[s], ((t / kStages) - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tc::tma_load_2d(st, &mp.a_hi, t * BK, m0, &full[s]);
        tc::tma_load_2d(st + kTileA, &mp.a_lo, t * BK, m0, &full[s]);
        if (!pair) {
          tc::tma_load_2d(st + 2 * kTileA, &mp.b0, t * BK, wr0, &full[s]);
        } else {
          tc::tma_load_2d(st + 2 * kTileA, &mp.b0, t * BK, wr0, &full[s]);
          tc::tma_load_2d(st + 2 * kTileA + kTileB / 2, &mp.b1, t * BK, wr0, &full[s]);
        }
      }
      // the CTA must not retire while its copies are in flight
      for (int u = (t > kStages ? t - kStages : 0); u < t; ++u)
        if (!mbar_wait(&full[u % kStages], (u / kStages) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      for (int t = 0; t < nk; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&full[s], (t / kStages) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        tc::fence_after_sync();
        const uint32_t st = smem_addr(smem + s * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ah = tc::sdesc_k128(st + kk * 32);
          const uint64_t al = tc::sdesc_k128(st + kTileA + kk * 32);
          const uint64_t b0 = tc::sdesc_k128(st + 2 * kTileA + kk * 32);
          const bool acc = (t > 0 || kk > 0);
          tc::mma_bf16(tmem, ah, b0, idesc, acc);
          tc::mma_bf16(tmem, al, b0, idesc, true);
          if (pair) {
            const uint64_t b1 = tc::sdesc_k128(st + 2 * kTileA + kTileB / 2 + kk * 32);
            tc::mma_bf16(tmem + 128, ah, b1, idesc, acc);
            tc::mma_bf16(tmem + 128, al, b1, idesc, true);
          }
        }
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(accum);  // also after a timeout: arrives once the issued MMAs have completed
    }
  } else {
    // epilogue: thread (warp w, lane i) owns token row m0 + 32 w + i
    // the TMEM loads are warp-collective: the whole warp takes the same branch
    const bool got = __all_sync(0xffffffffu, mbar_wait(accum, 0));
    if (!got && threadIdx.x == 0) set_guard(p.guard, kGuardWaitTimeout);
    tc::fence_after_sync();
    const int row = m0 + warp * 32 + lane;
    const bool live = warp * 32 + lane < mrows;  // the tile's own rows (grouped: not the next group's)
    const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
    if (got) {
      if (!pair) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tc::tmem_ld32(tbase + c0, v);
          if (!live) continue;
          float* y = p.y + (long long)row * p.ldy + n0 + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (n0 + c0 + j >= p.N) break;
            if (p.epi == kEpiResid) y[j] += v[j];
            else y[j] = v[j];
          }
        }
      } else {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float g[32], u[32];
          tc::tmem_ld32(tbase + c0, g);
          tc::tmem_ld32(tbase + 128 + c0, u);
          if (!live) continue;
          uint16_t* hh = p.h_hi + (long long)row * p.ldh + n0 + c0;
          uint16_t* hl = p.h_lo + (long long)row * p.ldh + n0 + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (n0 + c0 + j >= p.N) break;
            uint16_t a, b;
            split_bf16(siluf_(g[j]) * u[j], a, b);
            hh[j] = a;
            hl[j] = b;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Each row of x (FP32 [rows][ld_x], cols used) -> RMSNorm (gain g, or none)
// -> bf16 hi and lo parts [rows][ld_out].  One warp per row.
__global__ void k_norm_split(const float* __restrict__ x, int ld_x, const float* __restrict__ g, float eps, int rows,
                             int cols, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo, int ld_out) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const float* xr = x + (long long)warp * ld_x;
  float sc = 1.f;
  if (g) {
    float ss = 0.f;
    for (int i = lane; i < cols; i += 32) ss = fmaf(xr[i], xr[i], ss);
    ss = warp_sum(ss);
    sc = 1.0f / sqrtf(ss / (float)cols + eps);
  }
  uint16_t* h = hi + (long long)warp * ld_out;
  uint16_t* l = lo + (long long)warp * ld_out;
  for (int i = lane; i < cols; i += 32) {
    const float v = g ? xr[i] * sc * g[i] : xr[i];
    uint16_t a, b;
    split_bf16(v, a, b);
    h[i] = a;
    l[i] = b;
  }
}

}  // namespace

cudaError_t init() {
  cudaError_t e = cudaFuncSetAttribute(k_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess && !g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) e = cudaErrorNotSupported;
    if (e == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return e;
}

bool supported(int M, int N, int K) { return M > 0 && N > 0 && K > 0 && K % 8 == 0; }

cudaError_t launch(const Params& p, const uint16_t* a_hi, const uint16_t* a_lo, int lda, const uint16_t* w0,
                   const uint16_t* w1, int ldw, cudaStream_t st) {
  if (!g_encode || !supported(p.M, p.N, p.K) || lda < p.K || ldw < p.K) return cudaErrorInvalidValue;
  const bool grouped = p.tiles != nullptr;
  if (grouped && (!p.ntiles || p.max_tiles < 1 || p.n_groups < 1 || p.w_group_rows < p.N)) return cudaErrorInvalidValue;
  const bool pair = p.epi == kEpiSwigluSplit;
  if (pair && (!w1 || !p.h_hi || !p.h_lo)) return cudaErrorInvalidValue;
  if (!pair && !p.y) return cudaErrorInvalidValue;
  alignas(64) Maps mp;
  memset(&mp, 0, sizeof(mp));
  const int bn = pair ? 128 : 256;
  const long long wrows = grouped ? (long long)p.n_groups * p.w_group_rows : p.N;
  if (!encode(&mp.a_hi, a_hi, p.M, p.K, lda, BM) || !encode(&mp.a_lo, a_lo, p.M, p.K, lda, BM) ||
      !encode(&mp.b0, w0, wrows, p.K, ldw, bn) || (pair && !encode(&mp.b1, w1, wrows, p.K, ldw, bn)))
    return cudaErrorInvalidValue;
  const dim3 grid((p.N + bn - 1) / bn, grouped ? p.max_tiles : (p.M + BM - 1) / BM);
  return launch_k(k_gemm, grid, dim3(kThreads), (size_t)kSmem, st, false, p, mp);
}

cudaError_t norm_split(const float* x, int ld_x, const float* g, float eps, int rows, int cols, uint16_t* hi,
                       uint16_t* lo, int ld_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = (rows * 32 + 255) / 256;
  k_norm_split<<<blocks, 256, 0, st>>>(x, ld_x, g, eps, rows, cols, hi, lo, ld_out);
  return cudaGetLastError();
}

}  // namespace gemm
}  // namespace hy

// Tensor-core GEMM for the prompt (prefill) on sm_103a:
//     Y[m][n] = sum_k A[m][k] W[n][k]      (m: tokens, n: output rows)
// where the FP32 activations reach the tensor cores as two bf16 parts
// A = A_hi + A_lo (relative representation error ~2^-16) and W is the bf16
// weight matrix, so Y = A_hi W^T + A_lo W^T accumulates in FP32.
//
// Prefill is the one place of the step where the work is a dense contraction
// ("Beating llama.cpp from Scratch on Consumer AMD", Act 1: the prompt runs
// through batched kernels, one launch per layer for all its tokens).  Design:
//   * 128-token x 256-row output tiles (a SwiGLU pair: 128 rows of the gate
//     and of the up matrix); persistent CTAs (one per SM) take tiles in turn,
//     192 threads: warps 0-3 epilogue (TMEM lanes 0-127 = the tile's tokens),
//     warp 4 copies, warp 5 issues MMAs;
//   * the copy lane stages 64-wide K slices of A_hi, A_lo and W with 2D
//     tensor copies (TMA, 128-byte swizzle) into a 3-stage ring (64 KB each);
//   * one thread issues tcgen05.mma (M = 128, N = 256 or 2 x 128, K = 16) into
//     one of two FP32 accumulators of 256 TMEM columns (alternating by tile,
//     so that the epilogue of a tile overlaps the MMAs of the next) and
//     releases each ring stage with tcgen05.commit;
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
constexpr uint32_t kTmemCols = 512;  // two accumulators of 256 columns

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

// Output tile t of the launch (t = m tile x n tiles + n tile): its first A row,
// valid rows, first W row and first output column; false past the last tile
// (grouped: also at a bad table entry, with the guard set; every role of the
// CTA reads the same entries and stops at the same tile).
struct TileInfo {
  int m0, mrows, wr0, n0;
};
__device__ __forceinline__ bool tile_at(const Params& p, int t, int n_tiles, int BN, int total, TileInfo& ti) {
  if (t >= total) return false;
  const int mt = t / n_tiles;
  ti.n0 = (t % n_tiles) * BN;
  if (!p.tiles) {
    ti.m0 = mt * BM;
    ti.mrows = p.M - ti.m0;
    ti.wr0 = ti.n0;
    return true;
  }
  ti.m0 = p.tiles[3 * mt];
  ti.mrows = p.tiles[3 * mt + 1];
  const int g = p.tiles[3 * mt + 2];
  if (g < 0 || g >= p.n_groups || ti.m0 < 0 || ti.mrows < 1 || ti.mrows > BM || ti.m0 + ti.mrows > p.M) {
    if (threadIdx.x == 0) set_guard(p.guard, kGuardBadIndex);
    return false;
  }
  ti.wr0 = g * p.w_group_rows + ti.n0;
  return true;
}

// Persistent: CTA b takes output tiles b, b + grid, ... .  The ring of stages
// runs on across tiles; the accumulator alternates between two 256-column
// halves of TMEM, so the epilogue of one tile overlaps the MMAs of the next
// (tfull: the MMAs of a tile are done; tempty: the epilogue has read it).
__global__ void __launch_bounds__(kThreads, 1) k_gemm(const __grid_constant__ Params p, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool pair = p.epi == kEpiSwigluSplit;
  const int BN = pair ? 128 : 256;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int total = n_tiles * (p.tiles ? *p.ntiles : (p.M + BM - 1) / BM);
  if ((int)blockIdx.x >= total) return;
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  TileInfo ti;

  if (warp == 4) {
    if (lane == 0) {
      int q = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && tile_at(p, t, n_tiles, BN, total, ti); t += gridDim.x)
        for (int kk = 0; kk < nk; ++kk, ++q) {
          const int s = q % kStages;
          if (q >= kStages && !mbar_wait(&empty[s], ((q / kStages) - 1) & 1)) {
            set_guard(p.guard, kGuardWaitTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tc::tma_load_2d(st, &mp.a_hi, kk * BK, ti.m0, &full[s]);
          tc::tma_load_2d(st + kTileA, &mp.a_lo, kk * BK, ti.m0, &full[s]);
          tc::tma_load_2d(st + 2 * kTileA, &mp.b0, kk * BK, ti.wr0, &full[s]);
          if (pair) tc::tma_load_2d(st + 2 * kTileA + kTileB / 2, &mp.b1, kk * BK, ti.wr0, &full[s]);
        }
      // the CTA must not retire while its copies are in flight
      for (int u = (q > kStages ? q - kStages : 0); u < q; ++u)
        if (!mbar_wait(&full[u % kStages], (u / kStages) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int q = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && tile_at(p, t, n_tiles, BN, total, ti); t += gridDim.x, ++lt) {
        const int b = lt & 1, use = lt >> 1;
        if (use > 0 && !mbar_wait(&tempty[b], (use - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        tc::fence_after_sync();
        const uint32_t acc = tmem + (uint32_t)(b * 256);
        for (int kk = 0; kk < nk; ++kk, ++q) {
          const int s = q % kStages;
          if (!mbar_wait(&full[s], (q / kStages) & 1)) {
            set_guard(p.guard, kGuardWaitTimeout);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st = smem_addr(smem + s * kStageBytes);
#pragma unroll
          for (int k16 = 0; k16 < BK / 16; ++k16) {
            const uint64_t ah = tc::sdesc_k128(st + k16 * 32);
            const uint64_t al = tc::sdesc_k128(st + kTileA + k16 * 32);
            const uint64_t b0 = tc::sdesc_k128(st + 2 * kTileA + k16 * 32);
            const bool accum = (kk > 0 || k16 > 0);
            tc::mma_bf16(acc, ah, b0, idesc, accum);
            tc::mma_bf16(acc, al, b0, idesc, true);
            if (pair) {
              const uint64_t b1 = tc::sdesc_k128(st + 2 * kTileA + kTileB / 2 + k16 * 32);
              tc::mma_bf16(acc + 128, ah, b1, idesc, accum);
              tc::mma_bf16(acc + 128, al, b1, idesc, true);
            }
          }
          tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&tfull[b]);  // also after a timeout: arrives once the issued MMAs have completed
      }
      // every issued MMA has completed before TMEM is released
      tc::mma_commit(done);
      if (!mbar_wait(done, 0)) set_guard(p.guard, kGuardWaitTimeout);
    }
  } else {
    // epilogue: thread (warp w, lane i) owns token row m0 + 32 w + i of each tile; the TMEM loads are
    // warp-collective, so the whole warp takes the same branches
    int lt = 0;
    for (int t = blockIdx.x; tile_at(p, t, n_tiles, BN, total, ti); t += gridDim.x, ++lt) {
      const int b = lt & 1, use = lt >> 1;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&tfull[b], use & 1));
      if (!got) {
        if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
        break;
      }
      tc::fence_after_sync();
      const int row = ti.m0 + warp * 32 + lane;
      const bool live = warp * 32 + lane < ti.mrows;  // the tile's own rows (grouped: not the next group's)
      const uint32_t tbase = tmem + (uint32_t)(b * 256) + ((uint32_t)(warp * 32) << 16);
      if (!pair) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tc::tmem_ld32(tbase + c0, v);
          if (!live) continue;
          float* y = p.y + (long long)row * p.ldy + ti.n0 + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (ti.n0 + c0 + j >= p.N) break;
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
          uint16_t* hh = p.h_hi + (long long)row * p.ldh + ti.n0 + c0;
          uint16_t* hl = p.h_lo + (long long)row * p.ldh + ti.n0 + c0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (ti.n0 + c0 + j >= p.N) break;
            uint16_t a, c;
            split_bf16(siluf_(g[j]) * u[j], a, c);
            hh[j] = a;
            hl[j] = c;
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
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
  // persistent: at most one CTA per SM (its shared memory and all 512 TMEM columns)
  static int nsm_of[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (nsm_of[dev] == 0 && (e = cudaDeviceGetAttribute(&nsm_of[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long tiles = (long long)((p.N + bn - 1) / bn) * (grouped ? p.max_tiles : (p.M + BM - 1) / BM);
  const dim3 grid((unsigned)(tiles < nsm_of[dev] ? tiles : nsm_of[dev]));
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

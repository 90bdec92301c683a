// Batched decode GEMV on sm_103a: Y[b] = W * f(X[b]) for up to 8 token
// vectors b at once, W bf16 or 4-bit blocks, every weight byte read once per
// step for all tokens ("Beating llama.cpp from Scratch on Consumer AMD", Act 5
// and "Fourteen hours to 100 tokens per second": eight rows cost about 2.2
// times one row; "Flash-Next on Strix Halo", "Correctness fixes": the 4-bit
// block of 32 along K with a split-nibble +8 offset).
//
// With 8 token columns the product is a small dense contraction, so it runs
// on the tensor cores with mma.sync m16n8k16 (A = 16 weight rows x 16 k,
// B = 16 k x 8 tokens, FP32 accumulators):
//   * one copy lane streams 16-row tiles HBM -> shared memory with bulk copies
//     (TMA engine), one copy per row into a row stride padded by 16 bytes, so
//     that the fragment loads of 8 rows fall into 8 different bank groups;
//   * eight compute warps split the tile's K range; 4-bit weights are turned
//     into exact FP16 integers (nibble - 8) in registers (a magic-exponent OR
//     and one packed subtract), the block scale is applied to the FP32 result
//     of the block's two MMAs, so the weights are dequantised exactly;
//   * the token vectors are RMS-normalised per token and stored once per CTA
//     in shared memory as FP16 (4-bit weights) or bf16 (bf16 weights, the MMA
//     needs one operand type), in the K order the weight fragments use;
//   * per tile the eight warps' partial sums are reduced in a fixed order, and
//     the CTA's rows are finished at the end: store, residual add, SwiGLU or a
//     per-token argmax.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace bgemv {
namespace {

constexpr int kCT = kWarps * 32;

__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Two nibbles (bits 0..3 and 16..19 of v) -> FP16 pair (n - 8), exactly:
// 0x6400 | n is 1024 + n, minus 1032.
__device__ __forceinline__ uint32_t nib2_to_f16x2(uint32_t v) {
  const uint32_t h = (v & 0x000F000Fu) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Position of element k of a row in the staged token vector: bf16 weights
// keep k; 4-bit weights use, inside each 16-element half block, the order in
// which a lane's 32-bit nibble word feeds the A fragment (evens, then odds).
__device__ __forceinline__ int xperm(int fmt, int k) {
  if (fmt == kFmtBf16) return k;
  const int base = k & ~15, j = k & 15;
  return base + ((j & 1) ? 8 + (j >> 1) : (j >> 1));
}

struct Layout {
  int row_bytes;     // bytes of one weight row in the tile (padded)
  int scale_bytes;   // bytes of one row's scales (unpadded: one copy per tile); 0 for bf16
  int member_bytes;  // one pair member's 16 rows, then their scales
  int x_stride;      // bytes of one staged token vector (padded)
};

__device__ __forceinline__ Layout layout_of(const Params& p) {
  Layout L;
  if (p.fmt == kFmtBf16) {
    L.row_bytes = p.C * 2 + 16;
    L.scale_bytes = 0;
  } else {
    L.row_bytes = p.C / 2 + 16;
    L.scale_bytes = p.C / 16;
  }
  L.member_bytes = kTileRows * (L.row_bytes + L.scale_bytes);
  L.x_stride = p.C * 2 + 16;
  return L;
}

// Copy lane: rows [a, a + rows) of pair member j into the stage.
__device__ __forceinline__ void issue_tile(const Params& p, const Layout& L, int a, int rows, uint8_t* dst,
                                           uint64_t* bar, uint64_t pol) {
  const int npair = p.epi == kEpiSwiglu ? 2 : 1;
  const uint32_t wb = p.fmt == kFmtBf16 ? p.C * 2 : p.C / 2;
  const uint32_t sb = p.fmt == kFmtBf16 ? 0 : p.C / 16;
  mbar_arrive_expect_tx(bar, (uint32_t)rows * (wb + sb) * npair);
  for (int j = 0; j < npair; ++j) {
    uint8_t* m = dst + j * L.member_bytes;
    for (int r = 0; r < rows; ++r) bulk_g2s(m + r * L.row_bytes, p.W[j] + (long long)(a + r) * wb, wb, bar, pol);
    if (sb) bulk_g2s(m + kTileRows * L.row_bytes, p.S[j] + (long long)a * (sb / 2), rows * sb, bar, pol);
  }
}

// Compute threads: the token vectors, normalised per token, into xs (FP16 or
// bf16, permuted for 4-bit weights), zero for padding tokens.  s_red: >= B
// floats of scratch.
__device__ __forceinline__ void stage_inputs(const Params& p, const Layout& L, uint8_t* xs, float* s_red, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int b = 0; b < kMaxB; ++b) {
    uint8_t* row = xs + b * L.x_stride;
    if (b >= p.B) {
      for (int k = ctid; k < p.C / 2; k += kCT) reinterpret_cast<uint32_t*>(row)[k] = 0u;
      continue;
    }
    const float* src = nullptr;
    const uint16_t* emb = nullptr;
    if (p.in == kInEmbed) {
      int tok = p.tok[b];
      if (tok < 0 || tok >= p.vocab) {
        if (ctid == 0) set_guard(p.guard, kGuardBadIndex);
        tok = 0;
      }
      emb = p.embed + (long long)tok * p.C;
    } else {
      src = p.x + (long long)b * p.ldx;
    }
    auto val = [&](int k) { return emb ? bf16_to_f32(emb[k]) : src[k]; };
    float sc = 1.f;
    if (p.norm_g) {
      float ss = 0.f;
      for (int k = ctid; k < p.C; k += kCT) {
        const float v = val(k);
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_red[warp] = ss;
      named_barrier(1, kCT);
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += s_red[w];
      sc = 1.0f / sqrtf(t / (float)p.C + p.eps);
      named_barrier(1, kCT);  // s_red is reused by the next token
    }
    for (int k = ctid; k < p.C; k += kCT) {
      float v = val(k);
      if (p.in == kInEmbed && blockIdx.x == 0) p.x_out[(long long)b * p.ldx_out + k] = v;
      if (p.norm_g) v = v * sc * p.norm_g[k];
      const int pos = xperm(p.fmt, k);
      if (p.fmt == kFmtBf16) reinterpret_cast<uint16_t*>(row)[pos] = f32_to_bf16_rne(v);
      else reinterpret_cast<__half*>(row)[pos] = __float2half_rn(v);
    }
  }
  named_barrier(1, kCT);
}

// One warp's share of one pair member of a tile: 16 rows x 8 tokens, over the
// warp's K chunk [k0, k1) (multiples of 32).  d: the MMA accumulator.
__device__ __forceinline__ void tile_mma(const Params& p, const Layout& L, const uint8_t* m, const uint8_t* xs, int k0,
                                         int k1, float* d, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* xg = xs + g * L.x_stride;  // token g (the MMA's column n = g)
  if (p.fmt == kFmtBf16) {
    const uint8_t* r0 = m + g * L.row_bytes;
    const uint8_t* r8 = m + (g + 8) * L.row_bytes;
    for (int k = k0; k < k1; k += 16) {
      uint32_t a[4], b[2];
      a[0] = *reinterpret_cast<const uint32_t*>(r0 + (k + 2 * t) * 2);
      a[1] = *reinterpret_cast<const uint32_t*>(r8 + (k + 2 * t) * 2);
      a[2] = *reinterpret_cast<const uint32_t*>(r0 + (k + 8 + 2 * t) * 2);
      a[3] = *reinterpret_cast<const uint32_t*>(r8 + (k + 8 + 2 * t) * 2);
      b[0] = *reinterpret_cast<const uint32_t*>(xg + (k + 2 * t) * 2);
      b[1] = *reinterpret_cast<const uint32_t*>(xg + (k + 8 + 2 * t) * 2);
      mma_bf16(d, a, b);
    }
    return;
  }
  const uint8_t* r0 = m + g * L.row_bytes;
  const uint8_t* r8 = m + (g + 8) * L.row_bytes;
  const uint16_t* s0 = reinterpret_cast<const uint16_t*>(m + kTileRows * L.row_bytes + g * L.scale_bytes);
  const uint16_t* s8 = reinterpret_cast<const uint16_t*>(m + kTileRows * L.row_bytes + (g + 8) * L.scale_bytes);
  for (int k = k0; k < k1; k += 32) {
    const int blk = k >> 5;
    const uint32_t u0 = *reinterpret_cast<const uint32_t*>(r0 + blk * 16 + 4 * t);
    const uint32_t u8 = *reinterpret_cast<const uint32_t*>(r8 + blk * 16 + 4 * t);
    uint32_t a[4], b[2];
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    // low nibbles: elements 32 blk + 0..15
    a[0] = nib2_to_f16x2(u0);
    a[1] = nib2_to_f16x2(u8);
    a[2] = nib2_to_f16x2(u0 >> 8);
    a[3] = nib2_to_f16x2(u8 >> 8);
    b[0] = *reinterpret_cast<const uint32_t*>(xg + (k + 2 * t) * 2);
    b[1] = *reinterpret_cast<const uint32_t*>(xg + (k + 8 + 2 * t) * 2);
    mma_f16(e, a, b);
    // high nibbles: elements 32 blk + 16..31
    a[0] = nib2_to_f16x2(u0 >> 4);
    a[1] = nib2_to_f16x2(u8 >> 4);
    a[2] = nib2_to_f16x2(u0 >> 12);
    a[3] = nib2_to_f16x2(u8 >> 12);
    b[0] = *reinterpret_cast<const uint32_t*>(xg + (k + 16 + 2 * t) * 2);
    b[1] = *reinterpret_cast<const uint32_t*>(xg + (k + 24 + 2 * t) * 2);
    mma_f16(e, a, b);
    const float sg = f16_bits_to_f32(s0[blk]), sg8 = f16_bits_to_f32(s8[blk]);
    d[0] = fmaf(sg, e[0], d[0]);
    d[1] = fmaf(sg, e[1], d[1]);
    d[2] = fmaf(sg8, e[2], d[2]);
    d[3] = fmaf(sg8, e[3], d[3]);
  }
}

__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float ov, int oi) {
  if (ov > bv || (ov == bv && oi < bi)) {
    bv = ov;
    bi = oi;
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_bgemv(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout L = layout_of(p);
  const int npair = p.epi == kEpiSwiglu ? 2 : 1;
  const int nst = p.nstages;
  const int stage_bytes = npair * L.member_bytes;
  uint8_t* stages = smem;
  uint8_t* xs = smem + nst * stage_bytes;                               // [8][C] staged tokens
  float* part = reinterpret_cast<float*>(xs + kMaxB * L.x_stride);     // [2][npair][kWarps][16][8]
  float* red = part + 2 * npair * kWarps * kTileRows * kMaxB;           // [npair][rows_cta][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + npair * p.rows_cta_max * kMaxB);
  uint64_t* empty = full + kMaxStages;
  __shared__ float s_red[kWarps];
  __shared__ float s_bv[kWarps][kMaxB];
  __shared__ int s_bi[kWarps][kMaxB];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (p.R + kTileRows - 1) / kTileRows;
  const int t0 = (int)((long long)blockIdx.x * nt / p.ncta), t1 = (int)((long long)(blockIdx.x + 1) * nt / p.ncta);
  const int r0 = t0 * kTileRows, r1 = min(t1 * kTileRows, p.R);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kWarps) {
    pdl_launch_dependents();
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int t = 0;
      for (int a = r0; a < r1; a += kTileRows, ++t) {
        const int rows = min(kTileRows, r1 - a);
        const int s = t % nst, k = t / nst;
        if (t >= nst && !mbar_wait(&empty[s], (k - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        issue_tile(p, L, a, rows, stages + s * stage_bytes, &full[s], pol);
      }
      for (int u = (t > nst ? t - nst : 0); u < t; ++u)
        if (!mbar_wait(&full[u % nst], (u / nst) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  stage_inputs(p, L, xs, s_red, ctid);
  // K chunk of this warp (a multiple of 32 columns)
  const int nblk = p.C / 32;
  const int k0 = (int)((long long)warp * nblk / kWarps) * 32, k1 = (int)((long long)(warp + 1) * nblk / kWarps) * 32;
  const int g = lane >> 2, tq = lane & 3;
  bool ok = true;
  int t = 0;
  for (int a = r0; a < r1; a += kTileRows, ++t) {
    const int s = t % nst, k = t / nst;
    if (ok && !mbar_wait(&full[s], k & 1)) {
      if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
      ok = false;
    }
    float* pt = part + (t & 1) * npair * kWarps * kTileRows * kMaxB;
    for (int j = 0; j < npair; ++j) {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if (ok) tile_mma(p, L, stages + s * stage_bytes + j * L.member_bytes, xs, k0, k1, d, lane);
      float* pw = pt + (j * kWarps + warp) * kTileRows * kMaxB;
      pw[g * kMaxB + 2 * tq] = d[0];
      pw[g * kMaxB + 2 * tq + 1] = d[1];
      pw[(g + 8) * kMaxB + 2 * tq] = d[2];
      pw[(g + 8) * kMaxB + 2 * tq + 1] = d[3];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    named_barrier(1, kCT);
    // fixed-order sum over the warps' K chunks
    for (int e = ctid; e < npair * kTileRows * kMaxB; e += kCT) {
      const int j = e / (kTileRows * kMaxB), rr = e % (kTileRows * kMaxB);
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += pt[(j * kWarps + w) * kTileRows * kMaxB + rr];
      const int row = a - r0 + rr / kMaxB;
      if (row < r1 - r0) red[(j * p.rows_cta_max + row) * kMaxB + rr % kMaxB] = v;
    }
  }
  if (named_barrier_or(1, kCT, !ok)) return;  // one decision for all compute threads

  // ------------------------------------------------------------ epilogue
  const int rows_cta = r1 - r0;
  if (p.epi != kEpiArgmax) {
    for (int e = ctid; e < rows_cta * p.B; e += kCT) {
      const int row = e / p.B, b = e % p.B;
      const float v = red[row * kMaxB + b];
      float* y = p.y + (long long)b * p.ldy + r0 + row;
      if (p.epi == kEpiStore) *y = v;
      else if (p.epi == kEpiResid) *y += v;
      else *y = siluf_(v) * red[(p.rows_cta_max + row) * kMaxB + b];
    }
    return;
  }
  // per-token argmax: this CTA's candidates, then the last CTA merges
  for (int b = 0; b < p.B; ++b) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int row = ctid; row < rows_cta; row += kCT) {
      const float v = red[row * kMaxB + b];
      if (p.y) p.y[(long long)b * p.ldy + r0 + row] = v;
      argmax_merge(bv, bi, v, r0 + row);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) {
      s_bv[warp][b] = bv;
      s_bi[warp][b] = bi;
    }
  }
  named_barrier(1, kCT);
  if (ctid < p.B) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < kWarps; ++w) argmax_merge(bv, bi, s_bv[w][ctid], s_bi[w][ctid]);
    p.part_val[blockIdx.x * kMaxB + ctid] = bv;
    p.part_idx[blockIdx.x * kMaxB + ctid] = bi;
  }
  named_barrier(1, kCT);
  if (ctid == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(p.counter, 1u);
    s_last = (ticket == (unsigned)(p.ncta - 1));
  }
  named_barrier(1, kCT);
  if (!s_last) return;
  __threadfence();
  if (warp < p.B) {
    const int b = warp;
    float v = -INFINITY;
    int vi = 0x7fffffff;
    for (int c = lane; c < p.ncta; c += 32)
      argmax_merge(v, vi, __ldcg(p.part_val + c * kMaxB + b), __ldcg(p.part_idx + c * kMaxB + b));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
      argmax_merge(v, vi, ov, oi);
    }
    if (lane == 0) {
      p.ids_out[b] = vi;
      if (p.len_inc[b]) *p.len_inc[b] += 1;
    }
  }
  named_barrier(1, kCT);
  if (ctid == 0) *p.counter = 0u;
}

}  // namespace

Plan plan(int R, int C, int fmt, int epi, int nsm) {
  Plan pl = {};
  pl.ok = false;
  if (R <= 0 || C <= 0 || C % 32 != 0) return pl;
  if (fmt == kFmtQ4 && C % 256 != 0) return pl;  // scale rows stay 16-byte aligned
  const int npair = epi == kEpiSwiglu ? 2 : 1;
  const int row_bytes = fmt == kFmtBf16 ? C * 2 + 16 : C / 2 + 16;  // as the kernel's Layout
  const int scale_bytes = fmt == kFmtBf16 ? 0 : C / 16;
  const int stage_bytes = npair * kTileRows * (row_bytes + scale_bytes);
  const int ntiles = (R + kTileRows - 1) / kTileRows;
  pl.ncta = ntiles < nsm ? ntiles : nsm;
  const int tiles_cta = (ntiles + pl.ncta - 1) / pl.ncta;
  pl.rows_cta_max = tiles_cta * kTileRows;
  const int fixed = kMaxB * (C * 2 + 16) + 4 * (2 * npair * kWarps * kTileRows * kMaxB) +
                    4 * npair * pl.rows_cta_max * kMaxB + 2 * kMaxStages * 8;
  int ns = kInFlight / stage_bytes;
  ns = ns < 2 ? 2 : (ns > kMaxStages ? kMaxStages : ns);
  while (ns > 2 && fixed + ns * stage_bytes > kMaxSmem) --ns;
  pl.nstages = ns;
  pl.smem = fixed + ns * stage_bytes;
  pl.ok = pl.smem <= kMaxSmem;
  return pl;
}

cudaError_t init() {
  cudaError_t e = cudaFuncSetAttribute(k_bgemv<kFmtBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_bgemv<kFmtQ4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  return e;
}

cudaError_t launch(const Params& p0, const Plan& pl, cudaStream_t st, bool pdl) {
  if (!pl.ok || p0.B < 1 || p0.B > kMaxB) return cudaErrorInvalidValue;
  Params p = p0;
  p.ncta = pl.ncta;
  p.nstages = pl.nstages;
  p.rows_cta_max = pl.rows_cta_max;
  auto k = p.fmt == kFmtBf16 ? k_bgemv<kFmtBf16> : k_bgemv<kFmtQ4>;
  return launch_k(k, dim3(pl.ncta), dim3(kThreads), (size_t)pl.smem, st, pdl, p);
}

}  // namespace bgemv
}  // namespace hy

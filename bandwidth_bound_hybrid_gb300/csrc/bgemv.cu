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
//     in shared memory as FP16 (4-bit weights), or for bf16 weights (the MMA
//     needs one operand type) as two bf16 parts hi + lo, each multiplied by
//     the weights, so the products keep about 16 bits of the FP32 vector; in
//     the K order the weight fragments use;
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
  int x_parts;       // bf16 weights: the vector as hi + lo bf16 parts (two MMAs); FP16: one part
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
  L.x_parts = p.fmt == kFmtBf16 ? 2 : 1;
  return L;
}

// Tile t of the launch: its union entry u (0 for dense), first output row a
// (virtual row for kSrcUnionRows), row count, and the first weight row and
// scale row of each pair member.
struct TileSrc {
  int u, a, rows;
  const uint8_t* w[2];
  const uint16_t* sc[2];
};

__device__ __forceinline__ int checked_union_expert(const Params& p, int u) {
  int e = p.union_ids[u];
  if (e < 0) {  // never read outside the expert tensor (the router's ids are < n_experts)
    set_guard(p.guard, kGuardBadIndex);
    e = 0;
  }
  return e;
}

__device__ __forceinline__ int tiles_of(const Params& p, int U) {
  if (p.src == kSrcUnionRows) return (U + 1) * (p.slot_rows / kTileRows);
  if (p.src == kSrcUnionDown) return (U + 1) * (p.R / kTileRows);
  return (p.R + kTileRows - 1) / kTileRows;
}

__device__ __forceinline__ TileSrc tile_src(const Params& p, int t, int U) {
  TileSrc ts;
  const long long wb = p.fmt == kFmtBf16 ? (long long)p.C * 2 : p.C / 2;  // bytes of a weight row
  const long long sb = p.C / 32;                                           // scales of a row (fp16)
  int wrow;
  if (p.src == kSrcDense) {
    ts.u = 0;
    ts.a = t * kTileRows;
    ts.rows = min(kTileRows, p.R - ts.a);
    wrow = ts.a;
  } else if (p.src == kSrcUnionRows) {
    ts.a = t * kTileRows;
    ts.u = ts.a / p.slot_rows;
    ts.rows = kTileRows;
    wrow = ts.a - ts.u * p.slot_rows;
  } else {
    const int nrb = p.R / kTileRows;
    ts.u = t / nrb;
    ts.a = (t - ts.u * nrb) * kTileRows;
    ts.rows = kTileRows;
    wrow = ts.a;
  }
  for (int j = 0; j < 2; ++j) {
    const uint8_t* w = p.W[j];
    const uint16_t* sc = p.S[j];
    if (p.src != kSrcDense) {
      if (ts.u < U) {
        const long long e = checked_union_expert(p, ts.u);
        w = p.exp_base[j] ? p.exp_base[j] + e * p.exp_stride : nullptr;
        sc = p.exp_scale[j] ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.exp_scale[j]) +
                                                                 e * p.exp_sstride)
                            : nullptr;
      } else {
        w = p.sh_base[j];
        sc = p.sh_scale[j];
      }
    }
    ts.w[j] = w ? w + wrow * wb : nullptr;
    ts.sc[j] = sc ? sc + wrow * sb : nullptr;
  }
  return ts;
}

// Copy lane: the tile's rows of each pair member into the stage.
__device__ __forceinline__ void issue_tile(const Params& p, const Layout& L, const TileSrc& ts, uint8_t* dst,
                                           uint64_t* bar, uint64_t pol) {
  const int npair = p.epi == kEpiSwiglu ? 2 : 1;
  const uint32_t wb = p.fmt == kFmtBf16 ? p.C * 2 : p.C / 2;
  const uint32_t sb = p.fmt == kFmtBf16 ? 0 : p.C / 16;
  mbar_arrive_expect_tx(bar, (uint32_t)ts.rows * (wb + sb) * npair);
  for (int j = 0; j < npair; ++j) {
    uint8_t* m = dst + j * L.member_bytes;
    for (int r = 0; r < ts.rows; ++r) bulk_g2s(m + r * L.row_bytes, ts.w[j] + (long long)r * wb, wb, bar, pol);
    if (sb) bulk_g2s(m + kTileRows * L.row_bytes, ts.sc[j], ts.rows * sb, bar, pol);
  }
}

// Compute threads: the token vectors, normalised per token, into xs (FP16 or
// bf16, permuted for 4-bit weights), zero for padding tokens.  s_red: >= B
// floats of scratch.
__device__ __forceinline__ void stage_inputs(const Params& p, const Layout& L, uint8_t* xs, float* s_red, int ctid,
                                             long long x_off) {
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int b = 0; b < kMaxB; ++b) {
    uint8_t* row = xs + b * L.x_stride;
    if (b >= p.B) {
      for (int k = ctid; k < p.C / 2; k += kCT) {
        reinterpret_cast<uint32_t*>(row)[k] = 0u;
        if (L.x_parts == 2) reinterpret_cast<uint32_t*>(row + kMaxB * L.x_stride)[k] = 0u;
      }
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
      src = p.x + (long long)b * p.ldx + x_off;
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
      if (p.fmt == kFmtBf16) {  // v = hi + lo to ~16 bits: the products stay near FP32 accuracy
        const uint16_t hi = f32_to_bf16_rne(v);
        reinterpret_cast<uint16_t*>(row)[pos] = hi;
        reinterpret_cast<uint16_t*>(row + kMaxB * L.x_stride)[pos] = f32_to_bf16_rne(v - bf16_to_f32(hi));
      } else {
        reinterpret_cast<__half*>(row)[pos] = __float2half_rn(v);
      }
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
  const uint8_t* xl = xg + kMaxB * L.x_stride;  // its lo part (bf16 weights)
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
      b[0] = *reinterpret_cast<const uint32_t*>(xl + (k + 2 * t) * 2);
      b[1] = *reinterpret_cast<const uint32_t*>(xl + (k + 8 + 2 * t) * 2);
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
  float* part = reinterpret_cast<float*>(xs + L.x_parts * kMaxB * L.x_stride);  // [2][npair][kWarps][16][8]
  float* red = part + 2 * npair * kWarps * kTileRows * kMaxB;           // [npair][rows_cta][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + npair * p.rows_cta_max * kMaxB);
  uint64_t* empty = full + kMaxStages;
  __shared__ float s_red[kWarps];
  __shared__ float s_bv[kWarps][kMaxB];
  __shared__ int s_bi[kWarps][kMaxB];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tile range of this CTA; for MoE sources it depends on the union the
  // routing kernel wrote, so it is read after griddepcontrol.wait
  auto tile_range = [&](int& U, int& t0, int& t1) {
    U = 0;
    if (p.src != kSrcDense) {
      U = *p.n_union;
      if (U < 0 || U > kMaxUnion) {
        set_guard(p.guard, kGuardBadIndex);
        U = 0;
      }
    }
    const int nt = tiles_of(p, U);
    t0 = (int)((long long)blockIdx.x * nt / p.ncta);
    t1 = (int)((long long)(blockIdx.x + 1) * nt / p.ncta);
  };

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
      if (p.src != kSrcDense) pdl_wait();  // union and expert ids come from the routing kernel
      int U, t0, t1;
      tile_range(U, t0, t1);
      int n = 0;
      for (int t = t0; t < t1; ++t, ++n) {
        const int s = n % nst, k = n / nst;
        if (n >= nst && !mbar_wait(&empty[s], (k - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        issue_tile(p, L, tile_src(p, t, U), stages + s * stage_bytes, &full[s], pol);
      }
      for (int u = (n > nst ? n - nst : 0); u < n; ++u)
        if (!mbar_wait(&full[u % nst], (u / nst) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  int U, t0, t1;
  tile_range(U, t0, t1);
  const int r0 = (p.src == kSrcDense || p.src == kSrcUnionRows) ? t0 * kTileRows : 0;
  const int r1 = (p.src == kSrcDense) ? min(t1 * kTileRows, p.R) : (p.src == kSrcUnionRows ? t1 * kTileRows : 0);
  int staged_u = -1;
  if (p.src != kSrcUnionDown) {
    stage_inputs(p, L, xs, s_red, ctid, 0);
    staged_u = 0;
  }
  // K chunk of this warp (a multiple of 32 columns)
  const int nblk = p.C / 32;
  const int k0 = (int)((long long)warp * nblk / kWarps) * 32, k1 = (int)((long long)(warp + 1) * nblk / kWarps) * 32;
  const int g = lane >> 2, tq = lane & 3;
  bool ok = true;
  int n = 0;
  for (int t = t0; t < t1; ++t, ++n) {
    const TileSrc ts = tile_src(p, t, U);
    if (p.src == kSrcUnionDown && ts.u != staged_u) {  // the tile's expert input, for every token
      named_barrier(1, kCT);
      stage_inputs(p, L, xs, s_red, ctid, (long long)ts.u * p.C);
      staged_u = ts.u;
    }
    const int s = n % nst, k = n / nst;
    if (ok && !mbar_wait(&full[s], k & 1)) {
      if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
      ok = false;
    }
    float* pt = part + (n & 1) * npair * kWarps * kTileRows * kMaxB;
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
      const int b = rr % kMaxB, ri = rr / kMaxB;
      if (p.src == kSrcUnionDown) {
        // partial output of expert u for the tokens that selected it
        const int slot = (ts.u < U) ? p.slot_of[ts.u * kMaxB + b] : p.top_k;
        if (b < p.B && slot >= 0 && ri < ts.rows)
          p.part_out[((long long)b * (p.top_k + 1) + slot) * p.R + ts.a + ri] = v;
      } else {
        const int row = ts.a - r0 + ri;
        if (row < r1 - r0) red[(j * p.rows_cta_max + row) * kMaxB + b] = v;
      }
    }
  }
  if (named_barrier_or(1, kCT, !ok)) return;  // one decision for all compute threads
  if (p.src == kSrcUnionDown) return;

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

// One CTA: routing of every token, then the union of the selected experts.
__global__ void __launch_bounds__(256) k_route(const Route r) {
  __shared__ float lg[kMaxB][512];  // logits of up to 511 experts + the shared gate per token
  __shared__ int sel[kMaxB][16];
  __shared__ float selv[kMaxB][16];
  __shared__ int flag[512];
  __shared__ int pos[512];
  __shared__ int s_n;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int E = r.E, K = r.top_k;
  for (int b = 0; b < r.B; ++b)
    for (int e = tid; e <= E; e += blockDim.x) lg[b][e] = r.logits[(long long)b * r.ld + e];
  for (int e = tid; e < E; e += blockDim.x) flag[e] = 0;
  __syncthreads();
  // rank of every (token, expert): logits above it, or equal with a lower index
  for (int i = tid; i < r.B * E; i += blockDim.x) {
    const int b = i / E, e = i % E;
    const float v = lg[b][e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const float w = lg[b][f];
      rank += (w > v || (w == v && f < e)) ? 1 : 0;
    }
    if (rank < K) {
      sel[b][rank] = e;
      selv[b][rank] = v;
      flag[e] = 1;
    }
  }
  __syncthreads();
  if (tid < r.B) {  // softmax over the selected logits, sigmoid gate of the shared expert
    const int b = tid;
    const float m = selv[b][0];
    float den = 0.f;
    for (int k = 0; k < K; ++k) den += __expf(selv[b][k] - m);
    for (int k = 0; k < K; ++k) {
      r.w[b * (K + 1) + k] = __expf(selv[b][k] - m) / den;
      if (r.ids) r.ids[b * K + k] = sel[b][k];
    }
    r.w[b * (K + 1) + K] = sigmoidf_(lg[b][E]);
  }
  if (tid == 0) {  // ascending union (serial scan over at most 511 flags)
    int n = 0;
    for (int e = 0; e < E; ++e) {
      pos[e] = n;
      if (flag[e]) r.union_ids[n++] = e;
    }
    *r.n_union = n;
    s_n = n;
  }
  __syncthreads();
  const int U = s_n;
  for (int i = tid; i < (kMaxUnion + 1) * kMaxB; i += blockDim.x) r.slot_of[i] = -1;
  __syncthreads();
  for (int i = tid; i < r.B * K; i += blockDim.x) {
    const int b = i / K, k = i % K;
    r.slot_of[pos[sel[b][k]] * kMaxB + b] = k;
  }
  for (int b = tid; b < kMaxB; b += blockDim.x) r.slot_of[U * kMaxB + b] = K;
}

__global__ void k_moe_reduce(float* y, int ldy, const float* part, const float* w, int R, int B, int K) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R * B; i += gridDim.x * blockDim.x) {
    const int b = i / R, row = i % R;
    float acc = 0.f;
    for (int k = 0; k <= K; ++k) acc = fmaf(w[b * (K + 1) + k], part[((long long)b * (K + 1) + k) * R + row], acc);
    y[(long long)b * ldy + row] += acc;
  }
}

}  // namespace

cudaError_t route(const Route& r, cudaStream_t st, bool pdl) {
  if (r.B < 1 || r.B > kMaxB || r.E < 1 || r.E > 511 || r.top_k < 1 || r.top_k > 16 || r.B * r.top_k > kMaxUnion)
    return cudaErrorInvalidValue;
  return launch_k(k_route, dim3(1), dim3(256), 0, st, pdl, r);
}

cudaError_t moe_reduce(float* y, int ldy, const float* part, const float* w, int R, int B, int top_k, cudaStream_t st,
                       bool pdl) {
  const int n = R * B;
  return launch_k(k_moe_reduce, dim3((n + 255) / 256), dim3(256), 0, st, pdl, y, ldy, part, w, R, B, top_k);
}

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
  const int fixed = (fmt == kFmtBf16 ? 2 : 1) * kMaxB * (C * 2 + 16) + 4 * (2 * npair * kWarps * kTileRows * kMaxB) +
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

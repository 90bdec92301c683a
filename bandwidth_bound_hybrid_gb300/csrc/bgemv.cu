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
//   * the matrix is seen as 3D, {128-byte strip of a row, row, strip index},
//     and one copy lane streams stages of 16*GW rows x KS strips (16 KB, plus
//     2 KB of 4-bit scales) with one tensor copy each (TMA, 128-byte swizzle:
//     the fragment reads of 8 rows fall into 8 different bank groups without
//     padding); rows past the end of the matrix arrive as zeros;
//   * the 8 compute warps are GW row groups x KS strip lanes (GW * KS = 8);
//     warp (gw, ks) accumulates its 16 rows over strips ks, ks + KS, ... of
//     a row block in registers, so warps meet only at the end of a row block
//     (KS > 1: a fixed-order sum of the KS partials), not once per stage;
//   * 4-bit weights are turned into exact FP16 integers (nibble - 8) in
//     registers (a magic-exponent OR, then one packed subtract for the low
//     nibbles or one packed FMA by 1/16 for the high ones, in place) and the
//     block scale is applied to the FP32 result of the block's two MMAs, so
//     the weights are dequantised exactly;
//   * the token vectors are RMS-normalised per token (one warp per token) and
//     stored once per CTA in shared memory as FP16 (4-bit weights), or for
//     bf16 weights (the MMA needs one operand type) as two bf16 parts hi + lo,
//     each multiplied by the weights, so the products keep about 16 bits of
//     the FP32 vector; in the K order the weight fragments use;
//   * each row block is finished as soon as its last strip is in: store,
//     residual add, SwiGLU, per-(expert, token) partial, or a per-token
//     argmax candidate (merged across CTAs by the last one to finish).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace bgemv {

// Tensor maps of one launch, passed by value.
struct Maps {
  CUtensorMap w[2], s[2];    // the dense matrix, or the shared expert of a union source
  CUtensorMap ew[2], es[2];  // the routed experts of a union source, their rows stacked
};

namespace {

constexpr int kCT = kWarps * 32;
constexpr int kStrip = 128;      // bytes of a row in one strip
constexpr int kStageW = 16384;   // weight bytes of a stage member: 16 * GW rows x KS strips x 128 B
constexpr int kStageS = 2048;    // 4-bit scales of a stage member: 16 * GW rows x KS strips x 16 B
constexpr int kPartFloats = kWarps * kTileRows * kMaxB;  // one member's per-warp partials

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

// Tensor copy of box {0, c1, c2} of a 3D map into shared memory, completing
// on an mbarrier.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c1, int c2, uint64_t* bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// The staged token vectors: 8 rows of x_stride bytes, two parts for bf16
// weights.  Rows are padded so that the fragment reads of 8 tokens do not
// share banks: by 16 bytes for bf16 (32-bit reads), by 64 for 4-bit weights
// (128-bit reads, two token rows per quarter warp).
struct XLayout {
  int x_stride, x_parts;
};

// Four consecutive elements k..k+3 of a token vector (FP32 rows, 16-byte
// aligned or not, or a bf16 embedding row).
__device__ __forceinline__ float4 load4(const float* src, const uint16_t* emb, bool vec, int k) {
  if (emb) {
    const uint2 u = *reinterpret_cast<const uint2*>(emb + k);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
  }
  if (vec) return *reinterpret_cast<const float4*>(src + k);
  return make_float4(src[k], src[k + 1], src[k + 2], src[k + 3]);
}

// Elements k..k+3 (k a multiple of 4) into the staged row: bf16 hi + lo parts
// in element order, or FP16 in the order the 4-bit B fragments read them.
__device__ __forceinline__ void store4(int fmt, uint8_t* row, uint8_t* row_lo, int k, float4 v) {
  if (fmt == kFmtBf16) {
    const float f[4] = {v.x, v.y, v.z, v.w};
    uint16_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[i] = f32_to_bf16_rne(f[i]);
      l[i] = f32_to_bf16_rne(f[i] - bf16_to_f32(h[i]));
    }
    *reinterpret_cast<uint2*>(row + 2 * k) = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    *reinterpret_cast<uint2*>(row_lo + 2 * k) =
        make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
    return;
  }
  // 4-bit weights: the 32-element block k >> 5 occupies 64 bytes; lane t's
  // B fragments of the block's two MMAs (elements 4t, 4t+2 | 4t+1, 4t+3 |
  // 4t+16, 4t+18 | 4t+17, 4t+19, the order in which its nibble word feeds
  // the A fragments) are the 16 bytes at 16 t: elements k..k+3 (k a multiple
  // of 4) land as (k, k+2, k+1, k+3) at 16 t + 8 (k >= 16 in the block)
  const int e0 = k & 31;
  const __half2 p0 = __floats2half2_rn(v.x, v.z), p1 = __floats2half2_rn(v.y, v.w);
  *reinterpret_cast<uint2*>(row + (k >> 5) * 64 + 16 * ((e0 & 15) >> 2) + 8 * (e0 >> 4)) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1));
}

// Compute warps: token b = warp into xs, RMS-normalised when norm_g is set
// (FP16 in fragment order for 4-bit weights; bf16 hi + lo for bf16), zero for
// padding tokens.  Each warp loads its whole vector at once (up to 2048
// elements held in registers; longer vectors in two passes), so staging costs
// about one L2 round trip.  Ends with a barrier of the compute warps.
constexpr int kHold = 16;  // float4 per lane held in registers
static_assert(kWarps == kMaxB, "one compute warp per token");
__device__ __forceinline__ void stage_inputs(const Params& p, const XLayout& L, uint8_t* xs, int ctid,
                                             long long x_off) {
  const int b = ctid >> 5, lane = ctid & 31;
  uint8_t* row = xs + b * L.x_stride;
  uint8_t* row_lo = row + kMaxB * L.x_stride;
  const int ng = p.C / 4;  // groups of four elements
  if (b >= p.B) {
    for (int i = lane; i < ng; i += 32) {
      *reinterpret_cast<uint2*>(row + 8 * i) = make_uint2(0u, 0u);
      if (L.x_parts == 2) *reinterpret_cast<uint2*>(row_lo + 8 * i) = make_uint2(0u, 0u);
    }
    named_barrier(1, kCT);
    return;
  }
  const float* src = nullptr;
  const uint16_t* emb = nullptr;
  if (p.in == kInEmbed) {
    int tok = p.tok[b];
    if (tok < 0 || tok >= p.vocab) {
      if (lane == 0) set_guard(p.guard, kGuardBadIndex);
      tok = 0;
    }
    emb = p.embed + (long long)tok * p.C;
  } else {
    src = p.x + (long long)b * p.ldx + x_off;
  }
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  float* xo = (p.in == kInEmbed && blockIdx.x == 0) ? p.x_out + (long long)b * p.ldx_out : nullptr;
  const float* gn = p.norm_g;
  auto finish = [&](int k, float4 v, float sc) {
    if (xo) {
      xo[k] = v.x;
      xo[k + 1] = v.y;
      xo[k + 2] = v.z;
      xo[k + 3] = v.w;
    }
    if (gn) {
      v.x *= sc * gn[k];
      v.y *= sc * gn[k + 1];
      v.z *= sc * gn[k + 2];
      v.w *= sc * gn[k + 3];
    }
    store4(p.fmt, row, row_lo, k, v);
  };
  if (ng <= 32 * kHold) {
    float4 v[kHold];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
      const int i = lane + 32 * j;
      v[j] = i < ng ? load4(src, emb, vec, 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kHold; ++j)
      ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
    const float sc = gn ? 1.0f / sqrtf(warp_sum(ss) / (float)p.C + p.eps) : 1.f;
#pragma unroll
    for (int j = 0; j < kHold; ++j) {
      const int i = lane + 32 * j;
      if (i < ng) finish(4 * i, v[j], sc);
    }
  } else {
    float ss = 0.f;
    if (gn) {
      for (int i = lane; i < ng; i += 32) {
        const float4 v = load4(src, emb, vec, 4 * i);
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      }
    }
    const float sc = gn ? 1.0f / sqrtf(warp_sum(ss) / (float)p.C + p.eps) : 1.f;
    for (int i = lane; i < ng; i += 32) finish(4 * i, load4(src, emb, vec, 4 * i), sc);
  }
  named_barrier(1, kCT);
}


// Where a unit (one row block) comes from: union entry u (0 for dense), first
// output row a (virtual row for kSrcUnionRows), valid rows, the row
// coordinate in the maps and which maps.
struct UnitSrc {
  int u, a, rows, crow;
  bool routed;  // the routed-expert maps (else the dense / shared ones)
};

__device__ __forceinline__ int units_of(const Params& p, int U) {
  const int tr = kTileRows * p.gw;
  if (p.src == kSrcUnionRows) return (U + 1) * (p.slot_rows / tr);
  if (p.src == kSrcUnionDown) return (U + 1) * (p.R / tr);
  return (p.R + tr - 1) / tr;
}

__device__ __forceinline__ UnitSrc unit_src(const Params& p, const int* uids, int t, int U) {
  const int tr = kTileRows * p.gw;
  UnitSrc us;
  us.routed = false;
  if (p.src == kSrcDense) {
    us.u = 0;
    us.a = t * tr;
    us.rows = min(tr, p.R - us.a);
    us.crow = us.a;
    return us;
  }
  int r, per;
  if (p.src == kSrcUnionRows) {
    us.a = t * tr;
    us.u = us.a / p.slot_rows;
    r = us.a - us.u * p.slot_rows;
    per = p.slot_rows;
  } else {
    const int nrb = p.R / tr;
    us.u = t / nrb;
    us.a = (t - us.u * nrb) * tr;
    r = us.a;
    per = p.R;
  }
  us.rows = tr;
  us.crow = r;
  if (us.u < U) {
    int e = uids[us.u];
    if (e < 0 || e >= p.n_exp) {  // never address past the expert tensor
      set_guard(p.guard, kGuardBadIndex);
      e = 0;
    }
    us.crow = e * per + r;
    us.routed = true;
  }
  return us;
}

// One warp's MMAs over one strip of one stage member: its 16 rows (lines
// line0 and line0 + 8 of the member; line0 & 7 == g, the swizzle phase) x 8
// tokens, strip elements kb.. of the row.
template <int FMT>
__device__ __forceinline__ void strip_mma(const uint8_t* mem, const uint8_t* xs, const XLayout& L, int line0, int kb,
                                          float* d, int g, int t) {
  const uint8_t* l0 = mem + line0 * kStrip;
  const uint8_t* l8 = l0 + 8 * kStrip;
  const uint8_t* xg = xs + g * L.x_stride;  // token g (the MMA's column n = g)
  if (FMT == kFmtQ4) {
    // the strip's 8 block scales of rows g and g + 8 (16 bytes each)
    const uint4 sv0 = *reinterpret_cast<const uint4*>(mem + kStageW + line0 * 16);
    const uint4 sv8 = *reinterpret_cast<const uint4*>(mem + kStageW + (line0 + 8) * 16);
    const uint32_t sw0[4] = {sv0.x, sv0.y, sv0.z, sv0.w}, sw8[4] = {sv8.x, sv8.y, sv8.z, sv8.w};
    const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
    const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));    // -72
    // two nibbles in bits 0..3 and 16..19 (lo) or 4..7 and 20..23 (hi) of v
    // -> FP16 pair (n - 8), exactly: 0x6400 | n is 1024 + n, minus 1032;
    // 0x6400 | 16 n is 1024 + 16 n, times 1/16 minus 72
    auto lo2 = [&](uint32_t v) {
      const uint32_t h = (v & 0x000F000Fu) | 0x64006400u;
      const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), k1032);
      return *reinterpret_cast<const uint32_t*>(&r);
    };
    auto hi2 = [&](uint32_t v) {
      const uint32_t h = (v & 0x00F000F0u) | 0x64006400u;
      const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&h), k16th, km72);
      return *reinterpret_cast<const uint32_t*>(&r);
    };
    const uint8_t* xb = xg + (kb >> 5) * 64 + 16 * t;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // 32-element blocks of the strip
      const int off = ((j ^ g) << 4) + 4 * t;
      const uint32_t u0 = *reinterpret_cast<const uint32_t*>(l0 + off);
      const uint32_t u8 = *reinterpret_cast<const uint32_t*>(l8 + off);
      const uint4 bx = *reinterpret_cast<const uint4*>(xb + 64 * j);
      const uint32_t v0 = u0 >> 8, v8 = u8 >> 8;
      uint32_t a[4], b[2];
      float e[4] = {0.f, 0.f, 0.f, 0.f};
      // low nibbles: elements 0..15 of the block
      a[0] = lo2(u0);
      a[1] = lo2(u8);
      a[2] = lo2(v0);
      a[3] = lo2(v8);
      b[0] = bx.x;
      b[1] = bx.y;
      mma_f16(e, a, b);
      // high nibbles: elements 16..31
      a[0] = hi2(u0);
      a[1] = hi2(u8);
      a[2] = hi2(v0);
      a[3] = hi2(v8);
      b[0] = bx.z;
      b[1] = bx.w;
      mma_f16(e, a, b);
      const uint32_t w0 = sw0[j >> 1], w8 = sw8[j >> 1];
      const float sg = f16_bits_to_f32((uint16_t)((j & 1) ? (w0 >> 16) : (w0 & 0xFFFFu)));
      const float sg8 = f16_bits_to_f32((uint16_t)((j & 1) ? (w8 >> 16) : (w8 & 0xFFFFu)));
      d[0] = fmaf(sg, e[0], d[0]);
      d[1] = fmaf(sg, e[1], d[1]);
      d[2] = fmaf(sg8, e[2], d[2]);
      d[3] = fmaf(sg8, e[3], d[3]);
    }
  } else {
    const uint8_t* xl = xg + kMaxB * L.x_stride;  // the token's lo part
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 16-element steps of the 64-element strip
      const int o0 = (((2 * q) ^ g) << 4) + 4 * t, o1 = (((2 * q + 1) ^ g) << 4) + 4 * t;
      uint32_t a[4], b[2];
      a[0] = *reinterpret_cast<const uint32_t*>(l0 + o0);
      a[1] = *reinterpret_cast<const uint32_t*>(l8 + o0);
      a[2] = *reinterpret_cast<const uint32_t*>(l0 + o1);
      a[3] = *reinterpret_cast<const uint32_t*>(l8 + o1);
      const int k = kb + 16 * q;
      b[0] = *reinterpret_cast<const uint32_t*>(xg + (k + 2 * t) * 2);
      b[1] = *reinterpret_cast<const uint32_t*>(xg + (k + 8 + 2 * t) * 2);
      mma_bf16(d, a, b);
      b[0] = *reinterpret_cast<const uint32_t*>(xl + (k + 2 * t) * 2);
      b[1] = *reinterpret_cast<const uint32_t*>(xl + (k + 8 + 2 * t) * 2);
      mma_bf16(d, a, b);
    }
  }
}

__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float ov, int oi) {
  if (ov > bv || (ov == bv && oi < bi)) {
    bv = ov;
    bi = oi;
  }
}

// (value, index) as one integer that orders like the argmax: larger value
// first, then lower index; 0 = no candidate.
__device__ __forceinline__ unsigned long long am_key(float v, int i) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)i);
}
__device__ __forceinline__ void am_unkey(unsigned long long k, float& v, int& i) {
  if (k == 0ull) {
    v = -INFINITY;
    i = 0x7fffffff;
    return;
  }
  const uint32_t h = (uint32_t)(k >> 32);
  v = __uint_as_float((h & 0x80000000u) ? (h & 0x7fffffffu) : ~h);
  i = (int)(0xFFFFFFFFu - (uint32_t)k);
}

// Routing of every token of a batch from its router logits (logits [B][ld],
// row E of a token the shared gate), by the 8 compute warps' threads tid
// (synchronised with named barrier 1): warp b picks token b's top_k with
// warp_topk (largest logit, lowest index on ties: the same set and order as
// ranking all experts); the union of the picks is an ascending ballot scan
// over the experts' flags.
constexpr int kRouteMaxE = 512;  // experts + the shared gate per token
struct RouteShared {
  int sel[kMaxB][16];
  float selv[kMaxB][16];
  int flag[kRouteMaxE];
  int cnt[kRouteMaxE / 32 + 1];
  int pos[kRouteMaxE];
  int uid[kMaxUnion];  // the union, ascending
  int U;
};
// logits [B][ld]; the union also lands in rs.uid / rs.U.  publish: write the
// routing weights, ids, union and slot map to global memory (p.r_w, p.r_ids,
// p.union_ids, p.n_union, p.slot_of).  Ends with a barrier of the compute
// threads.
__device__ __noinline__ void route_tokens(const Params& p, const float* logits, int ld, RouteShared& rs, int tid,
                                          bool publish) {
  auto sync = [] { named_barrier(1, kCT); };
  const int warp = tid >> 5, lane = tid & 31;
  const int E = p.r_E, K = p.top_k;
  int* union_ids = const_cast<int*>(p.union_ids);
  int* slot_of = const_cast<int*>(p.slot_of);
  for (int e = tid; e < kRouteMaxE; e += kCT) rs.flag[e] = 0;
  sync();
  if (warp < p.B) {
    const int b = warp;
    auto logit = [&](int e) { return __ldcg(logits + (long long)b * ld + e); };
    if (E <= 128)
      warp_topk<4>(logit, E, K, rs.sel[b], rs.selv[b], lane);
    else if (E <= 256)
      warp_topk<8>(logit, E, K, rs.sel[b], rs.selv[b], lane);
    else
      warp_topk<kRouteMaxE / 32>(logit, E, K, rs.sel[b], rs.selv[b], lane);
    __syncwarp();
    if (lane < K) rs.flag[rs.sel[b][lane]] = 1;
    if (lane == 0 && publish) {  // softmax over the selected logits, sigmoid gate of the shared expert
      const float m = rs.selv[b][0];
      float den = 0.f;
      for (int k = 0; k < K; ++k) den += __expf(rs.selv[b][k] - m);
      for (int k = 0; k < K; ++k) {
        p.r_w[b * (K + 1) + k] = __expf(rs.selv[b][k] - m) / den;
        if (p.r_ids) p.r_ids[b * K + k] = rs.sel[b][k];
      }
      p.r_w[b * (K + 1) + K] = sigmoidf_(__ldcg(logits + (long long)b * ld + E));
    }
  }
  sync();
  const int nch = (E + 31) / 32;
  for (int c = warp; c < nch; c += kWarps) {
    const unsigned m = __ballot_sync(0xffffffffu, rs.flag[32 * c + lane] != 0);
    if (lane == 0) rs.cnt[c] = __popc(m);
  }
  sync();
  for (int c = warp; c < nch; c += kWarps) {
    int base = 0;
    for (int q = 0; q < c; ++q) base += rs.cnt[q];
    const int e = 32 * c + lane;
    const unsigned m = __ballot_sync(0xffffffffu, rs.flag[e] != 0);
    const int at = base + __popc(m & ((1u << lane) - 1u));
    rs.pos[e] = at;
    if (rs.flag[e]) {
      rs.uid[at] = e;
      if (publish) union_ids[at] = e;
    }
  }
  int U = 0;
  for (int q = 0; q < nch; ++q) U += rs.cnt[q];
  if (tid == 0) rs.U = U;
  if (publish) {
    if (tid == 0) {
      *const_cast<int*>(p.n_union) = U;
      if (p.union_count) atomicAdd(p.union_count, (unsigned long long)U);
    }
    for (int i = tid; i < (kMaxUnion + 1) * kMaxB; i += kCT) slot_of[i] = -1;
    sync();
    for (int i = tid; i < p.B * K; i += kCT) {
      const int b = i / K, k = i % K;
      slot_of[rs.pos[rs.sel[b][k]] * kMaxB + b] = k;
    }
    for (int b = tid; b < kMaxB; b += kCT) slot_of[U * kMaxB + b] = K;
  }
  sync();
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_bgemv(const __grid_constant__ Params p, const __grid_constant__ Maps mp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int npair = p.epi == kEpiSwiglu ? 2 : 1;
  const int nst = p.nstages, GW = p.gw, KS = p.ks, TR = kTileRows * p.gw;
  const int member = kStageW + (FMT == kFmtQ4 ? kStageS : 0);
  const int stage_bytes = npair * member;
  const int strip_elems = FMT == kFmtQ4 ? 256 : 64;
  const int spu = p.C / strip_elems / KS;  // stages per unit
  XLayout L;
  L.x_stride = p.C * 2 + (FMT == kFmtQ4 ? 64 : 16);
  L.x_parts = FMT == kFmtBf16 ? 2 : 1;
  uint8_t* stages = smem;                                                     // 1024-aligned members
  uint8_t* xs = smem + nst * stage_bytes;                                     // [parts][8][x_stride]
  float* part = reinterpret_cast<float*>(xs + L.x_parts * kMaxB * L.x_stride);  // [npair][8 warps][16][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + npair * kPartFloats);
  uint64_t* empty = full + kMaxStages;
  uint64_t* rbar = empty + kMaxStages;  // routing done (route_here)
  __shared__ unsigned long long s_key[kMaxB];
  __shared__ int s_last;
  __shared__ RouteShared s_route;
  const bool route_here = p.src == kSrcUnionRows && p.route_here;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the unit range of this CTA; for MoE sources it depends on the union: the
  // one this CTA routed (route_here), or the one the gate/up kernel published,
  // read after griddepcontrol.wait
  auto unit_range = [&](int& U, int& t0, int& t1) {
    U = 0;
    if (p.src != kSrcDense) {
      U = route_here ? s_route.U : *p.n_union;
      if (U < 0 || U > kMaxUnion) {
        set_guard(p.guard, kGuardBadIndex);
        U = 0;
      }
    }
    const int nt = units_of(p, U);
    t0 = (int)((long long)blockIdx.x * nt / p.ncta);
    t1 = (int)((long long)(blockIdx.x + 1) * nt / p.ncta);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(rbar, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < kMaxB) s_key[threadIdx.x] = 0ull;
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kWarps) {
    pdl_launch_dependents();
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      if (p.src != kSrcDense) pdl_wait();  // router logits, union and expert ids come from earlier kernels
      if (route_here && !mbar_wait(rbar, 0)) set_guard(p.guard, kGuardWaitTimeout);  // ... or from this CTA
      const int* uids = route_here ? s_route.uid : p.union_ids;
      int U, t0, t1;
      unit_range(U, t0, t1);
      const uint32_t tx = (uint32_t)(npair * member);
      int n = 0;
      bool alive = true;
      for (int t = t0; t < t1 && alive; ++t) {
        const UnitSrc us = unit_src(p, uids, t, U);
        for (int st = 0; st < spu; ++st, ++n) {
          const int s = n % nst, k = n / nst;
          if (n >= nst && !mbar_wait(&empty[s], (k - 1) & 1)) {
            set_guard(p.guard, kGuardWaitTimeout);
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], tx);
          for (int j = 0; j < npair; ++j) {
            uint8_t* dst = stages + s * stage_bytes + j * member;
            tma_load_3d(dst, us.routed ? &mp.ew[j] : &mp.w[j], us.crow, st * KS, &full[s], pol);
            if (FMT == kFmtQ4)
              tma_load_3d(dst + kStageW, us.routed ? &mp.es[j] : &mp.s[j], us.crow, st * KS, &full[s], pol);
          }
        }
      }
      // the CTA leaves only once its copies have landed
      for (int u = (n > nst ? n - nst : 0); u < n; ++u)
        if (!mbar_wait(&full[u % nst], (u / nst) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (route_here) {
    // every CTA routes the batch from the stored router logits (the same
    // result everywhere) for its copy lane; CTA 0 publishes the routing for
    // the down projection and the expert sum
    route_tokens(p, p.r_logits, p.r_ld, s_route, ctid, blockIdx.x == 0);
    if (ctid == 0) mbar_arrive(rbar);
  }
  const int* uids = route_here ? s_route.uid : p.union_ids;
  int U, t0, t1;
  unit_range(U, t0, t1);
  int staged_u = -1;
  if (p.src != kSrcUnionDown) {
    stage_inputs(p, L, xs, ctid, 0);
    staged_u = 0;
  }
  const int gw = warp / KS, ks = warp % KS;
  const int g = lane >> 2, tq = lane & 3;
  const int line0 = ks * TR + gw * kTileRows + g;  // TR is a multiple of 8: line0 & 7 == g
  float bv[2] = {-INFINITY, -INFINITY};  // argmax candidates of this thread's tokens
  int bi[2] = {0x7fffffff, 0x7fffffff};
  bool ok = true;
  int n = 0;
  for (int t = t0; t < t1; ++t) {
    const UnitSrc us = unit_src(p, uids, t, U);
    if (p.src == kSrcUnionDown && us.u != staged_u) {  // the unit's expert input, for every token
      named_barrier(1, kCT);
      stage_inputs(p, L, xs, ctid, (long long)us.u * p.C);
      staged_u = us.u;
    }
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int st = 0; st < spu; ++st, ++n) {
      const int s = n % nst, k = n / nst;
      if (ok && !mbar_wait(&full[s], k & 1)) {
        if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
        ok = false;
      }
      if (ok) {
        const int kb = (st * KS + ks) * strip_elems;
        strip_mma<FMT>(stages + s * stage_bytes, xs, L, line0, kb, d[0], g, tq);
        if (npair == 2) strip_mma<FMT>(stages + s * stage_bytes + member, xs, L, line0, kb, d[1], g, tq);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // finish one output (local row ri, token b) of the unit
    auto out = [&](int ri, int b, float v, float vu, int slot_b) {
      if (b >= p.B || ri >= us.rows) return;
      if (p.src == kSrcUnionDown) {
        const int slot = (us.u < U) ? p.slot_of[us.u * kMaxB + b] : p.top_k;
        if (slot >= 0) p.part_out[((long long)b * (p.top_k + 1) + slot) * p.R + us.a + ri] = v;
        return;
      }
      float* y = p.y ? p.y + (long long)b * p.ldy + us.a + ri : nullptr;
      if (p.epi == kEpiStore) *y = v;
      else if (p.epi == kEpiResid) *y += v;
      else if (p.epi == kEpiSwiglu) *y = siluf_(v) * vu;
      else {
        if (y) *y = v;
        argmax_merge(bv[slot_b], bi[slot_b], v, us.a + ri);
      }
    };
    if (KS == 1) {  // this warp holds whole rows: finish them from registers
      const int r0 = gw * kTileRows + g;
      out(r0, 2 * tq, d[0][0], d[1][0], 0);
      out(r0, 2 * tq + 1, d[0][1], d[1][1], 1);
      out(r0 + 8, 2 * tq, d[0][2], d[1][2], 0);
      out(r0 + 8, 2 * tq + 1, d[0][3], d[1][3], 1);
    } else {  // fixed-order sum of the KS strip lanes of each row group
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j == 1 && npair == 1) break;
        float* pw = part + j * kPartFloats + warp * kTileRows * kMaxB;
        pw[g * kMaxB + 2 * tq] = d[j][0];
        pw[g * kMaxB + 2 * tq + 1] = d[j][1];
        pw[(g + 8) * kMaxB + 2 * tq] = d[j][2];
        pw[(g + 8) * kMaxB + 2 * tq + 1] = d[j][3];
      }
      named_barrier(1, kCT);
      for (int e = ctid; e < TR * kMaxB; e += kCT) {  // b = ctid % 8 for every e of this thread
        const int b = e % kMaxB, ri = e / kMaxB;
        const int base = (ri / kTileRows) * KS * kTileRows * kMaxB + (ri % kTileRows) * kMaxB + b;
        float v = 0.f, vu = 0.f;
        for (int c = 0; c < KS; ++c) v += part[base + c * kTileRows * kMaxB];
        if (npair == 2)
          for (int c = 0; c < KS; ++c) vu += part[kPartFloats + base + c * kTileRows * kMaxB];
        out(ri, b, v, vu, 0);
      }
      named_barrier(1, kCT);
    }
  }
  if (named_barrier_or(1, kCT, !ok)) return;  // one decision for all compute threads
  if (p.epi != kEpiArgmax) return;

  // ------------------------------------------------------------ per-token argmax
  if (KS == 1) {
    if (bi[0] != 0x7fffffff) atomicMax(&s_key[2 * tq], am_key(bv[0], bi[0]));
    if (bi[1] != 0x7fffffff) atomicMax(&s_key[2 * tq + 1], am_key(bv[1], bi[1]));
  } else if (bi[0] != 0x7fffffff) {
    atomicMax(&s_key[ctid % kMaxB], am_key(bv[0], bi[0]));
  }
  named_barrier(1, kCT);
  if (ctid < p.B) {
    float v;
    int i;
    am_unkey(s_key[ctid], v, i);
    p.part_val[blockIdx.x * kMaxB + ctid] = v;
    p.part_idx[blockIdx.x * kMaxB + ctid] = i;
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

cudaError_t moe_reduce(float* y, int ldy, const float* part, const float* w, int R, int B, int top_k, cudaStream_t st,
                       bool pdl) {
  const int n = R * B;
  return launch_k(k_moe_reduce, dim3((n + 255) / 256), dim3(256), 0, st, pdl, y, ldy, part, w, R, B, top_k);
}

Plan plan(int R, int C, int fmt, int epi, int nsm, int row_mult) {
  Plan pl = {};
  pl.ok = false;
  const int strip_elems = fmt == kFmtQ4 ? 256 : 64;
  if (R <= 0 || C <= 0 || C % strip_elems != 0 || nsm <= 0) return pl;
  const int nstrips = C / strip_elems;
  const int npair = epi == kEpiSwiglu ? 2 : 1;
  const int stage_bytes = npair * (kStageW + (fmt == kFmtQ4 ? kStageS : 0));
  // row block of 16 * GW rows: the largest one whose units spread over the
  // SMs within 10% as evenly as the best choice (fewer row blocks need fewer
  // cross-warp sums)
  double score[4] = {0, 0, 0, 0};
  double best = 0;
  for (int i = 0; i < 4; ++i) {
    const int GW = 8 >> i, KS = kWarps / GW, TR = kTileRows * GW;
    if (nstrips % KS != 0 || (row_mult && row_mult % TR != 0)) continue;
    const long long units = (R + TR - 1) / TR;
    const long long per = (units + nsm - 1) / nsm;
    score[i] = (double)units / (double)(nsm * per) * (double)R / (double)(units * TR);
    if (score[i] > best) best = score[i];
  }
  int pick = -1;
  for (int i = 0; i < 4 && pick < 0; ++i)
    if (score[i] > 0 && score[i] >= 0.9 * best) pick = i;
  if (pick < 0) return pl;
  pl.gw = 8 >> pick;
  pl.ks = kWarps / pl.gw;
  const int TR = kTileRows * pl.gw;
  const long long units = (R + TR - 1) / TR;
  pl.ncta = (int)(units < nsm ? units : nsm);
  const int fixed = (fmt == kFmtBf16 ? 2 * kMaxB * (C * 2 + 16) : kMaxB * (C * 2 + 64)) + 4 * npair * kPartFloats +
                    (2 * kMaxStages + 1) * 8 +
                    1024;  // + alignment of the stages
  int ns = kInFlight / stage_bytes;
  ns = ns < 2 ? 2 : (ns > kMaxStages ? kMaxStages : ns);
  while (ns > 2 && fixed + ns * stage_bytes > kMaxSmem) --ns;
  pl.nstages = ns;
  pl.smem = fixed + ns * stage_bytes;
  pl.ok = pl.smem <= kMaxSmem;
  return pl;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// {128-byte strip, row, strip index} over `rows` rows of `width_bytes` of a
// matrix whose rows are `row_bytes` apart; box = 16 * GW rows x KS strips.
bool encode_w(CUtensorMap* m, const void* base, long long rows, int row_bytes, int TR, int KS, int width_bytes) {
  if (!base || rows <= 0 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kStrip, (cuuint64_t)rows, (cuuint64_t)(width_bytes / kStrip)};
  cuuint64_t str[2] = {(cuuint64_t)row_bytes, (cuuint64_t)kStrip};
  cuuint32_t box[3] = {(cuuint32_t)kStrip, (cuuint32_t)TR, (cuuint32_t)KS};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, str, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// The fp16 scales of the same rows (C columns of a row of ldw):
// {16 bytes (8 blocks) of a strip, row, strip index}.
bool encode_s(CUtensorMap* m, const void* base, long long rows, int C, int TR, int KS, int ldw) {
  if (!base || rows <= 0 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[3] = {16, (cuuint64_t)rows, (cuuint64_t)(C / 256)};
  cuuint64_t str[2] = {(cuuint64_t)(ldw / 16), 16};
  cuuint32_t box[3] = {16, (cuuint32_t)TR, (cuuint32_t)KS};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, str, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t init() {
  cudaError_t e = cudaFuncSetAttribute(k_bgemv<kFmtBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_bgemv<kFmtQ4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e == cudaSuccess && !g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) e = cudaErrorNotSupported;
    if (e == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return e;
}

cudaError_t launch(const Params& p0, const Plan& pl, cudaStream_t st, bool pdl) {
  if (!pl.ok || !g_encode || p0.B < 1 || p0.B > kMaxB) return cudaErrorInvalidValue;
  Params p = p0;
  p.ncta = pl.ncta;
  p.nstages = pl.nstages;
  p.gw = pl.gw;
  p.ks = pl.ks;
  const int TR = kTileRows * pl.gw;
  const int npair = p.epi == kEpiSwiglu ? 2 : 1;
  const int ldw = p.ldw > 0 ? p.ldw : p.C;  // a dense matrix may be a column slice of a wider one
  const int width_bytes = p.fmt == kFmtQ4 ? p.C / 2 : p.C * 2;
  const int row_bytes = p.fmt == kFmtQ4 ? ldw / 2 : ldw * 2;
  if (ldw < p.C || (p.src != kSrcDense && ldw != p.C) || (p.fmt == kFmtQ4 && ldw % 256)) return cudaErrorInvalidValue;
  alignas(64) Maps mp;
  memset(&mp, 0, sizeof(mp));
  for (int j = 0; j < npair; ++j) {
    if (p.src == kSrcDense) {
      if (!encode_w(&mp.w[j], p.W[j], p.R, row_bytes, TR, pl.ks, width_bytes)) return cudaErrorInvalidValue;
      if (p.fmt == kFmtQ4 && !encode_s(&mp.s[j], p.S[j], p.R, p.C, TR, pl.ks, ldw)) return cudaErrorInvalidValue;
      continue;
    }
    // union sources: the experts' matrices stacked, and the shared expert's
    const long long per = p.src == kSrcUnionRows ? p.slot_rows : p.R;
    if (p.n_exp < 1 || per % TR != 0 || p.exp_stride != per * row_bytes ||
        (p.fmt == kFmtQ4 && p.exp_sstride != per * (p.C / 16)))
      return cudaErrorInvalidValue;
    if (!encode_w(&mp.ew[j], p.exp_base[j], per * p.n_exp, row_bytes, TR, pl.ks, width_bytes) ||
        !encode_w(&mp.w[j], p.sh_base[j], per, row_bytes, TR, pl.ks, width_bytes))
      return cudaErrorInvalidValue;
    if (p.fmt == kFmtQ4 && (!encode_s(&mp.es[j], p.exp_scale[j], per * p.n_exp, p.C, TR, pl.ks, ldw) ||
                            !encode_s(&mp.s[j], p.sh_scale[j], per, p.C, TR, pl.ks, ldw)))
      return cudaErrorInvalidValue;
  }
  auto k = p.fmt == kFmtBf16 ? k_bgemv<kFmtBf16> : k_bgemv<kFmtQ4>;
  return launch_k(k, dim3(pl.ncta), dim3(kThreads), (size_t)pl.smem, st, pdl, p, mp);
}

}  // namespace bgemv
}  // namespace hy

// Device building blocks of the streaming GEMV, shared by the standalone GEMV
// kernel (gemv.cu) and the persistent decode-step kernel (step.cu).
//
// A GEMV phase: a CTA owns rows [r0, r1) of y = W * f(x).  A copy lane
// streams row tiles of W into a ring of shared-memory stages with bulk copies
// (TMA engine); eight compute warps hold their column slice of f(x) in
// registers and consume every tile, two (row, column-chunk) items per warp per
// pass with independent FMA chains and one paired butterfly reduction.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace gemv {

constexpr int kCT = kConsumerWarps * 32;  // compute threads

// Rows of the tile that starts at row a (expert slots are never straddled).
__device__ __forceinline__ int tile_rows_at(const Params& p, int src, int a, int r1) {
  int end = a + p.tile_rows;
  if (end > r1) end = r1;
  if (src == kSrcExpertRows) {
    const int slot_end = (a < p.top_k * p.slot_rows) ? (a / p.slot_rows + 1) * p.slot_rows : p.R;
    if (end > slot_end) end = slot_end;
  }
  return end - a;
}

__device__ __forceinline__ int checked_expert(const Params& p, int slot) {
  int e = p.moe_ids[slot];
  if (e < 0 || e >= p.n_experts) {  // never read outside the expert tensor
    set_guard(p.guard, kGuardBadIndex);
    e = 0;
  }
  return e;
}

// Address of row a of pair member j.
__device__ __forceinline__ const uint8_t* row_src(const Params& p, int src, int j, int a) {
  const long long rb = (long long)p.C * 2;
  if (src == kSrcDense) return p.W[j] + (long long)a * rb;
  if (a < p.top_k * p.slot_rows) {
    const int s = a / p.slot_rows;
    return p.exp_base[j] + (long long)checked_expert(p, s) * p.exp_stride + (long long)(a - s * p.slot_rows) * rb;
  }
  return p.sh_base[j] + (long long)(a - p.top_k * p.slot_rows) * rb;
}

// Copy lane: issue the tile [a, a + rows) into `dst`, completing on `bar`.
__device__ __forceinline__ void issue_tile(const Params& p, int src, int npair, int a, int rows, uint8_t* dst,
                                           uint64_t* bar, uint64_t pol) {
  if (src == kSrcExpertSegs) {
    const int nseg = p.top_k + 1;
    const uint32_t seg_bytes = (uint32_t)rows * p.seg_cols * 2;
    mbar_arrive_expect_tx(bar, seg_bytes * nseg);
    for (int g = 0; g < nseg; ++g) {
      const uint8_t* base = (g < p.top_k) ? p.exp_base[0] + (long long)checked_expert(p, g) * p.exp_stride : p.sh_base[0];
      bulk_g2s(dst + g * seg_bytes, base + (long long)a * p.seg_cols * 2, seg_bytes, bar, pol);
    }
  } else {
    const uint32_t bytes = (uint32_t)rows * p.C * 2;
    mbar_arrive_expect_tx(bar, bytes * npair);
    for (int j = 0; j < npair; ++j) bulk_g2s(dst + j * bytes, row_src(p, src, j, a), bytes, bar, pol);
  }
}

// Compute threads: the input vector f(x) into shared memory xs (RMSNorm when
// p.norm_g is set).  s_red: >= 8 floats of shared scratch.
__device__ __forceinline__ void load_input(const Params& p, int in, float* xs, float* s_red, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  int tok = 0;
  if (in == kInEmbed) {
    tok = p.tok[0];
    if (tok < 0 || tok >= p.vocab) {
      if (ctid == 0) set_guard(p.guard, kGuardBadIndex);
      tok = 0;
    }
  }
  float ss = 0.f;
  for (int c = ctid * 4; c < p.C; c += kCT * 4) {
    float4 v;
    if (in == kInX) {
      v = *reinterpret_cast<const float4*>(p.x + c);
    } else if (in == kInEmbed) {
      const uint2 e = *reinterpret_cast<const uint2*>(p.embed + (long long)tok * p.C + c);
      v = make_float4(bf16_lo(e.x), bf16_hi(e.x), bf16_lo(e.y), bf16_hi(e.y));
      if (blockIdx.x == 0) *reinterpret_cast<float4*>(p.x_out + c) = v;
    } else {  // kInMoeZ: routing-weighted expert activations
      const float w = p.moe_w[c / p.seg_cols];
      v = *reinterpret_cast<const float4*>(p.x + c);
      v.x *= w;
      v.y *= w;
      v.z *= w;
      v.w *= w;
    }
    *reinterpret_cast<float4*>(xs + c) = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (p.norm_g) {
    ss = warp_sum(ss);
    if (lane == 0) s_red[warp] = ss;
    named_barrier(1, kCT);
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) t += s_red[w];
    const float sc = 1.0f / sqrtf(t / (float)p.C + p.eps);
    for (int c = ctid; c < p.C; c += kCT) xs[c] = xs[c] * sc * p.norm_g[c];
  }
  named_barrier(1, kCT);
}

// Per-lane state of a compute warp: its column chunk, the input slice in
// registers, and the shared-memory offsets of its 16-byte vectors.
template <int VPL>
struct LaneSlice {
  float xr[VPL][8];
  int off[VPL];
  int segof[VPL];
  bool valid[VPL];
  int chunk, rg, nrg, seg_row_bytes;
};

template <int VPL>
__device__ __forceinline__ void lane_setup(const Params& p, int src, const float* xs, LaneSlice<VPL>& L, int warp,
                                           int lane) {
  L.chunk = warp % p.nchunk;
  L.rg = warp / p.nchunk;
  L.nrg = kConsumerWarps / p.nchunk;
  const int seg_cols = (src == kSrcExpertSegs) ? p.seg_cols : p.C;
  L.seg_row_bytes = seg_cols * 2;
  const int nvec = p.C / 8, seg_vecs = seg_cols / 8;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int lv = lane + 32 * j;
    const int v = L.chunk * p.chunk_vecs + lv;
    L.valid[j] = (lv < p.chunk_vecs) && (v < nvec);
    const int vv = L.valid[j] ? v : 0;
    L.segof[j] = vv / seg_vecs;
    L.off[j] = (vv % seg_vecs) * 16;
#pragma unroll
    for (int e = 0; e < 8; ++e) L.xr[j][e] = L.valid[j] ? xs[vv * 8 + e] : 0.f;
  }
}

// Consume one tile (rows [a, a + rows) of the CTA range starting at r0):
// partial dot products of this warp's column chunk go to red.
template <int VPL>
__device__ __forceinline__ void consume_tile(const Params& p, int src, int npair, const LaneSlice<VPL>& L,
                                             const uint8_t* st, int rows, int a, int r0, int rows_cta, float* red,
                                             int lane) {
  const int items = rows * npair;
  const int segstride = (src == kSrcExpertSegs) ? rows * L.seg_row_bytes : 0;
  for (int q = L.rg; q < items; q += 2 * L.nrg) {
    const int q2 = q + L.nrg;
    const bool has2 = q2 < items;
    const int j0 = q / rows, i0 = q - j0 * rows;
    const int qq = has2 ? q2 : q;
    const int j1 = qq / rows, i1 = qq - j1 * rows;
    const uint8_t* p0 = (src == kSrcExpertSegs) ? st + i0 * L.seg_row_bytes : st + (j0 * rows + i0) * p.C * 2;
    const uint8_t* p1 = (src == kSrcExpertSegs) ? st + i1 * L.seg_row_bytes : st + (j1 * rows + i1) * p.C * 2;
    uint4 w0[VPL], w1[VPL];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      if (L.valid[u]) {
        w0[u] = *reinterpret_cast<const uint4*>(p0 + L.segof[u] * segstride + L.off[u]);
        w1[u] = *reinterpret_cast<const uint4*>(p1 + L.segof[u] * segstride + L.off[u]);
      }
    }
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      if (L.valid[u]) {
        a0 += dot8(w0[u], L.xr[u]);
        a1 += dot8(w1[u], L.xr[u]);
      }
    }
    // paired butterfly: lanes 0..15 finish item q, lanes 16..31 item q2
    float keep = (lane < 16) ? a0 : a1;
    keep += __shfl_xor_sync(0xffffffffu, (lane < 16) ? a1 : a0, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    if (lane == 0) red[((j0 * rows_cta) + (a - r0) + i0) * p.nchunk + L.chunk] = keep;
    if (lane == 16 && has2) red[((j1 * rows_cta) + (a - r0) + i1) * p.nchunk + L.chunk] = keep;
  }
}

// Shared scratch of the epilogue.
struct EpiShared {
  float red[kConsumerWarps];
  int redi[kConsumerWarps];
  int sel[64];
  float selv[64];
  int last;
};

__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float ov, int oi) {
  if (ov > bv || (ov == bv && oi < bi)) {
    bv = ov;
    bi = oi;
  }
}

// Epilogue over the CTA's rows (after all tiles): store, residual add,
// SwiGLU, or argmax / router top-k finished by the last CTA to arrive (an
// atomic ticket: no CTA waits for another).
__device__ __forceinline__ void epilogue(const Params& p, int epi, const float* red, int r0, int rows_cta,
                                         EpiShared& sh, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  auto row_val = [&](int jj, int i) {
    float v = 0.f;
    for (int c = 0; c < p.nchunk; ++c) v += red[((jj * rows_cta) + i) * p.nchunk + c];
    return v;
  };
  if (epi == kEpiStore) {
    for (int i = ctid; i < rows_cta; i += kCT) p.y[r0 + i] = row_val(0, i);
    return;
  }
  if (epi == kEpiResid) {
    for (int i = ctid; i < rows_cta; i += kCT) p.y[r0 + i] += row_val(0, i);
    return;
  }
  if (epi == kEpiSwiglu) {
    for (int i = ctid; i < rows_cta; i += kCT) p.y[r0 + i] = siluf_(row_val(0, i)) * row_val(1, i);
    return;
  }
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = ctid; i < rows_cta; i += kCT) {
    const float v = row_val(0, i);
    if (epi == kEpiArgmax) {
      if (p.y) p.y[r0 + i] = v;
      argmax_merge(bv, bi, v, r0 + i);
    } else {
      p.router_logits[r0 + i] = v;
    }
  }
  if (epi == kEpiArgmax) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) {
      sh.red[warp] = bv;
      sh.redi[warp] = bi;
    }
    named_barrier(1, kCT);
    if (ctid == 0) {
      for (int w = 1; w < kConsumerWarps; ++w) argmax_merge(bv, bi, sh.red[w], sh.redi[w]);
      p.part_val[blockIdx.x] = bv;
      p.part_idx[blockIdx.x] = bi;
    }
  }
  if (ctid == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(p.counter, 1u);
    sh.last = (ticket == (unsigned)(p.ncta - 1));
  }
  named_barrier(1, kCT);
  if (!sh.last) return;
  __threadfence();
  if (epi == kEpiArgmax) {
    if (warp == 0) {
      float v = -INFINITY;
      int vi = 0x7fffffff;
      for (int c = lane; c < p.ncta; c += 32) argmax_merge(v, vi, __ldcg(p.part_val + c), __ldcg(p.part_idx + c));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
        argmax_merge(v, vi, ov, oi);
      }
      if (lane == 0) {
        *p.ids_out = vi;
        *p.counter = 0u;
        if (p.len_inc) *p.len_inc += 1;
      }
    }
    return;
  }
  // router: top-k over the E expert logits (FP32 compare, lowest index on
  // ties), softmax over the selected logits, sigmoid gate of the shared
  // expert's row ("Fourteen hours to 100 tokens per second", "The router with
  // 257 rows").
  const int E = p.n_experts;
  for (int kk = 0; kk < p.top_k; ++kk) {
    float v = -INFINITY;
    int vi = 0x7fffffff;
    for (int e = ctid; e < E; e += kCT) {
      bool taken = false;
      for (int q = 0; q < kk; ++q) taken |= (sh.sel[q] == e);
      if (!taken) argmax_merge(v, vi, __ldcg(p.router_logits + e), e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
      argmax_merge(v, vi, ov, oi);
    }
    if (lane == 0) {
      sh.red[warp] = v;
      sh.redi[warp] = vi;
    }
    named_barrier(1, kCT);
    if (ctid == 0) {
      for (int w = 1; w < kConsumerWarps; ++w) argmax_merge(v, vi, sh.red[w], sh.redi[w]);
      sh.sel[kk] = vi;
      sh.selv[kk] = v;
    }
    named_barrier(1, kCT);
  }
  if (ctid == 0) {
    const float m = sh.selv[0];
    float den = 0.f;
    for (int q = 0; q < p.top_k; ++q) den += __expf(sh.selv[q] - m);
    for (int q = 0; q < p.top_k; ++q) {
      p.out_ids[q] = sh.sel[q];
      p.out_w[q] = __expf(sh.selv[q] - m) / den;
      if (p.dbg_ids) p.dbg_ids[q] = sh.sel[q];
    }
    p.out_w[p.top_k] = sigmoidf_(__ldcg(p.router_logits + E));
    *p.counter = 0u;
  }
  if (p.dbg_logits)
    for (int e = ctid; e <= E; e += kCT) p.dbg_logits[e] = __ldcg(p.router_logits + e);
}

}  // namespace gemv
}  // namespace hy

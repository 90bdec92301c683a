// Device building blocks of the streaming GEMV kernel (gemv.cu).
//
// A CTA owns rows [r0, r1) of y = W * f(x).  A copy lane streams row tiles
// of W into a ring of shared-memory stages with bulk copies (TMA engine);
// the compute warps hold their column slice of f(x) in
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

// Copy lane: L2 prefetch of the tile [a, a + rows) (same addresses as issue_tile).
__device__ __forceinline__ void prefetch_tile(const Params& p, int src, int npair, int a, int rows) {
  if (src == kSrcExpertSegs) {
    const uint32_t seg_bytes = (uint32_t)rows * p.seg_cols * 2;
    for (int g = 0; g <= p.top_k; ++g) {
      const uint8_t* base = (g < p.top_k) ? p.exp_base[0] + (long long)checked_expert(p, g) * p.exp_stride : p.sh_base[0];
      bulk_prefetch_l2(base + (long long)a * p.seg_cols * 2, seg_bytes);
    }
  } else {
    const uint32_t bytes = (uint32_t)rows * p.C * 2;
    for (int j = 0; j < npair; ++j) bulk_prefetch_l2(row_src(p, src, j, a), bytes);
  }
}

// Copy lane: L2 prefetch of this CTA's share of the next kernels' first reads.
__device__ __forceinline__ void prefetch_next(const Params& p) {
  const int b = blockIdx.x;
  for (int i = 0; i < p.n_nx; ++i) {
    const PfSpan& s = p.nx[i];
    if (b >= s.ncta) continue;
    const long long r0 = (long long)b * s.rows / s.ncta, r1 = (long long)(b + 1) * s.rows / s.ncta;
    long long bytes = (r1 - r0) * s.row_bytes;
    if (bytes > s.bytes) bytes = s.bytes & ~15LL;
    const uint8_t* src = s.base + r0 * s.row_bytes;
    for (long long o = 0; o < bytes; o += 65536) bulk_prefetch_l2(src + o, (uint32_t)(bytes - o < 65536 ? bytes - o : 65536));
  }
}

// The input vector f(x) reaches shared memory by bulk copy from the copy
// lane, right after griddepcontrol.wait and ahead of all but the first weight
// tiles: a load issued by the compute warps would queue behind the whole ring
// already requested for this SM.  xs holds x (FP32) or the embedding row
// (bf16), gs the RMSNorm gain (requested before the wait: it is a weight), mw
// the routing weights of the MoE down projection.
__device__ __forceinline__ uint32_t input_bytes(const Params& p, int in) {
  uint32_t b = (in == kInEmbed) ? p.C * 2 : p.C * 4;
  if (in == kInMoeZ) b += ((p.top_k + 1) * 4 + 15) & ~15;
  return b;
}

// Copy lane, after griddepcontrol.wait.
__device__ __forceinline__ void issue_input(const Params& p, int in, float* xs, float* mw, uint64_t* xbar,
                                            uint64_t pol) {
  if (in == kInEmbed) {
    int tok = *p.tok;
    if (tok < 0 || tok >= p.vocab) {  // never read outside the embedding table
      set_guard(p.guard, kGuardBadIndex);
      tok = 0;
    }
    bulk_g2s(xs, p.embed + (long long)tok * p.C, p.C * 2, xbar, pol);
  } else {
    bulk_g2s(xs, p.x, p.C * 4, xbar, pol);
    if (in == kInMoeZ) bulk_g2s(mw, p.moe_w, ((p.top_k + 1) * 4 + 15) & ~15, xbar, pol);
  }
}

// Elements 8v .. 8v+7 of the input before normalisation, with 16-byte shared
// loads (a lane's 32 contiguous bytes in two accesses, not eight scalar ones
// that would hit the same banks as seven other lanes).
__device__ __forceinline__ void input_vec8(const Params& p, int in, const float* xs, const float* mw, int v,
                                           float* out) {
  if (in == kInEmbed) {
    const uint4 u = reinterpret_cast<const uint4*>(xs)[v];
    out[0] = bf16_lo(u.x);
    out[1] = bf16_hi(u.x);
    out[2] = bf16_lo(u.y);
    out[3] = bf16_hi(u.y);
    out[4] = bf16_lo(u.z);
    out[5] = bf16_hi(u.z);
    out[6] = bf16_lo(u.w);
    out[7] = bf16_hi(u.w);
    return;
  }
  const float4 a = reinterpret_cast<const float4*>(xs)[2 * v];
  const float4 b = reinterpret_cast<const float4*>(xs)[2 * v + 1];
  const float w = (in == kInMoeZ) ? mw[(8 * v) / p.seg_cols] : 1.f;
  out[0] = a.x * w;
  out[1] = a.y * w;
  out[2] = a.z * w;
  out[3] = a.w * w;
  out[4] = b.x * w;
  out[5] = b.y * w;
  out[6] = b.z * w;
  out[7] = b.w * w;
}

// Compute threads, once the input has landed: the RMSNorm scale (1 without a
// gain); CTA 0 of the embedding GEMV also initialises the residual stream.
// s_red: >= kConsumerWarps floats of shared scratch.
__device__ __forceinline__ float input_scale(const Params& p, int in, const float* xs, const float* mw, float* s_red,
                                             int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int nvec = p.C / 8;
  if (in == kInEmbed && blockIdx.x == 0)
    for (int v = ctid; v < nvec; v += kCT) {
      float e[8];
      input_vec8(p, in, xs, mw, v, e);
      reinterpret_cast<float4*>(p.x_out)[2 * v] = make_float4(e[0], e[1], e[2], e[3]);
      reinterpret_cast<float4*>(p.x_out)[2 * v + 1] = make_float4(e[4], e[5], e[6], e[7]);
    }
  if (!p.norm_g) return 1.f;
  float ss = 0.f;
  for (int v = ctid; v < nvec; v += kCT) {
    float e[8];
    input_vec8(p, in, xs, mw, v, e);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(e[i], e[i], ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) s_red[warp] = ss;
  named_barrier(1, kCT);
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) t += s_red[w];
  return 1.0f / sqrtf(t / (float)p.C + p.eps);
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
__device__ __forceinline__ void lane_setup(const Params& p, int src, int in, const float* xs, const float* gs,
                                           const float* mw, float sc, LaneSlice<VPL>& L, int warp, int lane) {
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
    float e8[8];
    input_vec8(p, in, xs, mw, vv, e8);
    if (p.norm_g) {
      const float4 g0 = reinterpret_cast<const float4*>(gs)[2 * vv];
      const float4 g1 = reinterpret_cast<const float4*>(gs)[2 * vv + 1];
      const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) e8[e] = e8[e] * sc * g[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) L.xr[j][e] = L.valid[j] ? e8[e] : 0.f;
  }
}

// dot of 8 bf16 (one 16-byte vector) with 8 FP32 values, accumulated into acc
__device__ __forceinline__ float dot8_acc(const uint4 w, const float* x, float acc) {
  acc = fmaf(bf16_lo(w.x), x[0], acc);
  acc = fmaf(bf16_hi(w.x), x[1], acc);
  acc = fmaf(bf16_lo(w.y), x[2], acc);
  acc = fmaf(bf16_hi(w.y), x[3], acc);
  acc = fmaf(bf16_lo(w.z), x[4], acc);
  acc = fmaf(bf16_hi(w.z), x[5], acc);
  acc = fmaf(bf16_lo(w.w), x[6], acc);
  acc = fmaf(bf16_hi(w.w), x[7], acc);
  return acc;
}

// Consume one tile (rows [a, a + rows) of the CTA range starting at r0): the
// partial dot products of this warp's column chunk go to red.  A warp owns
// the rows i = rg (mod nrg) of every tile and finishes two items per pass
// (rows i and i + nrg, or the gate and up rows of row i) with one paired
// butterfly; addresses advance by a fixed row stride, without divisions.
// FULL: every lane's VPL vectors lie inside its chunk (chunk_vecs == 32 VPL),
// so no vector is predicated off and a dense row's vectors sit 512 bytes apart.
template <int VPL, int SRC, int NPAIR, bool FULL>
__device__ __forceinline__ void consume_tile(const Params& p, const LaneSlice<VPL>& L, const uint8_t* st, int rows,
                                             int row0, int rows_cta, float* red, int lane) {
  // byte offset of this lane's vector u within a row, and the row stride
  int uoff[VPL];
  int stride;
  if (SRC == kSrcExpertSegs) {
    stride = L.seg_row_bytes;
#pragma unroll
    for (int u = 0; u < VPL; ++u) uoff[u] = L.segof[u] * rows * L.seg_row_bytes + L.off[u];
  } else {
    stride = p.C * 2;
#pragma unroll
    for (int u = 0; u < VPL; ++u) uoff[u] = FULL ? L.off[0] + 512 * u : L.off[u];
  }
  const int member_bytes = rows * stride;  // gate rows, then up rows (pairs)
  const int step = (NPAIR == 2) ? L.nrg : 2 * L.nrg;
  for (int i = L.rg; i < rows; i += step) {
    int i1, j1;
    const uint8_t* p0 = st + i * stride;
    const uint8_t* p1;
    bool has2;
    if (NPAIR == 2) {
      i1 = i;
      j1 = 1;
      has2 = true;
      p1 = p0 + member_bytes;
    } else {
      i1 = i + L.nrg;
      j1 = 0;
      has2 = i1 < rows;
      p1 = has2 ? st + i1 * stride : p0;
    }
    // four independent packed accumulator pairs: item x (vector parity)
    float e0[2] = {0.f, 0.f}, o0[2] = {0.f, 0.f}, e1[2] = {0.f, 0.f}, o1[2] = {0.f, 0.f};
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      if (FULL || L.valid[u]) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(p0 + uoff[u]);
        const uint4 w1 = *reinterpret_cast<const uint4*>(p1 + uoff[u]);
        dot8_acc2(w0, L.xr[u], e0[u & 1], o0[u & 1]);
        dot8_acc2(w1, L.xr[u], e1[u & 1], o1[u & 1]);
      }
    }
    const float a0 = (e0[0] + o0[0]) + (e0[1] + o0[1]);
    const float a1 = (e1[0] + o1[0]) + (e1[1] + o1[1]);
    // paired butterfly: lanes 0..15 finish the first item, lanes 16..31 the second
    float keep = (lane < 16) ? a0 : a1;
    keep += __shfl_xor_sync(0xffffffffu, (lane < 16) ? a1 : a0, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    if (lane == 0) red[(row0 + i) * p.nchunk + L.chunk] = keep;
    if (lane == 16 && has2) red[(j1 * rows_cta + row0 + i1) * p.nchunk + L.chunk] = keep;
  }
}

// Shared scratch of the epilogue.
struct EpiShared {
  float mw[kMaxTopK + 4];  // routing weights (bulk-copy destination: 16-byte multiple)
  int sel[kMaxTopK];
  float selv[kMaxTopK];
  float red[kConsumerWarps];
  int redi[kConsumerWarps];
  int last;
};

__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float ov, int oi) {
  if (ov > bv || (ov == bv && oi < bi)) {
    bv = ov;
    bi = oi;
  }
}

// One thread: softmax over the selected logits and the shared expert's gate
// sigmoid(gate_logit) into out_w [top_k + 1], the ids into out_ids (and the
// debug copy).
__device__ __forceinline__ void route_weights(const Params& p, const int* sel, const float* selv, float gate_logit) {
  const float m = selv[0];
  float den = 0.f;
  for (int q = 0; q < p.top_k; ++q) den += __expf(selv[q] - m);
  for (int q = 0; q < p.top_k; ++q) {
    p.out_ids[q] = sel[q];
    p.out_w[q] = __expf(selv[q] - m) / den;
    if (p.dbg_ids) p.dbg_ids[q] = sel[q];
  }
  p.out_w[p.top_k] = sigmoidf_(gate_logit);
}

// Epilogue over the CTA's rows (after all tiles): store, residual add,
// SwiGLU, or argmax finished by the last CTA to arrive (an atomic ticket: no
// CTA waits for another).
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
  // argmax: per-CTA best (row value, lowest index on ties), then the last CTA merges
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = ctid; i < rows_cta; i += kCT) {
    const float v = row_val(0, i);
    if (p.y) p.y[r0 + i] = v;
    argmax_merge(bv, bi, v, r0 + i);
  }
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
    __threadfence();
    const unsigned ticket = atomicAdd(p.counter, 1u);
    sh.last = (ticket == (unsigned)(p.ncta - 1));
  }
  named_barrier(1, kCT);
  if (!sh.last) return;
  __threadfence();
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
}

}  // namespace gemv
}  // namespace hy

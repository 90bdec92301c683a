// Streaming GEMV for batch-1 decode on sm_103a: y = W * f(x), W bf16 [R][C].
//
// Decode at M = 1 is a matrix-vector product and the weight stream is the
// whole cost ("Beating llama.cpp from Scratch on Consumer AMD", Act 0, pass 3
// and Act 6: weight GEMV kernels take 88.85% of the 4B decode time).  Design:
//   * persistent grid, one CTA per SM, each owning a contiguous row range;
//   * one copy warp streams row tiles HBM -> shared memory with bulk copies on
//     the TMA engine (cp.async.bulk, L2 evict-first), ~96 KB deep, completion
//     on mbarriers; tiles of the next kernel's weights start streaming before
//     griddepcontrol.wait releases the kernel (programmatic dependent launch);
//   * eight compute warps hold their slice of the (normalised) input vector in
//     registers, read 16-byte bf16 vectors from shared memory, accumulate in
//     FP32, and reduce with warp shuffles;
//   * fused prologues (RMSNorm, embedding gather, MoE weighted activations) and
//     epilogues (store, residual add, SwiGLU, argmax, router top-k).
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace gemv {

namespace {

struct TileWalk {
  // kSrcExpertRows: tiles never straddle an expert slot.
  __device__ __forceinline__ static int rows_of(const Params& p, int src, int a, int r1) {
    int end = a + p.tile_rows;
    if (end > r1) end = r1;
    if (src == kSrcExpertRows) {
      int slot_end = (a < p.top_k * p.slot_rows) ? (a / p.slot_rows + 1) * p.slot_rows : p.R;
      if (end > slot_end) end = slot_end;
    }
    return end - a;
  }
};

// Address of row `a` (first of a tile) of pair member j.
__device__ __forceinline__ const uint8_t* row_src(const Params& p, int src, int j, int a) {
  const long long rb = (long long)p.C * 2;
  if (src == kSrcDense) return p.W[j] + (long long)a * rb;
  // kSrcExpertRows
  if (a < p.top_k * p.slot_rows) {
    int s = a / p.slot_rows;
    int e = p.moe_ids[s];
    if (e < 0 || e >= p.n_experts) {  // never read outside the expert tensor
      set_guard(p.guard, kGuardBadIndex);
      e = 0;
    }
    return p.exp_base[j] + (long long)e * p.exp_stride + (long long)(a - s * p.slot_rows) * rb;
  }
  return p.sh_base[j] + (long long)(a - p.top_k * p.slot_rows) * rb;
}

template <int VPL, int SRC, int IN, int EPI>
__global__ void __launch_bounds__(kThreads, 1) k_gemv(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int kStages = p.nstages;
  uint8_t* stages = smem;
  float* xs = reinterpret_cast<float*>(smem + kStages * p.stage_bytes);
  float* red = xs + p.xs_floats;
  const int npair = (EPI == kEpiSwiglu) ? 2 : 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + ((p.rows_cta_max * npair * p.nchunk + 1) & ~1));
  uint64_t* empty = full + kMaxStages;
  __shared__ float s_red[kConsumerWarps];
  __shared__ int s_redi[kConsumerWarps];
  __shared__ float s_scale;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (int)((long long)blockIdx.x * p.R / p.ncta);
  const int r1 = (int)((long long)(blockIdx.x + 1) * p.R / p.ncta);
  const int nseg = (SRC == kSrcExpertSegs) ? p.top_k + 1 : 1;
  const int seg_cols = (SRC == kSrcExpertSegs) ? p.seg_cols : p.C;
  const int seg_row_bytes = seg_cols * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy warp
  // Lanes 0..nprod-1 each own the stages s with s % nprod == lane and issue
  // the tiles that land there (independent copy streams).
  if (warp == kConsumerWarps) {
    if (lane < p.nprod) {
      const uint64_t pol = l2_evict_first_policy();
      if (SRC != kSrcDense) pdl_wait();  // expert ids come from the router kernel
      int lastt[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) lastt[s] = -1;
      int t = 0;
      for (int a = r0; a < r1; ++t) {
        const int rows = TileWalk::rows_of(p, SRC, a, r1);
        const int s = t % kStages, k = t / kStages;
        if (s % p.nprod == lane) {
          if (t >= kStages && !mbar_wait(&empty[s], (k - 1) & 1)) {
            set_guard(p.guard, kGuardWaitTimeout);
            break;
          }
          uint8_t* dst = stages + s * p.stage_bytes;
          if (SRC == kSrcExpertSegs) {
            const uint32_t seg_bytes = (uint32_t)rows * seg_row_bytes;
            mbar_arrive_expect_tx(&full[s], seg_bytes * nseg);
            for (int g = 0; g < nseg; ++g) {
              const uint8_t* base;
              if (g < p.top_k) {
                int e = p.moe_ids[g];
                if (e < 0 || e >= p.n_experts) {
                  set_guard(p.guard, kGuardBadIndex);
                  e = 0;
                }
                base = p.exp_base[0] + (long long)e * p.exp_stride;
              } else {
                base = p.sh_base[0];
              }
              bulk_g2s(dst + g * seg_bytes, base + (long long)a * seg_row_bytes, seg_bytes, &full[s], pol);
            }
          } else {
            const uint32_t bytes = (uint32_t)rows * p.C * 2;
            mbar_arrive_expect_tx(&full[s], bytes * npair);
            for (int j = 0; j < npair; ++j) bulk_g2s(dst + j * bytes, row_src(p, SRC, j, a), bytes, &full[s], pol);
          }
          lastt[s] = t;
        }
        a += rows;
      }
      // Drain: the CTA must not retire while copies this lane issued are in flight.
      for (int s = 0; s < kStages; ++s)
        if (lastt[s] >= 0 && !mbar_wait(&full[s], (lastt[s] / kStages) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;  // 0..255
  const int nct = kConsumerWarps * 32;
  pdl_wait();
  pdl_launch_dependents();

  // prologue: the input vector into shared memory
  int tok = 0;
  if (IN == kInEmbed) {
    tok = p.tok[0];
    if (tok < 0 || tok >= p.vocab) {
      if (ctid == 0) set_guard(p.guard, kGuardBadIndex);
      tok = 0;
    }
  }
  float ss = 0.f;
  for (int c = ctid * 4; c < p.C; c += nct * 4) {
    float4 v;
    if (IN == kInX) {
      v = *reinterpret_cast<const float4*>(p.x + c);
    } else if (IN == kInEmbed) {
      const uint2 e = *reinterpret_cast<const uint2*>(p.embed + (long long)tok * p.C + c);
      v = make_float4(bf16_lo(e.x), bf16_hi(e.x), bf16_lo(e.y), bf16_hi(e.y));
      if (blockIdx.x == 0) *reinterpret_cast<float4*>(p.x_out + c) = v;
    } else {  // kInMoeZ: routing-weighted expert activations
      const int g = c / p.seg_cols;
      const float w = p.moe_w[g];
      v = *reinterpret_cast<const float4*>(p.x + c);
      v.x *= w; v.y *= w; v.z *= w; v.w *= w;
    }
    *reinterpret_cast<float4*>(xs + c) = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (p.norm_g) {
    ss = warp_sum(ss);
    if (lane == 0) s_red[warp] = ss;
    named_barrier(1, nct);
    if (ctid == 0) {
      float t = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w) t += s_red[w];
      s_scale = 1.0f / sqrtf(t / (float)p.C + p.eps);
    }
    named_barrier(1, nct);
    const float sc = s_scale;
    for (int c = ctid; c < p.C; c += nct) xs[c] = xs[c] * sc * p.norm_g[c];
  }
  named_barrier(1, nct);

  // this warp's column chunk and its input slice in registers
  const int chunk = warp % p.nchunk;
  const int rg = warp / p.nchunk, nrg = kConsumerWarps / p.nchunk;
  const int nvec = p.C / 8;
  const int seg_vecs = seg_cols / 8;
  float xr[VPL][8];
  int off[VPL];
  bool valid[VPL];
  int segof[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int lv = lane + 32 * j;
    const int v = chunk * p.chunk_vecs + lv;
    valid[j] = (lv < p.chunk_vecs) && (v < nvec);
    const int vv = valid[j] ? v : 0;
    segof[j] = vv / seg_vecs;
    off[j] = (vv % seg_vecs) * 16;
#pragma unroll
    for (int e = 0; e < 8; ++e) xr[j][e] = valid[j] ? xs[vv * 8 + e] : 0.f;
  }

  const int rows_cta = r1 - r0;
  bool abort = false;
  int t = 0;
  for (int a = r0; a < r1; ++t) {
    const int rows = TileWalk::rows_of(p, SRC, a, r1);
    const int s = t % kStages, k = t / kStages;
    if (!mbar_wait(&full[s], k & 1)) {
      if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
      abort = true;
      break;
    }
    const uint8_t* st = stages + s * p.stage_bytes;
    const int items = rows * npair;
    const int segstride = (SRC == kSrcExpertSegs) ? rows * seg_row_bytes : 0;
    auto item_ptr = [&](int q) -> const uint8_t* {
      const int j = q / rows, i = q - j * rows;
      return (SRC == kSrcExpertSegs) ? st + i * seg_row_bytes : st + (j * rows + i) * p.C * 2;
    };
    auto item_red = [&](int q) -> float* {
      const int j = q / rows, i = q - j * rows;
      return red + ((j * rows_cta) + (a - r0) + i) * p.nchunk + chunk;
    };
    // two items per pass: independent loads and FMA chains, then one paired
    // butterfly (lanes 0..15 finish item 0, lanes 16..31 item 1)
    for (int q = rg; q < items; q += 2 * nrg) {
      const int q2 = q + nrg;
      const bool has2 = q2 < items;
      const uint8_t* p0 = item_ptr(q);
      const uint8_t* p1 = has2 ? item_ptr(q2) : p0;
      uint4 w0[VPL], w1[VPL];
#pragma unroll
      for (int u = 0; u < VPL; ++u) {
        if (valid[u]) {
          w0[u] = *reinterpret_cast<const uint4*>(p0 + segof[u] * segstride + off[u]);
          w1[u] = *reinterpret_cast<const uint4*>(p1 + segof[u] * segstride + off[u]);
        }
      }
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int u = 0; u < VPL; ++u) {
        if (valid[u]) {
          a0 += dot8(w0[u], xr[u]);
          a1 += dot8(w1[u], xr[u]);
        }
      }
      float keep = (lane < 16) ? a0 : a1;
      keep += __shfl_xor_sync(0xffffffffu, (lane < 16) ? a1 : a0, 16);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
      if (lane == 0) *item_red(q) = keep;
      if (lane == 16 && has2) *item_red(q2) = keep;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    a += rows;
  }
  named_barrier(1, nct);
  if (abort) return;

  // ------------------------------------------------------------ epilogue
  auto row_val = [&](int jj, int i) {
    float v = 0.f;
    for (int c = 0; c < p.nchunk; ++c) v += red[((jj * rows_cta) + i) * p.nchunk + c];
    return v;
  };

  if (EPI == kEpiStore) {
    for (int i = ctid; i < rows_cta; i += nct) p.y[r0 + i] = row_val(0, i);
  } else if (EPI == kEpiResid) {
    for (int i = ctid; i < rows_cta; i += nct) p.y[r0 + i] += row_val(0, i);
  } else if (EPI == kEpiSwiglu) {
    for (int i = ctid; i < rows_cta; i += nct) {
      const float g = row_val(0, i), u = row_val(1, i);
      p.y[r0 + i] = siluf_(g) * u;
    }
  } else {
    // argmax / router: per-CTA part, then the last CTA to finish reduces.
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = ctid; i < rows_cta; i += nct) {
      const float v = row_val(0, i);
      if (EPI == kEpiArgmax) {
        if (p.y) p.y[r0 + i] = v;
        if (v > bv || (v == bv && r0 + i < bi)) { bv = v; bi = r0 + i; }
      } else {
        p.router_logits[r0 + i] = v;
      }
    }
    if (EPI == kEpiArgmax) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) { s_red[warp] = bv; s_redi[warp] = bi; }
      named_barrier(1, nct);
      if (ctid == 0) {
        for (int w = 1; w < kConsumerWarps; ++w)
          if (s_red[w] > bv || (s_red[w] == bv && s_redi[w] < bi)) { bv = s_red[w]; bi = s_redi[w]; }
        p.part_val[blockIdx.x] = bv;
        p.part_idx[blockIdx.x] = bi;
      }
    }
    // last-CTA ticket: no CTA ever waits for another
    if (ctid == 0) {
      __threadfence();
      const unsigned ticket = atomicAdd(p.counter, 1u);
      s_last = (ticket == (unsigned)(p.ncta - 1));
    }
    named_barrier(1, nct);
    if (!s_last) return;
    __threadfence();
    if (EPI == kEpiArgmax) {
      if (warp == 0) {
        float v = -INFINITY;
        int vi = 0x7fffffff;
        for (int c = lane; c < p.ncta; c += 32) {
          const float cv = __ldcg(p.part_val + c);
          const int ci = __ldcg(p.part_idx + c);
          if (cv > v || (cv == v && ci < vi)) { v = cv; vi = ci; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, o);
          const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
          if (ov > v || (ov == v && oi < vi)) { v = ov; vi = oi; }
        }
        if (lane == 0) {
          *p.ids_out = vi;
          *p.counter = 0u;
          if (p.len_inc) *p.len_inc += 1;
        }
      }
    } else {
      // router: top-k over the E expert logits (FP32 compare, lowest index on
      // ties), softmax over the selected logits, sigmoid gate of the shared
      // expert's row ("Fourteen hours to 100 tokens per second", "The router
      // with 257 rows").
      __shared__ int s_sel[64];
      __shared__ float s_selv[64];
      const int E = p.n_experts;
      for (int kk = 0; kk < p.top_k; ++kk) {
        float v = -INFINITY;
        int vi = 0x7fffffff;
        for (int e = ctid; e < E; e += nct) {
          bool taken = false;
          for (int q = 0; q < kk; ++q) taken |= (s_sel[q] == e);
          if (taken) continue;
          const float cv = __ldcg(p.router_logits + e);
          if (cv > v || (cv == v && e < vi)) { v = cv; vi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, o);
          const int oi = __shfl_xor_sync(0xffffffffu, vi, o);
          if (ov > v || (ov == v && oi < vi)) { v = ov; vi = oi; }
        }
        if (lane == 0) { s_red[warp] = v; s_redi[warp] = vi; }
        named_barrier(1, nct);
        if (ctid == 0) {
          for (int w = 1; w < kConsumerWarps; ++w)
            if (s_red[w] > v || (s_red[w] == v && s_redi[w] < vi)) { v = s_red[w]; vi = s_redi[w]; }
          s_sel[kk] = vi;
          s_selv[kk] = v;
        }
        named_barrier(1, nct);
      }
      if (ctid == 0) {
        float m = s_selv[0], den = 0.f;
        for (int q = 0; q < p.top_k; ++q) den += __expf(s_selv[q] - m);
        for (int q = 0; q < p.top_k; ++q) {
          p.out_ids[q] = s_sel[q];
          p.out_w[q] = __expf(s_selv[q] - m) / den;
          if (p.dbg_ids) p.dbg_ids[q] = s_sel[q];
        }
        p.out_w[p.top_k] = sigmoidf_(__ldcg(p.router_logits + E));
        *p.counter = 0u;
      }
      if (p.dbg_logits)
        for (int e = ctid; e <= E; e += nct) p.dbg_logits[e] = __ldcg(p.router_logits + e);
    }
  }
}

template <int SRC, int IN, int EPI>
void* pick_vpl(int vpl) {
  switch (vpl) {
    case 1: return (void*)k_gemv<1, SRC, IN, EPI>;
    case 2: return (void*)k_gemv<2, SRC, IN, EPI>;
    case 3: return (void*)k_gemv<3, SRC, IN, EPI>;
    case 4: return (void*)k_gemv<4, SRC, IN, EPI>;
    case 5: return (void*)k_gemv<5, SRC, IN, EPI>;
    case 8: return (void*)k_gemv<8, SRC, IN, EPI>;
    default: return nullptr;
  }
}

void* pick(int src, int in, int epi, int vpl) {
  if (src == kSrcDense && in == kInX && epi == kEpiStore) return pick_vpl<kSrcDense, kInX, kEpiStore>(vpl);
  if (src == kSrcDense && in == kInEmbed && epi == kEpiStore) return pick_vpl<kSrcDense, kInEmbed, kEpiStore>(vpl);
  if (src == kSrcDense && in == kInX && epi == kEpiResid) return pick_vpl<kSrcDense, kInX, kEpiResid>(vpl);
  if (src == kSrcDense && in == kInX && epi == kEpiSwiglu) return pick_vpl<kSrcDense, kInX, kEpiSwiglu>(vpl);
  if (src == kSrcDense && in == kInX && epi == kEpiArgmax) return pick_vpl<kSrcDense, kInX, kEpiArgmax>(vpl);
  if (src == kSrcDense && in == kInX && epi == kEpiRouter) return pick_vpl<kSrcDense, kInX, kEpiRouter>(vpl);
  if (src == kSrcExpertRows && in == kInX && epi == kEpiSwiglu) return pick_vpl<kSrcExpertRows, kInX, kEpiSwiglu>(vpl);
  if (src == kSrcExpertSegs && in == kInMoeZ && epi == kEpiResid) return pick_vpl<kSrcExpertSegs, kInMoeZ, kEpiResid>(vpl);
  return nullptr;
}

const int kCombos[][3] = {
    {kSrcDense, kInX, kEpiStore},   {kSrcDense, kInEmbed, kEpiStore},      {kSrcDense, kInX, kEpiResid},
    {kSrcDense, kInX, kEpiSwiglu},  {kSrcDense, kInX, kEpiArgmax},         {kSrcDense, kInX, kEpiRouter},
    {kSrcExpertRows, kInX, kEpiSwiglu}, {kSrcExpertSegs, kInMoeZ, kEpiResid},
};

}  // namespace

// Opt every instantiation in to the full dynamic shared memory once, so that
// launches (including those recorded into CUDA graphs) need no attribute call.
cudaError_t init() {
  const int vpls[] = {1, 2, 3, 4, 5, 8};
  for (const auto& c : kCombos)
    for (int v : vpls) {
      cudaError_t e = cudaFuncSetAttribute(pick(c[0], c[1], c[2], v), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kMaxSmem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

namespace {
// Tuning overrides (environment, read when a launch is planned).
int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  const int x = atoi(v);
  return x > 0 ? x : dflt;
}
}  // namespace

Plan plan(int R, int C, int npair, int nsm) {
  const int stage_target = env_int("HY_GEMV_STAGE_KB", kStageTarget / 1024) * 1024;
  const int in_flight = env_int("HY_GEMV_INFLIGHT_KB", kInFlight / 1024) * 1024;
  const int ctas_per_sm = env_int("HY_GEMV_CTAS_PER_SM", kCtasPerSm);
  const int nprod = env_int("HY_GEMV_PRODUCERS", kProducers);
  Plan pl = {};
  pl.ok = false;
  if (R <= 0 || C <= 0 || C % 8 != 0) return pl;
  const int nvec = C / 8;
  int nchunk = 1, vpl = 0;
  for (nchunk = 1; nchunk <= 8; nchunk *= 2) {
    const int cv = (nvec + nchunk - 1) / nchunk;
    vpl = (cv + 31) / 32;
    if (vpl <= 8) break;
  }
  if (nchunk > 8) return pl;
  if (vpl == 6 || vpl == 7) vpl = 8;
  const int row_bytes = C * 2 * npair;
  // Smallest column split whose minimum tile (enough row items for all eight
  // compute warps) fits the preferred stage size; a wider split keeps more of
  // the input vector per lane in registers.
  int tr_unit = 1;
  for (int nc = 1; nc <= 8; nc *= 2) {
    const int cv = (nvec + nc - 1) / nc;
    const int v = (cv + 31) / 32;
    if (v > 8) continue;
    const int unit_items = 2 * kConsumerWarps / nc;  // two items per warp per tile
    const int tu = (unit_items + npair - 1) / npair;
    nchunk = nc;
    vpl = v;
    tr_unit = tu;
    if (tu * row_bytes <= kStageCap) break;
  }
  if (vpl < 1 || vpl > 8) return pl;
  if (vpl == 6 || vpl == 7) vpl = 8;
  pl.nchunk = nchunk;
  pl.vpl = vpl;
  pl.chunk_vecs = (nvec + nchunk - 1) / nchunk;
  int tr = (stage_target / row_bytes / tr_unit) * tr_unit;
  if (tr < tr_unit) tr = tr_unit;
  if (tr * row_bytes > 2 * kStageCap) tr = 1;
  pl.tile_rows = tr;
  pl.stage_bytes = ((tr * row_bytes) + 127) & ~127;
  int ns = in_flight / pl.stage_bytes;
  ns = ns < 2 ? 2 : (ns > kMaxStages ? kMaxStages : ns);
  pl.nprod = nprod > ns ? ns : nprod;
  ns = (ns / pl.nprod) * pl.nprod;  // every producer lane owns the same number of stages
  pl.nstages = ns;
  pl.ncta = R < nsm * ctas_per_sm ? R : nsm * ctas_per_sm;
  pl.rows_cta_max = (R + pl.ncta - 1) / pl.ncta;
  pl.xs_floats = (C + 3) & ~3;
  const int red_floats = ((pl.rows_cta_max * npair * nchunk) + 1) & ~1;
  pl.smem = pl.nstages * pl.stage_bytes + 4 * (pl.xs_floats + red_floats) + 2 * kMaxStages * 8;
  pl.ok = pl.smem <= kMaxSmem;
  return pl;
}

cudaError_t launch(const Params& p0, const Plan& pl, int src, int in, int epi, cudaStream_t st, bool pdl) {
  void* k = pick(src, in, epi, pl.vpl);
  if (!k || !pl.ok) return cudaErrorInvalidValue;
  Params p = p0;
  p.ncta = pl.ncta;
  p.tile_rows = pl.tile_rows;
  p.nchunk = pl.nchunk;
  p.chunk_vecs = pl.chunk_vecs;
  p.stage_bytes = pl.stage_bytes;
  p.nstages = pl.nstages;
  p.nprod = pl.nprod;
  p.rows_cta_max = pl.rows_cta_max;
  p.xs_floats = pl.xs_floats;
  p.npair = (epi == kEpiSwiglu) ? 2 : 1;
  return launch_k(reinterpret_cast<void (*)(Params)>(k), dim3(pl.ncta), dim3(kThreads), (size_t)pl.smem, st, pdl, p);
}

}  // namespace gemv
}  // namespace hy

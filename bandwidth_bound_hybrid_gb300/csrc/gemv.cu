// Streaming GEMV for batch-1 decode on sm_103a: y = W * f(x), W bf16 [R][C].
//
// Decode at M = 1 is a matrix-vector product and the weight stream is the
// whole cost ("Beating llama.cpp from Scratch on Consumer AMD", Act 0, pass 3
// and Act 6: weight GEMV kernels take 88.85% of the 4B decode time).  Design:
//   * persistent grid, one CTA per SM, each owning a contiguous row range;
//   * one copy lane streams row tiles HBM -> shared memory with bulk copies on
//     the TMA engine (cp.async.bulk, L2 evict-first), ~180 KB deep, completion
//     on mbarriers; tiles of the next kernel's weights start streaming before
//     griddepcontrol.wait releases the kernel (programmatic dependent launch);
//     an optional L2 prefetch cursor runs ahead of the ring, then covers the
//     first rows the next kernels read;
//   * twelve compute warps hold their slice of the (normalised) input vector
//     in registers, read 16-byte bf16 vectors from shared memory, accumulate
//     in FP32, and reduce with warp shuffles;
//   * fused prologues (RMSNorm, embedding gather, MoE weighted activations) and
//     epilogues (store, residual add, SwiGLU, argmax).
#include <cstdlib>

#include "common.cuh"
#include "gemv_dev.cuh"
#include "kernels.h"

namespace hy {
namespace gemv {

namespace {

template <int VPL, int SRC, int IN, int EPI, bool FULL>
__global__ void __maxnreg__(kMaxRegs) k_gemv(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nst = p.nstages;
  uint8_t* stages = smem;
  float* xs = reinterpret_cast<float*>(smem + nst * p.stage_bytes);
  float* gs = xs + p.xs_floats;
  float* red = gs + p.gs_floats;
  constexpr int npair = (EPI == kEpiSwiglu) ? 2 : 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + ((p.rows_cta_max * npair * p.nchunk + 1) & ~1));
  uint64_t* empty = full + kMaxStages;
  uint64_t* xbar = empty + kMaxStages;
  uint64_t* rbar = xbar + 1;  // expert ids picked (routing in this kernel)
  __shared__ __align__(16) EpiShared esh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (int)((long long)blockIdx.x * p.R / p.ncta);
  const int r1 = (int)((long long)(blockIdx.x + 1) * p.R / p.ncta);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(xbar, 1);
    mbar_init(rbar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kConsumerWarps) {
    // A CTA releases its dependents once every thread has triggered or
    // exited: trigger here too, or the next kernel would launch only when the
    // copy lane retires at the end.
    pdl_launch_dependents();
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint64_t keep = l2_evict_last_policy();  // the input and gain are read by every CTA
      mbar_arrive_expect_tx(xbar, input_bytes(p, IN) + (p.norm_g ? p.C * 4 : 0));
      if (p.norm_g) bulk_g2s(gs, p.norm_g, p.C * 4, xbar, keep);
      // Dense weights do not depend on earlier kernels: pre_stages tiles go out
      // before griddepcontrol.wait; expert ids come from the router kernel.
      const int pre = (SRC == kSrcDense) ? p.pre_stages : 0;
      // q: p, with the expert ids this CTA picked (routing in this kernel)
      Params q = p;
      bool input_issued = false;
      int t = 0, pf = r0;                // pf: first row the L2 prefetch cursor has not covered
      bool next_done = false;
      const int row_bytes = (SRC == kSrcExpertSegs) ? (p.top_k + 1) * p.seg_cols * 2 : p.C * 2 * npair;
      for (int a = r0; a < r1; ++t) {
        if (!input_issued && t >= pre) {
          pdl_wait();
          issue_input(p, IN, xs, esh.mw, xbar, keep);
          input_issued = true;
          if (SRC == kSrcExpertRows && p.route_here) {
            if (!mbar_wait(rbar, 0)) {
              set_guard(p.guard, kGuardWaitTimeout);
              break;
            }
            q.moe_ids = esh.sel;
          }
        }
        const int rows = tile_rows_at(q, SRC, a, r1);
        const int s = t % nst, k = t / nst;
        if (t >= nst && !mbar_wait(&empty[s], (k - 1) & 1)) {
          set_guard(p.guard, kGuardWaitTimeout);
          break;
        }
        issue_tile(q, SRC, npair, a, rows, stages + s * p.stage_bytes, &full[s], pol);
        a += rows;
        if (p.pf_ahead > 0 && t + 1 >= nst && !next_done) {
          // once the ring is full, keep the prefetch cursor pf_ahead bytes
          // beyond what it has issued; past the last row, prefetch what the
          // next kernels read first
          if (pf < a) pf = a;
          while (pf < r1 && (long long)(pf - a) * row_bytes < p.pf_ahead) {
            const int pr = tile_rows_at(q, SRC, pf, r1);
            prefetch_tile(q, SRC, npair, pf, pr);
            pf += pr;
          }
          if (pf >= r1) {
            prefetch_next(p);
            next_done = true;
          }
        }
      }
      if (!input_issued) {  // fewer tiles than pre_stages
        pdl_wait();
        issue_input(p, IN, xs, esh.mw, xbar, keep);
      }
      if (!next_done) prefetch_next(p);
      // Drain: the CTA must not retire while copies it issued are in flight.
      if (!mbar_wait(xbar, 0)) set_guard(p.guard, kGuardWaitTimeout);
      for (int u = (t > nst ? t - nst : 0); u < t; ++u)
        if (!mbar_wait(&full[u % nst], (u / nst) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  if (SRC == kSrcExpertRows && p.route_here && warp == 0) {
    // every CTA picks the experts from the stored router logits (the same
    // result everywhere) and hands the ids to its copy lane; CTA 0 publishes
    // them and the routing weights for the down projection
    // the smallest per-lane list that holds the experts (its sort is the cost)
    auto logit = [&](int e) { return __ldcg(p.router_logits + e); };
    if (p.n_experts <= 128)
      warp_topk<4>(logit, p.n_experts, p.top_k, esh.sel, esh.selv, lane);
    else if (p.n_experts <= 256)
      warp_topk<8>(logit, p.n_experts, p.top_k, esh.sel, esh.selv, lane);
    else
      warp_topk<kMaxExperts / 32>(logit, p.n_experts, p.top_k, esh.sel, esh.selv, lane);
    if (blockIdx.x == 0 && p.dbg_logits)
      for (int e = lane; e <= p.n_experts; e += 32) p.dbg_logits[e] = __ldcg(p.router_logits + e);
    if (lane == 0) {
      if (blockIdx.x == 0) route_weights(p, esh.sel, esh.selv, __ldcg(p.router_logits + p.n_experts));
      mbar_arrive(rbar);
    }
  }
  if (!mbar_wait(xbar, 0) && ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
  const float sc = input_scale(p, IN, xs, esh.mw, esh.red, ctid);
  LaneSlice<VPL> L;
  lane_setup<VPL>(p, SRC, IN, xs, gs, esh.mw, sc, L, warp, lane);
  const int rows_cta = r1 - r0;
  bool abort = false;
  int t = 0;
  for (int a = r0; a < r1; ++t) {
    const int rows = tile_rows_at(p, SRC, a, r1);
    const int s = t % nst, k = t / nst;
    if (!mbar_wait(&full[s], k & 1)) {
      if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
      abort = true;
      break;
    }
    consume_tile<VPL, SRC, npair, FULL>(p, L, stages + s * p.stage_bytes, rows, a - r0, rows_cta, red, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    a += rows;
  }
  named_barrier(1, kCT);
  if (abort) return;
  epilogue(p, EPI, red, r0, rows_cta, esh, ctid);
}

template <int SRC, int IN, int EPI, bool FULL>
void* pick_vpl(int vpl) {
  switch (vpl) {
    case 1: return (void*)k_gemv<1, SRC, IN, EPI, FULL>;
    case 2: return (void*)k_gemv<2, SRC, IN, EPI, FULL>;
    case 3: return (void*)k_gemv<3, SRC, IN, EPI, FULL>;
    case 4: return (void*)k_gemv<4, SRC, IN, EPI, FULL>;
    case 5: return (void*)k_gemv<5, SRC, IN, EPI, FULL>;
    case 6: return (void*)k_gemv<6, SRC, IN, EPI, FULL>;
    case 8: return (void*)k_gemv<8, SRC, IN, EPI, FULL>;
    default: return nullptr;
  }
}

template <int SRC, int IN, int EPI>
void* pick_vpl(int vpl, bool full) {
  return full ? pick_vpl<SRC, IN, EPI, true>(vpl) : pick_vpl<SRC, IN, EPI, false>(vpl);
}

void* pick(int src, int in, int epi, int vpl, bool full) {
  if (src == kSrcDense && in == kInX && epi == kEpiStore) return pick_vpl<kSrcDense, kInX, kEpiStore>(vpl, full);
  if (src == kSrcDense && in == kInEmbed && epi == kEpiStore) return pick_vpl<kSrcDense, kInEmbed, kEpiStore>(vpl, full);
  if (src == kSrcDense && in == kInX && epi == kEpiResid) return pick_vpl<kSrcDense, kInX, kEpiResid>(vpl, full);
  if (src == kSrcDense && in == kInX && epi == kEpiSwiglu) return pick_vpl<kSrcDense, kInX, kEpiSwiglu>(vpl, full);
  if (src == kSrcDense && in == kInX && epi == kEpiArgmax) return pick_vpl<kSrcDense, kInX, kEpiArgmax>(vpl, full);
  if (src == kSrcExpertRows && in == kInX && epi == kEpiSwiglu) return pick_vpl<kSrcExpertRows, kInX, kEpiSwiglu>(vpl, full);
  if (src == kSrcExpertSegs && in == kInMoeZ && epi == kEpiResid) return pick_vpl<kSrcExpertSegs, kInMoeZ, kEpiResid>(vpl, full);
  return nullptr;
}

const int kCombos[][3] = {
    {kSrcDense, kInX, kEpiStore},   {kSrcDense, kInEmbed, kEpiStore},      {kSrcDense, kInX, kEpiResid},
    {kSrcDense, kInX, kEpiSwiglu},  {kSrcDense, kInX, kEpiArgmax},
    {kSrcExpertRows, kInX, kEpiSwiglu}, {kSrcExpertSegs, kInMoeZ, kEpiResid},
};

}  // namespace

// Opt every instantiation in to the full dynamic shared memory once, so that
// launches (including those recorded into CUDA graphs) need no attribute call.
cudaError_t init() {
  const int vpls[] = {1, 2, 3, 4, 5, 6, 8};
  for (const auto& c : kCombos)
    for (int v : vpls)
      for (int f = 0; f < 2; ++f) {
        cudaError_t e = cudaFuncSetAttribute(pick(c[0], c[1], c[2], v, f != 0),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
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

Plan plan(int R, int C, int npair, int nsm, bool norm) {
  const int stage_target = env_int("HY_GEMV_STAGE_KB", kStageTarget / 1024) * 1024;
  const int in_flight = env_int("HY_GEMV_INFLIGHT_KB", kInFlight / 1024) * 1024;
  const int ctas_per_sm = env_int("HY_GEMV_CTAS_PER_SM", kCtasPerSm);
  Plan pl = {};
  pl.ok = false;
  if (R <= 0 || C <= 0 || C % 8 != 0) return pl;
  const int nvec = C / 8;
  const int row_bytes = C * 2 * npair;
  // Column split nc (a divisor of the compute-warp count, so every warp has a
  // chunk and a row group): fewest lanes idle on a ragged last vector, then at
  // least two row items per warp per tile, then the fewest chunks.
  double best = 1e30;
  int tr_unit = 1;
  for (int nc = 1; nc <= kConsumerWarps; ++nc) {
    if (kConsumerWarps % nc) continue;
    const int cv = (nvec + nc - 1) / nc;
    int v = (cv + 31) / 32;
    if (v > 8) continue;
    if (v == 7) v = 8;
    const int nrg = kConsumerWarps / nc;
    int tu = (2 * nrg + npair - 1) / npair;        // rows for two items per warp
    if (tu * row_bytes > kStageCap) tu = (nrg + npair - 1) / npair;
    const int ipw = (tu * npair) / nrg;
    const double waste = 1.0 - (double)cv / (32.0 * v);
    // VPL above 5 does not fit the register cap without spills
    const double score = waste + 0.5 * (ipw < 2) + 0.001 * nc + (tu * row_bytes > kStageCap ? 1.0 : 0.0) + (v > 5 ? 0.2 : 0.0);
    if (score < best) {
      best = score;
      pl.nchunk = nc;
      pl.vpl = v;
      tr_unit = tu;
    }
  }
  if (pl.vpl < 1) return pl;
  pl.chunk_vecs = (nvec + pl.nchunk - 1) / pl.nchunk;
  pl.full = (pl.chunk_vecs == 32 * pl.vpl) && (pl.nchunk * pl.chunk_vecs == nvec);
  int tr = (stage_target / row_bytes / tr_unit) * tr_unit;
  if (tr < tr_unit) tr = tr_unit;
  if (tr * row_bytes > 2 * kStageCap) tr = 1;
  pl.tile_rows = tr;
  pl.stage_bytes = ((tr * row_bytes) + 127) & ~127;
  int ns = in_flight / pl.stage_bytes;
  ns = ns < 2 ? 2 : (ns > kMaxStages ? kMaxStages : ns);
  pl.nstages = ns;
  pl.ncta = R < nsm * ctas_per_sm ? R : nsm * ctas_per_sm;
  pl.rows_cta_max = (R + pl.ncta - 1) / pl.ncta;
  pl.xs_floats = (C + 3) & ~3;
  pl.gs_floats = norm ? pl.xs_floats : 0;
  pl.pre_stages = env_int("HY_GEMV_PRE_STAGES", kPreStages);
  const char* ps0 = getenv("HY_GEMV_PRE_STAGES");
  if (ps0 && *ps0 == '0') pl.pre_stages = 0;
  pl.pf_ahead = env_int("HY_GEMV_PREFETCH_KB", kPrefetchAhead / 1024) * 1024;
  const char* pf0 = getenv("HY_GEMV_PREFETCH_KB");
  if (pf0 && *pf0 == '0') pl.pf_ahead = 0;
  const int red_floats = ((pl.rows_cta_max * npair * pl.nchunk) + 1) & ~1;
  pl.smem = pl.nstages * pl.stage_bytes + 4 * (pl.xs_floats + pl.gs_floats + red_floats) + (2 * kMaxStages + 2) * 8;
  while (pl.smem > kMaxSmem && pl.nstages > 2) {
    pl.nstages -= 1;
    pl.smem -= pl.stage_bytes;
  }
  pl.ok = pl.smem <= kMaxSmem;
  return pl;
}

cudaError_t launch(const Params& p0, const Plan& pl, int src, int in, int epi, cudaStream_t st, bool pdl) {
  void* k = pick(src, in, epi, pl.vpl, pl.full);
  if (!k || !pl.ok) return cudaErrorInvalidValue;
  Params p = p0;
  p.ncta = pl.ncta;
  p.tile_rows = pl.tile_rows;
  p.nchunk = pl.nchunk;
  p.chunk_vecs = pl.chunk_vecs;
  p.stage_bytes = pl.stage_bytes;
  p.nstages = pl.nstages;
  p.pf_ahead = pl.pf_ahead;
  p.rows_cta_max = pl.rows_cta_max;
  p.xs_floats = pl.xs_floats;
  p.gs_floats = pl.gs_floats;
  p.pre_stages = pl.pre_stages;
  p.npair = (epi == kEpiSwiglu) ? 2 : 1;
  return launch_k(reinterpret_cast<void (*)(Params)>(k), dim3(pl.ncta), dim3(kThreads), (size_t)pl.smem, st, pdl, p);
}

}  // namespace gemv
}  // namespace hy

// The decode step as one persistent cooperative kernel on sm_103a.
//
// One CTA per SM runs the step's kernels (GEMVs, Gated DeltaNet step, split-KV
// attention; the same device code as their standalone kernels) as phases of a
// program held in device memory.  Phases are separated by a grid barrier: a
// CTA's compute warps arrive once they have finished a phase and wait until
// every CTA has arrived before they load the next phase's input.  The copy
// lane does not wait: weight and KV-cache tiles do not depend on the
// activations, so it keeps streaming the next phases' tiles into the ring as
// slots free up, and only the routed experts' tiles wait for the phase that
// picked them.  HBM stays busy across the barriers and no kernel launch, CTA
// start or grid drain separates the phases ("Beating llama.cpp from Scratch
// on Consumer AMD", Act 1: the decode step is a chain of small dependent
// kernels whose launch and drain costs add up; here the chain is one launch).
#include "attn_dev.cuh"
#include "common.cuh"
#include "gdn_dev.cuh"
#include "gemv_dev.cuh"
#include "kernels.h"

namespace hy {
namespace step {
namespace {

constexpr int kCT = kNW * 32;  // compute threads
static_assert(sizeof(Phase) % 16 == 0, "phase descriptors are bulk-copied");
constexpr int kGdnWarps = 8;   // a DeltaNet item: 16 state rows, 2 per warp
static_assert(gemv::kCT == kCT, "one set of compute warps");
static_assert(attn::kCWarps <= kNW && kGdnWarps <= kNW, "phase work fits the compute warps");

__device__ __forceinline__ void bar_arrive(unsigned* bar) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait until every CTA arrived `target` times in total.
__device__ __forceinline__ bool bar_wait(const unsigned* bar, unsigned target) {
  if (ld_acquire(bar) >= target) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire(bar) >= target) return true;
    if ((i & 255u) == 0) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitLimitNs) return false;
    }
  }
}

struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int nst, stage_bytes;
  __device__ __forceinline__ uint8_t* stage(uint32_t t) const { return base + (t % nst) * stage_bytes; }
};

// ------------------------------------------------------------ copy lane work

// Rows of CTA b in a GEMV phase.
__device__ __forceinline__ void gemv_rows(const gemv::Params& p, int b, int& r0, int& r1) {
  r0 = (int)((long long)b * p.R / p.ncta);
  r1 = (int)((long long)(b + 1) * p.R / p.ncta);
}

// L2 prefetch of the DeltaNet state rows CTA b updates in phase `ph` (the
// compute warps load them with plain loads).
__device__ __forceinline__ void prefetch_phase(const Phase& ph, int b) {
  if (ph.pf_bytes <= 0) return;
  if (ph.kind == kGdn) {
    const gdn::Params& d = ph.d;
    const int nrc = (d.dv + gdn::kRowsPerCta - 1) / gdn::kRowsPerCta;
    if (b >= d.nh * nrc) return;
    const int h = b % d.nh, rc = b / d.nh;
    const int rows = min(gdn::kRowsPerCta, d.dv - rc * gdn::kRowsPerCta);
    bulk_prefetch_l2(d.S + ((long long)h * d.dv + rc * gdn::kRowsPerCta) * d.dk, (uint32_t)rows * d.dk * 4);
  }
}

// ------------------------------------------------------------ compute work

// A phase descriptor into shared memory (all compute threads).
__device__ __forceinline__ void load_phase(const Program& pr, int i, Phase* dst, int ctid) {
  const uint4* src = reinterpret_cast<const uint4*>(pr.phases + i);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int k = ctid; k < (int)(sizeof(Phase) / 16); k += kCT) d[k] = __ldg(src + k);
}

// A GEMV phase's input vector (FP32, or the bf16 embedding row), the MoE
// routing weights and the RMSNorm gain into shared memory, with plain loads
// (not bulk copies, which would queue behind the tiles the copy lane already
// requested); what earlier phases wrote is read past L1.
__device__ __forceinline__ void load_input(const gemv::Params& p, int in, float* xs, float* gs, float* mw, int ctid) {
  if (in == gemv::kInEmbed) {
    int tok = __ldcg(p.tok);
    if (tok < 0 || tok >= p.vocab) {  // never read outside the embedding table
      if (ctid == 0) set_guard(p.guard, kGuardBadIndex);
      tok = 0;
    }
    const uint4* src = reinterpret_cast<const uint4*>(p.embed + (long long)tok * p.C);
    for (int v = ctid; v < p.C / 8; v += kCT) reinterpret_cast<uint4*>(xs)[v] = __ldg(src + v);
  } else {
    const float4* src = reinterpret_cast<const float4*>(p.x);
    for (int v = ctid; v < p.C / 4; v += kCT) reinterpret_cast<float4*>(xs)[v] = __ldcg(src + v);
    if (in == gemv::kInMoeZ)
      for (int k = ctid; k <= p.top_k; k += kCT) mw[k] = __ldcg(p.moe_w + k);
  }
  if (p.norm_g)
    for (int v = ctid; v < p.C / 4; v += kCT)
      reinterpret_cast<float4*>(gs)[v] = __ldg(reinterpret_cast<const float4*>(p.norm_g) + v);
  named_barrier(1, kCT);
}

// A wait that gives up sets *abort (shared); the CTA then skips the rest of
// the step but still passes every block barrier and grid arrival, so nothing
// waits forever.
template <int VPL, int SRC, int NPAIR>
__device__ __forceinline__ void gemv_tiles(const gemv::Params& p, const gemv::LaneSlice<VPL>& L, const Ring& rg,
                                           uint32_t& t, int r0, int r1, float* red, int lane, bool& ok,
                                           volatile int* abort) {
  const int rows_cta = r1 - r0;
  for (int a = r0; a < r1;) {
    const int rows = gemv::tile_rows_at(p, SRC, a, r1);
    const uint32_t s = t % rg.nst, k = t / rg.nst;
    if (ok && !mbar_wait(&rg.full[s], k & 1)) {
      if (lane == 0) set_guard(p.guard, kGuardWaitTimeout);
      ok = false;
      *abort = 1;
    }
    if (ok) gemv::consume_tile<VPL, SRC, NPAIR, true>(p, L, rg.stage(t), rows, a - r0, rows_cta, red, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&rg.empty[s]);
    a += rows;
    ++t;
  }
}

template <int VPL>
__device__ __forceinline__ void gemv_phase(const Phase& ph, const Ring& rg, uint32_t& t, uint8_t* region,
                                           gemv::EpiShared& esh, float* scratch, int ctid, bool& ok,
                                           volatile int* abort) {
  const gemv::Params& p = ph.g;
  const int warp = ctid >> 5, lane = ctid & 31;
  int r0, r1;
  gemv_rows(p, blockIdx.x, r0, r1);
  float* xs = reinterpret_cast<float*>(region);
  float* gs = xs + p.xs_floats;
  float* red = gs + p.gs_floats;
  load_input(p, ph.in, xs, gs, esh.mw, ctid);
  const float sc = gemv::input_scale(p, ph.in, xs, esh.mw, esh.red, ctid);
  gemv::LaneSlice<VPL> L;
  gemv::lane_setup<VPL>(p, ph.src, ph.in, xs, gs, esh.mw, sc, L, warp, lane);
  if (ph.src == gemv::kSrcDense) {
    if (ph.epi == gemv::kEpiSwiglu) gemv_tiles<VPL, gemv::kSrcDense, 2>(p, L, rg, t, r0, r1, red, lane, ok, abort);
    else gemv_tiles<VPL, gemv::kSrcDense, 1>(p, L, rg, t, r0, r1, red, lane, ok, abort);
  } else if (ph.src == gemv::kSrcExpertRows) {
    gemv_tiles<VPL, gemv::kSrcExpertRows, 2>(p, L, rg, t, r0, r1, red, lane, ok, abort);
  } else {
    gemv_tiles<VPL, gemv::kSrcExpertSegs, 1>(p, L, rg, t, r0, r1, red, lane, ok, abort);
  }
  // the copy lane may set *abort at any time: decide once, for all compute threads
  if (!named_barrier_or(1, kCT, *abort != 0)) gemv::epilogue(p, ph.epi, red, r0, r1 - r0, esh, scratch, ctid);
}

// A DeltaNet phase: items blockIdx.x, + gridDim.x, ...  The first item's
// state rows and conv taps (R, V) were loaded before the grid barrier: no
// earlier phase of the step writes them.
template <int EPL>
__device__ __forceinline__ void gdn_phase(const Phase& ph, uint8_t* region, int ctid, gdn::Rows<EPL, kGdnWarps>& R,
                                          gdn::ConvRegs<EPL, kGdnWarps>& V) {
  const gdn::Params& d = ph.d;
  const int nrc = (d.dv + gdn::kRowsPerCta - 1) / gdn::kRowsPerCta;
  auto& sh = *reinterpret_cast<gdn::ItemShared<EPL>*>(region);
  for (int b = blockIdx.x; b < d.nh * nrc; b += gridDim.x) {
    const int h = b % d.nh, rc = b / d.nh;
    if (b != (int)blockIdx.x) {
      gdn::load_rows<EPL, kGdnWarps>(d, h, rc, R, ctid);
      gdn::load_conv<EPL, kGdnWarps>(d, h, rc, V, ctid);
    }
    gdn::run_item<EPL, kGdnWarps>(d, h, rc, R, V, sh, ctid, [] __device__() { named_barrier(1, kGdnWarps * 32); });
  }
}

template <int HD, int G>
__device__ __forceinline__ void attn_phase(const Phase& ph, const Ring& rg, uint32_t& t, uint8_t* region,
                                           float* scratch, int ctid, bool& ok, volatile int* abort) {
  const attn::Params& p = ph.a;
  const int T = *p.len;
  for (int b = blockIdx.x; b < p.nkv * p.nsplit; b += gridDim.x) {
    const int g = b / p.nsplit, sp = b % p.nsplit;
    const attn::Item it = attn::item_of<HD>(p, T, sp);
    attn::WorkPtrs<HD, G> w;
    w.carve(region);
    attn::Acc<HD, G> A;
    attn::begin_item<HD, G>(p, g, T, it, w, A, ctid);
    for (int tt = 0; tt < it.ntiles; ++tt) {
      const uint32_t s = t % rg.nst, k = t / rg.nst;
      if (ok && !mbar_wait(&rg.full[s], k & 1)) {
        if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
        ok = false;
        *abort = 1;
      }
      // always run the tile (its block barriers must match across threads);
      // after a failed wait it reads stale, in-bounds shared memory
      const uint8_t* st = rg.stage(t);
      attn::process_tile<HD, G>(reinterpret_cast<const uint16_t*>(st),
                                reinterpret_cast<const uint16_t*>(st + attn::Tile<HD>::kBytesKV),
                                attn::tile_rows<HD>(it, tt), w, A, ctid);
      if (ctid == 0) mbar_arrive_cnt(&rg.empty[s], kNW);  // the stage's arrival count is kNW
      ++t;
    }
    if (it.has_new) attn::process_tile<HD, G>(w.kn, w.vn, 1, w, A, ctid);
    attn::end_item<HD, G>(p, g, sp, w, A, scratch, ctid);
  }
}

// Tiles of an attention phase this CTA streams (all compute warps count them).
template <int HD>
__device__ __forceinline__ int attn_tiles(const attn::Params& p) {
  const int T = *p.len;
  int n = 0;
  for (int b = blockIdx.x; b < p.nkv * p.nsplit; b += gridDim.x) n += attn::item_of<HD>(p, T, b % p.nsplit).ntiles;
  return n;
}

template <int HD, int G, int EPL>
__global__ void __maxnreg__(128) k_step(const Program pr) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(16) gemv::EpiShared esh;
  __shared__ volatile int s_abort;
  const int nst = pr.nstages;
  Ring rg;
  rg.base = smem;
  rg.nst = nst;
  rg.stage_bytes = pr.stage_bytes;
  uint8_t* region = smem + (size_t)nst * pr.stage_bytes;
  float* scratch = reinterpret_cast<float*>(region + pr.region_bytes);
  Phase* pbuf = reinterpret_cast<Phase*>(scratch + ((pr.scratch_floats + 3) & ~3));
  uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + 2);
  rg.full = bars;
  rg.empty = bars + kMaxStagesStep;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned nctas = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&rg.full[s], 1);
      mbar_init(&rg.empty[s], kNW);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kNW) {
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    uint32_t t = 0;
    bool ok = true;
    for (int ph_i = 0; ph_i < pr.nphases && ok; ++ph_i) {
      // read from global memory: this lane runs ahead of the compute warps'
      // descriptor copies
      const Phase& ph = pr.phases[ph_i];
      if (ph.after > 0) {  // tiles whose addresses an earlier phase decides
        if (!bar_wait(pr.bar, (unsigned)ph.after * nctas)) {
          set_guard(pr.guard, kGuardWaitTimeout);
          ok = false;
          s_abort = 1;
          break;
        }
      }
      if (s_abort) break;
      if (ph.kind == kGemv && (int)blockIdx.x < ph.g.ncta) {
        const gemv::Params& p = ph.g;
        const int npair = ph.epi == gemv::kEpiSwiglu ? 2 : 1;
        int r0, r1;
        gemv_rows(p, blockIdx.x, r0, r1);
        for (int a = r0; a < r1 && ok;) {
          const int rows = gemv::tile_rows_at(p, ph.src, a, r1);
          const uint32_t s = t % nst, k = t / nst;
          if (t >= (uint32_t)nst && !mbar_wait(&rg.empty[s], (k - 1) & 1)) {
            set_guard(pr.guard, kGuardWaitTimeout);
            ok = false;
            s_abort = 1;
            break;
          }
          gemv::issue_tile(p, ph.src, npair, a, rows, rg.stage(t), &rg.full[s], pol);
          a += rows;
          ++t;
        }
      } else if (ph.kind == kAttn) {
        const attn::Params& p = ph.a;
        const int T = *p.len;
        for (int b = blockIdx.x; b < p.nkv * p.nsplit && ok; b += gridDim.x) {
          const int g = b / p.nsplit;
          const attn::Item it = attn::item_of<HD>(p, T, b % p.nsplit);
          for (int tt = 0; tt < it.ntiles; ++tt) {
            const uint32_t s = t % nst, k = t / nst;
            if (t >= (uint32_t)nst && !mbar_wait(&rg.empty[s], (k - 1) & 1)) {
              set_guard(pr.guard, kGuardWaitTimeout);
              ok = false;
              s_abort = 1;
              break;
            }
            attn::issue_tile<HD>(p, g, it, tt, rg.stage(t), &rg.full[s], pol);
            ++t;
          }
        }
      } else if (ph.kind == kGdn) {
        prefetch_phase(ph, blockIdx.x);
      }
    }
    // Drain: the CTA must not retire while copies it issued are in flight.
    for (uint32_t u = (t > (uint32_t)nst ? t - nst : 0); u < t; ++u)
      if (!mbar_wait(&rg.full[u % nst], (u / nst) & 1)) set_guard(pr.guard, kGuardWaitTimeout);
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int ctid = threadIdx.x;
  uint32_t t = 0;
  load_phase(pr, 0, &pbuf[0], ctid);
  for (int ph_i = 0; ph_i < pr.nphases; ++ph_i) {
    named_barrier(2, kCT);  // descriptor ph_i is in shared memory
    gdn::Rows<EPL, kGdnWarps> R;
    gdn::ConvRegs<EPL, kGdnWarps> V;
    {
      // work that no earlier phase feeds, done while the others finish
      const Phase& ph = pbuf[ph_i & 1];
      if (ph.kind == kGdn && warp < kGdnWarps) {
        const gdn::Params& d = ph.d;
        const int b = blockIdx.x, nrc = (d.dv + gdn::kRowsPerCta - 1) / gdn::kRowsPerCta;
        if (b < d.nh * nrc && !s_abort) {
          gdn::load_rows<EPL, kGdnWarps>(d, b % d.nh, b / d.nh, R, ctid);
          gdn::load_conv<EPL, kGdnWarps>(d, b % d.nh, b / d.nh, V, ctid);
        }
      }
    }
    // the previous phase must be complete on every CTA
    bool failed = false;
    if (ph_i > 0 && ctid == 0 && !s_abort && !bar_wait(pr.bar, (unsigned)ph_i * nctas)) {
      set_guard(pr.guard, kGuardWaitTimeout);
      failed = true;
    }
    // every compute thread takes the same skip decision
    bool ok = !named_barrier_or(2, kCT, failed || s_abort != 0);
    const Phase& ph = pbuf[ph_i & 1];
    if (ok) {
      if (ph.kind == kGemv) {
        if ((int)blockIdx.x < ph.g.ncta) {
          switch (ph.vpl) {
            case 1: gemv_phase<1>(ph, rg, t, region, esh, scratch, ctid, ok, &s_abort); break;
            case 2: gemv_phase<2>(ph, rg, t, region, esh, scratch, ctid, ok, &s_abort); break;
            case 3: gemv_phase<3>(ph, rg, t, region, esh, scratch, ctid, ok, &s_abort); break;
            case 4: gemv_phase<4>(ph, rg, t, region, esh, scratch, ctid, ok, &s_abort); break;
            default: gemv_phase<5>(ph, rg, t, region, esh, scratch, ctid, ok, &s_abort); break;
          }
        }
      } else if (ph.kind == kGdn) {
        if (warp < kGdnWarps) gdn_phase<EPL>(ph, region, ctid, R, V);
      } else if (ph.kind == kCopy) {
        for (int i = blockIdx.x * kCT + ctid; i < ph.cn; i += gridDim.x * kCT) ph.cdst[i] = ph.csrc[i];
      } else {
        if (warp < attn::kCWarps) attn_phase<HD, G>(ph, rg, t, region, scratch, ctid, ok, &s_abort);
        else t += attn_tiles<HD>(ph.a);
      }
      if (!ok) s_abort = 1;
    }
    named_barrier(2, kCT);  // the CTA's part of the phase is done
    if (ctid == 0) {
      if (ph_i + 1 < pr.nphases) {
        bar_arrive(pr.bar);
      } else {
        // last arrival of the step resets the counter (nobody waits on it)
        const unsigned old = atomicAdd(pr.bar, 1u);
        if (old == (unsigned)pr.nphases * nctas - 1) atomicExch(pr.bar, 0u);
      }
    }
    // the next descriptor goes where the previous phase's was
    if (ph_i + 1 < pr.nphases) load_phase(pr, ph_i + 1, &pbuf[(ph_i + 1) & 1], ctid);
  }
}

template <int HD, int G, int EPL>
void* kern() {
  return (void*)k_step<HD, G, EPL>;
}

void* pick(int hd, int G, int epl) {
  if (hd == 64 && G == 2 && epl == 2) return kern<64, 2, 2>();
  if (hd == 128 && G == 4 && epl == 4) return kern<128, 4, 4>();
  if (hd == 256 && G == 8 && epl == 4) return kern<256, 8, 4>();
  return nullptr;
}

}  // namespace

bool supported(int hd, int G, int epl) { return pick(hd, G, epl) != nullptr; }

size_t attn_work_bytes(int hd, int G) {
#define HY_W(H_, G_) \
  if (hd == H_ && G == G_) return attn::Work<H_, G_>::total;
  HY_W(64, 2) HY_W(128, 4) HY_W(256, 8)
#undef HY_W
  return 0;
}

size_t gdn_work_bytes(int epl) {
  if (epl == 2) return sizeof(gdn::ItemShared<2>);
  if (epl == 4) return sizeof(gdn::ItemShared<4>);
  return 0;
}

int attn_stage_bytes(int hd) {
  if (hd == 64) return attn::Tile<64>::kStageBytes;
  if (hd == 128) return attn::Tile<128>::kStageBytes;
  return attn::Tile<256>::kStageBytes;
}

size_t smem_bytes(const Program& pr) {
  const size_t b = (size_t)pr.nstages * pr.stage_bytes + (((size_t)pr.region_bytes + 15) & ~(size_t)15) +
                   (size_t)((pr.scratch_floats + 3) & ~3) * 4 + 2 * sizeof(Phase) + 2 * kMaxStagesStep * 8;
  return b <= (size_t)kMaxSmem ? b : 0;
}

cudaError_t init() {
  const int cfg[][3] = {{64, 2, 2}, {128, 4, 4}, {256, 8, 4}};
  for (const auto& c : cfg) {
    cudaError_t e = cudaFuncSetAttribute(pick(c[0], c[1], c[2]), cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int blocks_per_sm(const Program& pr) {
  void* k = pick(pr.hd, pr.G, pr.epl);
  const size_t smem = smem_bytes(pr);
  if (!k || !smem) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch(const Program& pr, int nctas, cudaStream_t st) {
  void* k = pick(pr.hd, pr.G, pr.epl);
  const size_t smem = smem_bytes(pr);
  if (!k || !smem || pr.nstages > kMaxStagesStep) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reinterpret_cast<void (*)(Program)>(k), pr);
}

}  // namespace step
}  // namespace hy

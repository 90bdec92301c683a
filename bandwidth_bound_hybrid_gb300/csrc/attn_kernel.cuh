// The split-KV decode attention kernel template (device code in
// attn_dev.cuh), instantiated by attn.cu (one CTA per SM) and attn_pair.cu
// (two CTAs per SM).
#pragma once

#include "attn_dev.cuh"
#include "common.cuh"
#include "kernels.h"

namespace hy {
namespace attn {
namespace {

// PAIR: two CTAs share an SM (more warps to hide shared-memory and shuffle
// latency, for grids of more CTAs than SMs): a 5-stage ring and at most 112
// registers a thread, which only up to 4 query heads per kv head fit.
// Otherwise one CTA an SM with a 6-stage ring.
template <int HD, int G, bool PAIR = false>
struct Smem {
  static_assert(!PAIR || G <= 4, "a CTA pair per SM needs G <= 4");
  static constexpr int ring = PAIR ? kRing - 1 : kRing;
  static constexpr int min_blocks = PAIR ? 2 : 1;
  static constexpr size_t stages = (size_t)ring * Tile<HD>::kBytes;
  static constexpr size_t work = Work<HD, G>::total;
  static constexpr size_t bars = 2 * ring * 8;
  static constexpr size_t total = stages + ((work + 15) & ~(size_t)15) + bars + 64;
};

template <int HD, int G, bool KV8, bool PAIR>
__global__ void __launch_bounds__(kThreads, Smem<HD, G, PAIR>::min_blocks) k_attn(const Params p0) {
  Params p = p0;
  int sp = blockIdx.y;
  if (p0.nb > 0) {  // token blockIdx.z of a batch (or of grid row y, spread): its sequence's cache and scratch
    int z = blockIdx.z;
    if (p0.spread > 0) {
      z = spread_row(p0, blockIdx.y, &sp, &p.nsplit);
      if (p.mergers > p.nsplit) p.mergers = p.nsplit;
    }
    p.y = p0.y + (long long)z * p0.ld_y;
    p.o = p0.o + (long long)z * p0.ld_o;
    p.part = p0.part + (long long)z * p0.ld_part;
    p.counter = p0.counter + z * p0.nkv;
    p.K = p0.K_b[z];
    p.V = p0.V_b[z];
    p.Ks = p0.Ks_b[z];
    p.Vs = p0.Vs_b[z];
    p.len = p0.len_b[z];
    p.cap = p0.cap_b[z];
    p.cap_s = p0.cap_s_b[z];
    p.pages = p0.pages_b[z];
  }
  using S_ = Smem<HD, G, PAIR>;
  constexpr int R_ = S_::ring;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  WorkPtrs<HD, G> w;
  w.carve(smem + S_::stages);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S_::stages + ((S_::work + 15) & ~(size_t)15));
  uint64_t* empty = full + R_;

  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = *p.len;  // written only by the previous step's last kernel
  if (T < 0 || T >= p.cap) {  // the host checks capacity first; never touch memory past it
    if (threadIdx.x == 0) set_guard(p.guard, kGuardBadPosition);
    return;
  }
  const Item it = item_of<HD>(p, T, sp);

  if (threadIdx.x == 0) {
    for (int s = 0; s < R_; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);  // one arrival per compute warp
    }
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ copy lane
  if (warp == kCWarps) {
    pdl_launch_dependents();  // the CTA's trigger needs every thread (or its exit)
    if (lane == 0) {
      // issue order = consumption order: per chunk its K tiles, then its V tiles
      const uint64_t pol = l2_evict_first_policy();
      constexpr int CH = Tile<HD>::CH;
      int q = 0;
      bool ok = true;
      for (int t0 = 0; ok && t0 < it.ntiles; t0 += CH) {
        const int t1 = (t0 + CH < it.ntiles) ? t0 + CH : it.ntiles;
        for (int kv = 0; ok && kv < 2; ++kv)
          for (int t = t0; t < t1; ++t, ++q) {
            const int s = q % R_;
            if (q >= R_ && !mbar_wait(&empty[s], ((q / R_) - 1) & 1)) {
              set_guard(p.guard, kGuardWaitTimeout);
              ok = false;
              break;
            }
            issue_tile<HD, KV8>(p, g, it, t, kv, stages + s * Tile<HD>::kBytes, &full[s], pol);
          }
      }
      for (int u = (q > R_ ? q - R_ : 0); u < q; ++u)
        if (!mbar_wait(&full[u % R_], (u / R_) & 1)) set_guard(p.guard, kGuardWaitTimeout);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  // Per chunk: scores of its K tiles (each warp releases a tile as it is
  // done), one softmax pass, then P V over its V tiles.  The new row (held in
  // shared memory) is the last row of the last chunk.
  const int ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  Acc<HD, G> A;
  begin_item<HD, G, KV8>(p, g, T, it, w, A, ctid);
  constexpr int TP = Tile<HD>::TP, CH = Tile<HD>::CH;
  const int nchunks = it.ntiles > 0 ? (it.ntiles + CH - 1) / CH : 1;
  int q = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int t0 = c * CH, t1 = (t0 + CH < it.ntiles) ? t0 + CH : it.ntiles;
    const bool last = (c == nchunks - 1);
    int rows_c = 0;
    for (int t = t0; t < t1; ++t, ++q) {
      const int s = q % R_;
      if (!mbar_wait(&full[s], (q / R_) & 1)) {
        if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
        return;
      }
      const uint8_t* st = stages + s * Tile<HD>::kBytes;
      const int rows = tile_rows<HD>(it, t);
      const float* ks = KV8 ? reinterpret_cast<const float*>(st + scale_off<HD>()) + ((it.p0 + t * TP) & 3) : nullptr;
      tile_scores<HD, G, KV8>(reinterpret_cast<const uint16_t*>(st), rows, rows_c, w, A, ctid, ks);
      rows_c += rows;
      __syncwarp();
      if ((ctid & 31) == 0) mbar_arrive(&empty[s]);
    }
    const bool with_new = last && it.has_new;
    if (with_new) tile_scores<HD, G, KV8>(w.kn, 1, rows_c, w, A, ctid, w.kvs);
    named_barrier(1, kCT);
    chunk_softmax<HD, G>(rows_c + (with_new ? 1 : 0), w, A, ctid);
    int rb = 0;
    for (int t = t0; t < t1; ++t, ++q) {
      const int s = q % R_;
      if (!mbar_wait(&full[s], (q / R_) & 1)) {
        if (ctid == 0) set_guard(p.guard, kGuardWaitTimeout);
        return;
      }
      const uint8_t* st = stages + s * Tile<HD>::kBytes;
      const int rows = tile_rows<HD>(it, t);
      const float* vs = KV8 ? reinterpret_cast<const float*>(st + scale_off<HD>()) + ((it.p0 + t * TP) & 3) : nullptr;
      tile_pv<HD, G, KV8>(reinterpret_cast<const uint16_t*>(st), rows, rb, w, A, ctid, vs);
      rb += rows;
      __syncwarp();
      if ((ctid & 31) == 0) mbar_arrive(&empty[s]);
    }
    if (with_new) tile_pv<HD, G, KV8>(w.vn, 1, rows_c, w, A, ctid, w.kvs + 1);
    if (!last) named_barrier(1, kCT);  // the next chunk's scores overwrite w.sc
  }
  end_item<HD, G>(p, g, sp, w, A, ctid);
}

}  // namespace

// attn_pair.cu: the CTA-pair instantiations (G <= 4; nullptr otherwise).
void* pick_pair(int hd, int G, size_t* smem, bool kv8);
cudaError_t init_pair();

}  // namespace attn
}  // namespace hy

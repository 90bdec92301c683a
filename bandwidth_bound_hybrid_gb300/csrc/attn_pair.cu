// The CTA-pair instantiations of the decode attention kernel (two CTAs per
// SM, up to 4 query heads per kv head), used for grids of more CTAs than SMs.
#include "attn_kernel.cuh"

namespace hy {
namespace attn {
namespace {

template <int HD, int G>
void* kern_pair(bool kv8) {
  return kv8 ? (void*)k_attn<HD, G, true, true> : (void*)k_attn<HD, G, false, true>;
}

}  // namespace

void* pick_pair(int hd, int G, size_t* smem, bool kv8) {
#define HY_ATTN_PAIR(H_, G_)                 \
  if (hd == H_ && G == G_) {                 \
    *smem = Smem<H_, G_, true>::total;       \
    return kern_pair<H_, G_>(kv8);           \
  }
  HY_ATTN_PAIR(64, 1) HY_ATTN_PAIR(64, 2) HY_ATTN_PAIR(64, 4)
  HY_ATTN_PAIR(128, 1) HY_ATTN_PAIR(128, 2) HY_ATTN_PAIR(128, 4)
  HY_ATTN_PAIR(256, 1) HY_ATTN_PAIR(256, 2) HY_ATTN_PAIR(256, 4)
#undef HY_ATTN_PAIR
  return nullptr;
}

cudaError_t init_pair() {
  const int hds[] = {64, 128, 256};
  const int gs[] = {1, 2, 4};
  for (int h : hds)
    for (int gg : gs)
      for (int kv8 = 0; kv8 < 2; ++kv8) {
        size_t smem = 0;
        void* k = pick_pair(h, gg, &smem, kv8 != 0);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

}  // namespace attn
}  // namespace hy

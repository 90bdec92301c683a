// Gated DeltaNet decode step, in place, on sm_103a (standalone launch; the
// math and its sources are in gdn_dev.cuh).
//
// Grid: (heads, dv / 16); a CTA is one work item: 16 value rows of one head
// (4 warps x 4 rows).  The state rows, the conv taps and the conv history are
// loaded before griddepcontrol.wait: no earlier kernel of the same step writes
// them, so their latency overlaps the projection GEMV's tail and only the
// projection output is read after the wait.
#include "common.cuh"
#include "gdn_dev.cuh"
#include "kernels.h"

namespace hy {
namespace gdn {
namespace {

constexpr int kWarps = kThreads / 32;

template <int EPL>  // state elements per lane: dk / 32
__global__ void __launch_bounds__(kThreads) k_gdn(const Params p0) {
  __shared__ ItemShared<EPL> sh;
  const int h = blockIdx.x, rc = blockIdx.y;
  Params p = p0;
  if (p0.nb > 0) {  // token blockIdx.z of a batch: its sequence's state
    const int z = blockIdx.z;
    p.y = p0.y + (long long)z * p0.ld_y;
    p.o = p0.o + (long long)z * p0.ld_o;
    p.S = p0.S_b[z];
    p.conv_state = p0.conv_b[z];
    p.pos = p0.pos_b[z];
  }
  Rows<EPL, kWarps> R;
  ConvRegs<EPL, kWarps> V;
  load_rows<EPL, kWarps>(p, h, rc, R, threadIdx.x);  // pre-wait
  load_conv<EPL, kWarps>(p, h, rc, V, threadIdx.x);  // pre-wait
  pdl_launch_dependents();  // the next GEMV may stage its weights meanwhile
  pdl_wait();
  run_item<EPL, kWarps>(p, h, rc, R, V, sh, threadIdx.x, [] __device__() { __syncthreads(); });
}

}  // namespace

cudaError_t launch(const Params& p, cudaStream_t st, bool pdl) {
  if (p.dk % 32 != 0 || p.conv_k < 1 || p.conv_k > kMaxConvK) return cudaErrorInvalidValue;
  if (p.nb < 0 || p.nb > kMaxB) return cudaErrorInvalidValue;
  const dim3 grid(p.nh, (p.dv + kRowsPerCta - 1) / kRowsPerCta, p.nb > 0 ? p.nb : 1);
  switch (p.dk / 32) {
    case 2: return launch_k(k_gdn<2>, grid, dim3(kThreads), 0, st, pdl, p);
    case 4: return launch_k(k_gdn<4>, grid, dim3(kThreads), 0, st, pdl, p);
    case 8: return launch_k(k_gdn<8>, grid, dim3(kThreads), 0, st, pdl, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
}  // namespace hy

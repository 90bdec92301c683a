// hy_op_attention_noalloc: the decode attention of hy_op_attention with its
// scratch (the guard word, the per-kv-head last-CTA tickets and the per-split
// partial outputs) in a fixed array that the library holds in device memory,
// so that the call allocates nothing.
//
// For callers that cannot call cudaMalloc: code that runs under a host
// framework owning the whole device memory budget through its own pool, code
// on a latency path where an allocation (and its implicit synchronisation) is
// not allowed, and plug-ins whose host forbids allocations outside its
// allocator.  The array costs HY_NOALLOC_SCRATCH_BYTES on every GPU that loads
// the library, for the life of the process.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/hybrid.h"
#include "common.cuh"
#include "kernels.h"

using namespace hy;

namespace {

constexpr size_t kScratchBytes = HY_NOALLOC_SCRATCH_BYTES;
constexpr size_t kHeaderBytes = 256;  // guard word, then padding
constexpr int kMaxDevices = 64;

// Every call on a device shares this array and finds in it what the last call
// left.  Host code sees only a host-side stand-in for it: the device address
// comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
uint8_t* g_addr[kMaxDevices];
int g_nsm[kMaxDevices];

int err(int code, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return set_error(code, buf);
}

// Once per device, with that device current: the kernels' shared-memory
// limits and the array's device address.
int setup(uint8_t** addr, int* nsm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return err(HY_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return err(HY_ERR_UNSUPPORTED, "device index %d is beyond %d", dev, kMaxDevices - 1);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    int n = 0;
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err(HY_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if ((e = attn::init()) != cudaSuccess) return err(HY_ERR_CUDA, "attention set-up: %s", cudaGetErrorString(e));
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_scratch)) != cudaSuccess)
      return err(HY_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    g_nsm[dev] = n;
    g_addr[dev] = (uint8_t*)p;
  }
  *addr = g_addr[dev];
  *nsm = g_nsm[dev];
  return HY_OK;
}

}  // namespace

// Device address of the guard word in this device's array, or null before the
// first hy_op_attention_noalloc call on it (nothing to report then).
unsigned* hy::noalloc_guard() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return reinterpret_cast<unsigned*>(g_addr[dev]);
}

extern "C" int hy_op_attention_noalloc(const float* y_dev, void* K_dev, void* V_dev, int32_t cap, int32_t nq,
                                       int32_t nkv, int32_t hd, const int32_t* len_dev, const float* rope_table_dev,
                                       int32_t nsplit, float* o_dev, void* stream) {
  if (!y_dev || !K_dev || !V_dev || ((uintptr_t)K_dev & 15u) || ((uintptr_t)V_dev & 15u) || !len_dev ||
      !rope_table_dev || !o_dev || cap <= 0 || nkv <= 0 || nq <= 0 || nq % nkv)
    return err(HY_ERR_ARG, "bad attention arguments");
  if ((hd != 64 && hd != 128 && hd != 256) || nq / nkv > 8 || ((nq / nkv) & (nq / nkv - 1)))
    return err(HY_ERR_UNSUPPORTED, "attention: head_dim 64/128/256 and nq/nkv in {1,2,4,8}");
  uint8_t* base = nullptr;
  int nsm = 0;
  int rc = setup(&base, &nsm);
  if (rc != HY_OK) return rc;
  if (nsplit <= 0) nsplit = attn::auto_splits(nkv, nsm);
  // layout: [guard | pad to 256] [tickets, nkv words, padded to 256] [partials]
  const size_t tickets = ((size_t)nkv * 4 + 255) / 256 * 256;
  const size_t need = kHeaderBytes + tickets + attn::part_floats(nq, nkv, hd, nsplit) * 4;
  if (need > kScratchBytes)
    return err(HY_ERR_UNSUPPORTED, "attention scratch of %zu bytes exceeds the fixed array of %zu bytes", need,
               kScratchBytes);
  const cudaStream_t st = (cudaStream_t)stream;
  // the guard and the tickets must start at zero; partials are written before
  // they are read
  cudaError_t e = cudaMemsetAsync(base, 0, kHeaderBytes + tickets, st);
  if (e != cudaSuccess) return err(HY_ERR_CUDA, "clearing the scratch header: %s", cudaGetErrorString(e));
  attn::Params a;
  memset(&a, 0, sizeof(a));
  a.y = y_dev;
  a.K = (uint16_t*)K_dev;
  a.V = (uint16_t*)V_dev;
  a.len = len_dev;
  a.rope = (const float2*)rope_table_dev;
  a.cap = cap;
  a.nq = nq;
  a.nkv = nkv;
  a.hd = hd;
  a.nsplit = nsplit;
  a.scale = 1.0f / sqrtf((float)hd);
  a.guard = (unsigned*)base;
  a.counter = (unsigned*)(base + kHeaderBytes);
  a.part = (float*)(base + kHeaderBytes + tickets);
  a.o = o_dev;
  if ((e = attn::launch(a, st, false)) != cudaSuccess)
    return err(HY_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return HY_OK;
}

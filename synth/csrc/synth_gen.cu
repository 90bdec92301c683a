// Device (CUDA) copy of the seeded synthetic-input generator defined in
// synth/gen.py.  It holds none of the decode step's arithmetic: it fills
// multi-GB weight tensors in HBM so that large models need no host-side
// generation.  Bit-identical to the numpy definition and to synth_host.c
// (checked by the GPU tests).
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace {
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ULL;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ inline uint16_t f32_to_bf16(float f) {
  uint32_t b = __float_as_uint(f);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

__global__ void k_normal_bf16(uint16_t* dst, uint64_t n, uint64_t key, float scale, uint64_t start) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t w = mix64(key + (i + start + 1ULL) * kGolden);
    int64_t s = (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) + (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
    dst[i] = f32_to_bf16(__fmul_rn((float)(s - 131070), scale));
  }
}

__global__ void k_q4_packed(uint8_t* dst, uint64_t nbytes, uint64_t key) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < nbytes; i += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t w = mix64(key + (i / 8ULL + 1ULL) * kGolden);
    dst[i] = (uint8_t)((w >> (8 * (i % 8ULL))) & 0xFF);
  }
}

__global__ void k_q4_scales(uint16_t* dst, uint64_t nblocks, uint64_t key, float mult) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < nblocks; i += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t w = mix64(key + (i + 1ULL) * kGolden);
    float u = (float)((int64_t)(w & 0xFFFF) + 49152);
    dst[i] = __half_as_ushort(__float2half_rn(__fmul_rn(u, mult)));
  }
}

__global__ void k_uniform_ids(int32_t* dst, uint64_t n, uint64_t key, uint32_t upper, uint64_t start) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t w = mix64(key + (i + start + 1ULL) * kGolden);
    dst[i] = (int32_t)(((w >> 32) * (uint64_t)upper) >> 32);
  }
}

__global__ void k_fill_f32(float* dst, uint64_t n, float v) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) dst[i] = v;
}

inline unsigned grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  return (unsigned)(b < 152 * 64 ? (b == 0 ? 1 : b) : 152 * 64);
}
inline uint64_t key_of(uint64_t seed, uint64_t tid) { return mix64(seed * kGolden + tid); }
}  // namespace

extern "C" {
int synd_fill_normal_bf16(void* dst, uint64_t n, uint64_t seed, uint64_t tid, float scale, uint64_t start, void* stream) {
  if (n == 0) return 0;
  k_normal_bf16<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dst, n, key_of(seed, tid), scale, start);
  return (int)cudaGetLastError();
}
int synd_fill_q4_packed(void* dst, uint64_t nbytes, uint64_t seed, uint64_t tid, void* stream) {
  if (nbytes == 0) return 0;
  k_q4_packed<<<grid_for(nbytes), 256, 0, (cudaStream_t)stream>>>((uint8_t*)dst, nbytes, key_of(seed, tid));
  return (int)cudaGetLastError();
}
int synd_fill_q4_scales(void* dst, uint64_t nblocks, uint64_t seed, uint64_t tid, float mult, void* stream) {
  if (nblocks == 0) return 0;
  k_q4_scales<<<grid_for(nblocks), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dst, nblocks, key_of(seed, tid), mult);
  return (int)cudaGetLastError();
}
int synd_fill_uniform_ids(void* dst, uint64_t n, uint64_t seed, uint64_t tid, uint32_t upper, uint64_t start, void* stream) {
  if (n == 0) return 0;
  k_uniform_ids<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((int32_t*)dst, n, key_of(seed, tid), upper, start);
  return (int)cudaGetLastError();
}
int synd_fill_f32(void* dst, uint64_t n, float v, void* stream) {
  if (n == 0) return 0;
  k_fill_f32<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((float*)dst, n, v);
  return (int)cudaGetLastError();
}
}

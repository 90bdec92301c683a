// Shared device helpers for the sm_103a kernels: bf16 unpacking, warp
// reductions, mbarrier / bulk-copy (TMA engine) wrappers with bounded waits,
// and programmatic-dependent-launch (PDL) controls.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hy {

constexpr int kWarp = 32;

// Error word bits set by device-side guards; read back by the host.
enum GuardBits : unsigned {
  kGuardWaitTimeout = 1u << 0,   // an mbarrier wait ran past its time limit
  kGuardBadIndex = 1u << 1,      // a token id or expert id outside its range
  kGuardBadPosition = 1u << 2,   // a sequence position outside its cache capacity
};

// Time limit for any spin-wait inside a kernel (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_guard(unsigned* guard, unsigned bits) {
  if (guard) atomicOr(guard, bits);
}

// ------------------------------------------------------------------ PDL
// Wait until the preceding kernel in the stream (or graph) has completed and
// its writes are visible.  Every kernel calls this before touching any data a
// preceding kernel may write; only immutable weights (and state that no
// earlier kernel of the same step writes) are read before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream start launching (its pre-wait prologue
// only streams weights, so this may be issued early).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// dot of 8 bf16 (one 16-byte vector) with 8 fp32 values
__device__ __forceinline__ float dot8(const uint4 w, const float* x) {
  float a = bf16_lo(w.x) * x[0];
  a = fmaf(bf16_hi(w.x), x[1], a);
  a = fmaf(bf16_lo(w.y), x[2], a);
  a = fmaf(bf16_hi(w.y), x[3], a);
  a = fmaf(bf16_lo(w.z), x[4], a);
  a = fmaf(bf16_hi(w.z), x[5], a);
  a = fmaf(bf16_lo(w.w), x[6], a);
  a = fmaf(bf16_hi(w.w), x[7], a);
  return a;
}

// Two FP32 FMAs in one packed instruction (sm_100 family): (a0, a1) +=
// (w0 * x0, w1 * x1), each rounded once as fmaf would.
__device__ __forceinline__ void fma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
  asm("{\n .reg .b64 a, w, x;\n mov.b64 a, {%0, %1};\n mov.b64 w, {%2, %3};\n mov.b64 x, {%4, %5};\n"
      " fma.rn.f32x2 a, w, x, a;\n mov.b64 {%0, %1}, a;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// 8 bf16 (one 16-byte vector) times 8 FP32 values, accumulated into the pair
// (even elements, odd elements) with packed FMAs.
__device__ __forceinline__ void dot8_acc2(const uint4 w, const float* x, float& ae, float& ao) {
  fma2(ae, ao, bf16_lo(w.x), bf16_hi(w.x), x[0], x[1]);
  fma2(ae, ao, bf16_lo(w.y), bf16_hi(w.y), x[2], x[3]);
  fma2(ae, ao, bf16_lo(w.z), bf16_hi(w.z), x[4], x[5]);
  fma2(ae, ao, bf16_lo(w.w), bf16_hi(w.w), x[6], x[7]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + __expf(-x)); }

// ------------------------------------------------------------ top-k
// Unsigned key with the order of the FP32 value (-0 taken as +0, as an FP32
// compare does), and back.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// top_k of E logits (FP32 compare, lowest index on ties; a NaN ranks last) by
// one warp, in order (the same set and order as ranking all experts), E <=
// 32 * kPer.  Each lane holds logits lane, lane + 32, ... as order keys (slots past E get key
// 0, below every logit) and sorts them once, best first, with a bitonic
// network in registers; then each round takes the warp's best with two
// reductions (the largest key, then the lowest index holding it) and the
// winning lane shifts its list by one.  sel / selv (shared) receive ids and
// logits.
template <int kPer, typename Load>
__device__ __forceinline__ void warp_topk(Load load, int E, int K, int* sel, float* selv, int lane) {
  uint32_t key[kPer];
  uint32_t idx[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? load(e) : -INFINITY;
    key[i] = e < E ? order_key(x == x ? x : -INFINITY) : 0u;
    idx[i] = (uint32_t)e;
  }
  // bitonic sort, best first: a larger key, or an equal key and a lower index
#pragma unroll
  for (int k = 2; k <= kPer; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool i_better = key[i] > key[l] || (key[i] == key[l] && idx[i] < idx[l]);
          const bool want_i_first = (i & k) == 0;
          if (i_better != want_i_first) {
            const uint32_t tk = key[i], ti = idx[i];
            key[i] = key[l];
            idx[i] = idx[l];
            key[l] = tk;
            idx[l] = ti;
          }
        }
      }
    }
  }
  for (int q = 0; q < K; ++q) {
    const uint32_t gk = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t gi = __reduce_min_sync(0xffffffffu, key[0] == gk ? idx[0] : 0xffffffffu);
    if (lane == 0) {
      sel[q] = (int)gi;
      selv[q] = key_value(gk);
    }
    if (idx[0] == gi) {
#pragma unroll
      for (int i = 0; i + 1 < kPer; ++i) {
        key[i] = key[i + 1];
        idx[i] = idx[i + 1];
      }
      key[kPer - 1] = 0u;
      idx[kPer - 1] = 0xffffffffu;
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------ mbarrier / bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase of the given parity; false after kWaitLimitNs.
// The clock is read once every 1024 polls, not on every poll.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 0) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitLimitNs) return false;
    }
  }
}

// L2 policy for streamed-once weights: evict first, so KV, state and
// activations stay resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk global->shared copy on the TMA engine; completion is signalled on
// `bar` as transaction bytes.  dst, src and bytes must be 16-byte aligned.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (no destination, no
// completion); src and bytes 16-byte aligned.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier over a subset of warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns, to every participant, whether any of them
// passed pred = true (a decision all of them then take alike).
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

}  // namespace hy

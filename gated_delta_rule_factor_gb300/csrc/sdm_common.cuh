// Device helpers shared by the SDM kernels: sortable keys, warp bitonic sorts,
// accurate dot products, 16-byte row vectors of the bank / activation types and
// the kernel-side error flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

// ---------------------------------------------------------------- error flag

// Records the first kernel-side error code in the workspace flag; the access that
// raised it is skipped by the caller.  Never traps.
__device__ __forceinline__ void raise_error(int32_t *flag, int32_t code) {
  if (flag) atomicCAS(flag, 0, code);
}

// ---------------------------------------------------------------- sortable keys

// Monotone map of a float32 onto uint32 (larger float -> larger integer); -0 is
// first turned into +0 so that the two zeros compare equal, as IEEE comparison does.
__device__ __forceinline__ uint32_t ordered_bits(float x) {
  x = __fadd_rn(x, 0.0f);
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// ---------------------------------------------------------------- warp bitonic sort

// Sorts the 32*E 64-bit keys held by a warp (element i = lane*E + e) descending.
template <int E>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&key)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
        const int lj = j / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane * E + e;
          const uint64_t o = __shfl_xor_sync(0xffffffffu, key[e], lj);
          const bool desc = (i & k) == 0;
          const bool lower = (i & j) == 0;
          key[e] = (desc == lower) ? (key[e] > o ? key[e] : o) : (key[e] < o ? key[e] : o);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const int i = lane * E + e;
            const bool desc = (i & k) == 0;
            const uint64_t a = key[e], b = key[e | j];
            const bool sw = desc ? (a < b) : (a > b);
            key[e] = sw ? b : a;
            key[e | j] = sw ? a : b;
          }
        }
      }
    }
  }
}

// Two independent warp_sort_desc runs interleaved step by step (twice the work in
// flight per shuffle latency).
template <int E>
__device__ __forceinline__ void warp_sort_desc2(uint64_t (&ka)[E], uint64_t (&kb)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
        const int lj = j / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane * E + e;
          const uint64_t oa = __shfl_xor_sync(0xffffffffu, ka[e], lj);
          const uint64_t ob = __shfl_xor_sync(0xffffffffu, kb[e], lj);
          const bool keep_max = ((i & k) == 0) == ((i & j) == 0);
          ka[e] = keep_max ? (ka[e] > oa ? ka[e] : oa) : (ka[e] < oa ? ka[e] : oa);
          kb[e] = keep_max ? (kb[e] > ob ? kb[e] : ob) : (kb[e] < ob ? kb[e] : ob);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const int i = lane * E + e;
            const bool desc = (i & k) == 0;
            const uint64_t a = ka[e], b = ka[e | j], c = kb[e], d = kb[e | j];
            const bool sa = desc ? (a < b) : (a > b), sc = desc ? (c < d) : (c > d);
            ka[e] = sa ? b : a;
            ka[e | j] = sa ? a : b;
            kb[e] = sc ? d : c;
            kb[e | j] = sc ? c : d;
          }
        }
      }
    }
  }
}

// Keeps the 32*E largest of two descending lists: `key` becomes the descending
// merge of max(key[i], other[P-1-i]) (a bitonic sequence), P = 32*E.
template <int E>
__device__ __forceinline__ void warp_merge_top_desc(uint64_t (&key)[E], const uint64_t (&other)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint64_t o = __shfl_sync(0xffffffffu, other[E - 1 - e], 31 - lane);
    key[e] = key[e] > o ? key[e] : o;
  }
#pragma unroll
  for (int j = 16 * E; j > 0; j >>= 1) {
    if (j >= E) {
      const int lj = j / E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        const uint64_t o = __shfl_xor_sync(0xffffffffu, key[e], lj);
        key[e] = ((i & j) == 0) ? (key[e] > o ? key[e] : o) : (key[e] < o ? key[e] : o);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if ((e & j) == 0) {
          const uint64_t a = key[e], b = key[e | j];
          const bool sw = a < b;
          key[e] = sw ? b : a;
          key[e | j] = sw ? a : b;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- accurate dot products
//
// Factor scores are taken so that rounding them once to float32 almost always gives
// the correctly rounded dot product.  float32 inputs: the compensated dot product of
// Ogita, Rump and Oishi ("Accurate sum and dot product", SIAM J. Sci. Comput. 2005),
// an error-free product (Dekker/FMA) and Knuth's TwoSum per term.  bfloat16 inputs:
// their products are exact in float32, so 32-term blocks are accumulated with FMA and
// each block sum is folded into a TwoSum (sum, correction) pair.

struct Acc2 {
  float s, c;
};

__device__ __forceinline__ void two_sum_into(Acc2 &a, float x) {
  const float t = __fadd_rn(a.s, x);
  const float z = __fsub_rn(t, a.s);
  const float e = __fadd_rn(__fsub_rn(a.s, __fsub_rn(t, z)), __fsub_rn(x, z));
  a.s = t;
  a.c = __fadd_rn(a.c, e);
}

__device__ __forceinline__ void dot2_step(Acc2 &a, float x, float y) {
  const float p = __fmul_rn(x, y);
  const float pe = __fmaf_rn(x, y, -p);
  two_sum_into(a, p);
  a.c = __fadd_rn(a.c, pe);
}

__device__ __forceinline__ float acc2_value(const Acc2 &a) { return __fadd_rn(a.s, a.c); }

constexpr int kBf16Block = 32;  // terms per FMA block of the bfloat16 dot product

// ---------------------------------------------------------------- element types

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// A 16-byte vector of T (4 floats or 8 bfloat16) converted to / from float32 lanes.
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
};

template <typename T>
__device__ __forceinline__ void load_vec16(const T *p, float (&out)[Vec16<T>::N]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
  for (int i = 0; i < Vec16<T>::N; ++i) out[i] = to_f32(e[i]);
}

template <typename T>
__device__ __forceinline__ void store_vec16(T *p, const float (&in)[Vec16<T>::N]) {
  uint4 u;
  T *e = reinterpret_cast<T *>(&u);
#pragma unroll
  for (int i = 0; i < Vec16<T>::N; ++i) e[i] = from_f32<T>(in[i]);
  *reinterpret_cast<uint4 *>(p) = u;
}

// Loads / stores NV consecutive elements of T as 16-byte accesses (NV * sizeof(T) of 16
// or 32 bytes), one 8-byte access, or element by element.
template <typename T, int NV>
__device__ __forceinline__ void load_vec(const T *p, float (&out)[NV]) {
  if constexpr (NV * sizeof(T) == 32) {
    const uint4 u0 = *reinterpret_cast<const uint4 *>(p), u1 = *reinterpret_cast<const uint4 *>(p + NV / 2);
    const T *e0 = reinterpret_cast<const T *>(&u0), *e1 = reinterpret_cast<const T *>(&u1);
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      out[i] = to_f32(e0[i]);
      out[NV / 2 + i] = to_f32(e1[i]);
    }
  } else if constexpr (NV * sizeof(T) == 16) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int i = 0; i < NV; ++i) out[i] = to_f32(e[i]);
  } else if constexpr (NV * sizeof(T) == 8) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int i = 0; i < NV; ++i) out[i] = to_f32(e[i]);
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) out[i] = to_f32(p[i]);
  }
}

template <typename T, int NV>
__device__ __forceinline__ void store_vec(T *p, const float (&in)[NV]) {
  if constexpr (NV * sizeof(T) == 32) {
    uint4 u0, u1;
    T *e0 = reinterpret_cast<T *>(&u0), *e1 = reinterpret_cast<T *>(&u1);
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      e0[i] = from_f32<T>(in[i]);
      e1[i] = from_f32<T>(in[NV / 2 + i]);
    }
    *reinterpret_cast<uint4 *>(p) = u0;
    *reinterpret_cast<uint4 *>(p + NV / 2) = u1;
  } else if constexpr (NV * sizeof(T) == 16) {
    uint4 u;
    T *e = reinterpret_cast<T *>(&u);
#pragma unroll
    for (int i = 0; i < NV; ++i) e[i] = from_f32<T>(in[i]);
    *reinterpret_cast<uint4 *>(p) = u;
  } else if constexpr (NV * sizeof(T) == 8) {
    uint2 u;
    T *e = reinterpret_cast<T *>(&u);
#pragma unroll
    for (int i = 0; i < NV; ++i) e[i] = from_f32<T>(in[i]);
    *reinterpret_cast<uint2 *>(p) = u;
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) p[i] = from_f32<T>(in[i]);
  }
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async8(void *dst_smem, const void *src_gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src_gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Waits until at most N of this thread's committed cp.async groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_pending() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- mbarriers and bulk copies

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // a kernel gives up on a wait after 2 s

// Bounded wait for the mbarrier phase with the given parity; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = smem_addr(bar);
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 255) == 255 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Global -> shared bulk copy (bytes % 16 == 0, both addresses 16-byte aligned) that
// completes on an mbarrier.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Shared -> global bulk copy in the calling thread's current bulk group.
__device__ __forceinline__ void bulk_store(void *dst_gmem, const void *src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst_gmem),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Waits until this thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// Waits until at most N of this thread's newest bulk store groups are still reading
// shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read_pending() {
  asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}
// Waits until this thread's bulk stores are complete (their writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Orders this thread's earlier generic-proxy accesses before later async-proxy (bulk
// copy / TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// Arrives at named barrier `id` without waiting (a producer's signal to threads that
// bar.sync on it); the arriving threads' earlier memory accesses are ordered before it.
__device__ __forceinline__ void named_barrier_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

}  // namespace sdm

// topo_device.cuh -- device building blocks shared by the condensate-set
// attention kernels: PTX wrappers (mbarrier, TMA), bounded waits, the ranking
// key, and warp-level bitonic sort / merge in registers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace topo {

constexpr int kTile = 64;                        // keys per pipeline tile
constexpr int kConsumerWarps = 4;                // warps that score tiles
constexpr int kWarps = kConsumerWarps + 1;       // + one TMA producer warp
constexpr int kThreads = 32 * kWarps;
constexpr unsigned long long kWaitNs = 1000000000ull;  // every device wait gives up after 1 s
constexpr int kStatusTimeout = -5;               // TOPO_ERR_DEVICE_TIMEOUT
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- PTX ------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete; false after
// kWaitNs without completion (the caller records the timeout and bails out).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

// 2-D tiled TMA load (box of the tensor map) into shared memory; completion
// is signalled on `bar` as transaction bytes.  x must be 16-byte aligned in
// bytes (callers only pass multiples of 128 bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global to shared memory; completion is signalled on `bar` as transaction
// bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ elements -----

// element e of a 16-byte chunk, widened exactly to float
template <bool BF16>
__device__ __forceinline__ float chunk_elem(const uint4& w, int e) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
  if constexpr (BF16) {
    const uint32_t word = u[e >> 1];
    return __uint_as_float((e & 1) ? (word & 0xffff0000u) : (word << 16));
  } else {
    return __uint_as_float(u[e]);
  }
}

template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (BF16) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    return reinterpret_cast<const float*>(base)[i];
  }
}

// ---------------------------------------------------------- ranking key ----
//
// A candidate (score s, position j) is packed into one 64-bit key whose
// unsigned order is the ranking order: larger score first, then smaller j.
// The high word maps the float32 score monotonically onto uint32 (-0 ranks as
// +0); the low word is ~j.  Every finite score gives a key > 0, so 0 marks an
// empty slot.

__device__ __forceinline__ uint32_t ord_score(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t rank_key(float s, uint32_t j) {
  return (static_cast<uint64_t>(ord_score(s)) << 32) | static_cast<uint32_t>(~j);
}

__device__ __forceinline__ uint32_t key_pos(uint64_t key) { return ~static_cast<uint32_t>(key); }

// inverse of ord_score
__device__ __forceinline__ float ord_to_float(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ float key_score(uint64_t key) {
  return ord_to_float(static_cast<uint32_t>(key >> 32));
}

// ------------------------------------------------- warp bitonic networks ----
//
// A warp holds a list of N = 32*E 64-bit keys in registers, element i at
// register i / 32 of lane i % 32.

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Sort descending (bitonic sorting network).
template <int E>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&x)[E], int lane) {
  constexpr int N = 32 * E;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int J = j >> 5;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & J) continue;
          const bool desc = ((e * 32) & size) == 0;
          const uint64_t a = x[e], b = x[e | J];
          x[e] = desc ? umax64(a, b) : umin64(a, b);
          x[e | J] = desc ? umin64(a, b) : umax64(a, b);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t p = __shfl_xor_sync(kFull, x[e], j);
          const bool lower = (lane & j) == 0;
          const bool desc = ((e * 32 + lane) & size) == 0;
          x[e] = (lower == desc) ? umax64(x[e], p) : umin64(x[e], p);
        }
      }
    }
  }
}

// Sort floats descending across the warp (same network, 32-bit elements).
template <int E>
__device__ __forceinline__ void warp_sort_desc_f32(float (&x)[E], int lane) {
  constexpr int N = 32 * E;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int j = size >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int J = j >> 5;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & J) continue;
          const bool desc = ((e * 32) & size) == 0;
          const float a = x[e], b = x[e | J];
          x[e] = desc ? fmaxf(a, b) : fminf(a, b);
          x[e | J] = desc ? fminf(a, b) : fmaxf(a, b);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float p = __shfl_xor_sync(kFull, x[e], j);
          const bool lower = (lane & j) == 0;
          const bool desc = ((e * 32 + lane) & size) == 0;
          x[e] = (lower == desc) ? fmaxf(x[e], p) : fminf(x[e], p);
        }
      }
    }
  }
}

// a <- the N largest of (a U b), sorted descending; a and b sorted descending.
// max(a[i], b[N-1-i]) is bitonic and holds exactly those N elements; a
// half-cleaner cascade then sorts it.
template <int E>
__device__ __forceinline__ void warp_merge_desc(uint64_t (&a)[E], const uint64_t (&b)[E],
                                                int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint64_t br = __shfl_sync(kFull, b[E - 1 - e], 31 - lane);
    a[e] = umax64(a[e], br);
  }
#pragma unroll
  for (int j = 16 * E; j > 0; j >>= 1) {
    if (j >= 32) {
      const int J = j >> 5;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e & J) continue;
        const uint64_t x = a[e], y = a[e | J];
        a[e] = umax64(x, y);
        a[e | J] = umin64(x, y);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t p = __shfl_xor_sync(kFull, a[e], j);
        a[e] = ((lane & j) == 0) ? umax64(a[e], p) : umin64(a[e], p);
      }
    }
  }
}

// element i of a warp list (i uniform across the warp)
template <int E>
__device__ __forceinline__ uint64_t warp_list_get(const uint64_t (&x)[E], int i) {
  uint64_t v = 0;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (e == (i >> 5)) v = x[e];
  return __shfl_sync(kFull, v, i & 31);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

}  // namespace topo

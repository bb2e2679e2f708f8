// tc_bound_kernel.cu -- test-only kernel: one tcgen05 bf16 x bf16 -> float32
// MMA chain (M = 128 rows of A, N columns of B, K = d in steps of 16), the
// operation both tensor-core scorers of the library issue, with the operands
// written into shared memory in the library's own layout (K-major, 128-byte
// swizzle, through the same helpers).  The test compares D with the exact dot
// products to check the accumulation error bound the exact top-k selection
// relies on.  Built by tests/test_gpu_tc_bound.py; not part of the library.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc_device.cuh"
#include "topo_device.cuh"

namespace {

template <int D, int N>
struct TcbSmem {
  static constexpr int A = 0;                  // 128 x D bf16
  static constexpr int B = 128 * D * 2;        // N x D bf16
  static constexpr int BAR = B + N * D * 2;    // one mbarrier
  static constexpr int TSLOT = BAR + 8;        // TMEM base address
  static constexpr int TOTAL = TSLOT + 8 + 1024;  // + slack to align the base to 1024
};

// a: [128][D], b: [N][D] bfloat16 bits; d: [128][N] float32, d[i][j] =
// sum_c a[i][c] * b[j][c] as the tensor cores accumulate it.  One CTA of 128
// threads; status[0] = 1 if the MMA did not complete within the bounded wait.
template <int D, int N>
__global__ void __launch_bounds__(128, 1)
    tcb_kernel(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b, float* __restrict__ d,
               int* status) {
  using L = TcbSmem<D, N>;
  extern __shared__ uint8_t raw[];
  const uint32_t base = topo::smem_addr(raw);
  uint8_t* sm = raw + ((1024u - (base & 1023u)) & 1023u);
  uint8_t* sa = sm + L::A;
  uint8_t* sb = sm + L::B;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::TSLOT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < 128 * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    *reinterpret_cast<uint16_t*>(sa + topo::tc::sw128_offset_bf16(r, c, 128)) = a[i];
  }
  for (int i = tid; i < N * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    *reinterpret_cast<uint16_t*>(sb + topo::tc::sw128_offset_bf16(r, c, N)) = b[i];
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == 0) {
    topo::mbar_init(bar, 1);
    topo::fence_mbar_init();
  }
  if (warp == 0) {
    topo::tc::tmem_alloc(tslot, N < 32 ? 32u : (uint32_t)N);
    topo::tc::tmem_relinquish();
  }
  topo::tc::fence_before_sync();
  __syncthreads();
  topo::tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (tid == 0) {
    constexpr uint32_t idesc = topo::tc::idesc_bf16_f32(128, N);
    const uint32_t a0 = topo::smem_addr(sa), b0 = topo::smem_addr(sb);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t ao = a0 + (ks >> 2) * (128 * 128) + (ks & 3) * 32;
      const uint32_t bo = b0 + (ks >> 2) * (N * 128) + (ks & 3) * 32;
      topo::tc::mma_bf16(tmem, topo::tc::smem_desc_sw128(ao), topo::tc::smem_desc_sw128(bo),
                         idesc, ks > 0);
    }
    topo::tc::mma_commit(bar);
  }
  __syncwarp();
  const bool ok = topo::mbar_wait(bar, 0);
  topo::tc::fence_after_sync();
  if (ok) {
    const int row = warp * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      topo::tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      topo::tc::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) d[row * N + c0 + j] = v[j];
    }
  } else if (tid == 0) {
    status[0] = 1;
  }
  topo::tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    topo::tc::fence_after_sync();
    topo::tc::tmem_dealloc(tmem, N < 32 ? 32u : (uint32_t)N);
  }
}

template <int D, int N>
int launch(const void* a, const void* b, float* d, int* status, cudaStream_t st) {
  constexpr int smem = TcbSmem<D, N>::TOTAL;
  if (cudaFuncSetAttribute(tcb_kernel<D, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -4;
  tcb_kernel<D, N><<<1, 128, smem, st>>>(static_cast<const uint16_t*>(a),
                                         static_cast<const uint16_t*>(b), d, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

// d must hold 128 * n floats; a: 128 x dim, b: n x dim bf16 bits, all device
// pointers.  dim in {64, 128}, n in {16, 256}.  Returns 0, -1 (shape) or -4.
extern "C" int tcb_run(int dim, int n, const void* a, const void* b, float* d, int* status,
                       void* stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dim == 64 && n == 16) return launch<64, 16>(a, b, d, status, st);
  if (dim == 64 && n == 256) return launch<64, 256>(a, b, d, status, st);
  if (dim == 128 && n == 16) return launch<128, 16>(a, b, d, status, st);
  if (dim == 128 && n == 256) return launch<128, 256>(a, b, d, status, st);
  return -1;
}

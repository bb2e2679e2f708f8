// topo_noalloc.cu -- topo_attn_forward_noalloc: condensate-set attention for
// callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and have no
// way to obtain a device workspace: plugin hosts that own every allocation,
// and latency-critical loops where a cudaMalloc (which can synchronise the
// device) is not allowed once serving has started.  This entry point gives
// them the same computation as topo_attn_forward with its scratch (the split
// counters, per-split candidate lists and the status word) in a fixed-size
// array that lives in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds TOPO_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, so the device address is
// looked up with cudaGetSymbolAddress, once per device, with that device
// current, and that address is what the kernels receive.
#include <cuda_runtime.h>
#include <mutex>

#include "topo_attn.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[TOPO_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device); nullptr on failure.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_addr[dev] = ptr;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" int topo_attn_forward_noalloc(const topo_attn_params* p, const void* q, const void* k,
                                         const void* v, float* out, int32_t* idx, float* excl,
                                         topo_stream_t stream) {
  const size_t need = topo_attn_workspace_size(p);
  if (need == 0) {
    // invalid or unsupported parameters: let the regular entry point report which
    return topo_attn_forward(p, q, k, v, out, idx, excl, nullptr, 0, stream);
  }
  if (need > (size_t)TOPO_NOALLOC_SCRATCH_BYTES) return TOPO_ERR_SCRATCH_LIMIT;
  void* ws = scratch_on_current_device();
  if (!ws) return TOPO_ERR_CUDA;
  // topo_attn_forward clears the split counters it uses on `stream` before
  // its kernels run, so the previous call's contents do no harm.
  return topo_attn_forward(p, q, k, v, out, idx, excl, ws, (size_t)TOPO_NOALLOC_SCRATCH_BYTES,
                           stream);
}

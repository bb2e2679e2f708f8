// topo_launch.cuh -- typed launchers for the kernels of topo_kernels.cuh.
// Each (dtype, d) pair is instantiated in its own translation unit.
#pragma once

#include "topo_prefill.cuh"

namespace topo {

constexpr int kMaxSmem = 232448;  // opt-in shared memory per block on sm_100-class parts

template <auto Kern>
cudaError_t allow_smem() {
  static const cudaError_t e =
      cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  return e;
}

template <bool BF16, int D>
struct Launcher {
  static cudaError_t select(int NC, int KE, const CUtensorMap& mk, const Geom& G, dim3 grid,
                            int smem, cudaStream_t st);
  static cudaError_t excl(int NC, const CUtensorMap& mk, const Geom& G, dim3 grid, int smem,
                          cudaStream_t st);
  static cudaError_t dense(int NC, const CUtensorMap& mk, const CUtensorMap& mv, const Geom& G,
                           dim3 grid, int smem, cudaStream_t st);
  static cudaError_t pv(const Geom& G, long long nrows, cudaStream_t st);
  static cudaError_t compact(const Geom& G, void* k_out, void* v_out, cudaStream_t st);
  static cudaError_t select_tc(int NC, int KE, bool group, const CUtensorMap& mk128,
                               const Geom& G, dim3 grid, int smem, cudaStream_t st);
  // the tail of a kSplitTail select launch, as its programmatic dependent
  static cudaError_t tail_tc(int NC, int KE, bool group, const Geom& G, dim3 grid, int smem,
                             int scratch_bytes, cudaStream_t st);
  // dense attention on the tensor cores (bf16 only)
  static cudaError_t dense_tc(int NC, const CUtensorMap& mk128, const CUtensorMap& mv128,
                              const Geom& G, dim3 grid, int smem, cudaStream_t st);
  // chunked prefill on the tensor cores (bf16 only): K scale, scan, finalize, softmax
  static cudaError_t prefill(const CUtensorMap& mk128, const Geom& G, int scan_grid, int scan_smem,
                             int kmax_grid, bool do_pv, cudaStream_t st);
};

template <bool BF16, int D, int NC, int KE>
cudaError_t run_select(const CUtensorMap& mk, const Geom& G, dim3 grid, int smem,
                       cudaStream_t st) {
  constexpr auto kern = &topo_select_kernel<BF16, D, NC, KE>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(mk, G);
  return cudaGetLastError();
}

template <bool BF16, int D, int NC>
cudaError_t run_select_ke(int KE, const CUtensorMap& mk, const Geom& G, dim3 grid, int smem,
                          cudaStream_t st) {
  switch (KE) {
    case 1: return run_select<BF16, D, NC, 1>(mk, G, grid, smem, st);
    case 2: return run_select<BF16, D, NC, 2>(mk, G, grid, smem, st);
    case 4: return run_select<BF16, D, NC, 4>(mk, G, grid, smem, st);
    case 8: return run_select<BF16, D, NC, 8>(mk, G, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::select(int NC, int KE, const CUtensorMap& mk, const Geom& G,
                                      dim3 grid, int smem, cudaStream_t st) {
  switch (NC) {
    case 1: return run_select_ke<BF16, D, 1>(KE, mk, G, grid, smem, st);
    case 2: return run_select_ke<BF16, D, 2>(KE, mk, G, grid, smem, st);
    case 4: return run_select_ke<BF16, D, 4>(KE, mk, G, grid, smem, st);
    case 8: return run_select_ke<BF16, D, 8>(KE, mk, G, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int D, int NC>
cudaError_t run_excl(const CUtensorMap& mk, const Geom& G, dim3 grid, int smem, cudaStream_t st) {
  constexpr auto kern = &topo_excl_kernel<BF16, D, NC>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(mk, G);
  return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::excl(int NC, const CUtensorMap& mk, const Geom& G, dim3 grid,
                                    int smem, cudaStream_t st) {
  switch (NC) {
    case 1: return run_excl<BF16, D, 1>(mk, G, grid, smem, st);
    case 2: return run_excl<BF16, D, 2>(mk, G, grid, smem, st);
    case 4: return run_excl<BF16, D, 4>(mk, G, grid, smem, st);
    case 8: return run_excl<BF16, D, 8>(mk, G, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int D, int NC>
cudaError_t run_dense(const CUtensorMap& mk, const CUtensorMap& mv, const Geom& G, dim3 grid,
                      int smem, cudaStream_t st) {
  constexpr auto kern = &dense_kernel<BF16, D, NC>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(mk, mv, G);
  return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::dense(int NC, const CUtensorMap& mk, const CUtensorMap& mv,
                                     const Geom& G, dim3 grid, int smem, cudaStream_t st) {
  switch (NC) {
    case 1: return run_dense<BF16, D, 1>(mk, mv, G, grid, smem, st);
    case 2: return run_dense<BF16, D, 2>(mk, mv, G, grid, smem, st);
    case 4: return run_dense<BF16, D, 4>(mk, mv, G, grid, smem, st);
    case 8: return run_dense<BF16, D, 8>(mk, mv, G, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::pv(const Geom& G, long long nrows, cudaStream_t st) {
  const long long blocks = (nrows + 3) / 4;
  sparse_pv_kernel<BF16, D><<<(unsigned)blocks, 128, 0, st>>>(G);
  return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::compact(const Geom& G, void* k_out, void* v_out,
                                       cudaStream_t st) {
  const long long total = (long long)G.B * G.Hq * G.nq * (1 + (long long)G.W + G.topk) *
                          (Shape<BF16, D>::ROWB / 16);
  long long blocks = (total + 255) / 256;
  if (blocks > 148 * 16) blocks = 148 * 16;  // grid-stride beyond 16 blocks per SM
  if (blocks < 1) blocks = 1;
  compact_kv_kernel<BF16, D><<<(unsigned)blocks, 256, 0, st>>>(G, k_out, v_out);
  return cudaGetLastError();
}

template <int D, int NC, int KE, bool GROUP>
cudaError_t run_select_tc(const CUtensorMap& mk, const Geom& G, dim3 grid, int smem,
                          cudaStream_t st) {
  constexpr auto kern = &topo_select_tc_kernel<D, NC, KE, GROUP>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, smem, st>>>(mk, G);
  return cudaGetLastError();
}

template <int D, int NC, bool GROUP>
cudaError_t run_select_tc_ke(int KE, const CUtensorMap& mk, const Geom& G, dim3 grid, int smem,
                             cudaStream_t st) {
  if (KE == 1) return run_select_tc<D, NC, 1, GROUP>(mk, G, grid, smem, st);
  if constexpr (NC <= 4) {
    if (KE == 2) return run_select_tc<D, NC, 2, GROUP>(mk, G, grid, smem, st);
  }
  return cudaErrorInvalidValue;
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::select_tc(int NC, int KE, bool group, const CUtensorMap& mk128,
                                         const Geom& G, dim3 grid, int smem, cudaStream_t st) {
  if constexpr (!BF16) {
    return cudaErrorInvalidValue;
  } else {
    if (group) {
      // group-shared selection: at least two heads per selection column
      switch (NC) {
        case 2: return run_select_tc_ke<D, 2, true>(KE, mk128, G, grid, smem, st);
        case 4: return run_select_tc_ke<D, 4, true>(KE, mk128, G, grid, smem, st);
        case 8: return run_select_tc_ke<D, 8, true>(KE, mk128, G, grid, smem, st);
        case 16: return run_select_tc_ke<D, 16, true>(KE, mk128, G, grid, smem, st);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (NC) {
      case 1: return run_select_tc_ke<D, 1, false>(KE, mk128, G, grid, smem, st);
      case 2: return run_select_tc_ke<D, 2, false>(KE, mk128, G, grid, smem, st);
      case 4: return run_select_tc_ke<D, 4, false>(KE, mk128, G, grid, smem, st);
      case 8: return run_select_tc_ke<D, 8, false>(KE, mk128, G, grid, smem, st);
      case 16: return run_select_tc_ke<D, 16, false>(KE, mk128, G, grid, smem, st);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int D, int NC, int KE, bool GROUP>
cudaError_t run_tail_tc(const Geom& G, dim3 grid, int smem, int scratch_bytes, cudaStream_t st) {
  constexpr auto kern = &topo_tail_tc_kernel<D, NC, KE, GROUP>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, G, scratch_bytes);
}

template <int D, int NC, bool GROUP>
cudaError_t run_tail_tc_ke(int KE, const Geom& G, dim3 grid, int smem, int scratch_bytes,
                           cudaStream_t st) {
  if (KE == 1) return run_tail_tc<D, NC, 1, GROUP>(G, grid, smem, scratch_bytes, st);
  if constexpr (NC <= 4) {
    if (KE == 2) return run_tail_tc<D, NC, 2, GROUP>(G, grid, smem, scratch_bytes, st);
  }
  return cudaErrorInvalidValue;
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::tail_tc(int NC, int KE, bool group, const Geom& G, dim3 grid,
                                       int smem, int scratch_bytes, cudaStream_t st) {
  if constexpr (!BF16) {
    return cudaErrorInvalidValue;
  } else {
    if (group) {
      switch (NC) {
        case 2: return run_tail_tc_ke<D, 2, true>(KE, G, grid, smem, scratch_bytes, st);
        case 4: return run_tail_tc_ke<D, 4, true>(KE, G, grid, smem, scratch_bytes, st);
        case 8: return run_tail_tc_ke<D, 8, true>(KE, G, grid, smem, scratch_bytes, st);
        case 16: return run_tail_tc_ke<D, 16, true>(KE, G, grid, smem, scratch_bytes, st);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (NC) {
      case 1: return run_tail_tc_ke<D, 1, false>(KE, G, grid, smem, scratch_bytes, st);
      case 2: return run_tail_tc_ke<D, 2, false>(KE, G, grid, smem, scratch_bytes, st);
      case 4: return run_tail_tc_ke<D, 4, false>(KE, G, grid, smem, scratch_bytes, st);
      case 8: return run_tail_tc_ke<D, 8, false>(KE, G, grid, smem, scratch_bytes, st);
      case 16: return run_tail_tc_ke<D, 16, false>(KE, G, grid, smem, scratch_bytes, st);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int D, int NC>
cudaError_t run_dense_tc(const CUtensorMap& mk, const CUtensorMap& mv, const Geom& G, dim3 grid,
                         int smem, cudaStream_t st) {
  constexpr auto kern = &dense_tc_kernel<D, NC>;
  const cudaError_t e = allow_smem<kern>();
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, smem, st>>>(mk, mv, G);
  return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::dense_tc(int NC, const CUtensorMap& mk128,
                                        const CUtensorMap& mv128, const Geom& G, dim3 grid,
                                        int smem, cudaStream_t st) {
  if constexpr (!BF16) {
    return cudaErrorInvalidValue;
  } else {
    switch (NC) {
      case 1: return run_dense_tc<D, 1>(mk128, mv128, G, grid, smem, st);
      case 2: return run_dense_tc<D, 2>(mk128, mv128, G, grid, smem, st);
      case 4: return run_dense_tc<D, 4>(mk128, mv128, G, grid, smem, st);
      case 8: return run_dense_tc<D, 8>(mk128, mv128, G, grid, smem, st);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <bool BF16, int D>
cudaError_t Launcher<BF16, D>::prefill(const CUtensorMap& mk128, const Geom& G, int scan_grid,
                                       int scan_smem, int kmax_grid, bool do_pv,
                                       cudaStream_t st) {
  if constexpr (!BF16) {
    return cudaErrorInvalidValue;
  } else {
    const dim3 gk((unsigned)kmax_grid, (unsigned)(G.B * G.Hkv));
    prefill_kmax_kernel<D><<<gk, 256, 0, st>>>(G);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr auto scan = &prefill_scan_kernel<D>;
    e = allow_smem<scan>();
    if (e != cudaSuccess) return e;
    scan<<<scan_grid, kPfThreads, scan_smem, st>>>(mk128, G);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long ncolumns = (long long)G.B * G.Hkv * G.ncols;
    prefill_finalize_kernel<D><<<(unsigned)((ncolumns + 3) / 4), 128, 0, st>>>(G);
    e = cudaGetLastError();
    if (e != cudaSuccess || !do_pv) return e;
    const int pb_smem = PbSmem(D, G.W).total;
    if (pb_smem <= kMaxSmem) {
      // the window band of a block of rows fits in shared memory
      constexpr auto band = &prefill_pv_band_kernel<D>;
      e = allow_smem<band>();
      if (e != cudaSuccess) return e;
      const dim3 gb((unsigned)((G.nq + kPbRows - 1) / kPbRows), (unsigned)G.Hkv, (unsigned)G.B);
      band<<<gb, kPbWarps * 32, pb_smem, st>>>(G);
      return cudaGetLastError();
    }
    prefill_pv_kernel<D><<<(unsigned)((ncolumns + 3) / 4), 128, 0, st>>>(G);
    return cudaGetLastError();
  }
}

extern template struct Launcher<false, 64>;
extern template struct Launcher<false, 128>;
extern template struct Launcher<true, 64>;
extern template struct Launcher<true, 128>;

}  // namespace topo

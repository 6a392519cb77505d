// launch_table.cuh -- compile-time table of gemv_kernel<F, M>, M = 1..16.
// M is a template parameter so every accumulator lives in registers; the
// host picks the instantiation per call (no per-M compilation at run time).
#pragma once

#include <cuda_runtime.h>

#include "gemv_kernel.cuh"
#include "tc_kernel.cuh"

namespace qgemv {

template <class F>
struct LaunchTable {
  // Launched with programmatic stream serialization: the kernel may start
  // while the previous kernel on the stream drains; it runs its prologue
  // (barriers, tables, first weight copies) and then waits on the previous
  // grid (griddepcontrol.wait) before reading x or writing anything.
  template <int M>
  static cudaError_t launch_m(const GemvParams& p, int grid, cudaStream_t s) {
    // 227 KB per CTA, less room for the kernel's few static bytes
    static_assert(gemv_smem_bytes<F, M>() <= 227 * 1024 - 256, "shared memory budget exceeded");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(gemv_threads<M>());
    cfg.dynamicSmemBytes = gemv_smem_bytes<F, M>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<F, M>, p);
  }

  template <int M>
  static cudaError_t setup_m() {
    return cudaFuncSetAttribute(gemv_kernel<F, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gemv_smem_bytes<F, M>());
  }

  static int smem_bytes(int M) {
    switch (M) {
#define QGEMV_CASE(m) \
  case m:             \
    return gemv_smem_bytes<F, m>();
      QGEMV_CASE(1) QGEMV_CASE(2) QGEMV_CASE(3) QGEMV_CASE(4) QGEMV_CASE(5) QGEMV_CASE(6)
      QGEMV_CASE(7) QGEMV_CASE(8) QGEMV_CASE(9) QGEMV_CASE(10) QGEMV_CASE(11) QGEMV_CASE(12)
      QGEMV_CASE(13) QGEMV_CASE(14) QGEMV_CASE(15) QGEMV_CASE(16)
#undef QGEMV_CASE
    }
    return 0;
  }

  static cudaError_t setup() {
    cudaError_t e = cudaSuccess;
#define QGEMV_SETUP(m) \
  if (e == cudaSuccess) e = setup_m<m>();
    QGEMV_SETUP(1) QGEMV_SETUP(2) QGEMV_SETUP(3) QGEMV_SETUP(4) QGEMV_SETUP(5) QGEMV_SETUP(6)
    QGEMV_SETUP(7) QGEMV_SETUP(8) QGEMV_SETUP(9) QGEMV_SETUP(10) QGEMV_SETUP(11) QGEMV_SETUP(12)
    QGEMV_SETUP(13) QGEMV_SETUP(14) QGEMV_SETUP(15) QGEMV_SETUP(16)
#undef QGEMV_SETUP
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemv_tc_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem_bytes<F>());
    return e;
  }

  // M >= kTcMinM runs on the tensor cores (tc_kernel.cuh): one kernel for
  // every such M, the activations padded to 16 rows.
  static constexpr int kTcMinM = 5;

  static cudaError_t launch_tc(const GemvParams& p, int M, int grid, cudaStream_t s) {
    static_assert(tc_smem_bytes<F>() <= 227 * 1024 - 256, "shared memory budget exceeded");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_smem_bytes<F>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_tc_kernel<F>, p, M);
  }

  static cudaError_t launch(int M, const GemvParams& p, int grid, cudaStream_t s) {
    if (M >= kTcMinM && M <= kMaxM) return launch_tc(p, M, grid, s);
    switch (M) {
#define QGEMV_LAUNCH(m) \
  case m:               \
    return launch_m<m>(p, grid, s);
      QGEMV_LAUNCH(1) QGEMV_LAUNCH(2) QGEMV_LAUNCH(3) QGEMV_LAUNCH(4) QGEMV_LAUNCH(5)
      QGEMV_LAUNCH(6) QGEMV_LAUNCH(7) QGEMV_LAUNCH(8) QGEMV_LAUNCH(9) QGEMV_LAUNCH(10)
      QGEMV_LAUNCH(11) QGEMV_LAUNCH(12) QGEMV_LAUNCH(13) QGEMV_LAUNCH(14) QGEMV_LAUNCH(15)
      QGEMV_LAUNCH(16)
#undef QGEMV_LAUNCH
    }
    return cudaErrorInvalidValue;
  }
};

}  // namespace qgemv

// launch_table.cuh -- the kernels of a tile format and the choice between
// them by M (no per-M compilation at run time).
#pragma once

#include <cuda_runtime.h>

#include "gemv_kernel.cuh"
#include "mma_kernel.cuh"
#include "rowgroup_kernel.cuh"
#include "tc5_kernel.cuh"

namespace qgemv {

// M = 1: the CUDA-core kernel (gemv_kernel.cuh), or for table formats whose
// handle chose it the row-group kernel (rowgroup_kernel.cuh).  M = 2..16: the
// tensor-core kernel with register-level decode (mma_kernel.cuh), one
// activation block of 8 rows up to M = 8 (tile-parity geometry where the
// format has it), two above.  The tensor-core kernel computes every
// activation row on its own (a column of the MMA's B operand, the same
// instruction sequence, reduction tree and fix-up order for any M), so in
// batch-invariant mode M = 1 runs there too and a row's bits never depend on
// how many rows share the call.
template <class F>
struct LaunchTable {
  // Launched with programmatic stream serialization: the kernel may start
  // while the previous kernel on the stream drains; it runs its prologue
  // (barriers, tables, first weight copies) and then waits on the previous
  // grid (griddepcontrol.wait) before reading x or writing anything.
  static cudaLaunchConfig_t config(int grid, int threads, int smem, cudaStream_t s, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
  }

  static constexpr int kM1CtasPerSm = F::kCtasPerSm;

  static cudaError_t launch_m1(const RunParams& p, int grid, cudaStream_t s) {
    // 227 KB per SM shared by the CTAs, less room for each one's reserved and static bytes
    static_assert(F::kCtasPerSm * (gemv_smem_bytes<F, 1>() + 2048) <= 228 * 1024, "shared memory budget exceeded");
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = config(grid, gemv_threads<F, 1>(), gemv_smem_bytes<F, 1>(), s, attr);
    return cudaLaunchKernelEx(&cfg, wstream_kernel<F, 1>, p);
  }

  // The tensor-core kernel runs F::mma_ctas(NB) CTAs per SM: 1 (grid, plan)
  // or as many as the M = 1 kernel (grid_m1, plan_m1).  PAR: the tile-parity
  // geometry (F::mma_par), used for one activation block outside
  // batch-invariant mode.
  template <int NB, bool PAR = false>
  static cudaError_t launch_mma(const RunParams& p, int M, const LaunchGeom& g, cudaStream_t s) {
    static_assert(F::mma_ctas(NB) == 1 || F::mma_ctas(NB) == F::kCtasPerSm, "tensor-core grid");
    // batch invariance: both activation-block counts of the default geometry
    // are the same geometry
    static_assert(F::mma_ctas(1) == F::mma_ctas(2) && F::mma_spw(1) == F::mma_spw(2), "one geometry for all M");
    static_assert(F::mma_ctas(NB) * (mma_smem_bytes<F, NB, PAR>() + 2048) <= 228 * 1024,
                  "shared memory budget exceeded");
    RunParams q = p;
    q.plan = F::mma_ctas(NB) == 1 ? g.plan : g.plan_m1;
    const int grid = F::mma_ctas(NB) == 1 ? g.grid : g.grid_m1;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = config(grid, mma_threads<F, NB, PAR>(), mma_smem_bytes<F, NB, PAR>(), s, attr);
    return cudaLaunchKernelEx(&cfg, wstream_mma_kernel<F, NB, PAR>, q, M);
  }

  // M = 1, whole 32-row groups per CTA (table formats; the handle decides,
  // LaunchGeom::grid_rg).
  static cudaError_t launch_rg(const RunParams& p, int grid, cudaStream_t s) {
    static_assert(rg_smem_bytes<F>() + 2048 <= 228 * 1024, "shared memory budget exceeded");
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = config(grid, kRgThreads, rg_smem_bytes<F>(), s, attr);
    return cudaLaunchKernelEx(&cfg, rowgroup_stream_kernel<F>, p);
  }

  // GLU handles (gate and up interleaved; the GLU epilogues): M = 1 on the
  // CUDA-core kernel, on the M = 1 grid and its plan (made with 64-row
  // halves); M >= 2 in one launch of the tensor-core kernel for formats that
  // have its GLU form (F::kMmaGlu), else the CUDA-core kernel once per
  // activation row.
  static constexpr bool kMmaGlu = MmaGluOf<F>::value;
  static cudaError_t setup_glu() {
    cudaError_t e = cudaFuncSetAttribute(wstream_kernel<F, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gemv_smem_bytes<F, 1>());
    if constexpr (kMmaGlu) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wstream_mma_kernel<F, 1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 mma_smem_bytes<F, 1>());
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wstream_mma_kernel<F, 2, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 mma_smem_bytes<F, 2>());
    }
    return e;
  }
  template <int NB>
  static cudaError_t launch_mma_glu(const RunParams& p, int M, const LaunchGeom& g, cudaStream_t s) {
    RunParams q = p;
    q.residual = nullptr;
    q.plan = F::mma_ctas(NB) == 1 ? g.plan : g.plan_m1;
    const int grid = F::mma_ctas(NB) == 1 ? g.grid : g.grid_m1;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = config(grid, mma_threads<F, NB>(), mma_smem_bytes<F, NB>(), s, attr);
    return cudaLaunchKernelEx(&cfg, wstream_mma_kernel<F, NB, false, true>, q, M);
  }
  static cudaError_t launch_glu(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s) {
    if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
    if constexpr (kMmaGlu) {
      if (M >= 2) return M <= 8 ? launch_mma_glu<1>(p, M, g, s) : launch_mma_glu<2>(p, M, g, s);
    }
    for (int m = 0; m < M; ++m) {
      RunParams q = p;
      q.x = p.x + m * p.K;
      q.y = p.y + m * (p.N / 2);
      q.residual = nullptr;
      q.plan = g.plan_m1;
      cudaLaunchAttribute attr[1];
      const cudaLaunchConfig_t cfg = config(g.grid_m1, gemv_threads<F, 1>(), gemv_smem_bytes<F, 1>(), s, attr);
      const cudaError_t e = cudaLaunchKernelEx(&cfg, wstream_kernel<F, 1, true>, q);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }

  // The tensor-memory kernel (tc5_kernel.cuh; one CTA per SM, the handle's
  // grid and plan), for the formats that have it: MT = 8 accumulator columns
  // read back up to M = 8, 16 above.
  template <int MT>
  static cudaError_t launch_tc5(const RunParams& p, int M, const LaunchGeom& g, cudaStream_t s) {
    static_assert(tc5_smem_bytes<F, MT>() + 2048 <= 228 * 1024, "shared memory budget exceeded");
    RunParams q = p;
    q.plan = g.plan;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = config(g.grid, kTc5Threads, tc5_smem_bytes<F, MT>(), s, attr);
    return cudaLaunchKernelEx(&cfg, tc5_kernel<F, MT>, q, M);
  }

  static int smem_bytes(int M) {
    if (M == 1) return gemv_smem_bytes<F, 1>();
    if (M >= 2 && M <= 8) return F::mma_par(1) ? mma_smem_bytes<F, 1, true>() : mma_smem_bytes<F, 1>();
    if (M > 8 && M <= kMaxM) return mma_smem_bytes<F, 2>();
    return 0;
  }

  static cudaError_t setup() {
    cudaError_t e = cudaFuncSetAttribute(wstream_kernel<F, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gemv_smem_bytes<F, 1>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wstream_mma_kernel<F, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mma_smem_bytes<F, 1>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wstream_mma_kernel<F, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mma_smem_bytes<F, 2>());
    if constexpr (F::mma_par(1)) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wstream_mma_kernel<F, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 mma_smem_bytes<F, 1, true>());
    }
    if constexpr (F::kTileParity) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rowgroup_stream_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 rg_smem_bytes<F>());
    }
    if constexpr (Tc5<F>::kHas) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc5_kernel<F, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, tc5_smem_bytes<F, 8>());
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc5_kernel<F, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc5_smem_bytes<F, 16>());
    }
    return e;
  }

  static cudaError_t launch(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s,
                            bool batch_invariant) {
    RunParams q = p;
    if constexpr (Tc5<F>::kHas) {
      if (!batch_invariant && g.tc5_min_m > 0 && M >= g.tc5_min_m && M <= kMaxM)
        return M <= 8 ? launch_tc5<8>(q, M, g, s) : launch_tc5<16>(q, M, g, s);
    }
    if (M == 1 && !batch_invariant) {
      if constexpr (F::kTileParity) {
        if (g.grid_rg > 0) return launch_rg(q, g.grid_rg, s);
      }
      q.plan = g.plan_m1;
      return launch_m1(q, g.grid_m1, s);
    }
    if (M >= 1 && M <= 8) {
      if constexpr (F::mma_par(1)) {
        if (!batch_invariant) return launch_mma<1, true>(q, M, g, s);
      }
      return launch_mma<1>(q, M, g, s);
    }
    if (M > 8 && M <= kMaxM) return launch_mma<2>(q, M, g, s);
    return cudaErrorInvalidValue;
  }
};

}  // namespace qgemv

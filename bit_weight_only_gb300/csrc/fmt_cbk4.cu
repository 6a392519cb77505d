// fmt_cbk4.cu -- CBK4 (4-bit index into 16 fp16 centroids): re-layout,
// exact decode export and the GEMV launch table for M = 1..16.
#include "fmt_cbk.cuh"
#include "formats.h"
#include "launch_table.cuh"

namespace qgemv {
namespace {

using F = FmtCBK4;

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t nchunks = a.nRT * a.nKT * kRowsPerLane * 2 * kLaneSlots;
  cbk::prepare_kernel<F, 4><<<cbk::grid_for(nchunks, 256), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT,
                                                                       nchunks, a.tiles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.seg_of_rt == nullptr)  // one codebook (a GLU handle: the gate's, then the up's)
    return cudaMemcpyAsync(a.aux, a.codebooks, (a.glu ? 2 : 1) * 16 * sizeof(uint16_t), cudaMemcpyDeviceToDevice, s);
  cbk::expand_codebooks_kernel<16><<<cbk::grid_for(a.nRT * 16, 256), 256, 0, s>>>(
      a.codebooks, a.seg_of_rt, a.nRT, static_cast<uint16_t*>(a.aux));
  return cudaGetLastError();
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t* seg_of_rt, int64_t N, int64_t K,
                    int nKT, float* w, int glu, cudaStream_t s) {
  cbk::dequant_kernel<F, 4><<<cbk::grid_for(N * K, 256), 256, 0, s>>>(
      tiles, static_cast<const uint16_t*>(aux), seg_of_rt ? 16 : 0, glu ? 16 : 0, N, K, nKT, w);
  return cudaGetLastError();
}

// the regular launches and the GLU handles' kernels
cudaError_t setup_all() {
  cudaError_t e = LaunchTable<F>::setup();
  if (e == cudaSuccess) e = LaunchTable<F>::setup_glu();
  return e;
}

}  // namespace

const FormatOps* ops_cbk4() {
  static const FormatOps ops = {
      /*format=*/2, F::kKT, F::kTileBytes, /*aux_bytes=*/0,
      &LaunchTable<F>::smem_bytes, &setup_all, &LaunchTable<F>::launch,
      &prepare, &dequant, /*cb_entries=*/16, /*tile_rows=*/128, /*partial_stride=*/128 * 16,
      /*aux_per_row=*/0, /*m1_ctas_per_sm=*/LaunchTable<F>::kM1CtasPerSm,
      /*rowgroup=*/1, /*launch_x_int8=*/nullptr, /*row_tables=*/0, /*launch_xq=*/nullptr,
      /*launch_glu=*/&LaunchTable<F>::launch_glu, /*tc5_min_m=*/kTc5DefaultMinM, /*split_unit=*/SplitModeOf<F>::value};
  return &ops;
}

}  // namespace qgemv

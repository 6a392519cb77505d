// fmt_cbk4row.cu -- CBK4 with one fp32 codebook of 16 centroids per output
// row (FmtCBK4R): re-layout, exact decode export and the launches.
//
// Canonical input: indices as CBK4 (uint8 [N][K/2], k = 2j in the low
// nibble of byte j); codebooks fp32 [N][16], row n's 16 centroids together.
// Prepared: the CBK4 tiles, and the codebooks padded with zero rows to whole
// row tiles (row tile rt's 8 KB at aux + rt * 8 KB) with seg_of_rt[rt] = rt,
// so the CUDA-core kernel rebuilds its shared table at every row tile.
//
// The weights are fp32 centroids, which the f16 tensor-core path cannot
// take exactly, so every M runs the CUDA-core kernel: eight, two or one
// activation rows per launch (the weights are read once per launch).  A
// row's arithmetic is the same in the one- and two-row instantiations;
// the eight-row one adds the slices in another order (batch-invariant mode
// does not use it).
#include "fmt_cbk.cuh"
#include "formats.h"
#include "launch_table.cuh"

namespace qgemv {
namespace {

using F = FmtCBK4R;
constexpr int64_t kRowTileCbBytes = int64_t(kTileRows) * 16 * 4;  // 8 KB

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t nchunks = a.nRT * a.nKT * kRowsPerLane * 2 * kLaneSlots;
  cbk::prepare_kernel<F, 4><<<cbk::grid_for(nchunks, 256), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT,
                                                                       nchunks, a.tiles);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemsetAsync(a.aux, 0, a.nRT * kRowTileCbBytes, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(a.aux, a.codebooks, a.N * 16 * 4, cudaMemcpyDeviceToDevice, s);
  return e;
}

// w[n][k] = centroid idx(n, k) of row n, exact.
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, const float* __restrict__ cb, int64_t N,
                               int64_t K, int nKT, float* __restrict__ w) {
  const int64_t total = N * K;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = e / K, k = e % K;
    const int r = static_cast<int>(n % kTileRows);
    const int lane = r / kRowsPerLane, j = r % kRowsPerLane;
    const int64_t tile = (n / kTileRows) * nKT + k / F::kKT;
    const int kk = static_cast<int>(k % F::kKT);
    const int cw = kk / F::kKW, el = kk % F::kKW;
    const int byte_in_row = el / 2;  // 0..31
    const int h = byte_in_row / 16;
    const uint8_t byte = tiles[tile * F::kTileBytes + ((j * 2 + h) * kLaneSlots + cw * 32 + lane) * 16 +
                               byte_in_row % 16];
    const int idx = (el & 1) ? (byte >> 4) : (byte & 15);
    w[e] = cb[n * 16 + idx];
  }
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t*, int64_t N, int64_t K, int nKT,
                    float* w, int, cudaStream_t s) {
  dequant_kernel<<<cbk::grid_for(N * K, 256), 256, 0, s>>>(tiles, static_cast<const float*>(aux), N, K, nKT,
                                                           w);
  return cudaGetLastError();
}

template <int MB>
cudaError_t set_smem() {
  static_assert(gemv_smem_bytes<F, MB>() + 2048 <= 228 * 1024, "shared memory budget exceeded");
  return cudaFuncSetAttribute(wstream_kernel<F, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              gemv_smem_bytes<F, MB>());
}

cudaError_t setup() {
  cudaError_t e = set_smem<1>();
  if (e == cudaSuccess) e = set_smem<2>();
  if (e == cudaSuccess) e = set_smem<8>();
  if (e == cudaSuccess) e = LaunchTable<F>::setup_glu();
  return e;
}

int smem_bytes(int M) {
  return M == 1 ? gemv_smem_bytes<F, 1>() : (M < 8 ? gemv_smem_bytes<F, 2>() : gemv_smem_bytes<F, 8>());
}

template <int MB>
cudaError_t launch_rows(const RunParams& p, int m0, const LaunchGeom& g, cudaStream_t s) {
  RunParams q = p;
  q.x = p.x + m0 * p.K;
  q.y = p.y + m0 * p.N;
  q.residual = p.residual != nullptr ? p.residual + m0 * p.N : nullptr;
  q.plan = g.plan_m1;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      LaunchTable<F>::config(g.grid_m1, gemv_threads<F, MB>(), gemv_smem_bytes<F, MB>(), s, attr);
  return cudaLaunchKernelEx(&cfg, wstream_kernel<F, MB>, q);
}

// Eight activation rows per launch while eight remain (eight warps, one per
// slice, 248 registers), then two, then one for an odd last row (sixteen
// warps in tile parity).  The two geometries add a row's slices in
// different orders; batch-invariant mode keeps to the second, so that a
// row's bits never depend on M.
cudaError_t launch(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  for (int m0 = 0; m0 < M;) {
    const int mb = (M - m0 >= 8 && !batch_invariant) ? 8 : (M - m0 >= 2 ? 2 : 1);
    const cudaError_t e = mb == 8   ? launch_rows<8>(p, m0, g, s)
                          : mb == 2 ? launch_rows<2>(p, m0, g, s)
                                    : launch_rows<1>(p, m0, g, s);
    if (e != cudaSuccess) return e;
    m0 += mb;
  }
  return cudaSuccess;
}

}  // namespace

const FormatOps* ops_cbk4_row() {
  static const FormatOps ops = {
      /*format=*/8, F::kKT, F::kTileBytes, /*aux_bytes=*/0,
      &smem_bytes, &setup, &launch, &prepare, &dequant, /*cb_entries=*/F::kCbEntries, /*tile_rows=*/128,
      /*partial_stride=*/128 * 16, /*aux_per_row=*/0, /*m1_ctas_per_sm=*/F::kCtasPerSm, /*rowgroup=*/0,
      /*launch_x_int8=*/nullptr, /*row_tables=*/1, /*launch_xq=*/nullptr,
      /*launch_glu=*/&LaunchTable<F>::launch_glu, /*tc5_min_m=*/0, /*split_unit=*/SplitModeOf<F>::value};
  return &ops;
}

}  // namespace qgemv

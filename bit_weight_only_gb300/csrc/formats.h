// formats.h -- internal interface between the C ABI (qgemv_api.cu) and the
// per-format translation units.  Host-side declarations only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qgemv {

struct RunParams;
struct CtaPlan;  // gemv_kernel.cuh

// Canonical inputs already on the device, plus the prepared-layout geometry.
struct PrepareArgs {
  const uint8_t* packed;     // canonical packed bytes
  const uint16_t* scales;    // canonical fp16 scales or nullptr
  const uint16_t* codebooks; // canonical fp16 codebooks or nullptr
  int64_t N, K;
  int64_t nRT;               // row tiles
  int nKT;                   // k tiles per row tile
  uint8_t* tiles;            // out: nRT * nKT * tile_bytes
  void* aux;                 // out: format data (aux_bytes), may be nullptr
  int nseg;                  // codebooks (stacked handles; 1 otherwise)
  const int32_t* seg_of_rt;  // device [nRT] codebook of each row tile, or nullptr
  int glu = 0;               // GLU handle of a one-codebook format: codebooks = gate's, then up's
};

// Grids and stream-K plans of a handle: `grid`/`plan` for the tensor-core and
// AQLM kernels (one CTA per SM), `grid_m1`/`plan_m1` for the M = 1 CUDA-core
// kernel, which runs F::kCtasPerSm CTAs per SM (the same arrays when 1).
struct LaunchGeom {
  int grid;
  const CtaPlan* plan;
  int grid_m1;
  const CtaPlan* plan_m1;
  int grid_rg;  // M = 1 row-group kernel (table formats, whole rows per CTA): its grid, 0 if not used
  int tc5_min_m;  // calls with at least this many rows run the tensor-memory kernel (0: never)
};

struct FormatOps {
  int format;
  int kt;          // k per tile
  int tile_bytes;  // bytes per prepared tile
  int64_t aux_bytes;
  int (*smem_bytes)(int M);
  cudaError_t (*setup)();  // one-time kernel attributes
  // batch_invariant: every row's result must not depend on M (see
  // qgemv_set_batch_invariant); the kernels are chosen accordingly.
  cudaError_t (*launch)(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant);
  cudaError_t (*prepare)(const PrepareArgs& a, cudaStream_t s);
  // w_out[n*K + k] = exact decoded weight, read back from the prepared tiles
  // glu: a GLU handle of a one-codebook format (aux holds the gate then the
  // up codebook; rows 64..127 of every tile use the second)
  cudaError_t (*dequant)(const uint8_t* tiles, const void* aux, const int32_t* seg_of_rt, int64_t N,
                         int64_t K, int nKT, float* w_out, int glu, cudaStream_t s);
  int cb_entries = 0;               // fp16 entries per codebook (CBK4 16, CBK8 256)
  int tile_rows = 128;              // output rows per prepared tile
  int64_t partial_stride = 128 * 16;  // floats per stream-K partial slot
  int64_t aux_per_row = 0;          // aux bytes per output row, after aux_bytes
  int m1_ctas_per_sm = 1;           // CTAs per SM of the M = 1 kernel (LaunchGeom::grid_m1)
  int rowgroup = 0;                 // has the M = 1 row-group kernel (rowgroup_kernel.cuh)
  // PQ2_0 only: the run with INT8 activations (qgemv_set_x_int8), else nullptr
  cudaError_t (*launch_x_int8)(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s,
                               bool batch_invariant) = nullptr;
  // one codebook table per row tile, built from per-row codebooks (CBK4_ROW):
  // aux holds cb_entries fp16-sized units per row tile and seg_of_rt[rt] = rt
  int row_tables = 0;
  // PQ2_0 only: the run on prepared INT8 activations (qgemv_run_xq), else nullptr
  cudaError_t (*launch_xq)(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s,
                           bool batch_invariant) = nullptr;
  // Q4_0, PQ2_0: the fused SiLU(gate) * up run of a GLU handle (qgemv_create_glu), else nullptr
  cudaError_t (*launch_glu)(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s) = nullptr;
  // formats with the tensor-memory kernel (tc5_kernel.cuh): the smallest M
  // that runs it by default (0: not by default)
  int tc5_min_m = 0;
  // the stream-K split (stream_split): 0 spread, 1 or 2 front-loaded chunks;
  // the kernels' formula is the format's compile-time F::kSplitMode.
  // Measured (same box): front-loaded single tiles gain 2.5% on the 7B CBK4
  // stack (3% at M = 8), 7.5% on CBK4 11008x4096 and 11% on the PQ2_0
  // 5120/17408 model's projections at M = 1; Q4_0 is even at M = 1 and 2.7%
  // slower at M = 8, AQLM 2x8 12% slower: those two keep the spread.  Pairs
  // of tiles were no better than the spread for the tile-parity formats.
  int split_unit = 0;
};

// The formats that have the tensor-memory kernel (tc5_kernel.cuh).
inline bool has_tc5(int format) { return format >= 1 && format <= 4; }  // Q4_0, CBK4, CBK8, PQ2_0

const FormatOps* ops_q4_0();
const FormatOps* ops_pq2();
const FormatOps* ops_cbk4();
const FormatOps* ops_cbk8();
const FormatOps* ops_aqlm();
const FormatOps* ops_aqlm_mma();  // internal: the AQLM tensor-core layout
const FormatOps* ops_aqlm_1x16();
const FormatOps* ops_cbk4_row();
const FormatOps* ops_cbk8_row();

// Record the calling thread's last error (what qgemv_last_error returns);
// returns `code`.  QGEMV_OK clears it.
int report_error(int code, const char* msg);

// PQ2_0 INT8 activation quantizer: x fp16 [M][K] (K % 128 == 0) -> q int8
// [M][K], a fp32 [M][K/128]; the GEMV's own staging arithmetic.
cudaError_t quantize_x_int8(const void* x, int64_t M, int64_t K, int8_t* q, float* a, cudaStream_t s);

// PQ2_0 activation prologue: INT8 codes (staging order), scales and code
// sums of x fp16 [M][K] into xq (qgemv_xq_bytes), after the Hadamard mixing
// of blocks of hadamard_block (0: none, or 1024) with optional signs [K].
cudaError_t prepare_x_int8(const void* x, int64_t M, int64_t K, const int8_t* signs, int hadamard_block,
                           void* xq, cudaStream_t s);

// Q4_0 quantizer (canonical output).
cudaError_t quantize_q4_0(const float* w, int64_t N, int64_t K, uint8_t* out, cudaStream_t s);

}  // namespace qgemv

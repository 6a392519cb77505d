// fmt_aqlm_mma.cu -- AQLM 2x8 on the tensor cores, for calls with several
// activation rows.
//
// Same decoded weight as fmt_aqlm.cu ("Trapetum benchmarks", additive vector
// quantization):  w[n][8g + j] = s_n * (C0[c0(n, g)][j] + C1[c1(n, g)][j]).
// The per-group table path costs one table read per code byte and
// activation row, so its time grows with M.  Here the codebook vectors are
// the A operands of mma.m16n8k16 instead (wstream_mma_kernel, mma_kernel.cuh):
//
//     y[m][n] = s_n * sum_g ( <C0[c0(n, g)], x[m]_g> + <C1[c1(n, g)], x[m]_g> )
//
// with one MMA per codebook into the same fp32 accumulator, so every operand
// is an exact fp16 value (the two codebooks are never added in fp16), and
// the row scale multiplies the row's sum when it is stored.  The cost per
// code byte is two 8-byte table reads, whatever M is (up to 16).
//
// Tile: 128 rows x 1024 k (128 groups).  Slice s <-> groups 16s .. 16s+15;
// lane slot t = 32s + l <-> rows 4l .. 4l+3.  Codes [j][t][32 B]: the 32
// code bytes of row 4l + j for the slice, byte 16h + 2ks + cb = code cb of
// group 2ks + h of the slice.
//
// Fragment order.  The k16 step ks of a slice covers groups 2ks and 2ks+1.
// Fragment thread q (lane & 3) takes group 2ks + (q >> 1), weights
// j0 = 4 (q & 1) .. j0 + 3, in its fragment k slots (2q, 2q+1, 2q+8, 2q+9):
// k = 16 ks + 4q .. +3 of the slice, so its B fragment is x[16ks + 4q .. +3],
// one 8-byte load, and its A fragment pair of a row is one 8-byte table
// read.  Thread q loads the 16 code bytes of half q >> 1 of its rows.
//
// Table (64 KB on a 64 KB boundary of the shared window): entry e of
// codebook cb, copy r = 0..3, at byte  e * 256 + cb * 128 + r * 32, holds
// C_cb[e][0..7] twice.  Thread (gi, q) reads 8 bytes at
// e * 256 + cb * 128 + (gi & 3) * 32 + q * 8 = C_cb[e][4 (q & 1) .. +3]; the
// 16 lanes of each half-warp hit 16 distinct 8-byte slots of one 128-byte
// line whatever the codes, so the reads are conflict-free.  One byte
// permute of the code byte with the lane's key is the whole address.
#include "formats.h"
#include "mma_kernel.cuh"

namespace qgemv {
namespace {

struct FmtAQLM {
  static constexpr int kKW = 128;
  static constexpr int kKT = kKW * kSlices;                          // 1024
  static constexpr int kTileBytes = kLaneSlots * kRowsPerLane * 32;  // 32768
  static constexpr int kCtasPerSm = 1;
  static constexpr int kCbEntries = 0;  // one codebook pair per handle (no stacking)
  static constexpr int kCodebookBytes = 2 * 256 * 8 * 2;

  static constexpr int kMmaSharedBytes = kTableAlign;
  static constexpr int kMmaRowWords = 4;  // the 16 code bytes of the thread's half of the row
  static constexpr bool kMmaLateCodes = true;  // two activation blocks: one m-tile's codes live at a time
  static constexpr int kMmaCodebooks = 2;
  static constexpr bool kMmaRowScales = true;
  __device__ static const __half* mma_row_scales(const RunParams& p) {
    return reinterpret_cast<const __half*>(static_cast<const uint8_t*>(p.aux) + kCodebookBytes);
  }
  static constexpr int kMmaBlockSteps = 0;
  struct MmaScales {};
  static constexpr int kMmaXWords = 16;  // x[m][16 ks + 4q .. +3], ks = 0..7
  __host__ __device__ static constexpr int mma_spw(int) { return 1; }
  __host__ __device__ static constexpr int mma_ctas(int) { return 1; }
  // one activation block: tile parity (two halves of eight warps, alternate tiles)
  __host__ __device__ static constexpr bool mma_par(int nb) { return nb == 1; }
  __host__ __device__ static constexpr int mma_stages(int nb) { return nb == 1 ? 4 : 3; }
  __host__ __device__ static constexpr bool mma_prefetch_x(int) { return false; }  // registers (no gain measured)

  // table >> 16 in byte 2; (gi & 3) * 32 + q * 8 in byte 0 (codebook 1: + 128)
  __device__ static uint32_t mma_lut_key(uint32_t table, int lane) {
    return (table & 0xFFFF0000u) | static_cast<uint32_t>(((lane >> 2) & 3) * 32 + (lane & 3) * 8);
  }

  // 8192 eight-byte words; word v = 32 e + 16 cb + 4 r + 2 d + hh holds
  // C_cb[e][4 hh .. 4 hh + 3] (copy r, duplicate d).  Consecutive threads
  // store consecutive words: no bank conflict.
  template <int NT>
  __device__ static void mma_init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    for (int v = warp * 32 + lane; v < 8192; v += NT) {
      const int e = v >> 5, cbi = (v >> 4) & 1, hh = v & 1;
      const uint2 val = __ldg(reinterpret_cast<const uint2*>(cb + (cbi * 256 + e) * 8 + 4 * hh));
      *reinterpret_cast<uint2*>(lut + v * 8) = val;
    }
  }

  __device__ static void mma_load_row(const uint8_t* stage, int slice, int l, int j, int q, uint32_t (&w)[4]) {
    const int t = slice * 32 + l;
    const uint4 v = *reinterpret_cast<const uint4*>(stage + (j * kLaneSlots + t) * 32 + (q >> 1) * 16);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }

  // (C_cb[c][j0], C_cb[c][j0+1]) and (C_cb[c][j0+2], C_cb[c][j0+3]) of the
  // row's group of step ks: fragment k slots (2q, 2q+1) and (2q+8, 2q+9)
  __device__ static uint2 mma_frag(const uint32_t (&w)[4], int ks, uint32_t lut_key, int cb) {
    const uint32_t addr = lut_addr(w[ks >> 1], lut_key + 128u * cb, 2 * (ks & 1) + cb);
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
  }

  __device__ static void mma_load_x(uint32_t (&xw)[kMmaXWords], const unsigned short* row, int64_t K,
                                    int64_t kb, int q, bool vec) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) ld_x4(xw + 2 * ks, row, K, kb + 16 * ks + 4 * q, vec);
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    return make_uint2(xw[2 * ks], xw[2 * ks + 1]);
  }
};

using F = FmtAQLM;

int grid_for(int64_t work) {
  const int64_t b = (work + 255) / 256;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

// Canonical codes [N][K/8][2] -> tiles [rt][kt][j][t][32 B] (see above);
// bytes of rows >= N or groups >= K/8 are 0 (their x is 0 or the row is
// never stored).  One thread per 16-byte half row.
__global__ void prepare_kernel(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                               int64_t nvec, uint8_t* __restrict__ tiles) {
  const int64_t ng = K / 8;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < nvec;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tile = v / (F::kTileBytes / 16);
    const int w = static_cast<int>(v % (F::kTileBytes / 16));
    const int h = w & 1;
    const int t = (w >> 1) % kLaneSlots;
    const int j = (w >> 1) / kLaneSlots;
    const int slice = t >> 5, l = t & 31;
    const int64_t rt = tile / nKT;
    const int kt = static_cast<int>(tile % nKT);
    const int64_t n = rt * kTileRows + 4 * l + j;
    const int64_t g0 = int64_t(kt) * (F::kKT / 8) + slice * 16;
    uint8_t b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int ks = i >> 1, cb = i & 1;
      const int64_t g = g0 + 2 * ks + h;
      b[i] = (n < N && g < ng) ? canon[(n * ng + g) * 2 + cb] : 0;
    }
    uint4 o;
    o.x = b[0] | (b[1] << 8) | (b[2] << 16) | (uint32_t(b[3]) << 24);
    o.y = b[4] | (b[5] << 8) | (b[6] << 16) | (uint32_t(b[7]) << 24);
    o.z = b[8] | (b[9] << 8) | (b[10] << 16) | (uint32_t(b[11]) << 24);
    o.w = b[12] | (b[13] << 8) | (b[14] << 16) | (uint32_t(b[15]) << 24);
    reinterpret_cast<uint4*>(tiles)[v] = o;
  }
}

// Decode from this layout (the same exact value as the table layout's
// decoder: one fp32 rounding of s * (c0 + c1), computed exactly in fp64).
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, const uint8_t* __restrict__ aux,
                               int64_t N, int64_t K, int nKT, float* __restrict__ w_out) {
  const int64_t ng = K / 8;
  const __half* cbk = reinterpret_cast<const __half*>(aux);
  const __half* sc = reinterpret_cast<const __half*>(aux + F::kCodebookBytes);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < N * ng;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = i / ng, g = i % ng;
    const int64_t rt = n / kTileRows;
    const int r = static_cast<int>(n % kTileRows);
    const int l = r >> 2, j = r & 3;
    const int64_t kt = g / (F::kKT / 8);
    const int gs = static_cast<int>(g % (F::kKT / 8));
    const int slice = gs >> 4, gg = gs & 15;
    const int ks = gg >> 1, h = gg & 1;
    const uint8_t* row = tiles + (rt * nKT + kt) * F::kTileBytes + (int64_t(j) * kLaneSlots + slice * 32 + l) * 32;
    const int c0 = row[16 * h + 2 * ks], c1 = row[16 * h + 2 * ks + 1];
    const double s = __half2float(sc[n]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const double v0 = __half2float(cbk[c0 * 8 + e]);
      const double v1 = __half2float(cbk[(256 + c1) * 8 + e]);
      w_out[n * K + 8 * g + e] = static_cast<float>(s * (v0 + v1));
    }
  }
}

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t nvec = a.nRT * a.nKT * int64_t(F::kTileBytes / 16);
  prepare_kernel<<<grid_for(nvec), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT, nvec, a.tiles);
  cudaError_t e = cudaGetLastError();
  uint8_t* aux = static_cast<uint8_t*>(a.aux);
  if (e == cudaSuccess) e = cudaMemcpyAsync(aux, a.codebooks, F::kCodebookBytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(aux + F::kCodebookBytes, a.scales, 2 * a.N, cudaMemcpyDeviceToDevice, s);
  return e;
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t*, int64_t N, int64_t K, int nKT,
                    float* w_out, int, cudaStream_t s) {
  dequant_kernel<<<grid_for(N * (K / 8)), 256, 0, s>>>(tiles, static_cast<const uint8_t*>(aux), N, K, nKT,
                                                       w_out);
  return cudaGetLastError();
}

template <int NB, bool PAR = false>
cudaError_t launch_nb(const RunParams& p, int M, const LaunchGeom& g, cudaStream_t s) {
  static_assert(mma_smem_bytes<F, NB, PAR>() + 2048 <= 228 * 1024, "shared memory budget exceeded");
  RunParams q = p;
  q.plan = g.plan;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(mma_threads<F, NB, PAR>());
  cfg.dynamicSmemBytes = mma_smem_bytes<F, NB, PAR>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wstream_mma_kernel<F, NB, PAR>, q, M);
}

// Batch-invariant mode: every M runs the default geometry, the same
// instruction sequence per activation row (one B column each), so a row's
// bits do not depend on M.  Otherwise one activation block runs the
// tile-parity geometry.
cudaError_t launch(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant) {
  if (M >= 1 && M <= 8) return batch_invariant ? launch_nb<1>(p, M, g, s) : launch_nb<1, true>(p, M, g, s);
  if (M > 8 && M <= kMaxM) return launch_nb<2>(p, M, g, s);
  return cudaErrorInvalidValue;
}

int smem_bytes(int M) { return M <= 8 ? mma_smem_bytes<F, 1, true>() : mma_smem_bytes<F, 2>(); }

cudaError_t setup() {
  cudaError_t e = cudaFuncSetAttribute(wstream_mma_kernel<F, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       mma_smem_bytes<F, 1>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wstream_mma_kernel<F, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mma_smem_bytes<F, 2>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wstream_mma_kernel<F, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mma_smem_bytes<F, 1, true>());
  return e;
}

}  // namespace

// Internal format (not in the public enum): the AQLM handle's tensor-core
// companion, created and used by qgemv_api.cu.
const FormatOps* ops_aqlm_mma() {
  static const FormatOps ops = {
      /*format=*/6, F::kKT, F::kTileBytes, /*aux_bytes=*/F::kCodebookBytes,
      &smem_bytes, &setup, &launch, &prepare, &dequant,
      /*cb_entries=*/0, /*tile_rows=*/kTileRows, /*partial_stride=*/int64_t(kTileRows) * 16, /*aux_per_row=*/2,
      /*m1_ctas_per_sm=*/1};
  return &ops;
}

}  // namespace qgemv

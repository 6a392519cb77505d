// fmt_q4_0.cu -- Q4_0: re-layout (prepare), exact decode export, quantizer,
// and the launch table of the GEMV kernel for M = 1..16.
//
// Canonical Q4_0 ("Model quantization, read carefully", sections "The
// ladder" and "Anatomy of a block"; value (q - 8) * d and the quantizer
// d = signed-max / -8, q = clamp(round(w/d) + 8, 0..15) follow the ggml
// convention): per output row n, K/32 blocks of {fp16 d; uint8 qs[16]},
// byte i of qs holding element i (low nibble) and element i+16 (high).
#include <cuda_fp16.h>

#include "fmt_fields.cuh"
#include "formats.h"
#include "launch_table.cuh"

namespace qgemv {
namespace {

using F = FmtQ4_0;
constexpr int kBlockBytes = 18;

// Nibble q of element e (0..31) of a canonical block's qs[16].
__device__ __forceinline__ uint32_t canon_q(const uint8_t* qs, int e) {
  return e < 16 ? (qs[e] & 0xfu) : (qs[e - 16] >> 4);
}

// One thread per 32-bit code word of the prepared stream.  Word wi of half h
// of (row j, lane slot t) holds elements 8wi..8wi+7 of block 2*slice + h.
__global__ void prepare_codes(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                              int64_t nwords, uint32_t* __restrict__ tiles) {
  constexpr int kWordsPerTile = F::kTileBytes / 4;
  constexpr int kCodeWords = F::kCodeBytes / 4;
  const int64_t nb = K / 32;
  for (int64_t wa = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; wa < nwords;
       wa += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = wa / kCodeWords;
    const int off = static_cast<int>(wa % kCodeWords);
    const int chunk = off / 4, wi = off % 4;
    const int jh = chunk / kLaneSlots, t = chunk % kLaneSlots;
    const int j = jh / 2, h = jh % 2;
    const int cw = t / 32, lane = t % 32;
    const int64_t n = (tile / nKT) * kTileRows + kRowsPerLane * lane + j;
    const int64_t b = static_cast<int64_t>(tile % nKT) * (F::kKT / 32) + 2 * cw + h;
    uint32_t word = 0;
    if (n < N && b < nb) {
      const uint8_t* qs = canon + (n * nb + b) * kBlockBytes + 2;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) word |= canon_q(qs, 8 * wi + jj) << (4 * jj);
    }
    tiles[tile * kWordsPerTile + off] = word;
  }
}

// One thread per (tile, t): the eight fp16 scales [j][b] of rows 4l..4l+3,
// blocks 2*slice and 2*slice + 1.
__global__ void prepare_scales(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                               int64_t nitems, uint8_t* __restrict__ tiles) {
  const int64_t nb = K / 32;
  for (int64_t it = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; it < nitems;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = it / kLaneSlots;
    const int t = static_cast<int>(it % kLaneSlots);
    const int cw = t / 32, lane = t % 32;
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = (tile / nKT) * kTileRows + kRowsPerLane * lane + j;
      uint32_t hw[2] = {0, 0};
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int64_t b = static_cast<int64_t>(tile % nKT) * (F::kKT / 32) + 2 * cw + bb;
        if (n < N && b < nb) {
          const uint8_t* blk = canon + (n * nb + b) * kBlockBytes;
          hw[bb] = static_cast<uint32_t>(blk[0] | (blk[1] << 8));
        }
      }
      v[j] = hw[0] | (hw[1] << 16);
    }
    *reinterpret_cast<uint4*>(tiles + tile * F::kTileBytes + F::kCodeBytes + t * 16) =
        make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// Exact decode of every weight from the prepared tiles.
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, int64_t N, int64_t K, int nKT,
                               float* __restrict__ w) {
  const int64_t total = N * K;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = e / K, k = e % K;
    const int r = static_cast<int>(n % kTileRows);
    const int lane = r / kRowsPerLane, j = r % kRowsPerLane;
    const int64_t tile = (n / kTileRows) * nKT + k / F::kKT;
    const int kk = static_cast<int>(k % F::kKT);
    const int cw = kk / F::kKW, el = kk % F::kKW;
    const int h = el / 32, eb = el % 32;
    const int t = cw * 32 + lane;
    const uint8_t* tb = tiles + tile * F::kTileBytes;
    const uint32_t word =
        *reinterpret_cast<const uint32_t*>(tb + ((j * 2 + h) * kLaneSlots + t) * 16 + 4 * (eb / 8));
    const int q = static_cast<int>((word >> (4 * (eb % 8))) & 0xfu);
    const uint16_t hb = *reinterpret_cast<const uint16_t*>(tb + F::kCodeBytes + t * 16 + 2 * (2 * j + h));
    w[e] = static_cast<float>(q - 8) * h2f(hb);  // exact: 4-bit int x fp16 fits fp32
  }
}

// One thread per block of 32 weights.
__global__ void quantize_kernel(const float* __restrict__ w, int64_t nblocks,
                                uint8_t* __restrict__ out) {
  for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < nblocks;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float* v = w + b * 32;
    float amax = 0.f, absmax = 0.f;
    for (int i = 0; i < 32; ++i) {
      const float a = fabsf(v[i]);
      if (a > absmax) {
        absmax = a;
        amax = v[i];
      }
    }
    const float d = __fdiv_rn(amax, -8.0f);
    uint32_t q[32];
    for (int i = 0; i < 32; ++i) {
      int qi = 8;
      if (d != 0.0f) {
        qi = static_cast<int>(roundf(__fdiv_rn(v[i], d))) + 8;
        qi = qi < 0 ? 0 : (qi > 15 ? 15 : qi);
      }
      q[i] = static_cast<uint32_t>(qi);
    }
    // The block starts at an even byte offset: write it as nine 16-bit words
    // (fp16 d, then qs[2i] | qs[2i+1] << 8 with qs[i] = q_i | q_(i+16) << 4).
    uint16_t* blk = reinterpret_cast<uint16_t*>(out + b * kBlockBytes);
    blk[0] = __half_as_ushort(__float2half_rn(d));
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = q[2 * i] | (q[2 * i + 16] << 4);
      const uint32_t hi = q[2 * i + 1] | (q[2 * i + 17] << 4);
      blk[1 + i] = static_cast<uint16_t>(lo | (hi << 8));
    }
  }
}

int grid_for(int64_t items, int threads) {
  const int64_t g = (items + threads - 1) / threads;
  return static_cast<int>(g < 1 ? 1 : (g > 65536 ? 65536 : g));
}

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t T = a.nRT * a.nKT;
  const int64_t nwords = T * (F::kCodeBytes / 4);
  prepare_codes<<<grid_for(nwords, 256), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT, nwords,
                                                      reinterpret_cast<uint32_t*>(a.tiles));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nitems = T * kLaneSlots;
  prepare_scales<<<grid_for(nitems, 256), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT, nitems, a.tiles);
  return cudaGetLastError();
}

cudaError_t dequant(const uint8_t* tiles, const void*, const int32_t*, int64_t N, int64_t K, int nKT,
                    float* w, int, cudaStream_t s) {
  dequant_kernel<<<grid_for(N * K, 256), 256, 0, s>>>(tiles, N, K, nKT, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t quantize_q4_0(const float* w, int64_t N, int64_t K, uint8_t* out, cudaStream_t s) {
  const int64_t nblocks = N * (K / 32);
  quantize_kernel<<<grid_for(nblocks, 128), 128, 0, s>>>(w, nblocks, out);
  return cudaGetLastError();
}

namespace {
cudaError_t setup_all() {
  cudaError_t e = LaunchTable<F>::setup();
  if (e == cudaSuccess) e = LaunchTable<F>::setup_glu();
  return e;
}
}  // namespace

const FormatOps* ops_q4_0() {
  static const FormatOps ops = {
      /*format=*/1, F::kKT, F::kTileBytes, /*aux_bytes=*/0,
      &LaunchTable<F>::smem_bytes, &setup_all, &LaunchTable<F>::launch,
      &prepare, &dequant, /*cb_entries=*/0, /*tile_rows=*/128, /*partial_stride=*/128 * 16,
      /*aux_per_row=*/0, /*m1_ctas_per_sm=*/LaunchTable<F>::kM1CtasPerSm, /*rowgroup=*/0,
      /*launch_x_int8=*/nullptr, /*row_tables=*/0, /*launch_xq=*/nullptr,
      /*launch_glu=*/&LaunchTable<F>::launch_glu, /*tc5_min_m=*/kTc5DefaultMinM, /*split_unit=*/SplitModeOf<F>::value};
  return &ops;
}

}  // namespace qgemv

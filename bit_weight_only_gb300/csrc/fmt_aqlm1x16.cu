// fmt_aqlm1x16.cu -- AQLM 1x16: one codebook of 65,536 entries of 8 fp16
// values per matrix, one 16-bit code per group of 8 weights (2 bits per
// weight) and a per-row fp16 scale ("Trapetum benchmarks", the section on
// the PV-tuned Llama-2-70B in 1x16):
//
//     w[n][8g + j] = s_n * C[code(n, g)][j].
//
// The 1 MiB codebook does not fit in shared memory, so, as the page's
// kernel does, every looked-up entry is gathered from L2 (where the whole
// codebook stays resident) and the products are taken in fp32:
//   * one warp per output row at a time (rows grid-strided over the CTAs);
//     per chunk of 256 groups, lane l takes groups l, l + 32, ..., l + 224,
//     whose 8 codes the prepared layout keeps in the lane's 128-bit vector
//     (16 B, coalesced across the warp), so that a warp's activation loads
//     for one step are 32 consecutive groups' inputs (coalesced too);
//   * for each code the 16-byte entry is one 128-bit load, reused for every
//     activation row of the call, so each code and entry is read once per
//     call whatever M is;
//   * a lane sums its groups in a fixed order and the warp adds the lanes'
//     sums with a butterfly (commutative adds: every lane ends with the same
//     bits), then lane m stores row n of activation row m times s_n.  No
//     atomics and no split of a row: results are the same bits from run to
//     run and a row's bits do not depend on M.
// The bound is L2: each group costs a 32-byte sector for 16 useful bytes,
// against 2 bytes of codes from HBM.
//
// Prepared layout: each row padded with zero codes to a whole number of
// 256-code chunks (so every row starts 16-byte aligned), and inside a chunk
// the code of group 32e + l at position 8l + e (code_pos); aux = the
// codebook [65536][8] fp16, then the scales [N] fp16.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "formats.h"
#include "gemv_kernel.cuh"

namespace qgemv {
namespace a16 {

constexpr int kKC = 2048;                           // weights per prepared chunk
constexpr int kChunkCodes = kKC / 8;                // 256
constexpr int kChunkBytes = kChunkCodes * 2;        // 512
constexpr int64_t kCodebookBytes = 65536LL * 8 * 2;  // 1 MiB
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

// Position in the prepared row of the code of group g (lane l = g % 32 of
// its chunk's step e = (g % 256) / 32 holds it as element e of its vector).
__host__ __device__ __forceinline__ int64_t code_pos(int64_t g) {
  const int64_t gi = g % kChunkCodes;
  return g - gi + (gi % 32) * 8 + gi / 32;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = h2f(v.x & 0xffffu), f[1] = h2f(v.x >> 16);
  f[2] = h2f(v.y & 0xffffu), f[3] = h2f(v.y >> 16);
  f[4] = h2f(v.z & 0xffffu), f[5] = h2f(v.z >> 16);
  f[6] = h2f(v.w & 0xffffu), f[7] = h2f(v.w >> 16);
}

template <int MB>
// A register cap rather than launch bounds: left to itself the compiler
// gives the eight-row instantiation 48 registers and spills; 64 keep four
// CTAs of 256 threads per SM resident.
__global__ void __maxnreg__(64) aqlm1x16_kernel(const RunParams p, int M) {
  const uint4* cb = static_cast<const uint4*>(p.aux);
  const unsigned short* scales =
      reinterpret_cast<const unsigned short*>(static_cast<const uint8_t*>(p.aux) + kCodebookBytes);
  const unsigned int* xw = reinterpret_cast<const unsigned int*>(p.x);  // fp16 pairs (x is 4-byte aligned)
  // x 16-byte aligned (then every group's 8 inputs are, K being a multiple
  // of 8): one 128-bit load per group and activation row instead of four
  // 32-bit ones -- the loads, not the FMAs, fill the memory pipeline here
  // (8192 x 28672 at M = 1: 122 -> 291 GB/s).  Staging x in shared memory
  // instead measured slower (the lanes' 128-byte-apart reads conflict).
  const bool xvec = (reinterpret_cast<uintptr_t>(p.x) & 15u) == 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t G = p.K / 8;                        // groups (codes) per row
  const int64_t pitch = int64_t(p.nKT) * kChunkCodes;  // codes per prepared row
  const int nchunk = static_cast<int>((G + kChunkCodes - 1) / kChunkCodes);  // chunks holding real codes

  // Nothing above reads what an earlier kernel in the stream writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int64_t n = int64_t(blockIdx.x) * kWarps + warp; n < p.N; n += int64_t(gridDim.x) * kWarps) {
    const uint4* crow = reinterpret_cast<const uint4*>(p.tiles + n * pitch * 2);
    float acc[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[m] = 0.f;
    for (int ch = 0; ch < nchunk; ++ch) {
      const uint4 cv = __ldg(crow + ch * 32 + lane);
      const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
      uint4 ent[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ent[e] = __ldg(cb + ((cw[e >> 1] >> (16 * (e & 1))) & 0xffffu));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t g = int64_t(ch) * kChunkCodes + 32 * e + lane;
        if (g < G) {  // padding codes (0) past the row's end are not used
          float c[8];
          unpack8(ent[e], c);
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < M) {
              const unsigned int* xr = xw + (m * p.K + g * 8) / 2;
              const uint4 x8 = xvec ? __ldg(reinterpret_cast<const uint4*>(xr))
                                    : make_uint4(__ldg(xr), __ldg(xr + 1), __ldg(xr + 2), __ldg(xr + 3));
              const uint32_t x2[4] = {x8.x, x8.y, x8.z, x8.w};
              float d = 0.f;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                d = fmaf(c[2 * q], h2f(x2[q] & 0xffffu), d);
                d = fmaf(c[2 * q + 1], h2f(x2[q] >> 16), d);
              }
              acc[m] += d;
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
    const float s = h2f(__ldg(scales + n));
#pragma unroll
    for (int m = 0; m < MB; ++m)
      if (m < M && lane == m) store_y(p, m * p.N + n, __fmul_rn(acc[m], s));
  }
}

// One thread per prepared code: the canonical code, or 0 past the row's end.
__global__ void prepare_kernel(const uint16_t* __restrict__ canon, int64_t N, int64_t G, int nKT,
                               uint16_t* __restrict__ tiles) {
  const int64_t pitch = int64_t(nKT) * kChunkCodes;
  const int64_t total = N * pitch;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = e / pitch, g = e % pitch;
    tiles[n * pitch + code_pos(g)] = g < G ? canon[n * G + g] : static_cast<uint16_t>(0);
  }
}

// w[n][8g + j] = s_n * C[code][j]: a product of two fp16 values, exact in fp32.
__global__ void dequant_kernel(const uint16_t* __restrict__ tiles, const uint8_t* __restrict__ aux, int64_t N,
                               int64_t K, int nKT, float* __restrict__ w_out) {
  const unsigned short* cb = reinterpret_cast<const unsigned short*>(aux);
  const unsigned short* sc = reinterpret_cast<const unsigned short*>(aux + kCodebookBytes);
  const int64_t G = K / 8;
  const int64_t pitch = int64_t(nKT) * kChunkCodes;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < N * G;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = e / G, g = e % G;
    const uint32_t code = tiles[n * pitch + code_pos(g)];
    const float s = h2f(sc[n]);
#pragma unroll
    for (int j = 0; j < 8; ++j) w_out[n * K + 8 * g + j] = __fmul_rn(s, h2f(cb[code * 8 + j]));
  }
}

int grid_for(int64_t work) {
  const int64_t b = (work + 255) / 256;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  prepare_kernel<<<grid_for(a.N * a.nKT * int64_t(kChunkCodes)), 256, 0, s>>>(
      reinterpret_cast<const uint16_t*>(a.packed), a.N, a.K / 8, a.nKT, reinterpret_cast<uint16_t*>(a.tiles));
  cudaError_t e = cudaGetLastError();
  uint8_t* aux = static_cast<uint8_t*>(a.aux);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(aux, a.codebooks, kCodebookBytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(aux + kCodebookBytes, a.scales, 2 * a.N, cudaMemcpyDeviceToDevice, s);
  return e;
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t*, int64_t N, int64_t K, int nKT,
                    float* w_out, int, cudaStream_t s) {
  dequant_kernel<<<grid_for(N * (K / 8)), 256, 0, s>>>(reinterpret_cast<const uint16_t*>(tiles),
                                                       static_cast<const uint8_t*>(aux), N, K, nKT, w_out);
  return cudaGetLastError();
}

int smem_bytes(int) { return 0; }

cudaError_t setup() { return cudaSuccess; }

template <int MB>
cudaError_t launch_mb(const RunParams& p, int M, cudaStream_t s) {
  const int64_t blocks = (p.N + kWarps - 1) / kWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < 65535 ? blocks : 65535));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, aqlm1x16_kernel<MB>, p, M);
}

// One launch for all M rows (each code and entry read once per call); the
// instantiation only sizes the accumulators, so every M gives every row the
// same bits (batch invariant in either mode).
cudaError_t launch(int M, const RunParams& p, const LaunchGeom&, cudaStream_t s, bool) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  if (M == 1) return launch_mb<1>(p, M, s);
  if (M == 2) return launch_mb<2>(p, M, s);
  if (M <= 4) return launch_mb<4>(p, M, s);
  if (M <= 8) return launch_mb<8>(p, M, s);
  return launch_mb<16>(p, M, s);
}

}  // namespace a16

const FormatOps* ops_aqlm_1x16() {
  static const FormatOps ops = {
      /*format=*/7, a16::kKC, a16::kChunkBytes, /*aux_bytes=*/a16::kCodebookBytes,
      &a16::smem_bytes, &a16::setup, &a16::launch, &a16::prepare, &a16::dequant,
      /*cb_entries=*/0, /*tile_rows=*/1, /*partial_stride=*/1, /*aux_per_row=*/2};
  return &ops;
}

}  // namespace qgemv

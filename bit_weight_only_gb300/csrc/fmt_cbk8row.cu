// fmt_cbk8row.cu -- CBK8 with one fp32 codebook of 256 centroids per output
// row: the 8-bit LM head of the pages' own 4-bit files ("Trapetum
// benchmarks", "Model-level results": the new exporter's 8-bit head with
// 256-entry fp32 codebooks).  w[n][k] = C_n[idx(n, k)].
//
// A row's codebook (1 KB) is only used by that row, so there is no shared
// table to build per tile: one warp takes one output row at a time and puts
// the row's codebook in its own shared-memory slot, in four copies; lanes
// 8c .. 8c+7 read copy c, whose entry e sits at word e ^ 8c, so lanes of
// different copies never meet in a bank on equal indices (the lookups of a
// warp are otherwise random).  The entry address is one shift and one LOP3
// of the index word (the copy is 1 KB-aligned, the XOR folds into the LOP3).
// The activations of the launch's rows are staged once per CTA in shared
// memory as fp16 (zero-padded to a multiple of 16 inputs, so the padded
// index bytes past K meet x = 0), and the grid is persistent.
//   * lane l takes the 16-byte index vectors l, l + 32, ... of the row;
//   * products in fp32, two chains per activation row (even, odd k);
//   * the lanes' sums are added with an exactly commuting butterfly and lane
//     m stores activation row m: reproducible, no split of a row, and a
//     row's bits do not depend on M.
// Prepared layout: the index bytes, each row padded with zeros to whole
// 512-byte chunks; aux = the codebooks fp32 [N][256].
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "formats.h"
#include "gemv_kernel.cuh"

namespace qgemv {
namespace c8r {

constexpr int kKC = 512;        // index bytes per prepared chunk
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kCopies = 4;
constexpr int kCbSmem = kWarps * kCopies * 1024;  // 32 KB of codebook copies
constexpr int kSmemLimit = 220 * 1024;

__host__ __device__ constexpr int64_t kpad(int64_t K) { return (K + 15) / 16 * 16; }
__host__ __device__ constexpr int64_t smem_for(int mb, int64_t K) { return kCbSmem + 1024 + mb * kpad(K) * 2; }

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

template <int MB>
__global__ void __launch_bounds__(kThreads) rowcb8_kernel(const RunParams p, int M) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t K = p.K;
  const int64_t Kp = kpad(K);
  const int64_t pitch = (K + kKC - 1) / kKC * kKC;  // index bytes per prepared row
  // codebook copies first (1 KB-aligned), then x
  const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;
  uint8_t* cbw = smem + (base - smem_u32(smem)) + warp * kCopies * 1024;  // this warp's copies
  __half* sx = reinterpret_cast<__half*>(smem + (base - smem_u32(smem)) + kCbSmem);
  const uint32_t copy = static_cast<uint32_t>(lane >> 3);
  const uint32_t key = (smem_u32(cbw) + copy * 1024u) ^ (copy << 5);  // copy base, XOR skew of 8c words

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // stage x of the launch's rows (zero past K and past M)
  const unsigned short* xg = reinterpret_cast<const unsigned short*>(p.x);
  unsigned short* sxs = reinterpret_cast<unsigned short*>(sx);
  for (int64_t e = threadIdx.x; e < MB * Kp; e += kThreads) {
    const int64_t m = e / Kp, k = e % Kp;
    sxs[e] = (m < M && k < K) ? __ldg(xg + m * K + k) : static_cast<unsigned short>(0);
  }
  __syncthreads();

  const int nvec = static_cast<int>(Kp / 16);
  for (int64_t n = int64_t(blockIdx.x) * kWarps + warp; n < p.N; n += int64_t(gridDim.x) * kWarps) {
    // the row's codebook into the warp's four copies
    const float4* cbg = reinterpret_cast<const float4*>(static_cast<const float*>(p.aux) + n * 256);
    const float4 c0 = __ldg(cbg + 2 * lane), c1 = __ldg(cbg + 2 * lane + 1);
    const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    __syncwarp();  // every lane is done with the previous row's copies
#pragma unroll
    for (int c = 0; c < kCopies; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float*>(cbw + c * 1024)[(8 * lane + i) ^ (8 * c)] = cv[i];
    __syncwarp();

    const uint4* irow = reinterpret_cast<const uint4*>(p.tiles + n * pitch);
    float acc[MB][2];
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[m][0] = acc[m][1] = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 iv = __ldg(irow + v);
      const uint32_t iw[4] = {iv.x, iv.y, iv.z, iv.w};
      float w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // entry address of byte b of the word: (byte * 4) ^ key
        w[4 * q + 0] = lds_f32(((iw[q] << 2) & 0x3FCu) ^ key);
        w[4 * q + 1] = lds_f32(((iw[q] >> 6) & 0x3FCu) ^ key);
        w[4 * q + 2] = lds_f32(((iw[q] >> 14) & 0x3FCu) ^ key);
        w[4 * q + 3] = lds_f32(((iw[q] >> 22) & 0x3FCu) ^ key);
      }
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          const uint4* xr = reinterpret_cast<const uint4*>(sx + m * Kp + 16 * v);
          const uint4 xa = xr[0], xb = xr[1];
          const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc[m][0] = fmaf(w[2 * j], h2f(xw[j] & 0xffffu), acc[m][0]);
            acc[m][1] = fmaf(w[2 * j + 1], h2f(xw[j] >> 16), acc[m][1]);
          }
        }
      }
    }
    float r[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      r[m] = acc[m][0] + acc[m][1];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) r[m] += __shfl_xor_sync(0xffffffffu, r[m], off);
    }
#pragma unroll
    for (int m = 0; m < MB; ++m)
      if (m < M && lane == m) store_y(p, m * p.N + n, r[m]);
  }
}

// One thread per prepared index byte: the canonical byte, or 0 past K.
__global__ void prepare_kernel(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int64_t pitch,
                               uint8_t* __restrict__ tiles) {
  const int64_t total = N * pitch;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = e / pitch, k = e % pitch;
    tiles[e] = k < K ? canon[n * K + k] : static_cast<uint8_t>(0);
  }
}

__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, const float* __restrict__ cb, int64_t N,
                               int64_t K, int64_t pitch, float* __restrict__ w) {
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < N * K; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = e / K, k = e % K;
    w[e] = cb[n * 256 + tiles[n * pitch + k]];
  }
}

int grid_for(int64_t work) {
  const int64_t b = (work + 255) / 256;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t pitch = int64_t(a.nKT) * kKC;
  prepare_kernel<<<grid_for(a.N * pitch), 256, 0, s>>>(a.packed, a.N, a.K, pitch, a.tiles);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(a.aux, a.codebooks, a.N * 256 * 4, cudaMemcpyDeviceToDevice, s);
  return e;
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t*, int64_t N, int64_t K, int nKT,
                    float* w, int, cudaStream_t s) {
  dequant_kernel<<<grid_for(N * K), 256, 0, s>>>(tiles, static_cast<const float*>(aux), N, K, int64_t(nKT) * kKC,
                                                 w);
  return cudaGetLastError();
}

template <int MB>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(rowcb8_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

cudaError_t setup() {
  cudaError_t e = set_smem<1>();
  if (e == cudaSuccess) e = set_smem<2>();
  if (e == cudaSuccess) e = set_smem<4>();
  if (e == cudaSuccess) e = set_smem<8>();
  if (e == cudaSuccess) e = set_smem<16>();
  return e;
}

int smem_bytes(int) { return kSmemLimit; }

template <int MB>
cudaError_t launch_mb(const RunParams& p, int m0, int mrows, int sms, cudaStream_t s) {
  RunParams q = p;
  q.x = p.x + m0 * p.K;
  q.y = p.y + m0 * p.N;
  q.residual = p.residual != nullptr ? p.residual + m0 * p.N : nullptr;
  const int64_t smem = smem_for(MB, p.K);
  int64_t ctas = kSmemLimit / smem;
  ctas = ctas < 1 ? 1 : (ctas > 4 ? 4 : ctas);
  const int64_t want = (p.N + kWarps - 1) / kWarps;
  const int64_t grid = want < sms * ctas ? want : sms * ctas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rowcb8_kernel<MB>, q, mrows);
}

// Row blocks: the smallest instantiation (1, 2, 4, 8, 16 rows) that holds
// the remaining rows, halved while its staged activations do not fit;
// launch after launch.  A row's arithmetic is the same in every block size.
cudaError_t launch(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  const int sms = g.grid;  // min(tiles, SMs): the SM count for any matrix of at least that many rows
  for (int m0 = 0; m0 < M;) {
    const int rem = M - m0;
    int mb = 1;
    while (mb < rem) mb <<= 1;
    while (mb > 1 && smem_for(mb, p.K) > kSmemLimit) mb >>= 1;
    if (smem_for(mb, p.K) > kSmemLimit) return cudaErrorInvalidValue;  // K too large (checked at create)
    const int rows = mb < rem ? mb : rem;
    cudaError_t e = cudaSuccess;
    switch (mb) {
      case 16: e = launch_mb<16>(p, m0, rows, sms, s); break;
      case 8: e = launch_mb<8>(p, m0, rows, sms, s); break;
      case 4: e = launch_mb<4>(p, m0, rows, sms, s); break;
      case 2: e = launch_mb<2>(p, m0, rows, sms, s); break;
      default: e = launch_mb<1>(p, m0, rows, sms, s); break;
    }
    if (e != cudaSuccess) return e;
    m0 += rows;
  }
  return cudaSuccess;
}

}  // namespace c8r

const FormatOps* ops_cbk8_row() {
  static const FormatOps ops = {
      /*format=*/9, c8r::kKC, c8r::kKC, /*aux_bytes=*/0,
      &c8r::smem_bytes, &c8r::setup, &c8r::launch, &c8r::prepare, &c8r::dequant,
      /*cb_entries=*/0, /*tile_rows=*/1, /*partial_stride=*/1, /*aux_per_row=*/1024};
  return &ops;
}

}  // namespace qgemv

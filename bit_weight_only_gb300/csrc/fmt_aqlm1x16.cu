// fmt_aqlm1x16.cu -- AQLM 1x16: one codebook of 65,536 entries of 8 fp16
// values per matrix, one 16-bit code per group of 8 weights (2 bits per
// weight) and a per-row fp16 scale ("Trapetum benchmarks", the section on
// the PV-tuned Llama-2-70B in 1x16):
//
//     w[n][8g + j] = s_n * C[code(n, g)][j].
//
// The 1 MiB codebook does not fit in shared memory, so, as the page's
// kernel does, every looked-up entry is gathered from L2 (where the whole
// codebook stays resident) and the products (fp16 x fp16, exact) are summed
// in fp32:
//   * one warp per output row at a time (rows grid-strided over the CTAs);
//     per chunk of 256 groups, lane l takes groups l, l + 32, ..., l + 224,
//     whose 8 codes the prepared layout keeps in the lane's 128-bit vector
//     (16 B, coalesced across the warp), so that a warp's activation loads
//     for one step are 32 consecutive groups' inputs (coalesced too);
//   * for each code the 16-byte entry is one 128-bit load, reused for every
//     activation row of the call, so each code and entry is read once per
//     call whatever M is;
//   * for M > 1 the CTA's eight warps take their rows' chunks in step and
//     copy the activations of every 128 groups into shared memory once for
//     all eight rows (M = 1 reads them through L1, where they fit);
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

// Activation staging for M > 1: the CTA's eight warps walk their rows'
// chunks in step, and the inputs of every 128 groups (four steps of a chunk,
// one "unit") are copied once per CTA into shared memory with cp.async,
// double-buffered, instead of once per warp through L1: with a warp per row
// each of the eight rows of a CTA would otherwise read all M x K inputs
// (8 x 28672 at M = 8 is 458 KB, far beyond L1, so every warp re-read it
// from L2).  Lane l of step s reads the 16 bytes of group 32 s + l: 32
// consecutive 16-byte words, no bank conflict.  M = 1 keeps x in L1 (57 KB
// at K = 28672) and needs no barrier.  8192 x 28672 at M = 8: 720 -> 286 us
// with the staging, -> 251 us with the mixed-precision FMAs below.
constexpr int kUnitSteps = 4;
constexpr int kUnitGroups = 32 * kUnitSteps;  // 128
__host__ __device__ constexpr int x_stage_bytes(int MB) { return MB == 1 ? 0 : 2 * MB * kUnitGroups * 16; }

// d = fma(a.lo, b.lo, d), then d = fma(a.hi, b.hi, d): the mixed-precision
// FMA takes the fp16 halves as they are (the product of two fp16 values is
// exact, so this is fmaf on the values widened to fp32, without the two
// conversions).
__device__ __forceinline__ void fma_f16_pair(uint32_t a2, uint32_t b2, float& d) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(d)
      : "r"(a2), "r"(b2));
}

// The entry c (8 fp16) times x[m][8g .. 8g + 7]: a group's eight products
// summed in a fixed order (k = 8g, 8g + 1, ...), the same for every M and
// either source of x.
__device__ __forceinline__ float group_dot(const uint4& c8, const uint4& x8) {
  float d = 0.f;
  fma_f16_pair(c8.x, x8.x, d);
  fma_f16_pair(c8.y, x8.y, d);
  fma_f16_pair(c8.z, x8.z, d);
  fma_f16_pair(c8.w, x8.w, d);
  return d;
}

template <int MB>
// A register cap rather than launch bounds: left to itself the compiler
// gives the eight-row instantiation 48 registers and spills; 64 keep four
// CTAs of 256 threads per SM resident.  The sixteen-row form's 64 KB of
// staging buffers allow three CTAs per SM, so it may take 80 (no spill).
__global__ void __maxnreg__(MB > 8 ? 80 : 64) aqlm1x16_kernel(const RunParams p, int M) {
  const uint4* cb = static_cast<const uint4*>(p.aux);
  const unsigned short* scales =
      reinterpret_cast<const unsigned short*>(static_cast<const uint8_t*>(p.aux) + kCodebookBytes);
  const unsigned int* xw = reinterpret_cast<const unsigned int*>(p.x);  // fp16 pairs (x is 4-byte aligned)
  // x 16-byte aligned (then every group's 8 inputs are, K being a multiple
  // of 8): one 128-bit load (or copy) per group and activation row instead
  // of four 32-bit ones -- the loads, not the FMAs, fill the memory pipeline
  // here (8192 x 28672 at M = 1: 122 -> 291 GB/s).
  const bool xvec = (reinterpret_cast<uintptr_t>(p.x) & 15u) == 0;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t G = p.K / 8;                        // groups (codes) per row
  const int64_t pitch = int64_t(p.nKT) * kChunkCodes;  // codes per prepared row
  const int nchunk = static_cast<int>((G + kChunkCodes - 1) / kChunkCodes);  // chunks holding real codes

  // Nothing above reads what an earlier kernel in the stream writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // the eight entries of a lane's 16-byte code vector
  auto gather = [&](const uint4& cv, uint4 (&ent)[8]) {
    const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) ent[e] = __ldg(cb + ((cw[e >> 1] >> (16 * (e & 1))) & 0xffffu));
  };
  // lane m of the warp stores row n of activation row m, times s_n
  auto finish_row = [&](int64_t n, float (&acc)[MB]) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
    const float s = h2f(__ldg(scales + n));
#pragma unroll
    for (int m = 0; m < MB; ++m)
      if (m < M && lane == m) store_y(p, m * p.N + n, __fmul_rn(acc[m], s));
  };

  if constexpr (MB == 1) {
    for (int64_t n = int64_t(blockIdx.x) * kWarps + warp; n < p.N; n += int64_t(gridDim.x) * kWarps) {
      const uint4* crow = reinterpret_cast<const uint4*>(p.tiles + n * pitch * 2);
      float acc[1] = {0.f};
      // the codes of the next chunk are loaded a chunk ahead, so that the
      // gathers wait for L2 only, not for the code stream (8192 x 28672:
      // 146 -> 124 us; with M > 1 it measured slower and is not done)
      uint4 cv_next = __ldg(crow + lane);
      for (int ch = 0; ch < nchunk; ++ch) {
        uint4 ent[8];
        const uint4 cv = cv_next;
        if (ch + 1 < nchunk) cv_next = __ldg(crow + (ch + 1) * 32 + lane);
        gather(cv, ent);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int64_t g = int64_t(ch) * kChunkCodes + 32 * e + lane;
          if (g < G) {  // padding codes (0) past the row's end are not used
            const unsigned int* xr = xw + g * 4;
            const uint4 x8 = xvec ? __ldg(reinterpret_cast<const uint4*>(xr))
                                  : make_uint4(__ldg(xr), __ldg(xr + 1), __ldg(xr + 2), __ldg(xr + 3));
            acc[0] += group_dot(ent[e], x8);
          }
        }
      }
      finish_row(n, acc);
    }
  } else {
    extern __shared__ __align__(16) uint4 xsm[];  // [2 buffers][MB rows][kUnitGroups]
    const int nunits = 2 * nchunk;
    // Copy the inputs of unit u (groups 128 u .. 128 u + 127, those below G)
    // of every activation row into buffer u % 2; one commit group per unit.
    auto stage = [&](int u) {
      const int b = u & 1;
      const int64_t g0 = int64_t(u) * kUnitGroups;
      for (int idx = threadIdx.x; idx < M * kUnitGroups; idx += kThreads) {
        const int m = idx / kUnitGroups, i = idx % kUnitGroups;
        if (g0 + i < G) {
          const uint32_t dst = smem_u32(xsm + (b * MB + m) * kUnitGroups + i);
          const unsigned int* src = xw + (m * p.K + (g0 + i) * 8) / 2;
          if (xvec) {
            asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w)
              asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst + 4 * w), "l"(src + w) : "memory");
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    const int64_t step_rows = int64_t(gridDim.x) * kWarps;
    // the row loop is the same for every warp of the CTA (barriers inside);
    // a warp past the last row only helps with the copies
    if (int64_t(blockIdx.x) * kWarps < p.N) stage(0);
    for (int64_t nb = int64_t(blockIdx.x) * kWarps; nb < p.N; nb += step_rows) {
      const int64_t n = nb + warp;
      const bool live = n < p.N;
      const uint4* crow = reinterpret_cast<const uint4*>(p.tiles + (live ? n : 0) * pitch * 2);
      float acc[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[m] = 0.f;
      for (int ch = 0; ch < nchunk; ++ch) {
        uint4 ent[8];
        if (live) gather(__ldg(crow + ch * 32 + lane), ent);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int u = 2 * ch + h;  // buffer u % 2 == h
          // unit u has landed (each thread waits for its own copies, the
          // barrier for everyone's) and every warp is done with unit u - 1,
          // whose buffer the next copies overwrite
          asm volatile("cp.async.wait_group 0;" ::: "memory");
          __syncthreads();
          if (u + 1 < nunits)
            stage(u + 1);
          else if (nb + step_rows < p.N)
            stage(0);  // the CTA's next rows start with unit 0 (buffer 0)
          if (live) {
            const uint4* xb = xsm + h * MB * kUnitGroups;
#pragma unroll
            for (int s = 0; s < kUnitSteps; ++s) {
              const int e = kUnitSteps * h + s;
              const int64_t g = int64_t(ch) * kChunkCodes + 32 * e + lane;
              if (g < G) {
#pragma unroll
                for (int m = 0; m < MB; ++m)
                  if (m < M) acc[m] += group_dot(ent[e], xb[m * kUnitGroups + 32 * s + lane]);
              }
            }
          }
        }
      }
      if (live) finish_row(n, acc);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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

// the accumulator rows a call of M activation rows instantiates
constexpr int mb_of(int M) { return M == 1 ? 1 : (M == 2 ? 2 : (M <= 4 ? 4 : (M <= 8 ? 8 : 16))); }

int smem_bytes(int M) { return x_stage_bytes(mb_of(M)); }

// the sixteen-row staging buffers (64 KB) are above the default 48 KB
cudaError_t setup() {
  return cudaFuncSetAttribute(aqlm1x16_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, x_stage_bytes(16));
}

template <int MB>
cudaError_t launch_mb(const RunParams& p, int M, cudaStream_t s) {
  const int64_t blocks = (p.N + kWarps - 1) / kWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < 65535 ? blocks : 65535));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = x_stage_bytes(MB);
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

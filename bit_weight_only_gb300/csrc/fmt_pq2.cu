// fmt_pq2.cu -- PQ2_0: re-layout (prepare), exact decode export, the
// launch table of the GEMV kernel for M = 1..16, and the INT8-activation
// path (FmtPQ2I8) with its activation quantizer.
//
// Canonical PQ2_0 ("Making a ternary reasoning model fast in vLLM", section
// "Anatomy of a PQ2_0 block"): per output row n, K/128 blocks of
// {fp16 d; uint8 qs[32]} (34 bytes), byte j of qs holding elements
// 4j..4j+3 as two-bit codes read from the low end; code c decodes to
// (c - 1) * d, i.e. 0,1,2,3 -> -1,0,+1,+2.  The prepared layout keeps the same
// bytes, split into a code plane and a scale plane per tile, as the page's
// "prepared weights" do, so that every code row is 16-byte aligned.
#include "fmt_fields.cuh"
#include "formats.h"
#include "launch_table.cuh"

namespace qgemv {
namespace {

using F = FmtPQ2;
constexpr int kBlockBytes = 34;

__device__ __forceinline__ uint32_t canon_code(const uint8_t* qs, int e) {
  return (qs[e >> 2] >> (2 * (e & 3))) & 3u;
}

// One thread per 32-bit code word of the prepared stream.  Word i = 4h + wi
// of (row j, lane slot t) holds elements 16i..16i+15 of block `slice`.
__global__ void prepare_codes(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                              int64_t nwords, uint32_t* __restrict__ tiles) {
  constexpr int kWordsPerTile = F::kTileBytes / 4;
  constexpr int kCodeWords = F::kCodeBytes / 4;
  const int64_t nb = K / 128;
  for (int64_t wa = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; wa < nwords;
       wa += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = wa / kCodeWords;
    const int off = static_cast<int>(wa % kCodeWords);
    const int chunk = off / 4, wi = off % 4;
    const int jh = chunk / kLaneSlots, t = chunk % kLaneSlots;
    const int j = jh / 2, h = jh % 2;
    const int cw = t / 32, lane = t % 32;
    const int64_t n = (tile / nKT) * kTileRows + kRowsPerLane * lane + j;
    const int64_t b = static_cast<int64_t>(tile % nKT) * kSlices + cw;
    uint32_t word = 0;
    if (n < N && b < nb) {
      const uint8_t* qs = canon + (n * nb + b) * kBlockBytes + 2;
      const int e0 = 16 * (4 * h + wi);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) word |= canon_code(qs, e0 + jj) << (2 * jj);
    }
    tiles[tile * kWordsPerTile + off] = word;
  }
}

// One thread per (tile, t): the four fp16 scales of rows 4l..4l+3, block `slice`.
__global__ void prepare_scales(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                               int64_t nitems, uint8_t* __restrict__ tiles) {
  const int64_t nb = K / 128;
  for (int64_t it = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; it < nitems;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = it / kLaneSlots;
    const int t = static_cast<int>(it % kLaneSlots);
    const int cw = t / 32, lane = t % 32;
    const int64_t b = static_cast<int64_t>(tile % nKT) * kSlices + cw;
    uint16_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = (tile / nKT) * kTileRows + kRowsPerLane * lane + j;
      h[j] = 0;
      if (n < N && b < nb) {
        const uint8_t* p = canon + (n * nb + b) * kBlockBytes;
        h[j] = static_cast<uint16_t>(p[0] | (p[1] << 8));
      }
    }
    uint2 v;
    v.x = h[0] | (static_cast<uint32_t>(h[1]) << 16);
    v.y = h[2] | (static_cast<uint32_t>(h[3]) << 16);
    *reinterpret_cast<uint2*>(tiles + tile * F::kTileBytes + F::kCodeBytes + t * 8) = v;
  }
}

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
    const int i = el / 16, jj = el % 16;
    const int t = cw * 32 + lane;
    const uint8_t* tb = tiles + tile * F::kTileBytes;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(
        tb + ((j * 2 + i / 4) * kLaneSlots + t) * 16 + 4 * (i % 4));
    const int c = static_cast<int>((word >> (2 * jj)) & 3u);
    const uint16_t hb = *reinterpret_cast<const uint16_t*>(tb + F::kCodeBytes + t * 8 + 2 * j);
    w[e] = static_cast<float>(c - 1) * h2f(hb);  // exact
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

// ---- INT8 activations (FmtPQ2I8): the same tiles, the M = 1 kernel ----

using I8 = LaunchTable<FmtPQ2I8>;

template <int MB>
cudaError_t set_i8_smem() {
  static_assert(FmtPQ2I8::kCtasPerSm * (gemv_smem_bytes<FmtPQ2I8, MB>() + 2048) <= 228 * 1024,
                "shared memory budget exceeded");
  return cudaFuncSetAttribute(wstream_kernel<FmtPQ2I8, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              gemv_smem_bytes<FmtPQ2I8, MB>());
}

template <class FI, int MB>
cudaError_t set_i8_smem_of() {
  static_assert(FI::kCtasPerSm * (gemv_smem_bytes<FI, MB>() + 2048) <= 228 * 1024, "shared memory budget exceeded");
  return cudaFuncSetAttribute(wstream_kernel<FI, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              gemv_smem_bytes<FI, MB>());
}

// The INT8 tensor-core kernel (FmtPQ2Q8): one or two activation blocks.
template <int NB>
cudaError_t set_q8_smem() {
  static_assert(mma_smem_bytes<FmtPQ2Q8, NB>() + 2048 <= 228 * 1024, "shared memory budget exceeded");
  return cudaFuncSetAttribute(wstream_mma_kernel<FmtPQ2Q8, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              mma_smem_bytes<FmtPQ2Q8, NB>());
}

cudaError_t setup() {
  cudaError_t e = LaunchTable<F>::setup();
  if (e == cudaSuccess) e = set_q8_smem<1>();
  if (e == cudaSuccess) e = set_q8_smem<2>();
  if (e == cudaSuccess) e = set_i8_smem<1>();
  if (e == cudaSuccess) e = set_i8_smem<2>();
  if (e == cudaSuccess) e = set_i8_smem<4>();
  if (e == cudaSuccess) e = set_i8_smem_of<FmtPQ2I8P, 1>();
  if (e == cudaSuccess) e = set_i8_smem_of<FmtPQ2I8P, 2>();
  if (e == cudaSuccess) e = set_i8_smem_of<FmtPQ2I8P, 4>();
  if (e == cudaSuccess) e = LaunchTable<F>::setup_glu();
  return e;
}

// Activation rows [m0, m0 + MB) of the call in one launch of the CUDA-core
// kernel (the M = 1 grid and stream-K plan).
template <int MB>
cudaError_t launch_i8_rows(const RunParams& p, int m0, const LaunchGeom& g, cudaStream_t s) {
  RunParams q = p;
  q.x = p.x + m0 * p.K;
  q.y = p.y + m0 * p.N;
  q.residual = p.residual != nullptr ? p.residual + m0 * p.N : nullptr;
  q.plan = g.plan_m1;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      I8::config(g.grid_m1, gemv_threads<FmtPQ2I8, MB>(), gemv_smem_bytes<FmtPQ2I8, MB>(), s, attr);
  return cudaLaunchKernelEx(&cfg, wstream_kernel<FmtPQ2I8, MB>, q);
}

// Calls with at least this many activation rows run the integer path on the
// tensor cores (measured: the two-row CUDA-core kernel, one launch, is
// faster at M = 2; from M = 4 the tensor-core kernel, flat in M, is).
constexpr int kQ8MinM = 4;

// All M rows of a call on prepared activations (p.x: the codes, p.x_scale)
// in one launch of the tensor-core kernel (FmtPQ2Q8, the handle's
// one-CTA-per-SM grid and plan): every code read once per call.
cudaError_t launch_q8(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s) {
  RunParams q = p;
  q.plan = g.plan;
  cudaLaunchAttribute attr[1];
  if (M <= 8) {
    const cudaLaunchConfig_t cfg =
        I8::config(g.grid, mma_threads<FmtPQ2Q8, 1>(), mma_smem_bytes<FmtPQ2Q8, 1>(), s, attr);
    return cudaLaunchKernelEx(&cfg, wstream_mma_kernel<FmtPQ2Q8, 1>, q, M);
  }
  const cudaLaunchConfig_t cfg = I8::config(g.grid, mma_threads<FmtPQ2Q8, 2>(), mma_smem_bytes<FmtPQ2Q8, 2>(), s, attr);
  return cudaLaunchKernelEx(&cfg, wstream_mma_kernel<FmtPQ2Q8, 2>, q, M);
}

// M < kQ8MinM: the CUDA-core kernel, up to four rows per launch (each row
// with the same instructions and order in every instantiation).  From
// kQ8MinM rows (or in batch-invariant mode): the activation prologue into the
// handle's workspace, then the integer path on the tensor cores -- two
// launches, the weights read once.  Consecutive launches on the stream are
// ordered by the kernels' grid-dependency waits.
cudaError_t launch_x_int8(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  if ((M >= kQ8MinM || batch_invariant) && p.xq_ws != nullptr) {
    cudaError_t e = prepare_x_int8(p.x, M, p.K, nullptr, 0, p.xq_ws, s);
    if (e != cudaSuccess) return e;
    RunParams q = p;
    q.x = reinterpret_cast<const __half*>(p.xq_ws);
    q.x_scale = reinterpret_cast<const float*>(p.xq_ws + int64_t(M) * p.K);
    q.x_qsum = reinterpret_cast<const int32_t*>(p.xq_ws + int64_t(M) * p.K + 4 * int64_t(M) * (p.K / 128));
    return launch_q8(M, q, g, s);
  }
  int m0 = 0;
  while (m0 < M) {
    const int rem = M - m0;
    const int mb = rem >= 4 ? 4 : (rem >= 2 ? 2 : 1);
    const cudaError_t e = mb == 4   ? launch_i8_rows<4>(p, m0, g, s)
                          : mb == 2 ? launch_i8_rows<2>(p, m0, g, s)
                                    : launch_i8_rows<1>(p, m0, g, s);
    if (e != cudaSuccess) return e;
    m0 += mb;
  }
  return cudaSuccess;
}

// ---- prepared INT8 activations (FmtPQ2I8P) ----

// Rows [m0, m0 + MB) of a call on prepared activations in one launch.
template <int MB>
cudaError_t launch_xq_rows(const RunParams& p, int m0, const LaunchGeom& g, cudaStream_t s) {
  const int64_t G = p.K / 128;
  RunParams q = p;
  q.x = reinterpret_cast<const __half*>(reinterpret_cast<const uint8_t*>(p.x) + m0 * p.K);
  q.x_scale = p.x_scale + m0 * G;
  q.x_qsum = p.x_qsum + m0 * G;
  q.y = p.y + m0 * p.N;
  q.residual = p.residual != nullptr ? p.residual + m0 * p.N : nullptr;
  q.plan = g.plan_m1;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      I8::config(g.grid_m1, gemv_threads<FmtPQ2I8P, MB>(), gemv_smem_bytes<FmtPQ2I8P, MB>(), s, attr);
  return cudaLaunchKernelEx(&cfg, wstream_kernel<FmtPQ2I8P, MB>, q);
}

// As launch_x_int8: fewer than kQ8MinM rows on the CUDA-core kernel, more
// (or batch-invariant mode) in one launch of the tensor-core kernel.
cudaError_t launch_xq(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  if (M >= kQ8MinM || batch_invariant) return launch_q8(M, p, g, s);
  int m0 = 0;
  while (m0 < M) {
    const int rem = M - m0;
    const int mb = rem >= 4 ? 4 : (rem >= 2 ? 2 : 1);
    const cudaError_t e = mb == 4   ? launch_xq_rows<4>(p, m0, g, s)
                          : mb == 2 ? launch_xq_rows<2>(p, m0, g, s)
                                    : launch_xq_rows<1>(p, m0, g, s);
    if (e != cudaSuccess) return e;
    m0 += mb;
  }
  return cudaSuccess;
}

// Packed word of four INT8 codes, lowest byte first.
__device__ __forceinline__ uint32_t pack4(const int (&q)[4]) {
  return (static_cast<uint32_t>(q[0]) & 0xffu) | ((static_cast<uint32_t>(q[1]) & 0xffu) << 8) |
         ((static_cast<uint32_t>(q[2]) & 0xffu) << 16) | (static_cast<uint32_t>(q[3]) << 24);
}

// Prologue without mixing: one warp per group of 128, the GEMV staging's
// quantizer; lane l's packed word is word l of the group.
__global__ void prepare_x_plain_kernel(const unsigned short* __restrict__ x, int64_t groups, int64_t K,
                                       uint32_t* __restrict__ xq, float* __restrict__ xa,
                                       int32_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const int64_t ng = K / 128;
  const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t gi = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; gi < groups;
       gi += wstride) {
    const int64_t base = (gi / ng) * K + (gi % ng) * 128;
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) f[b] = h2f(__ldg(x + base + i8_pos(lane, b)));
    float a;
    int q[4], qsum;
    quant_i8_group(f, a, q, qsum);
    xq[base / 4 + lane] = pack4(q);
    if (lane == 0) {
      xa[gi] = a;
      xs[gi] = qsum;
    }
  }
}

// Prologue with the Hadamard mixing of each block of 1024 inputs, fused with
// the quantization.  One warp per block; lane l holds inputs 32l .. 32l+31
// of it.  The steps are the fp32 steps of the page's transform in its order:
// signs, butterflies h = 1 .. 16 inside the lane, h = 32 .. 512 across lanes
// (the lane whose bit is clear keeps u + w, the other u - w), then times
// 2^-5.  A group of 128 is four lanes: the scale and code sum are reduced
// over them, and each code goes to its staging position in the group.
__global__ void prepare_x_hadamard_kernel(const unsigned short* __restrict__ x, const int8_t* __restrict__ signs,
                                          int64_t blocks, int64_t K, uint8_t* __restrict__ xq,
                                          float* __restrict__ xa, int32_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / 1024;
  const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const unsigned int* xw = reinterpret_cast<const unsigned int*>(x);
  for (int64_t bi = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; bi < blocks;
       bi += wstride) {
    const int64_t b0 = (bi % nb) * 1024;                // block start within the row
    const int64_t base = (bi / nb) * K + b0 + 32 * lane;  // this lane's first input
    float v[32];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const unsigned int u = __ldg(xw + base / 2 + r);
      v[2 * r] = h2f(u & 0xffffu);
      v[2 * r + 1] = h2f(u >> 16);
    }
    if (signs != nullptr) {
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] = v[r] * static_cast<float>(__ldg(signs + b0 + 32 * lane + r));
    }
#pragma unroll
    for (int h = 1; h < 32; h <<= 1)
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (!(r & h)) {
          const float u = v[r], w = v[r + h];
          v[r] = u + w;
          v[r + h] = u - w;
        }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
      const bool upper = (lane & hl) != 0;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float other = __shfl_xor_sync(0xffffffffu, v[r], hl);
        v[r] = upper ? other - v[r] : v[r] + other;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      v[r] = v[r] * 0.03125f;
      amax = fmaxf(amax, fabsf(v[r]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float a = __fdiv_rn(amax, 127.0f);
    const int64_t gstart = (bi / nb) * K + b0 + 128 * (lane >> 2);  // this lane's group
    int qsum = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      int qv = 0;
      if (a != 0.0f) qv = min(127, max(-127, __float2int_rn(__fdiv_rn(v[r], a))));
      qsum += qv;
      const int e = 32 * (lane & 3) + r;                        // position in the group
      const int dst = 16 * (e >> 4) + 4 * (e & 3) + ((e >> 2) & 3);  // its staging position
      xq[gstart + dst] = static_cast<uint8_t>(qv);
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    if ((lane & 3) == 0) {
      const int64_t gi = gstart / 128;  // = m * K/128 + group
      xa[gi] = a;
      xs[gi] = qsum;
    }
  }
}

// One warp per group of 128 activations: the same quantizer as the GEMV's
// staging, written out in plain [M][K] order with the scales [M][K/128].
__global__ void quantize_x_int8_kernel(const unsigned short* __restrict__ x, int64_t groups, int64_t K,
                                       int8_t* __restrict__ q, float* __restrict__ a) {
  const int lane = threadIdx.x & 31;
  const int64_t ng = K / 128;
  const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t gi = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; gi < groups;
       gi += wstride) {
    const int64_t base = (gi / ng) * K + (gi % ng) * 128;
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) f[b] = h2f(__ldg(x + base + i8_pos(lane, b)));
    float sc;
    int qv[4], qsum;
    quant_i8_group(f, sc, qv, qsum);
#pragma unroll
    for (int b = 0; b < 4; ++b) q[base + i8_pos(lane, b)] = static_cast<int8_t>(qv[b]);
    if (lane == 0) a[gi] = sc;
  }
}

}  // namespace

const FormatOps* ops_pq2() {
  static const FormatOps ops = {
      /*format=*/4, F::kKT, F::kTileBytes, /*aux_bytes=*/0,
      &LaunchTable<F>::smem_bytes, &setup, &LaunchTable<F>::launch,
      &prepare, &dequant, /*cb_entries=*/0, /*tile_rows=*/128, /*partial_stride=*/128 * 16,
      /*aux_per_row=*/0, /*m1_ctas_per_sm=*/LaunchTable<F>::kM1CtasPerSm, /*rowgroup=*/0,
      /*launch_x_int8=*/&launch_x_int8, /*row_tables=*/0, /*launch_xq=*/&launch_xq,
      /*launch_glu=*/&LaunchTable<F>::launch_glu, /*tc5_min_m=*/kTc5DefaultMinM, /*split_unit=*/SplitModeOf<F>::value};
  static_assert(I8::kM1CtasPerSm == LaunchTable<F>::kM1CtasPerSm && FmtPQ2I8::kKT == F::kKT &&
                    FmtPQ2I8::kTileBytes == F::kTileBytes,
                "the INT8 path runs on the PQ2_0 handle's tiles, grid and plan");
  return &ops;
}

cudaError_t prepare_x_int8(const void* x, int64_t M, int64_t K, const int8_t* signs, int hadamard_block,
                           void* xq, cudaStream_t s) {
  uint8_t* q = static_cast<uint8_t*>(xq);
  float* xa = reinterpret_cast<float*>(q + M * K);
  int32_t* xs = reinterpret_cast<int32_t*>(q + M * K + 4 * M * (K / 128));
  const unsigned short* xh = static_cast<const unsigned short*>(x);
  if (hadamard_block == 0) {
    const int64_t groups = M * (K / 128);
    const int64_t blocks = (groups + 7) / 8;
    prepare_x_plain_kernel<<<static_cast<int>(blocks > 4096 ? 4096 : blocks), 256, 0, s>>>(
        xh, groups, K, reinterpret_cast<uint32_t*>(q), xa, xs);
  } else {
    const int64_t nblk = M * (K / 1024);
    const int64_t blocks = (nblk + 3) / 4;
    prepare_x_hadamard_kernel<<<static_cast<int>(blocks > 4096 ? 4096 : blocks), 128, 0, s>>>(
        xh, signs, nblk, K, q, xa, xs);
  }
  return cudaGetLastError();
}

cudaError_t quantize_x_int8(const void* x, int64_t M, int64_t K, int8_t* q, float* a, cudaStream_t s) {
  const int64_t groups = M * (K / 128);
  const int64_t blocks = (groups + 7) / 8;
  quantize_x_int8_kernel<<<static_cast<int>(blocks > 4096 ? 4096 : blocks), 256, 0, s>>>(
      static_cast<const unsigned short*>(x), groups, K, q, a);
  return cudaGetLastError();
}

}  // namespace qgemv

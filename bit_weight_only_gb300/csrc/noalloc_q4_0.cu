// noalloc_q4_0.cu -- an entry point for callers that cannot allocate device
// memory: a Q4_0 GEMV that reads the caller's canonical blocks directly and
// keeps its split-K scratch (partial sums and arrival counters) in one
// file-scope static device array of fixed size, so the call itself never
// allocates.  See qgemv_run_q4_0_noalloc in include/qgemv.h.
//
// Kernel: one CTA per (64-row block, 2048-input chunk).  A warp takes eight
// rows; within a Q4_0 block lane l decodes element l, (q - 8) * d exactly in
// fp32, and multiplies it by the chunk's activations staged in shared memory
// as fp32; each row is then reduced across the warp.  With one chunk the CTA
// writes y; with several, each CTA stores its partial sums in the static
// scratch, and the last CTA of a row block (an integer counter) adds the
// chunks in chunk order and writes y -- a fixed order, so repeated calls give
// identical bits.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "formats.h"
#include "qgemv.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB, held by every GPU that loads the library
constexpr int kRowsPerCta = 64;
constexpr int kChunkK = 2048;
constexpr int kThreads = 256;  // 8 warps x 8 rows
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol;
// the device address comes from cudaGetSymbolAddress (per device).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSetup {
  bool done = false;
  cudaError_t err = cudaSuccess;
  unsigned char* scratch = nullptr;  // device address of g_scratch
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;


__global__ void __launch_bounds__(kThreads)
q4_0_noalloc_kernel(const uint8_t* __restrict__ packed, int64_t N, int64_t K,
                    const __half* __restrict__ x, int M, float* __restrict__ y,
                    int* __restrict__ counters, float* __restrict__ partials, int nsplit) {
  extern __shared__ float xs[];  // [M][kChunkK]
  const int64_t rb = blockIdx.x;
  const int split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k0 = static_cast<int64_t>(split) * kChunkK;
  const int64_t kn = (K - k0 < kChunkK) ? (K - k0) : kChunkK;  // multiple of 32

  for (int i = threadIdx.x; i < M * kChunkK; i += kThreads) {
    const int m = i / kChunkK, kk = i % kChunkK;
    xs[i] = kk < kn ? __half2float(x[m * K + k0 + kk]) : 0.f;
  }
  __syncthreads();

  const int64_t nb = K / 32;
  float acc[8][16];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[r][m] = 0.f;

#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t n = rb * kRowsPerCta + warp * 8 + r;
    if (n >= N) continue;
    for (int64_t b = 0; b < kn / 32; ++b) {
      const uint8_t* blk = packed + (n * nb + k0 / 32 + b) * 18;
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(blk[0] | (blk[1] << 8))));
      const int q = lane < 16 ? (blk[2 + lane] & 15) : (blk[2 + lane - 16] >> 4);
      const float w = static_cast<float>(q - 8) * d;  // exact
      const float* xk = xs + b * 32 + lane;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (m < M) acc[r][m] = fmaf(w, xk[m * kChunkK], acc[r][m]);
    }
  }
  // reduce each (row, m) across the warp; lane m then holds row r's value for m
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t n = rb * kRowsPerCta + warp * 8 + r;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m >= M) continue;
      float v = acc[r][m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == m && n < N) {
        if (nsplit == 1) y[m * N + n] = v;
        else partials[(static_cast<int64_t>(split) * M + m) * N + n] = v;
      }
    }
  }
  if (nsplit == 1) return;

  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) last = (atomicAdd(&counters[rb], 1) == nsplit - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kRowsPerCta * M; i += kThreads) {
    const int64_t n = rb * kRowsPerCta + i % kRowsPerCta;
    const int m = i / kRowsPerCta;
    if (n >= N) continue;
    float v = 0.f;
    for (int s = 0; s < nsplit; ++s) v += __ldcg(partials + (static_cast<int64_t>(s) * M + m) * N + n);
    y[m * N + n] = v;
  }
  if (threadIdx.x == 0) counters[rb] = 0;
}

// Once per device, with that device current: the device address of the
// scratch array and the kernel's shared-memory limit.  Only a successful
// set-up is remembered: after a failure (for instance a first call made
// during a stream capture) the error is cleared from the thread's CUDA state
// and the next call tries again.
const DeviceSetup* setup_device(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    s.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.scratch), g_scratch);
    if (s.err == cudaSuccess)
      s.err = cudaFuncSetAttribute(q4_0_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   16 * kChunkK * static_cast<int>(sizeof(float)));
    if (s.err == cudaSuccess) {
      s.done = true;
    } else {
      s.scratch = nullptr;
      cudaGetLastError();
    }
  }
  return &s;
}

int fail(int code, const char* msg) { return qgemv::report_error(code, msg); }

}  // namespace

extern "C" int qgemv_run_q4_0_noalloc(const void* packed, int64_t N, int64_t K, const void* x,
                                      int M, float* y, void* stream) {
  if (!packed || !x || !y) return fail(QGEMV_ERR_ARG, "packed, x or y is NULL");
  if (N <= 0 || K <= 0 || K % 32) return fail(QGEMV_ERR_ARG, "K must be a positive multiple of 32");
  if (M < 1 || M > 16) return fail(QGEMV_ERR_ARG, "M outside [1, 16]");
  if ((reinterpret_cast<uintptr_t>(packed) & 1) || (reinterpret_cast<uintptr_t>(x) & 1) ||
      (reinterpret_cast<uintptr_t>(y) & 3))
    return fail(QGEMV_ERR_ALIGN, "packed and x must be 2-byte aligned, y 4-byte aligned");
  const int64_t nrb = (N + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t nsplit = (K + kChunkK - 1) / kChunkK;
  if (nrb > 2147483647 || nsplit > 65535) return fail(QGEMV_ERR_ARG, "shape too large");
  const size_t counter_bytes = (static_cast<size_t>(nrb) * sizeof(int) + 255) / 256 * 256;
  const size_t partial_bytes = nsplit > 1 ? static_cast<size_t>(nsplit) * M * N * sizeof(float) : 0;
  if (counter_bytes + partial_bytes > kScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "this shape needs %zu bytes of scratch (ceil(K/2048) * M * N * 4 + counters); the "
             "static scratch holds %zu",
             counter_bytes + partial_bytes, kScratchBytes);
    return fail(QGEMV_ERR_ARG, buf);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(QGEMV_ERR_CUDA, "no usable device");
  const DeviceSetup* s = setup_device(dev);
  if (!s->done) {
    char buf[256];
    snprintf(buf, sizeof(buf), "scratch set-up failed (retried on the next call): %s",
             cudaGetErrorString(s->err));
    return fail(QGEMV_ERR_CUDA, buf);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* counters = reinterpret_cast<int*>(s->scratch);
  float* partials = reinterpret_cast<float*>(s->scratch + counter_bytes);
  // The counters must start at zero; earlier calls leave them at zero, but a
  // call that failed midway might not, so clear them every time.
  e = cudaMemsetAsync(counters, 0, counter_bytes, st);
  if (e != cudaSuccess) return fail(QGEMV_ERR_CUDA, cudaGetErrorString(e));
  dim3 grid(static_cast<unsigned>(nrb), static_cast<unsigned>(nsplit));
  q4_0_noalloc_kernel<<<grid, kThreads, M * kChunkK * sizeof(float), st>>>(
      static_cast<const uint8_t*>(packed), N, K, static_cast<const __half*>(x), M, y, counters,
      partials, static_cast<int>(nsplit));
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(QGEMV_ERR_CUDA, cudaGetErrorString(e));
  return qgemv::report_error(QGEMV_OK, "");
}

// tc_kernel.cuh -- the tensor-core GEMV for M = 5..16 activation rows.
//
// Above a few activation rows the CUDA-core kernel is bound by its fp32
// FMAs (2 * M per weight).  Here the weights of each tile are decoded once
// into fp16 in shared memory and multiplied on the tensor cores
// (mma.m16n8k16, f16 x f16 -> f32), the activations padded to 16 rows:
//
//   * Same prepared tiles, TMA ring, stream-K split, CTA plans and polled
//     split-K fix-up as gemv_kernel.
//   * Sixteen warps, two per k-slice: warp (slice s, half h) covers slice s
//     of every tile for two of the four row groups (rows 4l + j, l = 0..31,
//     j = 2h, 2h + 1).  Lane l decodes its row of group j (the format's
//     tc_decode_row, exact fp16 values or integer codes) into a padded row of
//     a per-warp buffer (conflict-free 128-bit stores), then the warp runs
//     the MMAs of the group's four 8-row n-tiles with ldmatrix-loaded B
//     fragments.  Only __syncwarp orders a warp's decode and MMAs.
//   * A fragments (x, 16 x 16 per k step) are read from global memory into
//     registers, a tile ahead; rows m >= M and columns k >= K are zero.
//   * Formats with a block scale (Q4_0: 32 k, PQ2_0: 128 k) accumulate the
//     codes' products per block and add d * block into the fp32 accumulator,
//     so no value is rounded before the fp32 sums.
//   * At the end of a row tile the eight slices' partial results are added
//     in a fixed tree order through shared memory, then stored to y or to
//     the stream-K partial slots.
#pragma once

#include "gemv_kernel.cuh"

namespace qgemv {

constexpr int kTcHalves = 2;                   // warps per k-slice
constexpr int kTcGroups = 4 / kTcHalves;       // row groups per warp
constexpr int kTcWarps = kSlices * kTcHalves;  // 16
constexpr int kTcThreads = 32 * kTcWarps;      // 512

template <class F>
__host__ __device__ constexpr int tc_row_halfs() { return F::kKW + 8; }  // padded row, halfs
template <class F>
__host__ __device__ constexpr int tc_wbuf_bytes() { return 32 * tc_row_halfs<F>() * 2; }  // per warp
// tree reduction: (2 halves x 4 slices) warps x 32 lanes x 32 floats
constexpr int kTcRedBytes = kTcHalves * 4 * 32 * (kTcGroups * 16) * 4;
template <class F>
__host__ __device__ constexpr int tc_scratch_bytes() {
  return kTcWarps * tc_wbuf_bytes<F>() > kTcRedBytes ? kTcWarps * tc_wbuf_bytes<F>() : kTcRedBytes;
}
template <class F>
__host__ __device__ constexpr int tc_smem_bytes() {
  return F::kTcStages * F::kTileBytes + tc_scratch_bytes<F>() + F::kSharedBytes + 2 * F::kTcStages * 8;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp16 pair (x[m][k], x[m][k+1]), zero beyond M rows or K columns.
__device__ __forceinline__ uint32_t x_pair(const GemvParams& p, int M, int m, int64_t k) {
  if (m >= M || k >= p.K) return 0u;
  const unsigned short* row = reinterpret_cast<const unsigned short*>(p.x) + m * p.K;
  if ((p.K & 1) == 0) return __ldg(reinterpret_cast<const unsigned int*>(row + k));  // k even: aligned
  const uint32_t lo = __ldg(row + k);
  const uint32_t hi = k + 1 < p.K ? __ldg(row + k + 1) : 0u;
  return lo | (hi << 16);
}

// A fragments (16 rows x 16 k) of the warp's slice in k tile kt.
template <class F>
__device__ __forceinline__ void load_afrags(uint32_t (&a)[F::kKW / 16][4], const GemvParams& p, int M, int kt,
                                            int slice, int lane) {
  const int q = lane & 3, gi = lane >> 2;
  const int64_t kb = static_cast<int64_t>(kt) * F::kKT + slice * F::kKW + 2 * q;
#pragma unroll
  for (int ks = 0; ks < F::kKW / 16; ++ks) {
    const int64_t k = kb + 16 * ks;
    a[ks][0] = x_pair(p, M, gi, k);
    a[ks][1] = x_pair(p, M, gi + 8, k);
    a[ks][2] = x_pair(p, M, gi, k + 8);
    a[ks][3] = x_pair(p, M, gi + 8, k + 8);
  }
}

template <class F>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(const GemvParams p, int M) {
  constexpr int NS = F::kTcStages;
  constexpr int TB = F::kTileBytes;
  constexpr int KS = F::kKW / 16;  // k16 steps per slice
  constexpr int RH = tc_row_halfs<F>();
  constexpr int NT = kTcThreads;
  constexpr int BS = F::kTcBlockSteps;  // k16 steps per scale block, 0: none

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* scratch = smem + NS * TB;
  uint8_t* fsh = scratch + tc_scratch_bytes<F>();
  uint64_t* full = reinterpret_cast<uint64_t*>(fsh + F::kSharedBytes);
  uint64_t* empty = full + NS;
  __shared__ volatile int s_abort;
  __shared__ int s_seg[2];
  __shared__ __align__(16) CtaPlan s_plan;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int q = lane & 3, gi = lane >> 2;
  const int slice = warp % kSlices;
  const int hf = warp / kSlices;  // row groups 2 hf, 2 hf + 1
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t t0 = stream_split(c, p.T, G);
  const int64_t t1 = stream_split(c + 1, p.T, G);
  const int64_t ntiles = t1 - t0;
  const int64_t rt_first = div_fast(t0, p.nKT);

  // Barriers and the first tiles, as in gemv_kernel.
  const bool elected = (tid == 0);
  uint64_t pol = 0;
  int64_t n_issued = 0;
  if (elected) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTcWarps);
    }
    s_abort = 0;
    fence_mbarrier_init();
    pol = l2_policy_evict_first();
    for (; n_issued < NS - 1 && n_issued < ntiles; ++n_issued) {
      mbar_arrive_expect_tx(&full[n_issued], TB);
      bulk_g2s(ring + n_issued * TB, p.tiles + (t0 + n_issued) * TB, TB, &full[n_issued], pol);
    }
  }
  fetch_plan(&s_plan, p.plan, c, tid);
  if constexpr (F::kCbEntries > 0) {
    if (p.seg_of_rt != nullptr && tid == 0 && ntiles > 0) {
      const int64_t nRT = div_fast(p.T, p.nKT);
      s_seg[0] = __ldg(p.seg_of_rt + rt_first);
      s_seg[1] = rt_first + 1 < nRT ? __ldg(p.seg_of_rt + rt_first + 1) : s_seg[0];
    }
  }
  F::template init_shared<NT>(fsh, table_of<F>(p, rt_first), warp, lane);
  __syncthreads();

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t rt = rt_first;
  int kt = static_cast<int>(t0 - rt * p.nKT);
  uint32_t afr[KS][4];
  if (ntiles > 0) load_afrags<F>(afr, p, M, kt, slice, lane);

  // acc[jj][nt]: rows 32 nt + 4 (2q + e) + j with j = kTcGroups hf + jj,
  // e = 0, 1 (columns of the D fragment); [0..1] for activation row gi,
  // [2..3] for gi + 8.
  float acc[kTcGroups][4][4];
#pragma unroll
  for (int j = 0; j < kTcGroups; ++j)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.f;

  __half* wrow = reinterpret_cast<__half*>(scratch + warp * tc_wbuf_bytes<F>());
  const uint32_t wbuf_base = smem_u32(wrow);
  // ldmatrix.x4 row addresses: matrix i = lane >> 3 covers rows (lane & 7)
  // of the n-tile and k half ((i & 1) * 8) of k step (i >> 1).
  const uint32_t ldsm_off = ((lane & 7) * RH + ((lane >> 3) & 1) * 8 + (lane >> 4) * 16) * 2;

  int s = 0;
  uint32_t ph = 0;
  int su = static_cast<int>(n_issued % NS);
  uint32_t phu = static_cast<uint32_t>((n_issued / NS) & 1);
  for (int64_t i = 0; i < ntiles; ++i) {
    if constexpr (F::kCbEntries > 0) {
      if (p.seg_of_rt != nullptr && kt == 0 && i > 0) {
        __syncthreads();
        if (s_seg[1] != s_seg[0]) rebuild_table<F, NT>(fsh, table_of<F>(p, rt), warp, lane);
        __syncthreads();
        if (tid == 0) {
          const int64_t nRT = div_fast(p.T, p.nKT);
          s_seg[0] = s_seg[1];
          s_seg[1] = rt + 1 < nRT ? __ldg(p.seg_of_rt + rt + 1) : s_seg[0];
        }
      }
    }
    bool abort = s_abort != 0;
    if (elected && !abort && n_issued < ntiles) {
      if (n_issued >= NS && !mbar_wait_bounded(&empty[su], phu ^ 1)) {
        atomicOr(p.err, kErrTimeoutEmpty);
        s_abort = 1;
        abort = true;
      } else {
        mbar_arrive_expect_tx(&full[su], TB);
        bulk_g2s(ring + su * TB, p.tiles + (t0 + n_issued) * TB, TB, &full[su], pol);
        ++n_issued;
        if (++su == NS) { su = 0; phu ^= 1; }
      }
    }
    const int kt_next = (kt + 1 == p.nKT) ? 0 : kt + 1;
    uint32_t anext[KS][4];
    if (i + 1 < ntiles) load_afrags<F>(anext, p, M, kt_next, slice, lane);

    const bool ok = !abort && mbar_wait_bounded(&full[s], ph);
    if (!ok) {
      if (!abort && lane == 0) atomicOr(p.err, kErrTimeoutFull);
      s_abort = 1;
    } else {
      const uint8_t* stage = ring + s * TB;
#pragma unroll 1
      for (int jj = 0; jj < kTcGroups; ++jj) {
        const int j = kTcGroups * hf + jj;
        F::tc_decode_row(stage, slice, j, lane, fsh, reinterpret_cast<uint32_t*>(wrow + lane * RH));
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const uint32_t bbase = wbuf_base + nt * 8 * RH * 2 + ldsm_off;
          if constexpr (BS == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {
              uint32_t b[4];
              ldsm_x4(bbase + ks * 16 * 2, b);
              mma16816(acc[jj][nt], afr[ks], b[0], b[1]);
              mma16816(acc[jj][nt], afr[ks + 1], b[2], b[3]);
            }
          } else {
#pragma unroll
            for (int blk = 0; blk < KS / BS; ++blk) {
              float tmp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int ks = blk * BS; ks < (blk + 1) * BS; ks += 2) {
                uint32_t b[4];
                ldsm_x4(bbase + ks * 16 * 2, b);
                mma16816(tmp, afr[ks], b[0], b[1]);
                mma16816(tmp, afr[ks + 1], b[2], b[3]);
              }
              const float d0 = F::tc_scale(stage, slice, 8 * nt + 2 * q, j, blk);
              const float d1 = F::tc_scale(stage, slice, 8 * nt + 2 * q + 1, j, blk);
              acc[jj][nt][0] = fmaf(d0, tmp[0], acc[jj][nt][0]);
              acc[jj][nt][1] = fmaf(d1, tmp[1], acc[jj][nt][1]);
              acc[jj][nt][2] = fmaf(d0, tmp[2], acc[jj][nt][2]);
              acc[jj][nt][3] = fmaf(d1, tmp[3], acc[jj][nt][3]);
            }
          }
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (++s == NS) { s = 0; ph ^= 1; }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) afr[ks][e] = anext[ks][e];

    const bool row_end = (kt_next == 0) || (i + 1 == ntiles);
    const int64_t cur_rt = rt;
    kt = kt_next;
    if (kt_next == 0) ++rt;
    if (!row_end) continue;

    // ---- row-tile epilogue: add the eight slices' results in a fixed tree ----
    // red: [half][4 slots][kTcGroups * 4][32 lanes] float4
    float4* red = reinterpret_cast<float4*>(scratch);
    constexpr int kItems = kTcGroups * 4;
    named_bar_sync(1, NT);  // every warp is done with its row buffer
#pragma unroll 1
    for (int width = 4; width >= 1; width >>= 1) {
      if (slice >= width && slice < 2 * width) {
#pragma unroll
        for (int jj = 0; jj < kTcGroups; ++jj)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
            red[((hf * 4 + slice - width) * kItems + jj * 4 + nt) * 32 + lane] =
                make_float4(acc[jj][nt][0], acc[jj][nt][1], acc[jj][nt][2], acc[jj][nt][3]);
      }
      named_bar_sync(1, NT);
      if (slice < width) {
#pragma unroll
        for (int jj = 0; jj < kTcGroups; ++jj)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const float4 v = red[((hf * 4 + slice) * kItems + jj * 4 + nt) * 32 + lane];
            acc[jj][nt][0] += v.x;
            acc[jj][nt][1] += v.y;
            acc[jj][nt][2] += v.z;
            acc[jj][nt][3] += v.w;
          }
      }
      named_bar_sync(1, NT);
    }
    if (slice == 0) {
      const bool owner = (cur_rt * p.nKT >= t0) && ((cur_rt + 1) * p.nKT <= t1);
      const int side = (cur_rt * p.nKT <= t0) ? 0 : 1;
      float* my_part = p.partials + (c * 2 + side) * kPartialStride;
#pragma unroll
      for (int jj = 0; jj < kTcGroups; ++jj)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = gi + (e >> 1) * 8;
            const int r = 32 * nt + 4 * (2 * q + (e & 1)) + kTcGroups * hf + jj;
            if (m < M) {
              if (owner) {
                const int64_t n = cur_rt * kTileRows + r;
                if (n < p.N) p.y[m * p.N + n] = acc[jj][nt][e];
              } else {
                st_relaxed_f32(my_part + m * kTileRows + r, acc[jj][nt][e]);
              }
            }
          }
    }
#pragma unroll
    for (int j = 0; j < kTcGroups; ++j)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.f;
  }

  if (elected && s_abort != 0) {
    for (int64_t u = (n_issued > NS ? n_issued - NS : 0); u < n_issued; ++u)
      mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
  }

  // split row tiles: the shared polled-slot finisher, with M activation rows
  float* s_sub = reinterpret_cast<float*>(scratch);
  wait_plan();
  if (s_plan.seg_rt[0] >= 0) finish_segment<kTileRows, kMaxM, NT>(p, kPartialStride, s_plan, 0, nullptr, 1.0f, s_sub, tid, M);
  if (s_plan.seg_rt[1] >= 0) finish_segment<kTileRows, kMaxM, NT>(p, kPartialStride, s_plan, 1, nullptr, 1.0f, s_sub, tid, M);
}

}  // namespace qgemv

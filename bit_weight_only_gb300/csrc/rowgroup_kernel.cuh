// rowgroup_kernel.cuh -- the M = 1 CUDA-core kernel of the table formats
// (CBK4, CBK8) for matrices whose whole-row split balances as well as the
// stream-K split: no row is shared between CTAs, so there are no partial
// sums and no split-K finish.
//
// Work unit: one row group of a prepared 128-row tile (rows 4l + j,
// l = 0..31, for one j) over all of K -- 32 rows.  The tile layout
// [j][h][t][16 B] keeps a row group's codes of one k tile in two contiguous
// 4 KB pieces (h = 0, 1), so a unit streams 8 KB per k tile with plain TMA
// bulk copies from the same prepared tiles the other kernels read.  CTA c
// takes units [c*U/G, (c+1)*U/G) whole (U = 4 * row tiles).
//
// A stage holds kRgSub consecutive k tiles of a unit (32 KB).  As in
// wstream_kernel's tile parity, the sixteen warps form two halves that take
// alternate stages, one warp per slice, each half with its own pipeline over
// two of the four stages; a lane computes its one row of the unit for its
// slice (the format's tile_math with one row per lane), and at the end of a
// unit the sixteen slices' sums of each row are added in a fixed order and
// stored to y.  A warp stages the activations of a whole stage at once and
// fetches those of its next stage a stage ahead.  Every wait is bounded and
// reported as in wstream_kernel.
#pragma once

#include "gemv_kernel.cuh"

namespace qgemv {

constexpr int kRgSub = 4;                   // k tiles per stage
constexpr int kRgPiece = kLaneSlots * 16;   // 4096: one (j, h) piece of a tile
constexpr int kRgThreads = 512;

template <class F>
__host__ __device__ constexpr int rg_xs_floats() { return (F::kKW / 2) * 2; }  // per warp and k tile, M = 1
template <class F>
__host__ __device__ constexpr int rg_pre_bytes() {
  return kRgSub * 2 * kRgPiece                     // stage 0
         + 16 * kRgSub * rg_xs_floats<F>() * 4     // staged x, per warp and k tile of a stage
         + 16 * kTileRows * 4                      // per-slice row sums
         + 128;                                    // mbarriers
}
// Shared memory: stage 0, x, sums and barriers below the 64 KB-aligned
// table, the other three stages above it.
template <class F>
__host__ __device__ constexpr int rg_smem_bytes() {
  return kTableAlign + F::kSharedBytes + 3 * kRgSub * 2 * kRgPiece;
}

template <class F>
__global__ void __launch_bounds__(kRgThreads, 1) rowgroup_stream_kernel(const RunParams p) {
  constexpr int M = 1;
  constexpr int NS = 4;
  constexpr int SB = kRgSub * 2 * kRgPiece;  // stage bytes
  constexpr int NT = kRgThreads;
  constexpr int XS_FLOATS = rg_xs_floats<F>();
  static_assert(F::kTileBytes == kRowsPerLane * 2 * kRgPiece, "tile = four row groups of two pieces");
  static_assert(F::kSharedBytes == kTableAlign, "one 64 KB table");
  static_assert(rg_pre_bytes<F>() + kTablePreSlack <= kTableAlign, "pre-table layout");

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring0 = smem;
  float* xs_all = reinterpret_cast<float*>(smem + SB);
  float* red = xs_all + 16 * kRgSub * XS_FLOATS;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 16 * kTileRows);
  uint64_t* empty = full + NS;
  uint64_t* spare = empty + NS;  // takes the releases of a stage's earlier k tiles
  __shared__ volatile int s_abort;

  if (static_cast<int>(blockIdx.x) == p.skip_cta) return;  // test hook (QGEMV_FAULT_SKIP_CTA)
  const uint32_t base = smem_u32(smem);
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  const uint32_t R0 = (base + (kTableAlign - 1)) & ~uint32_t(kTableAlign - 1);
  if (R0 - base < uint32_t(rg_pre_bytes<F>()) || R0 + kTableAlign + (NS - 1) * SB > base + dyn) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
    return;
  }
  uint8_t* fsh = smem + (R0 - base);
  uint8_t* ringN = fsh + kTableAlign;
  auto stage_ptr = [&](int st) { return st == 0 ? ring0 : ringN + (st - 1) * SB; };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int slice = warp & 7;
  const int half = warp >> 3;
  const int nKT = static_cast<int>(p.nKT);
  const int64_t U = div_fast(p.T, p.nKT) * kRowsPerLane;  // units
  const int64_t G = gridDim.x;
  const int64_t u0 = stream_split<0>(blockIdx.x, U, G);
  const int64_t u1 = stream_split<0>(blockIdx.x + 1, U, G);
  const int nch = (nKT + kRgSub - 1) / kRgSub;  // stages per unit
  const int nq = static_cast<int>(u1 - u0) * nch;

  // Stage q of the run: unit u0 + q / nch, k tiles kt0 .. kt0 + nsub - 1.
  auto issue = [&](int q, uint64_t pol) {
    const int64_t u = u0 + q / nch;
    const int kt0 = (q % nch) * kRgSub;
    const int nsub = min(kRgSub, nKT - kt0);
    const int64_t rt = u >> 2;
    const int j = static_cast<int>(u & 3);
    const int st = q % NS;
    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nsub * 2 * kRgPiece));
    for (int cidx = 0; cidx < nsub; ++cidx)
      for (int h = 0; h < 2; ++h)
        bulk_g2s(stage_ptr(st) + (cidx * 2 + h) * kRgPiece,
                 p.tiles + (rt * p.nKT + kt0 + cidx) * F::kTileBytes + (j * 2 + h) * kRgPiece, kRgPiece,
                 &full[st], pol);
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);  // the eight warps of the stage's half
    }
    mbar_init(spare, 1);
    s_abort = 0;
    fence_mbarrier_init();
    // the first stage of each half only; the main loop fills the others
    // after the grid dependency (see wstream_kernel)
    const uint64_t pol = l2_policy_evict_first();
    for (int q = 0; q < 2 && q < nq; ++q) issue(q, pol);
  }
  const int64_t rt_first = u0 >> 2;
  F::template init_shared<NT>(fsh, table_of<F>(p, rt_first), warp, lane);
  __syncthreads();

  float* xs = xs_all + warp * kRgSub * XS_FLOATS;
  RowAcc<M, 1> acc;
  acc.init(red, 0, 0, lane);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const bool stacked = p.seg_of_rt != nullptr;
  // x of the warp's next stage (its kRgSub k tiles), a stage ahead
  typename F::XRegs xr[kRgSub];
  typename F::XScale xscale;  // per-lane activation scaling, the same for every tile
  F::x_scales(xscale, lane);
  auto kt_of_stage = [&](int q) { return (q % nch) * kRgSub; };
  auto load_stage_x = [&](int q) {
    const int kt = kt_of_stage(q);
#pragma unroll
    for (int cidx = 0; cidx < kRgSub; ++cidx)
      if (kt + cidx < nKT) F::template load_x<M>(xr[cidx], p, kt + cidx, slice, lane);
  };
  if (half < nq) load_stage_x(half);

  // Each half's first thread fills, at its stage q, the stage of its stage
  // q - 2 (released one stage ago; for q < 2 one not used yet) with stage
  // q + NS - 2; the prologue issued stages 0 and 1.
  const bool leader = (lane == 0) && (slice == 0);
  const uint64_t lpol = leader ? l2_policy_evict_first() : 0;
  int q_last = -1;  // leader: last stage of its parity issued
  for (int q = half; q < 2 && q < nq; q += 2) q_last = q;
  int64_t rt_prev = rt_first;
  for (int64_t u = u0; u < u1; ++u) {
    const int64_t rt = u >> 2;
    const int j = static_cast<int>(u & 3);
    if (stacked && rt != rt_prev) {  // a new row tile may use another codebook
      __syncthreads();
      if (__ldg(p.seg_of_rt + rt) != __ldg(p.seg_of_rt + rt_prev))
        rebuild_table<F, NT>(fsh, table_of<F>(p, rt), warp, lane);
      __syncthreads();
      rt_prev = rt;
    }
    const int qb = static_cast<int>(u - u0) * nch;
#pragma unroll 1
    for (int q = qb + ((qb ^ half) & 1); q < qb + nch; q += 2) {
      bool abort = s_abort != 0;
      const int qn = q + NS - 2;
      // stages 0 and 1 came from the prologue: never fill a stage twice
      if (leader && !abort && qn >= 2 && qn < nq) {
        if (qn >= NS && !mbar_wait_bounded(&empty[qn % NS], static_cast<uint32_t>(((qn - NS) / NS) & 1))) {
          atomicOr(p.err, kErrTimeoutEmpty);
          s_abort = 1;
          abort = true;
        } else {
          issue(qn, lpol);
          q_last = qn;
        }
      }
      const int st = q % NS;
      const int kt0 = kt_of_stage(q);
      const int nsub = min(kRgSub, nKT - kt0);
      // stage this stage's x, then fetch that of the warp's next stage
      float xsum[F::kSumGroups][M];
      __syncwarp();
#pragma unroll
      for (int cidx = 0; cidx < kRgSub; ++cidx)
        if (cidx < nsub) F::template stage_x<M>(xs + cidx * XS_FLOATS, xsum, xr[cidx], xscale, lane);
      __syncwarp();
      if (q + 2 < nq) load_stage_x(q + 2);
      const bool ok = !abort && mbar_wait_bounded(&full[st], static_cast<uint32_t>((q / NS) & 1));
      if (!ok) {
        if (!abort && lane == 0) atomicOr(p.err, kErrTimeoutFull);
        s_abort = 1;
      }
#pragma unroll 1
      for (int cidx = 0; ok && cidx < nsub; ++cidx) {
        // the stage is released after its last k tile's codes are loaded
        F::template tile_math<M, 1>(stage_ptr(st) + cidx * 2 * kRgPiece, xs + cidx * XS_FLOATS, xsum, acc, fsh,
                                    slice, 0, lane, cidx + 1 == nsub ? &empty[st] : spare);
      }
    }
    // end of the unit: add the sixteen slice sums of each row in a fixed order
    acc.flush(red, half * 8 + slice, 0, lane);
    named_bar_sync(1, NT);
    if (tid < 32) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 16; ++w) v += red[w * kTileRows + kRowsPerLane * tid];
      const int64_t n = rt * kTileRows + kRowsPerLane * tid + j;
      if (n < p.N) store_y(p, n, __fmul_rn(v, F::kOutScale));
    }
    named_bar_sync(1, NT);
    acc.reset();
  }
  // Never leave while a copy issued by this half may still be landing (only
  // after an aborted run): wait for the last fill of each of its stages.
  if (leader && s_abort != 0) {
    for (int q = q_last; q >= 0 && q > q_last - NS; q -= 2)
      mbar_wait_bounded(&full[q % NS], static_cast<uint32_t>((q / NS) & 1));
  }
}

}  // namespace qgemv

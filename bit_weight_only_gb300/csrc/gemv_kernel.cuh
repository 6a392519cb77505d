// gemv_kernel.cuh -- the CUDA-core weight-streaming GEMV kernel of the tile
// formats (Q4_0, PQ2_0, CBK4, CBK8, and PQ2_0 with INT8 activations), used
// for M = 1, and the stream-K finisher shared by every kernel.
//
//   y[m][n] = sum_k x[m][k] * w[n][k]      (1 <= M <= 16, fp32 accumulation)
//
// Design (a persistent grid: one CTA per SM, or two for formats without a
// table):
//   * The weights were re-laid out at create time into "tiles" of
//     kTileRows (128) output rows x F::kKT inputs, each tile one contiguous
//     run of F::kTileBytes bytes, stored in (row tile, k tile) order.  The
//     whole matrix is therefore one sequential byte stream.  Inside a tile,
//     the k range is cut into kSlices (8) slices of F::kKW inputs, and the
//     packed codes of slice s for rows 4l..4l+3 sit at lane slot t = 32s + l
//     (16 bytes per row), so one 128-bit shared load per row per lane and no
//     bank conflicts.
//   * The stream of T tiles is split evenly over the grid ("stream-K"): CTA
//     c owns tiles [c*T/G, (c+1)*T/G).  A row tile cut by CTA boundaries is
//     finished, after the main loop, by all of its contributors together:
//     each sums a slice of the rows from polled partial slots, in a fixed
//     order (no atomics, no fences; bitwise reproducible).
//   * TMA bulk copies (cp.async.bulk, evict-first L2 policy) fill a ring of
//     F::stages(M) shared-memory stages, signalled through mbarriers.  There
//     is no separate producer warp: one thread of a computing warp issues.
//   * Eight warps (one per slice; two CTAs per SM) or sixteen.  With sixteen
//     (the table formats) the two warps of a slice take alternate tiles
//     ("tile parity"), each for all four rows of its lanes; tile j sits in
//     stage j mod 4, so each half of the CTA owns every second stage and
//     runs its own pipeline.  Each lane loads its codes, releases the stage,
//     then decodes in registers and accumulates in fp32.  The activations of
//     the slice are staged per tile in a per-warp shared buffer (prefetched
//     from global one tile ahead), in the pre-scaled form the format's decode
//     wants.
//   * At the end of a row tile the slices' (and halves') partial sums are
//     added in a fixed order through shared memory and written to y (or to
//     the stream-K workspace).
// Every mbarrier wait is bounded; a timeout sets an error word, skips the
// remaining math and still meets every named barrier, so the kernel always
// returns.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "device_common.cuh"

namespace qgemv {

constexpr int kSlices = 8;                         // k slices per tile
constexpr int kLaneSlots = 32 * kSlices;           // 256 (slice, lane) slots
constexpr int kRowsPerLane = 4;
constexpr int kTileRows = 32 * kRowsPerLane;       // 128
constexpr int kMaxM = 16;
constexpr int kPartialStride = kTileRows * kMaxM;  // floats per partial slot

// Stream-K plan of one CTA, computed on the host when the handle is made:
// the row tiles (at most the first and the last of its run) that it shares
// with other CTAs, and its place among their contributors.
struct CtaPlan {
  int64_t seg_rt[2];     // shared row tiles, -1 if none
  int64_t seg_cf[2];     // first contributor of each
  int32_t seg_S[2];      // number of contributors
  int32_t seg_r0[2];     // this CTA's slice of the rows: [r0, r0 + nr)
  int32_t seg_nr[2];
  int32_t seg_flags[2];  // bit 0: the first contributor's run began earlier (its side-1 slot);
                         // bit 1: this CTA finishes the whole row tile (kWholeFinishItems)
};
static_assert(sizeof(CtaPlan) == 64, "CtaPlan is copied in 16-byte pieces");

struct RunParams {
  const uint8_t* tiles;  // prepared tiles (device)
  const __half* x;       // [M][K] fp16
  float* y;              // [M][N] fp32
  float* partials;       // [gridDim.x][2][partial stride], all ones between calls
  const CtaPlan* plan;   // [gridDim.x]
  const int32_t* seg_of_rt;  // stacked table formats and AQLM 2x8: [row tiles] segment of each; else null
  int* err;              // error word (kErr* bits)
  const void* aux;       // format data (codebooks ...)
  int64_t N, K;
  int64_t T;             // tiles in the stream = nRT * nKT
  int nKT;               // k tiles per row tile
  int skip_cta;          // test hook: this CTA does nothing (-1: none)
  const float* residual; // [M][N] fp32 added to y in the store (may be y itself), or null
  // PQ2_0 on prepared INT8 activations (x then points to their codes):
  // group scales and group code sums, [M][K/128]; null otherwise
  const float* x_scale;
  const int32_t* x_qsum;
  // PQ2_0 handles in INT8 mode: device workspace for the activation prologue
  // of runs with several rows (qgemv_xq_bytes(16, K) bytes), or null
  uint8_t* xq_ws;
};

// y[idx] = v, plus the residual in one fp32 add (never fused with the
// product that made v) when the call has one.  The residual element is read
// and y written by the same thread, so residual may alias y.
__device__ __forceinline__ void store_y(const RunParams& p, int64_t idx, float v) {
  p.y[idx] = p.residual != nullptr ? __fadd_rn(v, p.residual[idx]) : v;
}

// Warps per slice for a given M: two while the whole accumulator set of a
// lane fits in 128 registers, one above.
// A format with F::kCtasPerSm == 2 runs two independent CTAs of eight warps
// per SM instead (their phases differ, which hides more latency; only
// formats without a 64 KB table fit twice).
template <class F>
__host__ __device__ constexpr int wps_for(int M) { return (M <= 4 && F::kCtasPerSm == 1) ? 2 : 1; }

// x rows stored per k pair; padded so vector loads stay aligned.
__host__ __device__ constexpr int mpad(int M) { return M <= 2 ? M : (M + 3) / 4 * 4; }

// Row stride (floats) of the cross-slice reduction buffer.
__host__ __device__ constexpr int acc_stride(int M) { return M > 8 ? mpad(M) : M; }

// Accumulators of one lane's RPW rows over the k tiles of a row tile.
// M <= 8: registers.  M > 8: the lane's own rows of the slice's reduction
// buffer in shared memory, so the registers stay with the inner loop.
template <int M, int RPW, bool kInSmem = (M > 8)>
struct RowAcc;

template <int M, int RPW>
struct RowAcc<M, RPW, false> {
  float v[RPW][M];
  __device__ __forceinline__ void init(float*, int, int, int) { reset(); }
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int j = 0; j < RPW; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) v[j][m] = 0.f;
  }
  // row j (of the lane's RPW rows) += d * a
  __device__ __forceinline__ void add_row(int j, float d, const float (&a)[M]) {
#pragma unroll
    for (int m = 0; m < M; ++m) v[j][m] = fmaf(d, a[m], v[j][m]);
  }
  __device__ __forceinline__ void flush(float* red, int slice, int half, int lane) {
#pragma unroll
    for (int j = 0; j < RPW; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m)
        red[(slice * kTileRows + kRowsPerLane * lane + half * RPW + j) * M + m] = v[j][m];
  }
};

template <int M, int RPW>
struct RowAcc<M, RPW, true> {
  static constexpr int RS = acc_stride(M);
  float* rows;
  __device__ __forceinline__ void init(float* red, int slice, int half, int lane) {
    rows = red + (slice * kTileRows + kRowsPerLane * lane + half * RPW) * RS;
    reset();
  }
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < RPW * RS; i += 4)
      *reinterpret_cast<float4*>(rows + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __device__ __forceinline__ void add_row(int j, float d, const float (&a)[M]) {
    float* r = rows + j * RS;
#pragma unroll
    for (int m = 0; m < M; m += 4) {
      float4 o = lds128f(r + m);
      o.x = fmaf(d, a[m], o.x);
      if (m + 1 < M) o.y = fmaf(d, a[m + 1], o.y);
      if (m + 2 < M) o.z = fmaf(d, a[m + 2], o.z);
      if (m + 3 < M) o.w = fmaf(d, a[m + 3], o.w);
      *reinterpret_cast<float4*>(r + m) = o;
    }
  }
  __device__ __forceinline__ void flush(float*, int, int, int) {}
};

// Dynamic shared memory of wstream_kernel<F, M>.
// Tile parity (formats with F::kTileParity, which cannot run two CTAs per
// SM): the two warps of a slice take alternate tiles, each for all four rows
// of its lanes, instead of splitting the rows; the two halves of the CTA then
// do not wait on the same tile.  Their partial sums meet at the row-tile end.
template <class F, int M>
__host__ __device__ constexpr bool tile_parity() { return F::kTileParity && wps_for<F>(M) == 2; }
// partial-sum slots of the cross-slice reduction (per slice, and per half
// with tile parity)
template <class F, int M>
__host__ __device__ constexpr int red_slots() { return tile_parity<F, M>() ? 2 * kSlices : kSlices; }

// Table formats (a 64 KB lane-replicated table) place the table on a 64 KB
// boundary of the shared window, so that one PRMT of an index byte with
// (table >> 16, lane * 4) is the whole address of an entry, with no add per
// lookup.  Before the table ("pre", at most 64 KB less the window offset of
// the dynamic area): stage 0, the staged x, the reduction slots and the
// mbarriers; after it the other stages.  Formats without a table keep one
// block: ring, x, reduction slots, mbarriers.
constexpr int kTableAlign = 65536;
constexpr int kTablePreSlack = 4096;  // room left for the window offset of the dynamic area

template <class F, int M>
__host__ __device__ constexpr int gemv_red_bytes() { return red_slots<F, M>() * kTileRows * acc_stride(M) * 4; }

// Table formats whose pre-table part would not fit with the reduction slots
// (several activation rows) place the slots after the last stage instead.
template <class F, int M>
__host__ __device__ constexpr bool gemv_red_post() {
  return F::kSharedBytes != 0 && F::kTileBytes + kSlices * wps_for<F>(M) * (F::kKW / 2) * mpad(M) * 8 +
                                         gemv_red_bytes<F, M>() + (2 * F::stages(M) * 8 + 127) / 128 * 128 +
                                         kTablePreSlack > kTableAlign;
}

template <class F, int M>
__host__ __device__ constexpr int gemv_pre_bytes() {
  return F::kTileBytes                                             // stage 0
         + kSlices * wps_for<F>(M) * (F::kKW / 2) * mpad(M) * 8   // x pairs, per warp
         + (gemv_red_post<F, M>() ? 0 : gemv_red_bytes<F, M>())   // cross-slice reduction
         + (2 * F::stages(M) * 8 + 127) / 128 * 128;               // mbarriers (stage 1 stays 128-aligned)
}

template <class F, int M>
__host__ __device__ constexpr int gemv_smem_bytes() {
  return F::kSharedBytes == 0 ? gemv_pre_bytes<F, M>() + (F::stages(M) - 1) * F::kTileBytes
                              : kTableAlign + F::kSharedBytes + (F::stages(M) - 1) * F::kTileBytes +
                                    (gemv_red_post<F, M>() ? gemv_red_bytes<F, M>() : 0);
}

template <class F, int M>
__host__ __device__ constexpr int gemv_threads() { return 32 * kSlices * wps_for<F>(M); }

// Rows of shared row tile sg (of `rows`) that this CTA finishes.  When the
// whole tile is at most kWholeFinishItems items (rows x activation rows),
// one contributor finishes it alone: the one whose part of the row tile
// closes its run last (its plan flag), so that no CTA waits for a partial
// written at the end of another CTA's run except that one -- a contributor
// whose part opens its run stored it long before.  Larger tiles are split
// into the plan's even row slices over all contributors.  Every contributor
// of a segment decides alike (the rule depends on rows and mrows only).
constexpr int kWholeFinishItems = 256;
__device__ __forceinline__ void finish_slice(const CtaPlan& pl, int sg, int rows, int mrows, int& r0, int& nr) {
  if (rows * mrows <= kWholeFinishItems) {
    r0 = 0;
    nr = (pl.seg_flags[sg] & 2) ? rows : 0;
  } else {
    r0 = pl.seg_r0[sg];
    nr = pl.seg_nr[sg];
  }
}

// Finish one shared row tile (ROWS output rows) as described by a CtaPlan
// segment: sum rows [r0, r0 + nr) of each activation row over the S
// contributors starting at CTA cf.  A partial slot holds the empty mark (all
// ones, a pattern no fp32 add produces) until its writer stores the partial;
// the reader polls it with a bounded wait and marks it empty again.  The
// next launch writes partials only after its grid-dependency wait, i.e.
// after this launch has ended.  Up to 16 contributors one thread sums an
// item (row, m) alone; beyond that H threads sum contiguous runs of
// contributors and the H sub-sums are added in order.  The order depends
// only on the launch geometry, so results are bitwise reproducible.
// y = sum * out_scale, times the fp16 row scale when row_scales is not null.
template <int ROWS, int M, int NT>
__device__ __forceinline__ void finish_rows(const RunParams& p, int64_t stride, const CtaPlan& pl, int sg,
                                            const __half* row_scales, float out_scale, float* s_sub,
                                            int tid, int mrows = M) {
  const int64_t rt = pl.seg_rt[sg];
  const int64_t cf = pl.seg_cf[sg];
  const int S = pl.seg_S[sg];
  int r0, nr;
  finish_slice(pl, sg, ROWS, mrows, r0, nr);
  if (nr <= 0) return;  // another contributor finishes these rows
  constexpr int B = M > 8 ? 8 : 16;  // slots polled at once (registers)
  const int items = nr * mrows;
  const int H = (S <= 16 || items >= NT) ? 1 : NT / items;
  const int cpt = H == 1 ? S : (S + H - 1) / H;
  // slot of contributor cf + i: side 1 only for the first one, if its run began earlier
  const float* first_slot = p.partials + (cf * 2 + (pl.seg_flags[sg] & 1)) * stride;
  const float* base = p.partials + cf * 2 * stride;
  for (int t = tid; t < items * H; t += NT) {
    const int item = H == 1 ? t : t / H;
    const int h = H == 1 ? 0 : t - item * H;
    const int m = M == 1 ? 0 : item / nr;
    const int r = r0 + (M == 1 ? item : item - m * nr);  // M is mrows' upper bound
    const int64_t n = rt * ROWS + r;
    float sc = out_scale;
    if (row_scales != nullptr && h == 0 && n < p.N) sc *= __half2float(row_scales[n]);
    const int64_t off = m * ROWS + r;
    float sum = 0.f;
    for (int j0 = h * cpt; j0 < (h + 1) * cpt && j0 < S; j0 += B) {
      const int cnt = min(B, min((h + 1) * cpt, S) - j0);
      uint32_t bits[B];
      uint32_t pending = (1u << cnt) - 1u;
      auto slot = [&](int j) {
        const int i = j0 + j;
        return const_cast<float*>(i == 0 ? first_slot + off : base + int64_t(i) * 2 * stride + off);
      };
      unsigned long long t_start = 0;
      while (true) {
#pragma unroll
        for (int j = 0; j < B; ++j)
          if (pending & (1u << j)) bits[j] = ld_relaxed_u32(slot(j));
#pragma unroll
        for (int j = 0; j < B; ++j)
          if ((pending & (1u << j)) && bits[j] != kEmptySlot) pending &= ~(1u << j);
        if (!pending) break;
        // spin: each round is one L2 round trip; no sleep, whose granularity
        // is far coarser than the waits hidden here
        const unsigned long long now = global_timer_ns();
        if (t_start == 0) t_start = now;
        else if (now - t_start > kWaitLimitNs) {
          atomicOr(p.err, kErrTimeoutFixup);
          break;
        }
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        if (j < cnt) {
          sum += __uint_as_float(bits[j]);
          st_relaxed_u32(slot(j), kEmptySlot);
        }
      }
    }
    if (H == 1) {
      if (n < p.N) store_y(p, m * p.N + n, __fmul_rn(sum, sc));
    } else {
      s_sub[t] = sum;
      if (h == 0) s_sub[NT + item] = sc;
    }
  }
  if (H > 1) {
    __syncthreads();
    for (int item = tid; item < items; item += NT) {
      float sum = 0.f;
      for (int h = 0; h < H; ++h) sum += s_sub[item * H + h];
      const int m = item / nr;
      const int64_t n = rt * ROWS + r0 + item - m * nr;
      if (n < p.N) store_y(p, m * p.N + n, __fmul_rn(sum, s_sub[NT + item]));
    }
    __syncthreads();
  }
}

// Out-of-line copy for large M, whose main loop needs every register.
template <int ROWS, int M, int NT>
__device__ __noinline__ void finish_rows_call(const RunParams& p, int64_t stride, const CtaPlan& pl, int sg,
                                              const __half* row_scales, float out_scale, float* s_sub,
                                              int tid, int mrows) {
  finish_rows<ROWS, M, NT>(p, stride, pl, sg, row_scales, out_scale, s_sub, tid, mrows);
}

template <int ROWS, int M, int NT>
__device__ __forceinline__ void finish_segment(const RunParams& p, int64_t stride, const CtaPlan& pl, int sg,
                                               const __half* row_scales, float out_scale, float* s_sub,
                                               int tid, int mrows = M) {
  if constexpr (M > 8)
    finish_rows_call<ROWS, M, NT>(p, stride, pl, sg, row_scales, out_scale, s_sub, tid, mrows);
  else
    finish_rows<ROWS, M, NT>(p, stride, pl, sg, row_scales, out_scale, s_sub, tid, mrows);
}

// Finish the CTA's shared row tiles (the two plan segments) that it has
// rows of.  When it has two and neither needs the split-contributor sums
// (S <= 16), half the threads take each, so that the two waits for other
// CTAs' partials overlap instead of adding up.
template <int ROWS, int M, int NT>
__device__ __forceinline__ void finish_all(const RunParams& p, int64_t stride, const CtaPlan& pl,
                                           const __half* row_scales, float out_scale, float* s_sub, int tid,
                                           int mrows = M) {
  int r0, nr0, nr1;
  finish_slice(pl, 0, ROWS, mrows, r0, nr0);
  finish_slice(pl, 1, ROWS, mrows, r0, nr1);
  const bool s0 = pl.seg_rt[0] >= 0 && nr0 > 0, s1 = pl.seg_rt[1] >= 0 && nr1 > 0;
  if (s0 && s1 && pl.seg_S[0] <= 16 && pl.seg_S[1] <= 16) {
    const int sg = tid < NT / 2 ? 0 : 1;
    finish_segment<ROWS, M, NT / 2>(p, stride, pl, sg, row_scales, out_scale, s_sub, tid - sg * (NT / 2), mrows);
    return;
  }
  if (s0) finish_segment<ROWS, M, NT>(p, stride, pl, 0, row_scales, out_scale, s_sub, tid, mrows);
  if (s1) finish_segment<ROWS, M, NT>(p, stride, pl, 1, row_scales, out_scale, s_sub, tid, mrows);
}

// y[m][n] = SiLU(g) * u for a GLU handle (output width p.N / 2): SiLU(g) =
// g / (1 + e^-g) in fp32 (expf, IEEE division), then one fp32 product.
__device__ __forceinline__ void glu_store(const RunParams& p, int m, int64_t n, float g, float u) {
  const int64_t nout = p.N / 2;
  if (n < nout) p.y[m * nout + n] = __fmul_rn(g / (1.0f + expf(-g)), u);
}

// Finish a shared row tile of a GLU handle (plan segment sg, whose row slice
// counts gate/up row pairs, 0..63): for each pair and activation row, the
// gate and up sums over the S contributors in order, then SiLU(gate) * up.
// The gate and up slots of up to 8 contributors are polled at once (one L2
// round trip when they are there), each with a bounded wait; after a wait
// has given up, the rest of the thread's slots count as 0 and are not waited
// for, so a run whose partials never come ends after one time limit.
template <int M, int NT>
__device__ __noinline__ void finish_rows_glu(const RunParams& p, const CtaPlan& pl, int sg, float out_scale,
                                             int tid, int mrows = M) {
  const int64_t rt = pl.seg_rt[sg];
  const int64_t cf = pl.seg_cf[sg];
  const int S = pl.seg_S[sg];
  int r0, nr;
  finish_slice(pl, sg, kTileRows / 2, mrows, r0, nr);
  if (nr <= 0) return;
  constexpr int B = 8;  // contributors polled at once
  float* first_slot = p.partials + (cf * 2 + (pl.seg_flags[sg] & 1)) * kPartialStride;
  float* base = p.partials + cf * 2 * kPartialStride;
  bool gave_up = false;
  for (int t = tid; t < nr * mrows; t += NT) {
    const int m = t / nr;
    const int r = r0 + (t - m * nr);
    float g = 0.f, u = 0.f;
    for (int i0 = 0; i0 < S; i0 += B) {
      const int cnt = min(B, S - i0);
      // slot word 2j: gate row r of contributor i0 + j, 2j + 1: its up row
      auto slot = [&](int w) {
        const int i = i0 + (w >> 1);
        return (i == 0 ? first_slot : base + int64_t(i) * 2 * kPartialStride) + m * kTileRows + r +
               ((w & 1) ? kTileRows / 2 : 0);
      };
      uint32_t bits[2 * B];
      uint32_t pending = gave_up ? 0u : (1u << (2 * cnt)) - 1u;
#pragma unroll
      for (int w = 0; w < 2 * B; ++w) bits[w] = 0u;  // +0.0 for a slot given up on
      unsigned long long t_start = 0;
      while (pending) {
#pragma unroll
        for (int w = 0; w < 2 * B; ++w)
          if (pending & (1u << w)) bits[w] = ld_relaxed_u32(slot(w));
#pragma unroll
        for (int w = 0; w < 2 * B; ++w)
          if ((pending & (1u << w)) && bits[w] != kEmptySlot) pending &= ~(1u << w);
        if (!pending) break;
        const unsigned long long now = global_timer_ns();
        if (t_start == 0) {
          t_start = now;
        } else if (now - t_start > kWaitLimitNs) {
          atomicOr(p.err, kErrTimeoutFixup);
          gave_up = true;
#pragma unroll
          for (int w = 0; w < 2 * B; ++w)
            if (pending & (1u << w)) bits[w] = 0u;
          break;
        }
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        if (j < cnt) {
          g += __uint_as_float(bits[2 * j]);
          u += __uint_as_float(bits[2 * j + 1]);
          st_relaxed_u32(slot(2 * j), kEmptySlot);
          st_relaxed_u32(slot(2 * j + 1), kEmptySlot);
        }
      }
    }
    glu_store(p, m, rt * (kTileRows / 2) + r, __fmul_rn(g, out_scale), __fmul_rn(u, out_scale));
  }
}

// CTA c's share of a stream of T work units, in the split mode U of the
// format (a compile-time constant, so a kernel carries one formula).
// U = 0: [c T / G, (c + 1) T / G) (the larger runs spread evenly over the
// grid).  U = 1 or 2: chunks of U consecutive units (the last chunk may be
// short); with n = ceil(T / U) chunks, q = n / G and r = n % G, CTA c runs
// chunks [c q + min(c, r), (c + 1) q + min(c + 1, r)) -- the first r CTAs
// take one chunk more.  CTAs are placed in index order as SMs free up, so
// those with the extra chunk start first and the last-placed ones carry
// less.  32-bit divisions when the sizes fit.
template <int U>
__device__ __forceinline__ int64_t stream_split(int64_t c, int64_t T, int64_t G) {
  if constexpr (U == 0) {
    const int64_t prod = c * T;
    if (prod < (int64_t(1) << 31) && G < (int64_t(1) << 31))
      return static_cast<int64_t>(static_cast<uint32_t>(prod) / static_cast<uint32_t>(G));
    return prod / G;
  }
  const int64_t n = U == 1 ? T : (T + U - 1) / U;
  int64_t q;
  if (n < (int64_t(1) << 31) && G < (int64_t(1) << 31))
    q = static_cast<int64_t>(static_cast<uint32_t>(n) / static_cast<uint32_t>(G));
  else
    q = n / G;
  const int64_t r = n - q * G;
  const int64_t t = (c * q + (c < r ? c : r)) * U;
  return t < T ? t : T;
}

__device__ __forceinline__ int64_t div_fast(int64_t a, int64_t b) {
  if (a < (int64_t(1) << 31) && b < (int64_t(1) << 31))
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

// Start copying this CTA's plan into shared memory (four 16-byte pieces,
// asynchronous); wait_plan() must run before it is read.
__device__ __forceinline__ void fetch_plan(CtaPlan* s_plan, const CtaPlan* plan, int64_t c, int tid) {
  if (tid < 4) {
    const uint32_t dst = smem_u32(reinterpret_cast<uint8_t*>(s_plan) + 16 * tid);
    const void* src = reinterpret_cast<const uint8_t*>(plan + c) + 16 * tid;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n\tcp.async.commit_group;" ::"r"(dst), "l"(src)
                 : "memory");
  }
}

__device__ __forceinline__ void wait_plan() {
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
}

// The codebook of row tile rt (table formats): aux holds one codebook, or
// for a stacked handle one copy per row tile.
template <class F>
__device__ __forceinline__ const uint16_t* table_of(const RunParams& p, int64_t rt) {
  return static_cast<const uint16_t*>(p.aux) + (p.seg_of_rt != nullptr ? rt * F::kCbEntries : 0);
}

// GLU handles of the one-codebook table formats (F::kGluTables): the gate
// and up projections have a codebook each.  Their tables share the 64 KB
// region: a lane-replicated entry row is 256 bytes of which lanes use the
// first 128 (lane * 4), so the up table sits in the second 128 (a key with
// bit 7 set) and every lookup stays one conflict-free LDS.  The up rows of a
// tile (64..127) are those of lanes 16..31, or the odd m-tiles of the
// tensor-core kernel.
template <class F, class = void>
struct GluTables {
  static constexpr bool value = false;
};
template <class F>
struct GluTables<F, decltype(void(F::kGluTables))> {
  static constexpr bool value = F::kGluTables;
};
constexpr int kGluUpTable = 128;  // byte offset of the up table in each entry row

// Stacked table handles: the segment of the table built in shared memory
// (seg[0]), and the segment and codebook of the row tile after it (seg[1],
// cb), staged with cp.async ahead of time.  A global load at a row-tile
// change would stall the CTA for a loaded-memory round trip (over a
// microsecond while the weight stream saturates HBM), and the launch lasts
// as long as its latest CTA.  Codebooks of up to 256 entries are staged;
// larger ones (the per-row codebooks of a row tile, 8 KB) are read from
// global memory by the rebuild.
template <class F>
constexpr bool kStagedCb = F::kCbEntries > 0 && F::kCbEntries <= 256;

// The format's stream-K split mode (F::kSplitMode; 0 when absent).
template <class F, class = void>
struct SplitModeOf {
  static constexpr int value = 0;
};
template <class F>
struct SplitModeOf<F, decltype(void(F::kSplitMode))> {
  static constexpr int value = F::kSplitMode;
};

template <class F>
struct alignas(16) NextTable {
  int seg[2];
  int pad[2];
  uint16_t cb[kStagedCb<F> ? F::kCbEntries : 8];
};

// Stage the segment and codebook of row tile rt + 1 (rt itself if it is the
// last), and with first also rt's segment.  Threads 0 .. E/8 - 1 copy the
// codebook in 16-byte pieces, thread E/8 the segment numbers; every thread
// runs cp.async.wait_all and a barrier (advance_table) before any read.
template <class F>
__device__ __forceinline__ void prefetch_next_table(NextTable<F>* s, const RunParams& p, int64_t rt,
                                                    int64_t nRT, bool first, int tid) {
  constexpr int kPieces = kStagedCb<F> ? F::kCbEntries * 2 / 16 : 0;
  static_assert(kPieces * 16 == (kStagedCb<F> ? F::kCbEntries * 2 : 0), "codebook in 16-byte pieces");
  const int64_t rn = rt + 1 < nRT ? rt + 1 : rt;
  if (tid < kPieces) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n\tcp.async.commit_group;"
                 ::"r"(smem_u32(s->cb + 8 * tid)), "l"(table_of<F>(p, rn) + 8 * tid) : "memory");
  } else if (tid == kPieces) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&s->seg[1])), "l"(p.seg_of_rt + rn)
                 : "memory");
    if (first)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&s->seg[0])), "l"(p.seg_of_rt + rt)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
}

// At a row-tile change of a stacked handle (every thread; rt = the new row
// tile): rebuild the table from the staged codebook if the segment changes,
// then stage the next one.  Starts with a barrier (every warp is done with
// the old table) and leaves the staged data consumed.
template <class F, int NT, class Rebuild>
__device__ __forceinline__ void advance_table(NextTable<F>* s, const RunParams& p, int64_t rt, int tid,
                                              Rebuild&& rebuild) {
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int cur = s->seg[0], nxt = s->seg[1];
  if (nxt != cur) rebuild(kStagedCb<F> ? s->cb : table_of<F>(p, rt));
  __syncthreads();  // every thread has read s
  if (tid == 0) s->seg[0] = nxt;
  prefetch_next_table<F>(s, p, rt, div_fast(p.T, p.nKT), false, tid);
}

// Table rebuild at a segment change of a stacked handle: rare, so out of
// line, keeping the main loop's register allocation as without stacking.
template <class F, int NT>
__device__ __noinline__ void rebuild_table(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
  F::template init_shared<NT>(lut, cb, warp, lane);
}

// GLU: the handle's rows are a gate and an up projection interleaved in
// 64-row halves of every row tile (gate rows 64t .. 64t+63 are tile t's rows
// 0..63, the up rows the same, rows 64..127), and y[m][64t + r] =
// SiLU(gate) * up (glu_store, finish_rows_glu); p.N counts both halves.
template <class F, int M, bool GLU = false>
__global__ void __launch_bounds__(gemv_threads<F, M>(), F::kCtasPerSm) wstream_kernel(const RunParams p) {
  constexpr int NS = F::stages(M);
  constexpr int TB = F::kTileBytes;
  constexpr int MP = mpad(M);
  constexpr int WPS = wps_for<F>(M);
  constexpr int NT = gemv_threads<F, M>();
  constexpr bool PAR = tile_parity<F, M>();
  constexpr int RPW = PAR ? kRowsPerLane : kRowsPerLane / WPS;
  constexpr int XS_FLOATS = (F::kKW / 2) * MP * 2;  // per warp
  constexpr int RS = acc_stride(M);

  extern __shared__ __align__(128) uint8_t smem[];
  // stage s at ring0 (s = 0) or ringN + (s - 1) TB
  uint8_t* ring0 = smem;
  float* xs_all = reinterpret_cast<float*>(smem + TB);
  float* red = xs_all + kSlices * WPS * XS_FLOATS;  // or after the last stage (gemv_red_post)
  uint64_t* full = reinterpret_cast<uint64_t*>(gemv_red_post<F, M>() ? red : red + red_slots<F, M>() * kTileRows * RS);
  uint8_t* ringN;
  uint8_t* fsh;
  __shared__ volatile int s_abort;
  __shared__ NextTable<F> s_next;
  __shared__ __align__(16) CtaPlan s_plan;

  if (static_cast<int>(blockIdx.x) == p.skip_cta) return;  // test hook (QGEMV_FAULT_SKIP_CTA)
  if constexpr (F::kSharedBytes == 0) {
    ringN = smem + gemv_pre_bytes<F, M>();
    fsh = smem;  // unused
  } else {
    static_assert(F::kSharedBytes == kTableAlign, "one 64 KB table");
    static_assert(gemv_pre_bytes<F, M>() + kTablePreSlack <= kTableAlign, "pre-table layout");
    const uint32_t base = smem_u32(smem);
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t R0 = (base + (kTableAlign - 1)) & ~uint32_t(kTableAlign - 1);
    if (R0 - base < uint32_t(gemv_pre_bytes<F, M>()) ||
        R0 + kTableAlign + (NS - 1) * TB + (gemv_red_post<F, M>() ? gemv_red_bytes<F, M>() : 0) > base + dyn) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
      return;
    }
    fsh = smem + (R0 - base);
    ringN = fsh + kTableAlign;
    if constexpr (gemv_red_post<F, M>()) red = reinterpret_cast<float*>(ringN + (NS - 1) * TB);
  }
  uint64_t* empty = full + NS;
  auto stage_ptr = [&](int st) { return st == 0 ? ring0 : ringN + (st - 1) * TB; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slice = warp % kSlices;
  const int half = warp / kSlices;  // 0 when WPS == 1
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t t0 = stream_split<SplitModeOf<F>::value>(c, p.T, G);
  const int64_t t1 = stream_split<SplitModeOf<F>::value>(c + 1, p.T, G);

  const int64_t rt_first = div_fast(t0, p.nKT);

  // The elected thread initializes the barriers and at once starts filling
  // the ring NS - 1 tiles ahead of the math (with tile parity: the first
  // tile of each half), so the first tiles are in flight while the CTA
  // builds the format's tables.  With tile parity the stages after those
  // two are filled from the main loop: every tile issued before the grid
  // dependency resolves queues in HBM ahead of the first copies of the CTAs
  // that start last (those on the SMs the previous launch left last), and
  // the launch lasts as long as its latest CTA.
  constexpr int kPre = PAR ? 2 : NS - 1;
  const int64_t ntiles = t1 - t0;
  const bool elected = (tid == 0);
  uint64_t pol = 0;
  int64_t n_issued = 0;  // meaningful on the elected thread
  if (elected) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAR ? kSlices : kSlices * WPS);  // with tile parity one half uses a stage
    }
    s_abort = 0;
    fence_mbarrier_init();
    pol = l2_policy_evict_first();
    for (; n_issued < kPre && n_issued < ntiles; ++n_issued) {
      mbar_arrive_expect_tx(&full[n_issued], TB);
      bulk_g2s(stage_ptr(static_cast<int>(n_issued)), p.tiles + (t0 + n_issued) * TB, TB, &full[n_issued], pol);
    }
  }
  fetch_plan(&s_plan, p.plan, c, tid);
  // Table formats keep one codebook copy per row tile in aux (stacked
  // handles hold several codebooks); the first row tile's needs no lookup.
  // Stacked handles stage the next row tile's segment and codebook.
  if constexpr (F::kCbEntries > 0) {
    if (p.seg_of_rt != nullptr && ntiles > 0)
      prefetch_next_table<F>(&s_next, p, rt_first, div_fast(p.T, p.nKT), true, tid);
  }
  F::template init_shared<NT>(fsh, table_of<F>(p, rt_first), warp, lane);
  if constexpr (GLU && GluTables<F>::value)
    F::template init_shared<NT>(fsh + kGluUpTable, table_of<F>(p, rt_first) + F::kCbEntries, warp, lane);
  __syncthreads();
  // the table of the lane's rows (GLU: lanes 16..31 hold the up rows)
  uint8_t* const lane_table = fsh + (GLU && GluTables<F>::value && lane >= 16 ? kGluUpTable : 0);

  float* xs = xs_all + warp * XS_FLOATS;
  RowAcc<M, RPW> acc;
  // reduction slot and row half of this warp (tile parity: all rows, a slot per half)
  const int rslot = PAR ? half * kSlices + slice : slice;
  const int rhalf = PAR ? 0 : half;
  acc.init(red, rslot, rhalf, lane);

  // Programmatic dependent launch: the prologue above (barriers, tables, the
  // first weight copies) touches nothing a previous kernel in the stream
  // writes, so it may overlap that kernel's tail.  Everything below reads x
  // or writes global memory, so it waits for the previous grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Position of tile t0 in the stream, advanced incrementally below.
  int64_t rt = rt_first;
  const int nKT = static_cast<int>(p.nKT);
  int kt = static_cast<int>(t0 - rt * p.nKT);
  const int nt = static_cast<int>(ntiles);
  const bool stacked = F::kCbEntries > 0 && p.seg_of_rt != nullptr;
  // k-tile index k (< nKT + 2) reduced into [0, nKT)
  auto wrap_kt = [nKT](int k) {
    if (k >= nKT) k -= nKT;
    if (k >= nKT) k -= nKT;
    return k;
  };
  // x of the next tile this warp computes (tile parity: every second tile)
  constexpr int TSTEP = PAR ? 2 : 1;
  const int first = PAR ? half : 0;
  typename F::XRegs xr;
  if (first < nt) F::template load_x<M>(xr, p, wrap_kt(kt + first), slice, lane);
  typename F::XScale xscale;  // per-lane activation scaling, the same for every tile
  F::x_scales(xscale, lane);

  // A new row tile of a stacked handle may use another codebook: rebuild
  // the table once every warp is done with the old one.
  auto next_table = [&]() {
    if constexpr (F::kCbEntries > 0)
      advance_table<F, NT>(&s_next, p, rt, tid,
                           [&](const uint16_t* cb) { rebuild_table<F, NT>(fsh, cb, warp, lane); });
  };

  // The warp's part of tile j (stage st, fill parity par): stage its x,
  // prefetch the x of the warp's next tile (k-tile kt_pref), wait for the
  // codes, compute.
  auto compute_tile = [&](int j, int st, uint32_t par, int kt_pref, bool abort) {
    float xsum[F::kSumGroups][M];
    __syncwarp();
    F::template stage_x<M>(xs, xsum, xr, xscale, lane);
    __syncwarp();
    if (j + TSTEP < nt) F::template load_x<M>(xr, p, kt_pref, slice, lane);
    const bool ok = !abort && mbar_wait_bounded(&full[st], par);
    if (!ok) {
      if (!abort && lane == 0) atomicOr(p.err, kErrTimeoutFull);
      s_abort = 1;
    } else {
      F::template tile_math<M, RPW>(stage_ptr(st), xs, xsum, acc, lane_table, slice, rhalf, lane, &empty[st]);
    }
  };

  // Row-tile epilogue: add the slices' partials in slice order; the owner of
  // a whole row tile writes y, a contributor to a shared one its partials.
  auto row_epilogue = [&](int64_t cur_rt) {
    acc.flush(red, rslot, rhalf, lane);
    named_bar_sync(1, NT);
    const bool owner = (cur_rt * p.nKT >= t0) && ((cur_rt + 1) * p.nKT <= t1);
    const int side = (cur_rt * p.nKT <= t0) ? 0 : 1;
    float* my_part = p.partials + (c * 2 + side) * kPartialStride;
    if constexpr (GLU) {
      if (owner) {  // a gate row and its up row per item
        for (int o = tid; o < (kTileRows / 2) * M; o += NT) {
          const int r = o % (kTileRows / 2);
          const int m = o / (kTileRows / 2);
          float g = 0.f, u = 0.f;
#pragma unroll
          for (int w = 0; w < red_slots<F, M>(); ++w) {
            g += red[(w * kTileRows + r) * RS + m];
            u += red[(w * kTileRows + kTileRows / 2 + r) * RS + m];
          }
          glu_store(p, m, cur_rt * (kTileRows / 2) + r, __fmul_rn(g, F::kOutScale), __fmul_rn(u, F::kOutScale));
        }
      } else {
        for (int o = tid; o < kTileRows * M; o += NT) {
          const int r = o % kTileRows;
          const int m = o / kTileRows;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < red_slots<F, M>(); ++w) v += red[(w * kTileRows + r) * RS + m];
          st_relaxed_f32(my_part + m * kTileRows + r, v);
        }
      }
    } else {
    for (int o = tid; o < kTileRows * M; o += NT) {
      const int r = o % kTileRows;
      const int m = o / kTileRows;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < red_slots<F, M>(); ++w) v += red[(w * kTileRows + r) * RS + m];
      if (owner) {
        const int64_t n = cur_rt * kTileRows + r;
        if (n < p.N) store_y(p, m * p.N + n, __fmul_rn(v, F::kOutScale));
      } else {
        st_relaxed_f32(my_part + m * kTileRows + r, v);
      }
    }
    }
    named_bar_sync(1, NT);
    acc.reset();
  };

  if constexpr (PAR) {
    // Tile parity: tile j lives in stage j % NS and is computed by half
    // j % 2, so (NS even) each half owns every second stage.  Each half runs
    // its own pipeline over its own tiles: at its tile j its first thread
    // fills the stage of its tile j - 2 (released one tile ago; for j < 2 a
    // stage not used yet) with tile j + NS - 2.  The prologue issued tiles
    // 0 and 1.  Both halves walk the run row tile by row tile and meet at
    // each row-tile end.
    static_assert(NS % 2 == 0 && NS >= 4, "tile parity: each half owns every second stage");
    static_assert(kPre == 2, "the main loop fills stages 2 .. NS - 1 first");
    const bool leader = (lane == 0) && (slice == 0);
    const uint64_t lpol = leader ? l2_policy_evict_first() : 0;
    int u_last = -1;  // leader: last tile of its parity issued (by the prologue or by itself)
    for (int u = half; u < kPre && u < nt; u += 2) u_last = u;
    int i = 0;  // first tile of the current row tile segment
    while (i < nt) {
      if (stacked && i > 0) next_table();
      const int iend = i + min(nt - i, nKT - kt);
#pragma unroll 1
      for (int j = i + ((i ^ half) & 1); j < iend; j += 2) {
        bool abort = s_abort != 0;
        const int u = j + NS - 2;
        // tiles below kPre came from the prologue: never fill a stage twice
        if (leader && !abort && u >= kPre && u < nt) {
          const int su = u % NS;
          if (u >= NS && !mbar_wait_bounded(&empty[su], static_cast<uint32_t>(((u - NS) / NS) & 1))) {
            atomicOr(p.err, kErrTimeoutEmpty);
            s_abort = 1;
            abort = true;
          } else {
            mbar_arrive_expect_tx(&full[su], TB);
            bulk_g2s(stage_ptr(su), p.tiles + (t0 + u) * TB, TB, &full[su], lpol);
            u_last = u;
          }
        }
        compute_tile(j, j % NS, static_cast<uint32_t>((j / NS) & 1), wrap_kt(kt + (j - i) + 2), abort);
      }
      row_epilogue(rt);
      i = iend;
      kt = 0;
      ++rt;
    }
    // Never leave while a copy issued by this half may still be landing
    // (only possible after an aborted run): wait for the last fill of each
    // of the half's stages.
    if (leader && s_abort != 0) {
      for (int u = u_last; u >= 0 && u > u_last - NS; u -= 2)
        mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
    }
  } else {
    int s = 0;           // stage of the tile being computed
    uint32_t ph = 0;     // its fill parity
    int su = static_cast<int>(n_issued % NS);            // next stage to fill
    uint32_t phu = static_cast<uint32_t>((n_issued / NS) & 1);
    for (int i = 0; i < nt; ++i) {
      if (stacked && kt == 0 && i > 0) next_table();
      bool abort = s_abort != 0;

      // Refill: tile u = i + NS - 1 goes to the stage released by tile
      // u - NS = i - 1, whose codes every warp loaded one iteration ago.
      if (elected && !abort && n_issued < ntiles) {
        if (n_issued >= NS && !mbar_wait_bounded(&empty[su], phu ^ 1)) {
          atomicOr(p.err, kErrTimeoutEmpty);
          s_abort = 1;
          abort = true;
        } else {
          mbar_arrive_expect_tx(&full[su], TB);
          bulk_g2s(stage_ptr(su), p.tiles + (t0 + n_issued) * TB, TB, &full[su], pol);
          ++n_issued;
          if (++su == NS) { su = 0; phu ^= 1; }
        }
      }

      const int kt_next = (kt + 1 == nKT) ? 0 : kt + 1;
      compute_tile(i, s, ph, kt_next, abort);
      if (++s == NS) { s = 0; ph ^= 1; }

      const bool row_end = (kt_next == 0) || (i + 1 == nt);
      const int64_t cur_rt = rt;
      kt = kt_next;
      if (kt_next == 0) ++rt;
      if (row_end) row_epilogue(cur_rt);
    }

    // Never leave while a copy issued by this CTA may still be landing (only
    // possible after an aborted run; normally every issued tile was consumed).
    if (elected && s_abort != 0) {
      for (int64_t u = (n_issued > NS ? n_issued - NS : 0); u < n_issued; ++u)
        mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
    }
  }

  // Row tiles shared with other CTAs (at most the first and the last of the
  // run): every contributor finishes a slice of their rows from the polled
  // partial slots.  The cross-slice buffer (at least 2 * NT floats) is free
  // now and serves as the finishing scratch.
  static_assert(kSlices * kTileRows * RS >= 2 * NT, "finishing scratch");
  float* s_sub = red;
  wait_plan();
  if constexpr (GLU) {
    for (int sg = 0; sg < 2; ++sg)
      if (s_plan.seg_rt[sg] >= 0) finish_rows_glu<M, NT>(p, s_plan, sg, F::kOutScale, tid);
  } else {
    finish_all<kTileRows, M, NT>(p, kPartialStride, s_plan, nullptr, F::kOutScale, s_sub, tid);
  }
}

// ------------------------------------------------- activation staging ----
//
// Helpers for formats whose slice is 32 (one k per lane) or 64 (two k per
// lane) wide.  x is fp16 [M][K]; k >= K reads as 0.  stage_x converts to
// fp32, multiplies by the format's per-position power of two (exact) and
// stores pairs (x'[2q][m], x'[2q+1][m]) at xs[(q * MP + m) * 2 + {0,1}];
// xsum[m] is the plain sum of the slice's x[m][k] (all lanes get it).

template <int LPL>
struct XRegsT {
  unsigned short v[kMaxM][LPL];
};

template <int KW, int M, int LPL>
__device__ __forceinline__ void load_x_slice(XRegsT<LPL>& xr, const RunParams& p, int kt,
                                             int slice, int lane) {
  const int64_t kbase = static_cast<int64_t>(kt) * (KW * kSlices) + slice * KW + lane * LPL;
  const unsigned short* xb = reinterpret_cast<const unsigned short*>(p.x);
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const int64_t k = kbase + i;
      xr.v[m][i] = (k < p.K) ? __ldg(xb + m * p.K + k) : static_cast<unsigned short>(0);
    }
}

template <int M, int LPL, int SUBS>
__device__ __forceinline__ void stage_x_slice(float* xs, float (&xsum)[SUBS][M],
                                              const XRegsT<LPL>& xr, int lane,
                                              const float (&scale)[LPL]) {
  constexpr int MP = mpad(M);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const int kk = lane * LPL + i;  // position inside the slice
      const float v = h2f(xr.v[m][i]);
      s += v;
      xs[((kk >> 1) * MP + m) * 2 + (kk & 1)] = v * scale[i];
    }
    // sums over each group of 32 / SUBS consecutive lanes, then gathered so
    // every lane holds all SUBS group sums
#pragma unroll
    for (int off = 16 / SUBS; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
    for (int g = 0; g < SUBS; ++g) xsum[g][m] = __shfl_sync(0xffffffffu, s, g * (32 / SUBS));
  }
  if (MP > M) {  // keep padding lanes of the vector loads finite
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const int kk = lane * LPL + i;
#pragma unroll
      for (int m = M; m < MP; ++m) xs[((kk >> 1) * MP + m) * 2 + (kk & 1)] = 0.f;
    }
  }
}

// Load the x pairs of pair index q for all m: out[m] = (x'[2q][m], x'[2q+1][m]).
template <int M>
__device__ __forceinline__ void load_xpairs(const float* xs, int q, float2 (&out)[M]) {
  constexpr int MP = mpad(M);
  const float* b = xs + q * MP * 2;
  if constexpr (M == 1) {
    out[0] = *reinterpret_cast<const float2*>(b);
  } else {
#pragma unroll
    for (int m = 0; m < MP; m += 2) {
      const float4 v = lds128f(b + m * 2);
      if (m < M) out[m] = make_float2(v.x, v.y);
      if (m + 1 < M) out[m + 1] = make_float2(v.z, v.w);
    }
  }
}

// Load NP consecutive x pairs q0 .. q0+NP-1 (q0 even): 128-bit loads of two
// pairs at a time when M == 1.
template <int M, int NP>
__device__ __forceinline__ void load_xpair_run(const float* xs, int q0, float2 (&out)[NP][M]) {
  if constexpr (M == 1 && NP % 2 == 0) {
#pragma unroll
    for (int u = 0; u < NP; u += 2) {
      const float4 v = lds128f(xs + (q0 + u) * 2);
      out[u][0] = make_float2(v.x, v.y);
      out[u + 1][0] = make_float2(v.z, v.w);
    }
  } else {
#pragma unroll
    for (int u = 0; u < NP; ++u) load_xpairs<M>(xs, q0 + u, out[u]);
  }
}

__device__ __forceinline__ void release_stage(uint64_t* empty_bar, int lane) {
  __syncwarp();
  // lane 0 arrives (a predicated instruction, no divergent branch)
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %1, 0;\n\t"
      "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(empty_bar)),
      "r"(lane)
      : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

}  // namespace qgemv

// mma_kernel.cuh -- the tensor-core GEMV with register-level decode, for
// every M = 1..16.
//
//   y[m][n] = sum_k x[m][k] * w[n][k]
//
// is computed as D = W * X^T with mma.m16n8k16 (f16 x f16 -> f32): the
// weights are the 16 x 16 A operand (16 weight rows), the activations the
// 16 x 8 B operand (8 activation rows; two B operands for M > 8), so an
// activation block is padded to 8 rows, not 16.
//
//   * Same prepared tiles, TMA ring, stream-K split, CTA plans and polled
//     split-K fix-up as wstream_kernel.
//   * Two warps per group of F::mma_spw(NB) k-slices: warp (group g, half h)
//     covers slices g * spw .. of every tile, one after the other, for
//     row groups j = 2h, 2h + 1 (rows 4l + j, l = 0..31), as four 16-row
//     m-tiles (j = 2h + mt/2, l = 16 (mt & 1) + 0..15).  Formats without a
//     table use two slices per warp and run two CTAs of eight warps per SM,
//     whose phases differ; the table formats sixteen warps, one CTA per SM.
//   * Each thread reads the codes of its two fragment rows straight from the
//     stage (a few 32/64-bit loads per row, conflict-free) and decodes them
//     in registers into the A fragments -- no decoded copy of the weights is
//     stored anywhere.  Inside a k16 step the fragment's k order is a
//     permutation of the slice's k, chosen per format so that the decode is
//     cheapest; the B fragments (activations, read from global memory a tile
//     ahead) use the same permutation, so the products are unchanged.
//   * Formats with a block scale (Q4_0: 32 k, PQ2_0: 128 k) accumulate the
//     codes' products of a block (exact fp16 integers) and add d * block
//     into the fp32 accumulator; the D fragment's rows are the thread's own
//     weight rows, so the scales need no exchange.
//   * At the end of a row tile the eight slices' results are added in a
//     fixed tree order through shared memory, then stored to y or to the
//     stream-K partial slots.
//
//   * Additive formats (AQLM 2x8) make one A fragment per codebook and one
//     MMA each into the same accumulator; a per-row output scale is applied
//     when the row's sum is stored.
//
// Format hooks (members of the format struct): mma_stages(NB),
// mma_prefetch_x(NB), kMmaSharedBytes, kMmaBlockSteps (0: no scale), kMmaXWords,
// kMmaRowWords (code words per fragment row and slice), kMmaCodebooks,
// kMmaRowScales (and mma_row_scales), mma_init_shared, mma_lut_key (table
// formats), mma_load_row, mma_frag, mma_load_x, mma_bfrag and, with a block
// scale, MmaScales, mma_scales and mma_scale.
#pragma once

#include "gemv_kernel.cuh"

namespace qgemv {

constexpr int kMmaTiles = 4;  // 16-row m-tiles per warp

// Formats that, with two activation blocks, load each m-tile's code words
// just before its MMAs (F::kMmaLateCodes) instead of all four m-tiles' at
// the start of a slice: only one m-tile's codes are live, at the price of
// releasing the stage after the last m-tile.  Measured: no slower for AQLM
// (whose four code words per row would otherwise spill), 7% slower for CBK4.
// Formats whose activations are INT8 codes with a per-group scale
// (F::kMmaXCodes: the PQ2_0 integer path on prepared activations): the
// loader reads the codes and the D columns' scales (F::mma_load_x_q), and a
// block's sum is multiplied by its column's scale (F::mma_col_scale) before
// the row's block scale.
template <class F, class = void>
struct MmaXCodes {
  static constexpr bool value = false;
};
template <class F>
struct MmaXCodes<F, decltype(void(F::kMmaXCodes))> {
  static constexpr bool value = F::kMmaXCodes;
};

// Formats whose tensor-core kernel has the GLU form (F::kMmaGlu).
template <class F, class = void>
struct MmaGluOf {
  static constexpr bool value = false;
};
template <class F>
struct MmaGluOf<F, decltype(void(F::kMmaGlu))> {
  static constexpr bool value = F::kMmaGlu;
};

template <class F, class = void>
struct MmaLateCodes {
  static constexpr bool value = false;
};
template <class F>
struct MmaLateCodes<F, decltype(void(F::kMmaLateCodes))> {
  static constexpr bool value = F::kMmaLateCodes;
};
// Geometry.  Default: two warps per group of F::mma_spw(NB) k-slices (one
// slice per warp: 16 warps, one CTA per SM; two slices per warp: 8 warps, two
// CTAs per SM, F::mma_ctas(NB)).  Tile parity (PAR; one-CTA-per-SM formats):
// 16 warps in two halves that take alternate tiles, each half eight warps of
// two slices each, with four stages (two per half).
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_spw_of() { return PAR ? 2 : F::mma_spw(NB); }
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_stages_of() { return PAR ? 4 : F::mma_stages(NB); }
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_warps() { return PAR ? 16 : 2 * kSlices / F::mma_spw(NB); }
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_threads() { return 32 * mma_warps<F, NB, PAR>(); }

// tree reduction buffer: [4 slots][2 halves][4 m-tiles][NB][32 lanes] float4
template <int NB>
__host__ __device__ constexpr int mma_red_bytes() { return 4 * 2 * kMmaTiles * NB * 32 * 16; }

// Shared memory.  Formats without a table: the stages, the reduction
// buffer and the mbarriers, in that order.  Table formats (CBK4, CBK8): the
// 64 KB table starts on a 64 KB boundary of the shared window, so that one
// PRMT of the index byte with (table >> 16, lane * 4) is the whole address
// of an entry (no add per lookup).  Before the table ("pre", at most 64 KB
// less the window offset of the dynamic area): stage 0, the mbarriers and,
// for one activation block, the reduction buffer; after it the other stages
// and, for two blocks, the reduction buffer.
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_bar_bytes() { return 2 * mma_stages_of<F, NB, PAR>() * 8; }
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_pre_bytes() {
  return F::kTileBytes + mma_bar_bytes<F, NB, PAR>() + (NB == 1 ? mma_red_bytes<NB>() : 0);
}
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_post_bytes() {
  return (mma_stages_of<F, NB, PAR>() - 1) * F::kTileBytes + (NB == 1 ? 0 : mma_red_bytes<NB>());
}
template <class F, int NB, bool PAR = false>
__host__ __device__ constexpr int mma_smem_bytes() {
  return F::kMmaSharedBytes == 0
             ? mma_stages_of<F, NB, PAR>() * F::kTileBytes + mma_red_bytes<NB>() + mma_bar_bytes<F, NB, PAR>()
             : kTableAlign + F::kMmaSharedBytes + mma_post_bytes<F, NB, PAR>();
}

// Address of table entry (byte bsel of w) for the lane: key = (table >> 16)
// in byte 2, lane * 4 in byte 0; the index byte goes to byte 1.
__device__ __forceinline__ uint32_t lut_addr(uint32_t w, uint32_t key, int bsel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(key), "r"(w), "r"(0x3200u | ((4u + bsel) << 4)));
  return r;
}

__device__ __forceinline__ uint32_t lds32_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A * B (zero accumulator in)
__device__ __forceinline__ void mma_16816_c0(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// (a & mask) | 0x64006400: the two 16-bit fields as fp16 1024 + field
__device__ __forceinline__ uint32_t field_pair(uint32_t a, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(a), "r"(mask), "r"(0x64006400u));
  return r;
}

// fp16x2 a * s + c (exact for the small integers and powers of two used here)
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t s, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(s), "r"(c));
  return r;
}

// Code word q of each 16-byte half of row (l, j)'s slice chunk, from the
// codes region [j][h][t][16 B] (t = 32 slice + l).  A warp's eight rows of
// one half are 128 contiguous bytes, so each of the two loads is one
// conflict-free wavefront.
__device__ __forceinline__ void mma_row_words(const uint8_t* stage, int slice, int l, int j, int q,
                                              uint32_t (&w)[2]) {
  const int t = slice * 32 + l;
  w[0] = *reinterpret_cast<const uint32_t*>(stage + ((j * 2 + 0) * kLaneSlots + t) * 16 + 4 * q);
  w[1] = *reinterpret_cast<const uint32_t*>(stage + ((j * 2 + 1) * kLaneSlots + t) * 16 + 4 * q);
}

// Activation loads: `row` is x[m] (null for m >= M: zeros), K its length.
// x[m][k0 .. k0+3] as two fp16 pairs (k0 a multiple of 4); zero for k >= K.
// `vec`: x is 16-byte aligned and K % 8 == 0.
__device__ __forceinline__ void ld_x4(uint32_t* out, const unsigned short* row, int64_t K, int64_t k0, bool vec) {
  if (row == nullptr || k0 >= K) {
    out[0] = out[1] = 0u;
    return;
  }
  if (vec) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(row + k0));
    out[0] = v.x; out[1] = v.y;
    return;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t k = k0 + 2 * i;
    const uint32_t lo = k < K ? __ldg(row + k) : 0u;
    const uint32_t hi = k + 1 < K ? __ldg(row + k + 1) : 0u;
    out[i] = lo | (hi << 16);
  }
}

// x[m][k0 .. k0+7] as four fp16 pairs; zero for k >= K.  k0 is a multiple of
// 8; with `vec` the eight values are one aligned 16-byte load.
__device__ __forceinline__ void ld_x8(uint32_t* out, const unsigned short* row, int64_t K, int64_t k0, bool vec) {
  if (row == nullptr || k0 >= K) {
    out[0] = out[1] = out[2] = out[3] = 0u;
    return;
  }
  if (vec) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k0));
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t k = k0 + 2 * i;
    const uint32_t lo = k < K ? __ldg(row + k) : 0u;
    const uint32_t hi = k + 1 < K ? __ldg(row + k + 1) : 0u;
    out[i] = lo | (hi << 16);
  }
}

template <class F, int NT>
__device__ __noinline__ void mma_rebuild_table(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
  F::template mma_init_shared<NT>(lut, cb, warp, lane);
}

// GLU: the handle's rows are a gate and an up projection interleaved in
// 64-row halves of every row tile (as for wstream_kernel's GLU form), and
// the stores are y[m][64t + r] = SiLU(gate) * up.  A thread's m-tiles 2a and
// 2a + 1 hold the same rows of the two halves (l and l + 16, the same j), so
// each gate sum meets its up sum in one thread; split row tiles go through
// the pair finisher.
template <class F, int NB, bool PAR = false, bool GLU = false>
__global__ void __launch_bounds__(mma_threads<F, NB, PAR>(), F::mma_ctas(NB)) wstream_mma_kernel(const RunParams p, int M) {
  constexpr int NS = mma_stages_of<F, NB, PAR>();
  constexpr int TB = F::kTileBytes;
  constexpr int KS = F::kKW / 16;        // k16 steps per slice
  constexpr int BS = F::kMmaBlockSteps;  // k16 steps per scale block, 0: none
  constexpr int NBLK = BS > 0 ? KS / BS : 1;
  constexpr int XW = F::kMmaXWords;      // activation words per (thread, activation row)
  constexpr bool PF = F::mma_prefetch_x(NB);  // activations a tile ahead (registers permitting)
  constexpr int NT = mma_threads<F, NB, PAR>();
  constexpr int NW = mma_warps<F, NB, PAR>();
  constexpr int SPW = mma_spw_of<F, NB, PAR>();  // k-slices per warp
  constexpr int SG = kSlices / SPW;              // slice groups
  constexpr int TG = PAR ? 2 * SG : SG;          // partial sums per row added at a row-tile end
  static_assert(!PAR || (F::mma_ctas(NB) == 1 && NS % 2 == 0 && NS >= 4), "tile parity geometry");

  if (static_cast<int>(blockIdx.x) == p.skip_cta) return;  // test hook (QGEMV_FAULT_SKIP_CTA)
  extern __shared__ __align__(128) uint8_t smem[];
  // stage s at ring0 (s = 0) or ringN + (s - 1) TB
  uint8_t* ring0 = smem;
  uint8_t* ringN = smem + TB;
  float4* red;
  uint8_t* fsh;
  uint64_t* full;
  uint32_t lut_key = 0;  // table formats: the lane's entry address bits (F::mma_lut_key)
  if constexpr (F::kMmaSharedBytes == 0) {
    red = reinterpret_cast<float4*>(smem + NS * TB);
    fsh = smem;  // unused
    full = reinterpret_cast<uint64_t*>(smem + NS * TB + mma_red_bytes<NB>());
  } else {
    static_assert(F::kMmaSharedBytes == kTableAlign, "one 64 KB table");
    static_assert(mma_pre_bytes<F, NB, PAR>() + kTablePreSlack <= kTableAlign, "pre-table layout");
    const uint32_t base = smem_u32(smem);
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t R0 = (base + (kTableAlign - 1)) & ~uint32_t(kTableAlign - 1);
    if (R0 - base < uint32_t(mma_pre_bytes<F, NB, PAR>()) ||
        R0 + kTableAlign + mma_post_bytes<F, NB, PAR>() > base + dyn) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
      return;
    }
    fsh = smem + (R0 - base);
    ringN = fsh + kTableAlign;
    full = reinterpret_cast<uint64_t*>(smem + TB);
    red = reinterpret_cast<float4*>(NB == 1 ? smem + TB + mma_bar_bytes<F, NB, PAR>() : ringN + (NS - 1) * TB);
    lut_key = F::mma_lut_key(R0, static_cast<int>(threadIdx.x & 31u));
  }
  uint64_t* empty = full + NS;
  auto stage_ptr = [&](int64_t s) { return s == 0 ? ring0 : ringN + (s - 1) * TB; };
  __shared__ volatile int s_abort;
  __shared__ NextTable<F> s_next;
  __shared__ __align__(16) CtaPlan s_plan;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int q = lane & 3, gi = lane >> 2;
  // slice group sgrp (slices sgrp * SPW .. + SPW - 1), row half hf; with
  // tile parity, warp 8 par + 4 hf + sgrp computes the tiles j with j % 2 == par
  const int par = PAR ? warp >> 3 : 0;
  const int sgrp = PAR ? warp & 3 : warp % SG;
  const int hf = PAR ? (warp >> 2) & 1 : warp / SG;
  const int ti = par * SG + sgrp;  // index of the warp's partial sums in the row-tile tree
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t t0 = stream_split<SplitModeOf<F>::value>(c, p.T, G);
  const int64_t t1 = stream_split<SplitModeOf<F>::value>(c + 1, p.T, G);
  const int ntiles = static_cast<int>(t1 - t0);
  const int64_t rt_first = div_fast(t0, p.nKT);

  const bool elected = (tid == 0);
  uint64_t pol = 0;
  int n_issued = 0;
  if (elected) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAR ? NW / 2 : NW);  // with tile parity one half uses a stage
    }
    s_abort = 0;
    fence_mbarrier_init();
    pol = l2_policy_evict_first();
    // with tile parity the first tile of each half only: the other stages
    // are filled from the main loop, after the grid dependency (as in
    // wstream_kernel, so that the CTAs that start last find a short queue)
    for (; n_issued < (PAR ? 2 : NS - 1) && n_issued < ntiles; ++n_issued) {
      mbar_arrive_expect_tx(&full[n_issued], TB);
      bulk_g2s(stage_ptr(n_issued), p.tiles + (t0 + n_issued) * TB, TB, &full[n_issued], pol);
    }
  }
  fetch_plan(&s_plan, p.plan, c, tid);
  if constexpr (F::kCbEntries > 0) {
    if (p.seg_of_rt != nullptr && ntiles > 0)
      prefetch_next_table<F>(&s_next, p, rt_first, div_fast(p.T, p.nKT), true, tid);
  }
  F::template mma_init_shared<NT>(fsh, table_of<F>(p, rt_first), warp, lane);
  if constexpr (GLU && GluTables<F>::value)
    F::template mma_init_shared<NT>(fsh + kGluUpTable, table_of<F>(p, rt_first) + F::kCbEntries, warp, lane);
  __syncthreads();

  // The prologue touches nothing a previous kernel writes; x and the outputs
  // wait for the previous grid (programmatic dependent launch).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t rt = rt_first;
  int kt = static_cast<int>(t0 - rt * p.nKT);
  const bool xvec = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.K & 7) == 0;
  const bool xq_vec = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0;  // INT8: prepared rows of K bytes, K % 128 == 0
  // activation fragments of the thread's B rows m = gi + 8 nb for each of
  // its slices (a tile ahead when PF, else loaded at the top of each tile)
  uint32_t xw[SPW][NB][XW];
  const unsigned short* xrow[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
    xrow[nb] = gi + 8 * nb < M ? reinterpret_cast<const unsigned short*>(p.x) + (gi + 8 * nb) * p.K : nullptr;
  auto load_x = [&](uint32_t (&dst)[SPW][NB][XW], int ktile) {
#pragma unroll
    for (int ss = 0; ss < SPW; ++ss) {
      const int64_t kb = static_cast<int64_t>(ktile) * F::kKT + (sgrp * SPW + ss) * F::kKW;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if constexpr (MmaXCodes<F>::value)
          F::mma_load_x_q(dst[ss][nb], p, M, gi + 8 * nb, 8 * nb + 2 * q, kb, q, xq_vec);
        else
          F::mma_load_x(dst[ss][nb], xrow[nb], p.K, kb, q, xvec);
      }
    }
  };
  const int nKT = static_cast<int>(p.nKT);
  // k-tile index k (< nKT + 2) reduced into [0, nKT)
  auto wrap_kt = [nKT](int k) {
    if (k >= nKT) k -= nKT;
    if (k >= nKT) k -= nKT;
    return k;
  };
  if constexpr (PF) {
    if (par < ntiles) load_x(xw, wrap_kt(kt + par));
  }

  // acc[mt][nb]: D fragment of m-tile mt and activation block nb
  float acc[kMmaTiles][NB][4];
#pragma unroll
  for (int mt = 0; mt < kMmaTiles; ++mt)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nb][e] = 0.f;

  const int nt = ntiles;
  const bool stacked = F::kCbEntries > 0 && p.seg_of_rt != nullptr;
  // A new row tile of a stacked handle may use another codebook: rebuild the
  // table once every warp is done with the old one.
  auto next_table = [&]() {
    if constexpr (F::kCbEntries > 0)
      advance_table<F, NT>(&s_next, p, rt, tid,
                           [&](const uint16_t* cb) { mma_rebuild_table<F, NT>(fsh, cb, warp, lane); });
  };

  // The warp's part of the tile in stage st (fill parity fp), k-tile kt_cur:
  // activations (those of the warp's next tile, k-tile kt_pref, when PF),
  // wait for the codes, decode and multiply.
  auto compute_tile = [&](int st, uint32_t fp, int kt_cur, int kt_pref, bool pref, bool abort) {
    uint32_t xn[PF ? SPW : 1][PF ? NB : 1][PF ? XW : 1];
    if constexpr (PF) {
      if (pref) load_x(xn, kt_pref);
    } else {
      load_x(xw, kt_cur);
    }

      const bool ok = !abort && mbar_wait_bounded(&full[st], fp);
      if (!ok) {
        if (!abort && lane == 0) atomicOr(p.err, kErrTimeoutFull);
        s_abort = 1;
      } else {
        const uint8_t* stage = stage_ptr(st);
  #pragma unroll
        for (int ss = 0; ss < SPW; ++ss) {
          const int slice = sgrp * SPW + ss;
          // codes (and scales) of the thread's eight rows in this slice; after
          // the warp's last slice, release the stage
          uint32_t w[kMmaTiles][2][F::kMmaRowWords];
          typename F::MmaScales d[kMmaTiles][2];  // block scales of the rows, read per block
          auto load_mtile = [&](int mt) {
            const int j = 2 * hf + (mt >> 1);
            const int l = 16 * (mt & 1) + gi;
            F::mma_load_row(stage, slice, l, j, q, w[mt][0]);
            F::mma_load_row(stage, slice, l + 8, j, q, w[mt][1]);
            if constexpr (BS > 0) {
              F::mma_scales(stage, slice, l, j, d[mt][0]);
              F::mma_scales(stage, slice, l + 8, j, d[mt][1]);
            }
          };
          // MG m-tiles at a time, their MMAs interleaved so that consecutive
          // MMAs are independent (all four for one activation block; one for
          // two, which need twice the accumulators)
          constexpr int MG = NB == 1 ? kMmaTiles : 1;
          constexpr bool kLate = MG == 1 && MmaLateCodes<F>::value;
          if constexpr (!kLate) {
  #pragma unroll
            for (int mt = 0; mt < kMmaTiles; ++mt) load_mtile(mt);
            if (ss == SPW - 1) release_stage(&empty[st], lane);
          }
  #pragma unroll
          for (int mg = 0; mg < kMmaTiles; mg += MG) {
            if constexpr (kLate) {
              load_mtile(mg);
              if (ss == SPW - 1 && mg == kMmaTiles - 1) release_stage(&empty[st], lane);
            }
  #pragma unroll
            for (int blk = 0; blk < NBLK; ++blk) {
              float tmp[MG][NB][4];  // block sums (block formats); the first MMA writes them
  #pragma unroll
              for (int ks = blk * (BS > 0 ? BS : KS); ks < (blk + 1) * (BS > 0 ? BS : KS); ++ks) {
                // one A fragment per codebook (additive formats sum two); the
                // codebook loop is outside the m-tile loop so that MMAs into
                // the same accumulator are not adjacent
  #pragma unroll
                for (int cb = 0; cb < F::kMmaCodebooks; ++cb) {
  #pragma unroll
                  for (int mi = 0; mi < MG; ++mi) {
                    const int mt = mg + mi;
                    // GLU with two tables: the odd m-tiles hold the up rows
                    const uint32_t key = lut_key | (GLU && GluTables<F>::value && (mt & 1) ? kGluUpTable : 0);
                    const uint2 r0 = F::mma_frag(w[mt][0], ks, key, cb);  // row gi: (k lo pair, k hi pair)
                    const uint2 r1 = F::mma_frag(w[mt][1], ks, key, cb);  // row gi + 8
  #pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                      const uint2 bf = F::mma_bfrag(xw[ss][nb], ks);
                      if constexpr (BS > 0) {
                        static_assert(BS == 0 || F::kMmaCodebooks == 1, "block scales with one codebook");
                        if (ks == blk * BS)
                          mma_16816_c0(tmp[mi][nb], r0.x, r1.x, r0.y, r1.y, bf.x, bf.y);
                        else
                          mma_16816(tmp[mi][nb], r0.x, r1.x, r0.y, r1.y, bf.x, bf.y);
                      } else
                        mma_16816(acc[mt][nb], r0.x, r1.x, r0.y, r1.y, bf.x, bf.y);
                    }
                  }
                }
              }
              if constexpr (BS > 0) {
  #pragma unroll
                for (int mi = 0; mi < MG; ++mi)
  #pragma unroll
                  for (int nb = 0; nb < NB; ++nb) {
                    const int mt = mg + mi;
                    const float d0 = F::mma_scale(d[mt][0], blk), d1 = F::mma_scale(d[mt][1], blk);
                    if constexpr (MmaXCodes<F>::value) {
                      // the exact integer sum times the activation column's group scale
  #pragma unroll
                      for (int e = 0; e < 4; ++e)
                        tmp[mi][nb][e] = __fmul_rn(F::mma_col_scale(xw[ss][nb], e & 1), tmp[mi][nb][e]);
                    }
                    acc[mt][nb][0] = fmaf(d0, tmp[mi][nb][0], acc[mt][nb][0]);
                    acc[mt][nb][1] = fmaf(d0, tmp[mi][nb][1], acc[mt][nb][1]);
                    acc[mt][nb][2] = fmaf(d1, tmp[mi][nb][2], acc[mt][nb][2]);
                    acc[mt][nb][3] = fmaf(d1, tmp[mi][nb][3], acc[mt][nb][3]);
                  }
              }
            }
          }
        }
      }
    if constexpr (PF) {
#pragma unroll
      for (int ss = 0; ss < SPW; ++ss)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < XW; ++e) xw[ss][nb][e] = xn[ss][nb][e];
    }
  };

  // Row-tile epilogue: add the TG partial sums of every row in a fixed tree,
  // then store them to y or to the stream-K partial slots.
  auto row_epilogue = [&](int64_t cur_rt) {
  #pragma unroll 1
      for (int width = TG / 2; width >= 1; width >>= 1) {
        if (ti >= width && ti < 2 * width) {
  #pragma unroll
          for (int mt = 0; mt < kMmaTiles; ++mt)
  #pragma unroll
            for (int nb = 0; nb < NB; ++nb)
              red[(((ti - width) * 2 + hf) * kMmaTiles + mt) * NB * 32 + nb * 32 + lane] =
                  make_float4(acc[mt][nb][0], acc[mt][nb][1], acc[mt][nb][2], acc[mt][nb][3]);
        }
        named_bar_sync(1, NT);
        if (ti < width) {
  #pragma unroll
          for (int mt = 0; mt < kMmaTiles; ++mt)
  #pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const float4 v = red[((ti * 2 + hf) * kMmaTiles + mt) * NB * 32 + nb * 32 + lane];
              acc[mt][nb][0] += v.x;
              acc[mt][nb][1] += v.y;
              acc[mt][nb][2] += v.z;
              acc[mt][nb][3] += v.w;
            }
        }
        named_bar_sync(1, NT);
      }
      if (ti == 0) {
        const bool owner = (cur_rt * p.nKT >= t0) && ((cur_rt + 1) * p.nKT <= t1);
        const int side = (cur_rt * p.nKT <= t0) ? 0 : 1;
        float* my_part = p.partials + (c * 2 + side) * kPartialStride;
  #pragma unroll
        for (int mt = 0; mt < kMmaTiles; ++mt)
  #pragma unroll
          for (int nb = 0; nb < NB; ++nb)
  #pragma unroll
            for (int e = 0; e < 4; ++e) {
              // D element e: weight row gi (+8 for e >= 2), activation row 2q + (e & 1)
              const int m = 8 * nb + 2 * q + (e & 1);
              const int l = 16 * (mt & 1) + gi + (e >> 1) * 8;
              const int r = 4 * l + 2 * hf + (mt >> 1);
              if (m < M) {
                if (GLU && owner) {
                  // gate row r (m-tile mt, l < 16) with up row r + 64 (m-tile mt + 1)
                  if constexpr (GLU) {
                    if ((mt & 1) == 0) glu_store(p, m, cur_rt * (kTileRows / 2) + r, acc[mt][nb][e], acc[mt + 1][nb][e]);
                  }
                } else if (owner) {
                  const int64_t n = cur_rt * kTileRows + r;
                  if (n < p.N) {
                    if constexpr (F::kMmaRowScales)
                      store_y(p, m * p.N + n, __fmul_rn(__half2float(F::mma_row_scales(p)[n]), acc[mt][nb][e]));
                    else
                      store_y(p, m * p.N + n, acc[mt][nb][e]);
                  }
                } else {
                  st_relaxed_f32(my_part + m * kTileRows + r, acc[mt][nb][e]);
                }
              }
            }
      }
  #pragma unroll
      for (int mt = 0; mt < kMmaTiles; ++mt)
  #pragma unroll
        for (int nb = 0; nb < NB; ++nb)
  #pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][nb][e] = 0.f;
  };

  if constexpr (PAR) {
    // Tile parity: tile j sits in stage j % NS and is computed by half j % 2,
    // so each half owns every second stage and runs its own pipeline: at its
    // tile j its first thread fills the stage of its tile j - 2 (released
    // one tile ago; for j < 2 a stage not used yet) with tile j + NS - 2.
    // The prologue issued tiles 0 and 1.  Both halves walk the run row tile
    // by row tile and meet at each row-tile end.
    static_assert(!PAR || NS >= 4, "tile parity: two stages per half");
    const bool leader = (lane == 0) && ((warp & 7) == 0);
    const uint64_t lpol = leader ? l2_policy_evict_first() : 0;
    int u_last = -1;  // leader: last tile of its parity issued (by the prologue or by itself)
    for (int u = par; u < 2 && u < nt; u += 2) u_last = u;
    int i = 0;  // first tile of the current row tile segment
    while (i < nt) {
      if (stacked && i > 0) next_table();
      const int iend = i + min(nt - i, nKT - kt);
#pragma unroll 1
      for (int j = i + ((i ^ par) & 1); j < iend; j += 2) {
        bool abort = s_abort != 0;
        const int u = j + NS - 2;
        // tiles 0 and 1 came from the prologue: never fill a stage twice
        if (leader && !abort && u >= 2 && u < nt) {
          const int sn = u % NS;
          if (u >= NS && !mbar_wait_bounded(&empty[sn], static_cast<uint32_t>(((u - NS) / NS) & 1))) {
            atomicOr(p.err, kErrTimeoutEmpty);
            s_abort = 1;
            abort = true;
          } else {
            mbar_arrive_expect_tx(&full[sn], TB);
            bulk_g2s(stage_ptr(sn), p.tiles + (t0 + u) * TB, TB, &full[sn], lpol);
            u_last = u;
          }
        }
        const int ktj = kt + (j - i);
        compute_tile(j % NS, static_cast<uint32_t>((j / NS) & 1), ktj, wrap_kt(ktj + 2), j + 2 < nt, abort);
      }
      row_epilogue(rt);
      i = iend;
      kt = 0;
      ++rt;
    }
    // Never leave while a copy issued by this half may still be landing
    // (only after an aborted run): wait for the last fill of each of its stages.
    if (leader && s_abort != 0) {
      for (int u = u_last; u >= 0 && u > u_last - NS; u -= 2)
        mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
    }
  } else {
    int s = 0;
    uint32_t ph = 0;
    int su = static_cast<int>(n_issued % NS);
    uint32_t phu = static_cast<uint32_t>((n_issued / NS) & 1);
    for (int i = 0; i < nt; ++i) {
      if (stacked && kt == 0 && i > 0) next_table();
      bool abort = s_abort != 0;
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
      compute_tile(s, ph, kt, kt_next, i + 1 < nt, abort);
      if (++s == NS) { s = 0; ph ^= 1; }
      const bool row_end = (kt_next == 0) || (i + 1 == nt);
      const int64_t cur_rt = rt;
      kt = kt_next;
      if (kt_next == 0) ++rt;
      if (row_end) row_epilogue(cur_rt);
    }
    if (elected && s_abort != 0) {
      for (int u = (n_issued > NS ? n_issued - NS : 0); u < n_issued; ++u)
        mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
    }
  }

  // split row tiles: the shared polled-slot finisher, with M activation rows
  static_assert(mma_red_bytes<NB>() >= 2 * NT * 4, "finishing scratch");
  float* s_sub = reinterpret_cast<float*>(red);
  wait_plan();
  const __half* row_scales = nullptr;  // per-row output scales (F::kMmaRowScales), applied at the finish
  if constexpr (F::kMmaRowScales) row_scales = F::mma_row_scales(p);
  if constexpr (GLU) {
    for (int sg = 0; sg < 2; ++sg)
      if (s_plan.seg_rt[sg] >= 0) finish_rows_glu<8 * NB, NT>(p, s_plan, sg, 1.0f, tid, M);
  } else {
    finish_all<kTileRows, 8 * NB, NT>(p, kPartialStride, s_plan, row_scales, 1.0f, s_sub, tid, M);
  }
}

}  // namespace qgemv

// fmt_fields.cuh -- Q4_0 and PQ2_0: formats whose weight is an integer code
// times a per-block fp16 scale.
//
// Decode trick ("denormal fields").  In the prepared tiles every 32-bit word
// holds the codes of consecutive k (8 nibbles for Q4_0, 16 two-bit fields
// for PQ2_0).  A code sitting at bit p of a word, masked out with one AND,
// *is* the fp32 bit pattern of the subnormal q * 2^(p - 149), exactly.
// Multiplying it by x * 2^(109 - p) (the activation pre-scaled once per
// tile, an exact power-of-two scaling) gives x * q * 2^-40 exactly, so one
// AND plus one FMA per weight (half an FFMA2) decodes and accumulates.  Codes
// above bit 22 would reach the exponent field; those are first shifted down
// by 12 (one shift per word).  The code offset (q - 8 for Q4_0, c - 1 for
// PQ2_0) is applied once per block with the block sum of x:
//     sum_k x_k (q_k - off) = sum_k x_k q_k - off * sum_k x_k,
// and the per-row block scale d multiplies that difference.  Outputs carry a
// factor 2^-40 until the epilogue multiplies it back (exact).
//
// Formats: Q4_0 -- "Model quantization, read carefully" (localai blog),
// "Anatomy of a block": 32 weights, one fp16 scale, (q - 8) * d, 18 bytes.
// PQ2_0 -- "Making a ternary reasoning model fast in vLLM", "Anatomy of a
// PQ2_0 block": 128 weights, fp16 d, two-bit codes 0..3 -> -1, 0, +1, +2.
#pragma once

#include "gemv_kernel.cuh"

namespace qgemv {

constexpr int kFieldExp = -40;                       // outputs carry 2^kFieldExp
constexpr float kFieldOutScale = pow2f(-kFieldExp);  // 2^40

// 2^e as a float (exact for -126 <= e <= 127).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }


// ------------------------------------------------------------------ Q4_0 --
//
// Tile: 128 rows x 256 k.  Slice s <-> Q4_0 block s of the tile (32 k);
// lane slot t = 32s + l <-> rows 4l..4l+3.
//   codes  [j = 0..3][t][16 B]  row 4l+j, block s: word i holds k = 8i..8i+7
//          of the block, nibble jj at bits 4jj.
//   scales [t][4 x fp16]        d of rows 4l..4l+3, block s.
struct FmtQ4_0 {
  static constexpr int kKW = 32;
  static constexpr int kKT = kKW * kSlices;                   // 256
  static constexpr int kCodeBytes = kLaneSlots * kRowsPerLane * 16;
  static constexpr int kTileBytes = kCodeBytes + kLaneSlots * 8;  // 18432
  __host__ __device__ static constexpr int stages(int) { return 6; }
  static constexpr int kSharedBytes = 0;
  static constexpr float kOutScale = kFieldOutScale;
  using XRegs = XRegsT<1>;

  // bit position of the nibble of k = 8i + jj once extracted (jj >= 5 are
  // taken from the word shifted right by 12)
  __host__ __device__ static constexpr int field_pos(int jj) { return jj <= 4 ? 4 * jj : 4 * jj - 12; }

  __device__ static void init_shared(uint8_t*, const GemvParams&, int, int) {}

  template <int M>
  __device__ static void load_x(XRegs& xr, const GemvParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 1>(xr, p, kt, slice, lane);
  }

  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[M], const XRegs& xr, int lane) {
    stage_x_slice<M, 1>(xs, xsum, xr, lane,
                        [](int kk) { return exp2i(109 - field_pos(kk & 7)); });
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs, const float (&xsum)[M],
                                   RowAcc<M, RPW>& yacc, uint8_t*, int slice, int half, int lane,
                                   uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    uint4 cwd[RPW];
#pragma unroll
    for (int j = 0; j < RPW; ++j) cwd[j] = lds128(stage + ((j0 + j) * kLaneSlots + t) * 16);
    const uint2 sc = *reinterpret_cast<const uint2*>(stage + kCodeBytes + t * 8);
    release_stage(empty_bar, lane);

    // scales of this lane's rows j0..j0+RPW-1 (two fp16 per 32-bit word)
    float dr[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const uint32_t sw = (RPW == 4) ? (r < 2 ? sc.x : sc.y) : (half ? sc.y : sc.x);
      dr[r] = h2f((r & 1) ? (sw >> 16) : (sw & 0xffffu));
    }
    // code offset 8: subtract 8 * sum(x) (in the 2^-40 scaled domain)
    float off[M];
#pragma unroll
    for (int m = 0; m < M; ++m) off[m] = xsum[m] * (-8.0f * pow2f(kFieldExp));

    constexpr int RP = (M > 8 && RPW > 2) ? 2 : RPW;  // rows per pass (register budget)
#pragma unroll
    for (int pass = 0; pass < RPW / RP; ++pass) {
      float2 acc[RP][M];
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = make_float2(off[m], 0.f);
      constexpr int UI = (M > 8) ? 1 : 4;  // bound live ranges for large M
#pragma unroll UI
      for (int i = 0; i < 4; ++i) {
        uint32_t fld[RP][8];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const uint32_t wv = word_of(cwd[pass * RP + r], i);
          const uint32_t wh = wv >> 12;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            fld[r][jj] = (jj <= 4 ? wv : wh) & (0xfu << field_pos(jj));
        }
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          float2 xv[M];
          load_xpairs<M>(xs, 4 * i + pp, xv);
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const float2 w2 = make_float2(u2f(fld[r][2 * pp]), u2f(fld[r][2 * pp + 1]));
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = __ffma2_rn(w2, xv[m], acc[r][m]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        float a[M];
#pragma unroll
        for (int m = 0; m < M; ++m) a[m] = acc[r][m].x + acc[r][m].y;
        yacc.add_row(pass * RP + r, dr[pass * RP + r], a);
      }
    }
  }
};

// ----------------------------------------------------------------- PQ2_0 --
//
// Tile: 128 rows x 512 k (four PQ2 blocks).  Slice s <-> k 64s..64s+63,
// i.e. half (s & 1) of block s >> 1; lane slot t = 32s + l <-> rows 4l..4l+3.
//   codes  [j][t][16 B]  word i holds k = 16i..16i+15 of the slice, two-bit
//          field jj at bits 2jj.
//   scales [blk = 0..3][l][4 x fp16]  d of rows 4l..4l+3, block blk.
struct FmtPQ2 {
  static constexpr int kKW = 64;
  static constexpr int kKT = kKW * kSlices;                   // 512
  static constexpr int kCodeBytes = kLaneSlots * kRowsPerLane * 16;
  static constexpr int kTileBytes = kCodeBytes + 4 * 32 * 8;  // 17408
  __host__ __device__ static constexpr int stages(int) { return 6; }
  static constexpr int kSharedBytes = 0;
  static constexpr float kOutScale = kFieldOutScale;
  using XRegs = XRegsT<2>;

  __host__ __device__ static constexpr int field_pos(int jj) { return jj <= 10 ? 2 * jj : 2 * jj - 12; }

  __device__ static void init_shared(uint8_t*, const GemvParams&, int, int) {}

  template <int M>
  __device__ static void load_x(XRegs& xr, const GemvParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 2>(xr, p, kt, slice, lane);
  }

  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[M], const XRegs& xr, int lane) {
    stage_x_slice<M, 2>(xs, xsum, xr, lane,
                        [](int kk) { return exp2i(109 - field_pos(kk & 15)); });
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs, const float (&xsum)[M],
                                   RowAcc<M, RPW>& yacc, uint8_t*, int slice, int half, int lane,
                                   uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    uint4 cwd[RPW];
#pragma unroll
    for (int j = 0; j < RPW; ++j) cwd[j] = lds128(stage + ((j0 + j) * kLaneSlots + t) * 16);
    const uint2 sc =
        *reinterpret_cast<const uint2*>(stage + kCodeBytes + ((slice >> 1) * 32 + lane) * 8);
    release_stage(empty_bar, lane);

    // scales of this lane's rows j0..j0+RPW-1 (two fp16 per 32-bit word)
    float dr[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const uint32_t sw = (RPW == 4) ? (r < 2 ? sc.x : sc.y) : (half ? sc.y : sc.x);
      dr[r] = h2f((r & 1) ? (sw >> 16) : (sw & 0xffffu));
    }
    // code offset 1: subtract sum(x) (in the 2^-40 scaled domain)
    float off[M];
#pragma unroll
    for (int m = 0; m < M; ++m) off[m] = xsum[m] * (-pow2f(kFieldExp));

    constexpr int RP = (M > 8 && RPW > 2) ? 2 : RPW;
#pragma unroll
    for (int pass = 0; pass < RPW / RP; ++pass) {
      float2 acc[RP][M];
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = make_float2(off[m], 0.f);
      constexpr int UI = (M > 8) ? 1 : 4;  // bound live ranges for large M
#pragma unroll UI
      for (int i = 0; i < 4; ++i) {
        uint32_t wv[RP], wh[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          wv[r] = word_of(cwd[pass * RP + r], i);
          wh[r] = wv[r] >> 12;
        }
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
          float2 xv[M];
          load_xpairs<M>(xs, 8 * i + pp, xv);
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const int j0 = 2 * pp, j1 = 2 * pp + 1;
            const uint32_t f0 = (j0 <= 10 ? wv[r] : wh[r]) & (3u << field_pos(j0));
            const uint32_t f1 = (j1 <= 10 ? wv[r] : wh[r]) & (3u << field_pos(j1));
            const float2 w2 = make_float2(u2f(f0), u2f(f1));
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = __ffma2_rn(w2, xv[m], acc[r][m]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        float a[M];
#pragma unroll
        for (int m = 0; m < M; ++m) a[m] = acc[r][m].x + acc[r][m].y;
        yacc.add_row(pass * RP + r, dr[pass * RP + r], a);
      }
    }
  }
};

}  // namespace qgemv

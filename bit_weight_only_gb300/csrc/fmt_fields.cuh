// fmt_fields.cuh -- Q4_0 and PQ2_0: formats whose weight is an integer code
// times a per-block fp16 scale.
//
// Decode trick ("subnormal fields").  In the prepared tiles every 32-bit word
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
//
// Both use 32 code bytes per (row, lane slot) per tile: codes region
// [j = row 0..3 of the slot][h = 16-byte half][t = lane slot 0..255][16 B].
#pragma once

#include "gemv_kernel.cuh"
#include "mma_kernel.cuh"

namespace qgemv {

constexpr int kFieldExp = -40;                       // outputs carry 2^kFieldExp
constexpr float kFieldOutScale = pow2f(-kFieldExp);  // 2^40
constexpr int kCodeBytes32 = kRowsPerLane * 2 * kLaneSlots * 16;  // 32 KB of codes per tile

// 2^e as a float (exact for -126 <= e <= 127).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// The eight code words of rows j0 .. j0+R-1 of lane slot t.
template <int R>
__device__ __forceinline__ void load_codes32(const uint8_t* stage, int j0, int t,
                                             uint4 (&lo)[R], uint4 (&hi)[R]) {
#pragma unroll
  for (int j = 0; j < R; ++j) {
    lo[j] = lds128(stage + (((j0 + j) * 2 + 0) * kLaneSlots + t) * 16);
    hi[j] = lds128(stage + (((j0 + j) * 2 + 1) * kLaneSlots + t) * 16);
  }
}

__device__ __forceinline__ uint32_t word8(const uint4& lo, const uint4& hi, int i) {
  return i < 4 ? word_of(lo, i) : word_of(hi, i - 4);
}

// ------------------------------------------------------------------ Q4_0 --
//
// Tile: 128 rows x 512 k.  Slice s <-> Q4_0 blocks 2s, 2s+1 of the tile
// (64 k); lane slot t = 32s + l <-> rows 4l..4l+3.
//   codes  word i (0..7) of (row, slot) holds k = 8i..8i+7 of the slice,
//          nibble jj at bits 4jj; words 0-3 are block 2s, 4-7 block 2s+1.
//   scales [t][j = 0..3][b = 0..1] fp16: d of row 4l+j, block 2s+b.
struct FmtQ4_0 {
  static constexpr int kKW = 64;
  static constexpr int kKT = kKW * kSlices;                        // 512
  static constexpr int kCodeBytes = kCodeBytes32;
  static constexpr int kTileBytes = kCodeBytes + kLaneSlots * 16;  // 36864
  // M = 1 CUDA-core kernel: two CTAs of eight warps per SM, two stages each
  static constexpr int kCtasPerSm = 2;
  static constexpr bool kTileParity = false;
  __host__ __device__ static constexpr int stages(int) { return 2; }
  static constexpr int kSharedBytes = 0;
  static constexpr float kOutScale = kFieldOutScale;
  static constexpr int kSumGroups = 2;  // one offset sum per Q4_0 block of the slice

  // ---- register-decode tensor-core path (mma_kernel.cuh) ----
  // Thread q of a fragment row holds code word q of each block b of the
  // slice (k = 32b + 8q .. +7).  k16 step ks lies in block b = ks / 2;
  // with sub = ks % 2 its two k pairs are nibbles (2sub, 2sub + 4) and
  // (2sub + 1, 2sub + 5) of that word: one LOP3 makes each pair 1024 + code
  // (or 1024 + 16 code) as fp16, one HFMA2 turns it into code - 8, exactly.
  static constexpr int kMmaSharedBytes = 0;
  static constexpr int kMmaRowWords = 2;   // words q of the two 16-byte halves
  static constexpr int kMmaCodebooks = 1;
  static constexpr bool kMmaRowScales = false;
  static constexpr bool kMmaGlu = true;    // the GLU form of the tensor-core kernel
  __device__ static const __half* mma_row_scales(const RunParams&) { return nullptr; }
  static constexpr int kMmaBlockSteps = 2;
  static constexpr int kMmaXWords = 8;  // x[m][32b + 8q .. +7], b = 0, 1
  // two slices per warp, eight warps per CTA, two CTAs per SM, two stages each
  __host__ __device__ static constexpr int mma_spw(int) { return 2; }
  __host__ __device__ static constexpr int mma_ctas(int) { return 2; }
  __host__ __device__ static constexpr bool mma_par(int) { return false; }  // two CTAs per SM instead
  __host__ __device__ static constexpr int mma_stages(int) { return 2; }
  __host__ __device__ static constexpr bool mma_prefetch_x(int nb) { return nb == 1; }
  template <int NT>
  __device__ static void mma_init_shared(uint8_t*, const uint16_t*, int, int) {}
  __device__ static void mma_load_row(const uint8_t* stage, int slice, int l, int j, int q, uint32_t (&w)[2]) {
    mma_row_words(stage, slice, l, j, q, w);
  }
  struct MmaScales { uint32_t h2; };  // d of the row's two blocks, fp16 pair
  __device__ static void mma_scales(const uint8_t* stage, int slice, int l, int j, MmaScales& d) {
    const int t = slice * 32 + l;
    d.h2 = *reinterpret_cast<const uint32_t*>(stage + kCodeBytes + (t * 4 + j) * 4);
  }
  __device__ static float mma_scale(const MmaScales& d, int blk) { return h2f(blk ? d.h2 >> 16 : d.h2 & 0xFFFFu); }
  __device__ static uint2 mma_frag(const uint32_t (&w)[2], int ks, uint32_t, int) {
    const uint32_t wd = (ks & 1) ? (w[ks >> 1] >> 8) : w[ks >> 1];
    return make_uint2(hfma2_u32(field_pair(wd, 0x000F000Fu), 0x3C003C00u, 0xE408E408u),   // x1 - 1032
                      hfma2_u32(field_pair(wd, 0x00F000F0u), 0x2C002C00u, 0xD480D480u));  // /16 - 72
  }
  __device__ static void mma_load_x(uint32_t (&xw)[kMmaXWords], const unsigned short* row, int64_t K,
                                    int64_t kb, int q, bool vec) {
    ld_x8(xw, row, K, kb + 8 * q, vec);
    ld_x8(xw + 4, row, K, kb + 32 + 8 * q, vec);
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    const uint32_t* X = xw + 4 * (ks >> 1);  // (x0,x1) (x2,x3) (x4,x5) (x6,x7) of the block's 8 k
    const int sub = ks & 1;
    return make_uint2(prmt(X[sub], X[sub + 2], 0x5410u), prmt(X[sub], X[sub + 2], 0x7632u));
  }

  using XRegs = XRegsT<2>;

  // bit position of the nibble of k = 8i + jj once extracted (jj >= 5 are
  // taken from the word shifted right by 12)
  __host__ __device__ static constexpr int field_pos(int jj) { return jj <= 4 ? 4 * jj : 4 * jj - 12; }

  static constexpr int kCbEntries = 0;
  template <int NT>
  __device__ static void init_shared(uint8_t*, const uint16_t*, int, int) {}

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 2>(xr, p, kt, slice, lane);
  }

  struct XScale { float v[2]; };
  __device__ static void x_scales(XScale& sc, int lane) {
#pragma unroll
    for (int i = 0; i < 2; ++i) sc.v[i] = exp2i(109 - field_pos((2 * lane + i) & 7));
  }

  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[kSumGroups][M], const XRegs& xr,
                                 const XScale& sc, int lane) {
    stage_x_slice<M, 2, kSumGroups>(xs, xsum, xr, lane, sc.v);
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&xsum)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t*, int slice, int half, int lane, uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    // rows per pass (register budget): all rows for small M, fewer above
    constexpr int RP = (M > 12) ? 1 : ((M > 8 && RPW > 2) ? 2 : RPW);
    // For large M the codes are loaded pass by pass and the stage is released
    // after the last pass, to keep registers for the accumulators.
    constexpr bool kLate = RP < RPW;
    uint4 clo[RP], chi[RP];
    if (!kLate) load_codes32<RP>(stage, j0, t, clo, chi);
    const uint4 sc = lds128(stage + kCodeBytes + t * 16);
    if (!kLate) release_stage(empty_bar, lane);

    // scale of (row j0 + r, block b): fp16 number 2*(j0 + r) + b of sc
    float dr[RPW][2];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const uint32_t sw = (RPW == 4) ? word_of(sc, r) : (half ? word_of(sc, 2 + r) : word_of(sc, r));
      dr[r][0] = h2f(sw & 0xffffu);
      dr[r][1] = h2f(sw >> 16);
    }

#pragma unroll
    for (int pass = 0; pass < RPW / RP; ++pass) {
      if (kLate) {
        load_codes32<RP>(stage, j0 + pass * RP, t, clo, chi);
        if (pass == RPW / RP - 1) release_stage(empty_bar, lane);
      }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        // code offset 8: start from -8 * sum(x) (in the 2^-40 scaled domain)
        float2 acc[RP][M];
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
          for (int m = 0; m < M; ++m)
            acc[r][m] = make_float2(xsum[b][m] * (-8.0f * pow2f(kFieldExp)), 0.f);
        constexpr int UI = (M > 8) ? 1 : 4;  // bound live ranges for large M
#pragma unroll UI
        for (int ii = 0; ii < 4; ++ii) {
          const int i = 4 * b + ii;
          uint32_t fld[RP][8];
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const int rr = kLate ? r : pass * RP + r;
            const uint32_t wv = word8(clo[rr], chi[rr], i);
            const uint32_t wh = wv >> 12;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              fld[r][jj] = (jj <= 4 ? wv : wh) & (0xfu << field_pos(jj));
          }
          float2 xv[4][M];
          load_xpair_run<M, 4>(xs, 4 * i, xv);
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
#pragma unroll
            for (int r = 0; r < RP; ++r) {
              const float2 w2 = make_float2(u2f(fld[r][2 * pp]), u2f(fld[r][2 * pp + 1]));
#pragma unroll
              for (int m = 0; m < M; ++m) acc[r][m] = __ffma2_rn(w2, xv[pp][m], acc[r][m]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          float a[M];
#pragma unroll
          for (int m = 0; m < M; ++m) a[m] = acc[r][m].x + acc[r][m].y;
          yacc.add_row(pass * RP + r, dr[pass * RP + r][b], a);
        }
      }
    }
  }
};

// ----------------------------------------------------------------- PQ2_0 --
//
// Tile: 128 rows x 1024 k (eight PQ2 blocks).  Slice s <-> block s of the
// tile (128 k); lane slot t = 32s + l <-> rows 4l..4l+3.
//   codes  word i (0..7) of (row, slot) holds k = 16i..16i+15 of the block,
//          two-bit field jj at bits 2jj.
//   scales [t][j = 0..3] fp16: d of row 4l+j, block s.
struct FmtPQ2 {
  static constexpr int kKW = 128;
  static constexpr int kSplitMode = 1;  // front-loaded stream-K split
  static constexpr int kKT = kKW * kSlices;                       // 1024
  static constexpr int kCodeBytes = kCodeBytes32;
  static constexpr int kTileBytes = kCodeBytes + kLaneSlots * 8;  // 34816
  // M = 1 CUDA-core kernel: two CTAs of eight warps per SM, two stages each
  static constexpr int kCtasPerSm = 2;
  static constexpr bool kTileParity = false;
  __host__ __device__ static constexpr int stages(int) { return 2; }
  static constexpr int kSharedBytes = 0;
  static constexpr float kOutScale = kFieldOutScale;
  static constexpr int kSumGroups = 1;
  using XRegs = XRegsT<4>;

  // ---- register-decode tensor-core path (mma_kernel.cuh) ----
  // Thread q of a fragment row holds code word q of each half h of the
  // slice (word 4h + q: k = 64h + 16q .. +15).  k16 step ks uses the word of
  // half ks / 4; with sub = ks % 4
  // its two k pairs are fields (2sub, 2sub + 8) and (2sub + 1, 2sub + 9) of
  // that word.  Pair (f, f + 8), f' = f % 4, taken from the word shifted
  // right by 8 when f >= 4: one LOP3 gives 1024 + 4^f' c per half as fp16,
  // one HFMA2 (times 4^-f', minus 1024 4^-f' + 1) gives c - 1, exactly.
  static constexpr int kMmaSharedBytes = 0;
  static constexpr int kMmaRowWords = 2;   // words q of the two 16-byte halves
  static constexpr int kMmaCodebooks = 1;
  static constexpr bool kMmaRowScales = false;
  static constexpr bool kMmaGlu = true;    // the GLU form of the tensor-core kernel
  __device__ static const __half* mma_row_scales(const RunParams&) { return nullptr; }
  static constexpr int kMmaBlockSteps = 8;
  static constexpr int kMmaXWords = 16;  // x[m][64h + 16q .. +15], h = 0, 1
  // One slice per warp, sixteen warps, one CTA per SM for every M: two
  // slices per warp do not fit the activation registers of two blocks, and
  // one geometry for all M keeps the summation order (batch invariance).
  __host__ __device__ static constexpr int mma_spw(int) { return 1; }
  __host__ __device__ static constexpr int mma_ctas(int) { return 1; }
  // tile parity measured 2-5% slower for PQ2_0 (M = 2 and 8): not used
  __host__ __device__ static constexpr bool mma_par(int) { return false; }
  __host__ __device__ static constexpr int mma_stages(int) { return 5; }
  __host__ __device__ static constexpr bool mma_prefetch_x(int nb) { return nb == 1; }  // registers
  template <int NT>
  __device__ static void mma_init_shared(uint8_t*, const uint16_t*, int, int) {}
  __device__ static void mma_load_row(const uint8_t* stage, int slice, int l, int j, int q, uint32_t (&w)[2]) {
    mma_row_words(stage, slice, l, j, q, w);
  }
  struct MmaScales { float d; };  // d of the row's block (the whole slice)
  __device__ static void mma_scales(const uint8_t* stage, int slice, int l, int j, MmaScales& d) {
    const int t = slice * 32 + l;
    d.d = h2f(*reinterpret_cast<const uint16_t*>(stage + kCodeBytes + (t * 4 + j) * 2));
  }
  __device__ static float mma_scale(const MmaScales& d, int) { return d.d; }
  __device__ static uint32_t pq2_pair(uint32_t w, int f) {
    constexpr uint32_t kScale[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};  // 1, 1/4, 1/16, 1/64
    constexpr uint32_t kOff[4] = {0xE401E401u, 0xDC04DC04u, 0xD410D410u, 0xCC40CC40u};    // -1025, -257, -65, -17
    const int fp = f & 3;
    const uint32_t src = f >= 4 ? (w >> 8) : w;
    return hfma2_u32(field_pair(src, 0x00030003u << (2 * fp)), kScale[fp], kOff[fp]);
  }
  __device__ static uint2 mma_frag(const uint32_t (&w)[2], int ks, uint32_t, int) {
    const uint32_t wd = w[ks >> 2];
    const int sub = ks & 3;
    return make_uint2(pq2_pair(wd, 2 * sub), pq2_pair(wd, 2 * sub + 1));
  }
  __device__ static void mma_load_x(uint32_t (&xw)[kMmaXWords], const unsigned short* row, int64_t K,
                                    int64_t kb, int q, bool vec) {
#pragma unroll
    for (int i = 0; i < 4; ++i) ld_x8(xw + 4 * i, row, K, kb + 64 * (i >> 1) + 16 * q + 8 * (i & 1), vec);
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    const uint32_t* X = xw + 8 * (ks >> 2);  // (x0,x1) .. (x14,x15) of the word's 16 k
    const int sub = ks & 3;
    return make_uint2(prmt(X[sub], X[sub + 4], 0x5410u), prmt(X[sub], X[sub + 4], 0x7632u));
  }

  __host__ __device__ static constexpr int field_pos(int jj) { return jj <= 10 ? 2 * jj : 2 * jj - 12; }

  static constexpr int kCbEntries = 0;
  template <int NT>
  __device__ static void init_shared(uint8_t*, const uint16_t*, int, int) {}

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 4>(xr, p, kt, slice, lane);
  }

  struct XScale { float v[4]; };
  __device__ static void x_scales(XScale& sc, int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sc.v[i] = exp2i(109 - field_pos((4 * lane + i) & 15));
  }

  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[kSumGroups][M], const XRegs& xr,
                                 const XScale& sc, int lane) {
    stage_x_slice<M, 4, kSumGroups>(xs, xsum, xr, lane, sc.v);
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&xsum)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t*, int slice, int half, int lane, uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    constexpr int RP = (M > 12) ? 1 : ((M > 8 && RPW > 2) ? 2 : RPW);
    constexpr bool kLate = RP < RPW;  // see FmtQ4_0::tile_math
    uint4 clo[RP], chi[RP];
    if (!kLate) load_codes32<RP>(stage, j0, t, clo, chi);
    const uint2 sc = *reinterpret_cast<const uint2*>(stage + kCodeBytes + t * 8);
    if (!kLate) release_stage(empty_bar, lane);

    float dr[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const uint32_t sw = (RPW == 4) ? (r < 2 ? sc.x : sc.y) : (half ? sc.y : sc.x);
      dr[r] = h2f((r & 1) ? (sw >> 16) : (sw & 0xffffu));
    }

#pragma unroll
    for (int pass = 0; pass < RPW / RP; ++pass) {
      if (kLate) {
        load_codes32<RP>(stage, j0 + pass * RP, t, clo, chi);
        if (pass == RPW / RP - 1) release_stage(empty_bar, lane);
      }
      // code offset 1: start from -sum(x) (in the 2^-40 scaled domain)
      float2 acc[RP][M];
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = make_float2(xsum[0][m] * (-pow2f(kFieldExp)), 0.f);
      constexpr int UI = (M > 8) ? 1 : (M > 4 ? 2 : 8);
#pragma unroll UI
      for (int i = 0; i < 8; ++i) {
        uint32_t wv[RP], wh[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const int rr = kLate ? r : pass * RP + r;
          wv[r] = word8(clo[rr], chi[rr], i);
          wh[r] = wv[r] >> 12;
        }
#pragma unroll
        for (int ph = 0; ph < 2; ++ph) {
        float2 xv4[4][M];
        load_xpair_run<M, 4>(xs, 8 * i + 4 * ph, xv4);
#pragma unroll
        for (int pq = 0; pq < 4; ++pq) {
          const int pp = 4 * ph + pq;
          const float2 (&xv)[M] = xv4[pq];
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const int f0i = 2 * pp, f1i = 2 * pp + 1;
            const uint32_t f0 = (f0i <= 10 ? wv[r] : wh[r]) & (3u << field_pos(f0i));
            const uint32_t f1 = (f1i <= 10 ? wv[r] : wh[r]) & (3u << field_pos(f1i));
            const float2 w2 = make_float2(u2f(f0), u2f(f1));
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = __ffma2_rn(w2, xv[m], acc[r][m]);
          }
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

// -------------------------------------------- PQ2_0, INT8 activations --
//
// The integer path of "Making a ternary reasoning model fast in vLLM" (the
// section on quantising the activation too): every group of 128
// activations -- one PQ2_0 block's inputs, i.e. one slice of a tile -- is
// scaled to signed INT8, x_i ~ a q_i with
//     a = fl32(max |x_i| / 127),   q_i = clamp(rint(fl32(x_i / a)), -127, 127)
// (IEEE divisions, ties to even; a zero group has a = 0, q = 0), so the inner
// sum over the block's codes is an integer, and floating point is used once
// per block: y += d * (a * sum_i (c_i - 1) q_i).  Lossy by design; the
// weights are the plain PQ2_0 tiles.
//
// Staging puts the group's INT8 codes in the order the code words want:
// lane l holds x at k = 16 (l / 4) + 4 b + (l % 4), b = 0..3, so its four q
// packed into one word form, for code word i = l / 4 (k = 16 i .. 16 i + 15),
// the word Q_s (s = l % 4) whose byte b is q[16 i + 4 b + s].  A code word
// w holds field jj (k = 16 i + jj) at bits 2 jj, so byte b of
//     w & 0x03030303, w & 0x0C0C0C0C, (w >> 4) & 0x03030303, (w >> 4) & 0x0C0C0C0C
// is field 4b, 4 x field 4b+1, field 4b+2, 4 x field 4b+3: four DP4As against
// Q_0 .. Q_3 give sum c q over sixteen weights (the two "times 4" terms in
// their own accumulator, divided by 4 exactly at the end of the block).
// The offset c - 1 is applied with the group's sum of q.

// Warp-collective: the 128 values of one group, four per lane, to INT8.
// Every lane gets the group scale a and the group sum of q.
__device__ __forceinline__ void quant_i8_group(const float (&f)[4], float& a, int (&q)[4], int& qsum) {
  float am = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
  a = __fdiv_rn(am, 127.0f);
  int sum = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    int v = 0;
    if (a != 0.0f) v = min(127, max(-127, __float2int_rn(__fdiv_rn(f[b], a))));
    q[b] = v;
    sum += v;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  qsum = sum;
}

// Position (inside its group of 128) of lane l's b-th activation.
__host__ __device__ constexpr int i8_pos(int lane, int b) { return 16 * (lane >> 2) + 4 * b + (lane & 3); }

struct FmtPQ2I8 {
  static constexpr int kSplitMode = 1;  // the PQ2_0 handle's split (same plan)
  static constexpr int kKW = FmtPQ2::kKW;  // 128: one block, one INT8 group
  static constexpr int kKT = FmtPQ2::kKT;
  static constexpr int kCodeBytes = FmtPQ2::kCodeBytes;
  static constexpr int kTileBytes = FmtPQ2::kTileBytes;
  static constexpr int kCtasPerSm = 2;
  static constexpr bool kTileParity = false;
  __host__ __device__ static constexpr int stages(int) { return 2; }
  static constexpr int kSharedBytes = 0;
  static constexpr float kOutScale = 1.0f;
  static constexpr int kSumGroups = 2;  // [0]: the group's sum of q (exact in fp32), [1]: its scale a
  static constexpr int kCbEntries = 0;
  using XRegs = XRegsT<4>;
  struct XScale {};

  template <int NT>
  __device__ static void init_shared(uint8_t*, const uint16_t*, int, int) {}
  __device__ static void x_scales(XScale&, int) {}

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    const int64_t kbase = static_cast<int64_t>(kt) * kKT + slice * kKW;
    const unsigned short* xb = reinterpret_cast<const unsigned short*>(p.x);
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t k = kbase + i8_pos(lane, b);
        xr.v[m][b] = (k < p.K) ? __ldg(xb + m * p.K + k) : static_cast<unsigned short>(0);
      }
  }

  // xs (per warp): for each m, 32 words Q (128 bytes), word l from lane l.
  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[kSumGroups][M], const XRegs& xr, const XScale&,
                                 int lane) {
    uint32_t* xq = reinterpret_cast<uint32_t*>(xs);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) f[b] = h2f(xr.v[m][b]);
      float a;
      int q[4], qsum;
      quant_i8_group(f, a, q, qsum);
      xq[m * 32 + lane] = (static_cast<uint32_t>(q[0]) & 0xffu) | ((static_cast<uint32_t>(q[1]) & 0xffu) << 8) |
                          ((static_cast<uint32_t>(q[2]) & 0xffu) << 16) | (static_cast<uint32_t>(q[3]) << 24);
      xsum[0][m] = static_cast<float>(qsum);
      xsum[1][m] = a;
    }
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&xsum)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t*, int slice, int half, int lane, uint64_t* empty_bar) {
    static_assert(RPW == kRowsPerLane, "one warp per slice: the lane's four rows");
    // rows per pass: all four up to M = 2; above, two at a time (the codes of
    // the later rows are loaded, and the stage released, in the last pass)
    constexpr int RP = M > 2 ? 2 : RPW;
    const int t = slice * 32 + lane;
    const uint2 sc = *reinterpret_cast<const uint2*>(stage + kCodeBytes + t * 8);
    const uint8_t* xq = reinterpret_cast<const uint8_t*>(xs);
#pragma unroll
    for (int pass = 0; pass < RPW / RP; ++pass) {
      uint4 clo[RP], chi[RP];
      load_codes32<RP>(stage, pass * RP, t, clo, chi);
      if (pass == RPW / RP - 1) release_stage(empty_bar, lane);
      int lo[RP][M], hi[RP][M];
#pragma unroll
      for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) lo[r][m] = hi[r][m] = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4 Q[M];
#pragma unroll
        for (int m = 0; m < M; ++m) Q[m] = lds128(xq + m * 128 + 16 * i);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const uint32_t w = word8(clo[r], chi[r], i);
          const uint32_t w4 = w >> 4;
          const int c0 = static_cast<int>(w & 0x03030303u), c1 = static_cast<int>(w & 0x0C0C0C0Cu);
          const int c2 = static_cast<int>(w4 & 0x03030303u), c3 = static_cast<int>(w4 & 0x0C0C0C0Cu);
#pragma unroll
          for (int m = 0; m < M; ++m) {
            lo[r][m] = __dp4a(c0, static_cast<int>(Q[m].x), lo[r][m]);
            hi[r][m] = __dp4a(c1, static_cast<int>(Q[m].y), hi[r][m]);
            lo[r][m] = __dp4a(c2, static_cast<int>(Q[m].z), lo[r][m]);
            hi[r][m] = __dp4a(c3, static_cast<int>(Q[m].w), hi[r][m]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const int row = pass * RP + r;
        const uint32_t sw = row < 2 ? sc.x : sc.y;
        const float d = h2f((row & 1) ? (sw >> 16) : (sw & 0xffffu));
        float v[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          // hi is four times an integer, so the shift divides exactly
          const int inner = lo[r][m] + (hi[r][m] >> 2) - static_cast<int>(xsum[0][m]);
          v[m] = __fmul_rn(xsum[1][m], static_cast<float>(inner));
        }
        yacc.add_row(row, d, v);
      }
    }
  }
};

// PQ2_0 on prepared INT8 activations (qgemv_prepare_x_int8, which also
// applies the Hadamard mixing when asked): the codes of each group of 128
// are stored in the staging order (word l of a group is the word lane l
// stages), with the group's scale and code sum beside them, so staging is a
// copy and the quantization runs once per activation vector, not once per
// row tile.  The math is FmtPQ2I8's.
struct FmtPQ2I8P : FmtPQ2I8 {
  struct XRegs {
    uint32_t w[kMaxM];
    float a[kMaxM];
    int qs[kMaxM];
  };

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    const int64_t G = p.K / 128;
    const int64_t g = static_cast<int64_t>(kt) * kSlices + slice;  // the slice's group
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(p.x);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (g < G) {
        xr.w[m] = __ldg(xw + (m * p.K + g * 128) / 4 + lane);
        xr.a[m] = __ldg(p.x_scale + m * G + g);
        xr.qs[m] = __ldg(p.x_qsum + m * G + g);
      } else {  // past the row: no codes
        xr.w[m] = 0u;
        xr.a[m] = 0.f;
        xr.qs[m] = 0;
      }
    }
  }

  template <int M>
  __device__ static void stage_x(float* xs, float (&xsum)[kSumGroups][M], const XRegs& xr, const XScale&,
                                 int lane) {
    uint32_t* xq = reinterpret_cast<uint32_t*>(xs);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      xq[m * 32 + lane] = xr.w[m];
      xsum[0][m] = static_cast<float>(xr.qs[m]);
      xsum[1][m] = xr.a[m];
    }
  }
};

// ------------------------------- PQ2_0 integer path on the tensor cores --
//
// The integer path for several activation rows: PQ2_0 tiles and decode as
// FmtPQ2 (A = code - 1, exact fp16), and as B the prepared INT8 activations
// (qgemv_prepare_x_int8's layout) converted to fp16 in registers -- every
// INT8 value is an exact fp16 -- so the f16 MMA's fp32 block sum is the
// exact integer sum of (code - 1) times the INT8 codes (at most 2 * 127 *
// 128 in magnitude, far below 2^24).  The block (one slice, one INT8 group)
// then adds d * (a * inner) in fp32, the CUDA-core integer path's
// operations.  The f16 MMA rather than the INT8 one: this part's INT8
// tensor rate is far below its f16 rate.
//   Activations: thread q's k16 step 4h + sub needs, of its column's
//   inputs, k0 + {2sub, 2sub + 8} and k0 + {2sub + 1, 2sub + 9} with
//   k0 = 64h + 16q (FmtPQ2's fragment order).  The prepared group holds
//   input 16i + s + 4b at byte 16i + 4s + b, so the 16 bytes of word
//   i = 4h + q of the slice hold all of them: byte pairs (0, 2) and (4, 6)
//   for sub = 0, (8, 10) and (12, 14) for 1, (1, 3) and (5, 7) for 2,
//   (9, 11) and (13, 15) for 3.  A pair becomes fp16 with one PRMT (the
//   bytes, xor 0x80, under an exponent byte 0x64: 1024 + 128 + q) and one
//   HADD2 (- 1152).
struct FmtPQ2Q8 : FmtPQ2 {
  static constexpr bool kMmaXCodes = true;  // B from INT8 codes, a per-group column scale
  static constexpr int kMmaXWords = 10;     // the two 16-byte words of the halves, then a of the two D columns
  __host__ __device__ static constexpr bool mma_prefetch_x(int nb) { return nb == 1; }
  // Codes of prepared row mb (B column gi of the block) for the slice at kb
  // (words q and 4 + q of the group, 16 bytes each), and the group's scale
  // for D columns md and md + 1; zeros past M and K.
  __device__ static void mma_load_x_q(uint32_t (&xw)[kMmaXWords], const RunParams& p, int M, int mb, int md,
                                      int64_t kb, int q, bool vec) {
    const uint8_t* xq = reinterpret_cast<const uint8_t*>(p.x);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (mb < M && kb < p.K) {
        const uint8_t* src = xq + mb * p.K + kb + 64 * h + 16 * q;
        if (vec) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
          xw[4 * h] = v.x; xw[4 * h + 1] = v.y; xw[4 * h + 2] = v.z; xw[4 * h + 3] = v.w;
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) xw[4 * h + i] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) xw[4 * h + i] = 0u;
      }
    }
    const int64_t G = p.K / 128, g = kb / 128;
#pragma unroll
    for (int c = 0; c < 2; ++c)
      xw[8 + c] = (md + c < M && kb < p.K) ? __float_as_uint(__ldg(p.x_scale + (md + c) * G + g)) : 0u;
  }
  // the fp16 pair of signed bytes lo, hi of w (PRMT selector sel)
  __device__ static uint32_t i8_pair(uint32_t w, uint32_t sel) {
    const uint32_t t = prmt(w ^ 0x80808080u, 0x64646464u, sel);
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0xE480E480u));  // - 1152
    return r;
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    const uint32_t* W = xw + 4 * (ks >> 2);
    const int sub = ks & 3;
    const uint32_t sel = (sub & 2) ? 0x4341u : 0x4240u;  // bytes (1, 3) or (0, 2)
    const int w0 = (sub & 1) ? 2 : 0;                     // words (0, 1) or (2, 3)
    return make_uint2(i8_pair(W[w0], sel), i8_pair(W[w0 + 1], sel));
  }
  __device__ static float mma_col_scale(const uint32_t (&xw)[kMmaXWords], int c) { return __uint_as_float(xw[8 + c]); }
};

}  // namespace qgemv

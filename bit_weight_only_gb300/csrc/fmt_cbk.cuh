// fmt_cbk.cuh -- scalar codebook formats: CBK4 (4-bit index into 16 fp16
// centroids) and CBK8 (8-bit index into 256 fp16 centroids), one codebook
// per matrix ("Trapetum benchmarks", sections "Kernel microbenchmarks" and
// "Model-level results"; the 8-bit table is the LM head's).
//
// Decode: a table lookup in shared memory per index byte.  The table is
// replicated once per lane (entry e of lane l at byte e*256 + l*4), so the 32
// lanes of a warp always hit 32 different banks whatever their indices.  The
// table sits on a 64 KB boundary of the shared window, so the whole shared
// address of an entry is one PRMT of the index byte (-> bits 8..15) with the
// lane's key (table >> 16 -> bits 16..23, lane*4 -> bits 0..7).
//   CBK4: one byte = two indices (k even in the low nibble, k odd in the
//         high nibble); the entry is the fp16 pair (c[lo], c[hi]), and the
//         products with the fp16 activations accumulate in fp32 with the
//         mixed-precision FMA (f16 x f16 + f32; the product is exact).
//   CBK8: one byte = one index; the entry is c[idx] as fp32 and pairs of k
//         accumulate with FFMA2 against fp32 activation pairs.
#pragma once

#include "gemv_kernel.cuh"
#include "mma_kernel.cuh"

namespace qgemv {

constexpr int kLutBytes = 256 * 256;  // 256 entries x 64 four-byte slots

// Key of the lane's table entries for lut_addr: the table (on a 64 KB
// boundary of the shared window) >> 16 in byte 2, lane * 4 in byte 0.
__device__ __forceinline__ uint32_t lut_key_of(const uint8_t* lut, int lane) {
  return smem_u32(lut) | (static_cast<uint32_t>(lane) << 2);
}

// acc[0] += a.lo * b.lo, acc[1] += a.hi * b.hi  (f16 x f16 products, exact;
// f32 accumulation)
__device__ __forceinline__ void fma_f16x2_f32x2(uint32_t a2, uint32_t b2, float (&acc)[2]) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc[0]), "+f"(acc[1])
      : "r"(a2), "r"(b2));
}

// ------------------------------------------------------------------ CBK4 --
//
// Tile: 128 rows x 512 k.  Slice s <-> k 64s..64s+63, lane slot t = 32s + l
// <-> rows 4l..4l+3.  Codes [j][h][t][16 B]: the 32 canonical index bytes of
// row 4l+j for the slice, 16 per half h (byte b = k pair b: low nibble
// k = 2b, high nibble k = 2b+1).  Activations are staged as fp16 pairs: xs
// word (q * MP + m) = (x[2q][m], x[2q+1][m]).
struct FmtCBK4 {
  static constexpr int kKW = 64;
  static constexpr int kKT = kKW * kSlices;                              // 512
  static constexpr int kTileBytes = kLaneSlots * kRowsPerLane * 32;      // 32768
  static constexpr int kCtasPerSm = 1;  // the 64 KB table fits once per SM
  static constexpr bool kTileParity = true;  // so the two warps of a slice take alternate tiles
  __host__ __device__ static constexpr int stages(int M) { return M <= 4 ? 4 : 2; }
  static constexpr int kSharedBytes = kLutBytes;
  static constexpr int kCbEntries = 16;
  static constexpr int kSplitMode = 1;      // front-loaded stream-K split
  static constexpr bool kGluTables = true;  // GLU: the up table in each entry row's second half
  static constexpr bool kMmaGlu = true;     // the GLU form of the tensor-core kernel
  static constexpr float kOutScale = 1.0f;
  static constexpr int kSumGroups = 1;  // unused: codebook values carry no offset
  using XRegs = XRegsT<2>;

  // Warp w writes entries w, w + NT/32, ...; its 32 lanes write one entry's
  // 32 lane copies (32 consecutive words: no bank conflict).  The 16
  // centroids are read once per lane and passed around with shuffles.
  template <int NT>
  __device__ static void init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    constexpr int W = NT / 32;
    const uint32_t mine = cb[lane & 15];
#pragma unroll 4
    for (int e = warp; e < 256; e += W) {
      const uint32_t lo = __shfl_sync(0xffffffffu, mine, e & 15);
      const uint32_t hi = __shfl_sync(0xffffffffu, mine, e >> 4);
      *reinterpret_cast<uint32_t*>(lut + e * 256 + lane * 4) = lo | (hi << 16);
    }
  }

  // ---- register-decode tensor-core path (mma_kernel.cuh) ----
  // Thread q of a fragment row holds index word q of each half h of the
  // row's slice chunk (k = 32h + 8q .. +7); k16 step ks takes bytes 2(ks%2)
  // and 2(ks%2)+1 of word ks/2, i.e. k pairs (32h + 8q + 4(ks%2), +1) and
  // (.. + 2, +3) with h = ks/2, each one table read.
  static constexpr int kMmaSharedBytes = kLutBytes;
  // entry address bits of the lane: table >> 16 in byte 2, lane * 4 in byte 0
  __device__ static uint32_t mma_lut_key(uint32_t table, int lane) {
    return (table & 0xFFFF0000u) | (static_cast<uint32_t>(lane) << 2);
  }
  static constexpr int kMmaRowWords = 2;   // words q of the two 16-byte halves
  static constexpr int kMmaCodebooks = 1;
  static constexpr bool kMmaRowScales = false;
  __device__ static const __half* mma_row_scales(const RunParams&) { return nullptr; }
  static constexpr int kMmaBlockSteps = 0;
  struct MmaScales {};  // no block scale
  static constexpr int kMmaXWords = 8;  // x[m][32h + 8q .. +7], h = 0, 1
  // one slice per warp, sixteen warps per CTA; the 64 KB table fits once per SM
  __host__ __device__ static constexpr int mma_spw(int) { return 1; }
  __host__ __device__ static constexpr int mma_ctas(int) { return 1; }
  // one activation block: tile parity (two halves of eight warps, alternate tiles)
  __host__ __device__ static constexpr bool mma_par(int nb) { return nb == 1; }
  __host__ __device__ static constexpr int mma_stages(int nb) { return nb == 1 ? 4 : 3; }
  __host__ __device__ static constexpr bool mma_prefetch_x(int) { return true; }
  template <int NT>
  __device__ static void mma_init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    init_shared<NT>(lut, cb, warp, lane);
  }
  __device__ static void mma_load_row(const uint8_t* stage, int slice, int l, int j, int q, uint32_t (&w)[2]) {
    mma_row_words(stage, slice, l, j, q, w);
  }
  __device__ static uint2 mma_frag(const uint32_t (&w)[2], int ks, uint32_t lut_key, int) {
    const uint32_t wd = w[ks >> 1];
    const int b = 2 * (ks & 1);
    return make_uint2(lds32_at(lut_addr(wd, lut_key, b)), lds32_at(lut_addr(wd, lut_key, b + 1)));
  }
  __device__ static void mma_load_x(uint32_t (&xw)[kMmaXWords], const unsigned short* row, int64_t K,
                                    int64_t kb, int q, bool vec) {
    ld_x8(xw, row, K, kb + 8 * q, vec);
    ld_x8(xw + 4, row, K, kb + 32 + 8 * q, vec);
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    return make_uint2(xw[2 * ks], xw[2 * ks + 1]);
  }

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 2>(xr, p, kt, slice, lane);
  }

  struct XScale {};
  __device__ static void x_scales(XScale&, int) {}

  // fp16 pairs, unscaled: lane l holds k pair l of the slice
  template <int M>
  __device__ static void stage_x(float* xs, float (&)[kSumGroups][M], const XRegs& xr,
                                 const XScale&, int lane) {
    constexpr int MP = mpad(M);
    uint32_t* xw = reinterpret_cast<uint32_t*>(xs);
#pragma unroll
    for (int m = 0; m < MP; ++m)
      xw[lane * MP + m] = m < M ? (static_cast<uint32_t>(xr.v[m][0]) |
                                   (static_cast<uint32_t>(xr.v[m][1]) << 16)) : 0u;
  }

  template <int R>
  __device__ static void load_codes32(const uint8_t* stage, int j0, int t, uint4 (&lo)[R],
                                      uint4 (&hi)[R]) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      lo[j] = lds128(stage + (((j0 + j) * 2 + 0) * kLaneSlots + t) * 16);
      hi[j] = lds128(stage + (((j0 + j) * 2 + 1) * kLaneSlots + t) * 16);
    }
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t* lut, int slice, int half, int lane,
                                   uint64_t* empty_bar) {
    constexpr int MP = mpad(M);
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    uint4 clo[RPW], chi[RPW];
    load_codes32<RPW>(stage, j0, t, clo, chi);
    release_stage(empty_bar, lane);
    const uint32_t key = lut_key_of(lut, lane);
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs);

    // two accumulators per (row, m): even k and odd k, two independent chains
    float acc[RPW][M][2];
#pragma unroll
    for (int j = 0; j < RPW; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[j][m][0] = acc[j][m][1] = 0.f;
    constexpr int UI = (M > 8) ? 1 : (M > 4 ? 2 : 8);
#pragma unroll UI
    for (int i = 0; i < 8; ++i) {     // word i: k pairs 4i..4i+3
      uint4 x4 = make_uint4(0, 0, 0, 0);
      if constexpr (M == 1) x4 = *reinterpret_cast<const uint4*>(xw + 4 * i);
#pragma unroll
      for (int bp = 0; bp < 4; ++bp) {
        const int q = 4 * i + bp;
        uint32_t xp[M];
        if constexpr (M == 1) {
          xp[0] = word_of(x4, bp);
        } else {
#pragma unroll
          for (int m = 0; m < MP; m += 2) {
            const uint2 v = *reinterpret_cast<const uint2*>(xw + q * MP + m);
            if (m < M) xp[m] = v.x;
            if (m + 1 < M) xp[m + 1] = v.y;
          }
        }
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
          const uint32_t wv = i < 4 ? word_of(clo[j], i) : word_of(chi[j], i - 4);
          const uint32_t c2 = lds32_at(lut_addr(wv, key, bp));
#pragma unroll
          for (int m = 0; m < M; ++m) fma_f16x2_f32x2(c2, xp[m], acc[j][m]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      float a[M];
#pragma unroll
      for (int m = 0; m < M; ++m) a[m] = acc[j][m][0] + acc[j][m][1];
      yacc.add_row(j, 1.0f, a);
    }
  }
};

// ------------------------------------------------------------------ CBK8 --
//
// Tile: 128 rows x 256 k.  Slice s <-> k 32s..32s+31, lane slot t = 32s + l
// <-> rows 4l..4l+3.  Codes [j][h][t][16 B]: the 32 canonical index bytes of
// row 4l+j for the slice.  Activations are staged as fp32 pairs
// (x[2q][m], x[2q+1][m]).
struct FmtCBK8 {
  static constexpr int kKW = 32;
  static constexpr int kKT = kKW * kSlices;                              // 256
  static constexpr int kTileBytes = kLaneSlots * kRowsPerLane * 32;      // 32768
  static constexpr int kCtasPerSm = 1;  // the 64 KB table fits once per SM
  static constexpr bool kTileParity = true;  // so the two warps of a slice take alternate tiles
  __host__ __device__ static constexpr int stages(int M) { return M <= 4 ? 4 : 2; }
  static constexpr int kCbEntries = 256;
  static constexpr int kSplitMode = 1;      // front-loaded stream-K split
  static constexpr bool kGluTables = true;  // GLU: the up table in each entry row's second half
  static constexpr bool kMmaGlu = true;     // the GLU form of the tensor-core kernel
  static constexpr int kSharedBytes = kLutBytes;
  static constexpr float kOutScale = 1.0f;
  static constexpr int kSumGroups = 1;  // unused
  using XRegs = XRegsT<1>;

  // As for CBK4: warp w writes entries w + (NT/32)*j, one conflict-free row
  // of 32 lane copies each; lane l first reads centroids 32*i + l.
  template <int NT>
  __device__ static void init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    constexpr int W = NT / 32;
    float reg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) reg[i] = h2f(cb[32 * i + lane]);
#pragma unroll
    for (int j = 0; j < 256 / W; ++j) {
      const int e = warp + W * j;  // (W * j) >> 5 == e >> 5 since W divides 32
      const float v = __shfl_sync(0xffffffffu, reg[(W * j) >> 5], e & 31);
      *reinterpret_cast<float*>(lut + e * 256 + lane * 4) = v;
    }
  }

  // ---- register-decode tensor-core path (mma_kernel.cuh) ----
  // The table holds c[e] as fp16 (low half of the entry).  Thread q of a
  // fragment row holds index word q of each half h of the slice chunk (k =
  // 16h + 4q .. +3); k16 step ks takes word ks: k pairs (16ks + 4q, +1) and
  // (16ks + 4q + 2, +3).
  static constexpr int kMmaSharedBytes = kLutBytes;
  // entry address bits of the lane: table >> 16 in byte 2, lane * 4 in byte 0
  __device__ static uint32_t mma_lut_key(uint32_t table, int lane) {
    return (table & 0xFFFF0000u) | (static_cast<uint32_t>(lane) << 2);
  }
  static constexpr int kMmaRowWords = 2;   // words q of the two 16-byte halves
  static constexpr int kMmaCodebooks = 1;
  static constexpr bool kMmaRowScales = false;
  __device__ static const __half* mma_row_scales(const RunParams&) { return nullptr; }
  static constexpr int kMmaBlockSteps = 0;
  struct MmaScales {};  // no block scale
  static constexpr int kMmaXWords = 4;  // x[m][16h + 4q .. +3], h = 0, 1
  // one slice per warp, sixteen warps per CTA; the 64 KB table fits once per SM
  __host__ __device__ static constexpr int mma_spw(int) { return 1; }
  __host__ __device__ static constexpr int mma_ctas(int) { return 1; }
  // one activation block: tile parity (two halves of eight warps, alternate tiles)
  __host__ __device__ static constexpr bool mma_par(int nb) { return nb == 1; }
  __host__ __device__ static constexpr int mma_stages(int nb) { return nb == 1 ? 4 : 3; }
  __host__ __device__ static constexpr bool mma_prefetch_x(int) { return true; }
  template <int NT>
  __device__ static void mma_init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    constexpr int W = NT / 32;
    uint32_t reg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) reg[i] = cb[32 * i + lane];
#pragma unroll
    for (int j = 0; j < 256 / W; ++j) {
      const int e = warp + W * j;  // (W * j) >> 5 == e >> 5 since W divides 32
      const uint32_t v = __shfl_sync(0xffffffffu, reg[(W * j) >> 5], e & 31);
      *reinterpret_cast<uint32_t*>(lut + e * 256 + lane * 4) = v;
    }
  }
  __device__ static void mma_load_row(const uint8_t* stage, int slice, int l, int j, int q, uint32_t (&w)[2]) {
    mma_row_words(stage, slice, l, j, q, w);
  }
  __device__ static uint2 mma_frag(const uint32_t (&w)[2], int ks, uint32_t lut_key, int) {
    const uint32_t wd = w[ks];
    const uint32_t c0 = lds32_at(lut_addr(wd, lut_key, 0)), c1 = lds32_at(lut_addr(wd, lut_key, 1));
    const uint32_t c2 = lds32_at(lut_addr(wd, lut_key, 2)), c3 = lds32_at(lut_addr(wd, lut_key, 3));
    return make_uint2(prmt(c0, c1, 0x5410u), prmt(c2, c3, 0x5410u));
  }
  __device__ static void mma_load_x(uint32_t (&xw)[kMmaXWords], const unsigned short* row, int64_t K,
                                    int64_t kb, int q, bool vec) {
    ld_x4(xw, row, K, kb + 4 * q, vec);
    ld_x4(xw + 2, row, K, kb + 16 + 4 * q, vec);
  }
  __device__ static uint2 mma_bfrag(const uint32_t (&xw)[kMmaXWords], int ks) {
    return make_uint2(xw[2 * ks], xw[2 * ks + 1]);
  }

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 1>(xr, p, kt, slice, lane);
  }

  struct XScale {};
  __device__ static void x_scales(XScale&, int) {}

  template <int M>
  __device__ static void stage_x(float* xs, float (&)[kSumGroups][M], const XRegs& xr,
                                 const XScale&, int lane) {
    constexpr int MP = mpad(M);
#pragma unroll
    for (int m = 0; m < MP; ++m)
      xs[((lane >> 1) * MP + m) * 2 + (lane & 1)] = m < M ? h2f(xr.v[m][0]) : 0.f;
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t* lut, int slice, int half, int lane,
                                   uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    uint4 clo[RPW], chi[RPW];
    FmtCBK4::load_codes32<RPW>(stage, j0, t, clo, chi);
    release_stage(empty_bar, lane);
    const uint32_t key = lut_key_of(lut, lane);

    float2 acc[RPW][M];
#pragma unroll
    for (int j = 0; j < RPW; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[j][m] = make_float2(0.f, 0.f);
    constexpr int UI = (M > 8) ? 1 : (M > 4 ? 2 : 8);
#pragma unroll UI
    for (int i = 0; i < 8; ++i) {       // word i: k = 4i..4i+3 -> pairs 2i, 2i+1
      // both pairs of the word at once for M == 1 (one 128-bit load)
      float2 xv2[2][M];
      if constexpr (M == 1) load_xpair_run<M, 2>(xs, 2 * i, xv2);
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if constexpr (M > 1) load_xpairs<M>(xs, 2 * i + pp, xv2[pp]);
        const float2 (&xv)[M] = xv2[pp];
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
          const uint32_t wv = i < 4 ? word_of(clo[j], i) : word_of(chi[j], i - 4);
          const float2 w2 = make_float2(__uint_as_float(lds32_at(lut_addr(wv, key, 2 * pp))),
                                        __uint_as_float(lds32_at(lut_addr(wv, key, 2 * pp + 1))));
#pragma unroll
          for (int m = 0; m < M; ++m) acc[j][m] = __ffma2_rn(w2, xv[m], acc[j][m]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      float a[M];
#pragma unroll
      for (int m = 0; m < M; ++m) a[m] = acc[j][m].x + acc[j][m].y;
      yacc.add_row(j, 1.0f, a);
    }
  }
};

// ------------------------------------------------ CBK4, per-row codebooks --
//
// The pages' own 4-bit files ("Trapetum benchmarks", "Model-level results")
// carry one 16-centroid codebook per output row, in fp32.  Same tiles and
// indices as CBK4; the codebooks of a row tile (128 rows x 16 fp32, 8 KB)
// live in shared memory as T[j][c][l] = centroid c of row 4l + j (byte
// j*2048 + c*128 + l*4 of the 64 KB-aligned table region), so lane l's
// lookups always hit bank l whatever the indices.  A row tile's table is
// built when the CTA starts it (the stacked-handle machinery of wstream_kernel,
// with one segment per row tile).  The entry is fp32, so each weight is one
// lookup (the address: the index nibble shifted to bits 7..10 OR the lane's
// row base) and the products with fp32 activation pairs accumulate with
// FFMA2.  Tile parity as CBK4 (sixteen warps, alternate tiles).
struct FmtCBK4R {
  static constexpr int kKW = 64;
  static constexpr int kKT = kKW * kSlices;                              // 512
  static constexpr int kTileBytes = kLaneSlots * kRowsPerLane * 32;      // 32768
  static constexpr int kCtasPerSm = 1;
  static constexpr bool kTileParity = true;
  __host__ __device__ static constexpr int stages(int M) { return M <= 4 ? 4 : 2; }
  static constexpr int kSharedBytes = kLutBytes;    // the table region (8 KB of it used)
  static constexpr int kCbEntries = kTileRows * 16 * 2;  // fp16-sized units of a row tile's codebooks (8 KB)
  static constexpr int kSplitMode = 1;                   // front-loaded stream-K split
  static constexpr float kOutScale = 1.0f;
  static constexpr int kSumGroups = 1;  // unused
  using XRegs = XRegsT<2>;
  static_assert(kKT == FmtCBK4::kKT && kTileBytes == FmtCBK4::kTileBytes, "the CBK4 tiles");

  // cb: the row tile's codebooks, fp32 [128 rows][16]; entry e of the
  // table (word e) is T[j = e / 512][c = (e / 32) % 16][l = e % 32].
  template <int NT>
  __device__ static void init_shared(uint8_t* lut, const uint16_t* cb, int warp, int lane) {
    const float* cbf = reinterpret_cast<const float*>(cb);
    float* T = reinterpret_cast<float*>(lut);
    for (int e = warp * 32 + lane; e < kTileRows * 16; e += NT) {
      const int l = e & 31, c = (e >> 5) & 15, j = e >> 9;
      T[e] = __ldg(cbf + (kRowsPerLane * l + j) * 16 + c);
    }
  }

  template <int M>
  __device__ static void load_x(XRegs& xr, const RunParams& p, int kt, int slice, int lane) {
    load_x_slice<kKW, M, 2>(xr, p, kt, slice, lane);
  }

  struct XScale {};
  __device__ static void x_scales(XScale&, int) {}

  // fp32 pairs: lane l holds k pair l of the slice
  template <int M>
  __device__ static void stage_x(float* xs, float (&)[kSumGroups][M], const XRegs& xr, const XScale&,
                                 int lane) {
    constexpr int MP = mpad(M);
#pragma unroll
    for (int m = 0; m < MP; ++m)
      *reinterpret_cast<float2*>(xs + (lane * MP + m) * 2) =
          m < M ? make_float2(h2f(xr.v[m][0]), h2f(xr.v[m][1])) : make_float2(0.f, 0.f);
  }

  // Byte offset of the centroid of nibble n (0..7) of w in its row's table
  // column: the index times 128, at bits 7..10.
  template <int n>
  __device__ static uint32_t nib_off(uint32_t w) {
    if constexpr (4 * n >= 7) return (w >> (4 * n - 7)) & 0x780u;
    else return (w << (7 - 4 * n)) & 0x780u;
  }

  template <int M, int RPW>
  __device__ static void tile_math(const uint8_t* stage, const float* xs,
                                   const float (&)[kSumGroups][M], RowAcc<M, RPW>& yacc,
                                   uint8_t* lut, int slice, int half, int lane,
                                   uint64_t* empty_bar) {
    const int t = slice * 32 + lane;
    const int j0 = half * RPW;
    uint4 clo[RPW], chi[RPW];
    FmtCBK4::load_codes32<RPW>(stage, j0, t, clo, chi);
    release_stage(empty_bar, lane);
    // the table is 64 KB-aligned: bits 7..10 of every row base are free
    const uint32_t tbase = smem_u32(lut) + static_cast<uint32_t>(lane) * 4;

    float2 acc[RPW][M];
#pragma unroll
    for (int j = 0; j < RPW; ++j)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[j][m] = make_float2(0.f, 0.f);
    constexpr int UI = (M > 1) ? 2 : 8;
#pragma unroll UI
    for (int i = 0; i < 8; ++i) {  // word i: k pairs 4i..4i+3 (byte bp: k = 2(4i+bp), +1)
      float2 xv4[4][M];
      load_xpair_run<M, 4>(xs, 4 * i, xv4);
#pragma unroll
      for (int j = 0; j < RPW; ++j) {
        const uint32_t wv = i < 4 ? word_of(clo[j], i) : word_of(chi[j], i - 4);
        const uint32_t base = tbase + static_cast<uint32_t>(j0 + j) * 2048u;
        float2 w2[4];
        w2[0] = make_float2(__uint_as_float(lds32_at(base | nib_off<0>(wv))),
                            __uint_as_float(lds32_at(base | nib_off<1>(wv))));
        w2[1] = make_float2(__uint_as_float(lds32_at(base | nib_off<2>(wv))),
                            __uint_as_float(lds32_at(base | nib_off<3>(wv))));
        w2[2] = make_float2(__uint_as_float(lds32_at(base | nib_off<4>(wv))),
                            __uint_as_float(lds32_at(base | nib_off<5>(wv))));
        w2[3] = make_float2(__uint_as_float(lds32_at(base | nib_off<6>(wv))),
                            __uint_as_float(lds32_at(base | nib_off<7>(wv))));
#pragma unroll
        for (int bp = 0; bp < 4; ++bp)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[j][m] = __ffma2_rn(w2[bp], xv4[bp][m], acc[j][m]);
      }
    }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      float a[M];
#pragma unroll
      for (int m = 0; m < M; ++m) a[m] = acc[j][m].x + acc[j][m].y;
      yacc.add_row(j, 1.0f, a);
    }
  }
};

}  // namespace qgemv

namespace qgemv {
namespace cbk {

// Prepared code chunk (tile, j, h, t) <- 16 of the 32 canonical index bytes
// of row rt*128 + 4l + j covering the slice (half h); bytes past the row are 0.
template <class F, int kBitsPerIndex>
__global__ void prepare_kernel(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKT,
                               int64_t nchunks, uint8_t* __restrict__ tiles) {
  const int64_t row_bytes = K * kBitsPerIndex / 8;
  constexpr int kChunks = kRowsPerLane * 2 * kLaneSlots;
  for (int64_t ci = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; ci < nchunks;
       ci += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = ci / kChunks;
    const int rem = static_cast<int>(ci % kChunks);
    const int jh = rem / kLaneSlots, t = rem % kLaneSlots;
    const int j = jh / 2, h = jh % 2;
    const int cw = t / 32, lane = t % 32;
    const int64_t n = (tile / nKT) * kTileRows + kRowsPerLane * lane + j;
    const int64_t b0 = ((tile % nKT) * F::kKT + cw * F::kKW) * kBitsPerIndex / 8 + 16 * h;
    uint32_t w[4] = {0, 0, 0, 0};
    if (n < N) {
      for (int i = 0; i < 16; ++i) {
        const int64_t b = b0 + i;
        if (b < row_bytes) w[i / 4] |= static_cast<uint32_t>(canon[n * row_bytes + b]) << (8 * (i % 4));
      }
    }
    *reinterpret_cast<uint4*>(tiles + tile * F::kTileBytes + (jh * kLaneSlots + t) * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Exact decode (codebook entry of each index) from the prepared tiles; cb
// holds one codebook (cb_stride 0) or one copy per row tile (cb_stride =
// entries, stacked handles); up_off: offset of the codebook of rows 64..127
// of every tile (the up rows of a GLU handle), else 0.
template <class F, int kBitsPerIndex>
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, const uint16_t* __restrict__ cb,
                               int64_t cb_stride, int64_t up_off, int64_t N, int64_t K, int nKT,
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
    const int byte_in_row = el * kBitsPerIndex / 8;  // 0..31
    const int h = byte_in_row / 16;
    const uint8_t byte = tiles[tile * F::kTileBytes + ((j * 2 + h) * kLaneSlots + cw * 32 + lane) * 16 +
                               byte_in_row % 16];
    const int idx = kBitsPerIndex == 8 ? byte : ((el & 1) ? (byte >> 4) : (byte & 15));
    w[e] = h2f(cb[(n / kTileRows) * cb_stride + (r >= kTileRows / 2 ? up_off : 0) + idx]);
  }
}

// aux[rt][e] = codebook seg_of_rt[rt] entry e: one copy per row tile.
template <int E>
__global__ void expand_codebooks_kernel(const uint16_t* __restrict__ cbs, const int32_t* __restrict__ seg_of_rt,
                                        int64_t nRT, uint16_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nRT * E;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = cbs[static_cast<int64_t>(seg_of_rt[i / E]) * E + i % E];
}

inline int grid_for(int64_t items, int threads) {
  const int64_t g = (items + threads - 1) / threads;
  return static_cast<int>(g < 1 ? 1 : (g > 65536 ? 65536 : g));
}

}  // namespace cbk
}  // namespace qgemv

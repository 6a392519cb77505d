// fmt_aqlm.cu -- AQLM 2x8: two additive 256-entry codebooks of 8-vectors.
//
// Decoded weight ("Trapetum benchmarks", sections on additive vector
// quantization and the 2-bit 70B model): a row n is cut into groups of 8
// consecutive weights; group g is the sum of one 8-vector from each of two
// fp16 codebooks C0, C1 (256 x 8 each), picked by two uint8 codes, and the
// summed vector is multiplied by the row's fp16 scale s_n:
//
//     w[n][8g + j] = s_n * (C0[code0(n, g)][j] + C1[code1(n, g)][j]).
//
// GEMV by per-group tables (the pages' "LUT per group"): for activation row m
//
//     T_c[g][e] = sum_j C_c[e][j] * x[m][8g + j]        c = 0, 1; e = 0..255
//     y[m][n]   = s_n * sum_g ( T_0[g][code0(n, g)] + T_1[g][code1(n, g)] )
//
// so each code byte costs one table read and one add, and the scale is
// applied once per row.  The tables depend on x only, so one CTA builds them
// once per 128-input chunk and uses them for 2048 rows.
//
// Table layout and banks.  A chunk has 16 groups x 2 codebooks = 32 tables,
// "slot" tau = 2 * group + codebook.  Entry e of slot tau of buffer b lives
// at byte  R0 + e * 256 + b * 128 + tau * 4  of a 64 KB-aligned shared region
// R0: slot tau is always in bank tau.  Lane t, at step i of a row's 32 code
// bytes, reads slot (t + i) mod 32, so the 32 lanes of a read always hit 32
// different banks whatever the codes are.  The prepared code layout stores
// each row's 32 code bytes of a chunk already rotated by its lane: byte i of
// lane t is the code of slot (t + i) mod 32.  One byte permute then forms the
// whole shared address: [slot * 4 | code | R0 >> 16 | 0].
//
// The tables are built on the tensor cores: for a chunk, T^T = X (16 groups x
// 8) * C^T (8 x 256 entries) per codebook, 64 mma.m16n8k8 (f16 in, f32
// accumulate; the products of two fp16 values are exact).  Each warp keeps
// the B fragments of its 4 entry tiles in registers for the whole kernel.
// The n-tiles interleave the two codebooks so that the D fragments of a quad
// cover four different slots, which makes every table store conflict-free.
//
// Work split: row blocks of 2048 rows x chunks of 128 inputs ("units"),
// spread over a persistent grid stream-K style (each CTA a contiguous run of
// units).  Split row blocks are finished after the main loop by all their
// contributors, each summing a slice of rows from polled partial slots in a
// fixed order (finish_rows, gemv_kernel.cuh; deterministic).  Codes stream
// straight from HBM into registers (128-bit loads through an 8-row ring per
// lane); shared memory carries only the tables, whose reads are the binding
// on-chip resource.
//
// M > 1: a pass handles MB <= 2 activation rows (one 64 KB table slab each)
// and a call with M rows makes ceil(M / 2) passes over the codes.
//
// Stacked handles (several projections sharing K, e.g. gate|up): segment s
// has its own codebook pair; segments start on 2048-row blocks, so every
// row block has one pair.  aux = the nseg codebook pairs, the row scales,
// then the segment of every row block (seg_of_rt).  The warps load the B
// fragments of a row block's pair when the tables of its first unit are
// built (only when the segment changes).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "formats.h"
#include "gemv_kernel.cuh"

namespace qgemv {
namespace aqlm {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;       // 512
constexpr int kRPL = 4;                     // output rows per lane
constexpr int kRows = 32 * kWarps * kRPL;   // 2048 rows per row block
constexpr int kKC = 128;                    // inputs per chunk (16 groups)
constexpr int kPos = 32;                    // code bytes per row per chunk
constexpr int kTileBytes = kRows * kPos;    // 65536 bytes per unit
constexpr uint32_t kSlab = 65536;           // one activation row's tables (2 buffers)
constexpr int kMaxMB = 2;                   // activation rows per pass
constexpr int64_t kPartialStride = int64_t(kRows) * kMaxMB;
constexpr int kCodebookBytes = 2 * 256 * 8 * 2;
constexpr int kRing = 2 * kRPL;            // rows of codes per lane in the load ring
constexpr int kPreWait = 3;                // ring rows requested before the grid dependency wait

__host__ __device__ constexpr int smem_bytes_mb(int mb) { return 65536 + mb * 65536; }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

template <uint32_t OFF>
__device__ __forceinline__ float lds_at(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(addr), "n"(OFF));
  return v;
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Issued in program order with the code stream (volatile), so the small
// loads the table build needs are not queued behind the codes.
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// D (16 x 8, f32) = A (16 x 8, f16, row) * B (8 x 8, f16, col).
__device__ __forceinline__ void mma_16x8x8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%7,%7,%7,%7};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(b), "f"(0.f));
}

// Selector of the byte permute of step i (i = 4k + j = 3kk + jj): byte 0 is
// byte jj of the offset word, byte 1 byte j of the code word, byte 2 the
// offset word's region byte and byte 3 that byte's (zero) sign.
__host__ __device__ constexpr uint32_t step_sel(int i) {
  return static_cast<uint32_t>((4 + i % 3) | ((i & 3) << 4) | (7 << 8) | (15 << 12));
}

// One row's 32 code bytes of a chunk, tables in buffer BUF.
template <int MB, int BUF>
__device__ __forceinline__ void lookup_row(const uint4 (&cr)[2], const uint32_t (&L)[11], float2& acc) {
  constexpr uint32_t kOff = BUF * 128;
  const uint32_t w[8] = {cr[0].x, cr[0].y, cr[0].z, cr[0].w, cr[1].x, cr[1].y, cr[1].z, cr[1].w};
#pragma unroll
  for (int i = 0; i < kPos; i += 2) {
    const uint32_t a0 = prmt(w[i >> 2], L[i / 3], step_sel(i));
    const uint32_t a1 = prmt(w[(i + 1) >> 2], L[(i + 1) / 3], step_sel(i + 1));
    if constexpr (MB == 1) {
      acc = __fadd2_rn(acc, make_float2(lds_at<kOff>(a0), lds_at<kOff>(a1)));
    } else {
      acc = __fadd2_rn(acc, make_float2(lds_at<kOff>(a0), lds_at<kOff + kSlab>(a0)));
      acc = __fadd2_rn(acc, make_float2(lds_at<kOff>(a1), lds_at<kOff + kSlab>(a1)));
    }
  }
}

// Codebook pairs before the row scales in aux: one, or (stacked handles)
// one per segment, the last row block's segment being the last segment.
__device__ __forceinline__ int codebook_pairs(const int32_t* seg_of_rb, int64_t nRB) {
  return seg_of_rb != nullptr ? seg_of_rb[nRB - 1] + 1 : 1;
}

// STACKED: a handle with a codebook pair per segment (p.seg_of_rt set); a
// separate instantiation, so that the single-pair kernel carries none of it
// (with the segment checks folded in, 8192 x 28672 measured 18.0 -> 18.4 us).
template <int MB, bool STACKED>
__global__ void __launch_bounds__(kThreads, 1) aqlm_table_kernel(const RunParams p) {
  if (static_cast<int>(blockIdx.x) == p.skip_cta) return;  // test hook (QGEMV_FAULT_SKIP_CTA)
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_sub[2 * kThreads];
  __shared__ __align__(16) CtaPlan s_plan;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int q = lane & 3;     // mma thread-in-group
  const int gi = lane >> 2;   // mma group
  const int hi = q >> 1;
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t u0 = stream_split<0>(c, p.T, G);
  const int64_t u1 = stream_split<0>(c + 1, p.T, G);
  const int64_t nunits = u1 - u0;
  const int nKC = p.nKT;

  // The table region must start on a 64 KB boundary of the shared window.
  const uint32_t base = smem_u32(smem);
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  const uint32_t R0 = (base + 0xFFFFu) & ~0xFFFFu;
  if (R0 + MB * kSlab > base + dyn || (R0 >> 16) > 127u) {
    if (tid == 0) atomicOr(p.err, kErrSmemLayout);
    return;
  }

  fetch_plan(&s_plan, p.plan, c, tid);

  // Offset words: byte jj of L[k] is 4 * slot of step 3k + jj; byte 3 is R0 >> 16.
  uint32_t L[11];
#pragma unroll
  for (int k = 0; k < 11; ++k) {
    uint32_t v = (R0 >> 16) << 24;
#pragma unroll
    for (int jj = 0; jj < 3; ++jj) v |= static_cast<uint32_t>(4 * ((lane + 3 * k + jj) & 31)) << (8 * jj);
    L[k] = v;
  }

  // B fragments of this warp's entry tiles nt = 4 * warp + j.  Column n of a
  // tile is codebook (n >> 1) & 1, entry 4 * nt + 2 * (n >> 2) + (n & 1).
  // Stacked handles: the pair of segment seg (loaded by load_bf).
  const int32_t* seg_of_rb = p.seg_of_rt;
  const uint8_t* aux = static_cast<const uint8_t*>(p.aux);
  uint32_t bf[4];
  int bseg = 0;  // segment whose pair bf holds
  auto load_bf = [&](int seg) {
    const uint16_t* cb = reinterpret_cast<const uint16_t*>(aux + int64_t(seg) * kCodebookBytes);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int nt = 4 * warp + j;
      const int cbi = (gi >> 1) & 1;
      const int e = 4 * nt + 2 * (gi >> 2) + (gi & 1);
      bf[j] = ldg_u32(cb + (cbi * 256 + e) * 8 + 2 * q);
    }
    bseg = seg;
  };
  const __half* scales;
  if constexpr (STACKED) {
    scales = reinterpret_cast<const __half*>(aux + int64_t(codebook_pairs(seg_of_rb, p.T / nKC)) * kCodebookBytes);
    load_bf(nunits > 0 ? seg_of_rb[div_fast(u0, nKC)] : 0);
  } else {
    scales = reinterpret_cast<const __half*>(aux + kCodebookBytes);
    load_bf(0);
  }

  // Table store addresses: D values of this lane are slots 2 * gi + (q & 1)
  // (rows gi) and that + 16 (rows gi + 8), entries eA and eA + 1.
  const uint32_t tauX = 2 * (gi + 8 * hi) + (q & 1);
  const uint32_t tauY = 2 * (gi + 8 * (1 - hi)) + (q & 1);
  const uint32_t eA = 16 * warp + 2 * hi;
  const uint32_t stX = R0 + eA * 256 + tauX * 4;
  const uint32_t stY = R0 + eA * 256 + tauY * 4;

  // Codes stream through a ring of kRing rows per lane (two units): the
  // load of row-step s + kRing - 1 is issued when row-step s is consumed, so
  // about 112 KB per SM stay in flight.
  const uint64_t pol = l2_policy_evict_first();
  const int64_t nsteps = nunits * kRPL;
  auto load_row = [&](uint4 (&cr)[2], int64_t s) {
    const int64_t u = u0 + (s >> 2);
    const int r = static_cast<int>(s & 3);
    const uint8_t* t = p.tiles + u * kTileBytes + (r * 2) * 16 * 512 + warp * 512 + lane * 16;
    cr[0] = ldg_stream(t, pol);
    cr[1] = ldg_stream(t + 16 * 512, pol);
  };
  const int64_t ngroups = p.K / 8;
  auto load_xf = [&](uint32_t (&xf)[MB][2], int kc) {
    const int64_t g0 = static_cast<int64_t>(kc) * 16 + gi;
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      const __half* xm = p.x + m * p.K;
      xf[m][0] = (g0 < ngroups) ? ldg_u32(xm + 8 * g0 + 2 * q) : 0u;
      xf[m][1] = (g0 + 8 < ngroups) ? ldg_u32(xm + 8 * (g0 + 8) + 2 * q) : 0u;
    }
  };
  auto build = [&](const uint32_t (&xf)[MB][2], uint32_t bufoff) {
#pragma unroll
    for (int m = 0; m < MB; ++m) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float d[4];
        mma_16x8x8(d, xf[m][0], xf[m][1], bf[j]);
        const uint32_t o = m * kSlab + bufoff + 1024 * j;
        sts_f32(stX + o, hi ? d[2] : d[0]);
        sts_f32(stY + o, hi ? d[0] : d[2]);
        sts_f32(stX + o + 256, hi ? d[3] : d[1]);
        sts_f32(stY + o + 256, hi ? d[1] : d[3]);
      }
    }
  };

  uint4 ring[kRing][2];
  uint32_t xf[MB][2];
  float2 acc[kRPL];
#pragma unroll
  for (int r = 0; r < kRPL; ++r) acc[r] = make_float2(0.f, 0.f);

  // Row blocks this CTA shares with other CTAs (does not "own"): at most the
  // first and the last of its run.  Their partials are stored in the loop
  // and combined after it, with no fence or atomic inside the loop.
  auto owned = [&](int64_t r) { return r * nKC >= u0 && (r + 1) * nKC <= u1; };

  // Weights are constant: start the code stream before waiting on the
  // previous kernel in the stream.  x is read only after the wait, ahead of
  // the rest of the stream, so the first table build does not queue behind
  // the codes.
#pragma unroll
  for (int k = 0; k < kPreWait; ++k)
    if (k < nsteps) load_row(ring[k], k);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t rb = div_fast(u0, nKC);
  int kc = static_cast<int>(u0 - rb * nKC);
  auto next_kc = [&](int k) { return (k + 1 == nKC) ? 0 : k + 1; };
  if (nunits > 0) load_xf(xf, kc);
#pragma unroll
  for (int k = kPreWait; k < kRing - 1; ++k)
    if (k < nsteps) load_row(ring[k], k);
  if (nunits > 0) {
    build(xf, 0);
    if (nunits > 1) load_xf(xf, next_kc(kc));
  }
  __syncthreads();

  auto epilogue = [&](int64_t rbe) {
    const bool owner = owned(rbe);
    const int side = (rbe * nKC <= u0) ? 0 : 1;
    float* my_part = p.partials + (c * 2 + side) * kPartialStride;
#pragma unroll
    for (int r = 0; r < kRPL; ++r) {
      const int nl = r * 512 + warp * 32 + lane;
      const int64_t n = rbe * kRows + nl;
      float v[MB];
      if constexpr (MB == 1) {
        v[0] = acc[r].x + acc[r].y;
      } else {
        v[0] = acc[r].x;
        v[1] = acc[r].y;
      }
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (owner) {
          if (n < p.N) store_y(p, m * p.N + n, __fmul_rn(__half2float(scales[n]), v[m]));
        } else {
          st_relaxed_f32(my_part + m * kRows + nl, v[m]);
        }
      }
    }
  };

  // One unit: build the next unit's tables in the other buffer, look this
  // unit's rows up (refilling the ring), finish the row block if it ends.
  auto unit = [&](auto buf_tag, int64_t i) {
    constexpr int BUF = decltype(buf_tag)::value;
    const int k1 = next_kc(kc);
    if (i + 1 < nunits) {
      if constexpr (STACKED) {
        if (k1 == 0) {  // the next unit opens row block rb + 1
          const int sn = seg_of_rb[rb + 1];
          if (sn != bseg) load_bf(sn);
        }
      }
      build(xf, (1 - BUF) * 128);
      if (i + 2 < nunits) load_xf(xf, next_kc(k1));
    }
#pragma unroll
    for (int r = 0; r < kRPL; ++r) {
      const int64_t s = i * kRPL + r;
      constexpr int kBase = BUF * kRPL;
      if (s + kRing - 1 < nsteps) load_row(ring[(kBase + r + kRing - 1) % kRing], s + kRing - 1);
      lookup_row<MB, BUF>(ring[kBase + r], L, acc[r]);
    }
    if (k1 == 0 || i + 1 == nunits) {
      epilogue(rb);
#pragma unroll
      for (int r = 0; r < kRPL; ++r) acc[r] = make_float2(0.f, 0.f);
    }
    if (k1 == 0) ++rb;
    kc = k1;
    __syncthreads();
  };

  for (int64_t i = 0; i < nunits; i += 2) {
    unit(std::integral_constant<int, 0>{}, i);
    if (i + 1 < nunits) unit(std::integral_constant<int, 1>{}, i + 1);
  }

  // ---- split row blocks: every contributor finishes a slice of rows ----
  wait_plan();
  finish_all<kRows, MB, kThreads>(p, kPartialStride, s_plan, scales, 1.f, s_sub, tid);
}

// Canonical codes [N][K/8][2] -> prepared units (rotated per lane).
__global__ void prepare_kernel(const uint8_t* __restrict__ canon, int64_t N, int64_t K, int nKC,
                               int64_t nvec, uint8_t* __restrict__ tiles) {
  const int64_t ng = K / 8;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < nvec;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t u = v / (kTileBytes / 16);
    const int w = static_cast<int>(v % (kTileBytes / 16));
    const int lane = w & 31;
    const int warp = (w >> 5) & 15;
    const int rh = w >> 9;
    const int r = rh >> 1, h = rh & 1;
    const int64_t rb = u / nKC;
    const int kc = static_cast<int>(u % nKC);
    const int64_t n = rb * kRows + r * 512 + warp * 32 + lane;
    uint8_t b[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int slot = (lane + 16 * h + j) & 31;
      const int64_t g = int64_t(kc) * 16 + (slot >> 1);
      b[j] = (n < N && g < ng) ? canon[(n * ng + g) * 2 + (slot & 1)] : 0;
    }
    uint4 o;
    o.x = b[0] | (b[1] << 8) | (b[2] << 16) | (uint32_t(b[3]) << 24);
    o.y = b[4] | (b[5] << 8) | (b[6] << 16) | (uint32_t(b[7]) << 24);
    o.z = b[8] | (b[9] << 8) | (b[10] << 16) | (uint32_t(b[11]) << 24);
    o.w = b[12] | (b[13] << 8) | (b[14] << 16) | (uint32_t(b[15]) << 24);
    reinterpret_cast<uint4*>(tiles)[v] = o;
  }
}

// Decode one group of 8 weights per thread from the prepared layout.  The
// sum and product are exact in fp64 (fp16 operands), so the one rounding to
// fp32 gives the correctly rounded weight.
__global__ void dequant_kernel(const uint8_t* __restrict__ tiles, const uint8_t* __restrict__ aux,
                               const int32_t* __restrict__ seg_of_rb, int64_t N, int64_t K, int nKC,
                               float* __restrict__ w_out) {
  const int64_t ng = K / 8;
  const int64_t nRB = (N + kRows - 1) / kRows;
  const __half* sc = reinterpret_cast<const __half*>(aux + int64_t(codebook_pairs(seg_of_rb, nRB)) * kCodebookBytes);
  for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < N * ng;
       t += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = t / ng;
    const int64_t g = t % ng;
    const int64_t rb = n / kRows;
    const __half* cbk =
        reinterpret_cast<const __half*>(aux + int64_t(seg_of_rb != nullptr ? seg_of_rb[rb] : 0) * kCodebookBytes);
    const int nl = static_cast<int>(n % kRows);
    const int r = nl >> 9, warp = (nl >> 5) & 15, lane = nl & 31;
    const int64_t kc = g / 16;
    const int gg = static_cast<int>(g % 16);
    int code[2];
#pragma unroll
    for (int cbi = 0; cbi < 2; ++cbi) {
      const int i = (2 * gg + cbi - lane) & 31;  // byte i of the lane holds slot (lane + i) mod 32
      const int64_t off = (rb * nKC + kc) * kTileBytes + ((r * 2 + (i >> 4)) * 16 + warp) * 512 +
                          lane * 16 + (i & 15);
      code[cbi] = tiles[off];
    }
    const double s = __half2float(sc[n]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const double c0 = __half2float(cbk[code[0] * 8 + j]);
      const double c1 = __half2float(cbk[(256 + code[1]) * 8 + j]);
      w_out[n * K + 8 * g + j] = static_cast<float>(s * (c0 + c1));
    }
  }
}

int grid_for(int64_t work) {
  const int64_t b = (work + 255) / 256;
  return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

cudaError_t prepare(const PrepareArgs& a, cudaStream_t s) {
  const int64_t nvec = a.nRT * a.nKT * int64_t(kTileBytes / 16);
  prepare_kernel<<<grid_for(nvec), 256, 0, s>>>(a.packed, a.N, a.K, a.nKT, nvec, a.tiles);
  cudaError_t e = cudaGetLastError();
  uint8_t* aux = static_cast<uint8_t*>(a.aux);
  // the codebook pairs (one per segment), then the row scales
  const int64_t cb_bytes = int64_t(kCodebookBytes) * (a.seg_of_rt != nullptr ? a.nseg : 1);
  if (e == cudaSuccess) e = cudaMemcpyAsync(aux, a.codebooks, cb_bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(aux + cb_bytes, a.scales, 2 * a.N, cudaMemcpyDeviceToDevice, s);
  return e;
}

cudaError_t dequant(const uint8_t* tiles, const void* aux, const int32_t* seg_of_rb, int64_t N, int64_t K, int nKT,
                    float* w_out, int, cudaStream_t s) {
  dequant_kernel<<<grid_for(N * (K / 8)), 256, 0, s>>>(tiles, static_cast<const uint8_t*>(aux), seg_of_rb, N, K,
                                                       nKT, w_out);
  return cudaGetLastError();
}

int smem_bytes(int M) { return smem_bytes_mb(M >= 2 ? 2 : 1); }

cudaError_t setup() {
  cudaError_t e = cudaFuncSetAttribute(aqlm_table_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes_mb(1));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(aqlm_table_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes_mb(2));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(aqlm_table_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes_mb(1));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(aqlm_table_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes_mb(2));
  return e;
}

template <int MB>
cudaError_t launch_pass(const RunParams& p, int grid, cudaStream_t s) {
  static_assert(smem_bytes_mb(MB) <= 227 * 1024, "shared memory budget exceeded");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_mb(MB);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.seg_of_rt != nullptr ? cudaLaunchKernelEx(&cfg, aqlm_table_kernel<MB, true>, p)
                                : cudaLaunchKernelEx(&cfg, aqlm_table_kernel<MB, false>, p);
}

// Passes of two activation rows, and one for an odd last row.  The two pass
// kinds round differently, so in batch-invariant mode every row gets a
// one-row pass of its own.
cudaError_t launch(int M, const RunParams& p, const LaunchGeom& g, cudaStream_t s, bool batch_invariant) {
  cudaError_t e = cudaSuccess;
  const int grid = g.grid;
  for (int m0 = 0; m0 < M && e == cudaSuccess;) {
    RunParams q = p;
    q.plan = g.plan;
    q.x = p.x + int64_t(m0) * p.K;
    q.y = p.y + int64_t(m0) * p.N;
    q.residual = p.residual != nullptr ? p.residual + int64_t(m0) * p.N : nullptr;
    if (M - m0 >= 2 && !batch_invariant) {
      e = launch_pass<2>(q, grid, s);
      m0 += 2;
    } else {
      e = launch_pass<1>(q, grid, s);
      m0 += 1;
    }
  }
  return e;
}

}  // namespace aqlm

const FormatOps* ops_aqlm() {
  static const FormatOps ops = {
      /*format=*/5, aqlm::kKC, aqlm::kTileBytes, /*aux_bytes=*/aqlm::kCodebookBytes,
      &aqlm::smem_bytes, &aqlm::setup, &aqlm::launch, &aqlm::prepare, &aqlm::dequant,
      /*cb_entries=*/0, /*tile_rows=*/aqlm::kRows, /*partial_stride=*/aqlm::kPartialStride, /*aux_per_row=*/2};
  return &ops;
}

}  // namespace qgemv

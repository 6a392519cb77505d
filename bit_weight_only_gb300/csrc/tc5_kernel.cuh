// tc5_kernel.cuh -- the GEMV on the fifth-generation tensor cores (tcgen05)
// with the weights decoded into tensor memory, for the tile formats (Q4_0,
// PQ2_0, CBK4, CBK8).
//
//   y[m][n] = sum_k x[m][k] * w[n][k]        (1 <= M <= 16)
//
// computed per 128-row tile as D = W_tile . X^T with tcgen05.mma kind::f16
// (M = 128 weight rows, N = 16 activation rows, K = 16, fp32 accumulation):
//
//   * Same prepared tiles, TMA bulk copies, stream-K split, CTA plans and
//     polled split-K fix-up as the other kernels; one CTA per SM.  The
//     sixteenth warp to finish with a stage refills it, so no thread waits
//     for the others to free one.
//   * Four warpgroups of four warps.  Warpgroup G decodes slices 2G and
//     2G + 1 of every tile (a quarter of its k range) for all 128 rows: each
//     thread decodes one weight row -- the row whose codes its lane reads
//     without bank conflicts -- into exact fp16 values and stores them with
//     tcgen05.st into the A operand in tensor memory (its warp's 32 lanes).
//     Nothing decoded goes through shared memory: a decoded weight costs two
//     bytes of tensor-memory store instead of two bytes of shared-memory
//     store plus two of MMA read, which shared memory could not sustain at
//     the weight stream's rate.
//   * The activations of a chunk (64 k, 16 rows, padded with zeros beyond M
//     and K) are staged by the same warpgroup into shared memory in the MMA's
//     K-major layout, permuted within each group of k exactly as the decode
//     orders its fp16 pairs, so every product pairs the right x and w.
//   * Each warp signals an mbarrier when its part of a chunk's A and B is
//     stored; one lane of the warpgroup (a different warp for each chunk, or
//     each block of two chunks) waits for the four, issues the chunk's four
//     MMAs (K = 16 each) and commits them to the chunk's slot barrier, which
//     both frees the chunk's A and B slots and marks its blocks ready.
//   * Blocks: the fp32 accumulator of a block (Q4_0: 32 k, PQ2_0: 128 k, the
//     scale's span; CBK4: 128 k; CBK8: 64 k) is read back with tcgen05.ld by
//     the warpgroup one chunk later (so the MMA latency is hidden) and added
//     to the thread's fp32 row sums times the row's block scale (1 for the
//     codebook formats).  Codes, offsets and centroids are exact fp16, so
//     nothing is rounded before the fp32 sums.
//   * At a row-tile end the four warpgroups' row sums are added in a fixed
//     order and stored to y, or to the stream-K partial slots.
//
// Tensor memory: 512 columns per CTA, 128 per warpgroup: two A slots of 32
// columns (a chunk, 64 k as fp16 pairs) and up to four accumulator slots of
// 16 columns.  Every wait is bounded; on a timeout the kernel records the
// error, skips the remaining math, waits for its own MMAs and copies, frees
// tensor memory and returns.
//
// Measured on GB300 (8192 x 28672): correct at every M, but slower than the
// register-fed mma.sync kernel at every M, so the dispatcher does not use it
// by default (QGEMV_TC5 turns it on).  With at most 16 activation columns an
// MMA covers only 128 x 16 weights: issuing one costs a single thread about
// as long as its warpgroup takes to decode those 2048 weights, and the
// warpgroups spend most of the time waiting for the issuing lane (the
// tensor pipe is busy 4-7% of the time).
#pragma once

#include "fmt_cbk.cuh"
#include "fmt_fields.cuh"
#include "gemv_kernel.cuh"
#include "mma_kernel.cuh"

namespace qgemv {

constexpr int kTc5Threads = 512;     // four warpgroups
constexpr int kTc5ChunkK = 64;       // k per chunk (one A slot, four MMAs)
constexpr int kTc5BSlotBytes = 2048; // activations of one chunk: 4 k16 steps x 512 B
constexpr int kTc5ColsPerWg = 128;   // tensor-memory columns per warpgroup
constexpr int kTc5DCol0 = 64;        // first accumulator column of a warpgroup
// Calls with at least this many activation rows run this kernel by default
// (QGEMV_TC5 overrides it per handle).  0: never -- no M was measured at
// which it beats the mma.sync kernel.
constexpr int kTc5DefaultMinM = 0;

// ---------------------------------------------------------- tcgen05 PTX ----

__device__ __forceinline__ void tmem_alloc_512(uint32_t* dst_smem) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(dst_smem))
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_512(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(taddr) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive columns of the warp's 32 lanes (thread i -> lane base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Load MT (8 or 16) columns; the wait names the registers so that no use
// of them is scheduled before it.
template <int MT>
__device__ __forceinline__ void tmem_ld_wait(uint32_t taddr, uint32_t (&v)[MT]) {
  if constexpr (MT == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15])::"memory");
  } else {
    static_assert(MT == 8, "8 or 16 columns");
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                   "+r"(v[7])::"memory");
  }
}

// D[tmem] (+)= A[tmem] . B[smem]: kind::f16, fp16 A and B, fp32 D, M = 128,
// N = 16, both operands K-major.  Instruction descriptor: D format F32 (bit
// 4), A and B F16 (0), not transposed, N >> 3 at bits 17..22, M >> 4 at bits
// 24..28.
constexpr uint32_t kTc5InstrDesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(kTc5InstrDesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major: 8-row x 16-byte core
// matrices; `lbo` bytes between core matrices along K, `sbo` along N.
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// ------------------------------------------------------ format hooks -------
//
// Tc5<F>: per format
//   kCpw  chunks (64 k) of a warpgroup per tile; chunk c of warpgroup G
//         covers k0(G, c) .. + 63 of the tile.
//   kDpc  accumulator blocks completed per chunk (Q4_0: 2), or
//   kCpd  chunks per block (PQ2_0, CBK4: 2).
//   kXg   activations staged per item: 8 k (one 16-byte B row) or 16 k
//         (two rows, the PQ2_0 pairing (f, f + 8)).
//   decode(stage, c, G, lp, j, key, out, sc): the 32 A columns (fp16 pairs)
//         of chunk c for row 4 lp + j of the lane slot lp of its slice;
//         sc: the scales of the blocks the chunk completes.
//   bperm(lo, hi, out): the B row(s) of an item in the decode's k order.

template <class F>
struct Tc5 {
  static constexpr bool kHas = false;  // no tensor-memory kernel for this format
};

// Q4_0: chunk c = slice 2G + c (two blocks of 32 k).  Code word i (k 8i ..
// 8i + 7) gives the pairs (k, k + 4) for k = 8i .. 8i + 3, so a B row holds
// x0 x4 x1 x5 x2 x6 x3 x7 of its eight k.
template <>
struct Tc5<FmtQ4_0> {
  static constexpr bool kHas = true;
  static constexpr int kStages = 4;
  static constexpr int kCpw = 2, kDpc = 2, kCpd = 1, kXg = 8;
  static constexpr bool kTable = false;
  __device__ static int k0(int G, int c) { return (2 * G + c) * 64; }
  __device__ static void decode(const uint8_t* stage, int c, int G, int lp, int j, uint32_t, uint32_t* out,
                                float (&sc)[2]) {
    const int t = (2 * G + c) * 32 + lp;
    const uint4 lo = lds128(stage + ((j * 2 + 0) * kLaneSlots + t) * 16);
    const uint4 hi = lds128(stage + ((j * 2 + 1) * kLaneSlots + t) * 16);
    const uint32_t d2 = *reinterpret_cast<const uint32_t*>(stage + FmtQ4_0::kCodeBytes + (t * 4 + j) * 4);
    sc[0] = h2f(d2 & 0xFFFFu);
    sc[1] = h2f(d2 >> 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w = word8(lo, hi, i), wh = w >> 8;
      out[4 * i + 0] = hfma2_u32(field_pair(w, 0x000F000Fu), 0x3C003C00u, 0xE408E408u);   // (n0, n4) - 8
      out[4 * i + 1] = hfma2_u32(field_pair(w, 0x00F000F0u), 0x2C002C00u, 0xD480D480u);   // (n1, n5) - 8
      out[4 * i + 2] = hfma2_u32(field_pair(wh, 0x000F000Fu), 0x3C003C00u, 0xE408E408u);  // (n2, n6) - 8
      out[4 * i + 3] = hfma2_u32(field_pair(wh, 0x00F000F0u), 0x2C002C00u, 0xD480D480u);  // (n3, n7) - 8
    }
  }
  __device__ static void bperm(const uint4& x, const uint4&, uint4* out) {
    out[0] = make_uint4(prmt(x.x, x.z, 0x5410u), prmt(x.x, x.z, 0x7632u), prmt(x.y, x.w, 0x5410u),
                        prmt(x.y, x.w, 0x7632u));
  }
};

// PQ2_0: chunk c = half c % 2 of slice 2G + c / 2 (a block is a slice: two
// chunks).  Code word i of the half (k 16i .. 16i + 15) gives the pairs
// (k, k + 8), so the two B rows of a k16 step hold x0 x8 x1 x9 x2 x10 x3 x11
// and x4 x12 .. x7 x15.
template <>
struct Tc5<FmtPQ2> {
  static constexpr bool kHas = true;
  static constexpr int kStages = 4;
  static constexpr int kCpw = 4, kDpc = 1, kCpd = 2, kXg = 16;
  static constexpr bool kTable = false;
  __device__ static int k0(int G, int c) { return (2 * G + (c >> 1)) * 128 + (c & 1) * 64; }
  __device__ static void decode(const uint8_t* stage, int c, int G, int lp, int j, uint32_t, uint32_t* out,
                                float (&sc)[2]) {
    const int t = (2 * G + (c >> 1)) * 32 + lp;
    const uint4 v = lds128(stage + ((j * 2 + (c & 1)) * kLaneSlots + t) * 16);
    sc[0] = h2f(*reinterpret_cast<const uint16_t*>(stage + FmtPQ2::kCodeBytes + (t * 4 + j) * 2));
    sc[1] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = word_of(v, i);
#pragma unroll
      for (int f = 0; f < 8; ++f) out[8 * i + f] = FmtPQ2::pq2_pair(w, f);
    }
  }
  __device__ static void bperm(const uint4& lo, const uint4& hi, uint4* out) {
    out[0] = make_uint4(prmt(lo.x, hi.x, 0x5410u), prmt(lo.x, hi.x, 0x7632u), prmt(lo.y, hi.y, 0x5410u),
                        prmt(lo.y, hi.y, 0x7632u));
    out[1] = make_uint4(prmt(lo.z, hi.z, 0x5410u), prmt(lo.z, hi.z, 0x7632u), prmt(lo.w, hi.w, 0x5410u),
                        prmt(lo.w, hi.w, 0x7632u));
  }
};

// CBK4: chunk c = slice 2G + c; index byte b of the row's 32 is the k pair
// (2b, 2b + 1), one table read of the fp16 pair (c[lo], c[hi]).
template <>
struct Tc5<FmtCBK4> {
  static constexpr bool kHas = true;
  static constexpr int kStages = 3;
  static constexpr int kCpw = 2, kDpc = 1, kCpd = 2, kXg = 8;
  static constexpr bool kTable = true;
  __device__ static int k0(int G, int c) { return (2 * G + c) * 64; }
  __device__ static void decode(const uint8_t* stage, int c, int G, int lp, int j, uint32_t key, uint32_t* out,
                                float (&sc)[2]) {
    const int t = (2 * G + c) * 32 + lp;
    const uint4 lo = lds128(stage + ((j * 2 + 0) * kLaneSlots + t) * 16);
    const uint4 hi = lds128(stage + ((j * 2 + 1) * kLaneSlots + t) * 16);
    sc[0] = 1.f;
    sc[1] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w = word8(lo, hi, i);
#pragma unroll
      for (int b = 0; b < 4; ++b) out[4 * i + b] = lds32_at(lut_addr(w, key, b));
    }
  }
  __device__ static void bperm(const uint4& x, const uint4&, uint4* out) { out[0] = x; }
};

// CBK8: the chunk is slices 2G and 2G + 1 (32 k each); A column c is the k
// pair (2c, 2c + 1): two table reads of fp16 centroids, joined.
template <>
struct Tc5<FmtCBK8> {
  static constexpr bool kHas = true;
  static constexpr int kStages = 3;
  static constexpr int kCpw = 1, kDpc = 1, kCpd = 1, kXg = 8;
  static constexpr bool kTable = true;
  __device__ static int k0(int G, int) { return 2 * G * 32; }
  __device__ static void decode(const uint8_t* stage, int, int G, int lp, int j, uint32_t key, uint32_t* out,
                                float (&sc)[2]) {
    sc[0] = 1.f;
    sc[1] = 0.f;
#pragma unroll
    for (int ss = 0; ss < 2; ++ss) {
      const int t = (2 * G + ss) * 32 + lp;
      const uint4 lo = lds128(stage + ((j * 2 + 0) * kLaneSlots + t) * 16);
      const uint4 hi = lds128(stage + ((j * 2 + 1) * kLaneSlots + t) * 16);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w = word8(lo, hi, i);
        const uint32_t e0 = lds32_at(lut_addr(w, key, 0)), e1 = lds32_at(lut_addr(w, key, 1));
        const uint32_t e2 = lds32_at(lut_addr(w, key, 2)), e3 = lds32_at(lut_addr(w, key, 3));
        out[16 * ss + 2 * i + 0] = prmt(e0, e1, 0x5410u);
        out[16 * ss + 2 * i + 1] = prmt(e2, e3, 0x5410u);
      }
    }
  }
  __device__ static void bperm(const uint4& x, const uint4&, uint4* out) { out[0] = x; }
};

// ------------------------------------------------------------ geometry -----

template <class F>
__host__ __device__ constexpr int tc5_nd() { return Tc5<F>::kDpc == 2 ? 4 : 2; }  // accumulator slots per warpgroup
template <class F>
__host__ __device__ constexpr int tc5_bar_bytes() {
  return (Tc5<F>::kStages + 16) * 8 + 16;  // + the tensor-memory base
}
template <int MT>
__host__ __device__ constexpr int tc5_red_bytes() { return 3 * 128 * MT * 4; }  // warpgroups 1..3
constexpr int kTc5BBytes = 4 * 2 * kTc5BSlotBytes;                             // 16 KB

// Shared memory.  Without a table: the stages, B, the reduction buffer, the
// mbarriers.  Table formats: the 64 KB table on a 64 KB boundary (as in the
// other kernels); before it stage 0, B and the mbarriers, after it the other
// stages and the reduction buffer.
template <class F>
__host__ __device__ constexpr int tc5_pre_bytes() { return F::kTileBytes + kTc5BBytes + tc5_bar_bytes<F>(); }
template <class F, int MT>
__host__ __device__ constexpr int tc5_smem_bytes() {
  return Tc5<F>::kTable
             ? kTableAlign + kLutBytes + (Tc5<F>::kStages - 1) * F::kTileBytes + tc5_red_bytes<MT>()
             : Tc5<F>::kStages * F::kTileBytes + kTc5BBytes + tc5_red_bytes<MT>() + tc5_bar_bytes<F>();
}

// Row of the tile whose codes thread (warp quarter q, lane l) of a
// warpgroup decodes: lane slot lp = 8q + (l & 7) of the slice, row j = l >> 3
// of the slot, i.e. row 4 lp + j.  The eight lanes of each quarter warp read
// eight consecutive slots, so their 16-byte code loads do not conflict.
__host__ __device__ constexpr int tc5_row_of_lane(int L) { return 4 * (8 * (L >> 5) + (L & 7)) + ((L & 31) >> 3); }

template <class F, int MT>
__global__ void __launch_bounds__(kTc5Threads, 1) tc5_kernel(const RunParams p, int M) {
  using T = Tc5<F>;
  constexpr int NS = T::kStages;
  constexpr int TB = F::kTileBytes;
  constexpr int CPW = T::kCpw;
  constexpr int ND = tc5_nd<F>();
  constexpr int XV = T::kXg == 16 ? 2 : 1;  // 16-byte x vectors per staged item

  if (static_cast<int>(blockIdx.x) == p.skip_cta) return;  // test hook (QGEMV_FAULT_SKIP_CTA)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring0 = smem;
  uint8_t* ringN;
  uint8_t* bbuf;
  float* red;
  uint64_t* bars;
  uint8_t* fsh = smem;  // the table (table formats)
  uint32_t lut_key = 0;
  if constexpr (T::kTable) {
    static_assert(tc5_pre_bytes<F>() + kTablePreSlack <= kTableAlign, "pre-table layout");
    const uint32_t base = smem_u32(smem);
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t R0 = (base + (kTableAlign - 1)) & ~uint32_t(kTableAlign - 1);
    if (R0 - base < uint32_t(tc5_pre_bytes<F>()) ||
        R0 + kLutBytes + (NS - 1) * TB + tc5_red_bytes<MT>() > base + dyn) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
      return;
    }
    fsh = smem + (R0 - base);
    ringN = fsh + kLutBytes;
    bbuf = smem + TB;
    bars = reinterpret_cast<uint64_t*>(bbuf + kTc5BBytes);
    red = reinterpret_cast<float*>(ringN + (NS - 1) * TB);
    lut_key = F::mma_lut_key(R0, static_cast<int>(threadIdx.x & 31u));
  } else {
    ringN = smem + TB;
    bbuf = smem + NS * TB;
    red = reinterpret_cast<float*>(bbuf + kTc5BBytes);
    bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + tc5_red_bytes<MT>());
  }
  uint64_t* full = bars;                      // [NS]: a tile has landed
  uint64_t* afull = bars + NS;                // [G][2]: the four warps have stored a chunk's A and B
  uint64_t* aempty = bars + NS + 8;           // [G][2]: a chunk's MMAs are done (its A and B slots are free,
                                              // the blocks it completes are ready to read back)
  uint32_t* s_tbase = reinterpret_cast<uint32_t*>(bars + NS + 16);
  auto stage_ptr = [&](int s) { return s == 0 ? ring0 : ringN + (s - 1) * TB; };
  __shared__ volatile int s_abort;
  __shared__ NextTable<F> s_next;
  __shared__ int s_rel[4];      // warps done with the tile in each stage
  __shared__ int s_nissued;     // tiles whose copies were issued
  __shared__ __align__(16) CtaPlan s_plan;
  static_assert(NS <= 4, "release counters");

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = warp >> 2;     // warpgroup
  const int wq = warp & 3;     // warp of the warpgroup (its quarter of the tensor-memory lanes)
  const int wtid = tid & 127;  // = the thread's tensor-memory lane
  const int lp = 8 * wq + (lane & 7);
  const int jr = lane >> 3;
  const int64_t Gd = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t t0 = stream_split<SplitModeOf<F>::value>(c, p.T, Gd);
  const int64_t t1 = stream_split<SplitModeOf<F>::value>(c + 1, p.T, Gd);
  const int ntiles = static_cast<int>(t1 - t0);
  const int64_t rt_first = div_fast(t0, p.nKT);
  const uint64_t pol = l2_policy_evict_first();

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    for (int i = 0; i < 8; ++i) {
      mbar_init(&afull[i], 4);
      mbar_init(&aempty[i], 1);
    }
    for (int s = 0; s < 4; ++s) s_rel[s] = 0;
    s_abort = 0;
    fence_mbarrier_init();
    int n = 0;
    for (; n < NS && n < ntiles; ++n) {
      mbar_arrive_expect_tx(&full[n], TB);
      bulk_g2s(stage_ptr(n), p.tiles + (t0 + n) * TB, TB, &full[n], pol);
    }
    s_nissued = n;
  }
  fetch_plan(&s_plan, p.plan, c, tid);
  if constexpr (T::kTable) {
    if (p.seg_of_rt != nullptr && ntiles > 0)
      prefetch_next_table<F>(&s_next, p, rt_first, div_fast(p.T, p.nKT), true, tid);
    F::template mma_init_shared<kTc5Threads>(fsh, table_of<F>(p, rt_first), warp, lane);
  }
  if (warp == 0) tmem_alloc_512(s_tbase);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tbase;
  // this warpgroup's columns, this warp's lanes
  const uint32_t tcol = tbase + static_cast<uint32_t>(G * kTc5ColsPerWg);
  const uint32_t tlane = static_cast<uint32_t>(32 * wq) << 16;
  uint8_t* bslots = bbuf + G * 2 * kTc5BSlotBytes;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t rt = rt_first;
  int kt = static_cast<int>(t0 - rt * p.nKT);
  const int nKT = static_cast<int>(p.nKT);
  const bool xvec = (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.K & 7) == 0;
  const unsigned short* xb = reinterpret_cast<const unsigned short*>(p.x);

  // Activation items of this thread: per chunk one (XV = 1: row m, 8-k group
  // g of 8; warp wq stages the groups of k16 step wq) or, for 16-k items, one
  // per two chunks (row m, 16-k group g of 4).  xr[r][v]: item r of the
  // current tile, vector v.
  constexpr int NI = T::kXg == 16 ? CPW / 2 : CPW;
  auto item_of = [&](int r, int& chunk, int& m, int& g) {
    if constexpr (T::kXg == 16) {
      chunk = 2 * r + (wtid >> 6);
      m = wtid & 15;
      g = (wtid & 63) >> 4;
    } else {
      chunk = r;
      m = wtid & 15;
      g = wtid >> 4;
    }
  };
  auto load_x8 = [&](int m, int64_t k) -> uint4 {
    if (m >= M || k >= p.K) return make_uint4(0u, 0u, 0u, 0u);
    const unsigned short* row = xb + m * p.K;
    if (xvec) return __ldg(reinterpret_cast<const uint4*>(row + k));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t kk = k + 2 * i;
      const uint32_t lo = kk < p.K ? __ldg(row + kk) : 0u;
      const uint32_t hi = kk + 1 < p.K ? __ldg(row + kk + 1) : 0u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  };
  uint4 xr[NI][XV];
  auto load_x_tile = [&](uint4 (&dst)[NI][XV], int ktile) {
#pragma unroll
    for (int r = 0; r < NI; ++r) {
      int ch, m, g;
      item_of(r, ch, m, g);
      const int64_t k = static_cast<int64_t>(ktile) * F::kKT + T::k0(G, ch) + T::kXg * g;
#pragma unroll
      for (int v = 0; v < XV; ++v) dst[r][v] = load_x8(m, k + 8 * v);
    }
  };
  if (ntiles > 0) load_x_tile(xr, kt);

  float yacc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) yacc[m] = 0.f;

  int ci = 0;            // chunks of this warpgroup so far
  int nblk = 0;          // blocks completed so far (issued)
  int pend = 0;          // blocks completed by the previous chunk, not yet read back
  float pend_sc[2] = {0.f, 0.f};

  // Read back the pending blocks' accumulators (one load per block, one
  // wait) and add them, scaled by the rows' block scales.
  // The blocks were completed by chunk ci - 1, whose single commit (its
  // slot's completion barrier) covers every MMA of them: the issuing thread
  // issued all of a block's MMAs.
  auto drain = [&](bool abort) {
    if (pend == 0) return;
    const int pc = ci - 1;  // called after the chunk counter moved on
    const bool ok = !abort && mbar_wait_bounded(&aempty[G * 2 + (pc & 1)], static_cast<uint32_t>((pc >> 1) & 1));
    if (__all_sync(0xffffffffu, ok)) {  // warp-uniform: tcgen05.ld is a warp-wide instruction
      tc_fence_after();
      const int B0 = nblk - pend;
      uint32_t dv[MT];
      tmem_ld_wait<MT>(tlane + tcol + kTc5DCol0 + 16 * (B0 % ND), dv);
#pragma unroll
      for (int m = 0; m < MT; ++m) yacc[m] = fmaf(pend_sc[0], __uint_as_float(dv[m]), yacc[m]);
      if (pend == 2) {
        tmem_ld_wait<MT>(tlane + tcol + kTc5DCol0 + 16 * ((B0 + 1) % ND), dv);
#pragma unroll
        for (int m = 0; m < MT; ++m) yacc[m] = fmaf(pend_sc[1], __uint_as_float(dv[m]), yacc[m]);
      }
    } else if (!abort) {
      if (lane == 0) atomicOr(p.err, kErrTimeoutFull);
      s_abort = 1;
    }
    pend = 0;
  };

  const bool stacked = T::kTable && p.seg_of_rt != nullptr;
  auto next_table = [&]() {
    if constexpr (T::kTable)
      advance_table<F, kTc5Threads>(&s_next, p, rt, tid, [&](const uint16_t* cb) {
        mma_rebuild_table<F, kTc5Threads>(fsh, cb, warp, lane);
      });
  };

  // The warp is done with the codes of tile i (stage st): the sixteenth warp
  // to say so refills the stage with tile i + NS, so that no thread ever
  // waits for the others to free a stage.
  auto release_and_refill = [&](int i, int st, bool abort) {
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const int old = atomicAdd(&s_rel[st], 1);
      if (old == kTc5Threads / 32 - 1) {
        __threadfence_block();
        s_rel[st] = 0;
        const int u = i + NS;
        if (u < ntiles && !abort && s_abort == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive_expect_tx(&full[st], TB);
          bulk_g2s(stage_ptr(st), p.tiles + (t0 + u) * TB, TB, &full[st], pol);
          atomicMax(&s_nissued, u + 1);
        }
      }
    }
    __syncwarp();
  };

  // The warp's part of chunk ci of its warpgroup: wait until the A and B
  // slots are free, stage its B rows, decode its 32 weight rows into A, tell
  // the warpgroup's issuer, issue the chunk's MMAs if it is this warp's turn,
  // then read back the blocks the previous chunk completed.
  auto do_chunk = [&](const uint8_t* stage, int i, int st, int chk, bool abort) {
    const int as = ci & 1;
    const bool freed = abort || ci < 2 ||
                       mbar_wait_bounded(&aempty[G * 2 + as], static_cast<uint32_t>(((ci >> 1) - 1) & 1));
    if (!__all_sync(0xffffffffu, freed)) {  // warp-uniform, as tcgen05.st is warp-wide
      if (lane == 0) atomicOr(p.err, kErrTimeoutFull);
      s_abort = 1;
      abort = true;
    }
    uint8_t* bs = bslots + as * kTc5BSlotBytes;
    float sc[2] = {1.f, 0.f};
    if (!abort) {
#pragma unroll
      for (int r = 0; r < NI; ++r) {
        int ch, m, g;
        item_of(r, ch, m, g);
        if (ch != chk) continue;
        uint4 rows[2];
        T::bperm(xr[r][0], xr[r][XV - 1], rows);
        if constexpr (T::kXg == 16) {
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)
            *reinterpret_cast<uint4*>(bs + g * 512 + (m >> 3) * 256 + kb * 128 + (m & 7) * 16) = rows[kb];
        } else {
          *reinterpret_cast<uint4*>(bs + (g >> 1) * 512 + (m >> 3) * 256 + (g & 1) * 128 + (m & 7) * 16) = rows[0];
        }
      }
      uint32_t a[32];
      T::decode(stage, chk, G, lp, jr, lut_key, a, sc);
      tmem_st16(tlane + tcol + as * 32, a);
      tmem_st16(tlane + tcol + as * 32 + 16, a + 16);
    }
    if (chk == CPW - 1) release_and_refill(i, st, abort);
    if (!abort) {
      tmem_wait_st();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B, for the MMAs
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&afull[G * 2 + as]);
    // blocks this chunk completes, and the warp that issues it (per block:
    // a block's MMAs all come from one thread)
    const int done = T::kDpc == 2 ? 2 : ((T::kCpd == 2) ? (ci & 1) : 1);
    const int who = (T::kCpd == 2) ? ((ci >> 1) & 3) : (ci & 3);
    if (wq == who && lane == 0 && !abort) {
      if (mbar_wait_bounded(&afull[G * 2 + as], static_cast<uint32_t>((ci >> 1) & 1))) {
        tc_fence_after();
        // B of k16 step s at bs + 512 s: the descriptor's address field (in
        // 16-byte units, well inside its 14 bits) advances by 32 per step
        const uint64_t bdesc0 = smem_desc_kmajor(smem_u32(bs), 128, 256);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          int B;
          bool first;
          if constexpr (T::kDpc == 2) {
            B = nblk + (s >> 1);
            first = (s & 1) == 0;
          } else if constexpr (T::kCpd == 2) {
            B = nblk;
            first = (ci & 1) == 0 && s == 0;
          } else {
            B = nblk;
            first = s == 0;
          }
          const uint32_t dcol = tcol + kTc5DCol0 + 16 * (B % ND);
          umma_f16_tmem_a(dcol, tcol + as * 32 + 8 * s, bdesc0 + static_cast<uint64_t>(32 * s), !first);
        }
        umma_commit(&aempty[G * 2 + as]);
      } else {
        atomicOr(p.err, kErrTimeoutFull);
        s_abort = 1;
      }
    }
    __syncwarp();
    drain(abort);  // the blocks of chunk ci - 1
    pend = done;
    if (T::kDpc == 2) {
      pend_sc[0] = sc[0];
      pend_sc[1] = sc[1];
    } else if (done) {
      pend_sc[0] = sc[0];  // PQ2_0: both chunks of a block read the same scale
    }
    nblk += done;
    ++ci;
  };

  // Row-tile end: add the warpgroups' row sums in order (G = 0, 1, 2, 3) and
  // store them to y (a whole row tile) or to the partial slots.
  auto row_epilogue = [&](int64_t cur_rt, bool abort) {
    drain(abort);
    if (G > 0) {
      float* dst = red + ((G - 1) * 128 + wtid) * MT;
#pragma unroll
      for (int m = 0; m < MT; m += 4)
        *reinterpret_cast<float4*>(dst + m) = make_float4(yacc[m], yacc[m + 1], yacc[m + 2], yacc[m + 3]);
    }
    __syncthreads();
    if (G == 0) {
      const bool owner = (cur_rt * p.nKT >= t0) && ((cur_rt + 1) * p.nKT <= t1);
      const int side = (cur_rt * p.nKT <= t0) ? 0 : 1;
      float* my_part = p.partials + (c * 2 + side) * kPartialStride;
      const int r = tc5_row_of_lane(wtid);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = yacc[m];
#pragma unroll
        for (int g = 0; g < 3; ++g) v += red[(g * 128 + wtid) * MT + m];
        if (m < M) {
          if (owner) {
            const int64_t n = cur_rt * kTileRows + r;
            if (n < p.N) store_y(p, m * p.N + n, v);
          } else {
            st_relaxed_f32(my_part + m * kTileRows + r, v);
          }
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < MT; ++m) yacc[m] = 0.f;
  };

  for (int i = 0; i < ntiles; ++i) {
    if (stacked && kt == 0 && i > 0) next_table();
    const int st = i % NS;
    const int kt_next = (kt + 1 == nKT) ? 0 : kt + 1;
    uint4 xn[NI][XV];
    if (i + 1 < ntiles) load_x_tile(xn, kt_next);
    bool abort = __any_sync(0xffffffffu, s_abort != 0);
    if (!__all_sync(0xffffffffu, abort || mbar_wait_bounded(&full[st], static_cast<uint32_t>((i / NS) & 1)))) {
      if (lane == 0) atomicOr(p.err, kErrTimeoutFull);
      s_abort = 1;
      abort = true;
    }
    const uint8_t* stage = stage_ptr(st);
#pragma unroll 1
    for (int chk = 0; chk < CPW; ++chk) do_chunk(stage, i, st, chk, abort);
#pragma unroll
    for (int r = 0; r < NI; ++r)
#pragma unroll
      for (int v = 0; v < XV; ++v) xr[r][v] = xn[r][v];
    const bool row_end = (kt_next == 0) || (i + 1 == ntiles);
    const int64_t cur_rt = rt;
    kt = kt_next;
    if (kt_next == 0) ++rt;
    if (row_end) row_epilogue(cur_rt, s_abort != 0);
  }

  // Before leaving: every MMA of the warpgroup is done -- the last phase of
  // each A slot (chunks are issued by several threads, so a thread's own
  // last chunk need not be the slot's last) -- and no copy of this CTA is
  // still landing.
  if (wtid == 0) {
    for (int sl = 0; sl < 2; ++sl) {
      const int last = ci - 1 - ((ci - 1 - sl) & 1);  // the slot's last chunk
      if (last >= 0) mbar_wait_bounded(&aempty[G * 2 + sl], static_cast<uint32_t>((last >> 1) & 1));
    }
  }
  __syncthreads();
  if (tid == 0 && s_abort != 0) {
    const int n = s_nissued;
    for (int u = (n > NS ? n - NS : 0); u < n; ++u)
      mbar_wait_bounded(&full[u % NS], static_cast<uint32_t>((u / NS) & 1));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_512(tbase);
  }

  // split row tiles: the shared polled-slot finisher
  static_assert(tc5_red_bytes<MT>() >= 2 * kTc5Threads * 4, "finishing scratch");
  wait_plan();
  finish_all<kTileRows, MT, kTc5Threads>(p, kPartialStride, s_plan, nullptr, 1.0f, red, tid, M);
}

}  // namespace qgemv

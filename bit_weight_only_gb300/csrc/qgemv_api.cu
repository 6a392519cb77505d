// qgemv_api.cu -- the C ABI declared in include/qgemv.h.
//
// Host side only: argument checks, ownership of the device buffers of a
// handle, the per-format dispatch (format -> FormatOps, M -> kernel
// instantiation) and error reporting.  No exception crosses the ABI and no
// call aborts.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "formats.h"
#include "gemv_kernel.cuh"
#include "qgemv.h"

namespace {

constexpr uint32_t kMagic = 0x51474d56u;  // "QGMV"
// Internal format id: the tensor-core layout of an AQLM 2x8 matrix, held by
// every AQLM handle next to its table-path layout and used from
// kAqlmMmaMinM activation rows on (and for every M in batch-invariant mode).
constexpr int kAqlmMma = 6;
constexpr int kAqlmMmaMinM = 3;

thread_local char g_msg[512] = "";
thread_local int g_code = QGEMV_OK;

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  g_code = code;
  return code;
}

int ok() {
  g_msg[0] = '\0';
  g_code = QGEMV_OK;
  return QGEMV_OK;
}

int cuda_error(cudaError_t e, const char* what) {
  return set_error(QGEMV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

const qgemv::FormatOps* ops_for(int format) {
  switch (format) {
    case QGEMV_Q4_0: return qgemv::ops_q4_0();
    case QGEMV_PQ2_0: return qgemv::ops_pq2();
    case QGEMV_CBK4: return qgemv::ops_cbk4();
    case QGEMV_CBK8: return qgemv::ops_cbk8();
    case QGEMV_AQLM_2X8: return qgemv::ops_aqlm();
    case kAqlmMma: return qgemv::ops_aqlm_mma();
    case QGEMV_AQLM_1X16: return qgemv::ops_aqlm_1x16();
    case QGEMV_CBK4_ROW: return qgemv::ops_cbk4_row();
    case QGEMV_CBK8_ROW: return qgemv::ops_cbk8_row();
  }
  return nullptr;
}

// K granularity and canonical sizes per format.
int64_t k_multiple(int format) {
  switch (format) {
    case QGEMV_Q4_0: return 32;
    case QGEMV_CBK4: return 2;
    case QGEMV_CBK8: return 1;
    case QGEMV_PQ2_0: return 128;
    case QGEMV_AQLM_2X8: return 8;
    case kAqlmMma: return 8;
    case QGEMV_AQLM_1X16: return 8;
    case QGEMV_CBK4_ROW: return 2;
    case QGEMV_CBK8_ROW: return 1;
  }
  return 0;
}

int64_t scales_count(int format, int64_t N) {
  return format == QGEMV_AQLM_2X8 || format == kAqlmMma || format == QGEMV_AQLM_1X16 ? N : 0;
}

int64_t codebook_count(int format) {
  switch (format) {
    case QGEMV_CBK4: return 16;
    case QGEMV_CBK8: return 256;
    case QGEMV_AQLM_2X8: return 2 * 256 * 8;
    case kAqlmMma: return 2 * 256 * 8;
    case QGEMV_AQLM_1X16: return 65536 * 8;
    case QGEMV_CBK4_ROW: return 16;  // per output row, fp32
    case QGEMV_CBK8_ROW: return 256;  // per output row, fp32
  }
  return 0;
}

bool is_device_pointer(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear: plain host memory on some setups
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Fault hooks for tests, read when a handle is created (host side only;
// nothing on the device faults or hangs):
//   QGEMV_FAULT_ALLOC=n     the n-th device allocation of the create call
//                           fails as if the device were out of memory;
//   QGEMV_ROWGROUP=0|1      (not a fault) forbid or force the M = 1
//                           row-group kernel of the table formats, so that
//                           tests cover both M = 1 kernels on any shape;
//   QGEMV_TC5=n             (not a fault) runs with at least n activation
//                           rows use the tensor-memory kernel of the formats
//                           that have it (0: never, 1: every M), instead of
//                           the measured default, so that tests and the
//                           benchmark's crossover sweep reach both kernels;
//   QGEMV_FAULT_SKIP_CTA=c  the handle's runs launch CTA c as a no-op, so
//                           the CTAs that share a row tile with it never get
//                           its partial sums: their bounded fix-up waits run
//                           out and qgemv_status reports QGEMV_ERR_TIMEOUT.
int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return v && *v ? std::atoi(v) : dflt;
}
thread_local int g_alloc_count = 0;  // device allocations of the current create call
thread_local int g_alloc_fail = 0;   // QGEMV_FAULT_ALLOC of the current create call

cudaError_t dev_alloc(void** dst, size_t bytes) {
  if (++g_alloc_count == g_alloc_fail) {
    *dst = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(dst, bytes);
}

// Copy `bytes` from a host or device pointer into a fresh device buffer.
cudaError_t to_device(const void* src, size_t bytes, void** dst) {
  *dst = nullptr;
  if (bytes == 0) return cudaSuccess;
  cudaError_t e = dev_alloc(dst, bytes);
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(*dst, src, bytes, is_device_pointer(src) ? cudaMemcpyDeviceToDevice
                                                          : cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(*dst);
    *dst = nullptr;
  }
  return e;
}

// The stream-K split of T tiles over G CTAs: CTA c runs [c*T/G, (c+1)*T/G).
// A row tile (nKT consecutive tiles) that no single CTA covers is "shared";
// its contributors are the CTAs whose runs touch it.  Each gets an even
// slice of its rows to finish, and one of them the finisher flag (the
// kernels' finish_slice picks between the two by the tile's item count):
// the last contributor, unless the row tile opens that CTA's run (its part
// is then done early), in which case the one before it.  Computed once per
// handle so the kernels do no 64-bit divisions.
int64_t split_point(int64_t c, int64_t T, int64_t G, int64_t U) {
  if (U == 0) return c * T / G;
  const int64_t n = (T + U - 1) / U, q = n / G, r = n % G;
  const int64_t t = (c * q + (c < r ? c : r)) * U;
  return t < T ? t : T;
}
// the CTA whose run holds unit t
int64_t cta_of(int64_t t, int64_t T, int64_t G, int64_t U) {
  if (U == 0) return ((t + 1) * G - 1) / T;
  const int64_t n = (T + U - 1) / U, q = n / G, r = n % G, u = t / U;
  return u < r * (q + 1) ? u / (q + 1) : r + (u - r * (q + 1)) / q;
}

std::vector<qgemv::CtaPlan> plan_stream_k(int64_t T, int64_t G, int64_t nKT, int64_t rows, int64_t U) {
  std::vector<qgemv::CtaPlan> plan(static_cast<size_t>(G));
  for (int64_t c = 0; c < G; ++c) {
    qgemv::CtaPlan& pl = plan[static_cast<size_t>(c)];
    std::memset(&pl, 0, sizeof(pl));
    pl.seg_rt[0] = pl.seg_rt[1] = -1;
    const int64_t t0 = split_point(c, T, G, U), t1 = split_point(c + 1, T, G, U);
    if (t1 <= t0) continue;
    auto owned = [&](int64_t r) { return r * nKT >= t0 && (r + 1) * nKT <= t1; };
    const int64_t first = t0 / nKT, last = (t1 - 1) / nKT;
    int sg = 0;
    for (int64_t r : {first, last}) {
      if (owned(r) || (sg == 1 && r == first)) {
        ++sg;
        continue;
      }
      const int64_t cf = cta_of(r * nKT, T, G, U);
      const int64_t cl = cta_of((r + 1) * nKT - 1, T, G, U);
      pl.seg_rt[sg] = r;
      pl.seg_cf[sg] = cf;
      const int64_t S = cl - cf + 1, k = c - cf;
      pl.seg_S[sg] = static_cast<int32_t>(S);
      pl.seg_r0[sg] = static_cast<int32_t>(k * rows / S);
      pl.seg_nr[sg] = static_cast<int32_t>((k + 1) * rows / S - k * rows / S);
      const int64_t fin = split_point(cl + 1, T, G, U) > (r + 1) * nKT ? cl - 1 : cl;
      pl.seg_flags[sg] = (split_point(cf, T, G, U) < r * nKT ? 1 : 0) | (c == fin ? 2 : 0);
      ++sg;
    }
  }
  return plan;
}

std::once_flag g_setup_once[16];
cudaError_t g_setup_err[16];

}  // namespace

namespace qgemv {
int report_error(int code, const char* msg) {
  if (code == QGEMV_OK) return ok();
  return set_error(code, "%s", msg);
}
}  // namespace qgemv

struct qgemv_ctx {
  uint32_t magic;
  int format;
  int64_t N, K;
  const qgemv::FormatOps* ops;
  int64_t nRT;
  int nKT;
  int64_t T;
  int grid;      // tensor-core and AQLM kernels: min(T, SMs)
  int grid_m1;   // M = 1 CUDA-core kernel: min(T, SMs * m1_ctas_per_sm)
  int grid_rg;   // M = 1 row-group kernel (table formats): min(units, SMs), 0 if not used
  uint8_t* tiles;
  void* aux;
  float* partials;
  qgemv::CtaPlan* plan;     // [grid], then [grid_m1] for the M = 1 kernel if that grid differs
  qgemv::CtaPlan* plan_m1;
  int32_t* seg_of_rt;  // inside aux (stacked table formats and AQLM 2x8), else nullptr
  int* err;
  int batch_invariant;  // qgemv_set_batch_invariant
  int x_int8;           // qgemv_set_x_int8 (PQ2_0)
  int glu;              // qgemv_create_glu: gate and up interleaved, output SiLU(gate) * up
  int skip_cta;         // QGEMV_FAULT_SKIP_CTA test hook, -1 normally
  int tc5_min_m;        // runs of at least this many rows use the tensor-memory kernel (0: never)
  uint8_t* xq_ws;       // INT8 mode: the activation prologue's workspace (16 rows), allocated when turned on
  qgemv_ctx* mma;       // AQLM: the tensor-core companion (format kAqlmMma), else nullptr
};

extern "C" {

int64_t qgemv_packed_bytes(int format, int64_t N, int64_t K) {
  const int64_t km = k_multiple(format);
  if (km == 0 || N <= 0 || K <= 0 || K % km) return 0;
  switch (format) {
    case QGEMV_Q4_0: return N * (K / 32) * 18;
    case QGEMV_CBK4: return N * (K / 2);
    case QGEMV_CBK8: return N * K;
    case QGEMV_PQ2_0: return N * (K / 128) * 34;
    case QGEMV_AQLM_2X8: return N * (K / 8) * 2;
    case QGEMV_AQLM_1X16: return N * (K / 8) * 2;
    case QGEMV_CBK4_ROW: return N * (K / 2);
    case QGEMV_CBK8_ROW: return N * K;
  }
  return 0;
}

}  // extern "C"

static int64_t canonical_bytes(int format, int64_t N, int64_t K) {
  return qgemv_packed_bytes(format == kAqlmMma ? QGEMV_AQLM_2X8 : format, N, K);
}

static void free_handle(qgemv_ctx* h);

// Both create calls: `nseg` codebooks for the row segments `seg_rows`
// (one segment covering all N rows for qgemv_create).  `nested`: the
// companion of an AQLM handle, created within the same create call (the
// allocation fault counter keeps counting).
static qgemv_handle create_impl(int format, int64_t N, int64_t K, const void* packed, const void* scales,
                                const void* codebooks, int nseg, const int64_t* seg_rows,
                                bool nested = false, bool glu = false) {
  const qgemv::FormatOps* ops = ops_for(format);
  if (k_multiple(format) == 0) {
    set_error(QGEMV_ERR_ARG, "unknown format %d", format);
    return nullptr;
  }
  if (!ops) {
    set_error(QGEMV_ERR_ARG, "format %d is not built into this library", format);
    return nullptr;
  }
  if (N <= 0 || K <= 0 || K % k_multiple(format)) {
    set_error(QGEMV_ERR_ARG, "invalid shape N=%lld K=%lld for format %d (K must be a positive multiple of %lld)",
              (long long)N, (long long)K, format, (long long)k_multiple(format));
    return nullptr;
  }
  if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) {
    set_error(QGEMV_ERR_ARG, "N and K must be at most 2^31");
    return nullptr;
  }
  if (format == QGEMV_CBK8_ROW && K > 65536) {  // one activation row is staged in shared memory
    set_error(QGEMV_ERR_ARG, "CBK8_ROW takes K up to 65536 (got %lld)", (long long)K);
    return nullptr;
  }
  if (!packed) {
    set_error(QGEMV_ERR_ARG, "packed is NULL");
    return nullptr;
  }
  if ((scales_count(format, N) > 0) != (scales != nullptr)) {
    set_error(QGEMV_ERR_ARG, scales ? "format %d takes no scales" : "format %d needs scales", format);
    return nullptr;
  }
  if ((codebook_count(format) > 0) != (codebooks != nullptr)) {
    set_error(QGEMV_ERR_ARG, codebooks ? "format %d takes no codebooks" : "format %d needs codebooks",
              format);
    return nullptr;
  }

  std::call_once(g_setup_once[format], [&] { g_setup_err[format] = ops->setup(); });
  if (g_setup_err[format] != cudaSuccess) {
    cuda_error(g_setup_err[format], "kernel setup");
    return nullptr;
  }

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_error(e, "device query");
    return nullptr;
  }

  qgemv_ctx* h = new (std::nothrow) qgemv_ctx();
  if (!h) {
    set_error(QGEMV_ERR_NOMEM, "host allocation failed");
    return nullptr;
  }
  h->magic = kMagic;
  h->skip_cta = env_int("QGEMV_FAULT_SKIP_CTA", -1);
  h->tc5_min_m = qgemv::has_tc5(format) ? env_int("QGEMV_TC5", ops->tc5_min_m) : 0;
  if (h->tc5_min_m < 0 || h->tc5_min_m > qgemv::kMaxM) h->tc5_min_m = 0;
  if (!nested) {
    g_alloc_count = 0;
    g_alloc_fail = env_int("QGEMV_FAULT_ALLOC", 0);
  }
  h->format = format;
  h->glu = glu ? 1 : 0;
  h->N = N;
  h->K = K;
  h->ops = ops;
  h->nRT = (N + ops->tile_rows - 1) / ops->tile_rows;
  h->nKT = static_cast<int>((K + ops->kt - 1) / ops->kt);
  h->T = h->nRT * h->nKT;
  h->grid = static_cast<int>(h->T < sms ? h->T : sms);
  {
    const int64_t g1 = int64_t(sms) * ops->m1_ctas_per_sm;
    h->grid_m1 = static_cast<int>(h->T < g1 ? h->T : g1);
  }
  // The row-group kernel (whole 32-row groups per CTA, no split-K finish)
  // for matrices of at most one row group per SM whose busiest CTA then
  // streams no more than the stream-K split's busiest one.  Measured on the
  // 7B shapes: the 4096 x 4096 projection gains 10%; with several row groups
  // per CTA (q|k|v, gate|up) the per-group epilogues and codebook changes
  // cost more than the split-K finish they save.
  if (ops->rowgroup && !glu) {
    const int64_t U = h->nRT * 4, nch = (h->nKT + 3) / 4;
    const int64_t Grg = U < sms ? U : sms;
    const int64_t rg_bytes = (U + Grg - 1) / Grg * h->nKT * (ops->tile_bytes / 4);
    const int64_t sk_bytes = (h->T + h->grid_m1 - 1) / h->grid_m1 * ops->tile_bytes;
    bool use = nch >= 2 && U <= sms && nseg == 1 && rg_bytes <= sk_bytes;
    const int force = env_int("QGEMV_ROWGROUP", -1);
    if (force == 0) use = false;
    if (force == 1) use = true;
    h->grid_rg = use ? static_cast<int>(Grg) : 0;
  }
  const int slots_grid = h->grid > h->grid_m1 ? h->grid : h->grid_m1;  // partial slots for either grid
  const int n_plans = h->grid + (h->grid_m1 != h->grid ? h->grid_m1 : 0);
  // codebook segment of every row tile (table formats)
  std::vector<int32_t> seg_of_rt(static_cast<size_t>(h->nRT), 0);
  if (ops->row_tables) {  // a table of its own for every row tile
    for (int64_t r = 0; r < h->nRT; ++r) seg_of_rt[static_cast<size_t>(r)] = static_cast<int32_t>(r);
  } else {
    int64_t row = 0;
    for (int s = 0; s < nseg; ++s) {
      for (int64_t r = row; r < row + seg_rows[s]; r += ops->tile_rows)
        seg_of_rt[static_cast<size_t>(r / ops->tile_rows)] = s;
      row += seg_rows[s];
    }
  }

  void *d_packed = nullptr, *d_scales = nullptr, *d_cb = nullptr;
  auto cleanup = [&](int code, const char* what, cudaError_t ce) -> qgemv_handle {
    if (ce == cudaErrorMemoryAllocation) {
      cudaGetLastError();  // a real allocation failure is sticky in the last-error state
      set_error(QGEMV_ERR_NOMEM, "%s: out of device memory", what);
    } else if (ce != cudaSuccess) {
      cuda_error(ce, what);
    } else {
      set_error(code, "%s", what);
    }
    cudaFree(d_packed);
    cudaFree(d_scales);
    cudaFree(d_cb);
    cudaFree(h->tiles);
    cudaFree(h->aux);
    cudaFree(h->partials);
    cudaFree(h->plan);
    cudaFree(h->err);
    h->magic = 0;
    delete h;
    return nullptr;
  };

  e = to_device(packed, static_cast<size_t>(canonical_bytes(format, N, K)), &d_packed);
  if (e == cudaSuccess) e = to_device(scales, 2 * scales_count(format, N), &d_scales);
  const bool per_row_cb = format == QGEMV_CBK4_ROW || format == QGEMV_CBK8_ROW;
  // a GLU handle of a one-codebook format holds two codebooks (gate, up)
  const bool glu_tables = glu && ops->cb_entries > 0 && !ops->row_tables;
  const int64_t cb_bytes = per_row_cb ? 4 * codebook_count(format) * N  // fp32 per row
                                      : 2 * codebook_count(format) * nseg * (glu_tables ? 2 : 1);
  if (e == cudaSuccess) e = to_device(codebooks, static_cast<size_t>(cb_bytes), &d_cb);
  if (e != cudaSuccess) return cleanup(QGEMV_ERR_CUDA, "copying the canonical inputs", e);

  e = dev_alloc(reinterpret_cast<void**>(&h->tiles), static_cast<size_t>(h->T) * ops->tile_bytes);
  // table formats: one codebook, or (stacked) one copy per row tile followed
  // by the row tiles' segments
  const bool stacked = ops->cb_entries > 0 && (nseg > 1 || ops->row_tables);
  const int64_t table_bytes = int64_t(2) * ops->cb_entries * (stacked ? h->nRT : 1) * (glu_tables ? 2 : 1);
  // a stacked AQLM 2x8 handle: its segments' codebook pairs, the row scales,
  // then the segment of every 2048-row block (aligned to 4 bytes)
  const bool aqlm_stacked = format == QGEMV_AQLM_2X8 && nseg > 1;
  const int64_t aux_fixed = ops->aux_bytes * (aqlm_stacked ? nseg : 1) + ops->aux_per_row * N;
  const int64_t seg_map_off = (aux_fixed + 3) / 4 * 4;
  const int64_t aux_bytes = ops->cb_entries > 0 ? table_bytes + (stacked ? 4 * h->nRT : 0)
                                                : (aqlm_stacked ? seg_map_off + 4 * h->nRT : aux_fixed);
  if (e == cudaSuccess && aux_bytes > 0) e = dev_alloc(&h->aux, static_cast<size_t>(aux_bytes));
  if (e == cudaSuccess)
    e = dev_alloc(reinterpret_cast<void**>(&h->partials),
                  sizeof(float) * 2 * ops->partial_stride * static_cast<size_t>(slots_grid));
  if (e == cudaSuccess) e = dev_alloc(reinterpret_cast<void**>(&h->plan), sizeof(qgemv::CtaPlan) * n_plans);
  if (e == cudaSuccess) e = dev_alloc(reinterpret_cast<void**>(&h->err), sizeof(int));
  if (e == cudaSuccess && (stacked || aqlm_stacked)) {
    h->seg_of_rt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(h->aux) + (stacked ? table_bytes : seg_map_off));
    e = cudaMemcpy(h->seg_of_rt, seg_of_rt.data(), 4 * seg_of_rt.size(), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    // a GLU handle's shared row tiles are finished in gate/up row pairs
    const int plan_rows = glu ? ops->tile_rows / 2 : ops->tile_rows;
    std::vector<qgemv::CtaPlan> plan = plan_stream_k(h->T, h->grid, h->nKT, plan_rows, ops->split_unit);
    if (h->grid_m1 != h->grid) {
      const std::vector<qgemv::CtaPlan> plan1 = plan_stream_k(h->T, h->grid_m1, h->nKT, plan_rows, ops->split_unit);
      plan.insert(plan.end(), plan1.begin(), plan1.end());
    }
    e = cudaMemcpy(h->plan, plan.data(), sizeof(qgemv::CtaPlan) * plan.size(), cudaMemcpyHostToDevice);
    h->plan_m1 = h->grid_m1 != h->grid ? h->plan + h->grid : h->plan;
  }
  // partial slots start empty (all ones): the AQLM fix-up polls them
  if (e == cudaSuccess)
    e = cudaMemset(h->partials, 0xff, sizeof(float) * 2 * ops->partial_stride * static_cast<size_t>(slots_grid));
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(int));
  if (e != cudaSuccess) return cleanup(QGEMV_ERR_CUDA, "allocating the handle's device buffers", e);

  qgemv::PrepareArgs a;
  a.packed = static_cast<const uint8_t*>(d_packed);
  a.scales = static_cast<const uint16_t*>(d_scales);
  a.codebooks = static_cast<const uint16_t*>(d_cb);
  a.N = N;
  a.K = K;
  a.nRT = h->nRT;
  a.nKT = h->nKT;
  a.tiles = h->tiles;
  a.aux = h->aux;
  a.nseg = nseg;
  a.seg_of_rt = h->seg_of_rt;
  a.glu = glu_tables ? 1 : 0;
  e = ops->prepare(a, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cleanup(QGEMV_ERR_CUDA, "preparing the tiles", e);

  cudaFree(d_packed);
  cudaFree(d_scales);
  cudaFree(d_cb);
  // The tensor-core companion has one codebook pair; a stacked handle runs
  // the table kernel at every M instead (passes of two rows).
  if (format == QGEMV_AQLM_2X8 && !aqlm_stacked) {
    h->mma = create_impl(kAqlmMma, N, K, packed, scales, codebooks, 1, seg_rows, true);
    if (!h->mma) {  // the error is set
      free_handle(h);
      return nullptr;
    }
  }
  ok();
  return h;
}

extern "C" {

qgemv_handle qgemv_create(int format, int64_t N, int64_t K, const void* packed, const void* scales,
                          const void* codebooks) {
  if (format == kAqlmMma) {
    set_error(QGEMV_ERR_ARG, "unknown format %d", format);
    return nullptr;
  }
  const int64_t rows[1] = {N};
  return create_impl(format, N, K, packed, scales, codebooks, 1, rows);
}

qgemv_handle qgemv_create_stacked(int format, int nseg, const int64_t* seg_rows, int64_t K,
                                  const void* packed, const void* scales, const void* codebooks) {
  const qgemv::FormatOps* ops = ops_for(format);
  if (!ops || k_multiple(format) == 0) {
    set_error(QGEMV_ERR_ARG, "unknown format %d", format);
    return nullptr;
  }
  if (format == kAqlmMma || format == QGEMV_AQLM_1X16 || format == QGEMV_CBK4_ROW || format == QGEMV_CBK8_ROW) {
    set_error(QGEMV_ERR_ARG, "format %d cannot be stacked", format);
    return nullptr;
  }
  if (nseg < 1 || !seg_rows) {
    set_error(QGEMV_ERR_ARG, "nseg must be >= 1 with seg_rows given");
    return nullptr;
  }
  int64_t N = 0;
  for (int s = 0; s < nseg; ++s) {
    if (seg_rows[s] <= 0 || (s + 1 < nseg && seg_rows[s] % ops->tile_rows)) {
      set_error(QGEMV_ERR_ARG, "segment %d has %lld rows (must be > 0, and a multiple of %d but for the last)",
                s, (long long)seg_rows[s], ops->tile_rows);
      return nullptr;
    }
    N += seg_rows[s];
  }
  // codebook formats keep a codebook (AQLM 2x8: a codebook pair) per segment
  const bool per_seg_cb = ops->cb_entries > 0 || format == QGEMV_AQLM_2X8;
  return create_impl(format, N, K, packed, scales, codebooks, per_seg_cb ? nseg : 1, seg_rows);
}

qgemv_handle qgemv_create_glu(int format, int64_t N, int64_t K, const void* packed_gate, const void* packed_up,
                              const void* codebooks_gate, const void* codebooks_up) {
  const qgemv::FormatOps* ops = ops_for(format);
  if (!ops || format == kAqlmMma || ops->launch_glu == nullptr) {
    set_error(QGEMV_ERR_ARG,
              "format %d has no fused SiLU(gate) * up (Q4_0, PQ2_0, CBK4, CBK8 and CBK4_ROW have)", format);
    return nullptr;
  }
  if (!packed_gate || !packed_up) {
    set_error(QGEMV_ERR_ARG, "packed_gate or packed_up is NULL");
    return nullptr;
  }
  const bool row_cb = format == QGEMV_CBK4_ROW;  // per-row codebooks travel with their rows
  const bool has_cb = row_cb || ops->cb_entries > 0;
  if (has_cb != (codebooks_gate != nullptr && codebooks_up != nullptr) ||
      (!has_cb && (codebooks_gate != nullptr || codebooks_up != nullptr))) {
    set_error(QGEMV_ERR_ARG, has_cb ? "format %d needs both codebook arrays" : "format %d takes no codebooks",
              format);
    return nullptr;
  }
  const int64_t half = ops->tile_rows / 2;
  const int64_t row_bytes = qgemv_packed_bytes(format, 1, K);
  if (N <= 0 || N % half || row_bytes == 0 || N > (int64_t(1) << 30)) {
    set_error(QGEMV_ERR_ARG, "invalid GLU shape N=%lld K=%lld (N must be a positive multiple of %lld)",
              (long long)N, (long long)K, (long long)half);
    return nullptr;
  }
  // gate rows 64b .. 64b+63, then up rows 64b .. 64b+63, for every block b:
  // the canonical bytes of the interleaved 2N-row matrix
  g_alloc_count = 0;
  g_alloc_fail = env_int("QGEMV_FAULT_ALLOC", 0);
  void* inter = nullptr;
  void* inter_cb = nullptr;
  // interleave 64-row blocks of two row-major arrays of `rb` bytes per row
  auto interleave = [&](void* dst, const void* a, const void* b, int64_t rb) {
    const int64_t blk = half * rb;
    cudaError_t ce = cudaSuccess;
    for (int64_t i = 0; ce == cudaSuccess && i < N / half; ++i) {
      ce = cudaMemcpy(static_cast<uint8_t*>(dst) + (2 * i) * blk, static_cast<const uint8_t*>(a) + i * blk,
                      static_cast<size_t>(blk), cudaMemcpyDefault);
      if (ce == cudaSuccess)
        ce = cudaMemcpy(static_cast<uint8_t*>(dst) + (2 * i + 1) * blk, static_cast<const uint8_t*>(b) + i * blk,
                        static_cast<size_t>(blk), cudaMemcpyDefault);
    }
    return ce;
  };
  cudaError_t e = dev_alloc(&inter, static_cast<size_t>(2 * N * row_bytes));
  if (e == cudaSuccess) e = interleave(inter, packed_gate, packed_up, row_bytes);
  if (e == cudaSuccess && row_cb) e = dev_alloc(&inter_cb, static_cast<size_t>(2 * N * 16 * 4));
  if (e == cudaSuccess && row_cb) e = interleave(inter_cb, codebooks_gate, codebooks_up, 16 * 4);
  // one codebook per matrix: the gate's, then the up's (the kernels' two tables)
  const size_t cb1 = 2 * static_cast<size_t>(ops->cb_entries);
  if (e == cudaSuccess && !row_cb && has_cb) e = dev_alloc(&inter_cb, 2 * cb1);
  if (e == cudaSuccess && !row_cb && has_cb) e = cudaMemcpy(inter_cb, codebooks_gate, cb1, cudaMemcpyDefault);
  if (e == cudaSuccess && !row_cb && has_cb)
    e = cudaMemcpy(static_cast<uint8_t*>(inter_cb) + cb1, codebooks_up, cb1, cudaMemcpyDefault);
  if (e != cudaSuccess) {
    cudaFree(inter);
    cudaFree(inter_cb);
    if (e == cudaErrorMemoryAllocation) {
      cudaGetLastError();
      set_error(QGEMV_ERR_NOMEM, "interleaving gate and up: out of device memory");
    } else {
      cuda_error(e, "interleaving gate and up");
    }
    return nullptr;
  }
  const int64_t rows[1] = {2 * N};
  qgemv_handle h = create_impl(format, 2 * N, K, inter, nullptr, inter_cb, 1, rows, true, true);
  cudaFree(inter);
  cudaFree(inter_cb);
  return h;
}

static bool valid(qgemv_handle h) { return h && h->magic == kMagic; }

}  // extern "C"

// Kernel parameters of a run of handle h.
static qgemv::RunParams params_of(const qgemv_ctx* h, const void* x, float* y, const float* residual) {
  qgemv::RunParams p;
  p.tiles = h->tiles;
  p.x = static_cast<const __half*>(x);
  p.y = y;
  p.partials = h->partials;
  p.plan = h->plan;
  p.seg_of_rt = h->seg_of_rt;
  p.err = h->err;
  p.aux = h->aux;
  p.N = h->N;
  p.K = h->K;
  p.T = h->T;
  p.nKT = h->nKT;
  p.skip_cta = h->skip_cta;
  p.residual = residual;
  p.x_scale = nullptr;
  p.x_qsum = nullptr;
  p.xq_ws = h->xq_ws;
  return p;
}

static int check_run_args(qgemv_handle h, const void* x, int M, float* y, const float* residual) {
  if (!valid(h)) return set_error(QGEMV_ERR_ARG, "invalid handle");
  if (M < 1 || M > qgemv::kMaxM) return set_error(QGEMV_ERR_ARG, "M=%d outside [1, 16]", M);
  if (!x || !y) return set_error(QGEMV_ERR_ARG, "x or y is NULL");
  if ((reinterpret_cast<uintptr_t>(x) & 3) || (reinterpret_cast<uintptr_t>(y) & 3) ||
      (reinterpret_cast<uintptr_t>(residual) & 3))
    return set_error(QGEMV_ERR_ALIGN, "x, y and residual must be 4-byte aligned");
  return QGEMV_OK;
}

// Both run calls; `residual` is null for qgemv_run.
static int run_impl(qgemv_handle h, const void* x, int M, float* y, const float* residual, void* stream) {
  const int rc = check_run_args(h, x, M, y, residual);
  if (rc != QGEMV_OK) return rc;
  if (h->glu) {
    if (residual) return set_error(QGEMV_ERR_ARG, "a GLU handle takes no residual");
    const qgemv::RunParams p = params_of(h, x, y, nullptr);
    const qgemv::LaunchGeom g = {h->grid, h->plan, h->grid_m1, h->plan_m1, 0, 0};
    const cudaError_t e = h->ops->launch_glu(M, p, g, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "launching the GEMV kernel");
    return ok();
  }
  const bool inv = h->batch_invariant != 0;
  if (h->mma && (M >= kAqlmMmaMinM || inv)) h = h->mma;  // AQLM: the tensor-core layout
  const qgemv::RunParams p = params_of(h, x, y, residual);
  const qgemv::LaunchGeom g = {h->grid, h->plan, h->grid_m1, h->plan_m1, h->grid_rg, h->tc5_min_m};
  cudaError_t e = h->x_int8 ? h->ops->launch_x_int8(M, p, g, static_cast<cudaStream_t>(stream), inv)
                            : h->ops->launch(M, p, g, static_cast<cudaStream_t>(stream), inv);
  if (e != cudaSuccess) return cuda_error(e, "launching the GEMV kernel");
  return ok();
}

extern "C" {

int qgemv_run(qgemv_handle h, const void* x, int M, float* y, void* stream) {
  return run_impl(h, x, M, y, nullptr, stream);
}

int qgemv_run_residual(qgemv_handle h, const void* x, int M, float* y, const float* residual, void* stream) {
  if (!residual) return set_error(QGEMV_ERR_ARG, "residual is NULL");
  return run_impl(h, x, M, y, residual, stream);
}

int qgemv_set_batch_invariant(qgemv_handle h, int on) {
  if (!valid(h)) return set_error(QGEMV_ERR_ARG, "invalid handle");
  h->batch_invariant = on ? 1 : 0;
  return ok();
}

int qgemv_set_x_int8(qgemv_handle h, int on) {
  if (!valid(h)) return set_error(QGEMV_ERR_ARG, "invalid handle");
  if (h->ops->launch_x_int8 == nullptr || h->glu)
    return set_error(QGEMV_ERR_ARG, "INT8 activations need a PQ2_0 handle without GLU (format %d)", h->format);
  if (on && h->xq_ws == nullptr) {  // the prologue's workspace for runs of several rows
    void* ws = nullptr;
    const cudaError_t e = cudaMalloc(&ws, static_cast<size_t>(qgemv_xq_bytes(qgemv::kMaxM, h->K)));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return set_error(QGEMV_ERR_NOMEM, "INT8 activation workspace: %s", cudaGetErrorString(e));
    }
    h->xq_ws = static_cast<uint8_t*>(ws);
  }
  h->x_int8 = on ? 1 : 0;
  return ok();
}

int64_t qgemv_xq_bytes(int M, int64_t K) {
  if (M < 1 || K <= 0 || K % 128) return 0;
  return int64_t(M) * K + 8 * int64_t(M) * (K / 128);
}

int qgemv_prepare_x_int8(const void* x, int M, int64_t K, const int8_t* signs, int hadamard_block, void* xq,
                         void* stream) {
  if (!x || !xq) return set_error(QGEMV_ERR_ARG, "x or xq is NULL");
  if (M < 1 || K <= 0 || K % 128) return set_error(QGEMV_ERR_ARG, "M must be >= 1 and K a positive multiple of 128");
  if (hadamard_block != 0 && hadamard_block != 1024)
    return set_error(QGEMV_ERR_ARG, "hadamard_block must be 0 or 1024 (got %d)", hadamard_block);
  if (hadamard_block != 0 && K % hadamard_block)
    return set_error(QGEMV_ERR_ARG, "K=%lld is not a multiple of the Hadamard block", (long long)K);
  if (hadamard_block == 0 && signs)
    return set_error(QGEMV_ERR_ARG, "signs apply only with the Hadamard mixing");
  if ((reinterpret_cast<uintptr_t>(x) & 3) || (reinterpret_cast<uintptr_t>(xq) & 3))
    return set_error(QGEMV_ERR_ALIGN, "x and xq must be 4-byte aligned");
  cudaError_t e = qgemv::prepare_x_int8(x, M, K, signs, hadamard_block, xq, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "launching the activation prologue");
  return ok();
}

int qgemv_run_xq(qgemv_handle h, const void* xq, int M, float* y, const float* residual, void* stream) {
  const int rc = check_run_args(h, xq, M, y, residual);
  if (rc != QGEMV_OK) return rc;
  if (h->ops->launch_xq == nullptr || h->glu)
    return set_error(QGEMV_ERR_ARG, "prepared INT8 activations need a PQ2_0 handle without GLU (format %d)",
                     h->format);
  qgemv::RunParams p = params_of(h, xq, y, residual);
  const uint8_t* base = static_cast<const uint8_t*>(xq);
  p.x_scale = reinterpret_cast<const float*>(base + int64_t(M) * h->K);
  p.x_qsum = reinterpret_cast<const int32_t*>(base + int64_t(M) * h->K + 4 * int64_t(M) * (h->K / 128));
  const qgemv::LaunchGeom g = {h->grid, h->plan, h->grid_m1, h->plan_m1, h->grid_rg, 0};
  cudaError_t e = h->ops->launch_xq(M, p, g, static_cast<cudaStream_t>(stream), h->batch_invariant != 0);
  if (e != cudaSuccess) return cuda_error(e, "launching the GEMV kernel");
  return ok();
}

int qgemv_quantize_x_int8(const void* x, int M, int64_t K, int8_t* q_out, float* a_out, void* stream) {
  if (!x || !q_out || !a_out) return set_error(QGEMV_ERR_ARG, "x, q_out or a_out is NULL");
  if (M < 1 || K <= 0 || K % 128) return set_error(QGEMV_ERR_ARG, "M must be >= 1 and K a positive multiple of 128");
  if ((reinterpret_cast<uintptr_t>(x) & 1) || (reinterpret_cast<uintptr_t>(a_out) & 3))
    return set_error(QGEMV_ERR_ALIGN, "x must be 2-byte and a_out 4-byte aligned");
  cudaError_t e = qgemv::quantize_x_int8(x, M, K, q_out, a_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "launching the activation quantizer");
  return ok();
}

int qgemv_dequant(qgemv_handle h, float* w_out, void* stream) {
  if (!valid(h)) return set_error(QGEMV_ERR_ARG, "invalid handle");
  if (!w_out) return set_error(QGEMV_ERR_ARG, "w_out is NULL");
  cudaError_t e = h->ops->dequant(h->tiles, h->aux, h->seg_of_rt, h->N, h->K, h->nKT, w_out,
                                  h->glu && h->ops->cb_entries > 0 && !h->ops->row_tables,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "launching the decode kernel");
  return ok();
}

int qgemv_quantize_q4_0(const float* w, int64_t N, int64_t K, void* packed_out, void* stream) {
  if (!w || !packed_out) return set_error(QGEMV_ERR_ARG, "w or packed_out is NULL");
  if (N <= 0 || K <= 0 || K % 32) return set_error(QGEMV_ERR_ARG, "K must be a positive multiple of 32");
  cudaError_t e = qgemv::quantize_q4_0(w, N, K, static_cast<uint8_t*>(packed_out),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "launching the quantizer");
  return ok();
}

int qgemv_status(qgemv_handle h) {
  if (!valid(h)) return set_error(QGEMV_ERR_ARG, "invalid handle");
  cudaError_t e = cudaDeviceSynchronize();
  int err = 0;
  for (qgemv_ctx* k = h; k != nullptr && e == cudaSuccess; k = k->mma) {  // the handle and its companion
    int ek = 0;
    e = cudaMemcpy(&ek, k->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && ek) {
      // A run that gave up may have left partial slots written but unread.
      cudaMemset(k->partials, 0xff,
                 sizeof(float) * 2 * k->ops->partial_stride *
                     static_cast<size_t>(k->grid > k->grid_m1 ? k->grid : k->grid_m1));
      cudaMemset(k->err, 0, sizeof(int));
      err |= ek;
    }
  }
  if (e != cudaSuccess) return cuda_error(e, "reading the kernel status");
  if (err) {
    if (err & 4)
      return set_error(QGEMV_ERR_CUDA, "a kernel found its shared-memory window unusable (code %d)", err);
    return set_error(QGEMV_ERR_TIMEOUT, "a kernel gave up a bounded wait (code %d)", err);
  }
  return ok();
}

void qgemv_destroy(qgemv_handle h) {
  if (!valid(h)) return;
  cudaDeviceSynchronize();
  free_handle(h);
}

int qgemv_stream_k_plan(int64_t units, int grid, int64_t units_per_row_tile, int rows, int split_unit,
                        int64_t* out) {
  if (units <= 0 || grid <= 0 || units_per_row_tile <= 0 || rows <= 0 || out == nullptr ||
      units % units_per_row_tile != 0 || grid > units || split_unit < 0 || split_unit > 2)
    return set_error(QGEMV_ERR_ARG, "qgemv_stream_k_plan: bad sizes");
  const std::vector<qgemv::CtaPlan> plan = plan_stream_k(units, grid, units_per_row_tile, rows, split_unit);
  for (int c = 0; c < grid; ++c) {
    const qgemv::CtaPlan& pl = plan[static_cast<size_t>(c)];
    int64_t* o = out + static_cast<int64_t>(c) * 12;
    for (int s = 0; s < 2; ++s) {
      o[0 + s] = pl.seg_rt[s];
      o[2 + s] = pl.seg_cf[s];
      o[4 + s] = pl.seg_S[s];
      o[6 + s] = pl.seg_r0[s];
      o[8 + s] = pl.seg_nr[s];
      o[10 + s] = pl.seg_flags[s];
    }
  }
  return ok();
}

const char* qgemv_last_error(void) { return g_msg; }

int qgemv_last_error_code(void) { return g_code; }

}  // extern "C"

// A handle's device buffers, its companion's, and the handle itself.
static void free_handle(qgemv_ctx* h) {
  if (h->mma) free_handle(h->mma);
  cudaFree(h->tiles);
  cudaFree(h->aux);
  cudaFree(h->partials);
  cudaFree(h->plan);
  cudaFree(h->err);
  cudaFree(h->xq_ws);
  h->magic = 0;
  delete h;
}

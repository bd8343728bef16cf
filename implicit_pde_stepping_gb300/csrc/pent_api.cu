// C ABI of libpent: argument checks, plan lifecycle and dispatch to the kernels.
// Every declaration is documented in include/pent.h.
#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>
#include <cstring>
#include <new>

#include "pent_internal.cuh"

namespace pent {

static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
std::mutex g_prep_mu;
std::map<std::pair<const void*, int>, size_t> g_prep_smem;                 // limit set so far
std::map<std::tuple<const void*, int, size_t, int>, int> g_prep_occ;       // CTAs per SM
}  // namespace

cudaError_t kernel_prepare(const void* fn, size_t smem, int threads, int* per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_prep_mu);
  size_t& cur = g_prep_smem[{fn, dev}];
  if (smem > cur) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cur = smem;
  }
  if (per_sm) {
    const auto key = std::make_tuple(fn, dev, smem, threads);
    auto it = g_prep_occ.find(key);
    if (it == g_prep_occ.end()) {
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
      if (e != cudaSuccess) return e;
      it = g_prep_occ.emplace(key, n).first;
    }
    *per_sm = it->second;
  }
  return cudaSuccess;
}

namespace {

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline pent_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return PENT_OK;
  if (e == cudaErrorMemoryAllocation) return PENT_ERR_ALLOC;
  return PENT_ERR_CUDA;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Largest sweep length whose double-float tables fit in one CTA's shared memory.
constexpr int kMaxTwistedRows = 2560;

// The kernel variant a plan uses for `batch` systems.  fp64 plans run in
// double-float, and AUTO only picks kernels that keep the whole fp64 range
// (each system scaled by a power of two before it is converted): the
// fixed-grid partitioned kernel for non-cyclic plans that have its tables (at
// N = 1024, batch 65536: 0.329 ms, against 0.333 ms for the twisted kernel
// with twice the memory traffic), else the TwoSum partitioned kernels (one CTA
// per group of systems, or the multi-kernel form for long systems), else the
// native kernel.  The twisted kernel (PENT_VARIANT_THREAD_DF) runs only on
// request: it writes g over f as it goes and cannot rescale a system it has
// already started.
pent_variant resolve(const pent_plan_s& p, int batch) {
  (void)batch;
  if (p.variant != PENT_VARIANT_AUTO) return p.variant;
  if (p.dtype != PENT_F64) return PENT_VARIANT_THREAD;
  if (p.fg_ok && p.fg_use && p.sp_T > 0) return PENT_VARIANT_SPLIT;
  if (p.split_ok || p.split_big) return PENT_VARIANT_SPLIT;
  return PENT_VARIANT_THREAD;
}

// The twisted variant's tables, made once, synchronously, on the plan's
// device (its bands and plan-time scratch live in the arena).
cudaError_t ensure_twisted(pent_plan_s& p) {
  if (!p.twist_eligible || p.twist_built) return cudaSuccess;
  int tstatus = 0;
  cudaError_t e = factor_twisted(p.bands, p.N, p.cyclic, p.m, p.twtab, p.twist, p.work_area, p.status_area, 0);
  if (e == cudaSuccess) e = cudaMemcpy(&tstatus, p.status_area, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  p.twist_ok = (tstatus == 0);
  p.twist_built = 1;
  return cudaSuccess;
}

bool variant_exists(const pent_plan_s& p, pent_variant v) {
  switch (v) {
    case PENT_VARIANT_AUTO:
    case PENT_VARIANT_THREAD:
      return true;
    case PENT_VARIANT_THREAD_DF:
      return p.dtype == PENT_F64 && p.twist_ok;
    case PENT_VARIANT_SPLIT:
      return p.dtype == PENT_F64 && (p.split_ok || p.split_big);
    default:
      return false;
  }
}

// Whether nsteps of scheme `kind` run in the persistent multi-step kernel:
// two or more steps, the default or partitioned variant, a plan it supports
// (PENT_OPT_MULTI_STEP = 0 keeps one launch per step).
bool use_steps(const pent_plan_s& p, int nsteps, int kind) {
  if (nsteps < 2) return false;
  if (p.variant != PENT_VARIANT_AUTO && p.variant != PENT_VARIANT_SPLIT) return false;
  if (!p.steps_on) return false;
  return steps_supported(p, kind);
}

// Longest run of consecutive chunks whose row tables (L x kSpK float4) and
// chunk tables (kSpChunk doubles) are bitwise equal to those of the run's first
// chunk; recorded as dup_lo < c <= dup_hi (empty if no two neighbours match).
cudaError_t find_duplicate_chunks(pent_plan_s& p, int Mpad) {
  const int L = p.sp_L, P = p.sp_P;
  std::vector<float4> rows((size_t)Mpad * kSpK);
  std::vector<double> chunks((size_t)P * kSpChunk);
  cudaError_t e = cudaMemcpy(rows.data(), p.sptab, rows.size() * sizeof(float4), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(chunks.data(), p.spchunk, chunks.size() * sizeof(double), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  const size_t rb = (size_t)L * kSpK * sizeof(float4), cb = kSpChunk * sizeof(double);
  auto same = [&](int a, int b) {
    return std::memcmp(&rows[(size_t)a * L * kSpK], &rows[(size_t)b * L * kSpK], rb) == 0 &&
           std::memcmp(&chunks[(size_t)a * kSpChunk], &chunks[(size_t)b * kSpChunk], cb) == 0;
  };
  int best_lo = 0, best_hi = 0;
  for (int c = 1; c < P;) {
    if (!same(c - 1, c)) { ++c; continue; }
    const int lo = c - 1;
    while (c < P && same(lo, c)) ++c;
    if (c - 1 - lo > best_hi - best_lo) { best_lo = lo; best_hi = c - 1; }
  }
  p.dup_lo = best_lo;
  p.dup_hi = best_hi;
  return cudaSuccess;
}

// 8-row groups whose correction responses are below 2^-24 in every chunk (see
// pent_plan_s::cheap_k, cheap_m).  M1, M2 decay away from a chunk's start and K1, K2
// towards it, so the groups found are a prefix (K) and a suffix (M) of the chunk.
cudaError_t find_cheap_groups(pent_plan_s& p, int Mpad) {
  const int L = p.sp_L, P = p.sp_P, G = L / 8;
  std::vector<float4> rows((size_t)Mpad * kSpK);
  cudaError_t e = cudaMemcpy(rows.data(), p.sptab, rows.size() * sizeof(float4), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  std::vector<float> mM(L, 0.f), mK(L, 0.f);
  for (int c = 0; c < P; ++c)
    for (int j = 0; j < L; ++j) {
      const float4 m = rows[((size_t)c * L + j) * kSpK + 3], k = rows[((size_t)c * L + j) * kSpK + 4];
      mM[j] = std::max(mM[j], std::max(std::fabs(m.x), std::fabs(m.z)));
      mK[j] = std::max(mK[j], std::max(std::fabs(k.x), std::fabs(k.z)));
    }
  auto small = [&](const std::vector<float>& v, int g) {
    for (int j = 8 * g; j < 8 * g + 8; ++j)
      if (!(v[j] < 0x1p-24f)) return false;
    return true;
  };
  int gk = 0, gm = G;
  while (gk < G && small(mK, gk)) ++gk;
  while (gm > 0 && small(mM, gm - 1)) --gm;
  p.cheap_k = gk;
  p.cheap_m = gm;
  return cudaSuccess;
}

}  // namespace

// The solve kernel of the plan's variant for `batch` systems, in place on a
// device array with leading dimension batch.
cudaError_t solve_device(pent_plan_s& p, void* rhs, int batch, cudaStream_t st) {
  const pent_variant v = resolve(p, batch);
  if (p.dtype == PENT_F32) return shared_thread_f32(p, static_cast<float*>(rhs), batch, st);
  switch (v) {
    case PENT_VARIANT_THREAD: return shared_thread_f64(p, static_cast<double*>(rhs), batch, st);
    case PENT_VARIANT_THREAD_DF: return shared_twisted_df(p, static_cast<double*>(rhs), batch, st);
    case PENT_VARIANT_SPLIT:
      if (p.fg_ok && p.fg_use && p.sp_T > 0) return shared_fg(p, static_cast<double*>(rhs), batch, st);
      return p.split_ok ? shared_split_df(p, static_cast<double*>(rhs), batch, st)
                        : shared_split_big(p, static_cast<double*>(rhs), batch, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pent

using namespace pent;

extern "C" {

const char* pent_status_string(pent_status s) {
  switch (s) {
    case PENT_OK: return "PENT_OK";
    case PENT_ERR_INVALID_ARG: return "PENT_ERR_INVALID_ARG";
    case PENT_ERR_ZERO_PIVOT: return "PENT_ERR_ZERO_PIVOT";
    case PENT_ERR_CUDA: return "PENT_ERR_CUDA";
    case PENT_ERR_ALLOC: return "PENT_ERR_ALLOC";
    case PENT_ERR_UNSUPPORTED: return "PENT_ERR_UNSUPPORTED";
  }
  return "PENT_ERR_UNKNOWN";
}

unsigned long long pent_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

pent_status pent_sync(void* stream) {
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  return from_cuda(e);
}

void pent_destroy(pent_plan p) {
  if (!p) return;
  host_pipeline_release(*p);
  if (p->spsum) cudaFree(p->spsum);
  if (p->arena) cudaFree(p->arena);
  delete p;
}

pent_status pent_factor(const double* bands_host, int N, int batch, int cyclic, pent_dtype dtype,
                        pent_plan* out) {
  if (!out) return PENT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!bands_host || N < 1 || batch < 1 || (cyclic != 0 && cyclic != 1)) return PENT_ERR_INVALID_ARG;
  if (dtype != PENT_F64 && dtype != PENT_F32) return PENT_ERR_INVALID_ARG;
  if (cyclic && N < 5) return PENT_ERR_INVALID_ARG;
  if (N > (1 << 26)) return PENT_ERR_UNSUPPORTED;

  pent_plan_s* p = new (std::nothrow) pent_plan_s;
  if (!p) return PENT_ERR_ALLOC;
  p->N = N;
  p->M = cyclic ? N - 2 : N;
  p->batch = batch;
  p->cyclic = cyclic;
  p->dtype = dtype;
  cudaGetDevice(&p->device);

  // one arena: coef64 | tail64 | coef32 | tail32 | coefdf | taildf | bands | work | status
  const size_t nc = (size_t)kCoefCount * p->M;
  size_t off = 0;
  const size_t o_coef64 = off; off = round_up(off + nc * sizeof(double), 256);
  const size_t o_tail64 = off; off = round_up(off + kTailCount * sizeof(double), 256);
  const size_t o_coef32 = off; off = round_up(off + nc * sizeof(float), 256);
  const size_t o_tail32 = off; off = round_up(off + kTailCount * sizeof(float), 256);
  const size_t o_coefdf = off; off = round_up(off + nc * sizeof(float2), 256);
  const size_t o_taildf = off; off = round_up(off + kTailCount * sizeof(float2), 256);
  const size_t o_bands = off; off = round_up(off + 5 * (size_t)N * sizeof(double), 256);
  // partitioned variant: chunk length and count (P a multiple of 4, Mpad = L * P)
  const int spL = p->M >= 256 ? 32 : 16;
  const int spP = ((p->M + 4 * spL - 1) / (4 * spL)) * 4;
  const size_t Mpad = (size_t)spL * spP;
  // work: the partitioned tables' scratch (17 rows of Mpad), then the shared factor's
  // (4 rows of M), so that the two factor kernels can run at once
  const size_t wrow = Mpad > (size_t)p->M ? Mpad : (size_t)p->M;
  const size_t o_work = off; off = round_up(off + 22 * wrow * sizeof(double), 256);
  const size_t o_sptab = off; off = round_up(off + Mpad * kSpK * sizeof(float4), 256);
  const size_t o_spchunk = off; off = round_up(off + (size_t)spP * kSpChunk * sizeof(double), 256);
  const size_t o_spchunkdf = off; off = round_up(off + (size_t)spP * kSpChunk * sizeof(float2), 256);
  const size_t o_spextra = off; off = round_up(off + kSpExtra * sizeof(double), 256);
  const size_t o_status = off; off = round_up(off + 2 * sizeof(int), 256);
  const size_t o_kerr = off; off = round_up(off + sizeof(int), 256);
  const size_t o_sched = off; off = round_up(off + 2 * sizeof(unsigned), 256);
  const size_t o_twtab = off; off = round_up(off + (size_t)p->M * kTwK * sizeof(float4), 256);
  const size_t o_twist = off; off = round_up(off + kTwistCount * sizeof(double), 256);
  char* arena = nullptr;
  cudaError_t e = cudaMalloc(&arena, off);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return PENT_ERR_ALLOC;
  }
  p->arena = arena;
  p->coef64 = reinterpret_cast<double*>(arena + o_coef64);
  p->tail64 = reinterpret_cast<double*>(arena + o_tail64);
  p->coef32 = reinterpret_cast<float*>(arena + o_coef32);
  p->tail32 = reinterpret_cast<float*>(arena + o_tail32);
  p->coefdf = reinterpret_cast<float2*>(arena + o_coefdf);
  p->taildf = reinterpret_cast<float2*>(arena + o_taildf);
  p->twtab = reinterpret_cast<float4*>(arena + o_twtab);
  p->twist = reinterpret_cast<double*>(arena + o_twist);
  p->sptab = reinterpret_cast<float4*>(arena + o_sptab);
  p->spchunk = reinterpret_cast<double*>(arena + o_spchunk);
  p->spchunk_df = reinterpret_cast<float2*>(arena + o_spchunkdf);
  p->spextra = reinterpret_cast<double*>(arena + o_spextra);
  double* d_bands = reinterpret_cast<double*>(arena + o_bands);
  p->bands = d_bands;
  double* d_work = reinterpret_cast<double*>(arena + o_work);
  int* d_status = reinterpret_cast<int*>(arena + o_status);
  p->kern_err = reinterpret_cast<int*>(arena + o_kerr);
  p->sched = reinterpret_cast<unsigned*>(arena + o_sched);

  int status = 0;
  // The two factorisations (the native tables and the partitioned ones) are serial
  // sweeps of one thread or one CTA each; they run at once on two streams, each
  // with its own scratch and status word.
  const bool split_tables = dtype == PENT_F64 && p->M >= 16;
  int* d_status_split = d_status + 1;
  cudaStream_t fs[2] = {nullptr, nullptr};
  e = cudaMemset(arena, 0, off);
  if (e == cudaSuccess)
    e = cudaMemcpy(d_bands, bands_host, 5 * (size_t)N * sizeof(double), cudaMemcpyHostToDevice);
  // the non-blocking streams do not wait for the default stream's memset and copy
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  for (auto& q : fs)
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking);
  if (e == cudaSuccess)
    e = factor_shared(d_bands, N, cyclic, p->coef64, p->tail64, d_work + 18 * wrow, d_status, fs[0]);
  if (e == cudaSuccess)
    e = pack_coefficients(p->coef64, p->tail64, (int)nc, p->coef32, p->tail32, p->coefdf, p->taildf, fs[0]);
  if (e == cudaSuccess && split_tables)
    e = factor_split(d_bands, N, cyclic, spL, (int)Mpad, p->sptab, p->spchunk, p->spextra, d_work,
                     d_status_split, fs[1]);
  for (auto& q : fs)
    if (q) {
      const cudaError_t es = cudaStreamSynchronize(q);
      if (e == cudaSuccess) e = es;
      cudaStreamDestroy(q);
    }
  if (e == cudaSuccess) e = cudaMemcpy(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    cudaGetLastError();
    pent_destroy(p);
    return from_cuda(e);
  }
  if (status != 0) {
    pent_destroy(p);
    return PENT_ERR_ZERO_PIVOT;
  }
  // twisted double-float tables (fp64 plans whose sweep fits the kernel): made
  // when that variant is first selected, since the default path never uses them
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  p->work_area = d_work;
  p->status_area = d_status;
  if (dtype == PENT_F64 && p->M >= 8 && p->M <= kMaxTwistedRows) {
    p->m = p->M / 2;
    p->twist_eligible = 1;
  }
  // partitioned double-float tables
  {
    const int SB = (cyclic && spL == 32 && spP <= 32) ? 16 : 8;
    const bool fits = split_smem_bytes(spL, spP, SB, cyclic) <= 200 * 1024 && SB * spP <= 1024 && spP <= kSpMaxChunks &&
                      !(cyclic && spL == 32 && spP > 32);
    // tables for every fp64 plan of 16 rows or more: one kernel (tables in shared
    // memory) where they fit, else the two-kernel form for long systems
    if (split_tables) {
      p->sp_L = spL;
      p->sp_P = spP;
      int sstatus = 0;
      // the tables were made above, alongside the native factorisation
      e = cudaMemcpy(&sstatus, d_status_split, sizeof(int), cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) {
        cudaGetLastError();
        pent_destroy(p);
        return from_cuda(e);
      }
      const bool tables = (sstatus == 0);
      p->split_ok = tables && fits;
      if (tables) {
        double ex[2] = {0.0, 0.0};
        e = cudaMemcpy(ex, p->spextra + 18, sizeof(ex), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pent_destroy(p);
          return from_cuda(e);
        }
        p->sp_T = p->sp_T0 = (int)ex[0];
        p->reach0 = (int)ex[1];
        // the two-kernel form needs the truncated chunk couplings
        p->split_big = !fits && p->sp_T > 0;
      }
      // the chunk tables as double-float pairs, for the kernels that run the chunk
      // scan on the FP32 pipe (the two-kernel form, the partitioned one-step kernels
      // and the multi-step kernel)
      if (p->split_big || p->split_ok) {
        e = split_big_prepare(*p, 0);
        if (e == cudaSuccess) e = cudaStreamSynchronize(0);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pent_destroy(p);
          return from_cuda(e);
        }
      }
      // fixed-grid partitioned kernel: grid and correction groups
      if (tables) {
        e = fg_prepare(*p);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pent_destroy(p);
          return from_cuda(e);
        }
      }
      // correction-term groups of the multi-step kernel
      if (p->split_ok && p->sp_L % 8 == 0) {
        e = find_cheap_groups(*p, (int)Mpad);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pent_destroy(p);
          return from_cuda(e);
        }
        p->cheap_k0 = p->cheap_k;
        p->cheap_m0 = p->cheap_m;
      }
      // chunks with equal tables share one copy (long systems: in cache; the
      // multi-step kernel: one shared-memory slot)
      if (p->split_big || p->split_ok) {
        e = find_duplicate_chunks(*p, (int)Mpad);
        if (e != cudaSuccess) {
          cudaGetLastError();
          pent_destroy(p);
          return from_cuda(e);
        }
        p->dup_lo0 = p->dup_lo;
        p->dup_hi0 = p->dup_hi;
      }
    }
  }
  *out = p;
  return PENT_OK;
}

pent_status pent_set_variant(pent_plan p, pent_variant v) {
  if (!p) return PENT_ERR_INVALID_ARG;
  if (v == PENT_VARIANT_THREAD_DF) {
    const cudaError_t e = ensure_twisted(*p);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (!variant_exists(*p, v)) return PENT_ERR_UNSUPPORTED;
  p->variant = v;
  return PENT_OK;
}

pent_status pent_set_option(pent_plan p, pent_option opt, int v) {
  if (!p) return PENT_ERR_INVALID_ARG;
  auto in = [v](std::initializer_list<int> ok) {
    for (int o : ok)
      if (v == o) return true;
    return false;
  };
  auto put = [&](int k, double val) {
    cudaError_t e = cudaMemcpy(p->spextra + k, &val, sizeof(double), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) cudaGetLastError();
    return from_cuda(e);
  };
  switch (opt) {
    case PENT_OPT_FIXED_GRID:
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      p->fg_use = v;
      return PENT_OK;
    case PENT_OPT_SERIAL_CHUNK_SCAN: {
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      if (!p->split_ok) return p->split_big ? PENT_ERR_UNSUPPORTED : PENT_OK;
      const int T = v ? 0 : p->sp_T0;
      const pent_status st = put(18, (double)T);
      if (st == PENT_OK) p->sp_T = T;
      return st;
    }
    case PENT_OPT_BORDER_ALL_CHUNKS:
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      if (!p->cyclic || !(p->split_ok || p->split_big)) return PENT_OK;
      return put(19, v ? (double)p->sp_P : (double)p->reach0);
    case PENT_OPT_MULTI_STEP:
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      p->steps_on = v;
      return PENT_OK;
    case PENT_OPT_CHEAP_TERMS:
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      p->cheap_k = v ? p->cheap_k0 : 0;
      p->cheap_m = v ? p->cheap_m0 : 1 << 20;
      return PENT_OK;
    case PENT_OPT_CHUNK_DEDUP:
      if (!in({0, 1})) return PENT_ERR_INVALID_ARG;
      p->dup_lo = v ? p->dup_lo0 : 0;
      p->dup_hi = v ? p->dup_hi0 : 0;
      return PENT_OK;
    case PENT_OPT_TWISTED_RING:
      if (!in({0, 4, 6, 8, 12})) return PENT_ERR_INVALID_ARG;
      p->df_async = v;
      return PENT_OK;
    case PENT_OPT_STEPS_SYSTEMS:
      if (!in({0, 8, 16})) return PENT_ERR_INVALID_ARG;
      p->steps_sb = v;
      return PENT_OK;
    case PENT_OPT_TWISTED_SYSTEMS_PER_CTA:
      if (!in({64, 128, 160, 256, 320})) return PENT_ERR_INVALID_ARG;
      p->df_spb = v;
      return PENT_OK;
    case PENT_OPT_TWISTED_SYSTEMS_PER_THREAD:
      if (!in({1, 2})) return PENT_ERR_INVALID_ARG;
      p->df_spt = v;
      return PENT_OK;
    case PENT_OPT_TWISTED_PREFETCH_ROWS:
      if (!in({4, 8})) return PENT_ERR_INVALID_ARG;
      p->df_ku = v;
      return PENT_OK;
    case PENT_OPT_PERSISTENT_CTAS:
      if (v < 0) return PENT_ERR_INVALID_ARG;
      p->df_ctas = v;
      return PENT_OK;
  }
  return PENT_ERR_INVALID_ARG;
}

pent_status pent_plan_error(pent_plan p) {
  if (!p) return PENT_ERR_INVALID_ARG;
  int v = 0;
  const cudaError_t e = cudaMemcpy(&v, p->kern_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return from_cuda(e);
  }
  return v ? PENT_ERR_CUDA : PENT_OK;
}

pent_variant pent_get_variant(pent_plan p, int batch) {
  if (!p) return PENT_VARIANT_AUTO;
  return resolve(*p, batch);
}

pent_status pent_solve(pent_plan p, void* rhs, int batch, void* stream) {
  if (!p || !rhs || batch < 1) return PENT_ERR_INVALID_ARG;
  if (!aligned(rhs, 16)) return PENT_ERR_INVALID_ARG;
  if (p->dtype == PENT_F32 && resolve(*p, batch) != PENT_VARIANT_THREAD) return PENT_ERR_UNSUPPORTED;
  return from_cuda(solve_device(*p, rhs, batch, as_stream(stream)));
}

pent_status pent_solve_host(pent_plan p, const void* rhs_host, void* x_host, int batch, int chunks,
                            void* stream) {
  if (!p || !rhs_host || !x_host || batch < 1 || chunks < 0) return PENT_ERR_INVALID_ARG;
  if (p->dtype == PENT_F32 && resolve(*p, batch) != PENT_VARIANT_THREAD) return PENT_ERR_UNSUPPORTED;
  if (chunks == 0) {
    // 2-D copies keep the copy engines at full rate for rows of >= 128 KB, so
    // blocks are at least that wide; at most 8 blocks
    const size_t elem = p->dtype == PENT_F64 ? sizeof(double) : sizeof(float);
    const size_t row_bytes = (size_t)batch * elem;
    chunks = (int)(row_bytes / (128 * 1024));
    chunks = chunks < 1 ? 1 : chunks > 8 ? 8 : chunks;
  }
  return from_cuda(solve_host(*p, rhs_host, x_host, batch, chunks, as_stream(stream), solve_device));
}

size_t pent_factor_solve_work_bytes(int N, int batch, pent_dtype dtype) {
  if (N < 1 || batch < 1 || (dtype != PENT_F64 && dtype != PENT_F32)) return 0;
  return persys_work_bytes(N, batch, dtype);
}

pent_status pent_factor_solve_ex(const void* a, const void* b, const void* c, const void* d,
                                 const void* e, void* rhs, int N, int batch, pent_dtype dtype,
                                 pent_variant variant, int block_size, void* work, size_t work_bytes,
                                 int* info, void* stream) {
  if (!a || !b || !c || !d || !e || !rhs || N < 1 || batch < 1) return PENT_ERR_INVALID_ARG;
  if (block_size < 0 || (block_size > 0 && batch % block_size != 0)) return PENT_ERR_INVALID_ARG;
  if (dtype != PENT_F64 && dtype != PENT_F32) return PENT_ERR_INVALID_ARG;
  const void* ptrs[6] = {a, b, c, d, e, rhs};
  for (const void* q : ptrs)
    if (!aligned(q, 16)) return PENT_ERR_INVALID_ARG;
  const bool split_ok = dtype == PENT_F32 && persys_split_chunks(N) > 0;
  pent_variant v;
  switch (variant) {
    case PENT_VARIANT_AUTO:
      v = split_ok ? PENT_VARIANT_SPLIT : dtype == PENT_F64 ? PENT_VARIANT_THREAD_DF : PENT_VARIANT_THREAD;
      break;
    case PENT_VARIANT_THREAD: v = variant; break;
    case PENT_VARIANT_THREAD_DF:
      if (dtype != PENT_F64) return PENT_ERR_UNSUPPORTED;
      v = variant;
      break;
    case PENT_VARIANT_SPLIT:
      if (!split_ok) return PENT_ERR_UNSUPPORTED;
      v = variant;
      break;
    default: return PENT_ERR_INVALID_ARG;
  }
  if (v == PENT_VARIANT_SPLIT)
    return from_cuda(persys_split(a, b, c, d, e, rhs, N, batch, block_size, info, as_stream(stream)));
  if (!work || work_bytes < persys_work_bytes(N, batch, dtype) || !aligned(work, 256)) return PENT_ERR_INVALID_ARG;
  if (v == PENT_VARIANT_THREAD_DF)
    return from_cuda(persys_thread_df(a, b, c, d, e, rhs, N, batch, block_size, work, info, as_stream(stream)));
  return from_cuda(persys_thread(a, b, c, d, e, rhs, N, batch, block_size, dtype, work, info,
                                 as_stream(stream)));
}

pent_status pent_factor_solve(const void* a, const void* b, const void* c, const void* d,
                              const void* e, void* rhs, int N, int batch, pent_dtype dtype,
                              void* work, size_t work_bytes, int* info, void* stream) {
  // the scratch is checked where the chosen kernel needs it (pent_factor_solve_ex)
  return pent_factor_solve_ex(a, b, c, d, e, rhs, N, batch, dtype, PENT_VARIANT_AUTO, 0, work, work_bytes,
                              info, stream);
}

size_t pent_factor_solve_needs_work(int N, int batch, pent_dtype dtype) {
  if (N < 1 || batch < 1 || (dtype != PENT_F64 && dtype != PENT_F32)) return 0;
  if (dtype == PENT_F32 && persys_split_chunks(N) > 0) return 0;   // the partitioned kernel keeps all on chip
  return persys_work_bytes(N, batch, dtype);
}

size_t tri_factor_solve_work_bytes(int N, int batch, pent_dtype dtype) {
  if (N < 1 || batch < 1 || (dtype != PENT_F64 && dtype != PENT_F32)) return 0;
  return tri_work_bytes(N, batch, dtype);
}

pent_status tri_factor_solve(const void* a, const void* b, const void* c, void* rhs, int N, int batch,
                             pent_dtype dtype, pent_variant variant, int block_size, void* work,
                             size_t work_bytes, int* info, void* stream) {
  if (!a || !b || !c || !rhs || N < 1 || batch < 1) return PENT_ERR_INVALID_ARG;
  if (block_size < 0 || (block_size > 0 && batch % block_size != 0)) return PENT_ERR_INVALID_ARG;
  if (dtype != PENT_F64 && dtype != PENT_F32) return PENT_ERR_INVALID_ARG;
  const size_t elem = dtype == PENT_F64 ? sizeof(double) : sizeof(float);
  const void* ptrs[4] = {a, b, c, rhs};
  for (const void* q : ptrs)
    if (!aligned(q, elem)) return PENT_ERR_INVALID_ARG;
  const bool split_ok = dtype == PENT_F32 && tri_split_chunks(N) > 0;
  pent_variant v;
  switch (variant) {
    case PENT_VARIANT_AUTO:
      v = split_ok ? PENT_VARIANT_SPLIT : dtype == PENT_F64 ? PENT_VARIANT_THREAD_DF : PENT_VARIANT_THREAD;
      break;
    case PENT_VARIANT_THREAD: v = variant; break;
    case PENT_VARIANT_THREAD_DF:
      if (dtype != PENT_F64) return PENT_ERR_UNSUPPORTED;
      v = variant;
      break;
    case PENT_VARIANT_SPLIT:
      if (!split_ok) return PENT_ERR_UNSUPPORTED;
      v = variant;
      break;
    default: return PENT_ERR_INVALID_ARG;
  }
  if (v != PENT_VARIANT_SPLIT && (!work || work_bytes < tri_work_bytes(N, batch, dtype) || !aligned(work, 256)))
    return PENT_ERR_INVALID_ARG;
  if (v == PENT_VARIANT_THREAD_DF)
    return from_cuda(tri_solve_batch_df(a, b, c, rhs, N, batch, block_size, work, info, as_stream(stream)));
  return from_cuda(tri_solve_batch(a, b, c, rhs, N, batch, block_size, dtype, v == PENT_VARIANT_SPLIT, work, info,
                                   as_stream(stream)));
}

pent_status hyperdiffusion_step(pent_plan p, void* C, int batch, int nsteps, void* stream) {
  if (!p || !C || batch < 1 || nsteps < 0) return PENT_ERR_INVALID_ARG;
  if (!p->cyclic || p->dtype != PENT_F64) return PENT_ERR_INVALID_ARG;
  if (!aligned(C, 16)) return PENT_ERR_INVALID_ARG;
  // the multi-step kernel is arithmetic-bound (~160 instructions per point and
  // step); where the twisted kernel runs the single step it is memory-bound and
  // about twice as fast per step, so many steps use it one launch at a time
  if (resolve(*p, batch) != PENT_VARIANT_THREAD_DF && use_steps(*p, nsteps, 0))
    return from_cuda(steps_df(*p, static_cast<double*>(C), batch, nsteps, 0, 0.0, as_stream(stream)));
  for (int n = 0; n < nsteps; ++n) {
    const pent_status s = pent_solve(p, C, batch, stream);
    if (s != PENT_OK) return s;
  }
  return PENT_OK;
}

pent_status ch_step(pent_plan p, void* C, int batch, double dt_over_dx2, int nsteps, void* stream) {
  if (!p || !C || batch < 1 || nsteps < 0) return PENT_ERR_INVALID_ARG;
  if (!p->cyclic || p->dtype != PENT_F64) return PENT_ERR_INVALID_ARG;
  if (!aligned(C, 16)) return PENT_ERR_INVALID_ARG;
  // the partitioned double-float kernel unless the native one is requested
  const bool use_split = p->split_ok && p->N >= 8 &&
                         (p->variant == PENT_VARIANT_AUTO || p->variant == PENT_VARIANT_SPLIT ||
                          p->variant == PENT_VARIANT_THREAD_DF);
  if (use_steps(*p, nsteps, 1))
    return from_cuda(steps_df(*p, static_cast<double*>(C), batch, nsteps, 1, dt_over_dx2,
                              as_stream(stream)));
  for (int n = 0; n < nsteps; ++n) {
    const cudaError_t e =
        use_split ? ch_split_df(*p, static_cast<double*>(C), batch, dt_over_dx2, as_stream(stream))
                  : ch_thread_f64(*p, static_cast<double*>(C), batch, dt_over_dx2, as_stream(stream));
    if (e != cudaSuccess) return from_cuda(e);
  }
  return PENT_OK;
}

pent_status cn_step(pent_plan p, void* C, int batch, int nsteps, void* stream) {
  if (!p || !C || batch < 1 || nsteps < 0) return PENT_ERR_INVALID_ARG;
  if (!p->cyclic || p->dtype != PENT_F64) return PENT_ERR_INVALID_ARG;
  if (!aligned(C, 16)) return PENT_ERR_INVALID_ARG;
  // the partitioned double-float kernel unless the native one is requested
  const bool use_split = p->split_ok && (p->variant == PENT_VARIANT_AUTO ||
                                         p->variant == PENT_VARIANT_SPLIT ||
                                         p->variant == PENT_VARIANT_THREAD_DF);
  if (use_steps(*p, nsteps, 2))
    return from_cuda(steps_df(*p, static_cast<double*>(C), batch, nsteps, 2, 0.0, as_stream(stream)));
  for (int n = 0; n < nsteps; ++n) {
    const cudaError_t e = use_split ? cn_split_df(*p, static_cast<double*>(C), batch, as_stream(stream))
                                    : cn_thread_f64(*p, static_cast<double*>(C), batch, as_stream(stream));
    if (e != cudaSuccess) return from_cuda(e);
  }
  return PENT_OK;
}

}  // extern "C"

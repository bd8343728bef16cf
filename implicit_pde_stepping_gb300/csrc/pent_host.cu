// pent_solve_host: the shared-matrix solve with the right-hand sides and the
// solutions in host memory, the transfers overlapped with the solves.
//
// The batch is cut into chunks of systems.  Chunk k goes through three
// streams of the plan: a 2-D copy of its [N][w] column block from the host
// array (row pitch batch) into a compact device buffer, the solve of that
// buffer (leading dimension w), and the 2-D copy back.  Three staging buffers
// rotate, so the copy-in of chunk k+1, the solve of chunk k and the copy-out
// of chunk k-1 run at the same time; events order each chunk's three stages
// and the reuse of a buffer.  The caller's stream forks into the three streams
// and joins them at the end, so the call is ordered on the caller's stream like
// any other.
#include "pent_internal.cuh"

namespace pent {

void host_pipeline_release(pent_plan_s& p) {
  for (auto& s : p.hs)
    if (s) cudaStreamDestroy(s), s = nullptr;
  for (int k = 0; k < pent_plan_s::kHostRing; ++k) {
    if (p.hev_in[k]) cudaEventDestroy(p.hev_in[k]), p.hev_in[k] = nullptr;
    if (p.hev_solved[k]) cudaEventDestroy(p.hev_solved[k]), p.hev_solved[k] = nullptr;
    if (p.hev_out[k]) cudaEventDestroy(p.hev_out[k]), p.hev_out[k] = nullptr;
  }
  if (p.hev_fork) cudaEventDestroy(p.hev_fork), p.hev_fork = nullptr;
  if (p.hbuf) cudaFree(p.hbuf), p.hbuf = nullptr;
  p.hbuf_bytes = 0;
}

namespace {

cudaError_t ensure_pipeline(pent_plan_s& p, size_t bytes) {
  cudaError_t e = cudaSuccess;
  if (!p.hs[0]) {
    for (auto& s : p.hs)
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    for (int k = 0; k < pent_plan_s::kHostRing && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&p.hev_in[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.hev_solved[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.hev_out[k], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.hev_fork, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  if (p.hbuf_bytes < bytes) {
    if (p.hbuf) {
      // earlier calls may still use the old buffers
      for (auto& s : p.hs) cudaStreamSynchronize(s);
      cudaFree(p.hbuf);
      p.hbuf = nullptr;
      p.hbuf_bytes = 0;
    }
    e = cudaMalloc(&p.hbuf, bytes * pent_plan_s::kHostRing);
    if (e != cudaSuccess) return e;
    p.hbuf_bytes = bytes;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t solve_host(pent_plan_s& p, const void* in, void* out, int batch, int chunks, cudaStream_t st,
                       cudaError_t (*solve)(pent_plan_s&, void*, int, cudaStream_t)) {
  const size_t elem = p.dtype == PENT_F64 ? sizeof(double) : sizeof(float);
  // chunk width: a multiple of 64 systems (512-byte rows of fp64), at least 64
  long long cw = ((long long)batch + chunks - 1) / chunks;
  cw = (cw + 63) / 64 * 64;
  if (cw > batch) cw = batch;
  const size_t bytes = ((size_t)p.N * (size_t)cw * elem + 255) / 256 * 256;   // keeps every buffer aligned
  cudaError_t e = ensure_pipeline(p, bytes);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(p.hev_fork, st);
  for (auto& s : p.hs)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p.hev_fork, 0);
  const size_t hpitch = (size_t)batch * elem;
  int k = 0;
  for (long long s0 = 0; s0 < batch && e == cudaSuccess; s0 += cw, ++k) {
    const int w = (int)((batch - s0) < cw ? (batch - s0) : cw);
    const int r = k % pent_plan_s::kHostRing;
    char* buf = static_cast<char*>(p.hbuf) + (size_t)r * p.hbuf_bytes;
    const size_t dpitch = (size_t)w * elem;
    if (k >= pent_plan_s::kHostRing) e = cudaStreamWaitEvent(p.hs[0], p.hev_out[r], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(buf, dpitch, static_cast<const char*>(in) + s0 * elem, hpitch, dpitch, p.N,
                            cudaMemcpyHostToDevice, p.hs[0]);
    if (e == cudaSuccess) e = cudaEventRecord(p.hev_in[r], p.hs[0]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.hs[1], p.hev_in[r], 0);
    if (e == cudaSuccess) e = solve(p, buf, w, p.hs[1]);
    if (e == cudaSuccess) e = cudaEventRecord(p.hev_solved[r], p.hs[1]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.hs[2], p.hev_solved[r], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(static_cast<char*>(out) + s0 * elem, hpitch, buf, dpitch, dpitch, p.N,
                            cudaMemcpyDeviceToHost, p.hs[2]);
    if (e == cudaSuccess) e = cudaEventRecord(p.hev_out[r], p.hs[2]);
  }
  // join: the caller's stream waits for the last copy out (which follows every
  // earlier copy out on the same stream)
  if (e == cudaSuccess && k > 0) e = cudaStreamWaitEvent(st, p.hev_out[(k - 1) % pent_plan_s::kHostRing], 0);
  return e;
}

}  // namespace pent

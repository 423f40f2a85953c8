// Device-side planner: turns the caller's indptr arrays into per-request
// records and the list of work units (request, q tile, split-KV tile), so no
// plan ever travels from host to device.  One CTA; it also clears the status
// word.  The host sizes the launch from its mirrors of the same arrays; when
// the device arrays disagree, every unit is disabled and a status bit is set
// instead of reading or writing out of bounds.
#include "bia_internal.h"

namespace bia {

namespace {

constexpr int kPlanThreads = 1024;

struct ReqCounts {
  int64_t units, rows;
};

__device__ inline void request_geometry(const PlanArgs &a, int b, int32_t &q_start,
                                        int32_t &q_len, int32_t &kv_len) {
  if (a.qo_indptr) {
    q_start = a.qo_indptr[b];
    q_len = a.qo_indptr[b + 1] - q_start;
  } else {
    q_start = b;
    q_len = 1;
  }
  const int32_t pages = a.kv_indptr[b + 1] - a.kv_indptr[b];
  kv_len = pages > 0 ? (pages - 1) * a.page_size + a.kv_last_page_len[b] : 0;
}

__device__ inline ReqCounts request_counts(const PlanArgs &a, int32_t q_len, int32_t kv_len,
                                           int32_t &nsp) {
  ReqCounts c{0, 0};
  c.units = request_units(q_len, kv_len, a.tile_tokens, a.tiles_per_unit, a.causal, a.split,
                          &nsp);
  if (nsp > 1) c.rows = static_cast<int64_t>(q_len) * nsp;
  return c;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ int64_t s_units[kPlanThreads];
  __shared__ int64_t s_rows[kPlanThreads];
  __shared__ int s_ok;
  const int tid = threadIdx.x;
  const int per = (a.batch + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(a.batch, tid * per), hi = min(a.batch, lo + per);
  if (tid == 0) a.status[0] = 0;

  int64_t my_units = 0, my_rows = 0;
  for (int b = lo; b < hi; ++b) {
    int32_t q_start, q_len, kv_len, nsp;
    request_geometry(a, b, q_start, q_len, kv_len);
    ReqCounts c = request_counts(a, q_len, kv_len, nsp);
    my_units += c.units;
    my_rows += c.rows;
  }
  s_units[tid] = my_units;
  s_rows[tid] = my_rows;
  __syncthreads();
  // inclusive Hillis-Steele scan over the per-thread sums
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    int64_t u = tid >= off ? s_units[tid - off] : 0;
    int64_t r = tid >= off ? s_rows[tid - off] : 0;
    __syncthreads();
    s_units[tid] += u;
    s_rows[tid] += r;
    __syncthreads();
  }
  if (tid == 0) {
    s_ok = s_units[kPlanThreads - 1] == a.n_units_expected &&
           s_rows[kPlanThreads - 1] == a.part_rows_expected;
    if (!s_ok) atomicOr(a.status, kStatusPlanMismatch);
  }
  __syncthreads();
  if (!s_ok) {
    for (int64_t i = tid; i < a.n_units_expected; i += kPlanThreads)
      a.units[i] = Unit{-1, 0, 0, 0};
    return;
  }
  int64_t unit = s_units[tid] - my_units;
  int64_t row = s_rows[tid] - my_rows;
  for (int b = lo; b < hi; ++b) {
    int32_t q_start, q_len, kv_len, nsp;
    request_geometry(a, b, q_start, q_len, kv_len);
    ReqCounts c = request_counts(a, q_len, kv_len, nsp);
    ReqInfo r;
    r.q_start = q_start;
    r.q_len = q_len;
    r.kv_len = kv_len;
    r.nsp = nsp;
    r.rowbase = c.rows > 0 ? row : -1;
    r.page_base = a.kv_indptr[b];
    r.pad = 0;
    a.reqs[b] = r;
    const int32_t tiles = (q_len + a.tile_tokens - 1) / a.tile_tokens;
    const int32_t groups = (tiles + a.tiles_per_unit - 1) / a.tiles_per_unit;
    // last q tiles first: they carry the most keys
    for (int32_t gi = groups - 1; gi >= 0; --gi) {
      const int32_t t0 = gi * a.tiles_per_unit;
      const int32_t nt = min(a.tiles_per_unit, tiles - t0);
      const int32_t n = tile_splits(q_len, kv_len, t0 + nt - 1, a.tile_tokens, a.causal, a.split);
      for (int32_t s = 0; s < n; ++s) a.units[unit++] = Unit{b, t0, s, nt};
    }
    row += c.rows;
  }
}

} // namespace

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
  return cudaGetLastError();
}

} // namespace bia

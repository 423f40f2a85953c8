// Device-side planner: turns the caller's indptr arrays into per-request
// records and the list of work units (request, group of q tiles, split-KV
// tile), so no plan ever travels from host to device.  One CTA; it also clears
// the status word.
//
//   A. per request: lengths, q-tile groups, split tiles of the widest tile,
//      partial rows, streamed units of a single-token tail tile; block scans
//      give group offsets, partial-row bases and streamed-unit offsets, and
//      the streamed units are written here
//   B. per group (all threads): its split count
//   C. block scan of the split counts: each group's first unit
//   D. per group: its units (the request's last groups first: they carry the
//      most keys); for each split, one unit per CTA of a cluster
//
// The host sizes the launch either from its mirrors of the same arrays (the
// device plan must then match it exactly) or, for a bounded call, from
// per-request bounds (the launch then has room for every call within them:
// the units the actual lengths need come first and the rest are retired).
// Each request is also checked here (lengths, page counts, the bounds): when
// any check fails or the plan does not fit the launch, every unit is retired
// and a status bit is set instead of reading or writing out of bounds.
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kPlanThreads = 1024;

// Request b's q range and key count; false (and zero lengths) when its index
// arrays break a rule of the call: negative lengths, a last-page length
// outside 1..page_size, more than 2^30 keys, q_len > kv_len when causal, no
// key in a decode, or (bounded calls) lengths beyond the bounds.
__device__ inline bool request_geometry(const PlanArgs &a, int b, int32_t &q_start,
                                        int32_t &q_len, int32_t &kv_len) {
  int64_t ql;
  if (a.qo_indptr) {
    q_start = a.qo_indptr[b];
    ql = static_cast<int64_t>(a.qo_indptr[b + 1]) - q_start;
  } else {
    q_start = b;
    ql = 1;
  }
  const int64_t pages = static_cast<int64_t>(a.kv_indptr[b + 1]) - a.kv_indptr[b];
  const int32_t last = a.kv_last_page_len[b];
  const int64_t kl = pages > 0 ? (pages - 1) * a.page_size + last : 0;
  bool ok = ql >= 0 && pages >= 0 && (pages == 0 || (last >= 1 && last <= a.page_size)) &&
            kl <= INT32_MAX / 2 && ql <= INT32_MAX / 2 && (!a.causal || ql <= kl) &&
            (a.qo_indptr || kl > 0);
  if (a.bounded) ok = ok && ql <= a.max_q_len && kl <= a.max_kv_len;
  q_len = ok ? static_cast<int32_t>(ql) : 0;
  kv_len = ok ? static_cast<int32_t>(kl) : 0;
  return ok;
}

// Exclusive scan of one value per thread across the block; returns the
// thread's exclusive prefix and writes the block total to *total.  Two
// levels: a shuffle scan inside each warp, then a scan of the 32 warp totals
// by warp 0 (three block barriers instead of two per doubling step).
template <typename T>
__device__ T block_exclusive_scan(T v, T *scratch, T *total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  T incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T x = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) scratch[warp] = incl; // warp totals
  __syncthreads();
  if (warp == 0) {
    T w = scratch[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const T x = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += x;
    }
    scratch[lane] = w; // inclusive prefix of the warp totals
  }
  __syncthreads();
  const T before = warp > 0 ? scratch[warp - 1] : T(0);
  *total = scratch[kPlanThreads / 32 - 1];
  __syncthreads(); // scratch is reused by the next scan
  return before + incl - v;
}

__device__ inline int find_group_owner(const int32_t *group_off, int batch, int32_t g) {
  int lo = 0, hi = batch - 1; // largest b with group_off[b] <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (group_off[mid] <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ int64_t s_scan[kPlanThreads / 32];
  __shared__ int s_ok;
  const int tid = threadIdx.x;
  // The planner rewrites the workspace: it waits for the kernel before it in
  // the stream (it is launched chained, so only its launch overlaps that
  // kernel), then lets the attention kernel start launching (which waits
  // for this plan before reading it).
  grid_dep_wait();
  grid_dep_launch();
  const int32_t gt = group_tiles(a.tiles_per_unit, a.ctas);
  if (tid == 0) {
    a.status[0] = 0;
    a.status[kStatusWorkCounter] = 0;
  }

  // ---- A: per request
  const int per = (a.batch + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(a.batch, tid * per), hi = min(a.batch, lo + per);
  int64_t my_groups = 0, my_rows = 0, my_sunits = 0, my_merge = 0;
  bool bad = false;
  if (tid == 0) {
    bad = a.kv_indptr[0] < 0 || (a.qo_indptr && a.qo_indptr[0] != 0);
    if (a.bounded && a.qo_indptr) bad = bad || a.qo_indptr[a.batch] > a.max_total_q;
  }
  for (int b = lo; b < hi; ++b) {
    int32_t q_start, q_len, kv_len;
    bad = !request_geometry(a, b, q_start, q_len, kv_len) || bad;
    const int32_t tiles = (q_len + a.tile_tokens - 1) / a.tile_tokens;
    const int32_t nsp = tiles > 0 ? tile_splits(q_len, kv_len, tiles - 1, a.tile_tokens,
                                                a.causal, a.split) : 1;
    my_groups += (tensor_tiles(q_len, a.tile_tokens, a.stream) + gt - 1) / gt;
    if (nsp > 1) {
      my_rows += static_cast<int64_t>(q_len) * nsp;
      my_merge += q_len - merge_first_token(q_len, kv_len, a.tile_tokens, a.causal, a.split);
    }
    if (streamed_tail(q_len, a.tile_tokens, a.stream)) my_sunits += nsp;
  }
  const bool any_bad = __syncthreads_or(bad) != 0;
  int64_t total_groups, total_rows, total_sunits;
  int64_t group = block_exclusive_scan<int64_t>(my_groups, s_scan, &total_groups);
  int64_t row = block_exclusive_scan<int64_t>(my_rows, s_scan, &total_rows);
  int64_t sunit = block_exclusive_scan<int64_t>(my_sunits, s_scan, &total_sunits);
  int64_t total_merge;
  int64_t mrow = block_exclusive_scan<int64_t>(my_merge, s_scan, &total_merge);
  // every thread sees the same totals: the streamed units below are written
  // only when they fit the host-sized list
  const bool sizes_ok =
      !any_bad && (a.bounded ? total_groups <= a.n_groups_expected &&
                                   total_rows <= a.part_rows_expected &&
                                   total_sunits <= a.n_sunits_expected
                             : total_groups == a.n_groups_expected &&
                                   total_rows == a.part_rows_expected &&
                                   total_sunits == a.n_sunits_expected);
  if (tid == 0) {
    s_ok = sizes_ok;
    if (s_ok) a.group_off[a.batch] = static_cast<int32_t>(total_groups);
    a.status[kStatusMergeRows] = sizes_ok ? static_cast<int32_t>(total_merge) : 0;
  }
  for (int b = lo; b < hi; ++b) {
    int32_t q_start, q_len, kv_len;
    request_geometry(a, b, q_start, q_len, kv_len);
    const int32_t tiles = (q_len + a.tile_tokens - 1) / a.tile_tokens;
    const int32_t nsp = tiles > 0 ? tile_splits(q_len, kv_len, tiles - 1, a.tile_tokens,
                                                a.causal, a.split) : 1;
    if (streamed_tail(q_len, a.tile_tokens, a.stream)) {
      // the tail tile is the request's widest: its split count is nsp
      for (int32_t sp = 0; sp < nsp; ++sp)
        if (sizes_ok) a.sunits[sunit + sp] = Unit{b, q_len - 1, sp, 1};
      sunit += nsp;
    }
    const int64_t rows = nsp > 1 ? static_cast<int64_t>(q_len) * nsp : 0;
    ReqInfo r;
    r.q_start = q_start;
    r.q_len = q_len;
    r.kv_len = kv_len;
    r.nsp = nsp;
    r.rowbase = rows > 0 ? row : -1;
    r.page_base = a.kv_indptr[b];
    r.mbase = static_cast<int32_t>(mrow);
    a.reqs[b] = r;
    if (nsp > 1) mrow += q_len - merge_first_token(q_len, kv_len, a.tile_tokens, a.causal, a.split);
    a.group_off[b] = static_cast<int32_t>(group);
    group += (tensor_tiles(q_len, a.tile_tokens, a.stream) + gt - 1) / gt;
    row += rows;
  }
  __syncthreads();
  // the groups this call has (equal to the host's count unless bounded)
  const int32_t n_groups = sizes_ok ? static_cast<int32_t>(total_groups) : 0;

  // ---- B: split count of every group (reversed within its request)
  if (s_ok) {
    for (int32_t g = tid; g < n_groups; g += kPlanThreads) {
      const int b = find_group_owner(a.group_off, a.batch, g);
      const ReqInfo r = a.reqs[b];
      const int32_t tiles = tensor_tiles(r.q_len, a.tile_tokens, a.stream);
      const int32_t groups = (tiles + gt - 1) / gt;
      const int32_t gi = groups - 1 - (g - a.group_off[b]);
      const int32_t t0 = gi * gt;
      const int32_t nt = min(gt, tiles - t0);
      a.group_cnt[g] = a.ctas * tile_splits(r.q_len, r.kv_len, t0 + nt - 1, a.tile_tokens,
                                            a.causal, a.split);
    }
  }
  __syncthreads();

  // ---- C: exclusive scan of the split counts, in chunks of the block size
  int64_t carry = 0;
  for (int32_t base = 0; base < n_groups; base += kPlanThreads) {
    const int32_t g = base + tid;
    const int32_t v = (s_ok && g < n_groups) ? a.group_cnt[g] : 0;
    int64_t chunk_total;
    const int64_t excl = block_exclusive_scan<int64_t>(v, s_scan, &chunk_total);
    if (s_ok && g < n_groups) a.group_cnt[g] = static_cast<int32_t>(carry + excl);
    carry += chunk_total;
  }
  if (tid == 0 && s_ok && (a.bounded ? carry > a.n_units_expected : carry != a.n_units_expected))
    s_ok = 0;
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) atomicOr(a.status, kStatusPlanMismatch);
    for (int64_t i = tid; i < a.n_units_expected; i += kPlanThreads)
      a.units[i] = Unit{-1, 0, 0, 0};
    for (int64_t i = tid; i < a.n_sunits_expected; i += kPlanThreads)
      a.sunits[i] = Unit{-1, 0, 0, 0};
    // nothing will be computed: the outputs read NaN instead of stale values
    for (int64_t i = tid; i < a.out_elems; i += kPlanThreads) a.out[i] = 0x7fc0u; // bf16 NaN
    for (int64_t i = tid; a.lse && i < a.lse_elems; i += kPlanThreads) a.lse[i] = __int_as_float(0x7fc00000);
    return;
  }

  // ---- D: the units of every group
  for (int32_t g = tid; g < n_groups; g += kPlanThreads) {
    const int b = find_group_owner(a.group_off, a.batch, g);
    const ReqInfo r = a.reqs[b];
    const int32_t tiles = tensor_tiles(r.q_len, a.tile_tokens, a.stream);
    const int32_t groups = (tiles + gt - 1) / gt;
    const int32_t gi = groups - 1 - (g - a.group_off[b]);
    const int32_t t0 = gi * gt;
    const int32_t nt = min(gt, tiles - t0);
    const int32_t n = tile_splits(r.q_len, r.kv_len, t0 + nt - 1, a.tile_tokens, a.causal,
                                  a.split);
    int64_t u = a.group_cnt[g];
    for (int32_t s = 0; s < n; ++s)
      for (int32_t c = 0; c < a.ctas; ++c) {
        const int32_t tc = t0 + c * a.tiles_per_unit;
        a.units[u++] = Unit{b, tc, s, max(0, min(a.tiles_per_unit, tiles - tc))};
      }
  }
  // a bounded launch has room for more units than these lengths need: the
  // rest are retired (whole clusters, as the live count is a multiple of ctas)
  for (int64_t i = carry + tid; i < a.n_units_expected; i += kPlanThreads)
    a.units[i] = Unit{-1, 0, 0, 0};
  for (int64_t i = total_sunits + tid; i < a.n_sunits_expected; i += kPlanThreads)
    a.sunits[i] = Unit{-1, 0, 0, 0};
}

} // namespace

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, a);
}

} // namespace bia

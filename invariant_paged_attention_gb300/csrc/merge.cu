// Fixed-order log-sum-exp merge kernels.  One warp per output row (token,
// q head): lane i holds elements 4i..4i+3 (+128k), every split is folded in
// ascending order by fold_state, so the result depends only on the partial
// states, never on the grid.
#include "bia_internal.h"
#include "fold.cuh"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kMergeWarps = 8;

// Lane `lane` owns elements k*128 + 4*lane .. +3 of a D-wide row (k < V/4);
// lanes past the end of a short row hold zeros and store nothing.
template <int V>
__device__ __forceinline__ void load_state(const float *row, int D, int lane, float (&v)[V]) {
#pragma unroll
  for (int k = 0; k < V; k += 4) {
    const int e = (k / 4) * 128 + lane * 4;
    if (e < D) {
      const float4 x = __ldg(reinterpret_cast<const float4 *>(row + e));
      v[k] = x.x;
      v[k + 1] = x.y;
      v[k + 2] = x.z;
      v[k + 3] = x.w;
    } else {
      v[k] = v[k + 1] = v[k + 2] = v[k + 3] = 0.f;
    }
  }
}

template <int V>
__device__ __forceinline__ void store_row(uint16_t *out_row, int D, float *lse_out, int lane,
                                          float L, const float (&o)[V]) {
#pragma unroll
  for (int k = 0; k < V; k += 4) {
    const int e = (k / 4) * 128 + lane * 4;
    if (e < D) {
      uint2 w;
      w.x = pack_bf16(o[k], o[k + 1]);
      w.y = pack_bf16(o[k + 2], o[k + 3]);
      *reinterpret_cast<uint2 *>(out_row + e) = w;
    }
  }
  if (lse_out && lane == 0) *lse_out = L;
}

// The request owning global q token t: largest b with qo_indptr[b] <= t and a
// non-empty range.
__device__ __forceinline__ int owner(const int32_t *qo_indptr, int batch, int64_t t) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qo_indptr[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Merge of the split partials a prefill / decode call left in the workspace:
// one CTA per q token, its q heads spread over the warps.  A warp folds one
// row: lane s first loads the LSE of split s (all splits in flight at once),
// then the states are folded in ascending split order.  Rows whose q tile had
// a single split were written by the attention kernel and are skipped.
template <int V>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_partials_kernel(const AttnArgs a) {
  const int D = a.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait(); // the attention kernel's partials are complete
  const int64_t token = blockIdx.x;
  if (token >= a.total_rows) return;
  // a plan that failed its checks computed nothing (out already holds NaN)
  if (a.status[0] & kStatusPlanMismatch) return;
  const int b = a.qo_indptr ? owner(a.qo_indptr, a.batch, token) : static_cast<int>(token);
  const ReqInfo r = a.reqs[b];
  const int32_t t = static_cast<int32_t>(token - r.q_start);
  if (t >= r.q_len) return; // past the call's last token (a launch sized from bounds)
  const int32_t tile = t / a.tile_tokens;
  const int32_t n_tile = tile_splits(r.q_len, r.kv_len, tile, a.tile_tokens, a.causal, a.split);
  if (n_tile <= 1 || r.rowbase < 0) return;
  const int32_t p = a.causal ? r.kv_len - r.q_len + t : r.kv_len - 1;
  const int32_t n_row = min(n_tile, p / a.split + 1);
  const int64_t base = (r.rowbase + static_cast<int64_t>(t) * r.nsp) * a.Hq;
  for (int h = warp; h < a.Hq; h += kMergeWarps) {
    float L = -INFINITY;
    float o[V];
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = 0.f;
    for (int s0 = 0; s0 < n_row; s0 += 32) {
      const int n_here = min(32, n_row - s0);
      const float ls_lane = lane < n_here
          ? __ldg(a.part_lse + base + static_cast<int64_t>(s0 + lane) * a.Hq + h) : -INFINITY;
      for (int k = 0; k < n_here; ++k) {
        const float ls = __shfl_sync(0xffffffffu, ls_lane, k);
        if (ls == -INFINITY) continue;
        const int64_t idx = base + static_cast<int64_t>(s0 + k) * a.Hq + h;
        float v[V];
        load_state<V>(a.part_o + idx * D, D, lane, v);
        fold_state<V>(L, o, ls, v);
      }
    }
    if (L == -INFINITY) {
#pragma unroll
      for (int i = 0; i < V; ++i) o[i] = 0.f;
    }
    const int64_t row = token * a.Hq + h;
    store_row<V>(a.out + row * D, D, a.lse ? a.lse + row : nullptr, lane, L, o);
  }
}

// Public merge: v [n, S, H, D], s [n, S, H], optional per-row counts.
template <int V>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_states_kernel(const float *__restrict__ v, const float *__restrict__ s,
                        const int32_t *__restrict__ num_states, int64_t n, int32_t S, int32_t H,
                        int32_t D, uint16_t *__restrict__ out, float *__restrict__ out_lse) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (row >= n * H) return;
  const int64_t i = row / H;
  const int h = static_cast<int>(row - i * H);
  int32_t cnt = num_states ? num_states[i] : S;
  cnt = max(0, min(cnt, S));
  float L = -INFINITY;
  float o[V];
#pragma unroll
  for (int k = 0; k < V; ++k) o[k] = 0.f;
  for (int st = 0; st < cnt; ++st) {
    const int64_t idx = (i * S + st) * H + h;
    const float ls = __ldg(s + idx);
    if (ls == -INFINITY) continue;
    float x[V];
    load_state<V>(v + idx * D, D, lane, x);
    fold_state<V>(L, o, ls, x);
  }
  if (L == -INFINITY) {
#pragma unroll
    for (int k = 0; k < V; ++k) o[k] = 0.f;
  }
  store_row<V>(out + row * D, D, out_lse ? out_lse + row : nullptr, lane, L, o);
}

} // namespace

cudaError_t launch_merge_partials(const AttnArgs &a, cudaStream_t st) {
  if (a.total_rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.total_rows));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.D <= 128) return cudaLaunchKernelEx(&cfg, merge_partials_kernel<4>, a);
  if (a.D <= 256) // head_dim 256: eight floats per lane
    return cudaLaunchKernelEx(&cfg, merge_partials_kernel<8>, a);
  // the 512-wide latent rows of multi-head latent attention
  return cudaLaunchKernelEx(&cfg, merge_partials_kernel<16>, a);
}

cudaError_t launch_merge_states(const float *v, const float *s, const int32_t *num_states,
                                int64_t n, int32_t S, int32_t H, int32_t D, uint16_t *out,
                                float *out_lse, cudaStream_t st) {
  const int64_t rows = n * H;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps);
  if (D <= 128)
    merge_states_kernel<4><<<grid, kMergeWarps * 32, 0, st>>>(v, s, num_states, n, S, H, D,
                                                               out, out_lse);
  else if (D <= 256)
    merge_states_kernel<8><<<grid, kMergeWarps * 32, 0, st>>>(v, s, num_states, n, S, H, D,
                                                               out, out_lse);
  else
    merge_states_kernel<16><<<grid, kMergeWarps * 32, 0, st>>>(v, s, num_states, n, S, H, D,
                                                                out, out_lse);
  return cudaGetLastError();
}

} // namespace bia

// Paged-KV append: writes the key/value rows of a call's new tokens into
// their pages, the step that precedes an extend / prefill call over the same
// page tables.  One warp per new token: the token's Hkv*D row of K and of V is
// copied with 16-byte loads and stores (coalesced, read once, written once).
#include "bia_internal.h"

namespace bia {

namespace {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ int append_owner(const int32_t *indptr, int batch, int64_t t) {
  int lo = 0, hi = batch - 1; // largest b with indptr[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (indptr[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const AppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t token = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (token >= a.total_new) return;
  const int b = append_owner(a.append_indptr, a.batch, token);
  const int32_t n_new = a.append_indptr[b + 1] - a.append_indptr[b];
  const int32_t pages = a.kv_indptr[b + 1] - a.kv_indptr[b];
  const int32_t kv_len = pages > 0 ? (pages - 1) * a.page_size + a.kv_last_page_len[b] : 0;
  const int32_t pos = kv_len - n_new + static_cast<int32_t>(token - a.append_indptr[b]);
  if (pos < 0 || pos >= kv_len) { // the host checks n_new <= kv_len; never taken
    if (lane == 0 && a.status) atomicOr(a.status, kStatusBadPage);
    return;
  }
  const int32_t page = a.kv_indices[a.kv_indptr[b] + pos / a.page_size];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0 && a.status) atomicOr(a.status, kStatusBadPage);
    return;
  }
  const int64_t row_elems = static_cast<int64_t>(a.Hkv) * a.D; // one token, all kv heads
  const int64_t dst = (static_cast<int64_t>(page) * a.page_size + pos % a.page_size) * row_elems;
  const int64_t src = token * row_elems;
  const int64_t vecs = row_elems / 8; // 16-byte vectors
  for (int64_t i = lane; i < vecs; i += 32) {
    const uint4 k = __ldg(reinterpret_cast<const uint4 *>(a.k_new + src) + i);
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.v_new + src) + i);
    reinterpret_cast<uint4 *>(a.k_cache + dst)[i] = k;
    reinterpret_cast<uint4 *>(a.v_cache + dst)[i] = v;
  }
}

} // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
  if (a.total_new == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((a.total_new + kAppendWarps - 1) / kAppendWarps);
  append_kernel<<<grid, kAppendWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

} // namespace bia

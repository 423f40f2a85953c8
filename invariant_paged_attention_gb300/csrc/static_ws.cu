// Decode entry point that allocates nothing and takes no workspace argument.
//
// Some callers cannot hand this library a scratch buffer: plugin and
// extension interfaces of inference engines whose enqueue callbacks may not
// call cudaMalloc (an allocation there can synchronise the device, break a
// CUDA-graph capture in progress, or escape a memory budget the host fixed up
// front), and host programs that account for every byte of device memory
// before serving starts.  For them, bia_decode_paged_noalloc runs the same
// decode path as bia_decode_paged with its scratch space (device plan, split
// partials) placed in the file-scope array below, which the CUDA runtime
// reserves on every GPU that loads this library and keeps until the process
// exits.
#include <cstdio>
#include <mutex>

#include "../../include/bia.h"
#include "bia_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = BIA_DECODE_NOALLOC_SCRATCH_BYTES; // 64 MiB

// The scratch array.  In host code its name stands for a host-side shadow,
// not a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached for the life of the process
// (a cudaDeviceReset would leave the cached address stale).
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BIA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BIA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return BIA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return BIA_OK;
}

} // namespace

extern "C" {

int bia_decode_paged_noalloc(const bia_attn_desc *desc, const void *q, const void *k_cache,
                             const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                             const int32_t *kv_indices, const int32_t *kv_last_page_len,
                             const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                             int32_t batch, int32_t split_size, void *out, float *lse,
                             void *stream) {
  // every host-side check of bia_decode_paged first, with its status codes;
  // nothing touches the GPU until the call is known to be valid and to fit
  size_t need = 0;
  int rc = bia::decode_check(desc, q, k_cache, v_cache, num_pages, kv_indptr, kv_indices,
                             kv_last_page_len, kv_indptr_host, kv_last_page_len_host, batch,
                             split_size, out, lse, &need);
  if (rc != BIA_OK) return rc;
  if (need > kStaticScratchBytes) return BIA_ERR_WORKSPACE_TOO_SMALL;
  void *ws = nullptr;
  rc = scratch_address(&ws);
  if (rc != BIA_OK) return rc;
  return bia::decode_on_scratch(desc, q, k_cache, v_cache, num_pages, kv_indptr, kv_indices,
                                kv_last_page_len, kv_indptr_host, kv_last_page_len_host, batch,
                                split_size, ws, kStaticScratchBytes, out, lse, stream);
}

} // extern "C"

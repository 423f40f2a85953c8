// Internal declarations shared by the host entry points and the kernels of
// libbia.so: the workspace layout, the device plan records and the kernel
// launchers.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/bia.h"

#include <cuda.h> // CUtensorMap (a plain 128-byte struct; no driver-library link needed)
#include <cuda_runtime.h>

namespace bia {

// Status bits in the workspace status word.
constexpr int32_t kStatusBadPage = 1;     // a page index outside [0, num_pages)
constexpr int32_t kStatusPlanMismatch = 2; // device plan disagreed with the host-sized launch
constexpr int32_t kStatusTimeout = 4;      // a bounded device wait gave up

constexpr int kTileRows = 128; // q tile rows (GQA-packed)
constexpr int kKvBlock = 128;  // keys per block of the prefill inner loop
constexpr int kPrefillTilesPerUnit = 2; // q tiles sharing one K/V stream in a prefill CTA
// q tiles per prefill CTA for a head dim: one for 256 (its O fills half of TMEM)
inline int prefill_tiles_per_unit(int head_dim) {
  return head_dim == 256 ? 1 : kPrefillTilesPerUnit;
}
constexpr int kPrefillClusterCtas = 4; // prefill CTAs of a cluster sharing each K/V gather
constexpr int kMlaCkvDim = 512; // latent (value) width of multi-head latent attention
constexpr int kMlaKpeDim = 64;  // its rope key width

// Per-request record written by the plan kernel.
struct ReqInfo {
  int32_t q_start;  // first global q token
  int32_t q_len;    // q tokens in this call
  int32_t kv_len;   // keys
  int32_t nsp;      // split-KV tiles of the request's last q tile (max over tiles)
  int64_t rowbase;  // first partial row (rows of [Hq, D] fp32), -1 if none
  int32_t page_base;// kv_indptr[b]
  int32_t mbase;    // rows to merge (tokens of multi-split q tiles) of earlier requests
};
static_assert(sizeof(ReqInfo) == 32, "ReqInfo layout");

// One unit of work for one kv head (grid.y): q tiles tile .. tile+ntiles-1 of
// request b against split-KV tile `split`.  A streamed unit (one query token
// against one split tile, run by the decode kernel) holds the token's index
// within its request in `tile` and 1 in `ntiles`.
struct Unit {
  int32_t b, tile, split, ntiles;
};

// Byte offsets inside the caller's workspace.
struct WsLayout {
  size_t status = 0;   // int32[64]
  size_t reqs = 0;     // ReqInfo[batch]
  size_t group_off = 0; // int32[batch + 1]: first q-tile group of each request
  size_t group_cnt = 0; // int32[n_groups]: first unit of each group
  size_t units = 0;    // Unit[n_units]
  size_t sunits = 0;   // Unit[n_sunits]: streamed single-token q tiles
  size_t part_o = 0;   // float[part_rows * Hq * D]
  size_t part_lse = 0; // float[part_rows * Hq]
  size_t total = 0;
};

// Last absolute key position any row of q tile `tile` may see (-1: none).
// Rows of a tile are its tile_tokens consecutive in-call tokens; token t sits
// at position kv_len - q_len + t.
__host__ __device__ inline int32_t tile_last_key(int32_t q_len, int32_t kv_len, int32_t tile,
                                                 int32_t tile_tokens, int32_t causal) {
  if (!causal) return kv_len - 1;
  int32_t last_t = (tile + 1) * tile_tokens;
  if (last_t > q_len) last_t = q_len;
  return kv_len - q_len + last_t - 1;
}
// Split-KV tiles (anchored at key 0) a q tile touches; at least 1.
__host__ __device__ inline int32_t tile_splits(int32_t q_len, int32_t kv_len, int32_t tile,
                                               int32_t tile_tokens, int32_t causal,
                                               int32_t split) {
  int32_t last = tile_last_key(q_len, kv_len, tile, tile_tokens, causal);
  return last < 0 ? 1 : last / split + 1;
}

// First in-call token of a request whose q tile spans more than one split
// (q_len if none).  A tile's last key grows with the tile index (causal) or
// is the same for every tile, so such tiles are a suffix of the request: the
// rows the merge folds are tokens merge_first_token .. q_len-1.
__host__ __device__ inline int32_t merge_first_token(int32_t q_len, int32_t kv_len,
                                                     int32_t tile_tokens, int32_t causal,
                                                     int32_t split) {
  if (q_len <= 0 || kv_len - 1 < split) return q_len; // every key in split 0
  if (!causal) return 0;
  const int32_t need = split + 1 - (kv_len - q_len); // in-call tokens the tile must reach
  if (need > q_len) return q_len;
  const int32_t tile = need <= tile_tokens ? 0 : (need + tile_tokens - 1) / tile_tokens - 1;
  return tile * tile_tokens;
}

// Slot of the workspace status array holding the number of rows to merge
// (written by the planner; slot 0 is the status word).
constexpr int kStatusMergeRows = 1;
// Slot holding the work counter from which the persistent decode kernel's
// CTAs take their next (unit, kv head) item (zeroed by the planner).
constexpr int kStatusWorkCounter = 2;

// A prefill request whose last q tile holds a single token (a one-token
// extend, or the one-token tail of a longer chunk) has that tile streamed by
// the decode kernel, one query row per CTA, instead of filling G of the 128
// rows of a tensor-core tile.  The choice is a function of the tile alone (its
// token count), and every q-tile-aligned chunking of a request cuts the same
// tiles, so it holds the same way in any batch and any aligned chunking.
__host__ __device__ inline int32_t streamed_tail(int32_t q_len, int32_t tile_tokens,
                                                 int32_t stream) {
  return stream && tile_tokens > 1 && q_len % tile_tokens == 1 ? 1 : 0;
}
// q tiles of a request that run on the tensor-core prefill kernel.
__host__ __device__ inline int32_t tensor_tiles(int32_t q_len, int32_t tile_tokens,
                                                int32_t stream) {
  return (q_len + tile_tokens - 1) / tile_tokens - streamed_tail(q_len, tile_tokens, stream);
}

// Units of one request: its tensor q tiles grouped ctas * tiles_per_unit at a
// time, each group crossed with the split tiles its last (widest) q tile
// touches; a group's units for one split are `ctas` consecutive units (one per
// CTA of a cluster, tiles_per_unit tiles each; the last ones may hold no
// tile).  A streamed tail adds one streamed unit per split tile it touches
// (*stream_units).
__host__ __device__ inline int32_t group_tiles(int32_t tiles_per_unit, int32_t ctas) {
  return tiles_per_unit * ctas;
}
__host__ __device__ inline int64_t request_units(int32_t q_len, int32_t kv_len,
                                                 int32_t tile_tokens, int32_t tiles_per_unit,
                                                 int32_t ctas, int32_t causal, int32_t split,
                                                 int32_t stream, int32_t *max_splits,
                                                 int32_t *stream_units) {
  const int32_t tiles = (q_len + tile_tokens - 1) / tile_tokens;
  const int32_t tt = tensor_tiles(q_len, tile_tokens, stream);
  const int32_t gt = group_tiles(tiles_per_unit, ctas);
  int64_t units = 0;
  int32_t nsp = 1;
  for (int32_t t0 = 0; t0 < tt; t0 += gt) {
    const int32_t last = min(t0 + gt, tt) - 1;
    const int32_t n = tile_splits(q_len, kv_len, last, tile_tokens, causal, split);
    units += static_cast<int64_t>(n) * ctas;
    if (n > nsp) nsp = n;
  }
  int32_t ns = 0;
  if (tt < tiles) {
    ns = tile_splits(q_len, kv_len, tiles - 1, tile_tokens, causal, split);
    if (ns > nsp) nsp = ns;
  }
  if (max_splits) *max_splits = nsp;
  if (stream_units) *stream_units = ns;
  return units;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout make_layout(int batch, int64_t n_groups, int64_t n_units, int64_t n_sunits,
                            int64_t part_rows, int Hq, int D) {
  WsLayout w;
  w.status = 0;
  w.reqs = 256;
  w.group_off = align_up(w.reqs + sizeof(ReqInfo) * (size_t)batch, 256);
  w.group_cnt = align_up(w.group_off + sizeof(int32_t) * ((size_t)batch + 1), 256);
  w.units = align_up(w.group_cnt + sizeof(int32_t) * (size_t)n_groups, 256);
  w.sunits = align_up(w.units + sizeof(Unit) * (size_t)n_units, 256);
  w.part_o = align_up(w.sunits + sizeof(Unit) * (size_t)n_sunits, 256);
  w.part_lse = align_up(w.part_o + sizeof(float) * (size_t)part_rows * Hq * D, 256);
  w.total = align_up(w.part_lse + sizeof(float) * (size_t)part_rows * Hq, 256);
  return w;
}

struct PlanArgs {
  const int32_t *qo_indptr;  // NULL for decode (one token per request)
  const int32_t *kv_indptr;
  const int32_t *kv_last_page_len;
  int32_t batch, page_size, tile_tokens, tiles_per_unit, ctas, causal, split;
  int32_t stream; // 1: single-token tail tiles become streamed units (prefill)
  // 0: the launch was sized from the host mirrors and the device plan must
  // match it exactly; 1: it was sized from bounds (the *_expected counts are
  // capacities), every request must lie within them, and the units the
  // actual lengths do not need are retired
  int32_t bounded;
  int32_t max_q_len, max_kv_len; // per-request bounds (bounded calls)
  int64_t max_total_q;            // q tokens of the call (bounded calls)
  int64_t n_groups_expected, n_units_expected, n_sunits_expected, part_rows_expected;
  // the call's outputs: filled with NaN when the plan fails its checks, so a
  // failure shows in the data and not only in the status word
  uint16_t *out;
  int64_t out_elems;
  float *lse;      // may be NULL
  int64_t lse_elems;
  int32_t *status;
  ReqInfo *reqs;
  int32_t *group_off, *group_cnt;
  Unit *units, *sunits;
};

// Geometry of a call shared by the attention kernels.
struct AttnArgs {
  const uint16_t *q, *k_cache, *v_cache;
  const int32_t *kv_indices;
  const int32_t *qo_indptr; // NULL for decode
  int64_t num_pages;
  int32_t Hq, Hkv, D, G, page_shift, causal, split, tile_tokens;
  float scale_log2; // sm_scale * log2(e)
  int32_t batch;
  int64_t n_units;
  const ReqInfo *reqs;
  const Unit *units;
  float *part_o, *part_lse;
  int64_t total_rows; // total q tokens
  uint16_t *out;
  float *lse;
  int32_t *status;
  // TMA descriptors (prefill): q [total_q][Hq][D] in boxes of 64 columns x G
  // heads x tile_tokens tokens, and key / value rows [num_pages*page_size*Hkv,
  // D] in 64-column boxes one row high; all SW128
  CUtensorMap tm_q, tm_k, tm_v;
  int32_t q_rows, kv_rows; // row extents of the maps (a row >= extent reads as zeros)
  // head_dim 256 with pages of 16+ keys: the caches as 3-D maps [slots][Hkv][D]
  // in boxes of 64 columns x 1 head x 16 slots (16 consecutive keys of one page)
  CUtensorMap tm_k3, tm_v3;
  // multi-head latent attention on the tensor cores: q_pe rows [B*H, 64] in
  // 64 x 16-row boxes (tm_q then holds q_nope [B*H, 512] in the same boxes,
  // tm_k the ckv rows [num_pages*P, 512] in 64 x 1 boxes) and the kpe rows
  // [num_pages*P, 64] in 64 x 1 boxes
  CUtensorMap tm_qpe, tm_kpe;
  // multi-head latent attention (decode): q_pe [B, H, 64] and the rope rows
  // of the latent cache [num_pages, P, 64]; q holds q_nope, k_cache the ckv rows
  const uint16_t *q_pe, *kpe_cache;
  // optional custom mask (prefill): little-endian bit string of mask_words
  // 32-bit words; request b's [q_len, kv_len] bits start at bit mask_indptr[b]
  const uint32_t *mask;
  const int64_t *mask_indptr;
  int64_t mask_words;
};

// Paged-KV append: new token t of request b goes to position
// kv_len(b) - n_new(b) + (t - append_indptr[b]).
struct AppendArgs {
  const uint16_t *k_new, *v_new; // [total_new, Hkv, D]
  uint16_t *k_cache, *v_cache;
  const int32_t *append_indptr, *kv_indptr, *kv_indices, *kv_last_page_len;
  int64_t num_pages, total_new;
  int32_t batch, Hkv, D, page_size;
  int32_t *status; // may be NULL
};

// The decode of bia_decode_paged split in two for the static-scratch entry
// point: decode_check runs every host-side check of the call and reports the
// workspace bytes it needs (*need), enqueuing nothing; decode_on_scratch runs
// the call on the library's own scratch array (its residency is not checked:
// the address comes from the runtime for the current device).
int decode_check(const bia_attn_desc *desc, const void *q, const void *k_cache,
                 const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                 const int32_t *kv_indices, const int32_t *kv_last_page_len,
                 const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                 int32_t batch, int32_t split_size, void *out, float *lse, size_t *need);
int decode_on_scratch(const bia_attn_desc *desc, const void *q, const void *k_cache,
                      const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                      const int32_t *kv_indices, const int32_t *kv_last_page_len,
                      const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                      int32_t batch, int32_t split_size, void *scratch, size_t scratch_bytes,
                      void *out, float *lse, void *stream);

// Launch attribute of the kernels that follow the planner within a call:
// programmatic stream serialization (each waits in-kernel for its
// predecessor's completion, so its launch overlaps the predecessor's tail).
inline cudaLaunchAttribute chained_launch_attr() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s);
cudaError_t launch_append(const AppendArgs &a, cudaStream_t s);
cudaError_t launch_decode(const AttnArgs &a, cudaStream_t s);
// The tensor-core decode (head_dim 128, G in {1, 2, 4, 8}); launch_decode
// takes it whenever it applies.
bool decode_tc_supported(const AttnArgs &a);
cudaError_t launch_decode_tc(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_prefill(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_prefill_wide(const AttnArgs &a, cudaStream_t s); // head_dim 256
cudaError_t launch_mla_decode(const AttnArgs &a, cudaStream_t s);
// q heads per CTA of the MLA kernel: 32 when the head count is a multiple of
// 32, else 16 (the q tensor map's boxes are this many rows high)
inline int mla_head_group(int num_heads) { return num_heads % 32 == 0 ? 32 : 16; }
cudaError_t launch_merge_partials(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_merge_states(const float *v, const float *s, const int32_t *num_states,
                                int64_t n, int32_t S, int32_t H, int32_t D, uint16_t *out,
                                float *out_lse, cudaStream_t st);

} // namespace bia

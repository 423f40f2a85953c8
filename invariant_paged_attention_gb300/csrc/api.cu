// Host side of libbia.so: argument validation, workspace sizing and the
// launch sequence (device plan -> attention kernel -> merge of split
// partials) for each entry point of bia.h.  No allocation, no stream
// synchronisation (except bia_read_status, which exists to synchronise).
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <initializer_list>

#include <cudaTypedefs.h>

#include "../../include/bia.h"
#include "bia_internal.h"

namespace {

cudaEvent_t g_attn_begin = nullptr, g_attn_end = nullptr;

// A library-owned stream (one per host thread and device) onto which a prefill
// call forks its streamed single-token tiles, so that their key stream runs
// beside the tensor-core tiles of the same call; the fork waits for the plan
// and the call's stream waits for the fork before the merge, so the call is
// ordered on the caller's stream exactly as without it.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;

// The calling thread's side stream of the current device, created on first
// use; nullptr when it cannot be had (then the call stays on one stream).
// Nothing is created while `st` is being captured into a graph.
SideStream *side_stream(cudaStream_t st) {
  thread_local SideStream side[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream &s = side[dev];
  if (s.stream) return &s;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) {
    s.stream = nullptr;
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(s.stream);
    s.stream = nullptr;
    return nullptr;
  }
  return &s;
}
unsigned long long g_launches = 0;
thread_local char g_last_error[256] = "";

int fail(int status, const char *what, int code) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s (code %d)", what, code);
  return status;
}
int cuda_fail(const char *what, cudaError_t e) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, cudaGetErrorString(e));
  return BIA_ERR_CUDA;
}

using bia::PlanArgs;
using bia::AttnArgs;
using bia::WsLayout;

struct HostPlan {
  int64_t n_groups = 0;
  int64_t n_units = 0;
  int64_t n_sunits = 0; // streamed single-token q tiles x their split tiles
  int64_t part_rows = 0;
  int64_t total_q = 0;
};

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// True when a non-null pointer is not a multiple of `align` bytes (the
// kernels read int32 / fp32 words, int64 offsets and 16-byte vectors).
bool misaligned(const void *p, uintptr_t align) {
  return (reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0;
}

// Every non-null pointer of `ptrs` must be device memory of the current
// device.  The kernels read and write these addresses directly, and the
// prefill kernels' TMA gathers multicast each loaded row into every CTA of
// their cluster, which is defined here for this GPU's own memory only; a host
// buffer (pinned or not), managed memory or another GPU's peer-mapped buffer
// is refused with BIA_ERR_INVALID_ARG before anything is enqueued.
struct NamedPtr {
  const char *name;
  const void *p;
};
int check_resident(std::initializer_list<NamedPtr> ptrs) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  for (const NamedPtr &x : ptrs) {
    if (!x.p) continue;
    cudaPointerAttributes at{};
    e = cudaPointerGetAttributes(&at, x.p);
    if (e != cudaSuccess) {
      (void)cudaGetLastError(); // not sticky: keep it from reaching a later launch check
      return cuda_fail("cudaPointerGetAttributes", e);
    }
    if (at.type != cudaMemoryTypeDevice || at.device != dev) {
      std::snprintf(g_last_error, sizeof g_last_error,
                    "%s is not device memory of the current device %d (memory type %d, "
                    "device %d)",
                    x.name, dev, static_cast<int>(at.type), at.device);
      return BIA_ERR_INVALID_ARG;
    }
  }
  return BIA_OK;
}

int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

int check_desc(const bia_attn_desc *d) {
  if (!d) return BIA_ERR_INVALID_ARG;
  if (d->num_qo_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->page_size <= 0)
    return BIA_ERR_INVALID_ARG;
  if (d->num_qo_heads % d->num_kv_heads != 0) return BIA_ERR_UNSUPPORTED;
  const int G = d->num_qo_heads / d->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return BIA_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 96 && d->head_dim != 128 && d->head_dim != 256)
    return BIA_ERR_UNSUPPORTED;
  if (!is_pow2(d->page_size) || d->page_size > 256) return BIA_ERR_UNSUPPORTED;
  if (!(std::isfinite(d->sm_scale))) return BIA_ERR_INVALID_ARG;
  return BIA_OK;
}

// Validates the host mirrors and computes the same plan sizes the device
// planner will produce.  qo == nullptr: decode (one query per request).
// stream: single-token tail tiles become streamed units (prefill).
int host_plan(const bia_attn_desc *d, const int32_t *qo, const int32_t *kvp,
              const int32_t *last, int32_t batch, int32_t causal, int32_t split, int tile_tokens,
              int tiles_per_unit, int ctas, int stream, HostPlan *hp) {
  if (batch <= 0 || !kvp || !last) return BIA_ERR_INVALID_ARG;
  if (split <= 0 || split % bia::kKvBlock != 0) return BIA_ERR_UNSUPPORTED;
  if (qo && qo[0] != 0) return BIA_ERR_INVALID_ARG;
  if (kvp[0] < 0) return BIA_ERR_INVALID_ARG;
  HostPlan p;
  for (int b = 0; b < batch; ++b) {
    const int64_t q_len = qo ? static_cast<int64_t>(qo[b + 1]) - qo[b] : 1;
    const int64_t pages = static_cast<int64_t>(kvp[b + 1]) - kvp[b];
    if (q_len < 0 || pages < 0) return BIA_ERR_INVALID_ARG;
    if (pages > 0 && (last[b] < 1 || last[b] > d->page_size)) return BIA_ERR_INVALID_ARG;
    const int64_t kv_len = pages > 0 ? (pages - 1) * d->page_size + last[b] : 0;
    if (kv_len > INT32_MAX / 2) return BIA_ERR_UNSUPPORTED;
    if (causal && q_len > kv_len) return BIA_ERR_INVALID_ARG;
    if (!qo && kv_len == 0) return BIA_ERR_INVALID_ARG;
    int32_t nsp = 1, ns = 0;
    const int64_t tiles = bia::tensor_tiles(static_cast<int32_t>(q_len), tile_tokens, stream);
    const int64_t gt = bia::group_tiles(tiles_per_unit, ctas);
    p.n_groups += (tiles + gt - 1) / gt;
    p.n_units += bia::request_units(static_cast<int32_t>(q_len), static_cast<int32_t>(kv_len),
                                    tile_tokens, tiles_per_unit, ctas, causal, split, stream,
                                    &nsp, &ns);
    p.n_sunits += ns;
    if (nsp > 1) p.part_rows += q_len * nsp;
    p.total_q += q_len;
  }
  if (p.n_units > INT32_MAX) return BIA_ERR_UNSUPPORTED; // grid.x limit is 2^31-1
  if (p.n_sunits * d->num_kv_heads > INT32_MAX) return BIA_ERR_UNSUPPORTED;
  *hp = p;
  return BIA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no direct
// link against the driver library).  Looked up once; the initialisation of a
// function-local static is thread-safe, so concurrent first calls agree.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// A 2-D map over `rows` rows of `head_dim` bf16 (row pitch head_dim*2 bytes),
// 64-column x 1-row boxes with the 128-byte swizzle of the MMA operand tiles;
// coordinates outside the map read as zeros.
int encode_rows_map(CUtensorMap *map, const void *base, int64_t rows, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return -1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t estr[2] = {1, 1};
  return static_cast<int>(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// The paged cache [slots][Hkv][head_dim] bf16 as a 3-D map whose boxes are
// 64 columns x 1 kv head x 16 consecutive slots (128-byte swizzle); slots
// past the end read as zeros.
int encode_slots_map(CUtensorMap *map, const void *base, int64_t slots, int Hkv, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return -1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(Hkv) * head_dim * 2};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  return static_cast<int>(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// A 2-D map over `rows` rows of `cols` bf16 (row pitch cols*2 bytes) in boxes
// of 64 columns x box_rows rows, 128-byte swizzle; rows past the end read as
// zeros.
int encode_2d_map(CUtensorMap *map, const void *base, int64_t rows, int cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return -1;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return static_cast<int>(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// The q tiles of a prefill call as a 3-D map [total_q][Hq][head_dim]; a box
// of 64 columns x G heads x T tokens is one 64-column half of a 128-row q
// tile (rows = token-major (token, head) pairs, 128-byte swizzle); tokens past
// the end read as zeros.
int encode_q_map(CUtensorMap *map, const void *base, int64_t total_q, int Hq, int head_dim, int G,
                 int T) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return -1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(Hq) * head_dim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(T)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return static_cast<int>(enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

float effective_scale(const bia_attn_desc *d) {
  const float s = d->sm_scale > 0.f ? d->sm_scale : 1.0f / std::sqrt(static_cast<float>(d->head_dim));
  return s * 1.4426950408889634f;
}

// Custom mask of a prefill call (bia_prefill_paged_mask).
struct MaskArgs {
  const void *bits;               // device, 4-byte aligned
  size_t bytes;                   // size of the bit buffer
  const int64_t *indptr;          // device [batch+1] bit offsets
  const int64_t *indptr_host;     // host mirror
};

// Every request's [q_len, kv_len] bits lie inside the buffer's whole words.
int check_mask(const MaskArgs &m, const int32_t *qo, const int32_t *kvp, const int32_t *last,
               int32_t batch, int page_size) {
  if (!m.bits || !m.indptr || !m.indptr_host) return BIA_ERR_INVALID_ARG;
  if (misaligned(m.bits, 4) || misaligned(m.indptr, 8)) return BIA_ERR_INVALID_ARG;
  const int64_t total_bits = static_cast<int64_t>(m.bytes / 4) * 32;
  for (int b = 0; b < batch; ++b) {
    const int64_t q_len = static_cast<int64_t>(qo[b + 1]) - qo[b];
    const int64_t pages = static_cast<int64_t>(kvp[b + 1]) - kvp[b];
    const int64_t kv_len = pages > 0 ? (pages - 1) * page_size + last[b] : 0;
    const int64_t off = m.indptr_host[b];
    if (off < 0 || off > total_bits - q_len * kv_len) return BIA_ERR_INVALID_ARG;
  }
  return BIA_OK;
}

// Plan sizes that cover every call of `batch` requests within `bd` (a
// bounded call): the largest group, unit, streamed-unit and partial-row
// counts any such call can need, so that one launch configuration (and one
// captured CUDA graph) serves all of them.  The device planner fills the
// units the actual lengths need and retires the rest.
int bounded_plan(const bia_bounds *bd, int32_t batch, int32_t causal, int32_t split,
                 int tile_tokens, int tiles_per_unit, int ctas, int stream, bool decode,
                 HostPlan *hp) {
  if (!bd || batch <= 0) return BIA_ERR_INVALID_ARG;
  if (split <= 0 || split % bia::kKvBlock != 0) return BIA_ERR_UNSUPPORTED;
  const int64_t max_kv = bd->max_kv_len;
  int64_t max_q = decode ? 1 : bd->max_q_len;
  const int64_t total_q = decode ? batch : bd->max_total_q;
  if (max_kv < (decode ? 1 : 0) || max_q < 0 || total_q < 0) return BIA_ERR_INVALID_ARG;
  if (max_kv > INT32_MAX / 2 || max_q > INT32_MAX / 2) return BIA_ERR_UNSUPPORTED;
  if (causal && max_q > max_kv) max_q = max_kv; // a causal request has q_len <= kv_len
  if (max_q > total_q) max_q = total_q;
  const int64_t s_max = max_kv > 0 ? (max_kv + split - 1) / split : 1;
  const int64_t gt = bia::group_tiles(tiles_per_unit, ctas);
  const int64_t tiles_max = (max_q + tile_tokens - 1) / tile_tokens;
  HostPlan p;
  // sum over requests of ceil(q_len / (tile_tokens * gt)) is at most
  // batch + total_q / (tile_tokens * gt)
  p.n_groups = std::min<int64_t>(static_cast<int64_t>(batch) * ((tiles_max + gt - 1) / gt),
                                 batch + total_q / (tile_tokens * gt));
  p.n_units = p.n_groups * ctas * s_max;
  p.n_sunits = (stream && tile_tokens > 1) ? std::min<int64_t>(batch, total_q) * s_max : 0;
  p.part_rows = s_max > 1 ? std::min<int64_t>(static_cast<int64_t>(batch) * max_q, total_q) *
                                s_max
                          : 0;
  p.total_q = total_q;
  if (p.n_units > INT32_MAX) return BIA_ERR_UNSUPPORTED;
  *hp = p;
  return BIA_OK;
}

// Optional parts of an attention call.
struct CallOpts {
  const MaskArgs *mask = nullptr;
  const bia_bounds *bounds = nullptr; // bounded call: plan sized from bounds, no host mirrors
  bool ws_static = false;             // the workspace is the library's own scratch array
  size_t *need = nullptr;             // check only: report the workspace bytes and return
};

int run_attention(bool decode, const bia_attn_desc *desc, const void *q, const void *k_cache,
                  const void *v_cache, int64_t num_pages, const int32_t *qo_indptr,
                  const int32_t *kv_indptr, const int32_t *kv_indices,
                  const int32_t *kv_last_page_len, const int32_t *qo_host,
                  const int32_t *kvp_host, const int32_t *last_host, int32_t batch,
                  int32_t causal, int32_t split, void *workspace, size_t workspace_bytes,
                  void *out, float *lse, void *stream, const CallOpts &opt = CallOpts{}) {
  const MaskArgs *mask = opt.mask;
  const bool bounded = opt.bounds != nullptr;
  int rc = check_desc(desc);
  if (rc != BIA_OK) return rc;
  if (!q || !k_cache || !v_cache || !kv_indptr || !kv_indices || !kv_last_page_len || !out ||
      num_pages <= 0)
    return BIA_ERR_INVALID_ARG;
  if (!opt.need && !workspace) return BIA_ERR_INVALID_ARG;
  if (!decode && (!qo_indptr || (!bounded && !qo_host))) return BIA_ERR_INVALID_ARG;
  if (misaligned(workspace, 256)) return BIA_ERR_INVALID_ARG;
  if (misaligned(q, 16) || misaligned(k_cache, 16) || misaligned(v_cache, 16) ||
      misaligned(out, 16) || misaligned(lse, 4) || misaligned(qo_indptr, 4) ||
      misaligned(kv_indptr, 4) || misaligned(kv_indices, 4) || misaligned(kv_last_page_len, 4))
    return BIA_ERR_INVALID_ARG;
  if (split == 0) split = decode ? BIA_DECODE_SPLIT : BIA_PREFILL_SPLIT;
  const int G = desc->num_qo_heads / desc->num_kv_heads;
  const int tile_tokens = decode ? 1 : bia::kTileRows / G;
  const int tiles_per_unit = decode ? 1 : bia::prefill_tiles_per_unit(desc->head_dim);
  const int ctas = decode ? 1 : bia::kPrefillClusterCtas;
  const int stream_tail = decode ? 0 : 1;
  if (decode) causal = 1;
  HostPlan hp;
  rc = bounded ? bounded_plan(opt.bounds, batch, causal, split, tile_tokens, tiles_per_unit,
                              ctas, stream_tail, decode, &hp)
               : host_plan(desc, decode ? nullptr : qo_host, kvp_host, last_host, batch, causal,
                           split, tile_tokens, tiles_per_unit, ctas, stream_tail, &hp);
  if (rc != BIA_OK) return rc;
  if (decode && hp.n_units * desc->num_kv_heads > INT32_MAX) return BIA_ERR_UNSUPPORTED;
  if (mask) {
    rc = check_mask(*mask, qo_host, kvp_host, last_host, batch, desc->page_size);
    if (rc != BIA_OK) return rc;
  }
  const WsLayout w = bia::make_layout(batch, hp.n_groups, hp.n_units, hp.n_sunits,
                                      hp.part_rows, desc->num_qo_heads, desc->head_dim);
  if (opt.need) {
    *opt.need = w.total;
    return BIA_OK;
  }
  if (workspace_bytes < w.total) return BIA_ERR_WORKSPACE_TOO_SMALL;
  if (hp.total_q == 0) return BIA_OK;

  const int64_t q_rows = hp.total_q * desc->num_qo_heads;
  const int64_t kv_rows = num_pages * desc->page_size * desc->num_kv_heads;
  if (!decode && (q_rows >= INT32_MAX || kv_rows >= INT32_MAX)) return BIA_ERR_UNSUPPORTED;
  rc = check_resident({{"q", q},
                       {"k_cache", k_cache},
                       {"v_cache", v_cache},
                       {"out", out},
                       {"lse", lse},
                       {"qo_indptr", qo_indptr},
                       {"kv_indptr", kv_indptr},
                       {"kv_indices", kv_indices},
                       {"kv_last_page_len", kv_last_page_len},
                       {"mask", mask ? mask->bits : nullptr},
                       {"mask_indptr", mask ? mask->indptr : nullptr},
                       {"workspace", opt.ws_static ? nullptr : workspace}});
  if (rc != BIA_OK) return rc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  PlanArgs pa{};
  pa.qo_indptr = decode ? nullptr : qo_indptr;
  pa.kv_indptr = kv_indptr;
  pa.kv_last_page_len = kv_last_page_len;
  pa.batch = batch;
  pa.page_size = desc->page_size;
  pa.tile_tokens = tile_tokens;
  pa.tiles_per_unit = tiles_per_unit;
  pa.ctas = ctas;
  pa.causal = causal;
  pa.split = split;
  pa.stream = stream_tail;
  pa.bounded = bounded ? 1 : 0;
  if (bounded) {
    pa.max_q_len = decode ? 1 : opt.bounds->max_q_len;
    pa.max_kv_len = opt.bounds->max_kv_len;
    pa.max_total_q = hp.total_q;
  }
  pa.n_groups_expected = hp.n_groups;
  pa.n_units_expected = hp.n_units;
  pa.n_sunits_expected = hp.n_sunits;
  pa.part_rows_expected = hp.part_rows;
  pa.out = static_cast<uint16_t *>(out);
  pa.out_elems = hp.total_q * desc->num_qo_heads * desc->head_dim;
  pa.lse = lse;
  pa.lse_elems = hp.total_q * desc->num_qo_heads;
  pa.status = reinterpret_cast<int32_t *>(ws + w.status);
  pa.reqs = reinterpret_cast<bia::ReqInfo *>(ws + w.reqs);
  pa.group_off = reinterpret_cast<int32_t *>(ws + w.group_off);
  pa.group_cnt = reinterpret_cast<int32_t *>(ws + w.group_cnt);
  pa.units = reinterpret_cast<bia::Unit *>(ws + w.units);
  pa.sunits = reinterpret_cast<bia::Unit *>(ws + w.sunits);
  cudaError_t pe = bia::launch_plan(pa, st);
  if (pe != cudaSuccess) return cuda_fail("plan kernel launch", pe);
  __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);

  AttnArgs a{};
  a.q = static_cast<const uint16_t *>(q);
  a.k_cache = static_cast<const uint16_t *>(k_cache);
  a.v_cache = static_cast<const uint16_t *>(v_cache);
  a.kv_indices = kv_indices;
  a.qo_indptr = decode ? nullptr : qo_indptr;
  a.num_pages = num_pages;
  a.Hq = desc->num_qo_heads;
  a.Hkv = desc->num_kv_heads;
  a.D = desc->head_dim;
  a.G = G;
  a.page_shift = log2i(desc->page_size);
  a.causal = causal;
  a.split = split;
  a.tile_tokens = tile_tokens;
  a.scale_log2 = effective_scale(desc);
  a.batch = batch;
  a.n_units = hp.n_units;
  a.reqs = pa.reqs;
  a.units = pa.units;
  a.part_o = reinterpret_cast<float *>(ws + w.part_o);
  a.part_lse = reinterpret_cast<float *>(ws + w.part_lse);
  a.total_rows = hp.total_q;
  a.out = static_cast<uint16_t *>(out);
  a.lse = lse;
  a.status = pa.status;
  if (mask) {
    a.mask = static_cast<const uint32_t *>(mask->bits);
    a.mask_indptr = mask->indptr;
    a.mask_words = static_cast<int64_t>(mask->bytes / 4);
  }
  if (!decode) {
    a.q_rows = static_cast<int32_t>(q_rows);
    a.kv_rows = static_cast<int32_t>(kv_rows);
    int ce = encode_q_map(&a.tm_q, q, hp.total_q, desc->num_qo_heads, desc->head_dim, G,
                          tile_tokens);
    if (ce == 0) ce = encode_rows_map(&a.tm_k, k_cache, kv_rows, desc->head_dim);
    if (ce == 0) ce = encode_rows_map(&a.tm_v, v_cache, kv_rows, desc->head_dim);
    if (ce == 0 && desc->head_dim == 256 && desc->page_size >= 16) {
      const int64_t slots = num_pages * desc->page_size;
      ce = encode_slots_map(&a.tm_k3, k_cache, slots, desc->num_kv_heads, desc->head_dim);
      if (ce == 0) ce = encode_slots_map(&a.tm_v3, v_cache, slots, desc->num_kv_heads, desc->head_dim);
    }
    if (ce != 0) return fail(BIA_ERR_CUDA, "cuTensorMapEncodeTiled failed or unavailable", ce);
  }

  const bool profile = g_attn_begin != nullptr && g_attn_end != nullptr;
  if (profile) {
    const cudaError_t re = cudaEventRecord(g_attn_begin, st);
    if (re != cudaSuccess) return cuda_fail("profile event record", re);
  }
  // a prefill call with both kinds of tile forks its streamed single-token
  // tiles onto the side stream (after the plan) and joins it before the merge
  SideStream *side = !decode && hp.n_units > 0 && hp.n_sunits > 0 ? side_stream(st) : nullptr;
  if (side && (cudaEventRecord(side->fork, st) != cudaSuccess ||
               cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)) {
    // a stale handle (the device was reset): forget it, stay on one stream
    (void)cudaGetLastError();
    *side = SideStream{};
    side = nullptr;
  }
  cudaError_t e = decode                     ? bia::launch_decode(a, st)
                  : desc->head_dim == 256 ? bia::launch_prefill_wide(a, st)
                                          : bia::launch_prefill(a, st);
  if (e != cudaSuccess) return cuda_fail(decode ? "decode kernel launch" : "prefill kernel launch", e);
  if (hp.n_units > 0) __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  if (hp.n_sunits > 0) { // single-token q tiles of a prefill call, streamed
    AttnArgs sa = a;
    sa.units = pa.sunits;
    sa.n_units = hp.n_sunits;
    e = bia::launch_decode(sa, side ? side->stream : st);
    if (e != cudaSuccess) return cuda_fail("streamed-tile kernel launch", e);
    __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  }
  if (side) {
    cudaError_t je = cudaEventRecord(side->join, side->stream);
    if (je == cudaSuccess) je = cudaStreamWaitEvent(st, side->join, 0);
    if (je != cudaSuccess) return cuda_fail("side stream join", je);
  }
  if (profile) {
    const cudaError_t re = cudaEventRecord(g_attn_end, st);
    if (re != cudaSuccess) return cuda_fail("profile event record", re);
  }
  if (hp.part_rows > 0) {
    e = bia::launch_merge_partials(a, st);
    if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
    __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  }
  return BIA_OK;
}

size_t workspace_size(bool decode, const bia_attn_desc *desc, const int32_t *qo_host,
                      const int32_t *kvp_host, const int32_t *last_host, int32_t batch,
                      int32_t causal, int32_t split, const bia_bounds *bounds = nullptr) {
  if (check_desc(desc) != BIA_OK) return 0;
  if (!decode && !qo_host && !bounds) return 0;
  if (split == 0) split = decode ? BIA_DECODE_SPLIT : BIA_PREFILL_SPLIT;
  const int G = desc->num_qo_heads / desc->num_kv_heads;
  const int tile_tokens = decode ? 1 : bia::kTileRows / G;
  const int tiles_per_unit = decode ? 1 : bia::prefill_tiles_per_unit(desc->head_dim);
  const int ctas = decode ? 1 : bia::kPrefillClusterCtas;
  HostPlan hp;
  const int rc = bounds ? bounded_plan(bounds, batch, decode ? 1 : causal, split, tile_tokens,
                                       tiles_per_unit, ctas, decode ? 0 : 1, decode, &hp)
                        : host_plan(desc, decode ? nullptr : qo_host, kvp_host, last_host, batch,
                                    decode ? 1 : causal, split, tile_tokens, tiles_per_unit, ctas,
                                    decode ? 0 : 1, &hp);
  if (rc != BIA_OK) return 0;
  return bia::make_layout(batch, hp.n_groups, hp.n_units, hp.n_sunits, hp.part_rows,
                          desc->num_qo_heads, desc->head_dim)
      .total;
}

} // namespace

extern "C" {

int bia_prefill_paged(const bia_attn_desc *desc, const void *q, const void *k_cache,
                      const void *v_cache, int64_t num_pages, const int32_t *qo_indptr,
                      const int32_t *kv_indptr, const int32_t *kv_indices,
                      const int32_t *kv_last_page_len, const int32_t *qo_indptr_host,
                      const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                      int32_t batch, int32_t causal, int32_t split_size, void *workspace,
                      size_t workspace_bytes, void *out, float *lse, void *stream) {
  return run_attention(false, desc, q, k_cache, v_cache, num_pages, qo_indptr, kv_indptr,
                       kv_indices, kv_last_page_len, qo_indptr_host, kv_indptr_host,
                       kv_last_page_len_host, batch, causal ? 1 : 0, split_size, workspace,
                       workspace_bytes, out, lse, stream);
}

int bia_prefill_paged_mask(const bia_attn_desc *desc, const void *q, const void *k_cache,
                           const void *v_cache, int64_t num_pages, const int32_t *qo_indptr,
                           const int32_t *kv_indptr, const int32_t *kv_indices,
                           const int32_t *kv_last_page_len, const int32_t *qo_indptr_host,
                           const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                           int32_t batch, int32_t causal, int32_t split_size,
                           const void *mask, size_t mask_bytes, const int64_t *mask_indptr,
                           const int64_t *mask_indptr_host, void *workspace,
                           size_t workspace_bytes, void *out, float *lse, void *stream) {
  const MaskArgs m{mask, mask_bytes, mask_indptr, mask_indptr_host};
  CallOpts opt;
  opt.mask = &m;
  return run_attention(false, desc, q, k_cache, v_cache, num_pages, qo_indptr, kv_indptr,
                       kv_indices, kv_last_page_len, qo_indptr_host, kv_indptr_host,
                       kv_last_page_len_host, batch, causal ? 1 : 0, split_size, workspace,
                       workspace_bytes, out, lse, stream, opt);
}

size_t bia_prefill_workspace_size(const bia_attn_desc *desc, const int32_t *qo_indptr_host,
                                  const int32_t *kv_indptr_host,
                                  const int32_t *kv_last_page_len_host, int32_t batch,
                                  int32_t causal, int32_t split_size) {
  return workspace_size(false, desc, qo_indptr_host, kv_indptr_host, kv_last_page_len_host,
                        batch, causal ? 1 : 0, split_size);
}

int bia_decode_paged(const bia_attn_desc *desc, const void *q, const void *k_cache,
                     const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                     const int32_t *kv_indices, const int32_t *kv_last_page_len,
                     const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                     int32_t batch, int32_t split_size, void *workspace, size_t workspace_bytes,
                     void *out, float *lse, void *stream) {
  return run_attention(true, desc, q, k_cache, v_cache, num_pages, nullptr, kv_indptr,
                       kv_indices, kv_last_page_len, nullptr, kv_indptr_host,
                       kv_last_page_len_host, batch, 1, split_size, workspace, workspace_bytes,
                       out, lse, stream);
}

size_t bia_decode_workspace_size(const bia_attn_desc *desc, const int32_t *kv_indptr_host,
                                 const int32_t *kv_last_page_len_host, int32_t batch,
                                 int32_t split_size) {
  return workspace_size(true, desc, nullptr, kv_indptr_host, kv_last_page_len_host, batch, 1,
                        split_size);
}

int bia_prefill_paged_bounded(const bia_attn_desc *desc, const bia_bounds *bounds,
                              const void *q, const void *k_cache, const void *v_cache,
                              int64_t num_pages, const int32_t *qo_indptr,
                              const int32_t *kv_indptr, const int32_t *kv_indices,
                              const int32_t *kv_last_page_len, int32_t batch, int32_t causal,
                              int32_t split_size, void *workspace, size_t workspace_bytes,
                              void *out, float *lse, void *stream) {
  if (!bounds) return BIA_ERR_INVALID_ARG;
  CallOpts opt;
  opt.bounds = bounds;
  return run_attention(false, desc, q, k_cache, v_cache, num_pages, qo_indptr, kv_indptr,
                       kv_indices, kv_last_page_len, nullptr, nullptr, nullptr, batch,
                       causal ? 1 : 0, split_size, workspace, workspace_bytes, out, lse, stream,
                       opt);
}

size_t bia_prefill_bounded_workspace_size(const bia_attn_desc *desc, const bia_bounds *bounds,
                                          int32_t batch, int32_t causal, int32_t split_size) {
  if (!bounds) return 0;
  return workspace_size(false, desc, nullptr, nullptr, nullptr, batch, causal ? 1 : 0,
                        split_size, bounds);
}

int bia_decode_paged_bounded(const bia_attn_desc *desc, const bia_bounds *bounds, const void *q,
                             const void *k_cache, const void *v_cache, int64_t num_pages,
                             const int32_t *kv_indptr, const int32_t *kv_indices,
                             const int32_t *kv_last_page_len, int32_t batch, int32_t split_size,
                             void *workspace, size_t workspace_bytes, void *out, float *lse,
                             void *stream) {
  if (!bounds) return BIA_ERR_INVALID_ARG;
  CallOpts opt;
  opt.bounds = bounds;
  return run_attention(true, desc, q, k_cache, v_cache, num_pages, nullptr, kv_indptr,
                       kv_indices, kv_last_page_len, nullptr, nullptr, nullptr, batch, 1,
                       split_size, workspace, workspace_bytes, out, lse, stream, opt);
}

size_t bia_decode_bounded_workspace_size(const bia_attn_desc *desc, const bia_bounds *bounds,
                                         int32_t batch, int32_t split_size) {
  if (!bounds) return 0;
  return workspace_size(true, desc, nullptr, nullptr, nullptr, batch, 1, split_size, bounds);
}

int bia_merge_states(const float *v, const float *s, const int32_t *num_states, int64_t n,
                     int32_t num_states_max, int32_t num_heads, int32_t head_dim, void *out,
                     float *out_lse, void *stream) {
  if (n < 0 || num_states_max <= 0 || num_heads <= 0 || head_dim <= 0) return BIA_ERR_INVALID_ARG;
  if (head_dim % 4 != 0 || head_dim > 512) return BIA_ERR_UNSUPPORTED;
  if (n == 0) return BIA_OK;
  if (!v || !s || !out) return BIA_ERR_INVALID_ARG;
  if (misaligned(v, 16) || misaligned(out, 8) || misaligned(s, 4) || misaligned(out_lse, 4) ||
      misaligned(num_states, 4))
    return BIA_ERR_INVALID_ARG;
  const int rc = check_resident({{"v", v},
                                 {"s", s},
                                 {"num_states", num_states},
                                 {"out", out},
                                 {"out_lse", out_lse}});
  if (rc != BIA_OK) return rc;
  cudaError_t e = bia::launch_merge_states(v, s, num_states, n, num_states_max, num_heads,
                                           head_dim, static_cast<uint16_t *>(out), out_lse,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
  __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  return BIA_OK;
}

int bia_append_paged_kv(const bia_attn_desc *desc, const void *k_new, const void *v_new,
                        void *k_cache, void *v_cache, int64_t num_pages,
                        const int32_t *append_indptr, const int32_t *kv_indptr,
                        const int32_t *kv_indices, const int32_t *kv_last_page_len,
                        const int32_t *append_indptr_host, const int32_t *kv_indptr_host,
                        const int32_t *kv_last_page_len_host, int32_t batch, int32_t *status,
                        void *stream) {
  int rc = check_desc(desc);
  if (rc != BIA_OK) return rc;
  if (batch <= 0 || !append_indptr_host || !kv_indptr_host || !kv_last_page_len_host)
    return BIA_ERR_INVALID_ARG;
  if (append_indptr_host[0] != 0 || kv_indptr_host[0] < 0) return BIA_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    const int64_t n_new = static_cast<int64_t>(append_indptr_host[b + 1]) - append_indptr_host[b];
    const int64_t pages = static_cast<int64_t>(kv_indptr_host[b + 1]) - kv_indptr_host[b];
    if (n_new < 0 || pages < 0) return BIA_ERR_INVALID_ARG;
    const int32_t last = kv_last_page_len_host[b];
    if (pages > 0 && (last < 1 || last > desc->page_size)) return BIA_ERR_INVALID_ARG;
    const int64_t kv_len = pages > 0 ? (pages - 1) * desc->page_size + last : 0;
    if (kv_len > INT32_MAX / 2) return BIA_ERR_UNSUPPORTED;
    if (n_new > kv_len) return BIA_ERR_INVALID_ARG;
  }
  const int64_t total_new = append_indptr_host[batch];
  if (misaligned(status, 4)) return BIA_ERR_INVALID_ARG;
  if (total_new > 0) {
    if (!k_new || !v_new || !k_cache || !v_cache || !append_indptr || !kv_indptr ||
        !kv_indices || !kv_last_page_len || num_pages <= 0)
      return BIA_ERR_INVALID_ARG;
    if (misaligned(k_new, 16) || misaligned(v_new, 16) || misaligned(k_cache, 16) ||
        misaligned(v_cache, 16) || misaligned(append_indptr, 4) || misaligned(kv_indptr, 4) ||
        misaligned(kv_indices, 4) || misaligned(kv_last_page_len, 4))
      return BIA_ERR_INVALID_ARG;
  }
  if (total_new > 0 || status) {
    rc = check_resident({{"status", status},
                         {"k_new", total_new > 0 ? k_new : nullptr},
                         {"v_new", total_new > 0 ? v_new : nullptr},
                         {"k_cache", total_new > 0 ? k_cache : nullptr},
                         {"v_cache", total_new > 0 ? v_cache : nullptr},
                         {"append_indptr", total_new > 0 ? append_indptr : nullptr},
                         {"kv_indptr", total_new > 0 ? kv_indptr : nullptr},
                         {"kv_indices", total_new > 0 ? kv_indices : nullptr},
                         {"kv_last_page_len", total_new > 0 ? kv_last_page_len : nullptr}});
    if (rc != BIA_OK) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (status) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_fail("status reset", e);
  }
  if (total_new == 0) return BIA_OK;
  bia::AppendArgs a{};
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.k_cache = static_cast<uint16_t *>(k_cache);
  a.v_cache = static_cast<uint16_t *>(v_cache);
  a.append_indptr = append_indptr;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.kv_last_page_len = kv_last_page_len;
  a.num_pages = num_pages;
  a.total_new = total_new;
  a.batch = batch;
  a.Hkv = desc->num_kv_heads;
  a.D = desc->head_dim;
  a.page_size = desc->page_size;
  a.status = status;
  cudaError_t e = bia::launch_append(a, st);
  if (e != cudaSuccess) return cuda_fail("append kernel launch", e);
  __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  return BIA_OK;
}

} // extern "C"

namespace bia {

int decode_check(const bia_attn_desc *desc, const void *q, const void *k_cache,
                 const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                 const int32_t *kv_indices, const int32_t *kv_last_page_len,
                 const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                 int32_t batch, int32_t split_size, void *out, float *lse, size_t *need) {
  CallOpts opt;
  opt.need = need;
  return run_attention(true, desc, q, k_cache, v_cache, num_pages, nullptr, kv_indptr,
                       kv_indices, kv_last_page_len, nullptr, kv_indptr_host,
                       kv_last_page_len_host, batch, 1, split_size, nullptr, 0, out, lse,
                       nullptr, opt);
}

int decode_on_scratch(const bia_attn_desc *desc, const void *q, const void *k_cache,
                      const void *v_cache, int64_t num_pages, const int32_t *kv_indptr,
                      const int32_t *kv_indices, const int32_t *kv_last_page_len,
                      const int32_t *kv_indptr_host, const int32_t *kv_last_page_len_host,
                      int32_t batch, int32_t split_size, void *scratch, size_t scratch_bytes,
                      void *out, float *lse, void *stream) {
  CallOpts opt;
  opt.ws_static = true;
  return run_attention(true, desc, q, k_cache, v_cache, num_pages, nullptr, kv_indptr,
                       kv_indices, kv_last_page_len, nullptr, kv_indptr_host,
                       kv_last_page_len_host, batch, 1, split_size, scratch, scratch_bytes, out,
                       lse, stream, opt);
}

} // namespace bia

extern "C" {

namespace {
// Multi-head latent attention: validation and plan sizes as for the GQA
// decode (qo_host == nullptr, one query per request) or a causal extend of
// one-token q tiles (qo_host given), with one shared 512 + 64 wide latent
// "kv head".
// Tokens per q tile of an MLA call: an extend with 8 or 16 heads takes 32/Hq
// consecutive tokens per CTA (their heads fill the kernel's 32 columns and
// share each key block); a decode, or more heads, one token.
int mla_tile_tokens(int num_heads, bool extend) {
  return extend && num_heads < 32 && 32 % num_heads == 0 ? 32 / num_heads : 1;
}

int mla_plan(const bia_mla_desc *d, const int32_t *qo_host, const int32_t *kvp_host,
             const int32_t *last_host, int32_t batch, int32_t split, HostPlan *hp) {
  if (!d || d->page_size <= 0) return BIA_ERR_INVALID_ARG;
  if (d->num_heads <= 0 || d->num_heads % 8 != 0 || d->num_heads > 1024) return BIA_ERR_UNSUPPORTED;
  if (!is_pow2(d->page_size) || d->page_size > 256) return BIA_ERR_UNSUPPORTED;
  if (!std::isfinite(d->sm_scale)) return BIA_ERR_INVALID_ARG;
  const bia_attn_desc as_attn{d->num_heads, 1, BIA_MLA_CKV_DIM, d->page_size, d->sm_scale};
  return host_plan(&as_attn, qo_host, kvp_host, last_host, batch, 1, split,
                   mla_tile_tokens(d->num_heads, qo_host != nullptr), 1, 1, 0, hp);
}

size_t mla_workspace_size(const bia_mla_desc *desc, const int32_t *qo_host,
                          const int32_t *kvp_host, const int32_t *last_host, int32_t batch,
                          int32_t split) {
  HostPlan hp;
  if (mla_plan(desc, qo_host, kvp_host, last_host, batch, split, &hp) != BIA_OK) return 0;
  return bia::make_layout(batch, hp.n_groups, hp.n_units, 0, hp.part_rows, desc->num_heads,
                          BIA_MLA_CKV_DIM)
      .total;
}

// One MLA call: extend (qo_indptr given) or decode (qo_indptr == nullptr).
int run_mla(const bia_mla_desc *desc, const void *q_nope, const void *q_pe,
            const void *ckv_cache, const void *kpe_cache, int64_t num_pages,
            const int32_t *qo_indptr, const int32_t *kv_indptr, const int32_t *kv_indices,
            const int32_t *kv_last_page_len, const int32_t *qo_host, const int32_t *kvp_host,
            const int32_t *last_host, int32_t batch, int32_t split_size, void *workspace,
            size_t workspace_bytes, void *out, float *lse, void *stream) {
  const bool extend = qo_host != nullptr;
  if (!q_nope || !q_pe || !ckv_cache || !kpe_cache || !kv_indptr || !kv_indices ||
      !kv_last_page_len || !out || !workspace || num_pages <= 0 || (extend && !qo_indptr))
    return BIA_ERR_INVALID_ARG;
  if (misaligned(workspace, 256)) return BIA_ERR_INVALID_ARG;
  if (misaligned(q_nope, 16) || misaligned(q_pe, 16) || misaligned(ckv_cache, 16) ||
      misaligned(kpe_cache, 16) || misaligned(out, 16) || misaligned(lse, 4) ||
      misaligned(qo_indptr, 4) || misaligned(kv_indptr, 4) || misaligned(kv_indices, 4) ||
      misaligned(kv_last_page_len, 4))
    return BIA_ERR_INVALID_ARG;
  HostPlan hp;
  int rc = mla_plan(desc, qo_host, kvp_host, last_host, batch, split_size, &hp);
  if (rc != BIA_OK) return rc;
  const WsLayout w = bia::make_layout(batch, hp.n_groups, hp.n_units, 0, hp.part_rows,
                                      desc->num_heads, BIA_MLA_CKV_DIM);
  if (workspace_bytes < w.total) return BIA_ERR_WORKSPACE_TOO_SMALL;
  if (hp.total_q == 0) return BIA_OK;
  // tensor maps: the heads' q rows in 16-row boxes, the latent rows one row
  // per box (gathered)
  const int64_t q_rows = hp.total_q * desc->num_heads;
  const int64_t kv_rows = num_pages * desc->page_size;
  if (q_rows >= INT32_MAX || kv_rows >= INT32_MAX) return BIA_ERR_UNSUPPORTED;
  rc = check_resident({{"q_nope", q_nope},
                       {"q_pe", q_pe},
                       {"ckv_cache", ckv_cache},
                       {"kpe_cache", kpe_cache},
                       {"out", out},
                       {"lse", lse},
                       {"qo_indptr", extend ? qo_indptr : nullptr},
                       {"kv_indptr", kv_indptr},
                       {"kv_indices", kv_indices},
                       {"kv_last_page_len", kv_last_page_len},
                       {"workspace", workspace}});
  if (rc != BIA_OK) return rc;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  PlanArgs pa{};
  pa.qo_indptr = extend ? qo_indptr : nullptr;
  pa.kv_indptr = kv_indptr;
  pa.kv_last_page_len = kv_last_page_len;
  pa.batch = batch;
  pa.page_size = desc->page_size;
  const int mla_tt = mla_tile_tokens(desc->num_heads, extend);
  pa.tile_tokens = mla_tt;
  pa.tiles_per_unit = 1;
  pa.ctas = 1;
  pa.causal = 1;
  pa.split = split_size;
  pa.n_groups_expected = hp.n_groups;
  pa.n_units_expected = hp.n_units;
  pa.part_rows_expected = hp.part_rows;
  pa.out = static_cast<uint16_t *>(out);
  pa.out_elems = hp.total_q * desc->num_heads * BIA_MLA_CKV_DIM;
  pa.lse = lse;
  pa.lse_elems = hp.total_q * desc->num_heads;
  pa.status = reinterpret_cast<int32_t *>(ws + w.status);
  pa.reqs = reinterpret_cast<bia::ReqInfo *>(ws + w.reqs);
  pa.group_off = reinterpret_cast<int32_t *>(ws + w.group_off);
  pa.group_cnt = reinterpret_cast<int32_t *>(ws + w.group_cnt);
  pa.units = reinterpret_cast<bia::Unit *>(ws + w.units);
  cudaError_t e = bia::launch_plan(pa, st);
  if (e != cudaSuccess) return cuda_fail("plan kernel launch", e);
  __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);

  AttnArgs a{};
  a.q = static_cast<const uint16_t *>(q_nope);
  a.q_pe = static_cast<const uint16_t *>(q_pe);
  a.k_cache = static_cast<const uint16_t *>(ckv_cache);
  a.kpe_cache = static_cast<const uint16_t *>(kpe_cache);
  a.kv_indices = kv_indices;
  a.qo_indptr = pa.qo_indptr;
  a.num_pages = num_pages;
  a.Hq = desc->num_heads;
  a.Hkv = 1;
  a.D = BIA_MLA_CKV_DIM;
  a.G = desc->num_heads;
  a.page_shift = log2i(desc->page_size);
  a.causal = 1;
  a.split = split_size;
  a.tile_tokens = mla_tt;
  const float sc = desc->sm_scale > 0.f
                       ? desc->sm_scale
                       : 1.0f / std::sqrt(static_cast<float>(BIA_MLA_CKV_DIM + BIA_MLA_KPE_DIM));
  a.scale_log2 = sc * 1.4426950408889634f;
  a.batch = batch;
  a.n_units = hp.n_units;
  a.reqs = pa.reqs;
  a.units = pa.units;
  a.part_o = reinterpret_cast<float *>(ws + w.part_o);
  a.part_lse = reinterpret_cast<float *>(ws + w.part_lse);
  a.total_rows = hp.total_q;
  a.out = static_cast<uint16_t *>(out);
  a.lse = lse;
  a.status = pa.status;
  a.q_rows = static_cast<int32_t>(q_rows);
  a.kv_rows = static_cast<int32_t>(kv_rows);
  const int hg = mla_tt > 1 ? 32 : bia::mla_head_group(desc->num_heads);
  int ce = encode_2d_map(&a.tm_q, q_nope, q_rows, BIA_MLA_CKV_DIM, hg);
  if (ce == 0) ce = encode_2d_map(&a.tm_qpe, q_pe, q_rows, BIA_MLA_KPE_DIM, hg);
  if (ce == 0) ce = encode_2d_map(&a.tm_k, ckv_cache, kv_rows, BIA_MLA_CKV_DIM, 1);
  if (ce == 0) ce = encode_2d_map(&a.tm_kpe, kpe_cache, kv_rows, BIA_MLA_KPE_DIM, 1);
  if (ce != 0) return fail(BIA_ERR_CUDA, "cuTensorMapEncodeTiled failed or unavailable", ce);
  const bool profile = g_attn_begin != nullptr && g_attn_end != nullptr;
  if (profile) {
    const cudaError_t re = cudaEventRecord(g_attn_begin, st);
    if (re != cudaSuccess) return cuda_fail("profile event record", re);
  }
  e = bia::launch_mla_decode(a, st);
  if (e != cudaSuccess) return cuda_fail("mla kernel launch", e);
  if (hp.n_units > 0) __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  if (profile) {
    const cudaError_t re = cudaEventRecord(g_attn_end, st);
    if (re != cudaSuccess) return cuda_fail("profile event record", re);
  }
  if (hp.part_rows > 0) {
    e = bia::launch_merge_partials(a, st);
    if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
    __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  }
  return BIA_OK;
}
} // namespace

size_t bia_mla_decode_workspace_size(const bia_mla_desc *desc, const int32_t *kv_indptr_host,
                                     const int32_t *kv_last_page_len_host, int32_t batch,
                                     int32_t split_size) {
  return mla_workspace_size(desc, nullptr, kv_indptr_host, kv_last_page_len_host, batch,
                            split_size == 0 ? BIA_DECODE_SPLIT : split_size);
}

int bia_mla_decode_paged(const bia_mla_desc *desc, const void *q_nope, const void *q_pe,
                         const void *ckv_cache, const void *kpe_cache, int64_t num_pages,
                         const int32_t *kv_indptr, const int32_t *kv_indices,
                         const int32_t *kv_last_page_len, const int32_t *kv_indptr_host,
                         const int32_t *kv_last_page_len_host, int32_t batch, int32_t split_size,
                         void *workspace, size_t workspace_bytes, void *out, float *lse,
                         void *stream) {
  return run_mla(desc, q_nope, q_pe, ckv_cache, kpe_cache, num_pages, nullptr, kv_indptr,
                 kv_indices, kv_last_page_len, nullptr, kv_indptr_host, kv_last_page_len_host,
                 batch, split_size == 0 ? BIA_DECODE_SPLIT : split_size, workspace,
                 workspace_bytes, out, lse, stream);
}

size_t bia_mla_prefill_workspace_size(const bia_mla_desc *desc, const int32_t *qo_indptr_host,
                                      const int32_t *kv_indptr_host,
                                      const int32_t *kv_last_page_len_host, int32_t batch,
                                      int32_t split_size) {
  if (!qo_indptr_host) return 0;
  return mla_workspace_size(desc, qo_indptr_host, kv_indptr_host, kv_last_page_len_host, batch,
                            split_size == 0 ? BIA_PREFILL_SPLIT : split_size);
}

int bia_mla_prefill_paged(const bia_mla_desc *desc, const void *q_nope, const void *q_pe,
                          const void *ckv_cache, const void *kpe_cache, int64_t num_pages,
                          const int32_t *qo_indptr, const int32_t *kv_indptr,
                          const int32_t *kv_indices, const int32_t *kv_last_page_len,
                          const int32_t *qo_indptr_host, const int32_t *kv_indptr_host,
                          const int32_t *kv_last_page_len_host, int32_t batch, int32_t split_size,
                          void *workspace, size_t workspace_bytes, void *out, float *lse,
                          void *stream) {
  if (!qo_indptr_host) return BIA_ERR_INVALID_ARG;
  return run_mla(desc, q_nope, q_pe, ckv_cache, kpe_cache, num_pages, qo_indptr, kv_indptr,
                 kv_indices, kv_last_page_len, qo_indptr_host, kv_indptr_host,
                 kv_last_page_len_host, batch, split_size == 0 ? BIA_PREFILL_SPLIT : split_size,
                 workspace, workspace_bytes, out, lse, stream);
}

int32_t bia_q_tile_tokens(int32_t gqa_group) {
  if (gqa_group <= 0 || bia::kTileRows % gqa_group != 0) return 0;
  return bia::kTileRows / gqa_group;
}

const char *bia_status_string(int status) {
  switch (status) {
  case BIA_OK: return "ok";
  case BIA_ERR_INVALID_ARG: return "invalid argument";
  case BIA_ERR_UNSUPPORTED: return "unsupported configuration";
  case BIA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
  case BIA_ERR_CUDA: return "CUDA error";
  default: return "unknown status";
  }
}

int bia_read_status(const void *workspace, int32_t *status_out, void *stream) {
  if (!workspace || !status_out) return BIA_ERR_INVALID_ARG;
  const int rc = check_resident({{"workspace", workspace}});
  if (rc != BIA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail("status copy", e);
  e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? BIA_OK : cuda_fail("status copy synchronize", e);
}

void bia_set_profile_events(void *attn_begin, void *attn_end) {
  g_attn_begin = static_cast<cudaEvent_t>(attn_begin);
  g_attn_end = static_cast<cudaEvent_t>(attn_end);
}

uint64_t bia_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

const char *bia_last_error(void) { return g_last_error; }

} // extern "C"

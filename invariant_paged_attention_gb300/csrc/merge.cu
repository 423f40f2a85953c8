// Fixed-order log-sum-exp merge kernels.  One warp per output row (token,
// q head): lane i holds elements 4i..4i+3 (+128k), every split is folded in
// ascending order by fold_state, so the result depends only on the partial
// states, never on the grid.
#include <algorithm>

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

// load_state from shared memory.
template <int V>
__device__ __forceinline__ void load_state_smem(const float *row, int D, int lane, float (&v)[V]) {
#pragma unroll
  for (int k = 0; k < V; k += 4) {
    const int e = (k / 4) * 128 + lane * 4;
    if (e < D) {
      const float4 x = *reinterpret_cast<const float4 *>(row + e);
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

// The request owning merge row m: largest b with reqs[b].mbase <= m (requests
// with no rows to merge share the next one's mbase, and the largest index
// is the one with rows).
__device__ __forceinline__ int merge_owner(const ReqInfo *reqs, int batch, int64_t m) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (reqs[mid].mbase <= m)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Merge of the split partials a prefill / decode call left in the workspace.
// The planner lists the rows to merge: the tokens of q tiles that span more
// than one split (a suffix of each request), numbered across requests; a
// grid of two CTAs per SM takes them in contiguous ranges, a token at a time,
// its q heads spread over the warps.  A warp takes HB of its heads at a time: lane s
// loads the LSE of split s of each (all splits in flight at once), then the
// states of two splits of the HB heads are loaded together and folded
// in ascending split order, so a row's loads do not wait for the fold of the
// previous split.  Rows of single-split tiles were written by the attention
// kernel.
template <int V>
__global__ void __launch_bounds__(kMergeWarps * 32, 2)
    merge_partials_kernel(const AttnArgs a) {
  constexpr int kHb = V <= 4 ? 4 : V <= 8 ? 2 : 1; // heads a warp folds at once
  constexpr int kChunk = 2;                        // splits loaded at once
  const int D = a.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait(); // the attention kernel's partials (and the plan) are complete
  // a plan that failed its checks computed nothing (out already holds NaN)
  if (a.status[0] & kStatusPlanMismatch) return;
  const int64_t n_merge = a.status[kStatusMergeRows];
  // this CTA's rows: a contiguous range, its first owner found once, then
  // followed request by request
  const int64_t per = (n_merge + gridDim.x - 1) / gridDim.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t m1 = min(n_merge, m0 + per);
  if (m0 >= m1) return;
  int b = merge_owner(a.reqs, a.batch, m0);
  ReqInfo r = a.reqs[b];
  int32_t first = merge_first_token(r.q_len, r.kv_len, a.tile_tokens, a.causal, a.split);
  int64_t next = b + 1 < a.batch ? a.reqs[b + 1].mbase : INT64_MAX;
  for (int64_t m = m0; m < m1; ++m) {
    while (m >= next) { // the next request with rows (empty ones share its mbase)
      ++b;
      r = a.reqs[b];
      first = merge_first_token(r.q_len, r.kv_len, a.tile_tokens, a.causal, a.split);
      next = b + 1 < a.batch ? a.reqs[b + 1].mbase : INT64_MAX;
    }
    const int32_t t = first + static_cast<int32_t>(m - r.mbase);
    const int64_t token = static_cast<int64_t>(r.q_start) + t;
    const int32_t tile = t / a.tile_tokens;
    const int32_t n_tile = tile_splits(r.q_len, r.kv_len, tile, a.tile_tokens, a.causal, a.split);
    const int32_t p = a.causal ? r.kv_len - r.q_len + t : r.kv_len - 1;
    const int32_t n_row = min(n_tile, p / a.split + 1);
    const int64_t base = (r.rowbase + static_cast<int64_t>(t) * r.nsp) * a.Hq;
    for (int h0 = warp; h0 < a.Hq; h0 += kMergeWarps * kHb) {
      float L[kHb], o[kHb][V];
#pragma unroll
      for (int i = 0; i < kHb; ++i) {
        L[i] = -INFINITY;
#pragma unroll
        for (int e = 0; e < V; ++e) o[i][e] = 0.f;
      }
      for (int s0 = 0; s0 < n_row; s0 += 32) {
        const int n_here = min(32, n_row - s0);
        float ls_lane[kHb];
#pragma unroll
        for (int i = 0; i < kHb; ++i) {
          const int h = h0 + i * kMergeWarps;
          ls_lane[i] = lane < n_here && h < a.Hq
              ? __ldg(a.part_lse + base + static_cast<int64_t>(s0 + lane) * a.Hq + h) : -INFINITY;
        }
        for (int k0 = 0; k0 < n_here; k0 += kChunk) {
          float ls[kHb][kChunk], v[kHb][kChunk][V];
#pragma unroll
          for (int i = 0; i < kHb; ++i)
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
              const int h = h0 + i * kMergeWarps;
              ls[i][c] = __shfl_sync(0xffffffffu, ls_lane[i], (k0 + c) & 31);
              if (k0 + c < n_here && h < a.Hq && ls[i][c] != -INFINITY) {
                const int64_t idx = base + static_cast<int64_t>(s0 + k0 + c) * a.Hq + h;
                load_state<V>(a.part_o + idx * D, D, lane, v[i][c]);
              } else {
                ls[i][c] = -INFINITY; // fold_state skips it
              }
            }
#pragma unroll
          for (int i = 0; i < kHb; ++i)
#pragma unroll
            for (int c = 0; c < kChunk; ++c) fold_state<V>(L[i], o[i], ls[i][c], v[i][c]);
        }
      }
#pragma unroll
      for (int i = 0; i < kHb; ++i) {
        const int h = h0 + i * kMergeWarps;
        if (h >= a.Hq) break;
        if (L[i] == -INFINITY) {
#pragma unroll
          for (int e = 0; e < V; ++e) o[i][e] = 0.f;
        }
        const int64_t row = token * a.Hq + h;
        store_row<V>(a.out + row * D, D, a.lse ? a.lse + row : nullptr, lane, L[i], o[i]);
      }
    }
  }
}

// The same merge with the partial states streamed through shared memory:
// each (token, split, chunk of hc heads) block of partials is contiguous in
// the workspace (hc*D fp32 values, and hc LSE values), so one thread of a
// copy warp moves it with two bulk copies into a ring of stages while eight
// fold warps fold the stages in order: per head, splits ascending, exactly as
// merge_partials_kernel does (the same bits), with up to kMStages blocks in
// flight per CTA instead of what the registers of the fold warps can hold.
// Needs Hq % 4 == 0 (16-byte-aligned LSE blocks).
constexpr int kMStageO = 16384;  // partial values of one stage (<= 64 heads)
constexpr int kMStageL = 256;    // LSE values of one stage
constexpr int kMStages = 6;
constexpr int kMThreads = (kMergeWarps + 1) * 32; // fold warps + the copy warp
constexpr int kMSmem = kMStages * (kMStageO + kMStageL) + 2 * kMStages * 8;

// Heads of one stage: what fits kMStageO, a multiple of 8 (one head per fold
// warp and round), and at most 16/V rounds (the fold warps' registers).
__host__ __device__ inline int merge_chunk_heads(int Hq, int D) {
  const int V = D <= 128 ? 4 : D <= 256 ? 8 : 16;
  int hc = (kMStageO / (D * 4)) & ~7;
  if (hc > kMergeWarps * (16 / V)) hc = kMergeWarps * (16 / V);
  return Hq < hc ? Hq : hc;
}

template <int V>
__global__ void __launch_bounds__(kMThreads, 2) merge_stream_kernel(const AttnArgs a) {
  constexpr int kMaxHpw = 16 / V; // heads of a chunk per fold warp
  extern __shared__ __align__(128) uint8_t msm[];
  const uint32_t sbase = smem_u32(msm);
  auto stage_o = [&](int st) { return sbase + static_cast<uint32_t>(st) * kMStageO; };
  auto stage_l = [&](int st) {
    return sbase + kMStages * kMStageO + static_cast<uint32_t>(st) * kMStageL;
  };
  auto full = [&](int st) {
    return sbase + kMStages * (kMStageO + kMStageL) + 8u * static_cast<uint32_t>(st);
  };
  auto empty = [&](int st) { return full(kMStages) + 8u * static_cast<uint32_t>(st); };
  const int D = a.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  grid_dep_wait(); // the attention kernel's partials (and the plan) are complete
  if (a.status[0] & kStatusPlanMismatch) return;
  const int64_t n_merge = a.status[kStatusMergeRows];
  const int64_t per = (n_merge + gridDim.x - 1) / gridDim.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t m1 = min(n_merge, m0 + per);
  if (m0 >= m1) return;
  const int hc = merge_chunk_heads(a.Hq, D);
  const int n_hc = (a.Hq + hc - 1) / hc;
  if (threadIdx.x == 0) {
    for (int st = 0; st < kMStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kMergeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // both roles walk the same items: rows m0..m1-1, head chunks, splits
  int b = merge_owner(a.reqs, a.batch, m0);
  ReqInfo r = a.reqs[b];
  int32_t first = merge_first_token(r.q_len, r.kv_len, a.tile_tokens, a.causal, a.split);
  int64_t next = b + 1 < a.batch ? a.reqs[b + 1].mbase : INT64_MAX;
  uint32_t k = 0; // item counter: stage k % kMStages, its use k / kMStages
  bool ok = true;
  if (warp == kMergeWarps) {
    // ------------------------------------------------------------ copies
    if (lane == 0) {
      for (int64_t m = m0; m < m1 && ok; ++m) {
        while (m >= next) {
          ++b;
          r = a.reqs[b];
          first = merge_first_token(r.q_len, r.kv_len, a.tile_tokens, a.causal, a.split);
          next = b + 1 < a.batch ? a.reqs[b + 1].mbase : INT64_MAX;
        }
        const int32_t t = first + static_cast<int32_t>(m - r.mbase);
        const int32_t n_tile =
            tile_splits(r.q_len, r.kv_len, t / a.tile_tokens, a.tile_tokens, a.causal, a.split);
        const int32_t p = a.causal ? r.kv_len - r.q_len + t : r.kv_len - 1;
        const int32_t n_row = min(n_tile, p / a.split + 1);
        for (int ci = 0; ci < n_hc && ok; ++ci) {
          const int h0 = ci * hc, nh = min(hc, a.Hq - h0);
          for (int sp = 0; sp < n_row; ++sp, ++k) {
            const int st = static_cast<int>(k % kMStages);
            if (k >= kMStages && !mbar_wait(empty(st), ((k / kMStages) - 1) & 1, a.status)) {
              ok = false;
              break;
            }
            const int64_t row = (r.rowbase + static_cast<int64_t>(t) * r.nsp + sp) * a.Hq + h0;
            const uint32_t ob = static_cast<uint32_t>(nh * D * 4), lb = static_cast<uint32_t>(nh * 4);
            mbar_expect_tx(full(st), ob + lb);
            bulk_g2s(stage_o(st), a.part_o + row * D, ob, full(st));
            bulk_g2s(stage_l(st), a.part_lse + row, lb, full(st));
          }
        }
      }
      // no copy outlives the CTA: wait for the last use of every stage
      for (uint32_t j = k > kMStages ? k - kMStages : 0; j < k; ++j)
        mbar_wait(full(static_cast<int>(j % kMStages)), (j / kMStages) & 1, a.status);
    }
  } else {
    // ------------------------------------------------------------ folds
    for (int64_t m = m0; m < m1 && ok; ++m) {
      while (m >= next) {
        ++b;
        r = a.reqs[b];
        first = merge_first_token(r.q_len, r.kv_len, a.tile_tokens, a.causal, a.split);
        next = b + 1 < a.batch ? a.reqs[b + 1].mbase : INT64_MAX;
      }
      const int32_t t = first + static_cast<int32_t>(m - r.mbase);
      const int32_t n_tile =
          tile_splits(r.q_len, r.kv_len, t / a.tile_tokens, a.tile_tokens, a.causal, a.split);
      const int32_t p = a.causal ? r.kv_len - r.q_len + t : r.kv_len - 1;
      const int32_t n_row = min(n_tile, p / a.split + 1);
      const int64_t token = static_cast<int64_t>(r.q_start) + t;
      for (int ci = 0; ci < n_hc && ok; ++ci) {
        const int h0 = ci * hc, nh = min(hc, a.Hq - h0);
        float L[kMaxHpw], o[kMaxHpw][V];
#pragma unroll
        for (int i = 0; i < kMaxHpw; ++i) {
          L[i] = -INFINITY;
#pragma unroll
          for (int e = 0; e < V; ++e) o[i][e] = 0.f;
        }
        for (int sp = 0; sp < n_row; ++sp, ++k) {
          const int st = static_cast<int>(k % kMStages);
          if (!mbar_wait(full(st), (k / kMStages) & 1, a.status)) {
            ok = false;
            break;
          }
          const float *so = reinterpret_cast<const float *>(msm + st * kMStageO);
          const float *sl =
              reinterpret_cast<const float *>(msm + kMStages * kMStageO + st * kMStageL);
#pragma unroll
          for (int i = 0; i < kMaxHpw; ++i) {
            const int hh = warp + i * kMergeWarps;
            if (hh < nh) {
              const float ls = sl[hh];
              if (ls != -INFINITY) {
                float v[V];
                load_state_smem<V>(so + hh * D, D, lane, v);
                fold_state<V>(L[i], o[i], ls, v);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty(st));
        }
        if (!ok) break;
#pragma unroll
        for (int i = 0; i < kMaxHpw; ++i) {
          const int hh = warp + i * kMergeWarps;
          if (hh >= nh) break;
          if (L[i] == -INFINITY) {
#pragma unroll
            for (int e = 0; e < V; ++e) o[i][e] = 0.f;
          }
          const int64_t orow = token * a.Hq + h0 + hh;
          store_row<V>(a.out + orow * D, D, a.lse ? a.lse + orow : nullptr, lane, L[i], o[i]);
        }
      }
    }
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
  // two CTAs per SM (all resident at once) share out the rows the planner
  // lists (at most one per q token)
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(a.total_rows, 2LL * sms)));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.Hq % 4 == 0 && merge_chunk_heads(a.Hq, a.D) >= 1) { // streamed through shared memory
    static bool configured[3] = {false, false, false};
    const int vi = a.D <= 128 ? 0 : a.D <= 256 ? 1 : 2;
    const void *fn = vi == 0 ? reinterpret_cast<const void *>(merge_stream_kernel<4>)
                     : vi == 1 ? reinterpret_cast<const void *>(merge_stream_kernel<8>)
                               : reinterpret_cast<const void *>(merge_stream_kernel<16>);
    if (!configured[vi]) {
      const cudaError_t e =
          cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMSmem);
      if (e != cudaSuccess) return e;
      configured[vi] = true;
    }
    cfg.blockDim = dim3(kMThreads);
    cfg.dynamicSmemBytes = kMSmem;
    if (vi == 0) return cudaLaunchKernelEx(&cfg, merge_stream_kernel<4>, a);
    if (vi == 1) return cudaLaunchKernelEx(&cfg, merge_stream_kernel<8>, a);
    return cudaLaunchKernelEx(&cfg, merge_stream_kernel<16>, a);
  }
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

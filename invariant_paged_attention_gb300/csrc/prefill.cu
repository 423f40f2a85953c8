// Paged prefill / chunked-prefill extend on the tensor cores (tcgen05 + TMEM).
//
// One CTA computes one unit: a 128-row q tile of one kv head (128/G tokens x
// the G q heads that share the kv head, "sglang PR #43612", Summary: the
// 128-row q-tile grid) against one split-KV tile of its keys (fixed split,
// "sglang PR #10417 [POC] Support deterministic inference", Modifications).
// Keys are visited in 128-key blocks anchored at absolute key 0:
//   S = Q K^T       tcgen05.mma M=128 N=128 K=D, fp32 accumulator in TMEM
//   online softmax  one thread per row, reading its S row with tcgen05.ld
//   O (+)= P V      tcgen05.mma M=128 N=D K=128, O accumulated in TMEM
// Every per-row reduction boundary is a function of the absolute key
// position and the split size only, so a row's bits never depend on the
// batch, on which tile it shares, or on the grid.  A unit whose q tile has a
// single split writes the final bf16 output; otherwise it writes its fp32
// partial (o_s, lse_s) and the merge kernel folds them in split order.
//
// Shared memory holds Q, one K block, one V block and P, each as 128-byte
// swizzled (SW128) tiles: K-major for Q, K and P, MN-major for V.
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kThreads = 128;
constexpr int kAtom = kTileRows * 128; // one SW128 column of 128 rows x 64 bf16

template <int D>
struct PrefillSmem {
  static constexpr int kTile = kTileRows * D * 2;       // Q, K or V tile bytes
  static constexpr int kP = kTileRows * kKvBlock * 2;   // P tile bytes
  static constexpr int kQ = 0, kK = kTile, kV = 2 * kTile, kPoff = 3 * kTile;
  static constexpr int kBar = kPoff + kP;
  static constexpr int kBytes = kBar + 64;
  static constexpr int kAlloc = kBytes + 1024; // slack for 1024-byte alignment
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const AttnArgs a) {
  using L = PrefillSmem<D>;
  constexpr int QCH = D / 8; // 16-byte chunks per row
  constexpr uint32_t kIdescS = idesc_bf16(128, kKvBlock, false);
  constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
  constexpr uint32_t kTmemCols = 256;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem + L::kQ), sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV), sP = smem_u32(smem + L::kPoff);
  const uint32_t bar = smem_u32(smem + L::kBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kBar + 8);
  __shared__ int s_fail;

  if (blockIdx.x >= a.n_units) return;
  const Unit u = a.units[blockIdx.x];
  if (u.b < 0) return;
  const ReqInfo r = a.reqs[u.b];
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = a.G, T = a.tile_tokens;
  const int32_t t0 = u.tile * T;
  const int32_t last_key = tile_last_key(r.q_len, r.kv_len, u.tile, T, a.causal);
  const int32_t key_begin = u.split * a.split;
  const int32_t key_end = min(key_begin + a.split, last_key + 1);
  const int n_blocks = key_end > key_begin ? (key_end - key_begin + kKvBlock - 1) / kKvBlock : 0;

  // this thread's row of the tile
  const int32_t t_row = t0 + tid / G;
  const int h_row = kvh * G + tid % G;
  const bool row_valid = t_row < r.q_len;
  const int32_t p_row = a.causal ? r.kv_len - r.q_len + t_row : r.kv_len - 1;
  const int32_t vis_last = min(p_row, r.kv_len - 1);

  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    s_fail = 0;
  }
  // Q tile: row rr <-> (token t0 + rr/G, head kvh*G + rr%G); rows past q_len are zeros
  for (int idx = tid; idx < kTileRows * QCH; idx += kThreads) {
    const int rr = idx / QCH, c = idx % QCH;
    const int32_t tl = t0 + rr / G;
    const bool ok = tl < r.q_len;
    const uint16_t *src =
        ok ? a.q + (static_cast<int64_t>(r.q_start + tl) * a.Hq + kvh * G + rr % G) * D + c * 8
           : a.q;
    cp_async16(sQ + (c >> 3) * kAtom + sw128(rr, c & 7), src, ok);
  }
  cp_async_commit();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  float m = -INFINITY, l = 0.f;
  uint32_t phase = 0;
  bool failed = false;
  const int page_mask = (1 << a.page_shift) - 1;

  for (int kb = 0; kb < n_blocks && !failed; ++kb) {
    const int32_t key0 = key_begin + kb * kKvBlock;
    // ---- gather the K and V rows of this block (rows >= kv_len are zeros)
    for (int idx = tid; idx < kKvBlock * QCH; idx += kThreads) {
      const int kr = idx / QCH, c = idx % QCH;
      const int32_t key = key0 + kr;
      bool ok = key < r.kv_len;
      int64_t off = 0;
      if (ok) {
        const int32_t page = __ldg(a.kv_indices + r.page_base + (key >> a.page_shift));
        if (page < 0 || page >= a.num_pages) {
          atomicOr(a.status, kStatusBadPage);
          ok = false;
        } else {
          off = (((static_cast<int64_t>(page) << a.page_shift) + (key & page_mask)) * a.Hkv + kvh) *
                    D + c * 8;
        }
      }
      const uint32_t dst = (c >> 3) * kAtom + sw128(kr, c & 7);
      cp_async16(sK + dst, a.k_cache + off, ok);
      cp_async16(sV + dst, a.v_cache + off, ok);
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async();
    __syncthreads();

    // ---- S = Q K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk >> 2) * kAtom + (kk & 3) * 32;
        mma_bf16_ss(tS, desc_sw128(sQ + koff, 16, 1024), desc_sw128(sK + koff, 16, 1024),
                    kIdescS, kk > 0);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase, a.status)) failed = true;
    phase ^= 1;
    if (__syncthreads_or(failed)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // ---- online softmax of this row
    float x[kKvBlock];
#pragma unroll
    for (int j = 0; j < kKvBlock / 32; ++j) {
      uint32_t v[32];
      tmem_ld32(tS + lane_base + j * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[j * 32 + i] = __uint_as_float(v[i]);
    }
    float bm = -INFINITY;
#pragma unroll
    for (int c = 0; c < kKvBlock; ++c) {
      x[c] = (key0 + c <= vis_last) ? x[c] * a.scale_log2 : -INFINITY;
      bm = fmaxf(bm, x[c]);
    }
    const float m_new = fmaxf(m, bm);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2(m - m_use);
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < kKvBlock; ++c) {
      x[c] = ex2(x[c] - m_use);
      psum += x[c];
    }
    l = fmaf(l, alpha, psum);
    m = m_new;

    // ---- rescale the running O of this row (exact no-op when alpha == 1)
    if (kb > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        uint32_t v[32];
        tmem_ld32(tO + lane_base + j * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(tO + lane_base + j * 32, v);
      }
      tmem_wait_st();
    }

    // ---- P (bf16) to shared memory, K-major SW128
#pragma unroll
    for (int cc = 0; cc < kKvBlock / 8; ++cc) {
      uint4 w;
      w.x = pack_bf16(x[cc * 8 + 0], x[cc * 8 + 1]);
      w.y = pack_bf16(x[cc * 8 + 2], x[cc * 8 + 3]);
      w.z = pack_bf16(x[cc * 8 + 4], x[cc * 8 + 5]);
      w.w = pack_bf16(x[cc * 8 + 6], x[cc * 8 + 7]);
      const uint32_t dst = sP + (cc >> 3) * kAtom + sw128(tid, cc & 7);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w.x), "r"(w.y),
                   "r"(w.z), "r"(w.w)
                   : "memory");
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- O (+)= P V
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kKvBlock / 16; ++kk) {
        const uint32_t poff = (kk >> 2) * kAtom + (kk & 3) * 32;
        mma_bf16_ss(tO, desc_sw128(sP + poff, 16, 1024), desc_sw128(sV + kk * 2048, kAtom, 1024),
                    kIdescPV, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase, a.status)) failed = true;
    phase ^= 1;
    if (__syncthreads_or(failed)) {
      failed = true;
      break;
    }
    tc_fence_after();
  }

  // ---- epilogue: o_s = O / l, lse_s = ln(sum) ; final row or split partial
  const bool has = !failed && n_blocks > 0 && l > 0.f;
  const float lse = has ? __fmul_rn(__fadd_rn(m, lg2(l)), kLn2) : -INFINITY;
  const bool final_row = u.n_splits == 1;
  const int64_t out_row = static_cast<int64_t>(r.q_start + t_row) * a.Hq + h_row;
  const int64_t part_row =
      (r.rowbase + static_cast<int64_t>(t_row) * r.nsp + u.split) * a.Hq + h_row;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    float o[32];
    if (n_blocks > 0 && !failed) {
      uint32_t v[32];
      tmem_ld32(tO + lane_base + j * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = has ? __fdiv_rn(__uint_as_float(v[i]), l) : 0.f;
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0.f;
    }
    if (!row_valid) continue;
    if (final_row) {
      uint4 *dst = reinterpret_cast<uint4 *>(a.out + out_row * D + j * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16(o[q * 8 + 0], o[q * 8 + 1]);
        w.y = pack_bf16(o[q * 8 + 2], o[q * 8 + 3]);
        w.z = pack_bf16(o[q * 8 + 4], o[q * 8 + 5]);
        w.w = pack_bf16(o[q * 8 + 6], o[q * 8 + 7]);
        dst[q] = w;
      }
    } else {
      float4 *dst = reinterpret_cast<float4 *>(a.part_o + part_row * D + j * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
    }
  }
  if (row_valid) {
    if (final_row) {
      if (a.lse) a.lse[out_row] = lse;
    } else {
      a.part_lse[part_row] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_prefill_d(const AttnArgs &a, cudaStream_t s) {
  using L = PrefillSmem<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(static_cast<unsigned>(a.n_units), static_cast<unsigned>(a.Hkv));
  prefill_kernel<D><<<grid, kThreads, L::kAlloc, s>>>(a);
  return cudaGetLastError();
}

} // namespace

cudaError_t launch_prefill(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  return a.D == 128 ? launch_prefill_d<128>(a, s) : launch_prefill_d<64>(a, s);
}

} // namespace bia

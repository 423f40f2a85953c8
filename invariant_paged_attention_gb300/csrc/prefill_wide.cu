// Paged prefill / extend for head_dim 256 on the tensor cores.
//
// The same method as prefill.cu (128-row q tiles of 128/G tokens x G heads,
// "sglang PR #43612", Summary; fixed split-KV tiles merged in order, "sglang
// PR #10417 [POC] Support deterministic inference", Modifications; every
// reduction boundary anchored at absolute key 0), laid out for wide heads:
// the O accumulator of one q tile takes 256 TMEM columns, so a CTA computes
// one q tile, visits keys in 64-key blocks and double-buffers S (2 x 64
// columns) so that S of the next block runs while the softmax of this one
// does:
//   S(j) = Q K(j)^T   tcgen05.mma M=128 N=64 K=256 into S buffer j%2
//   softmax           one thread per row (softmax_rows.cuh), P as bf16 over
//                     the buffer's first 32 columns
//   O += P(j) V(j)    tcgen05.mma M=128 N=256, A = P from TMEM
// MMA order: S(0), S(1), then per block j: P.V(j), S(j+2).  A softmax that
// must rescale O first waits for the previous P.V (an mbarrier committed
// after every P.V).  Warps: 0-3 softmax + epilogue, 4 MMA issuer (owns
// TMEM), 5 TMA producer.  Like prefill.cu, four CTAs form a cluster over
// consecutive q tiles of one request, kv head and split, each gathering a
// quarter of every K/V block's rows (gather4) multicast into all four rings.
#include "bia_internal.h"
#include "ptx.cuh"
#include "softmax_rows.cuh"

namespace bia {

namespace {

constexpr int kD = 256;
constexpr int kKB = 64; // keys per block
constexpr int kCtasW = kPrefillClusterCtas;
constexpr uint16_t kMaskW = (1u << kCtasW) - 1;
constexpr int kMmaW = 4;
constexpr int kProdW = 5;
constexpr int kThreadsW = 192;
constexpr int kAtomQ = kTileRows * 128; // Q atom: 128 rows x 64 bf16
constexpr int kAtomKV = kKB * 128;      // K / V atom: 64 rows x 64 bf16
constexpr float kRescaleW = 8.0f;       // log2 units

struct SmemW {
  static constexpr int kQTile = kTileRows * kD * 2; // 64 KB
  static constexpr int kKVTile = kKB * kD * 2;      // 32 KB
  static constexpr int kQ = 0;
  static constexpr int kKV = kQTile;                // stage s: K at kKV + 2s*kKVTile, V after
  static constexpr int kBar = kKV + 4 * kKVTile;
  static constexpr int kQFull = 0, kKFull = 1, kVFull = 3, kKEmpty = 5, kVEmpty = 7,
                       kSFull = 9, kPFull = 11, kPVDone = 13, kODone = 14, kNumBars = 15;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAlloc = kSlot + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory per block");
};

template <bool MASK>
__global__ void __launch_bounds__(kThreadsW, 1)
    prefill_wide_kernel(const __grid_constant__ AttnArgs a) {
  using L = SmemW;
  constexpr uint32_t kIdescS = idesc_bf16(128, kKB, false);
  constexpr uint32_t kIdescPV = idesc_bf16(128, kD, true);
  constexpr uint32_t kTmemCols = 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  const uint32_t sQ = sbase + L::kQ;
  auto sK = [&](int st) { return sbase + L::kKV + (2 * st) * L::kKVTile; };
  auto sV = [&](int st) { return sbase + L::kKV + (2 * st + 1) * L::kKVTile; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kSlot);

  grid_dep_wait();   // the plan is complete
  grid_dep_launch(); // the next kernel of the call may start launching
  if (blockIdx.x >= a.n_units) return;
  const Unit u = a.units[blockIdx.x];
  if (u.b < 0) return; // plan mismatch: every unit of the launch is disabled
  const uint32_t rank = cluster_ctarank();
  const ReqInfo r = a.reqs[u.b];
  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, T = a.tile_tokens;
  const int32_t key_begin = u.split * a.split;

  struct Tile {
    int32_t tile, n_splits, n_blocks;
    bool has;
  };
  auto tile_of = [&](const Unit &w) {
    Tile x;
    x.tile = w.tile;
    const bool exists = w.ntiles > 0;
    x.n_splits = exists ? tile_splits(r.q_len, r.kv_len, x.tile, T, a.causal, a.split) : 0;
    x.has = exists && w.split < x.n_splits;
    const int32_t last = tile_last_key(r.q_len, r.kv_len, x.tile, T, a.causal);
    const int32_t end = min(key_begin + a.split, last + 1);
    x.n_blocks = (x.has && end > key_begin) ? (end - key_begin + kKB - 1) / kKB : 0;
    return x;
  };
  const Tile me = tile_of(u);
  // blocks the cluster moves: the union of all its CTAs' tiles
  int n_blocks = 0;
  const unsigned first = blockIdx.x - blockIdx.x % kCtasW;
#pragma unroll
  for (int c = 0; c < kCtasW; ++c) n_blocks = max(n_blocks, tile_of(a.units[first + c]).n_blocks);

  if (warp == kMmaW) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(bar(L::kQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), kCtasW); // one release from each CTA's MMAs
      mbar_init(bar(L::kVEmpty + s), kCtasW);
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 4);
    }
    mbar_init(bar(L::kPVDone), 1);
    mbar_init(bar(L::kODone), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kProdW && lane == 0 && me.has) {
    // the q tile (a local load) goes out before the cluster handshake
    mbar_expect_tx(bar(L::kQFull), L::kQTile);
#pragma unroll
    for (int h = 0; h < kD / 64; ++h)
      tma_load_3d(sQ + h * kAtomQ, &a.tm_q, 64 * h, kvh * G, r.q_start + me.tile * T,
                  bar(L::kQFull));
  }
  tc_fence_before();
  cluster_sync(); // every CTA's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S buffers [0,64) and [64,128), O [128,384)
  auto tS = [&](int b) { return tmem + 64u * b; };
  const uint32_t tO = tmem + 128u;

  if (warp == kProdW) {
    // ------------------------------------------------------------ TMA producer
    const int page_mask = (1 << a.page_shift) - 1;
    // this CTA's 16 rows of every 64-key block: lane = 4-row group x 64-col chunk
    constexpr int kGroups = kKB / kCtasW / 4;
    const int rg = lane % kGroups, hh = lane / kGroups;
    const bool issues = hh < kD / 64;
    const int32_t row0 = (kKB / kCtasW) * static_cast<int32_t>(rank) + 4 * rg;
    const uint32_t dst_off = static_cast<uint32_t>(hh * kAtomKV + (row0 / 4) * 512);
    auto fetch = [&](int j, int32_t (&pg)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t key = key_begin + j * kKB + row0 + i;
        pg[i] = (j < n_blocks && key < r.kv_len)
                    ? __ldg(a.kv_indices + r.page_base + (key >> a.page_shift)) : -1;
      }
    };
    int32_t pg[4];
    fetch(0, pg);
    for (int j = 0; j < n_blocks; ++j) {
      const int st = j & 1;
      int32_t rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t key = key_begin + j * kKB + row0 + i;
        rows[i] = a.kv_rows; // outside the map: zeros
        if (key < r.kv_len) {
          if (pg[i] < 0 || pg[i] >= a.num_pages)
            atomicOr(a.status, kStatusBadPage);
          else
            rows[i] = ((pg[i] << a.page_shift) + (key & page_mask)) * a.Hkv + kvh;
        }
      }
      // With pages of 16+ keys this CTA's 16 keys of the block are 16
      // consecutive slots of one page: when all of them are in the sequence
      // and the page is valid, they arrive as one tiled box per 64 columns
      // instead of 16 row gathers (the TMA issue rate of 128-byte row boxes
      // bounds this kernel); otherwise the rows are gathered one by one.
      const int32_t kb = key_begin + j * kKB + (kKB / kCtasW) * static_cast<int32_t>(rank);
      const int32_t pg0 = __shfl_sync(0xffffffffu, pg[0], 0); // lane 0 holds key kb's page
      const bool tiled = a.page_shift >= 4 && kb + kKB / kCtasW <= r.kv_len && pg0 >= 0 &&
                         pg0 < a.num_pages;
      const int32_t slot0 = (pg0 << a.page_shift) + (kb & page_mask);
      const uint32_t tile_off = static_cast<uint32_t>(lane * kAtomKV + (kb - key_begin - j * kKB) * 128);
      fetch(j + 1, pg);
      bool ok = j < 2 || mbar_wait(bar(L::kKEmpty + st), ((j >> 1) - 1) & 1, a.status);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(L::kKFull + st), L::kKVTile);
      __syncwarp();
      if (tiled) {
        if (lane < kD / 64)
          tma_load_3d_mc(sK(st) + tile_off, &a.tm_k3, 64 * lane, kvh, slot0, bar(L::kKFull + st),
                         kMaskW);
      } else if (issues) {
        tma_gather4_mc(sK(st) + dst_off, &a.tm_k, 64 * hh, rows[0], rows[1], rows[2], rows[3],
                       bar(L::kKFull + st), kMaskW);
      }
      ok = j < 2 || mbar_wait(bar(L::kVEmpty + st), ((j >> 1) - 1) & 1, a.status);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(L::kVFull + st), L::kKVTile);
      __syncwarp();
      if (tiled) {
        if (lane < kD / 64)
          tma_load_3d_mc(sV(st) + tile_off, &a.tm_v3, 64 * lane, kvh, slot0, bar(L::kVFull + st),
                         kMaskW);
      } else if (issues) {
        tma_gather4_mc(sV(st) + dst_off, &a.tm_v, 64 * hh, rows[0], rows[1], rows[2], rows[3],
                       bar(L::kVFull + st), kMaskW);
      }
    }
  } else if (warp == kMmaW) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int nb = me.n_blocks;
      bool ok = !me.has || mbar_wait(bar(L::kQFull), 0, a.status);
      auto wait_k = [&](int j) {
        ok = ok && mbar_wait(bar(L::kKFull + (j & 1)), (j >> 1) & 1, a.status);
        if (ok) tc_fence_after();
      };
      auto issue_s = [&](int j) { // S(j) into buffer j%2 from K stage j%2
        if (!ok) return;
        const int st = j & 1;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t c = (kk & 3) * 32;
          mma_bf16_ss(tS(j & 1), desc_sw128(sQ + (kk >> 2) * kAtomQ + c, 16, 1024),
                      desc_sw128(sK(st) + (kk >> 2) * kAtomKV + c, 16, 1024), kIdescS, kk > 0);
        }
        mma_commit(bar(L::kSFull + (j & 1)));
      };
      // K(j) / V(j) are released (to every CTA) iff block j + 2 refills
      // their stage, so every release is awaited and none reaches a CTA that
      // has left
      for (int j = 0; j < 2 && j < n_blocks; ++j) {
        wait_k(j);
        if (j < nb) issue_s(j);
        if (ok && j + 2 < n_blocks) mma_commit_mc(bar(L::kKEmpty + j), kMaskW);
      }
      for (int j = 0; j < n_blocks && ok; ++j) {
        const int st = j & 1;
        ok = mbar_wait(bar(L::kVFull + st), (j >> 1) & 1, a.status);
        if (ok && j < nb) ok = mbar_wait(bar(L::kPFull + (j & 1)), (j >> 1) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        if (j < nb) {
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            mma_bf16_ts(tO, tS(j & 1) + kk * 8, desc_sw128(sV(st) + kk * 2048, kAtomKV, 1024),
                        kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kPVDone));
          if (j == nb - 1) mma_commit(bar(L::kODone));
        }
        if (j + 2 < n_blocks) {
          mma_commit_mc(bar(L::kVEmpty + st), kMaskW);
          wait_k(j + 2);
          if (j + 2 < nb) issue_s(j + 2); // after P.V(j) has read buffer j%2
          if (ok && j + 4 < n_blocks) mma_commit_mc(bar(L::kKEmpty + st), kMaskW);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int gs = __ffs(G) - 1; // G is a power of two
    const int32_t t_row = me.tile * T + (row >> gs);
    const bool row_valid = me.has && t_row < r.q_len;
    const int32_t p_row = a.causal ? r.kv_len - r.q_len + t_row : r.kv_len - 1;
    const int32_t vis_last = min(p_row, r.kv_len - 1);
    constexpr bool use_mask = MASK;
    const int64_t mask_row =
        use_mask && row_valid ? a.mask_indptr[u.b] + static_cast<int64_t>(t_row) * r.kv_len : -1;
    float m = -INFINITY, l = 0.f; // running max (log2 units) and sum
    bool failed = false;
    for (int j = 0; j < me.n_blocks; ++j) {
      const int32_t key0 = key_begin + j * kKB;
      const int32_t n_vis = vis_last - key0 + 1;
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (use_mask) { // the row's 64 bits for this block AND n_vis
        if (mask_row >= 0) {
          const int64_t bit0 = mask_row + key0;
          const int64_t w0 = bit0 >> 5;
          const uint32_t sh = static_cast<uint32_t>(bit0 & 31);
          uint32_t wd[3];
#pragma unroll
          for (int i = 0; i < 3; ++i) wd[i] = w0 + i < a.mask_words ? __ldg(a.mask + w0 + i) : 0u;
#pragma unroll
          for (int w = 0; w < 2; ++w) vis[w] = __funnelshift_r(wd[w], wd[w + 1], sh);
        }
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int n = min(max(n_vis - 32 * w, 0), 32);
          vis[w] &= n >= 32 ? ~0u : ((1u << n) - 1u);
        }
      }
      if (!mbar_wait(bar(L::kSFull + (j & 1)), (j >> 1) & 1, a.status)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const bool full =
          __all_sync(0xffffffffu, use_mask ? (vis[0] & vis[1]) == ~0u : n_vis >= kKB);
      const uint32_t srow = tS(j & 1) + lane_base;
      float bm = full       ? row_block_max<kKB, kFull>(srow, n_vis, vis)
                 : use_mask ? row_block_max<kKB, kBits>(srow, n_vis, vis)
                            : row_block_max<kKB, kFirst>(srow, n_vis, vis);
      bm = bm == -INFINITY ? -INFINITY : bm * a.scale_log2;
      float m_use = m, alpha = 1.f;
      if (bm > m + kRescaleW || (m == -INFINITY && bm != -INFINITY)) {
        m_use = bm;
        alpha = ex2(m - bm); // 0 when m == -inf
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      const float psum = full ? row_block_p<kKB, kFull>(srow, n_vis, vis, a.scale_log2, m_sub)
                         : use_mask
                             ? row_block_p<kKB, kBits>(srow, n_vis, vis, a.scale_log2, m_sub)
                             : row_block_p<kKB, kFirst>(srow, n_vis, vis, a.scale_log2, m_sub);
      l = fmaf(l, alpha, psum);
      m = m_use;
      // rescale the running O row when the max moved, once P.V(j-1) is done
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!mbar_wait(bar(L::kPVDone), (j - 1) & 1, a.status)) failed = true;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(tO + lane_base + c * 16, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st16(tO + lane_base + c * 16, v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kPFull + (j & 1)));
    }
    // epilogue: o_s = O / l row by row into the (now idle) q buffer, then
    // copied out by whole rows so every global store is coalesced: bf16 rows
    // for a tile with one split, else fp32 partial rows in two passes
    if (me.has) {
      const bool have_o = __all_sync(0xffffffffu, !failed && me.n_blocks > 0 &&
                                                      mbar_wait(bar(L::kODone), 0, a.status));
      tc_fence_after();
      const bool nonzero = have_o && l > 0.f;
      const float lse = nonzero ? __fmul_rn(__fadd_rn(m, lg2(l)), kLn2) : -INFINITY;
      const float inv_l = nonzero ? __frcp_rn(l) : 0.f;
      const bool final_row = me.n_splits == 1;
      auto out_row_of = [&](int rr) {
        return static_cast<int64_t>(r.q_start + me.tile * T + (rr >> gs)) * a.Hq + kvh * G +
               (rr & (G - 1));
      };
      auto part_row_of = [&](int rr) {
        return (r.rowbase + static_cast<int64_t>(me.tile * T + (rr >> gs)) * r.nsp + u.split) *
                   a.Hq +
               kvh * G + (rr & (G - 1));
      };
      uint8_t *stage = smem + L::kQ; // 128 rows x 512 bytes
      constexpr int row_bytes = kD * 2;
      constexpr int chunks = row_bytes / 16;
      const int pass_cols = final_row ? kD : kD / 2;
      const int n_pass = kD / pass_cols;
      for (int ps = 0; ps < n_pass; ++ps) {
        uint4 *my = reinterpret_cast<uint4 *>(stage + row * row_bytes);
        const int nchunk = pass_cols / 32;
        const uint32_t obase = tO + lane_base + ps * pass_cols;
        uint32_t v[2][32];
        if (have_o) tmem_ld32(obase, v[0]);
#pragma unroll
        for (int c32 = 0; c32 < kD / 32; ++c32) {
          if (c32 >= nchunk) break;
          if (have_o) {
            tmem_wait_ld();
            if (c32 + 1 < nchunk) tmem_ld32(obase + (c32 + 1) * 32, v[(c32 + 1) & 1]);
          }
          const uint32_t(&x)[32] = v[c32 & 1];
          auto o = [&](int i) { return have_o ? __fmul_rn(__uint_as_float(x[i]), inv_l) : 0.f; };
          if (final_row) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              my[(c32 * 4 + q) ^ (row % chunks)] =
                  make_uint4(pack_bf16(o(q * 8 + 0), o(q * 8 + 1)),
                             pack_bf16(o(q * 8 + 2), o(q * 8 + 3)),
                             pack_bf16(o(q * 8 + 4), o(q * 8 + 5)),
                             pack_bf16(o(q * 8 + 6), o(q * 8 + 7)));
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              my[(c32 * 8 + q) ^ (row % chunks)] =
                  make_uint4(__float_as_uint(o(q * 4)), __float_as_uint(o(q * 4 + 1)),
                             __float_as_uint(o(q * 4 + 2)), __float_as_uint(o(q * 4 + 3)));
          }
        }
        bar_sync_named(1, 128);
        constexpr int rows_per_step = 128 / chunks;
#pragma unroll 4
        for (int r0 = 0; r0 < kTileRows; r0 += rows_per_step) {
          const int rr = r0 + row / chunks, c = row % chunks;
          const int c_lim = final_row ? chunks : (pass_cols * 4) / 16;
          if (me.tile * T + (rr >> gs) < r.q_len && c < c_lim) {
            const uint4 w =
                reinterpret_cast<const uint4 *>(stage + rr * row_bytes)[c ^ (rr % chunks)];
            if (final_row)
              reinterpret_cast<uint4 *>(a.out + out_row_of(rr) * kD)[c] = w;
            else
              reinterpret_cast<uint4 *>(a.part_o + part_row_of(rr) * kD + ps * pass_cols)[c] = w;
          }
        }
        bar_sync_named(1, 128); // the stage is rewritten by the next pass
      }
      if (row_valid) {
        if (final_row) {
          if (a.lse) a.lse[out_row_of(row)] = lse;
        } else {
          a.part_lse[part_row_of(row)] = lse;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaW) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool MASK>
cudaError_t launch_wide(const AttnArgs &a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_wide_kernel<MASK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SmemW::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_units), static_cast<unsigned>(a.Hkv));
  cfg.blockDim = dim3(kThreadsW);
  cfg.dynamicSmemBytes = SmemW::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCtasW;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = chained_launch_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_wide_kernel<MASK>, a);
}

} // namespace

cudaError_t launch_prefill_wide(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  if (a.n_units % kCtasW != 0) return cudaErrorInvalidValue; // the planner groups every unit
  return a.mask ? launch_wide<true>(a, s) : launch_wide<false>(a, s);
}

} // namespace bia

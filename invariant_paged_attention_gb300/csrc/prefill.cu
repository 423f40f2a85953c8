// Paged prefill / chunked-prefill extend on the tensor cores (tcgen05 + TMEM).
//
// A CTA computes one unit: up to two consecutive 128-row q tiles (A, B) of one
// request and one kv head (each tile = 128/G tokens x the G q heads of that kv
// head, "sglang PR #43612", Summary: the 128-row q-tile grid) against one
// split-KV tile of the request's keys ("sglang PR #10417 [POC] Support
// deterministic inference", Modifications: fixed split-KV).  The two tiles
// share every K/V block the CTA gathers.  Keys are visited in 128-key blocks
// anchored at absolute key 0:
//   S = Q K^T      tcgen05.mma M=128 N=128 K=D, operands in shared memory,
//                  fp32 accumulator in TMEM
//   softmax        one thread per row reads its S row (tcgen05.ld), masks by
//                  absolute key position, keeps a running max / sum, writes P
//                  as bf16 back into the S columns of TMEM (tcgen05.st)
//   O (+)= P V     tcgen05.mma with A = P read from TMEM, B = V in shared memory
// Warp roles (10 warps): 0-3 softmax + epilogue of tile A, 4-7 of tile B,
// 8 issues the MMAs (one thread) and owns TMEM, 9 loads the two q tiles (3-D
// TMA boxes of G heads x 128/G tokens) and gathers the paged K/V rows with TMA
// tile::gather4 (each gather fetches four rows of one 64-column half; rows
// past the sequence or on a bad page come from outside the tensor map and
// read as zeros) into a two-stage ring.  mbarriers order
// the roles; the MMA order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) lets one
// tile's softmax overlap the other tile's MMAs.
//
// kPrefillClusterCtas CTAs form a cluster: consecutive q-tile pairs of the
// same request, kv head and split.  They read the same K/V blocks, so each CTA
// gathers its share of every block's rows and multicasts them into all the
// cluster's rings; a stage is refilled once every CTA's MMAs have released it
// (multicast commits, barriers counting one arrival per CTA).  This divides
// the gather requests per SM, which bound the single-CTA version (small
// 128-byte rows, little of the L2 bandwidth used).  All CTAs walk the union
// of their tiles' blocks; a CTA waits for and releases the blocks its own
// tiles do not need without computing on them.
//
// Invariance: every reduction boundary is a function of absolute key
// positions and the split size.  A row's block sequence is the same in any
// tile (blocks past its position are fully masked: exact no-ops), its running
// max is rescaled only from its own history (lazy rescale when the max grows
// by more than 2^8), and each row of the M=128 MMA is computed on its own.
// A tile whose q rows touch a single split writes the final bf16 output;
// otherwise each unit writes an fp32 partial (o_s, lse_s) that the merge
// kernel folds in split order.
#include "bia_internal.h"
#include "ptx.cuh"
#include "softmax_rows.cuh"

namespace bia {

namespace {

constexpr int kCtas = kPrefillClusterCtas;
constexpr uint16_t kClusterMask = (1u << kCtas) - 1;
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp = 9;
constexpr int kThreads = 320;
constexpr int kAtom = kTileRows * 128; // one SW128 column block: 128 rows x 64 bf16
constexpr float kRescaleThreshold = 8.0f; // log2 units

template <int D>
struct Smem {
  static constexpr int kTile = kTileRows * D * 2; // one Q, K or V tile
  static constexpr int kQ0 = 0;
  static constexpr int kKV = 2 * kTile;              // stage s: K at kKV + 2s*kTile, V after it
  static constexpr int kBar = 6 * kTile;
  // barriers (8 bytes each)
  static constexpr int kQFull = 0, kKFull = 1, kVFull = 3, kKEmpty = 5, kVEmpty = 7,
                       kSFull = 9, kPFull = 11, kODone = 13, kNumBars = 15;
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kBytes = kSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

struct TileInfo {
  int32_t tile;       // q tile index in the request
  int32_t n_splits;   // split tiles this q tile touches
  int32_t n_blocks;   // 128-key blocks of this unit's split it needs
  bool has;           // the tile exists and touches this split
};

template <int D, bool MASK>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ AttnArgs a) {
  using L = Smem<D>;
  constexpr uint32_t kIdescS = idesc_bf16(128, kKvBlock, false);
  constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
  constexpr uint32_t kTmemCols = 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sbar = sbase + L::kBar;
  auto bar = [&](int i) { return sbar + 8u * static_cast<uint32_t>(i); };
  auto sQ = [&](int t) { return sbase + L::kQ0 + t * L::kTile; };
  auto sK = [&](int st) { return sbase + L::kKV + (2 * st) * L::kTile; };
  auto sV = [&](int st) { return sbase + L::kKV + (2 * st + 1) * L::kTile; };
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

  auto tile_info = [&](const Unit &w, int t) {
    TileInfo x;
    x.tile = w.tile + t;
    const bool exists = t < w.ntiles;
    x.n_splits = exists ? tile_splits(r.q_len, r.kv_len, x.tile, T, a.causal, a.split) : 0;
    x.has = exists && w.split < x.n_splits;
    const int32_t last = tile_last_key(r.q_len, r.kv_len, x.tile, T, a.causal);
    const int32_t end = min(key_begin + a.split, last + 1);
    x.n_blocks = (x.has && end > key_begin) ? (end - key_begin + kKvBlock - 1) / kKvBlock : 0;
    return x;
  };
  TileInfo ti[2];
  ti[0] = tile_info(u, 0);
  ti[1] = tile_info(u, 1);
  const bool any_tile = ti[0].has || ti[1].has;
  // blocks the cluster moves: the union of all its CTAs' tiles
  int n_blocks = 0;
  const unsigned first = blockIdx.x - blockIdx.x % kCtas;
#pragma unroll
  for (int c = 0; c < kCtas; ++c) {
    const Unit w = a.units[first + c];
    n_blocks = max(n_blocks, max(tile_info(w, 0).n_blocks, tile_info(w, 1).n_blocks));
  }

  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(bar(L::kQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), kCtas); // one release from each CTA's MMAs
      mbar_init(bar(L::kVEmpty + s), kCtas);
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 4);
      mbar_init(bar(L::kODone + s), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kProducerWarp && lane == 0 && any_tile) {
    // the q tiles (a local load) go out before the cluster handshake
    mbar_expect_tx(bar(L::kQFull), static_cast<uint32_t>(ti[0].has + ti[1].has) * L::kTile);
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (ti[t].has)
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sQ(t) + h * kAtom, &a.tm_q, 64 * h, kvh * G, r.q_start + ti[t].tile * T,
                      bar(L::kQFull));
  }
  // This CTA gathers its 1/kCtas share of every block's rows for all CTAs of
  // the cluster (producer lane = 4-row group x 64-column half); the first
  // block's page indices load while the cluster handshake runs.
  constexpr int kGroups = kKvBlock / kCtas / 4; // 4-row groups per CTA
  const int rg = lane % kGroups, hh = lane / kGroups;
  const int32_t row0 = (kKvBlock / kCtas) * static_cast<int32_t>(rank) + 4 * rg;
  auto fetch = [&](int j, int32_t (&pg)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int32_t key = key_begin + j * kKvBlock + row0 + i;
      pg[i] = (j < n_blocks && key < r.kv_len)
                  ? __ldg(a.kv_indices + r.page_base + (key >> a.page_shift)) : -1;
    }
  };
  int32_t pg[4] = {-1, -1, -1, -1};
  if (warp == kProducerWarp) fetch(0, pg);
  tc_fence_before();
  cluster_sync(); // every CTA's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S_A [0,128) S_B [128,256) O_A [256,256+D) O_B [256+D,256+2D)
  auto tS = [&](int t) { return tmem + 128u * t; };
  auto tO = [&](int t) { return tmem + 256u + static_cast<uint32_t>(D) * t; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    const int page_mask = (1 << a.page_shift) - 1;
    const bool issues = hh < D / 64;
    const uint32_t dst_off = static_cast<uint32_t>(hh * kAtom + (row0 / 4) * 512);
    for (int j = 0; j < n_blocks; ++j) {
      const int st = j & 1;
      int32_t rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t key = key_begin + j * kKvBlock + row0 + i;
        rows[i] = a.kv_rows; // outside the map: zeros
        if (key < r.kv_len) {
          if (pg[i] < 0 || pg[i] >= a.num_pages)
            atomicOr(a.status, kStatusBadPage);
          else
            rows[i] = ((pg[i] << a.page_shift) + (key & page_mask)) * a.Hkv + kvh;
        }
      }
      fetch(j + 1, pg); // in flight while this block's copies are issued
      bool ok = j < 2 || mbar_wait(bar(L::kKEmpty + st), ((j >> 1) - 1) & 1, a.status);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(L::kKFull + st), L::kTile); // every share lands here
      __syncwarp();
      if (issues)
        tma_gather4_mc(sK(st) + dst_off, &a.tm_k, 64 * hh, rows[0], rows[1], rows[2], rows[3],
                       bar(L::kKFull + st), kClusterMask);
      ok = j < 2 || mbar_wait(bar(L::kVEmpty + st), ((j >> 1) - 1) & 1, a.status);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(L::kVFull + st), L::kTile);
      __syncwarp();
      if (issues)
        tma_gather4_mc(sV(st) + dst_off, &a.tm_v, 64 * hh, rows[0], rows[1], rows[2], rows[3],
                       bar(L::kVFull + st), kClusterMask);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // shared-memory descriptors of the operand tiles, built once: a K step
      // only advances the start-address field (16-byte units; every address
      // is below 2^18, so the 14-bit field never carries), which keeps the
      // issue of each MMA to a few instructions
      const uint64_t dQ0 = desc_sw128(sQ(0), 16, 1024), dQ1 = desc_sw128(sQ(1), 16, 1024);
      const uint64_t dK0 = desc_sw128(sK(0), 16, 1024), dK1 = desc_sw128(sK(1), 16, 1024);
      const uint64_t dV0 = desc_sw128(sV(0), kAtom, 1024), dV1 = desc_sw128(sV(1), kAtom, 1024);
      bool ok = !any_tile || mbar_wait(bar(L::kQFull), 0, a.status);
      auto wait_k = [&](int j) {
        ok = ok && mbar_wait(bar(L::kKFull + (j & 1)), (j >> 1) & 1, a.status);
        if (ok) tc_fence_after();
      };
      auto issue_s = [&](int t, int j) {
        if (!ok) return;
        const int st = j & 1;
        const uint64_t dq = t ? dQ1 : dQ0, dk = st ? dK1 : dK0;
        const uint32_t ts = tS(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
          mma_bf16_ss(ts, dq + koff, dk + koff, kIdescS, kk > 0);
        }
        mma_commit(bar(L::kSFull + t));
      };
      auto issue_pv = [&](int t, int j, int nb, bool ready) {
        const int st = j & 1;
        ok = ok && (ready || mbar_wait(bar(L::kPFull + t), j & 1, a.status));
        if (!ok) return;
        tc_fence_after();
        const uint64_t dv = st ? dV1 : dV0;
        const uint32_t to = tO(t), ts = tS(t);
#pragma unroll
        for (int kk = 0; kk < kKvBlock / 16; ++kk)
          mma_bf16_ts(to, ts + kk * 8, dv + ((kk * 2048) >> 4), kIdescPV,
                      (j > 0 || kk > 0) ? 1u : 0u);
        if (j == nb - 1) mma_commit(bar(L::kODone + t));
      };
      // A stage is released (to every CTA) only when a later block will
      // refill it: block j is released iff j + 2 < n_blocks, so every
      // release is awaited and none reaches a CTA that has left.
      const int nb0 = ti[0].n_blocks, nb1 = ti[1].n_blocks;
      if (n_blocks > 0) wait_k(0);
      if (nb0 > 0) issue_s(0, 0);
      if (nb1 > 0) issue_s(1, 0);
      if (ok && 2 < n_blocks) mma_commit_mc(bar(L::kKEmpty + 0), kClusterMask);
      for (int j = 0; j < n_blocks && ok; ++j) {
        const int st = j & 1;
        // a barrier's answer takes ~170 cycles to come back even when its
        // phase is complete: ask the block's four barriers at once and use
        // the answers in order (a blocking bounded wait only where one is
        // not complete yet)
        const bool v_rdy = mbar_try(bar(L::kVFull + st), (j >> 1) & 1);
        const bool pa_rdy = j < nb0 && mbar_try(bar(L::kPFull + 0), j & 1);
        const bool k_rdy = j + 1 < n_blocks &&
                           mbar_try(bar(L::kKFull + ((j + 1) & 1)), ((j + 1) >> 1) & 1);
        const bool pb_rdy = j < nb1 && mbar_try(bar(L::kPFull + 1), j & 1);
        ok = v_rdy || mbar_wait(bar(L::kVFull + st), (j >> 1) & 1, a.status);
        if (!ok) break;
        if (j < nb0) issue_pv(0, j, nb0, pa_rdy);
        if (j + 1 < n_blocks) {
          ok = ok && (k_rdy || mbar_wait(bar(L::kKFull + ((j + 1) & 1)), ((j + 1) >> 1) & 1,
                                         a.status));
          if (ok) tc_fence_after();
        }
        if (j + 1 < nb0) issue_s(0, j + 1);
        if (j < nb1) issue_pv(1, j, nb1, pb_rdy);
        if (j + 1 < nb1) issue_s(1, j + 1);
        if (!ok) break;
        if (j + 2 < n_blocks) mma_commit_mc(bar(L::kVEmpty + st), kClusterMask);
        if (j + 3 < n_blocks) mma_commit_mc(bar(L::kKEmpty + ((j + 1) & 1)), kClusterMask);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const TileInfo me = t ? ti[1] : ti[0];
    const int32_t t_row = me.tile * T + row / G;
    const bool row_valid = me.has && t_row < r.q_len;
    const int32_t p_row = a.causal ? r.kv_len - r.q_len + t_row : r.kv_len - 1;
    const int32_t vis_last = min(p_row, r.kv_len - 1);
    // custom mask (MASK): bit (mask_indptr[b] + t_row * kv_len + key) of the
    // mask; rows past the request use none
    constexpr bool use_mask = MASK;
    const int64_t mask_row =
        use_mask && row_valid ? a.mask_indptr[u.b] + static_cast<int64_t>(t_row) * r.kv_len : -1;
    float m = -INFINITY, l = 0.f; // running max (log2 units) and sum
    bool failed = false;
    for (int j = 0; j < me.n_blocks; ++j) {
      const int32_t key0 = key_begin + j * kKvBlock;
      const int32_t n_vis = vis_last - key0 + 1; // columns the causal / length rule allows
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (use_mask) { // the row's 128 bits for this block (at any bit offset) AND n_vis
        if (mask_row >= 0) {
          const int64_t bit0 = mask_row + key0;
          const int64_t w0 = bit0 >> 5;
          const uint32_t sh = static_cast<uint32_t>(bit0 & 31);
          uint32_t wd[5];
#pragma unroll
          for (int i = 0; i < 5; ++i) wd[i] = w0 + i < a.mask_words ? __ldg(a.mask + w0 + i) : 0u;
#pragma unroll
          for (int w = 0; w < 4; ++w) vis[w] = __funnelshift_r(wd[w], wd[w + 1], sh);
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int n = min(max(n_vis - 32 * w, 0), 32);
          vis[w] &= n >= 32 ? ~0u : ((1u << n) - 1u);
        }
      }
      if (!mbar_wait(bar(L::kSFull + t), j & 1, a.status)) {
        failed = true;
        break;
      }
      tc_fence_after();
      // blocks every row of the warp sees in full skip the per-column test
      const bool full = __all_sync(
          0xffffffffu, use_mask ? (vis[0] & vis[1] & vis[2] & vis[3]) == ~0u : n_vis >= kKvBlock);
      const uint32_t srow = tS(t) + lane_base;
      float bm = full       ? row_block_max<kKvBlock, kFull>(srow, n_vis, vis)
                 : use_mask ? row_block_max<kKvBlock, kBits>(srow, n_vis, vis)
                            : row_block_max<kKvBlock, kFirst>(srow, n_vis, vis);
      bm = bm == -INFINITY ? -INFINITY : bm * a.scale_log2;
      float m_use = m, alpha = 1.f;
      if (bm > m + kRescaleThreshold || (m == -INFINITY && bm != -INFINITY)) {
        m_use = bm;
        alpha = ex2(m - bm); // 0 when m == -inf
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      const float psum = full       ? row_block_p<kKvBlock, kFull>(srow, n_vis, vis, a.scale_log2, m_sub)
                         : use_mask ? row_block_p<kKvBlock, kBits>(srow, n_vis, vis, a.scale_log2, m_sub)
                                    : row_block_p<kKvBlock, kFirst>(srow, n_vis, vis, a.scale_log2, m_sub);
      l = fmaf(l, alpha, psum);
      m = m_use;
      // rescale the running O row when the max moved (the previous P.V has
      // completed: S of this block was issued after it)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(tO(t) + lane_base + c * 16, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st16(tO(t) + lane_base + c * 16, v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kPFull + t));
    }
    // epilogue: o_s = O / l.  A tile with one split writes its bf16 rows
    // straight from the thread that owns each row (16-byte stores); fp32
    // partial rows go through the tile's q buffer (free once its last MMA is
    // done; two passes of D/2 columns, rows of D*2 bytes) and are copied out
    // by whole rows so that every global store is coalesced.
    if (me.has) {
      // warp-uniform (tcgen05.ld is warp-collective): a warp with a failed
      // wait writes zeros
      const bool have_o = __all_sync(0xffffffffu, !failed && me.n_blocks > 0 &&
                                                      mbar_wait(bar(L::kODone + t), 0, a.status));
      tc_fence_after();
      const bool nonzero = have_o && l > 0.f;
      const float lse = nonzero ? __fmul_rn(__fadd_rn(m, lg2(l)), kLn2) : -INFINITY;
      const float inv_l = nonzero ? __frcp_rn(l) : 0.f; // o_s = O * (1/l)
      const bool final_row = me.n_splits == 1;           // uniform over the tile
      const int gs = __ffs(G) - 1; // G is a power of two
      auto out_row_of = [&](int rr) {
        return static_cast<int64_t>(r.q_start + me.tile * T + (rr >> gs)) * a.Hq + kvh * G +
               (rr & (G - 1));
      };
      auto part_row_of = [&](int rr) {
        return (r.rowbase + static_cast<int64_t>(me.tile * T + (rr >> gs)) * r.nsp + u.split) *
                   a.Hq +
               kvh * G + (rr & (G - 1));
      };
      uint8_t *stage = smem + L::kQ0 + t * L::kTile; // 128 rows x D*2 bytes
      constexpr int row_bytes = D * 2;
      const int Dr = a.D; // head_dim 96 runs on the 128-wide layout, zero-padded
      constexpr int chunks = row_bytes / 16; // 16-byte chunks per staged row
      const int pass_cols = final_row ? D : D / 2;
      const int n_pass = D / pass_cols;
      for (int ps = 0; ps < n_pass; ++ps) {
        // this thread's row (fp32: chunk c staged at position c ^ (row %
        // chunks)); O read 32 columns at a time with the next load in flight
        uint4 *my = reinterpret_cast<uint4 *>(stage + row * row_bytes);
        const int nchunk = pass_cols / 32;
        const uint32_t obase = tO(t) + lane_base + ps * pass_cols;
        uint32_t v[2][32];
        if (have_o) tmem_ld32(obase, v[0]);
#pragma unroll
        for (int c32 = 0; c32 < D / 32; ++c32) {
          if (c32 >= nchunk) break;
          float o[32];
          if (have_o) {
            tmem_wait_ld();
            if (c32 + 1 < nchunk) tmem_ld32(obase + (c32 + 1) * 32, v[(c32 + 1) & 1]);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __fmul_rn(__uint_as_float(v[c32 & 1][i]), inv_l);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
          if (final_row) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack_bf16(o[q * 8 + 0], o[q * 8 + 1]);
              w.y = pack_bf16(o[q * 8 + 2], o[q * 8 + 3]);
              w.z = pack_bf16(o[q * 8 + 4], o[q * 8 + 5]);
              w.w = pack_bf16(o[q * 8 + 6], o[q * 8 + 7]);
              if (row_valid && c32 * 4 + q < Dr / 8)
                reinterpret_cast<uint4 *>(a.out + out_row_of(row) * Dr)[c32 * 4 + q] = w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              my[(c32 * 8 + q) ^ (row % chunks)] =
                  make_uint4(__float_as_uint(o[q * 4]), __float_as_uint(o[q * 4 + 1]),
                             __float_as_uint(o[q * 4 + 2]), __float_as_uint(o[q * 4 + 3]));
          }
        }
        if (final_row) continue; // one pass, written above
        bar_sync_named(1 + t, 128);
        // copy out: each warp takes 32 rows, chunks lanes per row
        const int tl = (warp & 3) * 32 + lane; // 0..127 within the tile's threads
        constexpr int rows_per_step = 128 / chunks; // rows the 128 threads cover per step
        // 16-byte chunks of real columns (4 fp32 each)
        const int c_lim = min(pass_cols, Dr - ps * pass_cols) / 4;
#pragma unroll 4
        for (int r0 = 0; r0 < kTileRows; r0 += rows_per_step) {
          const int rr = r0 + tl / chunks, c = tl % chunks;
          const int32_t t_rr = me.tile * T + (rr >> gs);
          if (t_rr < r.q_len && c < c_lim)
            reinterpret_cast<uint4 *>(a.part_o + part_row_of(rr) * Dr + ps * pass_cols)[c] =
                reinterpret_cast<const uint4 *>(stage + rr * row_bytes)[c ^ (rr % chunks)];
        }
        bar_sync_named(1 + t, 128); // the stage is rewritten by the next pass
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool MASK>
cudaError_t launch_prefill_d(const AttnArgs &a, cudaStream_t s) {
  using L = Smem<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, MASK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_units), static_cast<unsigned>(a.Hkv));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = chained_launch_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<D, MASK>, a);
}

} // namespace

cudaError_t launch_prefill(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  if (a.n_units % kCtas != 0) return cudaErrorInvalidValue; // the planner pairs every unit
  // head_dim 96 runs on the 128-wide layout: the tensor maps read columns
  // 96..127 as zeros, so S and the first 96 columns of O are unchanged
  if (a.mask)
    return a.D > 64 ? launch_prefill_d<128, true>(a, s) : launch_prefill_d<64, true>(a, s);
  return a.D > 64 ? launch_prefill_d<128, false>(a, s) : launch_prefill_d<64, false>(a, s);
}

} // namespace bia

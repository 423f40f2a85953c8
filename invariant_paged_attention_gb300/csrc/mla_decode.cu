// Batch-invariant multi-head latent attention (MLA) decode over a paged latent
// cache, on the tensor cores (tcgen05 + TMEM).  The pages' serving stack runs
// Kimi-Linear's MLA through a paged MLA wrapper that has no deterministic mode
// ("sglang PR #43612", Summary); this is the same computation with the decode
// path's invariance: fixed split-KV tiles of split_size keys anchored at key 0
// ("sglang PR #10417 [POC] Support deterministic inference", Modifications),
// their partials folded in ascending order by the merge kernel.
//
// Every q head attends to the shared latent rows: s = scale * (<q_nope, ckv>
// + <q_pe, kpe>), out = softmax(s) . ckv (the 512-wide latent row is also the
// value).  The MMAs take the keys as M and the heads as N: a decode query has
// 16 to 128 heads, far fewer than the 128 rows of an M=128 tile, while a
// 128-key block fills M exactly.
//
// One CTA per (query token, split tile, group of HG heads), HG = 32 when the
// head count is a multiple of 32, else 16; keys in 128-key blocks.  A decode call has one query token per request; an extend call
// (bia_mla_prefill_paged) runs each of its causal query tokens the same way,
// against the keys up to its own position, so a token's bits depend only on
// its request's keys and the split size: not on the batch, and not on how
// the extend is chunked.  Per block:
//   S^T = C Q^T     M=128 keys, N=HG heads, K=512+64: A = the latent rows
//                   (K-major, 64-column SW128 pieces), B = the group's
//                   q_nope / q_pe (K-major), fp32 accumulator in TMEM
//   softmax         thread t of a warpgroup = key t of the block (TMEM lane
//                   t) reads its warpgroup's HG/2 heads' scores; per-head block max =
//                   redux over the warp, then over the group's 4 warps through
//                   shared memory (the same value on every thread of the
//                   group); lazy online softmax (the running
//                   max moves only when the block max exceeds it by more than
//                   2^8; O is then rescaled in TMEM); P = 2^(s - m) as bf16
//                   into shared memory, row t = key t (MN-major operand;
//                   128-byte swizzle for 16 heads, 64-byte rows in the
//                   64-byte swizzle for 32)
//   O^T += C^T P^T  four accumulators of M=128 latent columns, N=HG heads,
//                   K=128 keys: A = the same latent pieces read MN-major
//                   (two 64-column pieces side by side), B = P
// Each thread keeps its own keys' partial row sums per head; the epilogue
// sums them (warp butterfly, then the 4 warps in order) and writes
// o = O^T / l and lse (bf16 rows for a request with one split, else fp32
// partials).
//
// Warp roles: 0-7 softmax + epilogue (two warpgroups of HG/2 heads each, a
// thread per key), 8 owns TMEM and issues every MMA from one thread, then the
// copy warps (eight for 16 heads, four for 32, within the registers the
// softmax threads of 32 heads need): one thread loads the group's q (2-D TMA
// boxes), and the copy threads move the paged latent rows with 16-byte cp.async
// straight into the swizzled operand layout (keys past the split or on a bad
// page are zero-filled; each thread's copies of a ring slot end with an
// arrival on the slot's barrier that fires when they land) into a ring of
// 32 KB slots (two ckv pieces: one P.V accumulator's operand) plus one slot
// for the rope piece.  A block's ckv pieces stay until its P.V is done; the
// ring holds the first slot of the next block meanwhile.  (An L2 prefetch of
// the rows two blocks ahead was measured slower, 3.29 against 3.85 TB/s at 16
// heads with the L2 flushed between calls: the prefetched lines were evicted
// before the copies reached them and DRAM read 1.36x the rows.)
//
// Measured (GB300, 16 heads): an M=128 N=16 MMA issues about every 90
// cycles, close to the N=128 rate, so a block's 68 MMAs take ~6k cycles; the
// softmax (~2.5k cycles) and the refill of the slots a P.V frees sit between
// them, and a block takes ~10k cycles (3.88 TB/s of latent rows at 64
// requests).  The MMA count per block does not depend on N, so a group of 32
// heads does the work of two groups of 16 in about the time of one: 64 heads
// 1.15 -> 1.76 TB/s and 128 heads 0.59 -> 0.92 TB/s, the same bits.
//
// Invariance: block boundaries are absolute key positions, every head's
// column of the MMAs is computed on its own, and the lazy-rescale decisions
// and all reductions depend only on the request's own keys in a fixed order,
// so a request's output bits do not depend on the batch.
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kKeys = 128;                   // keys per block: the MMA's M
constexpr int kPiece = kKeys * 128;          // 128 rows x 64 bf16, SW128
constexpr int kCkvPieces = kMlaCkvDim / 64;  // 8
constexpr int kPairs = 5;                    // ring slots of two ckv pieces
constexpr int kMmaWarpT = 8;
constexpr int kProdWarpT = 9;      // warps 9.. copy the latent rows
constexpr float kLazyT = 8.0f; // log2 units

// A CTA takes HG heads (the MMAs' N): 16, or 32 when the head count is a
// multiple of 32 (half the CTAs over the same rows and half the MMAs per
// head).  Two softmax warpgroups take HG/2 heads each.  For 32 heads P is
// kept with 64-byte rows in the 64-byte swizzle, and two copy warps instead of
// four leave the softmax threads the registers of their 16 heads.
template <int HG>
struct MlaCfg {
  static constexpr int kHs = HG / 2;                   // heads per softmax warpgroup
  static constexpr int kProdWarps = HG == 16 ? 8 : 4;  // copy warps
  static constexpr int kThreads = (kProdWarpT + kProdWarps) * 32;
  static constexpr int kPRow = HG == 16 ? 128 : 64;    // bytes per key row of P
  static constexpr int kTmemCols = HG == 16 ? 128 : 256;
};

template <int HG>
struct MlaSmem {
  static constexpr int kQPiece = HG * 128;             // HG heads x 64 columns
  static constexpr int kQ = 0;                         // 9 q pieces (8 ckv + rope)
  static constexpr int kP = kQ + 9 * kQPiece;          // P: 128 keys x kPRow-byte rows
  static constexpr int kRing = kP + kKeys * MlaCfg<HG>::kPRow; // kPairs slots of 2 pieces
  static constexpr int kKpe = kRing + kPairs * 2 * kPiece;
  static constexpr int kBar = kKpe + kPiece;
  static constexpr int bQFull = 0, bPairFull = 1, bPairEmpty = 1 + kPairs,
                       bKpeFull = 1 + 2 * kPairs, bKpeEmpty = bKpeFull + 1, bSFull = bKpeEmpty + 1,
                       bPFull = bSFull + 1, bPVDone = bPFull + 1, kNumBars = bPVDone + 1;
  static constexpr int kRed = kBar + 256;              // float [2][2 groups][4 warps][HG/2 heads]
  static constexpr int kLred = kRed + 2 * 4 * HG * 4;  // float [2 groups][4 warps][HG/2 heads]
  static constexpr int kSlot = kLred + 4 * HG * 4;
  static constexpr int kBytes = kSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kRing % 1024 == 0, "ring slots on the 128-byte swizzle period");
  static_assert(kNumBars * 8 <= 256, "barrier area");
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// Byte offset of 16-byte chunk c of key row t of P: the 128-byte swizzle of
// 128-byte rows (16 heads), or the 64-byte swizzle of 64-byte rows (32 heads:
// chunk bits 4-5 XOR address bits 7-8).
template <int HG>
__device__ __forceinline__ uint32_t p_chunk(uint32_t t, uint32_t c) {
  if constexpr (HG == 16) return sw128(t, c);
  else return t * 64u + ((c ^ ((t >> 1) & 3u)) << 4);
}

// TMEM load of n = HG/2 consecutive 32-bit columns (a warp's 32 lanes).
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 8) tmem_ld8(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 8) tmem_st8(taddr, r);
  else tmem_st16(taddr, r);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <int HG>
__global__ void __launch_bounds__(MlaCfg<HG>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ AttnArgs a) {
  using L = MlaSmem<HG>;
  constexpr int kHg = HG;
  constexpr int kHs = MlaCfg<HG>::kHs;
  constexpr int kProdThreads = MlaCfg<HG>::kProdWarps * 32;
  constexpr int kKeyStep = kProdThreads / 16; // keys between a copy thread's keys
  constexpr uint32_t kIdescS = idesc_bf16_ab(128, kHg, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_ab(128, kHg, true, true);
  constexpr uint32_t kTmemCols = MlaCfg<HG>::kTmemCols;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  auto pair_slot = [&](int s) { return sbase + L::kRing + static_cast<uint32_t>(s) * 2 * kPiece; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kSlot);

  grid_dep_wait();   // the plan is complete
  grid_dep_launch(); // the next kernel of the call may start launching
  // block = unit * head groups + head group: a unit's head groups run side by side
  const int n_hg = (a.Hq + kHg - 1) / kHg;
  const int64_t unit = blockIdx.x / n_hg;
  const int hg = static_cast<int>(blockIdx.x - unit * n_hg);
  if (unit >= a.n_units) return;
  const Unit u = a.units[unit];
  if (u.b < 0) return;
  const ReqInfo r = a.reqs[u.b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // u.tile: the q tile of T = a.tile_tokens consecutive tokens of the
  // request (T = 1: one token; a decode query is token 0).  With T > 1 (an
  // extend with T x Hq = HG) the group's columns are the T tokens' heads,
  // token-major, which are also consecutive rows of q and out.  Causal: token
  // tq sees keys 0 .. kv_len - q_len + tq; the tile walks the keys of its
  // last token, and each column stops at its own token's end.
  const int T = a.tile_tokens;
  const int32_t tq = u.tile * T;                   // the tile's first token
  const int32_t t_last = min(tq + T, r.q_len) - 1; // its last token
  const int32_t kv_end = r.kv_len - r.q_len + tq + 1; // keys of the first token
  const int64_t q_token = static_cast<int64_t>(r.q_start) + tq;
  const int32_t key_begin = u.split * a.split;
  const int32_t key_end = min(key_begin + a.split, kv_end + (t_last - tq));
  const int nb = key_end > key_begin ? (key_end - key_begin + kKeys - 1) / kKeys : 0;
  // columns of this group holding real (token, head) pairs (the rest are padding)
  const int h_real = min(kHg, (t_last + 1 - tq) * a.Hq - hg * kHg);

  if (warp == kMmaWarpT) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < kPairs; ++s) {
      mbar_init(bar(L::bPairFull + s), kProdThreads); // one arrival per copy thread
      mbar_init(bar(L::bPairEmpty + s), 1);
    }
    mbar_init(bar(L::bKpeFull), kProdThreads);
    mbar_init(bar(L::bKpeEmpty), 1);
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bPFull), 8); // one arrival per softmax warp
    mbar_init(bar(L::bPVDone), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S^T [0,HG) (lanes = keys), O^T of latent columns
  // 128*mb .. 128*mb+127 at [2HG+HG*mb, 3HG+HG*mb) (lanes = latent columns)
  const uint32_t tS = tmem;
  auto tO = [&](int mb) {
    return tmem + 2u * kHg + static_cast<uint32_t>(kHg) * static_cast<uint32_t>(mb);
  };

  if (warp >= kProdWarpT) {
    // ------------------------------------------------------------ producers
    const int pt = tid - kProdWarpT * 32; // 0..kProdThreads-1
    // rows past total_q * H read as zeros
    const int32_t q_row = static_cast<int32_t>(q_token * a.Hq + hg * kHg);
    if (pt == 0 && nb > 0) {
      mbar_expect_tx(bar(L::bQFull), 9u * L::kQPiece);
      for (int p = 0; p < kCkvPieces; ++p)
        tma_load_2d(sbase + L::kQ + p * L::kQPiece, &a.tm_q, 64 * p, q_row, bar(L::bQFull));
      tma_load_2d(sbase + L::kQ + kCkvPieces * L::kQPiece, &a.tm_qpe, 0, q_row, bar(L::bQFull));
    }
    // Thread pt copies 16-byte chunk cc of keys kb, kb+kKeyStep, ... of every
    // block (128/kKeyStep keys): of each pair's 256 bytes per key, and
    // (cc < 8) of the rope row; its page indices are fetched a block ahead.
    // Each copy group ends with an arrival that fires when the thread's copies
    // have landed (full barriers count the copy threads).
    const int cc = pt & 15, kb = pt >> 4;
    const int page_mask = (1 << a.page_shift) - 1;
    auto page_at = [&](int j, int k) -> int32_t {
      const int32_t key = key_begin + j * kKeys + k;
      return (j < nb && key < key_end)
                 ? __ldg(a.kv_indices + r.page_base + (key >> a.page_shift)) : -1;
    };
    constexpr int kNk = kKeys / kKeyStep; // keys per copy thread per block
    auto fetch = [&](int j, int32_t (&pg)[kNk]) {
#pragma unroll
      for (int n = 0; n < kNk; ++n) pg[n] = page_at(j, kb + kKeyStep * n);
    };
    // swizzle of chunk cc in key row k of a 128-byte-swizzled piece
    auto swz = [&](int n) {
      return static_cast<uint32_t>(((cc & 7) ^ ((kb + kKeyStep * n) & 7)) << 4);
    };
    int32_t pg_next[kNk];
    fetch(0, pg_next);
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
      int32_t rows[kNk]; // latent row of each of this thread's keys; -1: zeros
#pragma unroll
      for (int n = 0; n < kNk; ++n) {
        const int32_t key = key_begin + j * kKeys + kb + kKeyStep * n;
        rows[n] = -1;
        if (key < key_end) {
          if (pg_next[n] < 0 || pg_next[n] >= a.num_pages)
            atomicOr(a.status, kStatusBadPage);
          else
            rows[n] = (pg_next[n] << a.page_shift) + (key & page_mask);
        }
      }
      fetch(j + 1, pg_next); // in flight while this block's copies are issued
      // pair 0 (its slot frees first), the rope piece (free once the
      // previous block's S is done), then pairs 1-3
      for (int step = 0; step < kCkvPieces / 2 + 1 && ok; ++step) {
        if (step == 1) {
          if (j >= 1) {
            ok = mbar_wait(bar(L::bKpeEmpty), (j - 1) & 1, a.status);
            if (!ok) break;
          }
          if (cc < 8) {
            const uint32_t dbase = sbase + L::kKpe;
            const uint16_t *src0 = a.kpe_cache + cc * 8;
#pragma unroll
            for (int n = 0; n < kNk; ++n)
              cp_async16(dbase + (kb + kKeyStep * n) * 128 + swz(n),
                         src0 + static_cast<int64_t>(max(rows[n], 0)) * kMlaKpeDim, rows[n] >= 0);
          }
          cp_async_arrive(bar(L::bKpeFull));
          continue;
        }
        const int q = step == 0 ? 0 : step - 1;
        const int c = 4 * j + q, s = c % kPairs;
        if (c >= kPairs) {
          ok = mbar_wait(bar(L::bPairEmpty + s), ((c / kPairs) - 1) & 1, a.status);
          if (!ok) break;
        }
        const uint32_t dbase = pair_slot(s) + (cc >> 3) * kPiece;
        const uint16_t *src0 = a.k_cache + 128 * q + cc * 8;
#pragma unroll
        for (int n = 0; n < kNk; ++n)
          cp_async16(dbase + (kb + kKeyStep * n) * 128 + swz(n),
                     src0 + static_cast<int64_t>(max(rows[n], 0)) * kMlaCkvDim, rows[n] >= 0);
        cp_async_arrive(bar(L::bPairFull + s));
      }
    }
    cp_async_wait_all(); // no copy outlives the CTA
  } else if (warp == kMmaWarpT) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = nb == 0 || mbar_wait(bar(L::bQFull), 0, a.status);
      for (int j = 0; j < nb && ok; ++j) {
        // S^T = C Q^T: the eight ckv pieces, then the rope piece
        for (int q = 0; q < kCkvPieces / 2 && ok; ++q) {
          const int c = 4 * j + q, s = c % kPairs;
          ok = mbar_wait(bar(L::bPairFull + s), (c / kPairs) & 1, a.status);
          if (!ok) break;
          fence_proxy_async(); // the rows were written by cp.async (generic proxy)
          tc_fence_after();
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int piece = 2 * q + h2;
              mma_bf16_ss(tS, desc_sw128(pair_slot(s) + h2 * kPiece + kk * 32, 16, 1024),
                          desc_sw128(sbase + L::kQ + piece * L::kQPiece + kk * 32, 16, 1024),
                          kIdescS, (piece | kk) != 0 ? 1u : 0u);
            }
        }
        if (!ok) break;
        ok = mbar_wait(bar(L::bKpeFull), j & 1, a.status);
        if (!ok) break;
        fence_proxy_async();
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tS, desc_sw128(sbase + L::kKpe + kk * 32, 16, 1024),
                      desc_sw128(sbase + L::kQ + kCkvPieces * L::kQPiece + kk * 32, 16, 1024),
                      kIdescS, 1u);
        mma_commit(bar(L::bKpeEmpty));
        mma_commit(bar(L::bSFull));
        // O^T += C^T P^T, one accumulator per pair of ckv pieces
        ok = mbar_wait(bar(L::bPFull), j & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        // each pair is released as soon as its accumulator's MMAs are done
#pragma unroll
        for (int mb = 0; mb < kCkvPieces / 2; ++mb) {
          const int c = 4 * j + mb, s = c % kPairs;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            // P: 16 keys a step; 8-key groups 8*kPRow bytes apart
            const uint64_t dp =
                HG == 16 ? desc_sw128(sbase + L::kP + kk * 2048, kPiece, 1024)
                         : desc_sw64(sbase + L::kP + kk * 1024, 8192, 512);
            mma_bf16_ss(tO(mb), desc_sw128(pair_slot(s) + kk * 2048, kPiece, 1024), dp,
                        kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(L::bPairEmpty + s));
        }
        mma_commit(bar(L::bPVDone));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // two warpgroups, each owning 8 of the 16 heads; warp w%4 of a group
    // covers TMEM lanes (keys) 32(w%4)..+31
    const int gs = warp >> 2, qd = warp & 3;
    const int t = qd * 32 + lane; // key of the block = TMEM lane
    const int h0 = gs * kHs;      // first head of this group
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t gbar = 1 + gs; // the group's named barrier
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    float m[kHs], l[kHs];
#pragma unroll
    for (int h = 0; h < kHs; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    // A wait that runs out ends this thread's loop; it then still arrives at
    // the named barriers of the blocks it did not reach (drain below), so
    // every thread of the group makes the same nb + 1 arrivals and no
    // barrier waits for a thread that has left.
    bool failed = false;
    int drain_from = nb; // first block whose named barrier this thread has not passed
    for (int j = 0; j < nb; ++j) {
      if (!mbar_wait(bar(L::bSFull), j & 1, a.status)) {
        failed = true;
        drain_from = j;
        break;
      }
      tc_fence_after();
      uint32_t v[kHs];
      tmem_ld_n<kHs>(tS + h0 + lane_base, v);
      tmem_wait_ld();
      const int32_t key = key_begin + j * kKeys + t;
      float s[kHs];
#pragma unroll
      for (int h = 0; h < kHs; ++h) {
        // the column's token: tq + (h0 + h) / Hq when T > 1
        const int32_t lim = T > 1 ? min(key_end, kv_end + (h0 + h) / a.Hq) : key_end;
        s[h] = (key < lim && h0 + h < h_real) ? __uint_as_float(v[h]) * a.scale_log2 : -INFINITY;
      }
      // P against the running max, computed while the block max is exchanged
      // (the running max rarely moves: then these are the final values)
      float p[kHs];
#pragma unroll
      for (int h = 0; h < kHs; ++h) {
        const float ms = m[h] == -INFINITY ? 0.f : m[h];
        p[h] = s[h] == -INFINITY ? 0.f : ex2(s[h] - ms);
      }
      // block max per head: over the warp, then the group's 4 warps (the same
      // value on every thread of the group)
      float *rd = red + ((j & 1) * 2 + gs) * 4 * kHs;
      float mine = -INFINITY;
#pragma unroll
      for (int h = 0; h < kHs; ++h) {
        const float wm = warp_max(s[h]);
        mine = lane == h ? wm : mine;
      }
      if (lane < kHs) rd[qd * kHs + lane] = mine;
      bar_sync_named(gbar, 128);
      // lazy online softmax: the running max of a head moves only when the
      // block max exceeds it by more than 2^8; such a head's P is recomputed
      float bmv[kHs];
#pragma unroll
      for (int h4 = 0; h4 < kHs / 4; ++h4) {
        const float4 w0 = reinterpret_cast<const float4 *>(rd)[h4];
        const float4 w1 = reinterpret_cast<const float4 *>(rd + kHs)[h4];
        const float4 w2 = reinterpret_cast<const float4 *>(rd + 2 * kHs)[h4];
        const float4 w3 = reinterpret_cast<const float4 *>(rd + 3 * kHs)[h4];
        bmv[4 * h4 + 0] = fmaxf(fmaxf(w0.x, w1.x), fmaxf(w2.x, w3.x));
        bmv[4 * h4 + 1] = fmaxf(fmaxf(w0.y, w1.y), fmaxf(w2.y, w3.y));
        bmv[4 * h4 + 2] = fmaxf(fmaxf(w0.z, w1.z), fmaxf(w2.z, w3.z));
        bmv[4 * h4 + 3] = fmaxf(fmaxf(w0.w, w1.w), fmaxf(w2.w, w3.w));
      }
      uint32_t up = 0; // heads whose running max moves (the same on the group)
#pragma unroll
      for (int h = 0; h < kHs; ++h)
        if (bmv[h] > m[h] + kLazyT || (m[h] == -INFINITY && bmv[h] != -INFINITY)) up |= 1u << h;
      float alpha[kHs];
#pragma unroll
      for (int h = 0; h < kHs; ++h) alpha[h] = 1.f;
      const bool resc = up != 0;
      if (resc) {
#pragma unroll
        for (int h = 0; h < kHs; ++h) {
          if ((up >> h) & 1u) {
            alpha[h] = ex2(m[h] - bmv[h]); // 0 when m == -inf
            m[h] = bmv[h];
            p[h] = s[h] == -INFINITY ? 0.f : ex2(s[h] - m[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kHs; ++h) l[h] = fmaf(l[h], alpha[h], p[h]);
      // the previous P.V is done: P's buffer is free and O may be rescaled
      if (j > 0 && !mbar_wait(bar(L::bPVDone), (j - 1) & 1, a.status)) {
        failed = true;
        drain_from = j + 1;
        break;
      }
      tc_fence_after();
      if (j > 0 && resc) { // resc is the same on the group
#pragma unroll
        for (int mb = 0; mb < kCkvPieces / 2; ++mb) {
          uint32_t o[kHs];
          tmem_ld_n<kHs>(tO(mb) + h0 + lane_base, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kHs; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          tmem_st_n<kHs>(tO(mb) + h0 + lane_base, o);
        }
        tmem_wait_st();
      }
      // P row of key t: this group's heads are 16-byte chunks gs*kHs/8 .. of
      // the row (8 heads a chunk)
#pragma unroll
      for (int c = 0; c < kHs / 8; ++c)
        sts128(sbase + L::kP + p_chunk<HG>(t, gs * (kHs / 8) + c),
               make_uint4(pack_bf16(p[8 * c + 0], p[8 * c + 1]), pack_bf16(p[8 * c + 2], p[8 * c + 3]),
                          pack_bf16(p[8 * c + 4], p[8 * c + 5]), pack_bf16(p[8 * c + 6], p[8 * c + 7])));
      fence_proxy_async(); // P is read by the MMA (async proxy)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bPFull));
    }

    for (int j = drain_from; j < nb; ++j) bar_sync_named(gbar, 128);

    // ---- epilogue: l = sum of every thread's partial sums (warp butterfly,
    // then the group's 4 warps in order), o = O^T / l, lse = (m + log2 l) ln 2
    const bool have = __all_sync(0xffffffffu, !failed && nb > 0 &&
                                                  mbar_wait(bar(L::bPVDone), (nb - 1) & 1,
                                                            a.status));
    tc_fence_after();
#pragma unroll
    for (int h = 0; h < kHs; ++h)
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
    float *lr = reinterpret_cast<float *>(smem + L::kLred) + gs * 4 * kHs;
    float lw = 0.f;
#pragma unroll
    for (int h = 0; h < kHs; ++h) lw = lane == h ? l[h] : lw;
    if (lane < kHs) lr[qd * kHs + lane] = lw;
    bar_sync_named(gbar, 128);
    float inv[kHs];
    bool nz[kHs];
    float lse_mine = -INFINITY;
#pragma unroll
    for (int h = 0; h < kHs; ++h) {
      const float ls = __fadd_rn(__fadd_rn(__fadd_rn(lr[h], lr[kHs + h]), lr[2 * kHs + h]),
                                 lr[3 * kHs + h]);
      nz[h] = have && ls > 0.f;
      inv[h] = nz[h] ? __frcp_rn(ls) : 0.f;
      const float lse = nz[h] ? __fmul_rn(__fadd_rn(m[h], lg2(ls)), kLn2) : -INFINITY;
      lse_mine = t == h ? lse : lse_mine;
    }
    // one split for the whole tile: final rows (the merge folds a tile's rows
    // whenever the tile spans several splits)
    const bool single = (kv_end + (t_last - tq) - 1) / a.split == 0;
    const int64_t head0 = q_token * a.Hq + hg * kHg + h0;
    // partial row of column h0 + h: its token's rows of this split
    auto prow = [&](int h) {
      const int c = hg * kHg + h0 + h;
      const int tt = T > 1 ? c / a.Hq : 0;
      return (r.rowbase + static_cast<int64_t>(tq + tt) * r.nsp + u.split) * a.Hq +
             (T > 1 ? c % a.Hq : c);
    };
#pragma unroll
    for (int mb = 0; mb < kCkvPieces / 2; ++mb) {
      uint32_t o[kHs];
      if (have) {
        tmem_ld_n<kHs>(tO(mb) + h0 + lane_base, o);
        tmem_wait_ld();
      }
      const int d = mb * 128 + t; // latent column of this thread
#pragma unroll
      for (int h = 0; h < kHs; ++h) {
        if (h0 + h >= h_real) break;
        const float val = nz[h] ? __fmul_rn(__uint_as_float(o[h]), inv[h]) : 0.f;
        if (single)
          a.out[(head0 + h) * kMlaCkvDim + d] = to_bf16(val);
        else
          a.part_o[prow(h) * kMlaCkvDim + d] = val;
      }
    }
    if (t < kHs && h0 + t < h_real) {
      if (single) {
        if (a.lse) a.lse[head0 + t] = lse_mine;
      } else {
        a.part_lse[prow(t) + 0] = lse_mine;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpT) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int HG>
cudaError_t launch_mla_hg(const AttnArgs &a, cudaStream_t s) {
  using L = MlaSmem<HG>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<HG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t blocks = a.n_units * ((a.Hq + HG - 1) / HG);
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(MlaCfg<HG>::kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<HG>, a);
}

} // namespace

cudaError_t launch_mla_decode(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  return a.tile_tokens > 1 || mla_head_group(a.Hq) == 32 ? launch_mla_hg<32>(a, s)
                                                          : launch_mla_hg<16>(a, s);
}

} // namespace bia

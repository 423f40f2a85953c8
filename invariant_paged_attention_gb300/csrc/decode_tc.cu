// Split-KV paged decode for head_dim 128 on the tensor cores (tcgen05 +
// TMEM): the same units as decode.cu (request, split-KV tile, kv head; fixed
// split tiles anchored at key 0, "sglang PR #10417 [POC] Support
// deterministic inference", Modifications), with the keys as the MMAs' M and
// the G (1, 2, 4 or 8) query heads of the kv head as N (padded to 16):
//   S^T = K Q^T      M=128 keys of a block, N=16, K=128: A = the key rows
//                    (two 64-column SW128 pieces), B = the G heads' q rows
//   softmax          thread t = key t of the block (TMEM lane t) reads its
//                    G scores; per-head block max = redux over the warp, then
//                    over the 4 warps through shared memory; lazy online
//                    softmax (the running max moves only when the block max
//                    exceeds it by more than 2^8; O is then rescaled in
//                    TMEM); P = 2^(s - m) as bf16 rows of shared memory
//   O^T += V^T P^T   M=128 head-dim columns, N=16, K=128 keys: A = the value
//                    rows read MN-major, B = P (64-byte swizzle)
// A decode CTA on the CUDA cores streams a split at a rate its own instruction
// stream bounds; here a 128-key block is 16 MMAs, so one CTA per SM reads the
// cache at several times that rate.
//
// The kernel is persistent: one CTA per SM takes the work items (unit, kv
// head) from a counter (its first item is its own index; one copy thread
// takes the next item while the copies of the current one are issued and
// posts it to every role through a small mailbox in shared memory), so the
// CTAs finish together whatever the mix of item sizes, and the items a
// moment's CTAs work on stay neighbours (the kv heads of the same pages).
// Its roles run ahead across items: the copy warps
// stream the next item's q rows and key/value blocks while the MMAs finish
// the current one, S and P are double-buffered (the next block's S is
// computed while the softmax of this one runs), and O is double-buffered per
// item in TMEM (an item's epilogue overlaps the next item's MMAs).  Every item
// starts from a fresh state and its blocks, reductions and rescale decisions
// depend only on its own keys, so its bits do not depend on the batch, on the
// grid or on which CTA runs it.
//
// Warps: 0-3 softmax + epilogue, 4 owns TMEM and issues the MMAs (one
// thread), 5.. copy: 16-byte cp.async into the swizzled operand layouts, a
// ring of key blocks (a slot frees when its S is done) and one of value
// blocks (free when its P.V is done)
// (keys past the split, masked-off tails and bad pages are zero-filled; each
// copy group ends with an arrival that fires when the thread's copies land).
//
// Also runs the single-token q tiles a prefill call streams (with the
// prefill split size), with or without a custom mask: a masked key is left
// out of the softmax like a key past the end.
#include <algorithm>

#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kKeysT = 128;                 // keys per block: the MMA's M
constexpr int kDT = 128;                    // head_dim
constexpr int kPieceT = kKeysT * 128;       // 128 rows x 64 bf16, SW128
constexpr int kKStagesT = 3;                // key blocks in the key ring
constexpr int kVStagesT = 3;                // value blocks in the value ring
constexpr int kNT = 16;                     // the MMAs' N (heads, padded)
constexpr int kSoftWarpsT = 4;
constexpr int kMmaWarpTc = 4;
constexpr int kProdWarpTc = 5; // the first copy warp

// Copy warps for G heads: as many as the registers of the CTA allow (the copy
// rate grows with the number of threads issuing cp.async).
__host__ __device__ constexpr int tc_copy_warps(int G) { return G <= 4 ? 16 : 8; }
constexpr float kLazyTc = 8.0f; // log2 units

struct DecTcSmem {
  static constexpr int kQBuf = kNT * 128 * 2;          // 16 heads x 128 dims (2 pieces)
  static constexpr int kQ = 0;                         // 2 q buffers
  static constexpr int kPBuf = kKeysT * 64;            // 128 keys x 64-byte rows
  static constexpr int kP = kQ + 2 * kQBuf;            // 2 P buffers
  static constexpr int kStage = 2 * kPieceT;           // a block's key or value rows
  static constexpr int kKRing = kP + 2 * kPBuf;
  static constexpr int kVRing = kKRing + kKStagesT * kStage;
  static constexpr int kBar = kVRing + kVStagesT * kStage;
  // barriers
  static constexpr int bKFull = 0, bKEmpty = bKFull + kKStagesT, bVFull = bKEmpty + kKStagesT,
                       bVEmpty = bVFull + kVStagesT, bQFull = bVEmpty + kVStagesT,
                       bQEmpty = bQFull + 2, bSFull = bQEmpty + 2, bPFull = bSFull + 2,
                       bPVDone = bPFull + 2, bOFree = bPVDone + 2, bItemFull = bOFree + 2,
                       bItemEmpty = bItemFull + 4, kNumBars = bItemEmpty + 4;
  static constexpr int kRed = kBar + 256;              // float [2][4 warps][16 heads]
  static constexpr int kLred = kRed + 2 * 4 * kNT * 4; // float [4 warps][16 heads]
  static constexpr int kSlot = kLred + 4 * kNT * 4;
  static constexpr int kItems = kSlot + 16;            // int64 [4]: the item mailbox
  static constexpr int kBytes = kItems + 4 * 8;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kKRing % 1024 == 0, "rings on the 128-byte swizzle period");
  static_assert(kP % 512 == 0 && kPBuf % 512 == 0, "P on the 64-byte swizzle period");
  static_assert(kNumBars * 8 <= 256, "barrier area");
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

// Byte offset of 16-byte chunk c (8 heads) of key row t of P: 64-byte rows,
// the 64-byte swizzle (chunk bits 4-5 XOR address bits 7-8).
__device__ __forceinline__ uint32_t p_chunk64(uint32_t t, uint32_t c) {
  return t * 64u + ((c ^ ((t >> 1) & 3u)) << 4);
}

__device__ __forceinline__ void sts128_tc(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// TMEM load of the first NL columns (8 or 16) of a warp's 32 lanes.
template <int NL>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[NL]) {
  if constexpr (NL == 8) tmem_ld8(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int NL>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[NL]) {
  if constexpr (NL == 8) tmem_st8(taddr, r);
  else tmem_st16(taddr, r);
}

// The geometry of work item w (unit w / Hkv, kv head w % Hkv) every role
// derives the same way.
struct TcItem {
  bool live;          // false: a disabled unit (nothing computed or written)
  int kvh;
  Unit u;
  ReqInfo r;
  int32_t t;          // the query token's index in its request
  int32_t q_end;      // keys < q_end are visible
  int32_t key_begin, key_end;
  int nb;             // 128-key blocks
};

__device__ __forceinline__ TcItem tc_item(const AttnArgs &a, int64_t w) {
  TcItem it;
  const int64_t unit = w / a.Hkv;
  it.kvh = static_cast<int>(w - unit * a.Hkv);
  it.u = a.units[unit];
  it.live = it.u.b >= 0;
  it.nb = 0;
  if (!it.live) return it;
  it.r = a.reqs[it.u.b];
  it.t = it.u.tile;
  it.q_end = a.causal ? it.r.kv_len - it.r.q_len + it.t + 1 : it.r.kv_len;
  it.key_begin = it.u.split * a.split;
  it.key_end = min(it.key_begin + a.split, it.q_end);
  it.nb = it.key_end > it.key_begin ? (it.key_end - it.key_begin + kKeysT - 1) / kKeysT : 0;
  return it;
}

template <int G, bool MASK>
__global__ void __launch_bounds__((kProdWarpTc + tc_copy_warps(G)) * 32, 1)
    decode_tc_kernel(const __grid_constant__ AttnArgs a) {
  using L = DecTcSmem;
  constexpr int kProdThreadsT = tc_copy_warps(G) * 32;
  constexpr int kReaderWarps = tc_copy_warps(G) + 1 + kSoftWarpsT; // copy, MMA, softmax
  constexpr int kKeyStepT = kProdThreadsT / 16; // keys between a copy thread's keys
  constexpr int kNkT = kKeysT / kKeyStepT;      // keys a copy thread takes per block
  constexpr int NL = G <= 8 ? 8 : 16; // TMEM columns a softmax thread loads
  constexpr uint32_t kIdescS = idesc_bf16_ab(128, kNT, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_ab(128, kNT, true, true);
  constexpr uint32_t kTmemCols = 64;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  auto kstage = [&](int s) { return sbase + L::kKRing + static_cast<uint32_t>(s) * L::kStage; };
  auto vstage = [&](int s) { return sbase + L::kVRing + static_cast<uint32_t>(s) * L::kStage; };
  auto qbuf = [&](int i) { return sbase + L::kQ + static_cast<uint32_t>(i) * L::kQBuf; };
  auto pbuf = [&](int i) { return sbase + L::kP + static_cast<uint32_t>(i) * L::kPBuf; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kSlot);

  grid_dep_wait();   // the plan (and, for streamed tiles, the prefill kernel) is complete
  grid_dep_launch(); // the next kernel of the call may start launching
  const int64_t n_work = a.n_units * a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == kMmaWarpTc) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    for (int s = 0; s < kKStagesT; ++s) {
      mbar_init(bar(L::bKFull + s), kProdThreadsT); // one arrival per copy thread
      mbar_init(bar(L::bKEmpty + s), 1);
    }
    for (int s = 0; s < kVStagesT; ++s) {
      mbar_init(bar(L::bVFull + s), kProdThreadsT);
      mbar_init(bar(L::bVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bQFull + i), kProdThreadsT);
      mbar_init(bar(L::bQEmpty + i), 1);
      mbar_init(bar(L::bSFull + i), 1);
      mbar_init(bar(L::bPFull + i), kSoftWarpsT);
      mbar_init(bar(L::bPVDone + i), 1);
      mbar_init(bar(L::bOFree + i), kSoftWarpsT);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(L::bItemFull + i), 1);
      mbar_init(bar(L::bItemEmpty + i), kReaderWarps); // every warp that reads items
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S^T buffers [0,16) and [16,32) (lanes = keys); O^T buffers
  // [32,48) and [48,64) (lanes = head-dim columns)
  auto tS = [&](uint32_t jg) { return tmem + 16u * (jg & 1u); };
  auto tO = [&](uint32_t ig) { return tmem + 32u + 16u * (ig & 1u); };
  // the k-th item of this CTA, from mailbox slot k % 4 (-1: no more items, or
  // a wait that ran out); read by a whole warp, or by one thread (single)
  volatile int64_t *items = reinterpret_cast<volatile int64_t *>(smem + L::kItems);
  auto read_item = [&](uint32_t k, bool single) -> int64_t {
    const int s = static_cast<int>(k & 3u);
    int64_t w = -1;
    if (mbar_wait(bar(L::bItemFull + s), (k >> 2) & 1u, a.status)) w = items[s];
    if (!single) __syncwarp();
    if (single || lane == 0) mbar_arrive(bar(L::bItemEmpty + s));
    return w;
  };

  if (warp >= kProdWarpTc) {
    // ------------------------------------------------------------ copies
    // Thread pt copies 16-byte chunk cc of keys kb, kb+kKeyStepT, ... of a
    // block, of the key row and of the value row; its page indices are
    // fetched while the previous block's copies are issued.
    const int pt = tid - kProdWarpTc * 32;
    const int cc = pt & 15, kb = pt >> 4;
    const int page_mask = (1 << a.page_shift) - 1;
    const uint32_t piece_off = static_cast<uint32_t>(cc >> 3) * kPieceT;
    uint32_t jg = 0, ig = 0;
    bool ok = true;
    // copy thread 0 fetches the items: the first is the CTA's own index, each
    // next one is taken from the counter when the current item starts and
    // posted once the item's first block of copies is issued, so that the
    // copy warps find it waiting when they reach it (one item ahead)
    const bool fetcher = pt == 0;
    if (fetcher) {
      items[0] = blockIdx.x < n_work ? static_cast<int64_t>(blockIdx.x) : -1;
      mbar_arrive(bar(L::bItemFull + 0));
    }
    int32_t taken = 0;   // the counter's answer for the next item
    bool posted = false; // the next item is posted
    auto post_next = [&](uint32_t k) { // item k + 1
      if (!fetcher || posted) return;
      posted = true;
      int64_t nw = static_cast<int64_t>(gridDim.x) + taken;
      if (nw >= n_work) nw = -1;
      const uint32_t kn = k + 1;
      if (kn >= 4 && !mbar_wait(bar(L::bItemEmpty + (kn & 3u)), ((kn >> 2) - 1) & 1u, a.status))
        nw = -1;
      items[kn & 3u] = nw;
      mbar_arrive(bar(L::bItemFull + (kn & 3u)));
    };
    for (uint32_t k = 0; ok; ++k) {
      const int64_t w = read_item(k, false);
      if (w < 0) break;
      if (fetcher) taken = atomicAdd(a.status + kStatusWorkCounter, 1);
      posted = false;
      const TcItem it = tc_item(a, w);
      if (!it.live) {
        post_next(k);
        continue;
      }
      // q rows of the item's G heads (rows G..15 zero) into q buffer ig % 2
      if (ig >= 2 && !mbar_wait(bar(L::bQEmpty + (ig & 1)), ((ig >> 1) - 1) & 1, a.status)) {
        ok = false;
        break;
      }
      const int64_t q_row = static_cast<int64_t>(it.r.q_start) + it.t;
      for (int idx = pt; idx < kNT * 16; idx += kProdThreadsT) { // 16 rows x 16 chunks
        const int h = idx >> 4, c = idx & 15;
        const bool valid = h < G;
        const uint16_t *src = a.q + ((q_row * a.Hq + it.kvh * G + (valid ? h : 0)) * kDT + c * 8);
        cp_async16(qbuf(ig & 1) + (c >> 3) * (kNT * 128) + h * 128 +
                       ((static_cast<uint32_t>(c & 7) ^ static_cast<uint32_t>(h & 7)) << 4),
                   src, valid);
      }
      cp_async_arrive(bar(L::bQFull + (ig & 1)));
      ++ig;
      const int64_t mask_row =
          MASK ? a.mask_indptr[it.u.b] + static_cast<int64_t>(it.t) * it.r.kv_len : 0;
      // page of each of this thread's keys of block j (-1: not copied) and
      // which of them are visible; fetched a block ahead
      auto fetch = [&](int j, int32_t (&pg)[kNkT], uint32_t &vis) {
        vis = 0;
#pragma unroll
        for (int n = 0; n < kNkT; ++n) {
          const int32_t key = it.key_begin + j * kKeysT + kb + kKeyStepT * n;
          bool valid = j < it.nb && key < it.key_end;
          if constexpr (MASK) {
            if (valid) {
              const int64_t bit = mask_row + key;
              valid = (__ldg(a.mask + (bit >> 5)) >> (bit & 31)) & 1u;
            }
          }
          pg[n] = valid ? __ldg(a.kv_indices + it.r.page_base + (key >> a.page_shift)) : -1;
          vis |= static_cast<uint32_t>(valid) << n;
        }
      };
      int32_t pg_next[kNkT];
      uint32_t vis_next;
      fetch(0, pg_next, vis_next);
      for (int j = 0; j < it.nb; ++j, ++jg) {
        int32_t pg[kNkT];
#pragma unroll
        for (int n = 0; n < kNkT; ++n) pg[n] = pg_next[n];
        const uint32_t vis = vis_next;
        fetch(j + 1, pg_next, vis_next); // in flight while this block's copies are issued
        int64_t row[kNkT];
        uint32_t okeys = 0;
#pragma unroll
        for (int n = 0; n < kNkT; ++n) {
          const int32_t key = it.key_begin + j * kKeysT + kb + kKeyStepT * n;
          bool valid = (vis >> n) & 1u;
          if (valid && (pg[n] < 0 || pg[n] >= a.num_pages)) {
            atomicOr(a.status, kStatusBadPage);
            valid = false;
          }
          row[n] = valid ? ((static_cast<int64_t>(pg[n]) << a.page_shift) + (key & page_mask)) *
                                   a.Hkv + it.kvh
                         : 0;
          okeys |= static_cast<uint32_t>(valid) << n;
        }
        // key rows (their slot frees when the block's S is done), then value
        // rows (free when its P.V is done)
        for (int kv = 0; kv < 2; ++kv) {
          const int ns = kv == 0 ? kKStagesT : kVStagesT;
          const int s = static_cast<int>(jg % ns);
          const int eb = (kv == 0 ? L::bKEmpty : L::bVEmpty) + s;
          if (jg >= static_cast<uint32_t>(ns) &&
              !mbar_wait(bar(eb), ((jg / ns) - 1) & 1, a.status)) {
            ok = false;
            break;
          }
          const uint32_t base = (kv == 0 ? kstage(s) : vstage(s)) + piece_off;
          const uint16_t *src = (kv == 0 ? a.k_cache : a.v_cache) + cc * 8;
#pragma unroll
          for (int n = 0; n < kNkT; ++n) {
            const int k = kb + kKeyStepT * n;
            cp_async16(base + static_cast<uint32_t>(k) * 128 +
                           ((static_cast<uint32_t>(cc & 7) ^ static_cast<uint32_t>(k & 7)) << 4),
                       src + row[n] * kDT, (okeys >> n) & 1u);
          }
          cp_async_arrive(bar((kv == 0 ? L::bKFull : L::bVFull) + s));
        }
        if (!ok) break;
        post_next(k); // after the first block
      }
      post_next(k);
    }
    cp_async_wait_all(); // no copy outlives the CTA
  } else if (warp == kMmaWarpTc) {
    // ------------------------------------------------------------ MMA issuer
    // Per item: S(0), S(1), then per block j: P.V(j), S(j+2).
    if (lane == 0) {
      uint32_t jg = 0, ig = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t j_glob, uint32_t qb) {
        const int s = static_cast<int>(j_glob % kKStagesT);
        ok = mbar_wait(bar(L::bKFull + s), (j_glob / kKStagesT) & 1, a.status);
        if (!ok) return;
        fence_proxy_async(); // the rows were written by cp.async (generic proxy)
        tc_fence_after();
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tS(j_glob), desc_sw128(kstage(s) + p * kPieceT + kk * 32, 16, 1024),
                        desc_sw128(qb + p * (kNT * 128) + kk * 32, 16, 1024), kIdescS,
                        (p | kk) != 0 ? 1u : 0u);
        mma_commit(bar(L::bKEmpty + s));
        mma_commit(bar(L::bSFull + (j_glob & 1)));
      };
      for (uint32_t k = 0; ok; ++k) {
        const int64_t w = read_item(k, true);
        if (w < 0) break;
        const TcItem it = tc_item(a, w);
        if (!it.live) continue;
        const uint32_t qb = qbuf(ig & 1);
        ok = mbar_wait(bar(L::bQFull + (ig & 1)), (ig >> 1) & 1, a.status);
        if (!ok) break;
        fence_proxy_async();
        // the item's O buffer is free once the epilogue of item ig-2 read it
        if (ig >= 2) {
          ok = mbar_wait(bar(L::bOFree + (ig & 1)), ((ig >> 1) - 1) & 1, a.status);
          if (!ok) break;
        }
        const uint32_t j0 = jg;
        for (int j = 0; j < min(2, it.nb) && ok; ++j) issue_s(j0 + j, qb);
        for (int j = 0; j < it.nb && ok; ++j) {
          const uint32_t jj = j0 + j;
          const int s = static_cast<int>(jj % kVStagesT);
          ok = mbar_wait(bar(L::bVFull + s), (jj / kVStagesT) & 1, a.status);
          if (ok) ok = mbar_wait(bar(L::bPFull + (jj & 1)), (jj >> 1) & 1, a.status);
          if (!ok) break;
          fence_proxy_async();
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKeysT / 16; ++kk)
            mma_bf16_ss(tO(ig), desc_sw128(vstage(s) + kk * 2048, kPieceT, 1024),
                        desc_sw64(pbuf(jj & 1) + kk * 1024, 8192, 512), kIdescPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::bVEmpty + s));
          mma_commit(bar(L::bPVDone + (jj & 1)));
          if (j + 2 < it.nb) issue_s(jj + 2, qb);
        }
        if (!ok) break;
        // the q buffer is free once the item's S MMAs are done (committed
        // after its last P.V, which follows them)
        mma_commit(bar(L::bQEmpty + (ig & 1)));
        jg += it.nb;
        ++ig;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // A wait that runs out marks this thread failed; the named barriers of
    // the loop reduce the marks (bar.red.or), so the four warps leave the
    // loop at the same barrier and every barrier sees all 128 threads.
    const int qd = warp; // TMEM lanes (keys) 32qd..32qd+31
    const int t = qd * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    float *lr = reinterpret_cast<float *>(smem + L::kLred);
    uint32_t jg = 0, ig = 0;
    bool failed = false; // the same on every softmax thread
    for (uint32_t k = 0; !failed; ++k) {
      const int64_t w = read_item(k, false);
      // the four warps share named barriers: they stop together
      if (bar_any_named(1, 128, w < 0)) break;
      const TcItem it = tc_item(a, w);
      if (!it.live) continue;
      float m[G], l[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      const int64_t mask_row =
          MASK ? a.mask_indptr[it.u.b] + static_cast<int64_t>(it.t) * it.r.kv_len : 0;
      bool bad = false; // this thread's wait ran out
      for (int j = 0; j < it.nb; ++j, ++jg) {
        bad = bad || !mbar_wait(bar(L::bSFull + (jg & 1)), (jg >> 1) & 1, a.status);
        tc_fence_after();
        uint32_t v[NL];
        if (!bad) {
          tmem_ld_cols<NL>(tS(jg) + lane_base, v);
          tmem_wait_ld();
        }
        const int32_t key = it.key_begin + j * kKeysT + t;
        bool valid = !bad && key < it.key_end;
        if constexpr (MASK) {
          if (valid) {
            const int64_t bit = mask_row + key;
            valid = (__ldg(a.mask + (bit >> 5)) >> (bit & 31)) & 1u;
          }
        }
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = valid ? __uint_as_float(v[h]) * a.scale_log2 : -INFINITY;
        // P against the running max while the block max is exchanged
        float p[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float ms = m[h] == -INFINITY ? 0.f : m[h];
          p[h] = s[h] == -INFINITY ? 0.f : ex2(s[h] - ms);
        }
        float *rd = red + (jg & 1) * 4 * kNT;
        float mine = -INFINITY;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float wm = warp_max(s[h]);
          mine = lane == h ? wm : mine;
        }
        if (lane < G) rd[qd * kNT + lane] = mine;
        if (bar_any_named(1, 128, bad)) {
          failed = true;
          break;
        }
        float bmv[G];
#pragma unroll
        for (int h = 0; h < G; ++h)
          bmv[h] = fmaxf(fmaxf(rd[h], rd[kNT + h]), fmaxf(rd[2 * kNT + h], rd[3 * kNT + h]));
        uint32_t up = 0; // heads whose running max moves (the same on every thread)
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (bmv[h] > m[h] + kLazyTc || (m[h] == -INFINITY && bmv[h] != -INFINITY)) up |= 1u << h;
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) alpha[h] = 1.f;
        if (up != 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if ((up >> h) & 1u) {
              alpha[h] = ex2(m[h] - bmv[h]); // 0 when m == -inf
              m[h] = bmv[h];
              p[h] = s[h] == -INFINITY ? 0.f : ex2(s[h] - m[h]);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) l[h] = fmaf(l[h], alpha[h], p[h]);
        // P buffer jg % 2 is free once P.V(jg-2) is done; O may be rescaled
        // once P.V(jg-1) is done
        if (jg >= 2)
          bad = bad || !mbar_wait(bar(L::bPVDone + (jg & 1)), ((jg >> 1) - 1) & 1, a.status);
        if (j > 0 && up != 0) {
          bad = bad ||
                !mbar_wait(bar(L::bPVDone + ((jg - 1) & 1)), ((jg - 1) >> 1) & 1, a.status);
          tc_fence_after();
          if (!bad) {
            uint32_t o[NL];
            tmem_ld_cols<NL>(tO(ig) + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st_cols<NL>(tO(ig) + lane_base, o);
            tmem_wait_st();
          }
        }
        if (bad) continue; // the next barrier takes everyone out
        // P row of key t: 8 heads a 16-byte chunk (heads G..15 zero)
        float pz[kNT];
#pragma unroll
        for (int h = 0; h < kNT; ++h) pz[h] = h < G ? p[h] : 0.f;
#pragma unroll
        for (int c = 0; c < (G <= 8 ? 1 : 2); ++c)
          sts128_tc(pbuf(jg & 1) + p_chunk64(t, c),
                    make_uint4(pack_bf16(pz[8 * c], pz[8 * c + 1]),
                               pack_bf16(pz[8 * c + 2], pz[8 * c + 3]),
                               pack_bf16(pz[8 * c + 4], pz[8 * c + 5]),
                               pack_bf16(pz[8 * c + 6], pz[8 * c + 7])));
        fence_proxy_async(); // P is read by the MMA (async proxy)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bPFull + (jg & 1)));
      }
      if (failed) break;

      // ---- epilogue: l = sum of the threads' partial sums (warp butterfly,
      // then the 4 warps in order); o = O^T / l; lse = (m + log2 l) ln 2
      if (it.nb > 0) {
        const uint32_t jl = jg - 1; // the item's last block
        bad = bad || !mbar_wait(bar(L::bPVDone + (jl & 1)), (jl >> 1) & 1, a.status);
      }
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
      float lw = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) lw = lane == h ? l[h] : lw;
      // (also: the previous item's readers of lr are done)
      if (bar_any_named(1, 128, bad)) {
        failed = true;
        break;
      }
      if (lane < G) lr[qd * kNT + lane] = lw;
      bar_sync_named(1, 128);
      const bool have = it.nb > 0;
      float inv[G];
      bool nz[G];
      float lse_mine = -INFINITY;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float ls = __fadd_rn(__fadd_rn(__fadd_rn(lr[h], lr[kNT + h]), lr[2 * kNT + h]),
                                   lr[3 * kNT + h]);
        nz[h] = have && ls > 0.f;
        inv[h] = nz[h] ? __frcp_rn(ls) : 0.f;
        const float lse = nz[h] ? __fmul_rn(__fadd_rn(m[h], lg2(ls)), kLn2) : -INFINITY;
        lse_mine = t == h ? lse : lse_mine;
      }
      uint32_t o[NL];
#pragma unroll
      for (int h = 0; h < NL; ++h) o[h] = 0u;
      if (have) {
        tmem_ld_cols<NL>(tO(ig) + lane_base, o);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bOFree + (ig & 1))); // O read: the buffer is free
      const bool single = (it.q_end - 1) / a.split == 0; // one split: the final row
      const int64_t q_row = static_cast<int64_t>(it.r.q_start) + it.t;
      const int64_t head0 = q_row * a.Hq + it.kvh * G;
      const int64_t prow0 =
          (it.r.rowbase + static_cast<int64_t>(it.t) * it.r.nsp + it.u.split) * a.Hq + it.kvh * G;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float val = nz[h] ? __fmul_rn(__uint_as_float(o[h]), inv[h]) : 0.f;
        if (single)
          a.out[(head0 + h) * kDT + t] = to_bf16(val);
        else
          a.part_o[(prow0 + h) * kDT + t] = val;
      }
      if (t < G) {
        if (single) {
          if (a.lse) a.lse[head0 + t] = lse_mine;
        } else {
          a.part_lse[prow0 + t] = lse_mine;
        }
      }
      ++ig;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpTc) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G, bool MASK>
cudaError_t launch_tc(const AttnArgs &a, cudaStream_t s) {
  static bool configured = false;
  static int sms = 0;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G, MASK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecTcSmem::kAlloc);
    int dev = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t work = a.n_units * a.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(work, sms)));
  cfg.blockDim = dim3((kProdWarpTc + tc_copy_warps(G)) * 32);
  cfg.dynamicSmemBytes = DecTcSmem::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, MASK>, a);
}

template <int G>
cudaError_t launch_tc_g(const AttnArgs &a, cudaStream_t s) {
  return a.mask ? launch_tc<G, true>(a, s) : launch_tc<G, false>(a, s);
}

} // namespace

bool decode_tc_supported(const AttnArgs &a) {
  return a.D == kDT && (a.G == 1 || a.G == 2 || a.G == 4 || a.G == 8);
}

cudaError_t launch_decode_tc(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  switch (a.G) {
  case 1: return launch_tc_g<1>(a, s);
  case 2: return launch_tc_g<2>(a, s);
  case 4: return launch_tc_g<4>(a, s);
  case 8: return launch_tc_g<8>(a, s);
  default: return cudaErrorInvalidValue;
  }
}

} // namespace bia

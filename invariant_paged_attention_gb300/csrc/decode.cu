// Split-KV paged decode: one CTA per (request, split-KV tile, kv head), the kv
// heads of a (request, split) adjacent in the grid.
//
// The split's keys are cut into chunks of 8 consecutive keys; warp w of the
// CTA owns chunks w, w+8, w+16, ...  Each warp streams its chunks' key and
// value rows from the paged cache into its own ring of shared-memory stages
// with bulk asynchronous copies (one cp.async.bulk per 2*D-byte row, issued by
// 16 lanes, completion counted on the stage's mbarrier), keeping several
// kilobytes per warp in flight without holding registers; the page index of
// the next chunk is fetched one chunk ahead.  D/8 lanes read one row (16
// bytes each).  The G query heads of the kv head stay in registers as fp32
// pairs, pre-scaled by sm_scale * log2 e, and Q.K and P.V run on packed
// fp32x2 FMAs.  Every lane group keeps an online softmax per head over its own
// keys (a fixed function of the key index), rescaled lazily when its max grows
// by more than 2^8; lane groups and then warps are combined in a fixed order,
// so a request's partial and output have the same bits in any batch.  For 4
// heads of 128 columns (16 lanes a key) a chunk's 8 scores are computed first
// and the rescale is decided once per chunk and head, on the chunk max: the
// per-key compare, vote and branch were most of the non-FMA instructions of a
// stream that is issue-bound.  Other shapes do the same per chunk, or per
// sub-chunk when a chunk's scores would not fit in 16 registers per lane.
//
// The same kernel streams the single-token q tiles of a prefill call (a
// one-token extend, or a request's one-token tail tile) with the prefill
// split size: a unit then names its query token's index within the request,
// the keys it sees end at its causal position, and with a custom mask a key
// also needs its mask bit (a masked key is skipped exactly like a key past
// the end, so a mask that hides nothing visible gives the unmasked bits).
//
// The fixed split of 2048 keys per tile and the merge of the tiles' partials
// follow "sglang PR #10417 [POC] Support deterministic inference",
// Modifications (split-KV fixed to 2048 for decode).
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kWarps = 8;
constexpr int kThreadsDec = kWarps * 32;
constexpr int kChunk = 8;              // keys per chunk
constexpr float kLazyThreshold = 8.0f; // log2 units

template <int D>
struct DecSmem {
  static constexpr int kStages = D == 256 ? 2 : (D == 128 ? 3 : 5);
  static constexpr int kRow = D * 2;                  // bytes of one key row
  static constexpr int kStage = 2 * kChunk * kRow;    // K rows then V rows
  static constexpr int kRing = kStages * kStage;      // one warp's ring
  static constexpr int kBar = kWarps * kRing;         // mbarriers [warp][stage]
  static constexpr int kBytes = kBar + kWarps * kStages * 8;
  static constexpr int kAlloc = kBytes + 128;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

// Sums each of the G partial scores over the LPK lanes of a key group and
// leaves all G totals on every lane of the group (identical bits on each).
template <int G, int LPK>
__device__ __forceinline__ void group_reduce(float (&s)[G]) {
  if constexpr (G == 4 && LPK == 16) {
    const int sub = threadIdx.x & 15;
    const bool b3 = (sub >> 3) & 1, b2 = (sub >> 2) & 1;
    // reduce-scatter: the lane keeps heads {2*b3, 2*b3+1}, then head 2*b3+b2
    const float kx = b3 ? s[2] : s[0], ky = b3 ? s[3] : s[1];
    const float sx = b3 ? s[0] : s[2], sy = b3 ? s[1] : s[3];
    const float px = kx + __shfl_xor_sync(0xffffffffu, sx, 8);
    const float py = ky + __shfl_xor_sync(0xffffffffu, sy, 8);
    float c = (b2 ? py : px) + __shfl_xor_sync(0xffffffffu, b2 ? px : py, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    // all-gather: c is head 2*b3 + b2
    const float d = __shfl_xor_sync(0xffffffffu, c, 4); // head 2*b3 + !b2
    const float e = __shfl_xor_sync(0xffffffffu, c, 8); // head 2*!b3 + b2
    const float f = __shfl_xor_sync(0xffffffffu, d, 8); // head 2*!b3 + !b2
    const float lo = b2 ? d : c, hi = b2 ? c : d;        // heads 2*b3, 2*b3+1
    const float lo2 = b2 ? f : e, hi2 = b2 ? e : f;      // heads 2*!b3, 2*!b3+1
    s[0] = b3 ? lo2 : lo;
    s[1] = b3 ? hi2 : hi;
    s[2] = b3 ? lo : lo2;
    s[3] = b3 ? hi : hi2;
  } else {
#pragma unroll
    for (int off = 1; off < LPK; off <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] += __shfl_xor_sync(0xffffffffu, s[g], off);
  }
}

// G == 4, 16 lanes per key: a lane with sub bits b3, b2 holds its four
// partial scores in the order of heads 2b3+b2, 2b3+!b2, 2!b3+b2, 2!b3+!b2
// (own_head_order); sums them over the key's 16 lanes and leaves head
// (sub >> 2)'s total on lanes 4h..4h+3 of the group (identical bits on the
// four).  The per-lane head order makes every exchange select-free.
__device__ __forceinline__ int own_head_order(int j, int sub) {
  return 2 * ((j >> 1) ^ ((sub >> 3) & 1)) + ((j & 1) ^ ((sub >> 2) & 1));
}
__device__ __forceinline__ float reduce_scatter4(const float (&s)[4]) {
  const float px = s[0] + __shfl_xor_sync(0xffffffffu, s[2], 8);
  const float py = s[1] + __shfl_xor_sync(0xffffffffu, s[3], 8);
  float c = px + __shfl_xor_sync(0xffffffffu, py, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

template <int D, int G, bool MASK>
__global__ void __launch_bounds__(kThreadsDec, (G <= 4 ? 2 : 1))
    decode_kernel(const AttnArgs a) {
  using L = DecSmem<D>;
  constexpr int LPK = D / 8;         // lanes per key row
  constexpr int KPW = 32 / LPK;      // key rows per warp step
  constexpr int STEPS = kChunk / KPW; // steps per chunk
  constexpr int NS = L::kStages;
  // G == 4 with 16 lanes per key: the softmax state of head sub/4 lives on
  // lanes 4h..4h+3 of each lane group (m[0], l[0]); otherwise every lane keeps
  // all G states
  constexpr bool kOwnHead = (G == 4 && LPK == 16);
  // steps whose scores share one rescale decision: the whole chunk when its
  // scores fit in 16 registers per lane
  constexpr int SUB = STEPS * G <= 16 ? STEPS : 16 / G;
  static_assert(STEPS % SUB == 0, "sub-chunks");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const uint32_t sbase = smem_u32(smem);

  grid_dep_wait();   // the plan (and, for streamed tiles, the prefill kernel) is complete
  grid_dep_launch(); // the next kernel of the call may start launching
  // block = unit * Hkv + kv head: the kv heads of a unit run side by side
  const int64_t unit = blockIdx.x / a.Hkv;
  const int kvh = static_cast<int>(blockIdx.x - unit * a.Hkv);
  if (unit >= a.n_units) return;
  const Unit u = a.units[unit];
  if (u.b < 0) return;
  const ReqInfo r = a.reqs[u.b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPK, sub = lane % LPK;
  // the query: token t of the request (0 for decode); it sees keys < q_end
  const int32_t t = u.tile;
  const int32_t q_end = a.causal ? r.kv_len - r.q_len + t + 1 : r.kv_len;
  const int64_t q_row = static_cast<int64_t>(r.q_start) + t;
  const int32_t key_begin = u.split * a.split;
  const int32_t key_end = min(key_begin + a.split, q_end);
  // custom mask: bit (t, key) of the request's [q_len, kv_len] mask
  const int64_t mask_row = MASK ? a.mask_indptr[u.b] + static_cast<int64_t>(t) * r.kv_len : 0;
  const int n_chunks = (key_end - key_begin + kChunk - 1) / kChunk;
  const int my_chunks = warp < n_chunks ? (n_chunks - warp + kWarps - 1) / kWarps : 0;

  const uint32_t ring = sbase + warp * L::kRing;
  auto bar = [&](int s) { return sbase + L::kBar + 8u * (warp * NS + s); };
  auto sK = [&](int s) { return ring + s * L::kStage; };
  auto sV = [&](int s) { return ring + s * L::kStage + kChunk * L::kRow; };
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(bar(s), 1);
    fence_mbar_init();
  }
  // head_dim Dr < D (96 on the 128-wide layout): rows are copied Dr*2 bytes
  // into D*2-byte slots whose tails stay zero, and the q lanes past Dr hold 0
  const int Dr = a.D;
  const uint32_t row_copy = static_cast<uint32_t>(Dr) * 2;
  if (Dr < D) {
    for (int b = lane * 16; b < L::kRing; b += 32 * 16)
      asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(ring + b), "r"(0) : "memory");
    fence_proxy_async(); // the zeros precede the ring's bulk copies
  }
  __syncwarp();

  // ---- chunk loads: lanes 0..7 copy key rows, 8..15 the value rows of the
  // same keys; rows past the split or on a bad page are zero-filled instead
  const int kl_ld = lane & 7;
  const int page_mask = (1 << a.page_shift) - 1;
  auto page_of = [&](int i) -> int32_t { // page index of this lane's key in chunk i
    const int32_t key = key_begin + (warp + kWarps * i) * kChunk + kl_ld;
    if (lane >= 16 || i >= my_chunks || key >= key_end) return -1;
    return __ldg(a.kv_indices + r.page_base + (key >> a.page_shift));
  };
  int32_t pg_next = page_of(0);
  auto issue = [&](int i) {
    const int st = i % NS;
    const int32_t pg = pg_next;
    pg_next = page_of(i + 1);
    const int32_t key = key_begin + (warp + kWarps * i) * kChunk + kl_ld;
    bool ok = lane < 16 && key < key_end;
    if (ok && (pg < 0 || pg >= a.num_pages)) {
      atomicOr(a.status, kStatusBadPage);
      ok = false;
    }
    const uint32_t dst = (lane < 8 ? sK(st) : sV(st)) + kl_ld * L::kRow;
    if (lane < 16 && !ok) {
#pragma unroll
      for (int b = 0; b < L::kRow; b += 16)
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst + b), "r"(0) : "memory");
    }
    const int n_ok = __popc(__ballot_sync(0xffffffffu, ok));
    __syncwarp();
    if (lane == 0) mbar_expect_tx(bar(st), static_cast<uint32_t>(n_ok) * row_copy);
    __syncwarp();
    if (ok) {
      const int64_t off =
          (((static_cast<int64_t>(pg) << a.page_shift) + (key & page_mask)) * a.Hkv + kvh) * Dr;
      bulk_g2s(dst, (lane < 8 ? a.k_cache : a.v_cache) + off, row_copy, bar(st));
    }
  };
  for (int i = 0; i < NS && i < my_chunks; ++i) issue(i);

  // ---- queries of the group as fp32 pairs, pre-scaled by sm_scale * log2(e)
  // (G == 4 with 16 lanes a key: slot g holds head own_head_order(g, sub))
  uint64_t q2[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int hq = kOwnHead ? own_head_order(g, sub) : g;
    const uint4 w = sub * 8 < Dr ? *reinterpret_cast<const uint4 *>(
        a.q + (q_row * a.Hq + kvh * G + hq) * Dr + sub * 8)
                                 : make_uint4(0u, 0u, 0u, 0u);
    const uint64_t sc2 = f32x2(a.scale_log2, a.scale_log2);
    q2[g][0] = fmul2(bf16x2_to_f32x2(w.x), sc2);
    q2[g][1] = fmul2(bf16x2_to_f32x2(w.y), sc2);
    q2[g][2] = fmul2(bf16x2_to_f32x2(w.z), sc2);
    q2[g][3] = fmul2(bf16x2_to_f32x2(w.w), sc2);
  }
  float m[G], l[G];
  uint64_t o2[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) o2[g][k] = 0;
  }

  bool failed = false;
  for (int i = 0; i < my_chunks; ++i) {
    const int st = i % NS;
    if (!mbar_wait(bar(st), (i / NS) & 1, a.status)) {
      failed = true;
      break;
    }
    const int32_t key0 = key_begin + (warp + kWarps * i) * kChunk;
    if constexpr (kOwnHead) {
      // the chunk's scores first (this lane: head sub/4 of key s*KPW + grp),
      // then one lazy-rescale decision per chunk and head (the chunk max over
      // both key groups of the warp), then P.V
      float c[STEPS];
      bool vld[STEPS];
#pragma unroll
      for (int s = 0; s < STEPS; ++s) {
        const int kl = s * KPW + grp; // row of the chunk
        const uint4 kw = lds128(sK(st) + kl * L::kRow + sub * 16);
        const uint64_t k2[4] = {bf16x2_to_f32x2(kw.x), bf16x2_to_f32x2(kw.y),
                                bf16x2_to_f32x2(kw.z), bf16x2_to_f32x2(kw.w)};
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          uint64_t acc = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) ffma2(acc, q2[g][k], k2[k]);
          float x, y;
          f32x2_split(acc, x, y);
          sc[g] = x + y;
        }
        c[s] = reduce_scatter4(sc);
        bool valid = key0 + kl < key_end; // past the split's last key: no weight
        if constexpr (MASK) {
          const int64_t bit = mask_row + key0 + kl;
          valid = valid && ((__ldg(a.mask + (bit >> 5)) >> (bit & 31)) & 1u);
        }
        vld[s] = valid;
      }
      float cm = -INFINITY;
#pragma unroll
      for (int s = 0; s < STEPS; ++s) cm = vld[s] ? fmaxf(cm, c[s]) : cm;
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16)); // lanes l and l^16: the same head
      const bool resc = cm > m[0] + kLazyThreshold || (m[0] == -INFINITY && cm != -INFINITY);
      float alpha = 1.f;
      if (resc) {
        alpha = ex2(m[0] - cm); // 0 when m == -inf
        l[0] *= alpha;
        m[0] = cm;
      }
      const int base = lane & ~15;
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float ag = __shfl_sync(0xffffffffu, alpha, base + 4 * g);
          const uint64_t a2 = f32x2(ag, ag);
#pragma unroll
          for (int k = 0; k < 4; ++k) o2[g][k] = fmul2(o2[g][k], a2);
        }
      }
      float p[STEPS];
#pragma unroll
      for (int s = 0; s < STEPS; ++s) {
        p[s] = vld[s] ? ex2(c[s] - m[0]) : 0.f;
        l[0] += p[s];
      }
#pragma unroll
      for (int s = 0; s < STEPS; ++s) {
        const int kl = s * KPW + grp;
        const uint4 vw = lds128(sV(st) + kl * L::kRow + sub * 16);
        const uint64_t v2[4] = {bf16x2_to_f32x2(vw.x), bf16x2_to_f32x2(vw.y),
                                bf16x2_to_f32x2(vw.z), bf16x2_to_f32x2(vw.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = __shfl_sync(0xffffffffu, p[s], base + 4 * g);
          const uint64_t p2 = f32x2(pg, pg);
#pragma unroll
          for (int k = 0; k < 4; ++k) ffma2(o2[g][k], p2, v2[k]);
        }
      }
    } else {
      // as above with every lane holding all G scores: SUB steps' scores, one
      // rescale decision per head for them, then their P.V
#pragma unroll
      for (int s0 = 0; s0 < STEPS; s0 += SUB) {
        float sc[SUB][G];
        bool vld[SUB];
#pragma unroll
        for (int s = 0; s < SUB; ++s) {
          const int kl = (s0 + s) * KPW + grp; // row of the chunk
          const uint4 kw = lds128(sK(st) + kl * L::kRow + sub * 16);
          const uint64_t k2[4] = {bf16x2_to_f32x2(kw.x), bf16x2_to_f32x2(kw.y),
                                  bf16x2_to_f32x2(kw.z), bf16x2_to_f32x2(kw.w)};
#pragma unroll
          for (int g = 0; g < G; ++g) {
            uint64_t acc = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) ffma2(acc, q2[g][k], k2[k]);
            float x, y;
            f32x2_split(acc, x, y);
            sc[s][g] = x + y;
          }
          group_reduce<G, LPK>(sc[s]);
          bool valid = key0 + kl < key_end; // past the split's last key: no weight
          if constexpr (MASK) {
            const int64_t bit = mask_row + key0 + kl;
            valid = valid && ((__ldg(a.mask + (bit >> 5)) >> (bit & 31)) & 1u);
          }
          vld[s] = valid;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float cm = -INFINITY;
#pragma unroll
          for (int s = 0; s < SUB; ++s) cm = vld[s] ? fmaxf(cm, sc[s][g]) : cm;
#pragma unroll
          for (int off = LPK; off < 32; off <<= 1) // the warp's key groups
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
          if (cm > m[g] + kLazyThreshold || (m[g] == -INFINITY && cm != -INFINITY)) {
            const float alpha = ex2(m[g] - cm); // 0 when m == -inf
            l[g] *= alpha;
            const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
            for (int k = 0; k < 4; ++k) o2[g][k] = fmul2(o2[g][k], a2);
            m[g] = cm;
          }
        }
#pragma unroll
        for (int s = 0; s < SUB; ++s) {
          const int kl = (s0 + s) * KPW + grp;
          const uint4 vw = lds128(sV(st) + kl * L::kRow + sub * 16);
          const uint64_t v2[4] = {bf16x2_to_f32x2(vw.x), bf16x2_to_f32x2(vw.y),
                                  bf16x2_to_f32x2(vw.z), bf16x2_to_f32x2(vw.w)};
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float p = vld[s] ? ex2(sc[s][g] - m[g]) : 0.f;
            l[g] += p;
            const uint64_t p2 = f32x2(p, p);
#pragma unroll
            for (int k = 0; k < 4; ++k) ffma2(o2[g][k], p2, v2[k]);
          }
        }
      }
    }
    __syncwarp();
    fence_proxy_async(); // this warp's reads of the stage precede the refill
    if (i + NS < my_chunks) issue(i + NS);
  }

  if constexpr (kOwnHead) {
    const int base = lane & ~15;
    const float m_own = m[0], l_own = l[0];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = __shfl_sync(0xffffffffu, m_own, base + 4 * g);
      l[g] = __shfl_sync(0xffffffffu, l_own, base + 4 * g);
    }
  }
  float o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int k = 0; k < 4; ++k) f32x2_split(o2[g][k], o[g][2 * k], o[g][2 * k + 1]);

  // combine the KPW lane groups of the warp (butterfly: identical on every lane)
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
      const float M = fmaxf(m[g], mo);
      const float w1 = M == -INFINITY ? 0.f : ex2(m[g] - M);
      const float w2 = M == -INFINITY ? 0.f : ex2(mo - M);
      l[g] = l[g] * w1 + lo * w2;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float oo = __shfl_xor_sync(0xffffffffu, o[g][k], off);
        o[g][k] = o[g][k] * w1 + oo * w2;
      }
      m[g] = M;
    }
  }
  // every ring has drained: reuse the shared memory for the warp states
  __syncthreads();
  float *s_m = reinterpret_cast<float *>(smem);
  float *s_l = s_m + kWarps * G;
  float *s_o = s_l + kWarps * G; // [warp][g][D]
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (sub == 0) {
        s_m[warp * G + g] = failed ? -INFINITY : m[g];
        s_l[warp * G + g] = l[g];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) s_o[(warp * G + g) * D + sub * 8 + k] = o[g][k];
    }
  }
  __syncthreads();

  const bool single = (q_end - 1) / a.split == 0; // one split: the final row
  for (int e = threadIdx.x; e < G * D; e += kThreadsDec) {
    const int g = e / D, d = e % D;
    if (d >= Dr) continue;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kWarps; ++k) M = fmaxf(M, s_m[k * G + g]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < kWarps; ++k) {
        const float w = ex2(s_m[k * G + g] - M);
        Ls = fmaf(s_l[k * G + g], w, Ls);
        O = fmaf(s_o[(k * G + g) * D + d], w, O);
      }
    }
    const int h = kvh * G + g;
    const bool empty_row = !(Ls > 0.f);
    const float val = empty_row ? 0.f : __fdiv_rn(O, Ls);
    const float lse = empty_row ? -INFINITY : __fmul_rn(__fadd_rn(M, lg2(Ls)), kLn2);
    const int64_t row = q_row * a.Hq + h;
    if (single) {
      a.out[row * Dr + d] = to_bf16(val);
      if (a.lse && d == 0) a.lse[row] = lse;
    } else {
      const int64_t prow = (r.rowbase + static_cast<int64_t>(t) * r.nsp + u.split) * a.Hq + h;
      a.part_o[prow * Dr + d] = val;
      if (d == 0) a.part_lse[prow] = lse;
    }
  }
}

template <int D, int G, bool MASK>
cudaError_t launch_decode_dgm(const AttnArgs &a, cudaStream_t s) {
  using L = DecSmem<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, MASK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t blocks = a.n_units * a.Hkv;
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreadsDec);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {chained_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, G, MASK>, a);
}

template <int D, int G>
cudaError_t launch_decode_dg(const AttnArgs &a, cudaStream_t s) {
  return a.mask ? launch_decode_dgm<D, G, true>(a, s) : launch_decode_dgm<D, G, false>(a, s);
}

template <int D>
cudaError_t launch_decode_d(const AttnArgs &a, cudaStream_t s) {
  switch (a.G) {
  case 1: return launch_decode_dg<D, 1>(a, s);
  case 2: return launch_decode_dg<D, 2>(a, s);
  case 4: return launch_decode_dg<D, 4>(a, s);
  case 8: return launch_decode_dg<D, 8>(a, s);
  default: return cudaErrorInvalidValue;
  }
}

} // namespace

cudaError_t launch_decode(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  if (decode_tc_supported(a)) return launch_decode_tc(a, s);
  // head_dim 96 runs on the 128-wide layout, zero-padded
  if (a.D == 256) return launch_decode_d<256>(a, s);
  return a.D > 64 ? launch_decode_d<128>(a, s) : launch_decode_d<64>(a, s);
}

} // namespace bia

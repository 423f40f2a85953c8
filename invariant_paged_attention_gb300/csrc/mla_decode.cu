// Batch-invariant multi-head latent attention (MLA) decode over a paged latent
// cache.  The pages' serving stack runs Kimi-Linear's MLA through a paged MLA
// wrapper that has no deterministic mode ("sglang PR #43612", Summary); this
// is the same computation with the decode path's invariance: fixed split-KV
// tiles of split_size keys anchored at key 0 ("sglang PR #10417 [POC] Support
// deterministic inference", Modifications) folded in ascending order.
//
// Every q head attends to the shared latent rows: s = scale * (<q_nope, ckv>
// + <q_pe, kpe>), out = softmax(s) . ckv (the 512-wide latent row is also the
// value).  One CTA per (request, split tile, group of 8 or 16 heads): warps
// 0-7 each own 1 or 2 heads for all the split's keys, warp 8 streams the
// latent rows (ckv 1 KB + kpe 128 B per key) into a shared ring of 8-key
// stages with bulk copies.  A lane holds 16 of the 512 latent columns and 2 of
// the 64 rope columns of its heads' queries (fp32, pre-scaled by
// scale * log2 e) and of their outputs; a key's score is the butterfly sum of
// the 32 lanes' partial dot products (the same bits on every lane; four keys'
// sums reduced together), and each head runs its online softmax over groups
// of four keys in order, rescaled lazily when the group max exceeds the
// running max by more than 2^8.
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kDc = kMlaCkvDim;  // 512
constexpr int kDp = kMlaKpeDim;  // 64
constexpr int kMWarps = 8;       // consumer warps
constexpr int kMThreads = (kMWarps + 1) * 32;
constexpr int kMChunk = 8;       // keys per stage
constexpr int kMGroup = 4;       // keys whose scores are reduced together
constexpr int kMStages = 6;
constexpr float kMLazy = 8.0f;   // log2 units

struct MlaSmem {
  static constexpr int kCkvRow = kDc * 2;                        // 1024 bytes
  static constexpr int kKpeRow = kDp * 2;                        // 128 bytes
  static constexpr int kStage = kMChunk * (kCkvRow + kKpeRow);   // ckv rows then kpe rows
  static constexpr int kBar = kMStages * kStage;
  static constexpr int kFull = 0, kEmpty = kMStages, kNumBars = 2 * kMStages;
  static constexpr int kBytes = kBar + kNumBars * 8;
  static constexpr int kAlloc = kBytes + 128;
};

__device__ __forceinline__ uint4 lds128m(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
__device__ __forceinline__ uint32_t lds32m(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}

// HPW: heads per consumer warp (1 or 2); the CTA takes 8 * HPW heads.
template <int HPW>
__global__ void __launch_bounds__(kMThreads, 1) mla_decode_kernel(const AttnArgs a) {
  using L = MlaSmem;
  constexpr int HG = kMWarps * HPW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::kBar + 8u * static_cast<uint32_t>(i); };
  auto sCkv = [&](int st) { return sbase + st * L::kStage; };
  auto sKpe = [&](int st) { return sbase + st * L::kStage + kMChunk * L::kCkvRow; };

  const int n_groups = a.Hq / HG;
  const int64_t unit = blockIdx.x / n_groups;
  const int hg = static_cast<int>(blockIdx.x - unit * n_groups);
  if (unit >= a.n_units) return;
  const Unit u = a.units[unit];
  if (u.b < 0) return;
  const ReqInfo r = a.reqs[u.b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t key_begin = u.split * a.split;
  const int32_t key_end = min(key_begin + a.split, r.kv_len);
  const int n_chunks = (key_end - key_begin + kMChunk - 1) / kMChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), kMWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kMWarps) {
    // ---------------------------------------------------------- producer
    // lanes 0-7: the ckv rows of the stage's 8 keys, 8-15: their kpe rows;
    // keys past the split or on a bad page are zero-filled instead
    const int kl = lane & 7;
    const int page_mask = (1 << a.page_shift) - 1;
    for (int i = 0; i < n_chunks; ++i) {
      const int st = i % kMStages;
      if (i >= kMStages &&
          !mbar_wait(bar(L::kEmpty + st), (i / kMStages - 1) & 1, a.status))
        break;
      const int32_t key = key_begin + i * kMChunk + kl;
      bool ok = lane < 16 && key < key_end;
      int32_t pg = 0;
      if (ok) {
        pg = __ldg(a.kv_indices + r.page_base + (key >> a.page_shift));
        if (pg < 0 || pg >= a.num_pages) {
          atomicOr(a.status, kStatusBadPage);
          ok = false;
        }
      }
      const bool is_ckv = lane < 8;
      const uint32_t bytes = is_ckv ? L::kCkvRow : L::kKpeRow;
      const uint32_t dst = is_ckv ? sCkv(st) + kl * L::kCkvRow : sKpe(st) + kl * L::kKpeRow;
      if (lane < 16 && !ok) {
        for (uint32_t b = 0; b < bytes; b += 16)
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst + b), "r"(0) : "memory");
      }
      const unsigned okm = __ballot_sync(0xffffffffu, ok);
      const uint32_t tx = __popc(okm & 0xffu) * L::kCkvRow + __popc(okm & 0xff00u) * L::kKpeRow;
      fence_proxy_async(); // zero fills precede the stage's consumers' async view
      __syncwarp();
      if (lane == 0) mbar_expect_tx(bar(L::kFull + st), tx);
      __syncwarp();
      if (ok) {
        const int64_t slot = (static_cast<int64_t>(pg) << a.page_shift) + (key & page_mask);
        if (is_ckv)
          bulk_g2s(dst, a.k_cache + slot * kDc, bytes, bar(L::kFull + st));
        else
          bulk_g2s(dst, a.kpe_cache + slot * kDp, bytes, bar(L::kFull + st));
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int h0 = hg * HG + warp * HPW; // first head of this warp
  const uint64_t sc2 = f32x2(a.scale_log2, a.scale_log2);
  uint64_t qn[HPW][8], qp[HPW];
  float m[HPW], l[HPW];
  uint64_t o2[HPW][8];
#pragma unroll
  for (int k = 0; k < HPW; ++k) {
    const int64_t qrow = static_cast<int64_t>(r.q_start) * a.Hq + h0 + k;
    const uint4 w0 = *reinterpret_cast<const uint4 *>(a.q + qrow * kDc + lane * 16);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(a.q + qrow * kDc + lane * 16 + 8);
    const uint32_t wp = *reinterpret_cast<const uint32_t *>(a.q_pe + qrow * kDp + lane * 2);
    qn[k][0] = fmul2(bf16x2_to_f32x2(w0.x), sc2);
    qn[k][1] = fmul2(bf16x2_to_f32x2(w0.y), sc2);
    qn[k][2] = fmul2(bf16x2_to_f32x2(w0.z), sc2);
    qn[k][3] = fmul2(bf16x2_to_f32x2(w0.w), sc2);
    qn[k][4] = fmul2(bf16x2_to_f32x2(w1.x), sc2);
    qn[k][5] = fmul2(bf16x2_to_f32x2(w1.y), sc2);
    qn[k][6] = fmul2(bf16x2_to_f32x2(w1.z), sc2);
    qn[k][7] = fmul2(bf16x2_to_f32x2(w1.w), sc2);
    qp[k] = fmul2(bf16x2_to_f32x2(wp), sc2);
    m[k] = -INFINITY;
    l[k] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o2[k][i] = 0;
  }

  bool failed = false;
  for (int i = 0; i < n_chunks; ++i) {
    const int st = i % kMStages;
    if (!mbar_wait(bar(L::kFull + st), (i / kMStages) & 1, a.status)) {
      failed = true;
      break;
    }
    const int n_keys = min(kMChunk, key_end - (key_begin + i * kMChunk));
    // keys in groups of kMGroup: the group's scores are reduced together (their
    // shuffle chains overlap) and its max drives one lazy-rescale decision;
    // rows past the split's end are zero-filled and left out
    for (int k0 = 0; k0 < n_keys; k0 += kMGroup) {
      float sc[HPW][kMGroup];
#pragma unroll
      for (int q = 0; q < kMGroup; ++q) {
        const uint32_t row = sCkv(st) + (k0 + q) * L::kCkvRow + lane * 32;
        const uint4 c0 = lds128m(row);
        const uint4 c1 = lds128m(row + 16);
        const uint64_t p2 = bf16x2_to_f32x2(lds32m(sKpe(st) + (k0 + q) * L::kKpeRow + lane * 4));
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int k = 0; k < HPW; ++k) {
          uint64_t acc = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) ffma2(acc, qn[k][e], bf16x2_to_f32x2(cw[e]));
          ffma2(acc, qp[k], p2);
          float x, y;
          f32x2_split(acc, x, y);
          sc[k][q] = x + y;
        }
      }
      // butterfly sums over the warp: the same bits on every lane
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int k = 0; k < HPW; ++k)
#pragma unroll
          for (int q = 0; q < kMGroup; ++q) sc[k][q] += __shfl_xor_sync(0xffffffffu, sc[k][q], off);
      float pw[HPW][kMGroup];
#pragma unroll
      for (int k = 0; k < HPW; ++k) {
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kMGroup; ++q)
          if (k0 + q < n_keys) mx = fmaxf(mx, sc[k][q]);
        if (mx > m[k] + kMLazy || m[k] == -INFINITY) {
          const float alpha = ex2(m[k] - mx); // 0 when m == -inf
          l[k] *= alpha;
          const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 8; ++e) o2[k][e] = fmul2(o2[k][e], a2);
          m[k] = mx;
        }
#pragma unroll
        for (int q = 0; q < kMGroup; ++q) {
          pw[k][q] = k0 + q < n_keys ? ex2(sc[k][q] - m[k]) : 0.f;
          l[k] += pw[k][q];
        }
      }
      // P.V: the group's latent rows read again from shared memory
#pragma unroll
      for (int q = 0; q < kMGroup; ++q) {
        const uint32_t row = sCkv(st) + (k0 + q) * L::kCkvRow + lane * 32;
        const uint4 c0 = lds128m(row);
        const uint4 c1 = lds128m(row + 16);
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int k = 0; k < HPW; ++k) {
          const uint64_t pp = f32x2(pw[k][q], pw[k][q]);
#pragma unroll
          for (int e = 0; e < 8; ++e) ffma2(o2[k][e], pp, bf16x2_to_f32x2(cw[e]));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::kEmpty + st));
  }

  // epilogue: this warp's heads, one split: o = O / l, lse = (m + log2 l) ln 2
  const bool single = (r.kv_len - 1) / a.split == 0;
#pragma unroll
  for (int k = 0; k < HPW; ++k) {
    const int h = h0 + k;
    const bool nonzero = !failed && l[k] > 0.f;
    const float lse = nonzero ? __fmul_rn(__fadd_rn(m[k], lg2(l[k])), kLn2) : -INFINITY;
    float o[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) f32x2_split(o2[k][e], o[2 * e], o[2 * e + 1]);
    const int64_t row = static_cast<int64_t>(r.q_start) * a.Hq + h;
    if (single) {
      uint4 w[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = nonzero ? __fdiv_rn(o[q * 8 + e], l[k]) : 0.f;
        w[q] = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                          pack_bf16(v[6], v[7]));
      }
      uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * kDc + lane * 16);
      dst[0] = w[0];
      dst[1] = w[1];
      if (a.lse && lane == 0) a.lse[row] = lse;
    } else {
      const int64_t prow = (r.rowbase + u.split) * a.Hq + h;
      float4 *dst = reinterpret_cast<float4 *>(a.part_o + prow * kDc + lane * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = nonzero ? __fdiv_rn(o[q * 4 + e], l[k]) : 0.f;
        dst[q] = make_float4(v[0], v[1], v[2], v[3]);
      }
      if (lane == 0) a.part_lse[prow] = lse;
    }
  }
}

template <int HPW>
cudaError_t launch_mla_hpw(const AttnArgs &a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<HPW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         MlaSmem::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t blocks = a.n_units * (a.Hq / (kMWarps * HPW));
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  mla_decode_kernel<HPW><<<static_cast<unsigned>(blocks), kMThreads, MlaSmem::kAlloc, s>>>(a);
  return cudaGetLastError();
}

} // namespace

cudaError_t launch_mla_decode(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  // 16 heads per CTA when they divide evenly, else 8
  return a.Hq % 16 == 0 ? launch_mla_hpw<2>(a, s) : launch_mla_hpw<1>(a, s);
}

} // namespace bia

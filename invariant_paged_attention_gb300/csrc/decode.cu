// Split-KV paged decode: one CTA per (request, split-KV tile, kv head).
//
// The G query heads that share a kv head are kept in registers; the split's
// keys stream through the CTA as 16-byte vector loads, D/8 lanes per key row
// so every 32-byte sector of a row is consumed by one load instruction.  Each
// lane group keeps an online softmax state for the keys it owns (a fixed
// function of the key index), and the 8 warps' states are combined in a
// fixed order at the end.  Nothing depends on the grid, so a request's
// partial (and its output) has the same bits in any batch.
//
// The fixed split of 2048 keys per tile and the merge of the tiles' partials
// follow "sglang PR #10417 [POC] Support deterministic inference",
// Modifications (split-KV fixed to 2048 for decode).
#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

namespace {

constexpr int kDecodeWarps = 8;
constexpr int kDecodeSteps = 4; // key rows per lane group per iteration

__device__ __forceinline__ uint4 ld_stream(const uint16_t *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4 w, float (&f)[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <int D, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32, (G <= 4 ? 2 : 1))
    decode_kernel(const AttnArgs a) {
  constexpr int LPK = D / 8;        // lanes per key row
  constexpr int KPW = 32 / LPK;     // key rows per warp per load step
  constexpr int U = kDecodeSteps;
  constexpr int KEYS_PER_ITER = kDecodeWarps * KPW * U;
  constexpr int NSTATE = kDecodeWarps; // one combined state per warp

  __shared__ float s_m[NSTATE][G];
  __shared__ float s_l[NSTATE][G];
  __shared__ __align__(16) float s_o[NSTATE][G][D];

  if (blockIdx.x >= a.n_units) return;
  const Unit u = a.units[blockIdx.x];
  if (u.b < 0) return;
  const ReqInfo r = a.reqs[u.b];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPK, sub = lane % LPK;
  const int32_t key_begin = u.split * a.split;
  const int32_t key_end = min(key_begin + a.split, r.kv_len);

  // queries of the group, pre-scaled by sm_scale * log2(e)
  float q[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint16_t *src =
        a.q + (static_cast<int64_t>(r.q_start) * a.Hq + kvh * G + g) * D + sub * 8;
    float f[8];
    unpack8(*reinterpret_cast<const uint4 *>(src), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[g][i] = f[i] * a.scale_log2;
  }

  float m[G], l[G], o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[g][i] = 0.f;
  }

  const int page_mask = (1 << a.page_shift) - 1;
  for (int32_t it = key_begin; it < key_end; it += KEYS_PER_ITER) {
    uint4 kw[U], vw[U];
    bool ok[U];
#pragma unroll
    for (int s = 0; s < U; ++s) {
      const int32_t key = it + (warp * U + s) * KPW + grp;
      ok[s] = key < key_end;
      int64_t off = 0;
      if (ok[s]) {
        const int32_t page = __ldg(a.kv_indices + r.page_base + (key >> a.page_shift));
        if (page < 0 || page >= a.num_pages) {
          atomicOr(a.status, kStatusBadPage);
          ok[s] = false;
        } else {
          off = ((static_cast<int64_t>(page) << a.page_shift) + (key & page_mask)) * a.Hkv + kvh;
          off = off * D + sub * 8;
        }
      }
      if (ok[s]) {
        kw[s] = ld_stream(a.k_cache + off);
        vw[s] = ld_stream(a.v_cache + off);
      } else {
        kw[s] = make_uint4(0, 0, 0, 0);
        vw[s] = make_uint4(0, 0, 0, 0);
      }
    }
    // scores
    float sc[U][G];
#pragma unroll
    for (int s = 0; s < U; ++s) {
      float kf[8];
      unpack8(kw[s], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(q[g][i], kf[i], acc);
        sc[s][g] = acc;
      }
    }
#pragma unroll
    for (int off = 1; off < LPK; off <<= 1) {
#pragma unroll
      for (int s = 0; s < U; ++s)
#pragma unroll
        for (int g = 0; g < G; ++g) sc[s][g] += __shfl_xor_sync(0xffffffffu, sc[s][g], off);
    }
    // online softmax over this lane group's U keys
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = m[g];
#pragma unroll
      for (int s = 0; s < U; ++s) {
        if (!ok[s]) sc[s][g] = -INFINITY;
        mx = fmaxf(mx, sc[s][g]);
      }
      if (mx == -INFINITY) continue;
      const float alpha = ex2(m[g] - mx);
      float psum = 0.f;
      float p[U];
#pragma unroll
      for (int s = 0; s < U; ++s) {
        p[s] = ex2(sc[s][g] - mx);
        psum += p[s];
      }
      l[g] = fmaf(l[g], alpha, psum);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[g][i] *= alpha;
      m[g] = mx;
#pragma unroll
      for (int s = 0; s < U; ++s) {
        float vf[8];
        unpack8(vw[s], vf);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[g][i] = fmaf(p[s], vf[i], o[g][i]);
      }
    }
  }

  // combine the KPW lane groups of the warp (butterfly; lane group 0 keeps
  // the result that is published)
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
      const float M = fmaxf(m[g], mo);
      const float w1 = M == -INFINITY ? 0.f : ex2(m[g] - M);
      const float w2 = M == -INFINITY ? 0.f : ex2(mo - M);
      l[g] = fmaf(l[g], w1, lo * w2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float oo = __shfl_xor_sync(0xffffffffu, o[g][i], off);
        o[g][i] = fmaf(o[g][i], w1, oo * w2);
      }
      m[g] = M;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (sub == 0) {
        s_m[warp][g] = m[g];
        s_l[warp][g] = l[g];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) s_o[warp][g][sub * 8 + i] = o[g][i];
    }
  }
  __syncthreads();

  // combine the NSTATE states in index order; thread handles (g, d) pairs
  for (int e = threadIdx.x; e < G * D; e += kDecodeWarps * 32) {
    const int g = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < NSTATE; ++k) M = fmaxf(M, s_m[k][g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < NSTATE; ++k) {
        const float w = ex2(s_m[k][g] - M);
        L = fmaf(s_l[k][g], w, L);
        O = fmaf(s_o[k][g][d], w, O);
      }
    }
    const int h = kvh * G + g;
    const bool empty = !(L > 0.f);
    const float val = empty ? 0.f : __fdiv_rn(O, L);
    const float lse = empty ? -INFINITY : __fmul_rn(__fadd_rn(M, lg2(L)), kLn2);
    const int64_t row = static_cast<int64_t>(r.q_start) * a.Hq + h;
    if ((r.kv_len - 1) / a.split == 0) { // a single split: final row
      a.out[row * D + d] = to_bf16(val);
      if (a.lse && d == 0) a.lse[row] = lse;
    } else {
      const int64_t prow = (r.rowbase + u.split) * a.Hq + h;
      a.part_o[prow * D + d] = val;
      if (d == 0) a.part_lse[prow] = lse;
    }
  }
}

template <int D>
cudaError_t launch_decode_d(const AttnArgs &a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(a.n_units), static_cast<unsigned>(a.Hkv));
  dim3 block(kDecodeWarps * 32);
  switch (a.G) {
  case 1: decode_kernel<D, 1><<<grid, block, 0, s>>>(a); break;
  case 2: decode_kernel<D, 2><<<grid, block, 0, s>>>(a); break;
  case 4: decode_kernel<D, 4><<<grid, block, 0, s>>>(a); break;
  case 8: decode_kernel<D, 8><<<grid, block, 0, s>>>(a); break;
  default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

} // namespace

cudaError_t launch_decode(const AttnArgs &a, cudaStream_t s) {
  if (a.n_units == 0) return cudaSuccess;
  return a.D == 128 ? launch_decode_d<128>(a, s) : launch_decode_d<64>(a, s);
}

} // namespace bia

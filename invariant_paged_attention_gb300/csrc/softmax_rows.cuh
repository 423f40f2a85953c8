// The softmax of one block of one S row, for the prefill kernels: one thread
// per row, S read from TMEM (tcgen05.ld), P written back as bf16 pairs over
// the row's first columns (tcgen05.st).  Templated on the block width KB
// (columns) and on which columns the row uses.
#pragma once

#include "bia_internal.h"
#include "ptx.cuh"

namespace bia {

// Whether column c of the block is visible: bit c of the 128-bit set vis.
__device__ __forceinline__ bool col_visible(const uint32_t (&vis)[4], int c) {
  return (vis[c >> 5] >> (c & 31)) & 1u;
}

// Which columns of a block a row uses: kFull every column, kFirst the first
// n_vis (causal / length limit), kBits the columns in a 128-bit set (custom
// mask).
enum ColMode { kFull, kFirst, kBits };

template <int MODE>
__device__ __forceinline__ bool col_used(int c, int32_t n_vis, const uint32_t (&vis)[4]) {
  if constexpr (MODE == kFull) return true;
  else if constexpr (MODE == kFirst) return c < n_vis;
  else return col_visible(vis, c);
}

// Max of this thread's row of S (KB fp32 columns at taddr) over the columns
// MODE selects.  Batches of 64 columns: two loads, one wait each.
template <int KB, int MODE>
__device__ __forceinline__ float row_block_max(uint32_t taddr, int32_t n_vis,
                                               const uint32_t (&vis)[4]) {
  static_assert(KB % 64 == 0 && KB <= 128, "block of 64 or 128 columns");
  float bm = -INFINITY;
#pragma unroll
  for (int h = 0; h < KB / 64; ++h) {
    uint32_t v0[32], v1[32];
    if constexpr (MODE == kFull) { // every column counts: the load reduces them
      float m0, m1;
      tmem_ld32_max(taddr + h * 64, v0, m0);
      tmem_ld32_max(taddr + h * 64 + 32, v1, m1);
      tmem_wait_ld();
      bm = fmax3(bm, m0, m1);
    } else {
      tmem_ld32(taddr + h * 64, v0);
      tmem_ld32(taddr + h * 64 + 32, v1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (col_used<MODE>(h * 64 + i, n_vis, vis)) bm = fmaxf(bm, __uint_as_float(v0[i]));
        if (col_used<MODE>(h * 64 + 32 + i, n_vis, vis)) bm = fmaxf(bm, __uint_as_float(v1[i]));
      }
    }
  }
  return bm;
}

// P = 2^(s*scale - m_sub) of this thread's row (zero in the columns MODE
// leaves out), written as bf16 pairs over the first KB/2 columns of the same
// TMEM row; returns the row sum of the fp32 P.
template <int KB, int MODE>
__device__ __forceinline__ float row_block_p(uint32_t taddr, int32_t n_vis,
                                             const uint32_t (&vis)[4], float scale,
                                             float m_sub) {
  const uint64_t scale2 = f32x2(scale, scale);
  const uint64_t neg2 = f32x2(-m_sub, -m_sub);
  uint64_t psum2 = 0;
#pragma unroll
  for (int c = 0; c < KB / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float x0, x1;
      f32x2_split(ffma2r(f32x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), scale2, neg2),
                  x0, x1);
      float p0 = ex2(x0), p1 = ex2(x1);
      if constexpr (MODE != kFull) {
        if (!col_used<MODE>(c * 32 + i, n_vis, vis)) p0 = 0.f;
        if (!col_used<MODE>(c * 32 + i + 1, n_vis, vis)) p1 = 0.f;
      }
      psum2 = fadd2(psum2, f32x2(p0, p1));
      pk[i / 2] = pack_bf16(p0, p1);
    }
    tmem_st16(taddr + c * 16, pk);
  }
  float ps0, ps1;
  f32x2_split(psum2, ps0, ps1);
  return ps0 + ps1;
}

} // namespace bia

// The Forecast projection, the fourth per-layer projection (bittide thread; techwalker
// section 二): f[b, r] = bf16(sum_c W[r, c] h[b, c]), one 128-wide head per KV group.
//
// A skinny GEMM (M = batch, N = G*d rows, K = hidden) bound by reading W, run on m16n8k16
// bf16 MMAs with the sequences as M. One CTA of 256 threads computes one tile of 8 rows x
// kProjSeqs sequences over the whole hidden dimension (MMA rows past kProjSeqs carry zeros):
// warp w takes the 32-wide K chunks w, w + 8, w + 16, ..., issuing the 16-byte loads of
// kProjUnroll chunks before their MMAs (at hidden 4096 all 16 of a warp's chunks: one round of
// loads, one memory round trip); the eight warps' partial tiles are then added in warp order
// through shared memory. Tiles of 8 sequences keep a thread's loads of that one round within
// its registers (W row and one hidden-state row per chunk). The contraction index may be
// permuted as long as A and B use the same permutation, so in each chunk lane (g, c) loads 8
// consecutive elements of W row g and of h rows g and g+8 (those that exist) and feeds
// elements 0-3 to one MMA and 4-7 to the next. Every launch that projects (the standalone
// projection and the decode prologue) runs this same arithmetic, so their forecasts agree bit
// for bit.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kProjWarps = 8;
constexpr int kProjThreads = kProjWarps * 32;
constexpr int kProjUnroll = 16;
// Sequences per tile (the MMA's M rows that carry data: 16, 8 or 4). With 8, a thread loads
// one hidden-state row per chunk, so kProjUnroll = 16 chunks fit its registers.
constexpr int kProjSeqs = 8;
static_assert(kProjSeqs == 16 || kProjSeqs == 8 || kProjSeqs == 4, "sequences per projection tile");

// CTAs of a projection of `rows` W rows (a multiple of 8) for `batch` sequences.
__host__ __device__ __forceinline__ int proj_ctas(int rows, int batch) {
  return (rows / 8) * ((batch + kProjSeqs - 1) / kProjSeqs);
}

struct ProjShared {
  float red[kProjWarps][16][8];
};

__device__ __forceinline__ uint4 proj_ld16(const __nv_bfloat16* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

// Tile (rows n_tile*8 .. +8, sequences m_tile*kProjSeqs .. +kProjSeqs) by threads 0..255 of
// the CTA, which synchronise with named barrier `bar` (256 threads).
__device__ __forceinline__ void project_rows(const ProjectArgs& a, int n_tile, int m_tile, ProjShared& sh,
                                             int bar) {
  const int n0 = n_tile * 8;
  const int m0 = m_tile * kProjSeqs;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* wrow = a.W + (size_t)(n0 + g) * a.hidden;
  const bool has0 = g < kProjSeqs && (m0 + g) < a.batch, has1 = g + 8 < kProjSeqs && (m0 + g + 8) < a.batch;
  const __nv_bfloat16* h0 = a.h + (size_t)(has0 ? m0 + g : 0) * a.hidden;
  const __nv_bfloat16* h1 = a.h + (size_t)(has1 ? m0 + g + 8 : 0) * a.hidden;
  const int n_chunks = a.hidden / 32;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int ch = warp; ch < n_chunks; ch += kProjWarps * kProjUnroll) {
    uint4 w[kProjUnroll], x[kProjUnroll], y[kProjUnroll];
#pragma unroll
    for (int u = 0; u < kProjUnroll; ++u) {
      const int cc = ch + u * kProjWarps;
      const bool in = cc < n_chunks;
      const int k = cc * 32 + 8 * c;
      w[u] = in ? proj_ld16(wrow + k) : z;
      x[u] = (in && has0) ? proj_ld16(h0 + k) : z;
      y[u] = (in && has1) ? proj_ld16(h1 + k) : z;
    }
#pragma unroll
    for (int u = 0; u < kProjUnroll; ++u) {
      mma_16816(acc, x[u].x, y[u].x, x[u].y, y[u].y, w[u].x, w[u].y);
      mma_16816(acc, x[u].z, y[u].z, x[u].w, y[u].w, w[u].z, w[u].w);
    }
  }
  // acc: (row g, cols 2c, 2c+1) and (row g+8, cols 2c, 2c+1); rows = sequences, cols = W rows
  sh.red[warp][g][2 * c] = acc[0];
  sh.red[warp][g][2 * c + 1] = acc[1];
  sh.red[warp][g + 8][2 * c] = acc[2];
  sh.red[warp][g + 8][2 * c + 1] = acc[3];
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kProjThreads) : "memory");
  if (t < 128) {
    const int m = t >> 3, n = t & 7;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kProjWarps; ++w) s += sh.red[w][m][n];
    if (m < kProjSeqs && m0 + m < a.batch) a.f[(size_t)(m0 + m) * a.rows + n0 + n] = __float2bfloat16_rn(s);
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kProjThreads) : "memory");   // red is free again
}

}  // namespace sparda

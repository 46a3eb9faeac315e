// The Forecast projection, the fourth per-layer projection (bittide thread; techwalker
// section 二): f[b, r] = bf16(sum_c W[r, c] h[b, c]), one 128-wide head per KV group.
//
// It is a skinny GEMM (M = batch, N = G*d rows, K = hidden) bound by reading W, run on
// m16n8k16 bf16 MMAs. grid (N/8 row tiles, 4 K-splits, M/16 sequence tiles); the four
// K-splits of a tile form a thread-block cluster. Each CTA's 8 warps take interleaved
// 32-wide K chunks of its quarter, issue all their 16-byte loads first, then the MMAs. The
// contraction index may be permuted as long as A and B use the same permutation, so in each
// chunk lane (g, c) loads 8 consecutive elements of W row g and of h rows g and g+8 and feeds
// elements 0-3 to one MMA and 4-7 to the next. Warps reduce through shared memory; the
// cluster's rank-0 CTA adds the other three CTAs' partial tiles through distributed shared
// memory and writes bf16.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kProjWarps = 8;
constexpr int kProjThreads = kProjWarps * 32;
constexpr int kProjSplit = 4;
constexpr int kProjUnroll = 4;

struct ProjShared {
  float red[kProjWarps][16][8];
  float part[16][8];
};

__device__ __forceinline__ uint4 proj_ld16(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// One CTA of the projection: rows n_tile*8 .. +8 of W, sequences m_tile*16 .. +16, the
// quarter `split` of the hidden dimension. The four CTAs of a (row, sequence) tile form a
// thread-block cluster in which CTA rank r holds quarter r; rank 0 writes the tile.
__device__ __forceinline__ void project_cta(const ProjectArgs& a, int n_tile, int split, int m_tile,
                                            ProjShared& sh) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int n0 = n_tile * 8;
  const int m0 = m_tile * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* wrow = a.W + (size_t)(n0 + g) * a.hidden;
  const bool has0 = (m0 + g) < a.batch, has1 = (m0 + g + 8) < a.batch;
  const __nv_bfloat16* h0 = a.h + (size_t)(has0 ? m0 + g : 0) * a.hidden;
  const __nv_bfloat16* h1 = a.h + (size_t)(has1 ? m0 + g + 8 : 0) * a.hidden;
  const int n_chunks = a.hidden / 32;
  const int q0 = n_chunks * split / kProjSplit, q1 = n_chunks * (split + 1) / kProjSplit;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int ch = q0 + warp; ch < q1; ch += kProjWarps * kProjUnroll) {
    uint4 w[kProjUnroll], x[kProjUnroll], y[kProjUnroll];
#pragma unroll
    for (int u = 0; u < kProjUnroll; ++u) {
      const int cc = ch + u * kProjWarps;
      const bool in = cc < q1;
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
  __syncthreads();
  if (threadIdx.x < 128) {
    const int m = threadIdx.x >> 3, n = threadIdx.x & 7;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kProjWarps; ++w) s += sh.red[w][m][n];
    sh.part[m][n] = s;
  }
  cluster.sync();                      // every CTA's partial tile is in its shared memory
  if (cluster.block_rank() == 0 && threadIdx.x < 128) {
    const int m = threadIdx.x >> 3, n = threadIdx.x & 7;
    float s = sh.part[m][n];
#pragma unroll
    for (int r = 1; r < kProjSplit; ++r) s += cluster.map_shared_rank(&sh.part[0][0], r)[m * 8 + n];
    if (m0 + m < a.batch) a.f[(size_t)(m0 + m) * a.rows + n0 + n] = __float2bfloat16_rn(s);
  }
  cluster.sync();                      // keep every CTA's tile alive until rank 0 has read it
}

}  // namespace sparda

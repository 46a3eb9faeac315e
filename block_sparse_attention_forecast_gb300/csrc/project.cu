// The Forecast projection, the fourth per-layer projection (bittide thread; techwalker
// section 二): f[b, r] = bf16(sum_c W[r, c] h[b, c]), one 128-wide head per KV group.
//
// It is a skinny GEMM (M = batch, N = G*d rows, K = hidden), run on m16n8k16 bf16 MMAs.
// CTA (n-tile of 8 rows, m-tile of 16 sequences), 8 warps splitting K in 32-wide chunks.
// The contraction index may be permuted as long as A and B use the same permutation, so in
// each 32-wide chunk lane (g, c) loads 8 consecutive elements (16 bytes) of W row g and of
// h rows g and g+8, and feeds elements 0-3 to the first MMA and 4-7 to the second: every
// load is a coalesced 16-byte vector and no shared-memory staging is needed.
#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kProjWarps = 8;

__device__ __forceinline__ uint4 ld16(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__global__ void __launch_bounds__(kProjWarps * 32) forecast_project_kernel(const ProjectArgs a) {
  __shared__ float red[kProjWarps][16][8];
  const int n0 = blockIdx.x * 8;
  const int m0 = blockIdx.y * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* wrow = a.W + (size_t)(n0 + g) * a.hidden;
  const bool has0 = (m0 + g) < a.batch, has1 = (m0 + g + 8) < a.batch;
  const __nv_bfloat16* h0 = a.h + (size_t)(has0 ? m0 + g : 0) * a.hidden;
  const __nv_bfloat16* h1 = a.h + (size_t)(has1 ? m0 + g + 8 : 0) * a.hidden;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int k0 = warp * 32; k0 < a.hidden; k0 += kProjWarps * 32) {
    const uint4 w = ld16(wrow + k0 + 8 * c);
    const uint4 x = has0 ? ld16(h0 + k0 + 8 * c) : z;
    const uint4 y = has1 ? ld16(h1 + k0 + 8 * c) : z;
    mma_16816(acc, x.x, y.x, x.y, y.y, w.x, w.y);
    mma_16816(acc, x.z, y.z, x.w, y.w, w.z, w.w);
  }
  // acc: (row g, cols 2c, 2c+1) and (row g+8, cols 2c, 2c+1); rows = sequences, cols = W rows
  red[warp][g][2 * c] = acc[0];
  red[warp][g][2 * c + 1] = acc[1];
  red[warp][g + 8][2 * c] = acc[2];
  red[warp][g + 8][2 * c + 1] = acc[3];
  __syncthreads();
  if (threadIdx.x < 128) {
    const int m = threadIdx.x >> 3, n = threadIdx.x & 7;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kProjWarps; ++w) s += red[w][m][n];
    if (m0 + m < a.batch) a.f[(size_t)(m0 + m) * a.rows + n0 + n] = __float2bfloat16_rn(s);
  }
}

void launch_forecast_project(const ProjectArgs& a, cudaStream_t s) {
  dim3 grid(a.rows / 8, (a.batch + 15) / 16);
  forecast_project_kernel<<<grid, kProjWarps * 32, 0, s>>>(a);
}

}  // namespace sparda

// The baseline, query-driven selector that SparDA replaces (bittide thread, the paragraph on
// the standard selector; 10100 "先把痛点讲透"): every query head of a GQA group scores every
// compressed key, each head's scores go through a softmax over the windows, the per-head
// probabilities are summed over the group, and the sums are max-pooled onto blocks for the
// same top-k as the Forecast selector. Built as the comparison point for the selector A/B.
//
// Kernel 1, grid (64-window tiles, sequence-groups), 4 warps: the tile of compressed keys is
// one 64 x 128 bf16 box pair loaded by TMA with the 128-byte swizzle (the layout of a K block
// in the attention kernel); z = Q ck^T for the group's 16 heads runs on m16n8k16 bf16 MMAs,
// in the exp2 domain (scale log2(e)/sqrt(d)). It stores z and, per head, the tile's maximum
// and sum of exp2(z - max).
// Kernel 2, one CTA of 256 threads per sequence-group: combines the tile statistics into each
// head's softmax normaliser, forms s[i] = sum_h exp2(z[h][i] - M_h) / L_h in shared memory,
// max-pools the windows 4j-1 .. 4j+3 onto block j, and runs the exact top-k.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace sparda {

constexpr int kMhTile = 64;
constexpr int kMhThreads = 128;

int multihead_tiles(int w_cap) { return (w_cap + kMhTile - 1) / kMhTile; }

__device__ __forceinline__ uint32_t mh_swz(const uint8_t* tile, int r, int chunk) {
  return smem_addr(tile + (chunk >> 3) * (kBlockBytes / 2) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kMhThreads) multihead_scores_kernel(
    const MultiheadArgs a, const __grid_constant__ CUtensorMap mck) {
  __shared__ __align__(1024) uint8_t tile[kBlockBytes];
  __shared__ uint64_t bar;
  __shared__ float red_m[4][kHeads], red_l[4][kHeads];
  const int bg = blockIdx.y, tl = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int T = a.seq_len[bg / a.G];
  const bool valid = T >= 1 && T <= a.max_ctx;
  const int W = valid ? num_windows(T - 1) : 0;
  const int i0 = tl * kMhTile;
  float2* st = a.stats + ((size_t)bg * a.n_tiles + tl) * kHeads;
  if (i0 >= W) {
    if (tid < kHeads) st[tid] = make_float2(-INFINITY, 0.f);
    return;
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, kBlockBytes);
    const int row = bg * a.W_cap + i0;
    tma_load_2d(tile, &mck, 0, row, &bar);
    tma_load_2d(tile + kBlockBytes / 2, &mck, 64, row, &bar);
  }
  uint32_t qf[8][4];
  {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)bg * kHeads + g) * kHeadDim);
    const uint32_t* q1 = q0 + 8 * (kHeadDim / 2);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = q0[8 * ks + cq];
      qf[ks][1] = q1[8 * ks + cq];
      qf[ks][2] = q0[8 * ks + 4 + cq];
      qf[ks][3] = q1[8 * ks + 4 + cq];
    }
  }
  __syncthreads();
  const bool ok = __syncthreads_and(mbar_wait(&bar, 0, a.err));
  float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if (ok) {
    const int r = 16 * warp + (lane & 7) + ((lane >> 4) << 3);
    const int hi = (lane >> 3) & 1;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(mh_swz(tile, r, 2 * ks + hi), b0, b1, b2, b3);
      mma_16816(sc[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
      mma_16816(sc[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
    }
  }
  const float sl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
  float* z = a.z + (size_t)bg * kHeads * a.W_cap;
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + 16 * warp + 8 * nt + 2 * cq + (e & 1);
      const int h = (e < 2) ? g : g + 8;
      const float v = (i < W && ok) ? sc[nt][e] * sl2 : -INFINITY;
      sc[nt][e] = v;
      if (i < W) z[(size_t)h * a.W_cap + i] = v;
      if (e < 2) m0 = fmaxf(m0, v); else m1 = fmaxf(m1, v);
    }
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  const float b0 = (m0 == -INFINITY) ? 0.f : m0, b1 = (m1 == -INFINITY) ? 0.f : m1;
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    l0 += exp2f(sc[nt][0] - b0) + exp2f(sc[nt][1] - b0);
    l1 += exp2f(sc[nt][2] - b1) + exp2f(sc[nt][3] - b1);
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (cq == 0) {
    red_m[warp][g] = m0;
    red_l[warp][g] = l0;
    red_m[warp][g + 8] = m1;
    red_l[warp][g + 8] = l1;
  }
  __syncthreads();
  if (tid < kHeads) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][tid]);
    const float base = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) L += exp2f(red_m[w][tid] - base) * red_l[w][tid];
    st[tid] = make_float2(M, L);
  }
}

// (m1, l1) + (m2, l2) of the same head: one softmax normaliser over both parts.
__device__ __forceinline__ float2 lse_combine(float2 x, float2 y) {
  const float M = fmaxf(x.x, y.x);
  if (M == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(M, x.y * exp2f(x.x - M) + y.y * exp2f(y.x - M));
}

__global__ void __launch_bounds__(kTopkThreads, 1) multihead_pool_topk_kernel(const MultiheadArgs a) {
  extern __shared__ float s_win[];                 // [W_cap] summed probabilities
  __shared__ TopkShared sh;
  __shared__ float s_M[kHeads], s_invL[kHeads];
  const int bg = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int T = a.seq_len[bg / a.G];
  const bool valid = T >= 1 && T <= a.max_ctx;
  if (!valid && t == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
  const int W = valid ? num_windows(T - 1) : 0;
  const int nb = valid ? (T - 1) / kBlock + 1 : 0;
  const int n_used = (W + kMhTile - 1) / kMhTile;
  // each warp owns heads 2w and 2w+1: fold the tile statistics
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = 2 * warp + hh;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int tl = lane; tl < n_used; tl += 32) acc = lse_combine(acc, a.stats[((size_t)bg * a.n_tiles + tl) * kHeads + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float2 other;
      other.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
      other.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
      acc = lse_combine(acc, other);
    }
    if (lane == 0) {
      s_M[h] = acc.x;
      s_invL[h] = acc.y > 0.f ? 1.f / acc.y : 0.f;
    }
  }
  __syncthreads();
  const float* z = a.z + (size_t)bg * kHeads * a.W_cap;
  for (int i = t; i < W; i += kTopkThreads) {
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < kHeads; ++h) s += exp2f(z[(size_t)h * a.W_cap + i] - s_M[h]) * s_invL[h];
    s_win[i] = s;
  }
  __syncthreads();
  float* S = a.block_scores + (size_t)bg * a.nb_cap;
  for (int j = t; j < nb; j += kTopkThreads) {
    float m = -INFINITY;
#pragma unroll
    for (int d = -1; d <= 3; ++d) {
      const int w = kWinPerBlock * j + d;
      if (w >= 0 && w < W) m = fmaxf(m, s_win[w]);
    }
    S[j] = m;
  }
  __syncthreads();
  topk_select(S, a.idx + (size_t)bg * (a.topk + 2), a.cnt + bg, a.topk, a.max_ctx, T, sh);
}

void launch_multihead_select(const MultiheadArgs& a, const CUtensorMap& mck, int bg_count, cudaStream_t s) {
  dim3 g1(a.n_tiles, bg_count);
  multihead_scores_kernel<<<g1, kMhThreads, 0, s>>>(a, mck);
  const int smem = a.W_cap * (int)sizeof(float);
  cudaFuncSetAttribute(multihead_pool_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  multihead_pool_topk_kernel<<<bg_count, kTopkThreads, smem, s>>>(a);
}

}  // namespace sparda

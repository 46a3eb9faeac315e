// Block-sparse GQA decode attention (bittide thread: the next layer's own queries attend the
// blocks the forecast picked; techwalker section 六: SparDA leaves the sparse attention
// computation itself unchanged).
//
// grid (n_split, B*G), 128 threads (4 warps). CTA `split` of a (sequence, group) owns the
// selected blocks [split*kBPC, split*kBPC + kBPC). Thread 0 issues, per block, four tiled
// TMA loads (K and V, two 64-column halves each, 128-byte swizzle) onto one mbarrier. Warp w
// handles tokens 16w .. 16w+15 of every block: S = Q K^T with the group's 16 query heads as
// the M dimension of m16n8k16 bf16 MMAs, an online softmax in float32 (exp2 domain), then
// O += P V with P re-packed from the S accumulators. The four warps' partial results are
// merged in shared memory; with several splits each CTA stores (O, max, sum) to the
// workspace and the last CTA of the (sequence, group) merges them (log-sum-exp weights).
#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kAttnThreads = 128;
constexpr int kBPC = 2;                            // selected blocks per CTA
constexpr int kSlotBytes = 2 * kBlockBytes;        // K + V of one block
constexpr int kCombineBytes = 4 * (kHeads * kHeadDim + 2 * kHeads) * 4;
constexpr int kAttnSmem = 1024 /*align slack*/ + 1024 /*barriers*/ +
                          (kBPC * kSlotBytes > kCombineBytes ? kBPC * kSlotBytes : kCombineBytes);

int attn_blocks_per_cta() { return kBPC; }

// Shared-memory address of 16-byte chunk `chunk` (0..15 over the 128 dims) of row `r` of a
// K or V block staged as two 64-row x 128-byte halves with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t swz(const uint8_t* tile, int r, int chunk) {
  return smem_addr(tile + (chunk >> 3) * (kBlockBytes / 2) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kAttnThreads) sparse_attn_kernel(
    const AttnArgs a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
    const __grid_constant__ CUtensorMap hk, const __grid_constant__ CUtensorMap hv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* slots = smem + 1024;
  __shared__ bool s_last;

  const int bg = blockIdx.y;
  const int b = bg / a.G;
  const int split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;

  const int T = a.seq_len[b];
  const bool valid = (T >= 1 && T <= a.max_ctx);
  const int tb = valid ? (T - 1) / kBlock : 0;
  const int n_sel = valid ? min(max(a.cnt[bg], 0), a.kslots) : 0;
  const int s0 = split * kBPC;
  const int s1 = min(s0 + kBPC, n_sel);
  const int32_t* idx = a.idx + (size_t)bg * a.kslots;
  const float sl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)

  if (s0 < s1) {
    if (tid == 0) {
      for (int i = 0; i < s1 - s0; ++i) mbar_init(&bars[i], 1);
      fence_mbar_init();
      for (int i = 0; i < s1 - s0; ++i) {
        const int s = s0 + i;
        int j = idx[s];
        if (j < 0 || j > tb) {
          atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
          j = 0;
        }
        const CUtensorMap* tk = &mk;
        const CUtensorMap* tv = &mv;
        int row;
        if (!a.offload) {
          row = (bg * a.max_ctx) + j * kBlock;
        } else if (j == 0 || j == tb) {
          tk = &hk;
          tv = &hv;
          row = (bg * kHotSlots + hot_slot(j)) * kBlock;
        } else {
          row = (bg * a.kslots + s) * kBlock;
        }
        uint8_t* dst = slots + i * kSlotBytes;
        mbar_arrive_expect_tx(&bars[i], kSlotBytes);
        tma_load_2d(dst, tk, 0, row, &bars[i]);
        tma_load_2d(dst + kBlockBytes / 2, tk, 64, row, &bars[i]);
        tma_load_2d(dst + kBlockBytes, tv, 0, row, &bars[i]);
        tma_load_2d(dst + kBlockBytes + kBlockBytes / 2, tv, 64, row, &bars[i]);
      }
    }
    // A fragments of Q (16 heads x 128 dims) for the 8 k-steps of 16 dims.
    uint32_t qf[8][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)bg * kHeads + g) * kHeadDim);
      const uint32_t* q1 = q0 + 8 * (kHeadDim / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[ks][0] = q0[8 * ks + c];
        qf[ks][1] = q1[8 * ks + c];
        qf[ks][2] = q0[8 * ks + 4 + c];
        qf[ks][3] = q1[8 * ks + 4 + c];
      }
    }
    __syncthreads();   // barriers initialised

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int i = 0; i < s1 - s0; ++i) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[i], 0, a.err));
      if (!ok) break;
      int j = idx[s0 + i];
      if (j < 0 || j > tb) j = 0;
      const uint8_t* Kt = slots + i * kSlotBytes;
      const uint8_t* Vt = Kt + kBlockBytes;

      // S = Q K^T over this warp's 16 tokens (two n-tiles of 8).
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int r = 16 * warp + (lane & 7) + ((lane >> 4) << 3);
        const int hi = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(swz(Kt, r, 2 * ks + hi), b0, b1, b2, b3);
          mma_16816(sc[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
          mma_16816(sc[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
        }
      }
      // Scale into the exp2 domain and mask tokens at or beyond T.
      const int tok0 = j * kBlock + 16 * warp + 2 * c;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = tok0 + 8 * nt + (e & 1);
          sc[nt][e] = (pos < T) ? sc[nt][e] * sl2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
      m0 = mn0;
      m1 = mn1;
      float p[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = exp2f(sc[nt][0] - base0);
        p[nt][1] = exp2f(sc[nt][1] - base0);
        p[nt][2] = exp2f(sc[nt][2] - base1);
        p[nt][3] = exp2f(sc[nt][3] - base1);
      }
      float ps0 = p[0][0] + p[0][1] + p[1][0] + p[1][1];
      float ps1 = p[0][2] + p[0][3] + p[1][2] + p[1][3];
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      // P (16 heads x 16 tokens) as the A operand of O += P V.
      const uint32_t pa0 = pack_bf16(p[0][0], p[0][1]);
      const uint32_t pa1 = pack_bf16(p[0][2], p[0][3]);
      const uint32_t pa2 = pack_bf16(p[1][0], p[1][1]);
      const uint32_t pa3 = pack_bf16(p[1][2], p[1][3]);
      {
        const int r = 16 * warp + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int hi = lane >> 4;
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(swz(Vt, r, 2 * np + hi), b0, b1, b2, b3);
          mma_16816(o[2 * np], pa0, pa1, pa2, pa3, b0, b1);
          mma_16816(o[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
    }

    // Merge the four warps' partial results.
    __syncthreads();   // all warps are done with the staged blocks
    float* cO = reinterpret_cast<float*>(slots);                     // [4][16][128]
    float* cM = cO + 4 * kHeads * kHeadDim;                          // [4][16]
    float* cL = cM + 4 * kHeads;                                     // [4][16]
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      float* r0p = cO + (warp * kHeads + g) * kHeadDim + 8 * n + 2 * c;
      float* r1p = r0p + 8 * kHeadDim;
      r0p[0] = o[n][0];
      r0p[1] = o[n][1];
      r1p[0] = o[n][2];
      r1p[1] = o[n][3];
    }
    if (c == 0) {
      cM[warp * kHeads + g] = m0;
      cM[warp * kHeads + g + 8] = m1;
      cL[warp * kHeads + g] = l0;
      cL[warp * kHeads + g + 8] = l1;
    }
    __syncthreads();
    const int col = tid;   // one output dim per thread
    for (int h = 0; h < kHeads; ++h) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, cM[w * kHeads + h]);
      const float base = (M == -INFINITY) ? 0.f : M;
      float O = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float wt = exp2f(cM[w * kHeads + h] - base);
        O += wt * cO[(w * kHeads + h) * kHeadDim + col];
        L += wt * cL[w * kHeads + h];
      }
      if (gridDim.x == 1) {
        a.out[((size_t)bg * kHeads + h) * kHeadDim + col] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
      } else {
        a.part_o[(((size_t)bg * a.n_split + split) * kHeads + h) * kHeadDim + col] = O;
        if (col == 0) {
          a.part_ml[((size_t)bg * a.n_split + split) * 2 * kHeads + h] = M;
          a.part_ml[((size_t)bg * a.n_split + split) * 2 * kHeads + kHeads + h] = L;
        }
      }
    }
  }

  if (gridDim.x == 1) {
    if (s0 >= s1)   // nothing selected: zero output
      for (int h = 0; h < kHeads; ++h)
        a.out[((size_t)bg * kHeads + h) * kHeadDim + tid] = __float2bfloat16_rn(0.f);
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(a.counters + bg, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n_used = (n_sel + kBPC - 1) / kBPC;
  const int col = tid;
  for (int h = 0; h < kHeads; ++h) {
    float M = -INFINITY;
    for (int sp = 0; sp < n_used; ++sp)
      M = fmaxf(M, __ldcg(a.part_ml + ((size_t)bg * a.n_split + sp) * 2 * kHeads + h));
    const float base = (M == -INFINITY) ? 0.f : M;
    float O = 0.f, L = 0.f;
    for (int sp = 0; sp < n_used; ++sp) {
      const float* ml = a.part_ml + ((size_t)bg * a.n_split + sp) * 2 * kHeads;
      const float wt = exp2f(__ldcg(ml + h) - base);
      O += wt * __ldcg(a.part_o + (((size_t)bg * a.n_split + sp) * kHeads + h) * kHeadDim + col);
      L += wt * __ldcg(ml + kHeads + h);
    }
    a.out[((size_t)bg * kHeads + h) * kHeadDim + col] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
  }
  if (tid == 0) a.counters[bg] = 0u;
}

void launch_sparse_attn(const AttnArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& hk, const CUtensorMap& hv, int bg_count,
                        cudaStream_t s) {
  cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  dim3 grid(a.n_split, bg_count);
  sparse_attn_kernel<<<grid, kAttnThreads, kAttnSmem, s>>>(a, mk, mv, hk, hv);
}

}  // namespace sparda

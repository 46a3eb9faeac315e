// Chunked prefill: the Forecast selector and the baseline multi-head selector applied to
// 64-token query chunks, and causal block-sparse prefill attention.
//
// The pages report prefill as well as decode figures (bittide thread and abstract: up to
// 1.25x faster prefill; techwalker section 五: in prefill the block-sparse attention is the
// main cost, the block selection grows with the context and nears it at 128K, and the
// Forecast indexer cuts the selection cost by up to 2.5x). The prefill selection rule is a
// reading: chunk c (tokens 64c .. 64c+63) shares one selection, scores the compressed keys
// complete before it (windows i < W_c = num_windows(64c)), keeps blocks 0 and c and the
// top-k of blocks 1 .. c-1. The Forecast score of a window sums the decode score over the
// chunk's tokens, s_c[i] = sum_t f_t . ck_i = (sum_t f_t) . ck_i; the baseline sums each
// (token, head) query's softmax over the windows. Every token attends its chunk's blocks up
// to its own position.
//
// Kernels:
//   prefill_forecast_score_kernel  per (sequence-group, 16-chunk tile): the chunks' summed
//       forecasts (float32) against 64-window tiles of compressed keys staged in shared memory
//       by cp.async (double buffered), float32 FMA on CUDA cores (128 FMAs per window and
//       chunk, exact bf16 inputs), max-pooled onto blocks in shared memory; block scores to
//       the workspace.
//   prefill_topk_kernel            one top-k CTA per (sequence-group, chunk) (topk.cuh).
//   prefill_multihead_kernel       the baseline: per (sequence-group, chunk), for each of
//       8 slices of 8 tokens, two passes over TMA-staged 64-window tiles on bf16 mma.sync
//       (a warp = one token's 16 heads): the per-row log-sum-exp, then the column sums of the
//       normalised probabilities, added in a fixed order into the chunk's window sums in
//       shared memory; then max-pool and the top-k in the same CTA.
//   prefill_attn_tc_kernel         per (sequence-group, chunk, 16-token slice): two 128-row
//       query tiles on the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor
//       memory), the chunk's selected K/V blocks through a TMA ring, causal in the chunk's own
//       block (described at the kernel).
#include "common.cuh"
#include "kernels.h"
#include "tc05.cuh"
#include "topk.cuh"

namespace sparda {

namespace {

// ------------------------------------------------------------------ shared helpers
constexpr int kPfChunks = 16;                 // chunk rows per forecast-scoring CTA
constexpr int kPfWin = 64;                    // windows per tile
constexpr int kPfThreads = 256;
constexpr int kCkStride = kHeadDim + 8;       // bf16 per padded shared row: 272 B, no conflicts

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const int n = pred ? 16 : 0;                // 0: the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)), "l"(gmem), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ bool valid_len(int T, int max_ctx) { return T >= 1 && T <= max_ctx; }

}  // namespace

// ==================================================================== Forecast scoring
__global__ void __launch_bounds__(kPfThreads) prefill_forecast_score_kernel(const PrefillArgs a) {
  __shared__ __align__(16) float fs[kPfChunks][kHeadDim];            // summed forecasts
  __shared__ __align__(16) __nv_bfloat16 ckt[2][kPfWin][kCkStride];  // window tiles
  __shared__ float sw[kPfChunks][kPfWin + 1];                        // [.][0] = halo window
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int bg = blockIdx.y, b = bg / a.G, g = bg % a.G;
  const int n_ct = (a.nb_cap + kPfChunks - 1) / kPfChunks;
  const int c0 = (n_ct - 1 - (int)blockIdx.x) * kPfChunks;          // the longest rows first
  const int T = a.seq_len[b];
  if (!valid_len(T, a.max_ctx)) {
    if (t == 0 && blockIdx.x == 0 && g == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int nc = (T + kBlock - 1) / kBlock;
  if (c0 >= nc) return;
  const int c_last = min(c0 + kPfChunks, nc) - 1;

  // ---- the chunks' summed forecasts: thread t sums 8 dims of chunk t/16 over its tokens
  {
    const int r = t >> 4, d8 = (t & 15) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int p0 = (c0 + r) * kBlock;
    const int p1 = min(p0 + kBlock, T);
    const size_t row_stride = (size_t)a.G * kHeadDim;
    const __nv_bfloat16* fp = a.f + ((size_t)b * a.max_ctx * a.G + g) * kHeadDim + d8;
#pragma unroll 8
    for (int p = p0; p < p1; ++p) {
      const uint4 v = *reinterpret_cast<const uint4*>(fp + (size_t)p * row_stride);
      acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
      acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
      acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
      acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) fs[r][d8 + e] = acc[e];
  }
  if (t < kPfChunks) sw[t][0] = -INFINITY;                            // no window before tile 0

  // ---- window tiles, double buffered
  const int W_last = num_windows(kBlock * c_last);
  const int n_wt = (W_last + kPfWin - 1) / kPfWin;
  const __nv_bfloat16* ckg = a.ck + (size_t)bg * a.W_cap * kHeadDim;
  auto load_tile = [&](int m, int buf) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = e * kPfThreads + t;                               // 16-byte chunk of the tile
      const int r = q >> 4, c16 = q & 15;
      const int i = m * kPfWin + r;
      const bool in = i < W_last;
      cp_async16(&ckt[buf][r][c16 * 8], ckg + (size_t)(in ? i : 0) * kHeadDim + c16 * 8, in);
    }
    cp_async_commit();
  };
  if (n_wt > 0) load_tile(0, 0);
  const int r0 = warp, r1 = warp + 8;                                 // chunk rows of this thread
  const int Wr0 = num_windows(kBlock * (c0 + r0)), Wr1 = num_windows(kBlock * (c0 + r1));
  for (int m = 0; m < n_wt; ++m) {
    const int buf = m & 1;
    if (m + 1 < n_wt) {
      load_tile(m + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();                                                  // tile m and fs visible
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;                 // [row][window]
    const __nv_bfloat16* k0 = &ckt[buf][lane][0];
    const __nv_bfloat16* k1 = &ckt[buf][lane + 32][0];
#pragma unroll 4
    for (int d = 0; d < kHeadDim; d += 8) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(k0 + d);
      const uint4 u1 = *reinterpret_cast<const uint4*>(k1 + d);
      const float4 fa0 = *reinterpret_cast<const float4*>(&fs[r0][d]);
      const float4 fb0 = *reinterpret_cast<const float4*>(&fs[r0][d + 4]);
      const float4 fa1 = *reinterpret_cast<const float4*>(&fs[r1][d]);
      const float4 fb1 = *reinterpret_cast<const float4*>(&fs[r1][d + 4]);
      const float x0[8] = {bf16_lo(u0.x), bf16_hi(u0.x), bf16_lo(u0.y), bf16_hi(u0.y),
                           bf16_lo(u0.z), bf16_hi(u0.z), bf16_lo(u0.w), bf16_hi(u0.w)};
      const float x1[8] = {bf16_lo(u1.x), bf16_hi(u1.x), bf16_lo(u1.y), bf16_hi(u1.y),
                           bf16_lo(u1.z), bf16_hi(u1.z), bf16_lo(u1.w), bf16_hi(u1.w)};
      const float f0[8] = {fa0.x, fa0.y, fa0.z, fa0.w, fb0.x, fb0.y, fb0.z, fb0.w};
      const float f1[8] = {fa1.x, fa1.y, fa1.z, fa1.w, fb1.x, fb1.y, fb1.z, fb1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s00 = fmaf(f0[e], x0[e], s00);
        s01 = fmaf(f0[e], x1[e], s01);
        s10 = fmaf(f1[e], x0[e], s10);
        s11 = fmaf(f1[e], x1[e], s11);
      }
    }
    const int i0 = m * kPfWin + lane, i1 = i0 + 32;
    sw[r0][1 + lane] = i0 < Wr0 ? s00 : -INFINITY;
    sw[r0][33 + lane] = i1 < Wr0 ? s01 : -INFINITY;
    sw[r1][1 + lane] = i0 < Wr1 ? s10 : -INFINITY;
    sw[r1][33 + lane] = i1 < Wr1 ? s11 : -INFINITY;
    __syncthreads();
    // max-pool: block j = 16m + jj takes windows 4j-1 .. 4j+3 (local 4jj .. 4jj+4 with the
    // halo window in column 0); thread t: chunk row t/16, block t%16
    {
      const int r = t >> 4, jj = t & 15, j = m * 16 + jj;
      float S = sw[r][4 * jj];
#pragma unroll
      for (int e = 1; e <= 4; ++e) S = fmaxf(S, sw[r][4 * jj + e]);
      const int c = c0 + r;
      if (c <= c_last && j < a.nb_cap && j <= c)
        a.block_scores[((size_t)bg * a.nb_cap + c) * a.nb_cap + j] = S;
    }
    __syncthreads();                                                  // sw read before the halo moves
    if (t < kPfChunks) sw[t][0] = sw[t][kPfWin];
  }
}

__global__ void __launch_bounds__(kTopkThreads) prefill_topk_kernel(const PrefillArgs a) {
  __shared__ TopkShared sh;
  const int bg = blockIdx.y, b = bg / a.G, c = blockIdx.x;
  const int T = a.seq_len[b];
  const int kslots = a.topk + 2;
  int32_t* idx = a.idx + ((size_t)bg * a.nb_cap + c) * kslots;
  int32_t* cnt = a.cnt + (size_t)bg * a.nb_cap + c;
  if (!valid_len(T, a.max_ctx) || c * kBlock >= T) {
    // no such chunk: an empty selection
    for (int s = threadIdx.x; s < kslots; s += blockDim.x) idx[s] = -1;
    if (threadIdx.x == 0) *cnt = 0;
    return;
  }
  // the decode rule for a context whose current token lies in block c: tail block c, windows
  // before the chunk (the scores were written for exactly those)
  topk_select(a.block_scores + ((size_t)bg * a.nb_cap + c) * a.nb_cap, idx, cnt, a.topk, a.max_ctx,
              c * kBlock + 1, sh);
}

// ==================================================================== tensor-core helpers
namespace {

constexpr int kPaConsumerWarps = 8;
constexpr int kPaThreads = (kPaConsumerWarps + 1) * 32;     // 8 consumer warps + producer
constexpr int kMhStages = 6;
constexpr int kMhTileBytes = kBlockBytes;                    // 64 windows x 128 dims bf16
// [align slack][barriers][ring][per-warp column sums, 2 buffers][top-k scratch][window sums]
constexpr int kMhFixedSmem = 1024 + 1024 + kMhStages * kMhTileBytes + 2 * kPaConsumerWarps * 64 * 4 +
                             ((int)sizeof(TopkShared) + 15) / 16 * 16;
__host__ __device__ constexpr int mh_smem_bytes(int w_cap) { return kMhFixedSmem + 4 * w_cap; }
static_assert(mh_smem_bytes(kMaxCtx / kWinStride) <= 227 * 1024, "the baseline prefill selector fits shared memory");

// Shared address of 16-byte chunk `chunk` (0..15 over the 128 dims) of row r of a 64-row
// tile staged by TMA as two 64-column halves with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_addr(const uint8_t* tile, int r, int chunk) {
  return smem_addr(tile + (chunk >> 3) * (kBlockBytes / 2) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kPaConsumerWarps * 32) : "memory");
}

// The A fragments of one token's 16 query heads (rows = heads, k = dims), from global memory.
__device__ __forceinline__ void load_q_frags(const __nv_bfloat16* q16, int lane, uint32_t (&qf)[8][4]) {
  const int g = lane >> 2, cq = lane & 3;
  const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q16 + (size_t)g * kHeadDim);
  const uint32_t* q1 = q0 + 8 * (kHeadDim / 2);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qf[ks][0] = q0[8 * ks + cq];
    qf[ks][1] = q1[8 * ks + cq];
    qf[ks][2] = q0[8 * ks + 4 + cq];
    qf[ks][3] = q1[8 * ks + 4 + cq];
  }
}

// S[16 heads x 64 rows of the tile] = Q . tile^T; sc[n] is n-tile n (rows 8n .. 8n+7 of the
// tile) in the m16n8 accumulator layout.
__device__ __forceinline__ void qk_tile(const uint32_t (&qf)[8][4], const uint8_t* tile, int lane, float (&sc)[8][4]) {
#pragma unroll
  for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
  const int hi = (lane >> 3) & 1;
#pragma unroll
  for (int wq = 0; wq < 4; ++wq) {
    const int r = 16 * wq + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz_addr(tile, r, 2 * ks + hi), b0, b1, b2, b3);
      mma_16816(sc[2 * wq], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
      mma_16816(sc[2 * wq + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
    }
  }
}

}  // namespace

// ==================================================================== baseline multi-head
__global__ void __launch_bounds__(kPaThreads, 1) prefill_multihead_kernel(const PrefillArgs a,
                                                                          const __grid_constant__ CUtensorMap mck) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMhStages;
  uint8_t* ring = smem + 1024;
  float* part = reinterpret_cast<float*>(ring + kMhStages * kMhTileBytes);    // [2][8 warps][64]
  TopkShared& sh = *reinterpret_cast<TopkShared*>(part + 2 * kPaConsumerWarps * 64);
  float* win_sum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(&sh) +
                                            ((int)sizeof(TopkShared) + 15) / 16 * 16);   // [W_cap]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bg = blockIdx.y, b = bg / a.G, g = bg % a.G;
  const int c = a.nb_cap - 1 - (int)blockIdx.x;                // the longest chunks first
  const int T = a.seq_len[b];
  const int kslots = a.topk + 2;
  const size_t row = (size_t)bg * a.nb_cap + c;
  if (!valid_len(T, a.max_ctx) || c * kBlock >= T) {
    if (!valid_len(T, a.max_ctx) && tid == 0 && blockIdx.x == 0 && g == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    for (int s = tid; s < kslots; s += blockDim.x) a.idx[row * kslots + s] = -1;
    if (tid == 0) a.cnt[row] = 0;
    return;
  }
  const int Wc = num_windows(c * kBlock);
  const int n_wt = (Wc + 63) / 64;
  const int n_tok = min(kBlock, T - c * kBlock);
  const int n_sl = (n_tok + kPaConsumerWarps - 1) / kPaConsumerWarps;
  const int n_loads = n_sl * 2 * n_wt;                           // slices x passes x tiles

  if (tid == 0) {
    for (int i = 0; i < kMhStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPaConsumerWarps);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < Wc; i += blockDim.x) win_sum[i] = 0.f;
  __syncthreads();

  if (warp == kPaConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mck);
      for (int it = 0; it < n_loads; ++it) {
        const int m = it % n_wt;
        const int stage = it % kMhStages;
        if (it >= kMhStages && !mbar_wait(&empty[stage], ((it / kMhStages) & 1) ^ 1, a.err)) break;
        uint8_t* dst = ring + stage * kMhTileBytes;
        const int rr = bg * a.W_cap + m * 64;
        mbar_arrive_expect_tx(&full[stage], kMhTileBytes);
        tma_load_2d(dst, &mck, 0, rr, &full[stage]);
        tma_load_2d(dst + kBlockBytes / 2, &mck, 64, rr, &full[stage]);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cq = lane & 3;
    const float zl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    bool ok = true;
    int it = 0, tile_no = 0;
    for (int s = 0; s < n_sl; ++s) {
      const int tok = c * kBlock + s * kPaConsumerWarps + warp;
      const bool active = tok < T;
      uint32_t qf[8][4];
      if (active) {
        load_q_frags(a.q + (((size_t)b * a.max_ctx + tok) * a.G + g) * kHeads * kHeadDim, lane, qf);
      }
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      for (int pass = 0; pass < 2; ++pass) {
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
        for (int m = 0; m < n_wt; ++m, ++it) {
          const int stage = it % kMhStages;
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (it / kMhStages) & 1, a.err));
          float sc[8][4];
          if (ok && active) {
            qk_tile(qf, ring + stage * kMhTileBytes, lane, sc);
            const int ibase = m * 64 + 2 * cq;
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                sc[n][e] = (ibase + 8 * n + (e & 1)) < Wc ? sc[n][e] * zl2 : -INFINITY;
          }
          __syncwarp();
          if (lane == 0) bar_arrive(&empty[stage]);
          if (pass == 0) {
            if (ok && active) {
              float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
              for (int n = 0; n < 8; ++n) {
                mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
                mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
              }
              mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
              mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
              mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
              mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
              const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
              const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
              const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
              float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
              for (int n = 0; n < 8; ++n) {
                ps0 += exp2f(sc[n][0] - base0) + exp2f(sc[n][1] - base0);
                ps1 += exp2f(sc[n][2] - base1) + exp2f(sc[n][3] - base1);
              }
              ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
              ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
              ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
              ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
              l0 = l0 * exp2f(m0 - base0) + ps0;
              l1 = l1 * exp2f(m1 - base1) + ps1;
              m0 = mn0;
              m1 = mn1;
            }
          } else {
            // normalised probabilities summed over this token's 16 heads, per window
            float cs[8][2];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
              cs[n][0] = cs[n][1] = 0.f;
              if (ok && active) {
                const float b0 = (m0 == -INFINITY) ? 0.f : m0, b1 = (m1 == -INFINITY) ? 0.f : m1;
                cs[n][0] = exp2f(sc[n][0] - b0) * inv0 + exp2f(sc[n][2] - b1) * inv1;
                cs[n][1] = exp2f(sc[n][1] - b0) * inv0 + exp2f(sc[n][3] - b1) * inv1;
              }
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                cs[n][e] += __shfl_xor_sync(0xffffffffu, cs[n][e], 4);
                cs[n][e] += __shfl_xor_sync(0xffffffffu, cs[n][e], 8);
                cs[n][e] += __shfl_xor_sync(0xffffffffu, cs[n][e], 16);
              }
            }
            float* pw = part + ((tile_no & 1) * kPaConsumerWarps + warp) * 64;
            if (lane < 4) {
#pragma unroll
              for (int n = 0; n < 8; ++n) {
                pw[8 * n + 2 * lane] = cs[n][0];
                pw[8 * n + 2 * lane + 1] = cs[n][1];
              }
            }
            consumers_sync();
            // the eight tokens' sums, added in warp order into the chunk's window sums
            if (tid < 64) {
              const float* pb = part + (tile_no & 1) * kPaConsumerWarps * 64;
              float acc = 0.f;
#pragma unroll
              for (int w = 0; w < kPaConsumerWarps; ++w) acc += pb[w * 64 + tid];
              const int i = m * 64 + tid;
              if (i < Wc) win_sum[i] += acc;
            }
            ++tile_no;
          }
        }
      }
    }
    consumers_sync();
    // max-pool onto blocks j <= c (windows 4j-1 .. 4j+3 below Wc), then the top-k
    float* S = a.block_scores + row * a.nb_cap;
    for (int j = tid; j <= c; j += kPaConsumerWarps * 32) {
      float v = -INFINITY;
      for (int i = max(0, 4 * j - 1); i <= min(Wc - 1, 4 * j + 3); ++i) v = fmaxf(v, win_sum[i]);
      S[j] = v;
    }
    __threadfence_block();
    consumers_sync();
    topk_select(S, a.idx + row * kslots, a.cnt + row, a.topk, a.max_ctx, c * kBlock + 1, sh);
  }
}

// ==================================================================== block-sparse attention, tcgen05
// Causal block-sparse prefill attention on the fifth-generation tensor cores. A CTA holds two
// query tiles of 128 rows (8 tokens x 16 heads each, row 16i + h), 16 tokens of one chunk,
// which share every K/V block it loads, and takes the chunk's selected blocks two at a time
// (a pair: 128 keys; an odd last block is paired with itself, its second copy masked):
//   warp 0, one thread: TMA loads of the two Q tiles (once) and of each pair's K and V into a
//       2-stage ring of full / empty mbarriers (a stage: K and V of both blocks, the second
//       block's rows after the first's, so that each pair is one 128-key operand);
//   warp 1: allocates the 512 tensor-memory columns (per tile 128 columns of S, which P
//       overwrites, and 128 of O) and, from one thread, issues per pair p and tile t
//       S_t,p = Q_t K_p^T (M 128, N 128, 8 K steps of 16) and O_t += P_t,p V_p (M 128, N 128,
//       8 K steps; P read from tensor memory, V M/N-major from shared memory), each completion
//       signalled by tcgen05.commit on an mbarrier; S_t,p+1 is issued right after
//       O_t += P_t,p V_p, whose read of P it must follow (one thread's tcgen05.mma run in issue
//       order), so the tensor cores work on one tile while the other tile's softmax runs;
//   warps 2-5 (tile 0) and 6-9 (tile 1), one thread per row (tensor-memory lane): the row
//       maximum of S_t,p over the keys the token may see (the chunk's own block is masked
//       after the token), an online softmax in the exp2 domain whose running maximum is only
//       moved (and O rescaled in tensor memory) when it grows by more than 2^8, then P_t,p as
//       bf16 pairs into the first 64 of S's columns (a second pass over S, block by block: P
//       never overwrites S that is still unread); at the end O / l.
// Every mbarrier phase a thread waits for can only be followed by the barrier's next phase
// after that thread itself has arrived somewhere (a parity wait tells phase k from phase k+2
// only if k+1 cannot have completed behind its back): s_full's next phase needs the issuer
// to have seen this warp's P, pv_done's next phase this warp's next P, and each warp waits
// pv_done's phases in order.
namespace {
// The softmax warps' waits: the library's bounded wait, or (SPARDA_TC_SPIN) a bounded loop of
// try_wait without the suspend-time hint.
__device__ __forceinline__ bool sm_wait(uint64_t* bar, uint32_t parity, int* err) {
#ifdef SPARDA_TC_SPIN
  for (uint32_t i = 0; i < (kWaitPolls << 4); ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  atomicOr(err, SPARDA_DEV_WAIT_TIMEOUT);
  return false;
#else
  return mbar_wait(bar, parity, err);
#endif
}

// 2^x by the PTX instruction ex2.approx.ftz.f32 (one MUFU operation; the PTX ISA bounds its
// relative error by 2^-22). Results below 2^-126 flush to zero, which the softmax cannot
// notice: the running maximum it subtracts is a logit it has already summed, so every row's
// sum is at least 1.
__device__ __forceinline__ float ex2_ftz(float x) {
#ifdef SPARDA_TC_LIBM_EXP2
  return exp2f(x);
#else
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
#endif
}

constexpr int kTcTiles = 2;
constexpr int kTcTokens = 8 * kTcTiles;                     // tokens per CTA
constexpr int kTcSlices = kBlock / kTcTokens;               // CTAs per chunk
constexpr int kTcStages = 2;                                // ring stages, one pair each
constexpr int kTcHalf = kBlockBytes / 2;                    // 64 rows x 64 dims of one block: 8 KiB
constexpr int kTcPart = 2 * kTcHalf;                        // the pair's 128 rows of one 64-dim half
constexpr int kTcStageBytes = 4 * kTcPart;                  // K lo, K hi, V lo, V hi: 64 KiB
constexpr int kTcQBytes = 128 * kRowBytes;                  // 32 KiB per tile: 128 rows x 128 dims
constexpr int kTcSmem = 1024 /*align*/ + 1024 /*barriers*/ + kTcTiles * kTcQBytes + kTcStages * kTcStageBytes;
static_assert(kTcSmem <= 227 * 1024, "the tcgen05 prefill attention fits shared memory");
constexpr int kTcThreads = (2 + 4 * kTcTiles) * 32;
constexpr uint32_t kTcCols = 512;
constexpr float kRescaleLog2 = 8.f;                         // move the running max past 2^8 growth
}  // namespace

__global__ void __launch_bounds__(kTcThreads, 1) prefill_attn_tc_kernel(const PrefillArgs a,
                                                                       const __grid_constant__ CUtensorMap mq,
                                                                       const __grid_constant__ CUtensorMap mk,
                                                                       const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* kv_full = q_full + 1;                           // [stages]
  uint64_t* kv_empty = kv_full + kTcStages;                 // [stages]
  uint64_t* s_full = kv_empty + kTcStages;                  // [tile]
  uint64_t* p_full = s_full + kTcTiles;                     // [tile]
  uint64_t* pv_done = p_full + kTcTiles;                    // [tile]
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(pv_done + kTcTiles);
  uint8_t* qs = smem + 1024;                                // [tile] 32 KiB
  uint8_t* ring = qs + kTcTiles * kTcQBytes;                // [stage] 64 KiB

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bg = blockIdx.y, b = bg / a.G, g = bg % a.G;
  const int c = blockIdx.x / kTcSlices, sl = blockIdx.x % kTcSlices;
  const int T = a.seq_len[b];
  if (!valid_len(T, a.max_ctx)) {
    if (tid == 0 && blockIdx.x == 0 && g == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int tok0 = c * kBlock + sl * kTcTokens;
  if (tok0 >= T) return;                                     // CTA-uniform
  const int kslots = a.topk + 2;
  const size_t row = (size_t)bg * a.nb_cap + c;
  const int n_sel = min(max(a.cnt[row], 0), kslots);
  const int n_pairs = (n_sel + 1) / 2;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&pv_done[t], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tc05::alloc(tmem_base_sh, kTcCols);
    tc05::relinquish();
  }
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = *tmem_base_sh;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      mbar_arrive_expect_tx(q_full, kTcTiles * kTcQBytes);
      const int qrow0 = (((b * a.max_ctx) + tok0) * a.G + g) * kHeads;
      const int tok_stride = a.G * kHeads;
      for (int i = 0; i < kTcTokens; ++i) {
        const int qr = qrow0 + i * tok_stride;
        uint8_t* qt = qs + (i >> 3) * kTcQBytes + (i & 7) * 16 * 128;
        tma_load_2d(qt, &mq, 0, qr, q_full);
        tma_load_2d(qt + kTcQBytes / 2, &mq, 64, qr, q_full);
      }
      for (int p = 0; p < n_pairs && ok; ++p) {
        const int stage = p % kTcStages;
        if (p >= kTcStages) ok = mbar_wait(&kv_empty[stage], ((p / kTcStages) & 1) ^ 1, a.err);
        if (!ok) break;
        uint8_t* dst = ring + stage * kTcStageBytes;
        mbar_arrive_expect_tx(&kv_full[stage], kTcStageBytes);
        for (int h = 0; h < 2; ++h) {
          const int s = min(2 * p + h, n_sel - 1);         // an odd last block is loaded twice
          int j = a.idx[row * kslots + s];
          if (j < 0 || j > c) {
            atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
            j = 0;
          }
          const int rr = bg * a.max_ctx + j * kBlock;
          tma_load_2d(dst + h * kTcHalf, &mk, 0, rr, &kv_full[stage]);
          tma_load_2d(dst + kTcPart + h * kTcHalf, &mk, 64, rr, &kv_full[stage]);
          tma_load_2d(dst + 2 * kTcPart + h * kTcHalf, &mv, 0, rr, &kv_full[stage]);
          tma_load_2d(dst + 3 * kTcPart + h * kTcHalf, &mv, 64, rr, &kv_full[stage]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every MMA in one fixed order: S_0,0 and S_1,0, then per pair p and
    // tile t (0, then 1) O_t += P_t,p V_p once the softmax has written
    // P_t,p, followed by S_t,p+1 once pair p+1 is in shared memory (after the O update that
    // read P_t,p from the same columns: one thread's MMAs run in issue order). Each wait
    // blocks on exactly the barrier it needs. A pair's ring stage is released once both
    // tiles' O += P V have read it.
    if (lane == 0) {
      constexpr uint32_t id_qk = tc05::idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t id_pv = tc05::idesc_bf16(128, 128, 0, 1);
      const uint32_t q_addr = smem_addr(qs), ring_addr = smem_addr(ring);
      auto issue_qk = [&](int t, int pq) {
        const uint32_t kb = ring_addr + (pq % kTcStages) * kTcStageBytes;
        const uint32_t qa = q_addr + t * kTcQBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32;
          const uint64_t da = tc05::smem_desc(qa + half * (kTcQBytes / 2) + off, 16, 1024);
          const uint64_t db = tc05::smem_desc(kb + half * kTcPart + off, 16, 1024);
          tc05::mma_bf16_ss(tmem + 256 * t, da, db, id_qk, kk > 0 ? 1u : 0u);
        }
        tc05::commit(&s_full[t]);
      };
      ok = mbar_wait(q_full, 0, a.err);
      if (ok && n_pairs > 0) ok = mbar_wait(&kv_full[0], 0, a.err);
      if (ok && n_pairs > 0) {
        tc05::fence_after();
        issue_qk(0, 0);
        issue_qk(1, 0);
      }
      for (int pp = 0; ok && pp < n_pairs; ++pp) {
#pragma unroll
        for (int t = 0; t < kTcTiles; ++t) {
          ok = mbar_wait(&p_full[t], pp & 1, a.err);
          if (!ok) break;
          tc05::fence_after();
          const uint32_t vb = ring_addr + (pp % kTcStages) * kTcStageBytes + 2 * kTcPart;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t db = tc05::smem_desc(vb + kk * 2048, kTcPart, 1024);
            tc05::mma_bf16_ts(tmem + 256 * t + 128, tmem + 256 * t + 8 * kk, db, id_pv,
                              (pp > 0 || kk > 0) ? 1u : 0u);
          }
          tc05::commit(&pv_done[t]);
          if (pp + 1 < n_pairs) {
            const int pq = pp + 1;
            ok = mbar_wait(&kv_full[pq % kTcStages], (pq / kTcStages) & 1, a.err);
            if (!ok) break;
            tc05::fence_after();
            issue_qk(t, pq);
          }
        }
        if (ok) tc05::commit(&kv_empty[pp % kTcStages]);   // both tiles' O += P V of pair pp
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int t = (warp - 2) >> 2;                           // query tile
    const int quarter = warp & 3;                            // tensor-memory lanes 32q .. 32q+31
    const int r = quarter * 32 + lane;                       // row: token r/16 of the tile, head r%16
    const int tok = tok0 + 8 * t + (r >> 4);
    const float sl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + 256 * t + lane_off;          // S, then P
    const uint32_t t_o = t_s + 128;
    // the chunk's block indices, lane i holding entries i and 32 + i (read before the loop: no
    // global load on the per-pair path)
    int jreg0 = lane < n_sel ? a.idx[row * kslots + lane] : 0;
    int jreg1 = lane + 32 < n_sel ? a.idx[row * kslots + lane + 32] : 0;
    float m_used = -INFINITY, l = 0.f;
    for (int p = 0; p < n_pairs; ++p) {
      // the pair's two blocks; -1: the second copy of an odd last block (every key masked)
      int jb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int s = 2 * p + h;
        const int j = __shfl_sync(0xffffffffu, s < 32 ? jreg0 : jreg1, s & 31);
        jb[h] = s >= n_sel ? -1 : ((j < 0 || j > c) ? 0 : j);
      }
      if (ok) ok = __all_sync(0xffffffffu, sm_wait(&s_full[t], p & 1, a.err));
      if (!ok) {
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&p_full[t]);
        continue;
      }
      tc05::fence_after();
      // One pass over S, block by block: the block's row maximum over the keys this token may
      // see (only the chunk's own block has keys after some of the tile's tokens), then its P
      // into columns 32h .. 32h+31, after the S columns 64h .. 64h+63 it comes from (and every
      // S column below) have been read. The running maximum moves only on the first block or
      // when it grows by more than 2^8; then O (which holds P_{p-1} V_{p-1} once pv_done's
      // phase p-1 is in) and, on the pair's second block, the first block's P are rescaled.
      bool pv_waited = (p == 0);
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = jb[h];
        uint32_t pk[32];
        if (j < 0) {                                           // warp-uniform
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = 0u;
        } else {
          float x[64];
          tc05::ld32(t_s + 64 * h, *reinterpret_cast<float(*)[32]>(x));
          tc05::ld32(t_s + 64 * h + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          tc05::wait_ld();
          if (j == c) {
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = (j * kBlock + e <= tok) ? x[e] : -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
          for (int e = 8; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], x[e]);
          const float mb = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
          const bool first = (m_used == -INFINITY);
          const bool grow = first || mb > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, grow)) {
            const float mn = grow ? (first ? mb : fmaxf(m_used, mb)) : m_used;
            const float alpha = first ? 0.f : ex2_ftz(m_used - mn);
            if (!pv_waited) {
              // O += P_{p-1} V_{p-1} is complete (S_p was issued after it): take the phase
              ok = __all_sync(0xffffffffu, sm_wait(&pv_done[t], (p - 1) & 1, a.err)) && ok;
              pv_waited = true;
              tc05::fence_after();
            }
            if (p > 0) {                                       // O holds earlier pairs
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                float o[32];
                tc05::ld32(t_o + 32 * q4, o);
                tc05::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= alpha;
                tc05::st32(t_o + 32 * q4, o);
              }
            }
            if (h == 1 && jb[0] >= 0) {                        // the first block's P, written
              float pa[32];
              tc05::wait_st();                                 // (its store is complete)
              tc05::ld32(t_s, pa);
              tc05::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const uint32_t u = __float_as_uint(pa[e]);
                pa[e] = __uint_as_float(pack_bf16(__uint_as_float(u << 16) * alpha,
                                                  __uint_as_float(u & 0xffff0000u) * alpha));
              }
              tc05::st32(t_s, pa);
            }
            tc05::wait_st();
#pragma unroll
            for (int e = 0; e < 8; ++e) ps[e] *= alpha;
            l *= alpha;
            m_used = mn;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float p0 = ex2_ftz(fmaf(x[2 * e], sl2, -m_used)), p1 = ex2_ftz(fmaf(x[2 * e + 1], sl2, -m_used));
            ps[e & 7] += p0 + p1;
            pk[e] = pack_bf16(p0, p1);
          }
        }
        tc05::st32(t_s + 32 * h, *reinterpret_cast<const float(*)[32]>(pk));
      }
      tc05::wait_st();
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      // pv_done's phase p-1 in turn (long complete) before this warp's P_p can complete phase p
      if (!pv_waited) ok = __all_sync(0xffffffffu, sm_wait(&pv_done[t], (p - 1) & 1, a.err)) && ok;
      tc05::fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&p_full[t]);
    }
    // ---- epilogue: O / l of this row (token tok, head r % 16), once the last O += P V is done
    // (its phase n_pairs-1 is the barrier's last; n_pairs-2 was waited for at the last pair)
    if (ok && n_pairs > 0) ok = __all_sync(0xffffffffu, sm_wait(&pv_done[t], (n_pairs - 1) & 1, a.err));
    if (ok && n_pairs > 0) {
      tc05::fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.out + ((((size_t)b * a.max_ctx + tok) * a.G + g) * kHeads + (r & 15)) * kHeadDim);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float o[32];
        __syncwarp();                                          // tcgen05.ld is warp-aligned
        tc05::ld32(t_o + 32 * q4, o);
        tc05::wait_ld();
        if (tok < T) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[4 * q4 + e] = make_uint4(pack_bf16(o[8 * e] * inv, o[8 * e + 1] * inv),
                                         pack_bf16(o[8 * e + 2] * inv, o[8 * e + 3] * inv),
                                         pack_bf16(o[8 * e + 4] * inv, o[8 * e + 5] * inv),
                                         pack_bf16(o[8 * e + 6] * inv, o[8 * e + 7] * inv));
        }
      }
    }
  }
  // every tensor-memory access of this CTA is done before the allocating warp frees it
  tc05::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::dealloc(tmem, kTcCols);
  }
}

// ==================================================================== launches
void launch_prefill_forecast_select(const PrefillArgs& a, int batch, cudaStream_t s) {
  const int n_ct = (a.nb_cap + kPfChunks - 1) / kPfChunks;
  prefill_forecast_score_kernel<<<dim3(n_ct, batch * a.G), kPfThreads, 0, s>>>(a);
  prefill_topk_kernel<<<dim3(a.nb_cap, batch * a.G), kTopkThreads, 0, s>>>(a);
}

void launch_prefill_multihead_select(const PrefillArgs& a, const CUtensorMap& mck, int batch, cudaStream_t s) {
  const int smem = mh_smem_bytes(a.W_cap);
  cudaFuncSetAttribute(prefill_multihead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  prefill_multihead_kernel<<<dim3(a.nb_cap, batch * a.G), kPaThreads, smem, s>>>(a, mck);
}


void launch_prefill_attn_tc(const PrefillArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, int batch, cudaStream_t s) {
  cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  prefill_attn_tc_kernel<<<dim3(a.nb_cap * kTcSlices, batch * a.G), kTcThreads, kTcSmem, s>>>(a, mq, mk, mv);
}

}  // namespace sparda

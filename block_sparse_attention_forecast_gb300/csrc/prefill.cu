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
// The softmax warps' waits: the library's bounded wait (try_wait with a suspend-time hint; a
// polling loop of test_wait measured slower, its thread taking issue slots from the softmax).
__device__ __forceinline__ bool sm_wait(uint64_t* bar, uint32_t parity, int* err) {
  return mbar_wait(bar, parity, err);
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 2^x by the PTX instruction ex2.approx.ftz.f32 (one MUFU operation; the PTX ISA bounds its
// relative error by 2^-22). Results below 2^-126 flush to zero, which the softmax cannot
// notice: the running maximum it subtracts is a logit it has already summed, so every row's
// sum is at least 1.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// ==================================================================== baseline multi-head, tcgen05
// The baseline chunk selector on the fifth-generation tensor cores. One CTA per (sequence-
// group, chunk), the longest chunks first. The chunk's 1024 query rows (64 tokens x 16 heads)
// are taken two 128-row tiles at a time (a tile: 8 tokens, row 16i + h; an odd last tile is
// paired with a tile of rows past the prompt, which count for nothing). For each pair, two
// passes over the chunk's windows, 128 at a time:
//   warp 0, one thread: TMA loads of the pair's Q tiles (once per pair, after the pair before
//       has been read) and of each 128-window tile of compressed keys into a ring;
//   warp 1: allocates 512 tensor-memory columns (per tile an S double buffer of 2 x 128) and,
//       from one thread, issues per window tile and query tile S = Q CK^T (M 128, N 128, 8 K
//       steps), each completion signalled by tcgen05.commit;
//   warps 2-9, one thread per row: pass 1 keeps the row's running maximum and sum of
//       2^(s - max) over the windows (logits scaled by log2(e)/sqrt(d)); pass 2 forms
//       p = 2^(s - max) / sum and sums it over the rows: within a warp by a butterfly that
//       leaves lane l the sums of windows 2l, 2l+1 of each 64, then over the eight warps in a
//       fixed order into the chunk's window sums in shared memory.
// Then the max-pool onto blocks and the exact top-k, as in the Forecast selector. Every wait
// is bounded; each parity wait can only be followed by the barrier's next phase after the
// waiting thread has itself arrived somewhere.
namespace {
constexpr int kMtTiles = 2;
constexpr int kMtWin = 128;                                 // windows per S tile
constexpr int kMtCkBytes = kMtWin * kRowBytes;              // 32 KiB
constexpr int kMtQBytes = 128 * kRowBytes;                  // 32 KiB per query tile
constexpr int kMtThreads = (2 + 4 * kMtTiles) * 32;         // 320
constexpr int kMtPartFloats = 2 * 4 * kMtTiles * kMtWin;    // [2 buffers][8 warps][128 windows]
constexpr uint32_t kMtCols = 512;
static_assert((int)sizeof(TopkShared) <= kMtTiles * kMtQBytes, "the top-k scratch fits over the query tiles");
// [align slack][barriers][Q tiles][ring][column sums][window sums]
__host__ __device__ constexpr int mt_smem_bytes(int w_cap, int stages) {
  return 1024 + 1024 + kMtTiles * kMtQBytes + stages * kMtCkBytes + kMtPartFloats * 4 + (4 * w_cap + 15) / 16 * 16;
}
__host__ __device__ constexpr int mt_stages(int w_cap) { return mt_smem_bytes(w_cap, 3) <= 227 * 1024 ? 3 : 2; }
static_assert(mt_smem_bytes(kMaxCtx / kWinStride, 2) <= 227 * 1024, "the baseline prefill selector fits shared memory");

// Sum of v over the 32 lanes, per index: lane l gets the sums of entries 2l and 2l+1 (a
// transposing butterfly: each step a lane keeps one half of its entries, adds the partner's
// copy of that half, and hands the other half over).
__device__ __forceinline__ void lane_colsum64(float (&v)[64], int lane, float& s0, float& s1) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool up = lane & 16;
    const float give = up ? v[i] : v[i + 32];
    const float keep = up ? v[i + 32] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool up = lane & 8;
    const float give = up ? v[i] : v[i + 16];
    const float keep = up ? v[i + 16] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 4;
    const float give = up ? v[i] : v[i + 8];
    const float keep = up ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 2;
    const float give = up ? v[i] : v[i + 4];
    const float keep = up ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 1;
    const float give = up ? v[i] : v[i + 2];
    const float keep = up ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 1);
  }
  s0 = v[0];
  s1 = v[1];
}

__device__ __forceinline__ void mt_softmax_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(4 * kMtTiles * 32) : "memory");
}
}  // namespace

__global__ void __launch_bounds__(kMtThreads, 1) prefill_multihead_tc_kernel(const PrefillArgs a, int n_st,
                                                                            const __grid_constant__ CUtensorMap mq,
                                                                            const __grid_constant__ CUtensorMap mck) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* q_free = q_full + 1;
  uint64_t* kv_full = q_free + 1;                           // [stages]
  uint64_t* kv_empty = kv_full + 3;                         // [stages]
  uint64_t* s_full = kv_empty + 3;                          // [tile][2]
  uint64_t* s_free = s_full + 2 * kMtTiles;                 // [tile][2]
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(s_free + 2 * kMtTiles);
  uint8_t* qs = smem + 1024;                                // [tile] 32 KiB
  uint8_t* ring = qs + kMtTiles * kMtQBytes;                // [stage] 32 KiB
  float* part = reinterpret_cast<float*>(ring + n_st * kMtCkBytes);   // [2][8 warps][128]
  float* win_sum = part + kMtPartFloats;                    // [W_cap]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bg = blockIdx.y, b = bg / a.G, g = bg % a.G;
  const int c = a.nb_cap - 1 - (int)blockIdx.x;               // the longest chunks first
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
  const int n_wt = (Wc + kMtWin - 1) / kMtWin;
  const int n_tok = min(kBlock, T - c * kBlock);
  const int n_rp = (n_tok + 8 * kMtTiles - 1) / (8 * kMtTiles);  // pairs of 8-token tiles
  const int n_steps = 2 * n_wt;                                   // per pair: two passes

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int i = 0; i < n_st; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2 * kMtTiles; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < Wc; i += blockDim.x) win_sum[i] = 0.f;
  if (warp == 1) {
    tc05::alloc(tmem_base_sh, kMtCols);
    tc05::relinquish();
  }
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = *tmem_base_sh;
  bool ok = true;

  if (n_wt > 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mck);
      int gs = 0;
      for (int rp = 0; rp < n_rp && ok; ++rp) {
        if (rp > 0) ok = mbar_wait(q_free, (rp - 1) & 1, a.err);    // the pair before has been read
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, kMtTiles * kMtQBytes);
        for (int i = 0; i < 8 * kMtTiles; ++i) {
          const int tok = c * kBlock + 8 * kMtTiles * rp + i;          // < max_ctx: a row past T counts for nothing
          const int qr = (((b * a.max_ctx) + tok) * a.G + g) * kHeads;
          uint8_t* qt = qs + (i >> 3) * kMtQBytes + (i & 7) * 16 * 128;
          tma_load_2d(qt, &mq, 0, qr, q_full);
          tma_load_2d(qt + kMtQBytes / 2, &mq, 64, qr, q_full);
        }
        for (int s = 0; s < n_steps && ok; ++s, ++gs) {
          const int stage = gs % n_st;
          if (gs >= n_st) ok = mbar_wait(&kv_empty[stage], ((gs / n_st) & 1) ^ 1, a.err);
          if (!ok) break;
          const int rr = bg * a.W_cap + (s % n_wt) * kMtWin;
          uint8_t* dst = ring + stage * kMtCkBytes;
          mbar_arrive_expect_tx(&kv_full[stage], kMtCkBytes);
          tma_load_2d(dst, &mck, 0, rr, &kv_full[stage]);
          tma_load_2d(dst + kMtCkBytes / 4, &mck, 0, rr + 64, &kv_full[stage]);
          tma_load_2d(dst + kMtCkBytes / 2, &mck, 64, rr, &kv_full[stage]);
          tma_load_2d(dst + 3 * kMtCkBytes / 4, &mck, 64, rr + 64, &kv_full[stage]);
        }
      }
    }
  } else if (n_wt > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = tc05::idesc_bf16(128, kMtWin, 0, 0);
      const uint32_t q_addr = smem_addr(qs), ring_addr = smem_addr(ring);
      int gs = 0;
      for (int rp = 0; rp < n_rp && ok; ++rp) {
        ok = mbar_wait(q_full, rp & 1, a.err);
        for (int s = 0; s < n_steps && ok; ++s, ++gs) {
          const int stage = gs % n_st;
          ok = mbar_wait(&kv_full[stage], (gs / n_st) & 1, a.err);
          for (int t = 0; t < kMtTiles && ok; ++t) {
            const int sb = 2 * t + (gs & 1);
            if (gs >= 2) ok = mbar_wait(&s_free[sb], ((gs >> 1) - 1) & 1, a.err);   // read two steps ago
            if (!ok) break;
            tc05::fence_after();
            const uint32_t kb = ring_addr + stage * kMtCkBytes;
            const uint32_t qa = q_addr + t * kMtQBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32;
              const uint64_t da = tc05::smem_desc(qa + half * (kMtQBytes / 2) + off, 16, 1024);
              const uint64_t db = tc05::smem_desc(kb + half * (kMtCkBytes / 2) + off, 16, 1024);
              tc05::mma_bf16_ss(tmem + 256 * t + 128 * (gs & 1), da, db, id_qk, kk > 0 ? 1u : 0u);
            }
            tc05::commit(&s_full[sb]);
          }
          if (ok) tc05::commit(&kv_empty[stage]);                  // both tiles' S read the stage
        }
        if (ok) tc05::commit(q_free);                              // every S of the pair read Q
      }
    }
  } else if (n_wt > 0 && warp >= 2) {
    // ------------------------------------------------------------ softmax, one row per thread
    const int t = (warp - 2) >> 2;                           // query tile
    const int quarter = warp & 3;                            // tensor-memory lanes 32q .. 32q+31
    const int r = quarter * 32 + lane;                       // row: token r/16 of the tile, head r%16
    const int wi = warp - 2;                                 // this warp's slot in the column sums
    const float zl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int st = tid - 64;                                 // 0 .. 255 over the softmax warps
    int gs = 0;
    for (int rp = 0; rp < n_rp; ++rp) {
      const int tok = c * kBlock + 8 * kMtTiles * rp + 8 * t + (r >> 4);
      const bool live = tok < T;
      float M = -INFINITY, L = 0.f, invL = 0.f;
      for (int s = 0; s < n_steps; ++s, ++gs) {
        const bool pass2 = s >= n_wt;
        const int m = s - (pass2 ? n_wt : 0);
        const int nvalid = min(kMtWin, Wc - m * kMtWin);     // windows of this tile below Wc
        const int sb = 2 * t + (gs & 1);
        if (ok) ok = __all_sync(0xffffffffu, sm_wait(&s_full[sb], (gs >> 1) & 1, a.err));
        if (ok) tc05::fence_after();
        float* pw = part + ((gs & 1) * 4 * kMtTiles + wi) * kMtWin;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[64];
          if (ok) {
            const uint32_t ta = tmem + 256 * t + 128 * (gs & 1) + 64 * h + lane_off;
            tc05::ld32(ta, *reinterpret_cast<float(*)[32]>(x));
            tc05::ld32(ta + 32, *reinterpret_cast<float(*)[32]>(x + 32));
            tc05::wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = 0.f;
          }
          if (64 * (h + 1) > nvalid) {                       // warp-uniform: windows past Wc
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = (64 * h + e < nvalid) ? x[e] : -INFINITY;
          }
          if (!pass2) {
            float m8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
            for (int e = 8; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], x[e]);
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * zl2;
            const float mn = fmaxf(M, mx);
            if (mn != -INFINITY) {
              float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int e = 0; e < 64; ++e) ps[e & 7] += ex2_ftz(fmaf(x[e], zl2, -mn));
              L = L * ex2_ftz(M - mn) + (((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7])));
              M = mn;
            }
          } else {
            // p = 2^(s - max) / sum, 0 for rows past the prompt and windows past Wc
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = live ? ex2_ftz(fmaf(x[e], zl2, -M)) * invL : 0.f;
            float s0, s1;
            lane_colsum64(x, lane, s0, s1);
            *reinterpret_cast<float2*>(pw + 64 * h + 2 * lane) = make_float2(s0, s1);
          }
        }
        tc05::fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&s_free[sb]);
        if (s == n_wt - 1) invL = L > 0.f ? 1.f / L : 0.f;
        if (pass2) {
          // the eight warps' sums of this window tile, added in warp order
          mt_softmax_sync();
          if (st < kMtWin) {
            const float* pb = part + (gs & 1) * 4 * kMtTiles * kMtWin;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 4 * kMtTiles; ++w) acc += pb[w * kMtWin + st];
            if (st < nvalid) win_sum[m * kMtWin + st] += acc;
          }
        }
      }
    }
  }
  // ---- every thread: the window sums are complete once every role has left its loop
  tc05::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after();
    tc05::dealloc(tmem, kMtCols);
  }
  if (warp < 8) {
    // max-pool onto blocks j <= c (windows 4j-1 .. 4j+3 below Wc), then the top-k (threads
    // 0 .. 255; its scratch over the query tiles, free now)
    float* S = a.block_scores + row * a.nb_cap;
    for (int j = tid; j <= c; j += 256) {
      float v = -INFINITY;
      for (int i = max(0, 4 * j - 1); i <= min(Wc - 1, 4 * j + 3); ++i) v = fmaxf(v, win_sum[i]);
      S[j] = v;
    }
    __threadfence_block();
    topk_sync();
    TopkShared& sh = *reinterpret_cast<TopkShared*>(qs);
    topk_select(S, a.idx + row * kslots, a.cnt + row, a.topk, a.max_ctx, c * kBlock + 1, sh);
  }
}

// ==================================================================== launches
void launch_prefill_forecast_select(const PrefillArgs& a, int batch, cudaStream_t s) {
  const int n_ct = (a.nb_cap + kPfChunks - 1) / kPfChunks;
  prefill_forecast_score_kernel<<<dim3(n_ct, batch * a.G), kPfThreads, 0, s>>>(a);
  prefill_topk_kernel<<<dim3(a.nb_cap, batch * a.G), kTopkThreads, 0, s>>>(a);
}

void launch_prefill_multihead_select(const PrefillArgs& a, const CUtensorMap& mq, const CUtensorMap& mck, int batch,
                                     cudaStream_t s) {
  const int n_st = mt_stages(a.W_cap);
  const int smem = mt_smem_bytes(a.W_cap, n_st);
  cudaFuncSetAttribute(prefill_multihead_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  prefill_multihead_tc_kernel<<<dim3(a.nb_cap, batch * a.G), kMtThreads, smem, s>>>(a, n_st, mq, mck);
}


void launch_prefill_attn_tc(const PrefillArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, int batch, cudaStream_t s) {
  cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  prefill_attn_tc_kernel<<<dim3(a.nb_cap * kTcSlices, batch * a.G), kTcThreads, kTcSmem, s>>>(a, mq, mk, mv);
}

}  // namespace sparda

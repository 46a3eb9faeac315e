// Exact top-k block selection shared by the Forecast selector and the baseline multi-head
// selector: keep block 0, the tail block and the topk highest-scoring other blocks, ties to
// the lower block index; output sorted ascending and padded with -1.
#pragma once

#include "common.cuh"

namespace sparda {

constexpr int kTopkWarps = 8;
constexpr int kTopkThreads = kTopkWarps * 32;                      // 256
constexpr int kMaxBlocksPerSeq = kMaxCtx / kBlock;                 // 4096
constexpr int kKeysPerThread = kMaxBlocksPerSeq / kTopkThreads;    // 16

__device__ __forceinline__ void topk_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kTopkThreads) : "memory");
}

// Inclusive prefix sum over the 256 consumer threads; `warp_tot` is 8 words of shared
// memory. *total gets the sum over all consumers.
__device__ __forceinline__ int topk_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  topk_sync();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    const int x = warp_tot[w];
    if (w < warp) before += x;
    all += x;
  }
  topk_sync();
  *total = all;
  return v + before;
}

constexpr int kMaxList = 512;          // candidates ranked exactly by the fast path
static_assert(kMaxTopk <= 64, "the chosen blocks fit TopkShared::sel");

// Order-preserving 32-bit key of a block score, with -0 keyed as +0 so that equal scores get
// equal keys (ties then go to the lower block, as for any other equal pair). Every NaN, of
// either sign and any payload, is keyed as the largest key, above +inf: all NaNs rank alike,
// above every number, and none can take key 0, the key of a non-candidate. Every other
// score's key lies strictly between.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  else if ((u & 0x7fffffffu) > 0x7f800000u) u = 0x7fffffffu;
  return ordered_key(__uint_as_float(u));
}

struct TopkShared {
  unsigned hist[256];
  int warp_tot[kTopkWarps];
  uint32_t warp_th[kTopkWarps];
  int warp_bad[kTopkWarps];
  uint32_t prefix;
  int krem;
  int last;
  uint64_t lp[kMaxList];               // listed candidates: score key << 32 | ~block
  int sel[64];                         // the chosen blocks, by rank
  unsigned char flag[kMaxBlocksPerSeq];
};

// Top-k of one (sequence, group) by 256 threads (threads 0-255 of the CTA, synchronised with
// named barrier 1), from the block scores S[0 .. nb) in global memory. Writes idx[0 .. topk+2)
// (block 0, the chosen blocks ascending, the tail block; -1 padded) and *cnt_out.
//
// Thread t holds the scores of blocks t, t + 256, t + 512, ... (each warp load is one
// contiguous 128-byte line). Fast path, four barriers in all:
//   * a threshold that at least k candidates reach: each warp takes the q-th largest of its
//     32 lane maxima (q = ceil(k / 8)) by q warp-wide max reductions of order-preserving keys,
//     and the threshold is the smallest of the 8 warps' values. Every warp holds at least q
//     candidates at or above its own value, so at least 8q >= k reach the threshold, and every
//     candidate of the top k is among them (a warp with fewer than q candidate lanes lowers the
//     threshold to take every candidate);
//   * those candidates -- a few dozen for real score distributions -- listed in shared memory
//     by ballots and per-warp counts;
//   * their exact ranks (score descending, block ascending) by comparing each candidate's
//     packed key (score key above, inverted block index below: one 64-bit order) with every
//     other, one thread per candidate over broadcast loads; each chosen block written at its
//     rank, and then placed by counting the chosen blocks below it.
// If more than kMaxList candidates reach the threshold (near-constant scores), or a candidate
// score is not finite, a 4-pass radix select on order-preserving 32-bit keys takes over and
// the output is assembled from per-block flags. Either way the result is exact and ties go to
// the lower block index.
template <int KPT>
static __device__ void topk_select_impl(const float* S, int32_t* idx, int32_t* cnt_out, int topk, int max_ctx,
                                        int T, TopkShared& sh) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // The loads of the whole score row (max_ctx / 64 entries: each stays inside it) do not wait
  // for T, so they share one memory round trip with the caller's read of the sequence length.
  const int nb_row = max_ctx / kBlock;
  float v[KPT];
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const int j = e * kTopkThreads + t;
    v[e] = j < nb_row ? __ldcg(S + j) : 0.f;
  }
  const int kslots = topk + 2;
  const bool valid = (T >= 1 && T <= max_ctx);
  const int tb = valid ? (T - 1) / kBlock : -1;
  const int nb = tb + 1;
  const int n_cand = max(0, tb - 1);
  const int k_eff = min(topk, n_cand);
  bool isc[KPT];
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const int j = e * kTopkThreads + t;
    isc[e] = j >= 1 && j < tb;
    if (!isc[e]) v[e] = 0.f;
  }

  if (k_eff > 0 && k_eff < n_cand) {
    // keys of the candidates, 0 for the others
    uint32_t key[KPT];
    uint32_t lane_max = 0u;
    bool bad = false;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      key[e] = 0u;
      if (isc[e]) {
        bad |= !isfinite(v[e]);
        key[e] = score_key(v[e]);
        lane_max = max(lane_max, key[e]);
      }
    }
    // the q-th largest lane maximum of this warp, the lanes counted with multiplicity
    const int quota = (k_eff + kTopkWarps - 1) / kTopkWarps;
    uint32_t th = 1u, cur = lane_max;
    int got = 0;
    for (int r = 0; r < quota; ++r) {             // warp-uniform: m and got are
      const uint32_t m = __reduce_max_sync(0xffffffffu, cur);
      if (m == 0u) {                              // fewer than quota candidate lanes: all
        th = 1u;
        break;
      }
      got += __popc(__ballot_sync(0xffffffffu, cur == m));
      th = m;
      if (got >= quota) break;
      if (cur == m) cur = 0u;
    }
    const bool warp_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      sh.warp_th[warp] = th;
      sh.warp_bad[warp] = warp_bad ? 1 : 0;
    }
    topk_sync();
    uint32_t theta = 0xffffffffu;
    bool any_bad = false;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      theta = min(theta, sh.warp_th[w]);
      any_bad |= sh.warp_bad[w] != 0;
    }
    // list the candidates at or above the threshold, in (warp, e, lane) order: one ballot per
    // register slot, per-warp totals exchanged once
    unsigned bal[KPT];
    int wcount = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      bal[e] = __ballot_sync(0xffffffffu, key[e] >= theta);
      wcount += __popc(bal[e]);
    }
    if (lane == 0) sh.warp_tot[warp] = wcount;
    topk_sync();
    int p = 0, c = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      const int x = sh.warp_tot[w];
      if (w < warp) p += x;
      c += x;
    }
    if (!any_bad && c <= kMaxList) {                // CTA-uniform
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        if (key[e] >= theta) {
          const uint32_t j = (uint32_t)(e * kTopkThreads + t);
          sh.lp[p + __popc(bal[e] & below)] = ((uint64_t)key[e] << 32) | (uint64_t)(~j);
        }
        p += __popc(bal[e]);
      }
      topk_sync();
      // exact rank of each listed candidate: the number of listed packed keys above its own
      for (int i = t; i < c; i += kTopkThreads) {
        const uint64_t mine = sh.lp[i];
        int rank = 0;
#pragma unroll 8
        for (int m = 0; m < c; ++m) rank += sh.lp[m] > mine ? 1 : 0;
        if (rank < k_eff) sh.sel[rank] = (int)~(uint32_t)mine;
      }
      topk_sync();
      // output: block 0, the chosen blocks in ascending order, the tail block (tb >= 2 here)
      if (t < k_eff) {
        const int ji = sh.sel[t];
        int pos = 0;
#pragma unroll 8
        for (int m = 0; m < k_eff; ++m) pos += sh.sel[m] < ji ? 1 : 0;
        idx[1 + pos] = ji;
      }
      if (t == 0) {
        idx[0] = 0;
        idx[k_eff + 1] = tb;
        *cnt_out = k_eff + 2;
      }
      for (int s = k_eff + 2 + t; s < kslots; s += kTopkThreads) idx[s] = -1;
      return;
    }
  }
  // -------------------------------------------------------------- flag-based paths
  // every candidate chosen (k_eff == n_cand), or the radix select for near-constant scores
  for (int j = t; j < nb; j += kTopkThreads) sh.flag[j] = (j == 0 || j == tb) ? 1 : 0;   // forced blocks
  topk_sync();
  if (k_eff == n_cand) {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (isc[e]) sh.flag[e * kTopkThreads + t] = 1;
  } else if (k_eff > 0) {
    uint32_t key[KPT];
#pragma unroll
    for (int e = 0; e < KPT; ++e) key[e] = isc[e] ? score_key(v[e]) : 0u;
    uint32_t prefix = 0u, mask = 0u;
    int krem = k_eff;
    for (int shift = 24; shift >= 0; shift -= 8) {
      sh.hist[t] = 0u;
      topk_sync();
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        const bool in = key[e] != 0u && (key[e] & mask) == prefix;
        if (in) atomicAdd(&sh.hist[(key[e] >> shift) & 255u], 1u);
      }
      topk_sync();
      const int hv = (int)sh.hist[255 - t];
      int tot;
      const int incl = topk_scan(hv, sh.warp_tot, &tot);
      if (incl - hv < krem && incl >= krem) {
        sh.prefix = prefix | ((uint32_t)(255 - t) << shift);
        sh.krem = krem - (incl - hv);
      }
      topk_sync();
      prefix = sh.prefix;
      krem = sh.krem;
      mask |= 255u << shift;
    }
    // keys above the k-th key are chosen; of the keys equal to it, the krem of lowest block
    // index. Thread t's equal keys sit at blocks t, t + 256, ...: count, per e, the equal keys
    // of all threads at earlier e or, at the same e, lower t.
    int eq_before = 0;                    // equal keys at blocks below this thread's current one
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const bool eq = key[e] != 0u && key[e] == prefix;
      int tot_e;
      const int incl_e = topk_scan(eq ? 1 : 0, sh.warp_tot, &tot_e);
      if (key[e] != 0u && key[e] > prefix) sh.flag[e * kTopkThreads + t] = 1;
      if (eq && eq_before + incl_e - 1 < krem) sh.flag[e * kTopkThreads + t] = 1;
      eq_before += tot_e;
    }
  }
  topk_sync();
  // the selected blocks in ascending order: thread t scans the contiguous range of blocks
  // [t*per, t*per + per)
  const int per = (nb + kTopkThreads - 1) / kTopkThreads;
  const int jb = t * per;
  int my_sel = 0;
  for (int e = 0; e < per; ++e)
    if (jb + e < nb) my_sel += sh.flag[jb + e];
  int total;
  int pos = topk_scan(my_sel, sh.warp_tot, &total) - my_sel;
  for (int e = 0; e < per; ++e)
    if (jb + e < nb && sh.flag[jb + e] && pos < kslots) idx[pos++] = jb + e;
  for (int s = total + t; s < kslots; s += kTopkThreads) idx[s] = -1;
  if (t == 0) *cnt_out = min(total, kslots);
}


// Thread t holds the scores of blocks t, t + 256, ...: 8 of them up to 2048 blocks (128K
// tokens), 16 beyond. The two instantiations run the same steps; the smaller one does half
// the register work in every phase.
static __device__ void topk_select(const float* S, int32_t* idx, int32_t* cnt_out, int topk, int max_ctx,
                                   int T, TopkShared& sh) {
  if (max_ctx / kBlock <= 8 * kTopkThreads)
    topk_select_impl<8>(S, idx, cnt_out, topk, max_ctx, T, sh);
  else
    topk_select_impl<kKeysPerThread>(S, idx, cnt_out, topk, max_ctx, T, sh);
}

}  // namespace sparda

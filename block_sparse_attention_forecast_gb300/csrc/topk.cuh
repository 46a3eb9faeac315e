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

struct TopkShared {
  unsigned hist[256];
  int warp_tot[kTopkWarps];
  float red_lo[kTopkWarps], red_hi[kTopkWarps];
  uint32_t prefix;
  int krem;
  int last;
  int bstar;
  int n_ge;
  float lv[kMaxList];
  int lj[kMaxList];
  int lr[kMaxList];                    // exact rank of each listed candidate
  unsigned char flag[kMaxBlocksPerSeq];
};

// Bucket of a candidate score in the 256 equal slices of [lo, hi]: floor((x - lo) * scale),
// taken as the low mantissa bits of 2^23 + that product added with rounding down (an FP32
// add instead of a float-to-int conversion). Monotone non-decreasing in x (a subtraction, a
// positive scaling and a rounded-down add, each monotone), so every candidate in a higher
// bucket outscores every candidate in a lower one.
__device__ __forceinline__ int score_bucket(float x, float lo, float scale) {
  const float y = __fadd_rd(fmaxf((x - lo) * scale, 0.f), 8388608.f);
  return min(255, __float_as_int(y) & 0x7fffff);
}

// Top-k of one (sequence, group) by 256 threads (threads 0-255 of the CTA, synchronised with
// named barrier 1), from the block scores S[0 .. nb) in global memory. Writes idx[0 .. topk+2)
// (block 0, the chosen blocks ascending, the tail block; -1 padded) and *cnt_out.
//
// Thread t holds the scores of blocks t, t + 256, t + 512, ... (each warp load is one
// contiguous 128-byte line). Fast path: min/max of the candidate scores; a 256-bucket
// histogram over that range (shared-memory atomics); the bucket that holds the k-th score,
// found by a scan from the top; the candidates at or above that bucket -- a few dozen for real
// score distributions -- listed in shared memory by ballots and per-warp counts; their exact ranks
// (score descending, block ascending) by pairwise comparison; and the output position of each
// chosen block by counting the chosen blocks below it. If more than kMaxList candidates share
// those buckets (near-constant scores), a 4-pass radix select on order-preserving 32-bit keys
// takes over and the output is assembled from per-block flags. Either way the result is exact
// and ties go to the lower block index.
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
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (isc[e]) {
        lo = fminf(lo, v[e]);
        hi = fmaxf(hi, v[e]);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      sh.red_lo[warp] = lo;
      sh.red_hi[warp] = hi;
    }
    sh.hist[t] = 0u;
    topk_sync();
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      lo = fminf(lo, sh.red_lo[w]);
      hi = fmaxf(hi, sh.red_hi[w]);
    }
    const float scale = 256.f / (hi - lo);
    bool fast = hi > lo && isfinite(lo) && isfinite(hi) && isfinite(scale);   // CTA-uniform
    int bk[KPT];
    if (fast) {
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        bk[e] = isc[e] ? score_bucket(v[e], lo, scale) : -1;
        if (isc[e]) atomicAdd(&sh.hist[bk[e]], 1u);
      }
      topk_sync();
      const int hv = (int)sh.hist[255 - t];      // thread t looks at bucket 255 - t
      int tot;
      const int incl = topk_scan(hv, sh.warp_tot, &tot);
      if (incl - hv < k_eff && incl >= k_eff) {
        sh.bstar = 255 - t;
        sh.n_ge = incl;
      }
      topk_sync();
      fast = sh.n_ge <= kMaxList;
    }
    if (fast) {
      const int bstar = sh.bstar;
      // list the candidates at or above bucket bstar, in (warp, e, lane) order: one ballot
      // per register slot, per-warp totals exchanged once
      unsigned bal[KPT];
      int wcount = 0;
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        bal[e] = __ballot_sync(0xffffffffu, bk[e] >= bstar);
        wcount += __popc(bal[e]);
      }
      if (lane == 0) sh.warp_tot[warp] = wcount;
      topk_sync();
      int p = 0;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w)
        if (w < warp) p += sh.warp_tot[w];
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int e = 0; e < KPT; ++e) {
        if (bk[e] >= bstar) {
          const int q = p + __popc(bal[e] & below);
          sh.lv[q] = v[e];
          sh.lj[q] = e * kTopkThreads + t;
        }
        p += __popc(bal[e]);
      }
      topk_sync();
      // exact rank of each listed candidate: `split` threads share one candidate, each
      // scanning a slice of the list
      const int c = sh.n_ge;
      const int split = c <= 32 ? 8 : (c <= 64 ? 4 : (c <= 128 ? 2 : 1));
      for (int i0 = 0; i0 < c * split; i0 += kTopkThreads) {
        const int q = i0 + t;
        const int i = q / split, part = q % split;
        int rank = 0;
        if (i < c) {
          const float vi = sh.lv[i];
          const int ji = sh.lj[i];
          for (int m = part; m < c; m += split) {
            const float vm = sh.lv[m];
            rank += (vm > vi) || (vm == vi && sh.lj[m] < ji);
          }
        }
        for (int o = 1; o < split; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (i < c && part == 0) sh.lr[i] = rank;
      }
      topk_sync();
      // output: block 0, the chosen blocks in ascending order, the tail block (tb >= 2 here)
      for (int i0 = 0; i0 < c * split; i0 += kTopkThreads) {
        const int q = i0 + t;
        const int i = q / split, part = q % split;
        int pos = 0;
        bool chosen = false;
        int ji = 0;
        if (i < c) {
          chosen = sh.lr[i] < k_eff;
          ji = sh.lj[i];
          if (chosen)
            for (int m = part; m < c; m += split) pos += (sh.lr[m] < k_eff && sh.lj[m] < ji);
        }
        for (int o = 1; o < split; o <<= 1) pos += __shfl_xor_sync(0xffffffffu, pos, o);
        if (chosen && part == 0) idx[1 + pos] = ji;
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
    for (int e = 0; e < KPT; ++e) key[e] = isc[e] ? ordered_key(v[e]) : 0u;
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

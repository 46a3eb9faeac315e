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
  int n_list;
  float lv[kMaxList];
  int lj[kMaxList];
  unsigned char flag[kMaxBlocksPerSeq];
};

// Bucket of a candidate score in the 256 equal slices of [lo, hi]. Monotone non-decreasing
// in x (a subtraction and a positive scaling, each rounded), so every candidate in a higher
// bucket outscores every candidate in a lower one.
__device__ __forceinline__ int score_bucket(float x, float lo, float scale) {
  return min(255, max(0, __float2int_rd((x - lo) * scale)));
}

// Top-k of one (sequence, group) by 256 threads (threads 0-255 of the CTA, synchronised with
// named barrier 1), from the block scores S[0 .. nb) in global memory. Writes idx[0 .. topk+2)
// (sorted, -1 padded) and *cnt_out. Fast path: min/max of the candidate scores, a
// 256-bucket histogram over that range, the bucket that holds the k-th score, then exact
// ranks (score descending, block ascending) among the candidates at or above that bucket --
// a few dozen for real score distributions. If more than kMaxList candidates share those
// buckets (near-constant scores), a 4-pass radix select on order-preserving 32-bit keys
// takes over. Either way the result is exact and ties go to the lower block index.
static __device__ void topk_select(const float* S, int32_t* idx, int32_t* cnt_out, int topk, int max_ctx,
                            int T, TopkShared& sh) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int kslots = topk + 2;
  const bool valid = (T >= 1 && T <= max_ctx);
  const int tb = valid ? (T - 1) / kBlock : -1;
  const int nb = tb + 1;
  const int per = (nb + kTopkThreads - 1) / kTopkThreads;
  const int jb = t * per;
  const int n_cand = max(0, tb - 1);
  const int k_eff = min(topk, n_cand);

  float v[kKeysPerThread];
  bool isc[kKeysPerThread];
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int j = jb + e;
    isc[e] = e < per && j >= 1 && j < tb;
    v[e] = isc[e] ? __ldcg(S + j) : 0.f;
    if (e < per && j < nb) sh.flag[j] = (j == 0 || j == tb) ? 1 : 0;   // the forced blocks
  }

  if (k_eff == n_cand) {
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e)
      if (isc[e]) sh.flag[jb + e] = 1;
  } else if (k_eff > 0) {
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int e = 0; e < kKeysPerThread; ++e)
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
    if (t == 0) sh.n_list = 0;
    topk_sync();
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      lo = fminf(lo, sh.red_lo[w]);
      hi = fmaxf(hi, sh.red_hi[w]);
    }
    const float scale = 256.f / (hi - lo);
    bool fast = hi > lo && isfinite(lo) && isfinite(hi) && isfinite(scale);   // CTA-uniform
    if (fast) {
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) {
        if (e >= per) break;                       // per is the same in every thread
        const unsigned d = isc[e] ? (unsigned)score_bucket(v[e], lo, scale) : 256u;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (isc[e] && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], (unsigned)__popc(peers));
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
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) {
        if (e >= per) break;                       // per is the same in every thread
        const bool in = isc[e] && score_bucket(v[e], lo, scale) >= bstar;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&sh.n_list, __popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (in) {
          const int p = base + __popc(bal & ((1u << lane) - 1u));
          sh.lv[p] = v[e];
          sh.lj[p] = jb + e;
        }
      }
      topk_sync();
      // exact rank of each listed candidate (score descending, block ascending): `split`
      // threads share one candidate, each scanning a slice of the list
      const int c = sh.n_list;
      const int split = c <= 32 ? 8 : (c <= 64 ? 4 : (c <= 128 ? 2 : 1));
      for (int i0 = 0; i0 < c * split; i0 += kTopkThreads) {
        const int q = i0 + t;
        const int i = q / split, part = q % split;
        int rank = 0;
        int ji = 0;
        if (i < c) {
          const float vi = sh.lv[i];
          ji = sh.lj[i];
          for (int m = part; m < c; m += split) {
            const float vm = sh.lv[m];
            rank += (vm > vi) || (vm == vi && sh.lj[m] < ji);
          }
        }
        for (int o = 1; o < split; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (i < c && part == 0 && rank < k_eff) sh.flag[ji] = 1;
      }
    } else {
      // radix select on order-preserving keys
      uint32_t key[kKeysPerThread];
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) key[e] = isc[e] ? ordered_key(v[e]) : 0u;
      uint32_t prefix = 0u, mask = 0u;
      int krem = k_eff;
      for (int shift = 24; shift >= 0; shift -= 8) {
        sh.hist[t] = 0u;
        topk_sync();
#pragma unroll
        for (int e = 0; e < kKeysPerThread; ++e) {
          const bool in = key[e] != 0u && (key[e] & mask) == prefix;
          const unsigned d = in ? (key[e] >> shift) & 255u : 256u;
          const unsigned peers = __match_any_sync(0xffffffffu, d);
          if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], (unsigned)__popc(peers));
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
      int my_eq = 0;
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) my_eq += (key[e] != 0u && key[e] == prefix);
      int dummy;
      int rank = topk_scan(my_eq, sh.warp_tot, &dummy) - my_eq;
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e) {
        if (key[e] == 0u) continue;
        if (key[e] > prefix) {
          sh.flag[jb + e] = 1;
        } else if (key[e] == prefix) {
          if (rank < krem) sh.flag[jb + e] = 1;
          ++rank;
        }
      }
    }
  }
  topk_sync();
  // the selected blocks in ascending order
  int my_sel = 0;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e)
    if (e < per && jb + e < nb) my_sel += sh.flag[jb + e];
  int total;
  int pos = topk_scan(my_sel, sh.warp_tot, &total) - my_sel;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e)
    if (e < per && jb + e < nb && sh.flag[jb + e] && pos < kslots) idx[pos++] = jb + e;
  for (int s = total + t; s < kslots; s += kTopkThreads) idx[s] = -1;
  if (t == 0) *cnt_out = min(total, kslots);
}


}  // namespace sparda

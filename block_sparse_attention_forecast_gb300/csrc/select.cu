// The Forecast selector (bittide thread: one forecast head per GQA group, no softmax;
// techwalker section 二; 10100 "SparDA 的解法"): score every compressed key of the target
// layer with the group's forecast vector, max-pool the window scores onto 64-token blocks and
// keep the top-k blocks plus block 0 and the tail block.
//
// One kernel. A CTA owns `chunk_blocks` consecutive blocks of one (sequence, group): it
// stages the contiguous run of compressed keys those blocks need with one bulk TMA copy,
// scores them (8 lanes per window, float32), max-pools them and writes the block scores to
// the workspace. The last CTA of the (sequence, group) to finish -- found with a counter in
// the workspace, which it resets -- selects the top-k by a 4-pass radix select on
// order-preserving 32-bit keys and writes the sorted block list.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kSelThreads = 256;
constexpr int kMaxBlocksPerSeq = kMaxCtx / kBlock;                 // 4096
constexpr int kKeysPerThread = kMaxBlocksPerSeq / kSelThreads;     // 16
constexpr int kSmemHeader = 128;                                   // mbarrier + padding

size_t smem_select_bytes(int chunk_blocks) {
  const int nw = kWinPerBlock * chunk_blocks + 1;
  return kSmemHeader + (size_t)nw * kRowBytes + (size_t)nw * sizeof(float);
}

int select_chunk_blocks(int nb_cap, int bg_count) {
  // Aim at about four resident CTAs per SM over 152 SMs; chunks of 16 .. 64 blocks.
  const long total = (long)nb_cap * bg_count;
  int ch = 16;
  while (ch < 64 && total / ch > 152L * 4) ch *= 2;
  return ch;
}

// Inclusive prefix sum over the 256 threads of the CTA; `warp_tot` is 8 words of shared
// memory. Returns the inclusive sum; *total gets the CTA-wide sum.
__device__ __forceinline__ int cta_inclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kSelThreads / 32; ++w) {
    const int x = warp_tot[w];
    if (w < warp) before += x;
    all += x;
  }
  __syncthreads();  // warp_tot may be reused right after
  *total = all;
  return v + before;
}

__device__ void select_topk(const SelectArgs& a, int bg, int T) {
  __shared__ unsigned hist[256];
  __shared__ int warp_tot[kSelThreads / 32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_krem;

  const int t = threadIdx.x;
  const int kslots = a.topk + 2;
  int32_t* idx = a.idx + (size_t)bg * kslots;
  const bool valid = (T >= 1 && T <= a.max_ctx);
  const int tb = valid ? (T - 1) / kBlock : -1;
  const int nb = tb + 1;
  const int per = (nb + kSelThreads - 1) / kSelThreads;
  const int jb = t * per;
  const float* S = a.block_scores + (size_t)bg * a.nb_cap;

  uint32_t key[kKeysPerThread];
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int j = jb + e;
    key[e] = (e < per && j >= 1 && j < tb) ? ordered_key(__ldcg(S + j)) : 0u;
  }
  const int n_cand = max(0, tb - 1);
  const int k_eff = min(a.topk, n_cand);

  // Threshold: a candidate is kept when key > thr, or key == thr and fewer than take_eq
  // equal keys sit at lower block indices.
  uint32_t thr;
  int take_eq;
  if (k_eff == n_cand) {
    thr = 0u;
    take_eq = 0;
  } else if (k_eff == 0) {
    thr = 0xffffffffu;
    take_eq = 0;
  } else {
    uint32_t prefix = 0u, mask = 0u;
    int krem = k_eff;
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist[t] = 0u;
      __syncthreads();
#pragma unroll
      for (int e = 0; e < kKeysPerThread; ++e)
        if (key[e] != 0u && (key[e] & mask) == prefix) atomicAdd(&hist[(key[e] >> shift) & 255u], 1u);
      __syncthreads();
      const int v = (int)hist[255 - t];      // thread t looks at digit 255 - t
      int tot;
      const int incl = cta_inclusive_scan(v, warp_tot, &tot);
      const int excl = incl - v;
      if (excl < krem && incl >= krem) {
        s_prefix = prefix | ((uint32_t)(255 - t) << shift);
        s_krem = krem - excl;
      }
      __syncthreads();
      prefix = s_prefix;
      krem = s_krem;
      mask |= 255u << shift;
    }
    thr = prefix;
    take_eq = krem;
  }

  int my_eq = 0;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) my_eq += (key[e] != 0u && key[e] == thr);
  int dummy;
  int rank = cta_inclusive_scan(my_eq, warp_tot, &dummy) - my_eq;

  bool sel[kKeysPerThread];
  int my_sel = 0;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e) {
    const int j = jb + e;
    bool s = false;
    if (e < per && j < nb) {
      if (j == 0 || j == tb) {
        s = true;
      } else if (key[e] != 0u) {
        if (key[e] > thr) {
          s = true;
        } else if (key[e] == thr) {
          s = rank < take_eq;
          ++rank;
        }
      }
    }
    sel[e] = s;
    my_sel += s;
  }
  int total;
  int pos = cta_inclusive_scan(my_sel, warp_tot, &total) - my_sel;
#pragma unroll
  for (int e = 0; e < kKeysPerThread; ++e)
    if (sel[e] && pos < kslots) idx[pos++] = jb + e;
  for (int s = total + t; s < kslots; s += kSelThreads) idx[s] = -1;
  if (t == 0) a.cnt[bg] = min(total, kslots);
}

__global__ void __launch_bounds__(kSelThreads) forecast_select_kernel(const SelectArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint8_t* tile = smem + kSmemHeader;
  const int CH = a.chunk_blocks;
  const int nw_max = kWinPerBlock * CH + 1;
  float* s_sc = reinterpret_cast<float*>(tile + (size_t)nw_max * kRowBytes);
  __shared__ bool s_last;

  const int bg = blockIdx.y;
  const int b = bg / a.G;
  const int t = threadIdx.x;
  const int T = a.seq_len[b];
  const bool valid = (T >= 1 && T <= a.max_ctx);
  if (!valid && t == 0 && blockIdx.x == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);

  const int nb = valid ? (T - 1) / kBlock + 1 : 0;
  const int W = valid ? num_windows(T - 1) : 0;
  const int j0 = blockIdx.x * CH;
  const int j1 = min(j0 + CH, nb);
  if (j0 < j1) {
    const int w0 = max(0, kWinPerBlock * j0 - 1);
    const int w1 = min(W, kWinPerBlock * j1);
    const int nw = w1 - w0;
    bool ok = true;
    if (nw > 0) {
      if (t == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)nw * kRowBytes;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(tile, a.ck + ((size_t)bg * a.W_cap + w0) * kHeadDim, bytes, bar);
      }
      // forecast slice of this thread: dims 8c..8c+7 and 64+8c..64+8c+7
      const int c = t & 7;
      float fr[16];
      {
        const uint4* fp = reinterpret_cast<const uint4*>(a.f + (size_t)bg * kHeadDim);
        const uint4 u0 = fp[c], u1 = fp[8 + c];
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          fr[2 * e] = bf16_lo(w[e]);
          fr[2 * e + 1] = bf16_hi(w[e]);
        }
      }
      __syncthreads();                       // mbarrier initialised before anyone waits
      ok = __syncthreads_and(mbar_wait(bar, 0, a.err));   // uniform across the CTA
      if (ok) {
        const int wl = t >> 3;               // 32 windows per pass, 8 lanes each
        for (int base = 0; base < nw; base += kSelThreads / 8) {
          const int i = base + wl;
          float acc = 0.f;
          if (i < nw) {
            const uint8_t* row = tile + (size_t)i * kRowBytes;
            const uint4 x0 = *reinterpret_cast<const uint4*>(row + 16 * c);
            const uint4 x1 = *reinterpret_cast<const uint4*>(row + 128 + 16 * c);
            const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc = fmaf(fr[2 * e], bf16_lo(w[e]), acc);
              acc = fmaf(fr[2 * e + 1], bf16_hi(w[e]), acc);
            }
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 4);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          if (c == 0 && i < nw) s_sc[i] = acc;
        }
      }
      __syncthreads();
    }
    float* S = a.block_scores + (size_t)bg * a.nb_cap;
    for (int jj = t; jj < j1 - j0; jj += kSelThreads) {
      const int j = j0 + jj;
      const int lo = max(kWinPerBlock * j - 1, 0);
      const int hi = min(kWinPerBlock * j + 3, W - 1);
      float m = -INFINITY;
      if (ok)
        for (int i = lo; i <= hi; ++i) m = fmaxf(m, s_sc[i - w0]);
      S[j] = m;
    }
  }

  // The last CTA of this (sequence, group) selects.
  __threadfence();
  __syncthreads();
  if (t == 0) {
    const unsigned prev = atomicAdd(a.counters + bg, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  select_topk(a, bg, T);
  if (t == 0) a.counters[bg] = 0u;
}

void launch_forecast_select(const SelectArgs& a, int bg_count, cudaStream_t s) {
  const size_t smem = smem_select_bytes(a.chunk_blocks);
  cudaFuncSetAttribute(forecast_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem_select_bytes(64));
  dim3 grid((a.nb_cap + a.chunk_blocks - 1) / a.chunk_blocks, bg_count);
  forecast_select_kernel<<<grid, kSelThreads, smem, s>>>(a);
}

}  // namespace sparda

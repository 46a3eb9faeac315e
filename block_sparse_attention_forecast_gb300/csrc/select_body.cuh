// The Forecast selector (bittide thread: one forecast head per GQA group, no softmax;
// techwalker section 二; 10100 "SparDA 的解法"): score every compressed key of the target
// layer with the group's forecast vector, max-pool the window scores onto 64-token blocks
// (windows 4j-1 .. 4j+3 overlap block j) and keep the top-k blocks plus block 0 and the tail
// block.
//
// Persistent kernel, one CTA per SM. The work is the list of (sequence-group, block) units,
// B*G*nb_cap of them; CTA c owns the contiguous range [U*c/grid, U*(c+1)/grid), cut into
// sub-chunks of up to 31 blocks that never cross a group boundary. Warp 8 is the producer:
// one lane streams the compressed keys each sub-chunk needs -- its 124 windows plus the one
// to their left, which the first block's max-pool also reads -- with one bulk TMA copy into
// a 6-stage shared-memory ring guarded by full/empty mbarriers. Warps 0-7 consume in two
// groups of four that take alternate sub-chunks: 4 lanes per window, 16-byte shared loads,
// four independent float32 FMA chains against the group's forecast held in registers, a
// 2-step shuffle reduction, then (after one group barrier) the max-pool of each block from
// its five windows and a store of the block scores. Window scores are double-buffered per
// group, so one barrier per sub-chunk suffices.
//
// When a CTA finishes its part of a (sequence, group), it bumps that group's counter in the
// workspace; the last of the covering CTAs selects the top-k (exact; ties to the lower block
// index, see select_topk) and writes the sorted list.
// Because ranges are contiguous, that selection overlaps the producer's loads for the next
// group; only the last group of the last CTA is a tail.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace sparda {

constexpr int kSelConsumerWarps = 8;
constexpr int kSelGroupWarps = 4;                         // two groups take alternate sub-chunks
constexpr int kSelConsumers = kSelConsumerWarps * 32;     // 256
constexpr int kSelGroupThreads = kSelGroupWarps * 32;     // 128
constexpr int kSelThreads = kSelConsumers + 32;
constexpr int kSubBlocks = 31;                            // blocks per sub-chunk
constexpr int kSubRows = kWinPerBlock * kSubBlocks + 1;   // 125 windows: 4 passes of 32
constexpr int kSelStages = 6;
// the two consumer groups take alternate sub-chunks: an even stage count keeps every stage
// with one group (a phase-parity wait cannot tell a stage's next phase from its last one)
static_assert(kSelStages % 2 == 0, "each ring stage must belong to one consumer group");
constexpr int kSelStageBytes = kSubRows * kRowBytes;
// Queue ids a producer of the queue-fed selection holds before their use (see sel_cta_dyn).
constexpr int kSelIdAhead = 2;
constexpr int kSelSmem = 128 /*align slack*/ + 128 /*barriers*/ + kSelStages * kSelStageBytes;


__device__ __forceinline__ void sel_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSelConsumers) : "memory");
}

__device__ __forceinline__ void group_sync(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "n"(kSelGroupThreads) : "memory");
}

// Barrier of consumer group grp (128 threads) that also returns whether v holds in every one
// of its threads.
__device__ __forceinline__ bool group_all(int grp, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)v), "r"(2 + grp), "n"(kSelGroupThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void sel_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ int sel_cta_of_unit(long long u, int grid, long long U) {
  return (int)(((u + 1) * grid - 1) / U);
}

// Per (sequence, group) constants.
struct SelGroup {
  int T, nb, W;
  bool valid;
};

__device__ __forceinline__ SelGroup sel_group(const SelectArgs& a, int bg) {
  SelGroup gr;
  gr.T = a.seq_len[bg / a.G];
  gr.valid = gr.T >= 1 && gr.T <= a.max_ctx;
  gr.nb = gr.valid ? (gr.T - 1) / kBlock + 1 : 0;
  gr.W = gr.valid ? num_windows(gr.T - 1) : 0;
  return gr;
}

// Window scores of one staged sub-chunk by a consumer group: 4 lanes per window (lane c takes
// dims 8c + 32k), 16-byte shared loads, four independent FMA chains against the forecast fr
// held in registers, then a 2-step shuffle. sw[i] gets window i of the tile (i < kSubRows).
__device__ __forceinline__ void sel_score_windows(const uint8_t* tile, int nw, const float (&fr)[32], float* sw,
                                                  int c, int wl, bool ok) {
  for (int base = 0; base < kSubRows; base += kSelGroupThreads / 4) {
    const int i = base + wl;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (ok && i < nw) {
      const uint8_t* row = tile + (size_t)i * kRowBytes + 16 * c;
      const uint4 x0 = *reinterpret_cast<const uint4*>(row);
      const uint4 x1 = *reinterpret_cast<const uint4*>(row + 64);
      const uint4 x2 = *reinterpret_cast<const uint4*>(row + 128);
      const uint4 x3 = *reinterpret_cast<const uint4*>(row + 192);
      const uint32_t w0v[4] = {x0.x, x0.y, x0.z, x0.w}, w1v[4] = {x1.x, x1.y, x1.z, x1.w};
      const uint32_t w2v[4] = {x2.x, x2.y, x2.z, x2.w}, w3v[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a0 = fmaf(fr[2 * e], bf16_lo(w0v[e]), a0);
        a0 = fmaf(fr[2 * e + 1], bf16_hi(w0v[e]), a0);
        a1 = fmaf(fr[8 + 2 * e], bf16_lo(w1v[e]), a1);
        a1 = fmaf(fr[8 + 2 * e + 1], bf16_hi(w1v[e]), a1);
        a2 = fmaf(fr[16 + 2 * e], bf16_lo(w2v[e]), a2);
        a2 = fmaf(fr[16 + 2 * e + 1], bf16_hi(w2v[e]), a2);
        a3 = fmaf(fr[24 + 2 * e], bf16_lo(w3v[e]), a3);
        a3 = fmaf(fr[24 + 2 * e + 1], bf16_hi(w3v[e]), a3);
      }
    }
    float acc = (a0 + a1) + (a2 + a3);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (c == 0 && i < kSubRows) sw[i] = acc;
  }
}

// The forecast slice of lane c (dims 8c + 32k, k < 4) of one group, from 128 bf16 at fp.
__device__ __forceinline__ void sel_load_forecast(const uint4* fp, int c, float (&fr)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = fp[c + 4 * k];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      fr[8 * k + 2 * e] = bf16_lo(w[e]);
      fr[8 * k + 2 * e + 1] = bf16_hi(w[e]);
    }
  }
}

// The work of CTA `cta` of `grid` CTAs that share the selection units.
__device__ __forceinline__ void sel_cta(const SelectArgs& a, int cta, int grid) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kSelStages;
  uint8_t* ring = smem + 128;
  __shared__ float s_win[2][2][kSubRows + 3];    // [group][buffer][window]
  __shared__ TopkShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long U = (long long)a.n_units;
  const long long J0 = U * cta / grid, J1 = U * (cta + 1) / grid;

  if (tid == 0) {
    for (int i = 0; i < kSelStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kSelGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSelConsumerWarps) {
    // -------------------------------------------------------------- producer
    if (lane != 0) return;
    int it = 0;
    for (long long u = J0; u < J1;) {
      const int bg = (int)(u / a.nb_cap);
      const long long seg_end = min(J1, (long long)(bg + 1) * a.nb_cap);
      const SelGroup gr = sel_group(a, bg);
      const int jseg0 = (int)(u - (long long)bg * a.nb_cap);
      const int jseg1 = (int)(seg_end - (long long)bg * a.nb_cap);
      u = seg_end;
      for (int j0 = jseg0; j0 < min(jseg1, gr.nb); j0 += kSubBlocks) {
        const int j1 = min(min(j0 + kSubBlocks, jseg1), gr.nb);
        const int w0 = max(0, kWinPerBlock * j0 - 1);
        const int w1 = min(gr.W, kWinPerBlock * j1);
        const int stage = it % kSelStages;
        if (it >= kSelStages && !mbar_wait(&empty[stage], ((it / kSelStages) & 1) ^ 1, a.err)) return;
        if (w1 > w0) {
          const uint32_t bytes = (uint32_t)(w1 - w0) * kRowBytes;
          mbar_arrive_expect_tx(&full[stage], bytes);
          bulk_load(ring + stage * kSelStageBytes, a.ck + ((size_t)bg * a.W_cap + w0) * kHeadDim, bytes,
                    &full[stage]);
        } else {
          sel_arrive(&full[stage]);             // nothing to load: complete the phase
        }
        ++it;
      }
    }
    if (a.l2_prefetch) {
      // this CTA's slice of the buffer the next launches read, into L2 (16-byte granules)
      const size_t g16 = a.l2_prefetch_bytes / 16;
      const size_t b0 = g16 * cta / grid * 16, b1 = g16 * (cta + 1) / grid * 16;
      const char* base = static_cast<const char*>(a.l2_prefetch);
      for (size_t off = b0; off < b1; off += 32768) {
        const uint32_t n = (uint32_t)min((size_t)32768, b1 - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + off), "r"(n) : "memory");
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int t = tid;
  const int grp = warp / kSelGroupWarps;          // takes sub-chunks it % 2 == grp
  const int gt = t % kSelGroupThreads;            // thread within the group
  const int c = gt & 3;                           // lane within a window: dims 8c + 32k
  const int wl = gt >> 2;                         // window of this thread within a pass
  int it = 0, nbuf = 0;
  bool first_seg = true;
  bool ok = true;                      // false after a wait ran out: skip compute, keep pace
  for (long long u = J0; u < J1;) {
    const int bg = (int)(u / a.nb_cap);
    const long long seg_end = min(J1, (long long)(bg + 1) * a.nb_cap);
    const SelGroup gr = sel_group(a, bg);
    if (!gr.valid && t == 0 && u == (long long)bg * a.nb_cap) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    const int jseg0 = (int)(u - (long long)bg * a.nb_cap);
    const int jseg1 = (int)(seg_end - (long long)bg * a.nb_cap);
    u = seg_end;
    // forecast slice of this thread (written by the kernel before this one in the stream)
    if (first_seg) {
      grid_dep_wait();
      first_seg = false;
    }
    float fr[32];
    sel_load_forecast(reinterpret_cast<const uint4*>(a.f + (size_t)bg * kHeadDim), c, fr);
    float* S = a.block_scores + (size_t)bg * a.nb_cap;
    for (int j0 = jseg0; j0 < min(jseg1, gr.nb); j0 += kSubBlocks, ++it) {
      if ((it & 1) != grp) continue;
      const int j1 = min(min(j0 + kSubBlocks, jseg1), gr.nb);
      const int w0 = max(0, kWinPerBlock * j0 - 1);      // tile row 0
      const int w1 = min(gr.W, kWinPerBlock * j1);
      const int nw = max(0, w1 - w0);
      const int stage = it % kSelStages;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (it / kSelStages) & 1, a.err));
      const uint8_t* tile = ring + stage * kSelStageBytes;
      float* sw = s_win[grp][nbuf & 1];
      sel_score_windows(tile, nw, fr, sw, c, wl, ok);
      __syncwarp();
      if ((t & 31) == 0) sel_arrive(&empty[stage]);
      group_sync(grp);                              // this sub-chunk's window scores complete
      if (gt < j1 - j0) {                           // block j uses windows 4j-1 .. 4j+3 below W
        const int j = j0 + gt;
        float m = -INFINITY;
        if (ok) {
#pragma unroll
          for (int d = -1; d <= 3; ++d) {
            const int w = kWinPerBlock * j + d;
            if (w >= 0 && w < gr.W) m = fmaxf(m, sw[w - w0]);
          }
        }
        S[j] = m;
      }
      ++nbuf;                                       // alternate buffers: no second barrier
    }
    if (!a.do_topk) continue;        // the top-k runs in a later launch (decode prologue)
    // this CTA's part of the group is done: count it; the last covering CTA selects
    const long long first_u = (long long)bg * a.nb_cap, last_u = first_u + a.nb_cap - 1;
    const int n_cover = sel_cta_of_unit(last_u, grid, U) - sel_cta_of_unit(first_u, grid, U) + 1;
    sel_sync();                                     // block scores of all consumers stored
    if (t == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(a.counters + bg, 1u);
      sh.last = (prev == (unsigned)(n_cover - 1));
      if (sh.last) a.counters[bg] = 0u;
      __threadfence();
    }
    sel_sync();
    if (sh.last)
      topk_select(a.block_scores + (size_t)bg * a.nb_cap, a.idx + (size_t)bg * (a.topk + 2), a.cnt + bg,
                  a.topk, a.max_ctx, gr.T, sh);
    sel_sync();
  }
}


// Dynamic variant, for the scores-only selection of the fused launch: the sub-chunks (31
// blocks of one (sequence, group)) are handed out one at a time from a counter in the
// workspace, so CTAs that start late or stream slowly take fewer of them and the selection
// CTAs finish together. The producer writes each stage's (group, blocks) beside it; the
// consumers keep every group's forecast in shared memory (bg_count * 256 bytes after the
// ring). The counter is reset by the last producer to finish (queue[1] counts them).
__device__ __forceinline__ void sel_cta_dyn(const SelectArgs& a, int cta, int grid) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kSelStages;
  uint8_t* ring = smem + 128;
  uint8_t* ftab = ring + kSelStages * kSelStageBytes;      // [bg_count][128] bf16 forecasts
  __shared__ float s_win[2][2][kSubRows + 3];               // [group][buffer][window]
  __shared__ int4 s_meta[kSelStages];                       // (bg, j0, j1, W); bg < 0: no more

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bg_count = a.n_units / a.nb_cap;
  const int ipg = (a.nb_cap + kSubBlocks - 1) / kSubBlocks;  // sub-chunks per group
  const int n_items = bg_count * ipg;

  if (tid == 0) {
    for (int i = 0; i < kSelStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kSelGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSelConsumerWarps) {
    // -------------------------------------------------------------- producer
    if (lane != 0) return;
    int it = 0;
    int ends = 0;                               // end markers pushed (one per consumer group)
    // Queue ids are taken kSelIdAhead ahead of their use, so that the atomic's round trip
    // (about a microsecond under load, longer when the counter's memory sits far from the SM)
    // overlaps the wait for a free stage instead of adding to it.
    int pend[kSelIdAhead];
#pragma unroll
    for (int k = 0; k < kSelIdAhead; ++k) pend[k] = (int)atomicAdd(a.queue, 1u);
    while (ends < 2) {
      int4 m = make_int4(-1, 0, 0, 0);
      int w0 = 0, w1 = 0;
      if (ends == 0) {
        const int id = pend[0];
#pragma unroll
        for (int k = 0; k + 1 < kSelIdAhead; ++k) pend[k] = pend[k + 1];
        pend[kSelIdAhead - 1] = id < n_items ? (int)atomicAdd(a.queue, 1u) : n_items;
        if (id < n_items) {
          const int bg = id / ipg, j0 = (id % ipg) * kSubBlocks;
          const SelGroup gr = sel_group(a, bg);
          if (!gr.valid && j0 == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
          if (j0 >= gr.nb) continue;            // past this sequence's blocks: nothing to do
          m = make_int4(bg, j0, min(j0 + kSubBlocks, gr.nb), gr.W);
          w0 = max(0, kWinPerBlock * m.y - 1);
          w1 = min(gr.W, kWinPerBlock * m.z);
        }
      }
      const int stage = it % kSelStages;
      if (it >= kSelStages && !mbar_wait(&empty[stage], ((it / kSelStages) & 1) ^ 1, a.err)) break;
      s_meta[stage] = m;
      if (m.x >= 0 && w1 > w0) {
        const uint32_t bytes = (uint32_t)(w1 - w0) * kRowBytes;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_load(ring + stage * kSelStageBytes, a.ck + ((size_t)m.x * a.W_cap + w0) * kHeadDim, bytes,
                  &full[stage]);
      } else {
        sel_arrive(&full[stage]);               // (releases the stage's meta) nothing to load
      }
      if (m.x < 0) ++ends;
      ++it;
    }
    if (atomicAdd(a.queue + 1, 1u) == (unsigned)(grid - 1)) {   // every producer has finished
      a.queue[0] = 0u;
      a.queue[1] = 0u;
    }
    if (a.l2_prefetch) {
      const size_t g16 = a.l2_prefetch_bytes / 16;
      const size_t b0 = g16 * cta / grid * 16, b1 = g16 * (cta + 1) / grid * 16;
      const char* base = static_cast<const char*>(a.l2_prefetch);
      for (size_t off = b0; off < b1; off += 32768) {
        const uint32_t n = (uint32_t)min((size_t)32768, b1 - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + off), "r"(n) : "memory");
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int t = tid;
  const int grp = warp / kSelGroupWarps;          // takes stages it % 2 == grp
  const int gt = t % kSelGroupThreads;
  const int c = gt & 3;
  const int wl = gt >> 2;
  // the forecasts of every group (written by the kernel before this one in the stream)
  grid_dep_wait();
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.f);
    uint4* dst = reinterpret_cast<uint4*>(ftab);
    for (int i = t; i < bg_count * (kHeadDim * 2 / 16); i += kSelConsumers) dst[i] = __ldcg(src + i);
  }
  sel_sync();
  int nbuf = 0;
  for (int it = grp;; it += 2) {
    const int stage = it % kSelStages;
    // every warp of the group leaves the loop at the same stage: on a wait that ran out (in
    // any of them) or at the end marker
    if (!group_all(grp, mbar_wait(&full[stage], (it / kSelStages) & 1, a.err))) break;
    const int4 m = s_meta[stage];
    if (m.x < 0) break;                           // no more sub-chunks for this group
    const int bg = m.x, j0 = m.y, j1 = m.z, W = m.w;
    const int w0 = max(0, kWinPerBlock * j0 - 1);
    const int nw = max(0, min(W, kWinPerBlock * j1) - w0);
    float fr[32];
    sel_load_forecast(reinterpret_cast<const uint4*>(ftab + (size_t)bg * kHeadDim * 2), c, fr);
    float* sw = s_win[grp][nbuf & 1];
    sel_score_windows(ring + stage * kSelStageBytes, nw, fr, sw, c, wl, true);
    __syncwarp();
    if ((t & 31) == 0) sel_arrive(&empty[stage]);
    group_sync(grp);                              // this sub-chunk's window scores complete
    if (gt < j1 - j0) {
      const int j = j0 + gt;
      float mx = -INFINITY;
#pragma unroll
      for (int d = -1; d <= 3; ++d) {
        const int w = kWinPerBlock * j + d;
        if (w >= 0 && w < W) mx = fmaxf(mx, sw[w - w0]);
      }
      a.block_scores[(size_t)bg * a.nb_cap + j] = mx;
    }
    ++nbuf;
  }
}

}  // namespace sparda

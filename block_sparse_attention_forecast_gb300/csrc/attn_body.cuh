// Block-sparse GQA decode attention (bittide thread: the next layer's own queries attend the
// blocks the forecast picked; techwalker section 六: SparDA leaves the sparse attention
// computation itself unchanged).
//
// Persistent kernel, one CTA per SM. The work is the list of (sequence-group, slot) units,
// B*G*(topk+2) of them; CTA c owns the contiguous range [U*c/grid, U*(c+1)/grid), so every
// CTA streams the same number of 64-token blocks and a (sequence, group) is split over a few
// neighbouring CTAs.
//
// Warp 8 is the producer. Its 32 lanes read the metadata of 32 units at a time (sequence
// length, selection count, block index) in parallel; lane 0 then issues, for every selected
// block, four tiled TMA loads (K and V, two 64-column halves each, 128-byte swizzle) into a
// 4-stage shared-memory ring guarded by full/empty mbarriers, and records the block index
// beside the stage. Warps 0-7 consume in two groups of four that take alternate blocks, so
// every SM sub-partition has two warps to switch between. Within a group, warp w takes
// tokens 16w .. 16w+15 of its block: S = Q K^T with the group's 16 query heads as the M
// dimension of m16n8k16 bf16 MMAs, an online softmax in float32 (exp2 domain), then O += P V
// with P re-packed from the S accumulators.
//
// At the end of a (sequence, group) in its range a CTA merges its eight warps' partial
// results through shared memory (one write, one read of a padded buffer). A group covered by
// one CTA is written out directly. Otherwise, in the cluster form (kClusterMerge: the standalone
// launch with a whole number of CTAs per group, each group one thread-block cluster), each CTA
// pushes its (O, max, sum) of every head into the shared memory of the CTA that owns the head,
// and after one cluster barrier each combines its share of the heads; in the general form each covering CTA stores (O, max, sum) to the workspace and
// the last one to arrive (a counter in the workspace, which it resets) merges them with
// log-sum-exp weights. Because ranges are contiguous, that merge overlaps the producer's loads
// for the next group.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "timeline.cuh"

namespace sparda {

constexpr int kGroupWarps = 4;
constexpr int kConsumerWarps = 2 * kGroupWarps;
constexpr int kConsumers = kConsumerWarps * 32;             // 256
constexpr int kAttnThreads = kConsumers + 32;
constexpr int kStages = 4;
// The two consumer groups take alternate ring slots, so with an even stage count each stage
// is only ever consumed by one group. With an odd count a group could wait, by phase parity,
// for a stage's next phase while the other group's current phase is still open: the parity
// wait cannot tell the two apart and would pass early.
static_assert(kStages % 2 == 0, "each ring stage must belong to one consumer group");
constexpr int kSlotBytes = 2 * kBlockBytes;                 // K + V of one block
constexpr int kMStride = kHeadDim + 8;      // merge-buffer row stride (floats): no bank conflicts
constexpr int kMergeFloats = kConsumerWarps * (kHeads * kMStride + 2 * kHeads);
constexpr int kMaxInlineSeg = 8;           // partials the last arriver keeps in registers
constexpr int kAttnSmem = 1024 /*align slack*/ + 1024 /*header*/ + kStages * kSlotBytes +
                          kMergeFloats * 4;
// The cluster form's receive area, after the merge buffer: for each head h, the sg partials
// (O, max, sum) that the cluster's CTAs push to the CTA owning h (rank h % sg), at entry
// (h / sg) * sg + source rank: below ceil(16 / sg) * sg <= 16 + sg - 1 entries.
constexpr int kMaxClusterCtas = 8;
constexpr int kRecvEntries = kHeads + kMaxClusterCtas - 1;
constexpr int kRecvFloats = kRecvEntries * kHeadDim + 2 * kRecvEntries;
constexpr int kAttnClusterSmem = kAttnSmem + kRecvFloats * 4;

// Shared-memory address of 16-byte chunk `chunk` (0..15 over the 128 dims) of row `r` of a
// K or V block staged as two 64-row x 128-byte halves with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t swz(const uint8_t* tile, int r, int chunk) {
  return smem_addr(tile + (chunk >> 3) * (kBlockBytes / 2) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// CTA whose unit range contains unit u (ranges start at floor(U*c/grid)).
__device__ __forceinline__ int cta_of_unit(long long u, int grid, long long U) {
  return (int)(((u + 1) * grid - 1) / U);
}

struct GroupInfo {
  int T, tb, n_sel;
};

// Both loads are issued before either is looked at (one memory round trip, not two).
__device__ __forceinline__ GroupInfo group_info(const AttnArgs& a, int bg) {
  GroupInfo gi;
  gi.T = a.seq_len[bg / a.G];
  const int cnt = a.cnt[bg];
  const bool valid = gi.T >= 1 && gi.T <= a.max_ctx;
  gi.tb = valid ? (gi.T - 1) / kBlock : 0;
  gi.n_sel = valid ? min(max(cnt, 0), a.kslots) : 0;
  return gi;
}

// The work of CTA c of `grid` CTAs that share the attention units. The tensor maps live in
// the calling kernel's parameter space. kClusterMerge: CTA c is rank c % seg_per_group of a
// cluster of seg_per_group CTAs that covers group c / seg_per_group (seg_per_group >= 2), and
// every thread of the CTA reaches the merge's one cluster barrier. tl_first (timeline
// build only): thread 0 stores there the time its first block arrived.
template <bool kClusterMerge = false>
__device__ __forceinline__ void attn_cta(const AttnArgs& a, const CUtensorMap* mk, const CUtensorMap* mv,
                                         const CUtensorMap* hk, const CUtensorMap* hv, int c, int grid,
                                         unsigned long long* tl_first = nullptr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  int* stage_j = reinterpret_cast<int*>(empty + kStages);      // block index per stage
  int* s_flag = stage_j + kStages;
  uint8_t* ring = smem + 1024;
  float* mO = reinterpret_cast<float*>(ring + kStages * kSlotBytes);    // [8][16][kMStride]
  float* mM = mO + kConsumerWarps * kHeads * kMStride;                  // [8][16]
  float* mL = mM + kConsumerWarps * kHeads;                             // [8][16]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long U = (long long)a.n_units;
  // this CTA's units: an equal share of one group's slots, or a contiguous balanced range
  const int sg = a.seg_per_group;
  const int u0 = sg > 0 ? (c / sg) * a.kslots + a.kslots * (c % sg) / sg : (int)(U * c / grid);
  const int u1 = sg > 0 ? (c / sg) * a.kslots + a.kslots * (c % sg + 1) / sg : (int)(U * (c + 1) / grid);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(mk);
      prefetch_tensormap(mv);
      if (a.offload) {
        prefetch_tensormap(hk);
        prefetch_tensormap(hv);
      }
    }
    // the selection and the caches were written by the kernels before this one in the stream
    // (the decode prologue's top-k and append)
    grid_dep_wait();
    int it = 0;
    for (int base = u0; base < u1; base += 32) {
      // lane i prepares unit base + i
      const int u = base + lane;
      bool v = false;
      int j = 0, row = 0, hot = 0;
      if (u < u1) {
        const int bg = u / a.kslots;
        const int j_raw = a.idx[u];              // in bounds for every unit: loaded with the two below
        const GroupInfo gi = group_info(a, bg);
        if (u - bg * a.kslots < gi.n_sel) {
          v = true;
          j = j_raw;
          if (j < 0 || j > gi.tb) {
            atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
            j = 0;
          }
          if (!a.offload) {
            row = bg * a.max_ctx + j * kBlock;
          } else if (j == 0 || j == gi.tb) {
            hot = 1;
            row = (bg * kHotSlots + hot_slot(j)) * kBlock;
          } else if (a.stage_slot) {
            int cs = a.stage_slot[u];             // its block-cache slot
            if (cs < 0 || cs >= a.stage_slots) {
              atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
              cs = 0;
            }
            row = (bg * a.stage_slots + cs) * kBlock;
          } else {
            row = u * kBlock;                   // staging slot (bg, s) = unit u
          }
        }
      }
      unsigned vmask = __ballot_sync(0xffffffffu, v);
      while (vmask) {
        const int i = __ffs(vmask) - 1;
        vmask &= vmask - 1;
        const int jj = __shfl_sync(0xffffffffu, j, i);
        const int rr = __shfl_sync(0xffffffffu, row, i);
        const int hh = __shfl_sync(0xffffffffu, hot, i);
        int ok = 1;
        if (lane == 0) {
          const int stage = it % kStages;
          if (it >= kStages) ok = mbar_wait(&empty[stage], ((it / kStages) & 1) ^ 1, a.err);
          if (ok) {
            const CUtensorMap* tk = hh ? hk : mk;
            const CUtensorMap* tv = hh ? hv : mv;
            uint8_t* dst = ring + stage * kSlotBytes;
            stage_j[stage] = jj;
            mbar_arrive_expect_tx(&full[stage], kSlotBytes);
            tma_load_2d(dst, tk, 0, rr, &full[stage]);
            tma_load_2d(dst + kBlockBytes / 2, tk, 64, rr, &full[stage]);
            tma_load_2d(dst + kBlockBytes, tv, 0, rr, &full[stage]);
            tma_load_2d(dst + kBlockBytes + kBlockBytes / 2, tv, 64, rr, &full[stage]);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {  // a wait ran out: no further loads
          if constexpr (!kClusterMerge) return;
          base = u1;
          break;
        }
        ++it;
      }
    }
    if constexpr (kClusterMerge) cluster_sync();   // the consumers' merge barrier
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = warp / kGroupWarps;         // 0 or 1: takes blocks it % 2 == grp
  const int wq = warp % kGroupWarps;          // token quarter of the block
  const int g = lane >> 2, cq = lane & 3;
  const float sl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
  const int t = tid;                                              // 0..255
  int it = 0;
  // A wait that runs out sets the device error word; that warp then skips all further
  // compute but keeps walking the same loop, so the named barriers stay matched.
  bool ok = true;
  // The workspace may still be in use by the kernel before this one in the stream (a launch
  // that may overlap it): no partial or counter is written before that kernel completes.
  grid_dep_wait();
  for (int u = u0; u < u1;) {
    const int bg = u / a.kslots;
    const int seg_end = min(u1, (bg + 1) * a.kslots);
    const GroupInfo gi = group_info(a, bg);
    const int s_begin = u - bg * a.kslots;
    const int s_stop = min(seg_end - bg * a.kslots, gi.n_sel);
    u = seg_end;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    if (s_begin < s_stop) {
      uint32_t qf[8][4];
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)bg * kHeads + g) * kHeadDim);
      const uint32_t* q1 = q0 + 8 * (kHeadDim / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qf[ks][0] = q0[8 * ks + cq];
        qf[ks][1] = q1[8 * ks + cq];
        qf[ks][2] = q0[8 * ks + 4 + cq];
        qf[ks][3] = q1[8 * ks + 4 + cq];
      }
      for (int s = s_begin; s < s_stop; ++s, ++it) {
        if ((it & 1) != grp) continue;
        const int stage = it % kStages;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (it / kStages) & 1, a.err));
        if (!ok) continue;
#ifdef SPARDA_TIMELINE
        if (tid == 0 && tl_first && *tl_first == 0) *tl_first = tl_now();
#endif
        const int j = stage_j[stage];
        const uint8_t* Kt = ring + stage * kSlotBytes;
        const uint8_t* Vt = Kt + kBlockBytes;

        // S = Q K^T, two independent accumulator chains per n-tile
        float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int r = 16 * wq + (lane & 7) + ((lane >> 4) << 3);
          const int hi = (lane >> 3) & 1;
#pragma unroll
          for (int ks = 0; ks < 8; ks += 2) {
            uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
            ldsm_x4(swz(Kt, r, 2 * ks + hi), b0, b1, b2, b3);
            ldsm_x4(swz(Kt, r, 2 * ks + 2 + hi), c0, c1, c2, c3);
            mma_16816(sa[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
            mma_16816(sa[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            mma_16816(sb[0], qf[ks + 1][0], qf[ks + 1][1], qf[ks + 1][2], qf[ks + 1][3], c0, c1);
            mma_16816(sb[1], qf[ks + 1][0], qf[ks + 1][1], qf[ks + 1][2], qf[ks + 1][3], c2, c3);
          }
        }
        float sc[2][4];
        const int tok0 = j * kBlock + 16 * wq + 2 * cq;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = tok0 + 8 * nt + (e & 1);
            sc[nt][e] = (pos < gi.T) ? (sa[nt][e] + sb[nt][e]) * sl2 : -INFINITY;
          }
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
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
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
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
        const uint32_t pa0 = pack_bf16(p[0][0], p[0][1]);
        const uint32_t pa1 = pack_bf16(p[0][2], p[0][3]);
        const uint32_t pa2 = pack_bf16(p[1][0], p[1][1]);
        const uint32_t pa3 = pack_bf16(p[1][2], p[1][3]);
        {
          const int r = 16 * wq + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int hi = lane >> 4;
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(swz(Vt, r, 2 * np + hi), b0, b1, b2, b3);
            mma_16816(o[2 * np], pa0, pa1, pa2, pa3, b0, b1);
            mma_16816(o[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
    }

    // ---------------------------------------------------------- merge the eight warps
    consumer_sync();                           // the merge buffer is free again
    {
      float* myO = mO + (warp * kHeads + g) * kMStride + 2 * cq;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        *reinterpret_cast<float2*>(myO + 8 * n) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(myO + 8 * n + 8 * kMStride) = make_float2(o[n][2], o[n][3]);
      }
      if (cq == 0) {
        mM[warp * kHeads + g] = m0;
        mM[warp * kHeads + g + 8] = m1;
        mL[warp * kHeads + g] = l0;
        mL[warp * kHeads + g + 8] = l1;
      }
    }
    consumer_sync();
    // thread t: head h = t / 16, dims d0 .. d0+7
    const int h = t >> 4, d0 = (t & 15) * 8;
    float Mh = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) Mh = fmaxf(Mh, mM[w * kHeads + h]);
    const float baseh = (Mh == -INFINITY) ? 0.f : Mh;
    float Oh[8], Lh = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) Oh[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float wt = exp2f(mM[w * kHeads + h] - baseh);
      Lh += wt * mL[w * kHeads + h];
      const float4* src = reinterpret_cast<const float4*>(mO + (w * kHeads + h) * kMStride + d0);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float4 x = src[e];
        Oh[4 * e] += wt * x.x;
        Oh[4 * e + 1] += wt * x.y;
        Oh[4 * e + 2] += wt * x.z;
        Oh[4 * e + 3] += wt * x.w;
      }
    }
    if constexpr (kClusterMerge) {
      // this CTA's (O, max, sum) of head h pushed into the receive area of the CTA that owns
      // h (rank h % sg); after one cluster barrier each CTA combines its heads' sg partials
      // from its own shared memory, and no CTA reads another's, so none has to stay resident
      float* rO = mL + kConsumerWarps * kHeads;            // [kRecvEntries][128 dims]
      float* rM = rO + kRecvEntries * kHeadDim;            // [kRecvEntries]
      float* rL = rM + kRecvEntries;                       // [kRecvEntries]
      const uint32_t rank = cluster_rank();
      const int entry = (h / sg) * sg + (int)rank;
      const uint32_t owner = (uint32_t)(h % sg);
      st_cluster_f4(rO + entry * kHeadDim + d0, owner, make_float4(Oh[0], Oh[1], Oh[2], Oh[3]));
      st_cluster_f4(rO + entry * kHeadDim + d0 + 4, owner, make_float4(Oh[4], Oh[5], Oh[6], Oh[7]));
      if ((t & 15) == 0) {
        st_cluster_f(rM + entry, owner, Mh);
        st_cluster_f(rL + entry, owner, Lh);
      }
      cluster_sync();                          // every partial of the cluster's heads is in place
      if (h % sg == (int)rank) {
        const int e0 = (h / sg) * sg;
        float Mx = -INFINITY;
        for (int q = 0; q < sg; ++q) Mx = fmaxf(Mx, rM[e0 + q]);
        const float base = (Mx == -INFINITY) ? 0.f : Mx;
        float acc[8], L = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int q = 0; q < sg; ++q) {
          const float wt = exp2f(rM[e0 + q] - base);
          L += wt * rL[e0 + q];
          const float4* src = reinterpret_cast<const float4*>(rO + (e0 + q) * kHeadDim + d0);
          const float4 x0 = src[0], x1 = src[1];
          acc[0] += wt * x0.x; acc[1] += wt * x0.y; acc[2] += wt * x0.z; acc[3] += wt * x0.w;
          acc[4] += wt * x1.x; acc[5] += wt * x1.y; acc[6] += wt * x1.z; acc[7] += wt * x1.w;
        }
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pk[e] = pack_bf16(L > 0.f ? acc[2 * e] / L : 0.f, L > 0.f ? acc[2 * e + 1] / L : 0.f);
        *reinterpret_cast<uint4*>(a.out + ((size_t)bg * kHeads + h) * kHeadDim + d0) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      continue;
    }
    const long long first = (long long)bg * a.kslots, last = first + a.kslots - 1;
    const int c_first = sg > 0 ? (c / sg) * sg : cta_of_unit(first, grid, U);
    const int n_seg = sg > 0 ? sg : cta_of_unit(last, grid, U) - c_first + 1;
    uint4* outp = reinterpret_cast<uint4*>(a.out + ((size_t)bg * kHeads + h) * kHeadDim + d0);
    if (n_seg == 1) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        pk[e] = pack_bf16(Lh > 0.f ? Oh[2 * e] / Lh : 0.f, Lh > 0.f ? Oh[2 * e + 1] / Lh : 0.f);
      *outp = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      continue;
    }
    const int seg = c - c_first;
    float4* po = reinterpret_cast<float4*>(a.part_o + (((size_t)bg * a.kslots + seg) * kHeads + h) * kHeadDim + d0);
    po[0] = make_float4(Oh[0], Oh[1], Oh[2], Oh[3]);
    po[1] = make_float4(Oh[4], Oh[5], Oh[6], Oh[7]);
    if ((t & 15) == 0) {
      float* pml = a.part_ml + ((size_t)bg * a.kslots + seg) * 2 * kHeads;
      pml[h] = Mh;
      pml[kHeads + h] = Lh;
    }
    consumer_sync();                           // every consumer's partial stores are issued
    if (t == 0) {
      // release: this CTA's partials (ordered by the barrier) before the count; acquire:
      // the other CTAs' partials before the merge below
      unsigned prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                   : "=r"(prev) : "l"(a.counters + bg) : "memory");
      *s_flag = (prev == (unsigned)(n_seg - 1));
      if (*s_flag) a.counters[bg] = 0u;
    }
    consumer_sync();
    if (!*s_flag) continue;
    // last arriver: merge the n_seg partials of this group
    const float* pml0 = a.part_ml + (size_t)bg * a.kslots * 2 * kHeads;
    const float* po0 = a.part_o + (size_t)bg * a.kslots * kHeads * kHeadDim + h * kHeadDim + d0;
    float acc[8], L = 0.f, M = -INFINITY;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < n_seg; s0 += kMaxInlineSeg) {
      // issue every load of up to kMaxInlineSeg partials before combining them
      float pm[kMaxInlineSeg], pl[kMaxInlineSeg];
      float4 px[kMaxInlineSeg][2];
#pragma unroll
      for (int q = 0; q < kMaxInlineSeg; ++q) {
        const bool in = s0 + q < n_seg;
        const int sg = in ? s0 + q : s0;
        pm[q] = in ? __ldcg(pml0 + sg * 2 * kHeads + h) : -INFINITY;
        pl[q] = __ldcg(pml0 + sg * 2 * kHeads + kHeads + h);
        const float4* src = reinterpret_cast<const float4*>(po0 + (size_t)sg * kHeads * kHeadDim);
        px[q][0] = __ldcg(src);
        px[q][1] = __ldcg(src + 1);
      }
      float Mn = M;
#pragma unroll
      for (int q = 0; q < kMaxInlineSeg; ++q) Mn = fmaxf(Mn, pm[q]);
      const float base = (Mn == -INFINITY) ? 0.f : Mn;
      const float sc = exp2f(M - base);         // rescale what was merged so far
      L *= sc;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= sc;
#pragma unroll
      for (int q = 0; q < kMaxInlineSeg; ++q) {
        const float wt = exp2f(pm[q] - base);
        L += wt * pl[q];
        acc[0] += wt * px[q][0].x; acc[1] += wt * px[q][0].y;
        acc[2] += wt * px[q][0].z; acc[3] += wt * px[q][0].w;
        acc[4] += wt * px[q][1].x; acc[5] += wt * px[q][1].y;
        acc[6] += wt * px[q][1].z; acc[7] += wt * px[q][1].w;
      }
      M = Mn;
    }
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      pk[e] = pack_bf16(L > 0.f ? acc[2 * e] / L : 0.f, L > 0.f ? acc[2 * e + 1] / L : 0.f);
    *outp = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}


}  // namespace sparda

// The baseline, query-driven selector that SparDA replaces (bittide thread, the paragraph on
// the standard selector; 10100 "先把痛点讲透"): every query head of a GQA group scores every
// compressed key, each head's scores go through a softmax over the windows, the per-head
// probabilities are summed over the group, and the sums are max-pooled onto blocks for the
// same top-k as the Forecast selector. Built as the comparison point for the selector A/B,
// engineered like the Forecast selector: the compressed keys are read from HBM once, and no
// per-head score leaves the chip.
//
// One thread-block cluster of NC CTAs per sequence-group (NC = 1 .. 8, chosen so that the
// clusters fill the GPU and each CTA's share of the windows fits in shared memory). CTA r of
// the cluster owns a contiguous range of 64-window tiles:
//   * a producer warp streams its tiles by TMA (one 64 x 128 bf16 box pair, 128-byte
//     swizzle) into a ring of full/empty mbarriers;
//   * two groups of four consumer warps take alternate tiles; warp w of a group computes the
//     logits of windows 16w .. 16w+15 for the group's 16 heads on m16n8k16 bf16 MMAs
//     (exp2 domain, scale log2(e)/sqrt(d)), keeps them in shared memory (float32, 16 heads x
//     the CTA's windows) and folds them into a running per-head (max, sum of exp2);
//   * the CTAs exchange their per-head (max, sum) through distributed shared memory, so every
//     CTA holds each head's softmax normaliser over all windows;
//   * each CTA forms s[i] = sum_h exp2(z[h][i] - M_h) / L_h for its windows, takes the score of
//     the window just before its range from the previous CTA (distributed shared memory),
//     max-pools windows 4j-1 .. 4j+3 onto its blocks and writes them to the workspace;
//   * after a cluster barrier (release / acquire), CTA 0 runs the exact top-k (topk.cuh).
// The bytes moved per sequence-group are the compressed keys once, the queries, the block
// scores and the selection: those of the Forecast selector plus the 16 query heads.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace sparda {

constexpr int kMhTile = 64;                                   // windows per tile
constexpr int kMhGroupWarps = 4;
constexpr int kMhConsumerWarps = 2 * kMhGroupWarps;
constexpr int kMhThreads = (kMhConsumerWarps + 1) * 32;       // + producer warp
constexpr int kMhStages = 4;                                  // even: one consumer group per stage
static_assert(kMhStages % 2 == 0, "each ring stage must belong to one consumer group");
constexpr int kMhMaxCluster = 8;
constexpr int kMhMaxTilesPerCta = 32;                         // 2048 windows of logits per CTA

int multihead_tiles(int w_cap) { return (w_cap + kMhTile - 1) / kMhTile; }

namespace {

__device__ __forceinline__ uint32_t mh_swz(const uint8_t* tile, int r, int chunk) {
  return smem_addr(tile + (chunk >> 3) * (kBlockBytes / 2) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mh_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kMhConsumerWarps * 32) : "memory");
}

// (m1, l1) + (m2, l2) of the same head: one softmax normaliser (sum of exp2(x - m)) over both.
__device__ __forceinline__ float2 lse_combine(float2 x, float2 y) {
  const float M = fmaxf(x.x, y.x);
  if (M == -INFINITY) return make_float2(-INFINITY, 0.f);
  return make_float2(M, x.y * exp2f(x.x - M) + y.y * exp2f(y.x - M));
}

struct MhLayout {
  int zstride;                   // floats per head row of logits (tiles x 64 + 8)
  size_t ring, z, s, stat, red, misc, topk, total;
};

__host__ __device__ inline MhLayout mh_layout(int tiles_per_cta) {
  MhLayout L;
  L.zstride = tiles_per_cta * kMhTile + 8;   // = 8 (mod 32): conflict-free float2 stores
  L.ring = 1024;
  L.z = L.ring + (size_t)kMhStages * kBlockBytes;
  L.s = L.z + (size_t)kHeads * L.zstride * 4;
  L.stat = L.s + ((size_t)tiles_per_cta * kMhTile + 4) * 4;
  L.stat = (L.stat + 15) & ~(size_t)15;
  L.red = L.stat + kHeads * 8;
  L.misc = L.red + (size_t)kMhConsumerWarps * kHeads * 8;
  L.topk = L.misc + 256;                          // misc: 1 + 16 + 16 floats
  L.total = L.topk + sizeof(TopkShared) + 1024;   // + alignment slack of the dynamic base
  return L;
}

}  // namespace

__global__ void __launch_bounds__(kMhThreads, 1) multihead_select_kernel(const MultiheadArgs a,
                                                                        const __grid_constant__ CUtensorMap mck) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const MhLayout Ly = mh_layout(a.tiles_per_cta);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMhStages;
  uint8_t* ring = smem + Ly.ring;
  float* z = reinterpret_cast<float*>(smem + Ly.z);                 // [16][zstride]
  float* s = reinterpret_cast<float*>(smem + Ly.s);                 // [1 + windows]: s[0] halo
  float2* stat = reinterpret_cast<float2*>(smem + Ly.stat);         // this CTA's (max, sum) per head
  float2* red = reinterpret_cast<float2*>(smem + Ly.red);           // [8 warps][16 heads]
  float* misc = reinterpret_cast<float*>(smem + Ly.misc);           // [0]: last window score; [1..16]: M; [17..32]: 1/L
  TopkShared& sh = *reinterpret_cast<TopkShared*>(smem + Ly.topk);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int ncl = a.cluster;
  const int bg = blockIdx.x / ncl;
  const int T = a.seq_len[bg / a.G];
  const bool valid = T >= 1 && T <= a.max_ctx;
  if (!valid && rank == 0 && tid == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
  const int W = valid ? num_windows(T - 1) : 0;
  const int nb = valid ? (T - 1) / kBlock + 1 : 0;
  const int n_used = (W + kMhTile - 1) / kMhTile;                   // tiles with a window
  const int tpr = (n_used + ncl - 1) / ncl;
  const int tl0 = min((int)rank * tpr, n_used), tl1 = min(tl0 + tpr, n_used);
  const int n_my = tl1 - tl0;
  const int w0 = tl0 * kMhTile;                                     // first window of this CTA

  if (tid == 0) {
    for (int i = 0; i < kMhStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMhGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kMhConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mck);
      for (int it = 0; it < n_my; ++it) {
        const int stage = it % kMhStages;
        if (it >= kMhStages && !mbar_wait(&empty[stage], ((it / kMhStages) & 1) ^ 1, a.err)) break;
        const int row = bg * a.W_cap + (tl0 + it) * kMhTile;
        uint8_t* dst = ring + stage * kBlockBytes;
        mbar_arrive_expect_tx(&full[stage], kBlockBytes);
        tma_load_2d(dst, &mck, 0, row, &full[stage]);
        tma_load_2d(dst + kBlockBytes / 2, &mck, 64, row, &full[stage]);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int grp = warp / kMhGroupWarps, wq = warp % kMhGroupWarps;
    const int g = lane >> 2, cq = lane & 3;
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
    const float sl2 = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    float2 st0 = make_float2(-INFINITY, 0.f), st1 = make_float2(-INFINITY, 0.f);   // heads g, g+8
    bool ok = true;
    for (int it = 0; it < n_my; ++it) {
      if ((it & 1) != grp) continue;
      const int stage = it % kMhStages;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (it / kMhStages) & 1, a.err));
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (ok) {
        const uint8_t* tile = ring + stage * kBlockBytes;
        const int r = 16 * wq + (lane & 7) + ((lane >> 4) << 3);
        const int hi = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(mh_swz(tile, r, 2 * ks + hi), b0, b1, b2, b3);
          mma_16816(sc[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
          mma_16816(sc[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mh_arrive(&empty[stage]);
      // logits of windows il .. il+1 (local), heads g and g+8; windows past W are -inf
      float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int il = it * kMhTile + 16 * wq + 8 * nt + 2 * cq;
        const int ig = w0 + il;
        const float v0 = (ok && ig < W) ? sc[nt][0] * sl2 : -INFINITY;
        const float v1 = (ok && ig + 1 < W) ? sc[nt][1] * sl2 : -INFINITY;
        const float v2 = (ok && ig < W) ? sc[nt][2] * sl2 : -INFINITY;
        const float v3 = (ok && ig + 1 < W) ? sc[nt][3] * sl2 : -INFINITY;
        *reinterpret_cast<float2*>(z + (size_t)g * Ly.zstride + il) = make_float2(v0, v1);
        *reinterpret_cast<float2*>(z + (size_t)(g + 8) * Ly.zstride + il) = make_float2(v2, v3);
        sc[nt][0] = v0; sc[nt][1] = v1; sc[nt][2] = v2; sc[nt][3] = v3;
        m0 = fmaxf(m0, fmaxf(v0, v1));
        m1 = fmaxf(m1, fmaxf(v2, v3));
      }
      const float b0 = m0 == -INFINITY ? 0.f : m0, b1 = m1 == -INFINITY ? 0.f : m1;
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        l0 += exp2f(sc[nt][0] - b0) + exp2f(sc[nt][1] - b0);
        l1 += exp2f(sc[nt][2] - b1) + exp2f(sc[nt][3] - b1);
      }
      st0 = lse_combine(st0, make_float2(m0, l0));
      st1 = lse_combine(st1, make_float2(m1, l1));
    }
    // this CTA's per-head (max, sum): over the 4 lanes of a row, then over the 8 warps
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      st0 = lse_combine(st0, make_float2(__shfl_xor_sync(0xffffffffu, st0.x, o), __shfl_xor_sync(0xffffffffu, st0.y, o)));
      st1 = lse_combine(st1, make_float2(__shfl_xor_sync(0xffffffffu, st1.x, o), __shfl_xor_sync(0xffffffffu, st1.y, o)));
    }
    if (cq == 0) {
      red[warp * kHeads + g] = st0;
      red[warp * kHeads + g + 8] = st1;
    }
    consumers_sync();
    if (tid < kHeads) {
      float2 acc = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int w = 0; w < kMhConsumerWarps; ++w) acc = lse_combine(acc, red[w * kHeads + tid]);
      stat[tid] = acc;
    }
  }
  cluster_sync();                                               // #1: every CTA's stat is set

  // every head's normaliser over the whole cluster
  if (tid < kHeads) {
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int r = 0; r < ncl; ++r) acc = lse_combine(acc, ld_cluster_f2(&stat[tid], (uint32_t)r));
    misc[1 + tid] = acc.x == -INFINITY ? 0.f : acc.x;
    misc[17 + tid] = acc.y > 0.f ? 1.f / acc.y : 0.f;
  }
  __syncthreads();
  // s[i] = sum_h exp2(z[h][i] - M_h) / L_h over this CTA's windows (-inf past W, for the pool)
  const int nw = n_my * kMhTile;
  for (int il = tid; il < nw; il += kMhThreads) {
    float v = -INFINITY;
    if (w0 + il < W) {
      v = 0.f;
#pragma unroll
      for (int h = 0; h < kHeads; ++h) v += exp2f(z[(size_t)h * Ly.zstride + il] - misc[1 + h]) * misc[17 + h];
    }
    s[1 + il] = v;
  }
  __syncthreads();
  if (tid == 0) misc[0] = nw > 0 ? s[nw] : -INFINITY;          // the last window, for the next CTA
  cluster_sync();                                               // #2: every CTA's last window is set

  // max-pool: this CTA's blocks are those whose first full window (4j) lies in its range; the
  // CTA with the last used tile also takes the blocks past it (no window: -inf, or the forced
  // tail). Window 4j-1 of its first block comes from the previous CTA.
  if (tid == 0) s[0] = (rank > 0 && n_my > 0) ? ld_cluster_f(&misc[0], rank - 1) : -INFINITY;
  __syncthreads();
  {
    const int j0 = w0 / kWinPerBlock;
    const bool last = (n_my > 0 && tl1 == n_used) || (n_used == 0 && rank == 0);
    const int j1 = last ? nb : min(nb, (w0 + nw) / kWinPerBlock);
    float* S = a.block_scores + (size_t)bg * a.nb_cap;
    for (int j = j0 + tid; j < j1; j += kMhThreads) {
      float m = -INFINITY;
#pragma unroll
      for (int d = -1; d <= 3; ++d) {
        const int il = kWinPerBlock * j + d - w0;               // local window, -1 = the halo
        if (il >= -1 && il < nw) m = fmaxf(m, s[1 + il]);
      }
      S[j] = m;
    }
  }
  cluster_sync();                                               // #3: every block score is written
  if (rank == 0 && warp < kMhConsumerWarps)
    topk_select(a.block_scores + (size_t)bg * a.nb_cap, a.idx + (size_t)bg * (a.topk + 2), a.cnt + bg, a.topk,
                a.max_ctx, T, sh);
}

namespace {
int mh_sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 152;
  }
  return n[dev];
}
}  // namespace

// Cluster size for a launch: the fewest CTAs whose shared memory holds a (sequence, group)'s
// logits, raised (in powers of two, up to 8) while the clusters of all groups still fit the
// GPU in one wave.
int multihead_cluster_size(int n_tiles_cap, int bg_count) {
  int nc = 1;
  while (nc < kMhMaxCluster && (n_tiles_cap + nc - 1) / nc > kMhMaxTilesPerCta) nc *= 2;
  while (nc < kMhMaxCluster && 2 * nc * bg_count <= mh_sm_count()) nc *= 2;
  return nc;
}

size_t multihead_smem_bytes(int tiles_per_cta) { return mh_layout(tiles_per_cta).total; }

void launch_multihead_select(const MultiheadArgs& a, const CUtensorMap& mck, int bg_count, cudaStream_t s) {
  const size_t smem = multihead_smem_bytes(a.tiles_per_cta);
  cudaFuncSetAttribute(multihead_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.cluster * bg_count);
  cfg.blockDim = dim3(kMhThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, multihead_select_kernel, a, mck);
}

}  // namespace sparda

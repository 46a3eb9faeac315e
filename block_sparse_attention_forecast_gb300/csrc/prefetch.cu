// The offload gather (bittide thread: the next layer's blocks are fetched from CPU memory on
// a separate CUDA stream while the current layer computes; techwalker section 三: a
// persistent kernel with a small, fixed set of copy CTAs reads host memory directly through
// unified virtual addressing, 16 CTAs below batch 32 and 32 from batch 32 on).
//
// A fixed grid of n_ctas CTAs walks the (sequence, group, slot) items with a grid stride.
// Each item is one selected block that lives only in host memory: its 16 KiB of K and
// 16 KiB of V are read over the host link with 16-byte non-caching loads and written to the
// item's staging slot in device memory. Block 0 and the tail block are skipped: the
// attention reads them from the hot buffers.
//
// A copy CTA is small -- 128 threads and no shared memory, each keeping sixteen 16-byte
// loads (32 KiB per CTA) in flight -- so that it fits on an SM beside one CTA of the persistent
// select or attention kernels, which run while the gather streams; a larger copy CTA would
// keep those kernels' CTAs off its SM for the whole gather.
#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kGatherThreads = 128;
constexpr int kVecPerBlock = kBlockBytes / 16;                 // 1024 16-byte vectors
constexpr int kInFlight = 8;                                   // per tensor (K and V) per pass
constexpr int kPasses = kVecPerBlock / (kGatherThreads * kInFlight);   // 2

__device__ __forceinline__ uint4 ld_host(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copies one 64-token block of K and V (16 KiB each) from host memory to device memory, by
// the 128 threads of a copy CTA: kPasses rounds of kInFlight 16-byte loads per tensor and
// thread, all issued before their stores.
__device__ __forceinline__ void copy_block(const __nv_bfloat16* hk, const __nv_bfloat16* hv, size_t src,
                                           __nv_bfloat16* dk_base, __nv_bfloat16* dv_base, size_t dst, int t) {
  const uint4* sk = reinterpret_cast<const uint4*>(hk + src);
  const uint4* sv = reinterpret_cast<const uint4*>(hv + src);
  uint4* dk = reinterpret_cast<uint4*>(dk_base + dst);
  uint4* dv = reinterpret_cast<uint4*>(dv_base + dst);
#pragma unroll
  for (int pass = 0; pass < kPasses; ++pass) {
    const int base = pass * kGatherThreads * kInFlight + t;
    uint4 rk[kInFlight], rv[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      rk[u] = ld_host(sk + base + u * kGatherThreads);
      rv[u] = ld_host(sv + base + u * kGatherThreads);
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      dk[base + u * kGatherThreads] = rk[u];
      dv[base + u * kGatherThreads] = rv[u];
    }
  }
}

__global__ void __launch_bounds__(kGatherThreads) prefetch_kernel(const PrefetchArgs a) {
  const int n_items = a.B * a.G * a.kslots;
  const int t = threadIdx.x;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int bg = item / a.kslots;
    const int s = item - bg * a.kslots;
    const int T = a.seq_len[bg / a.G];
    if (T < 1 || T > a.max_ctx) {
      if (t == 0 && s == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
      continue;
    }
    if (s >= min(a.cnt[bg], a.kslots)) continue;
    const int tb = (T - 1) / kBlock;
    const int j = a.idx[(size_t)bg * a.kslots + s];
    if (j == 0 || j == tb) continue;
    if (j < 0 || j > tb) {
      if (t == 0) atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
      continue;
    }
    copy_block(a.hk, a.hv, ((size_t)bg * a.max_ctx + (size_t)j * kBlock) * kHeadDim, a.sk, a.sv,
               ((size_t)bg * a.kslots + s) * kBlock * kHeadDim, t);
  }
}

void launch_prefetch(const PrefetchArgs& a, int n_ctas, cudaStream_t s) {
  prefetch_kernel<<<n_ctas, kGatherThreads, 0, s>>>(a);
}

// ------------------------------------------------------------------ cross-step block cache
// An extension beyond the pages: each (sequence, group) of an offloaded layer keeps the blocks
// it gathered at earlier steps in n_cache slots of HBM, and only blocks that are not there
// yet cross the host link. cache_blocks[bg][c] names the block held in slot c (-1: none).
//
// cache_gather_kernel: one CTA per (sequence, group). Its first warp assigns the slots: a
// selected block (not block 0 or the tail block, which the hot ring supplies) already held in
// a slot keeps it (a hit); every other selected block (a miss) takes, in order of its position
// in idx, the lowest slot whose block is not selected at this step; fetch[bg][c] = the block
// slot c must receive (-1: none), slot[bg][s] = the cache slot of idx entry s (-1 for block 0,
// the tail block and padding). After a CTA barrier the CTA copies the group's misses on
// kCacheStreams copy streams of 128 threads. Only this CTA reads or writes the group's slot
// table, so the assignment and the copies need no ordering across CTAs, and the gather is one
// launch: a separate assignment launch ahead of the copies stalled every layer's gather stream
// (the offloaded step with every block a miss took 25 ms instead of 20).
constexpr int kCacheMaxSlots = 128;                 // 4 words of 32 lanes (n_cache at most)
static_assert(kCacheMaxSlots == 4 * 32, "the assignment keeps each lane's slots in four words");
constexpr int kCacheStreams = 4;
constexpr int kCacheThreads = kCacheStreams * kGatherThreads;   // 512

// The slot assignment of (sequence, group) bg by one warp.
__device__ __forceinline__ void assign_group(const CacheArgs& a, int bg, int lane) {
  const int T = a.seq_len[bg / a.G];
  const bool valid = T >= 1 && T <= a.max_ctx;
  if (!valid && lane == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
  const int tb = valid ? (T - 1) / kBlock : -1;
  const int n = valid ? min(max(a.cnt[bg], 0), a.kslots) : 0;
  int32_t* cb = a.cache_blocks + (size_t)bg * a.n_cache;
  // the blocks held in this lane's slots (c = lane + 32m)
  int held[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int c = lane + 32 * m;
    held[m] = c < a.n_cache ? cb[c] : -2;
  }
  // the selected blocks that need a slot (idx entries s = lane, lane + 32)
  int js[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    int j = -1;
    if (s < n) {
      j = a.idx[(size_t)bg * a.kslots + s];
      if (j < 0 || j > tb) {
        atomicOr(a.err, SPARDA_DEV_BAD_INDEX);
        j = -1;
      } else if (j == 0 || j == tb) {
        j = -1;                                     // the hot ring holds it
      }
    }
    js[h] = j;
  }
  // hits: the slot already holding each selected block; keep[m] bit lane: slot selected
  unsigned keep[4] = {0u, 0u, 0u, 0u};
  int myslot[2] = {-1, -1};
  int n_miss_before = 0, my_miss_rank[2] = {-1, -1};
  for (int s = 0; s < a.kslots; ++s) {               // warp-uniform loop over idx entries
    const int j = __shfl_sync(0xffffffffu, js[s >> 5], s & 31);
    if (j < 0) continue;
    int slot = -1;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const unsigned b = __ballot_sync(0xffffffffu, held[m] == j);
      if (b && slot < 0) {
        slot = 32 * m + __ffs(b) - 1;
        keep[m] |= 1u << (__ffs(b) - 1);
      }
    }
    if ((s & 31) == lane) {
      if (slot >= 0) myslot[s >> 5] = slot;
      else my_miss_rank[s >> 5] = n_miss_before;
    }
    if (slot < 0) ++n_miss_before;
  }
  // the r-th miss takes the r-th slot not kept (slots past n_cache are never free)
  unsigned freem[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int lim = a.n_cache - 32 * m;
    const unsigned in = lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : ((1u << lim) - 1u));
    freem[m] = in & ~keep[m];
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (my_miss_rank[h] >= 0) {
      int r = my_miss_rank[h], slot = -1;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int pc = __popc(freem[m]);
        if (slot < 0 && r < pc) {
          unsigned x = freem[m];
          for (int q = 0; q < r; ++q) x &= x - 1;  // drop the r lowest free slots
          slot = 32 * m + __ffs(x) - 1;
        } else if (slot < 0) {
          r -= pc;
        }
      }
      myslot[h] = slot;                             // n_cache >= topk: a free slot exists
    }
  }
  __syncwarp();
  // outputs: fetch list cleared, then the misses' slots; the slot of every idx entry
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int c = lane + 32 * m;
    if (c < a.n_cache) a.fetch[(size_t)bg * a.n_cache + c] = -1;
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    if (s < a.kslots) a.slot[(size_t)bg * a.kslots + s] = js[h] >= 0 ? myslot[h] : -1;
    if (js[h] >= 0 && my_miss_rank[h] >= 0 && myslot[h] >= 0) {
      a.fetch[(size_t)bg * a.n_cache + myslot[h]] = js[h];
      cb[myslot[h]] = js[h];
    }
  }
  if (a.stats && lane == 0) {
    atomicAdd(a.stats, (unsigned long long)(__popc(keep[0]) + __popc(keep[1]) + __popc(keep[2]) + __popc(keep[3])));
    atomicAdd(a.stats + 1, (unsigned long long)n_miss_before);
  }
}

__global__ void __launch_bounds__(kCacheThreads) cache_gather_kernel(const CacheArgs a) {
  const int bg = blockIdx.x;
  if (threadIdx.x < 32) assign_group(a, bg, threadIdx.x);
  __syncthreads();                                 // the fetch list is written
  const int stream = threadIdx.x / kGatherThreads, t = threadIdx.x % kGatherThreads;
  for (int c = stream; c < a.n_cache; c += kCacheStreams) {
    const size_t item = (size_t)bg * a.n_cache + c;
    const int j = a.fetch[item];
    if (j < 0) continue;
    copy_block(a.hk, a.hv, ((size_t)bg * a.max_ctx + (size_t)j * kBlock) * kHeadDim, a.ck_cache, a.cv_cache,
               item * kBlock * kHeadDim, t);
  }
}

void launch_cache_gather(const CacheArgs& a, cudaStream_t s) {
  cache_gather_kernel<<<a.B * a.G, kCacheThreads, 0, s>>>(a);
}

}  // namespace sparda

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
    const size_t src = ((size_t)bg * a.max_ctx + (size_t)j * kBlock) * kHeadDim;
    const size_t dst = ((size_t)bg * a.kslots + s) * kBlock * kHeadDim;
    const uint4* sk = reinterpret_cast<const uint4*>(a.hk + src);
    const uint4* sv = reinterpret_cast<const uint4*>(a.hv + src);
    uint4* dk = reinterpret_cast<uint4*>(a.sk + dst);
    uint4* dv = reinterpret_cast<uint4*>(a.sv + dst);
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
}

void launch_prefetch(const PrefetchArgs& a, int n_ctas, cudaStream_t s) {
  prefetch_kernel<<<n_ctas, kGatherThreads, 0, s>>>(a);
}

}  // namespace sparda
